#!/usr/bin/env python
"""Benchmark of the trellis decode-and-multiply path on one GB300 (sm_103a).

Default workload: the dense gated MLP at decode, 5120 -> 17408 -> 5120 with
gate 2-bit, up 3-bit and down 3-bit trellis codes, one token.  One step is one
full MLP application (input rotations, two trellis GEMV launches, the fused
SiLU-gate middle, the output rotation) on device-resident inputs.

Prints ONE JSON line.  `value` is decode GEMV throughput in GB/s of
algorithmic bytes (code words + side vectors + activations) per step;
`roofline` rates the dominant kernel (the trellis GEMV) against the measured
HBM copy bandwidth and `roofline_issue` against the instruction-issue bound
of its decode; `e2e` is the same metric through the C ABI with host buffers
and the copies inside the timed region; `cpu_baseline` is the CPU oracle on a
bounded sample of the same workload.  The `prefill` object holds the other
half of the metric, measured in the same process: the tcgen05 prefill GEMM at
2048 tokens, 5120 -> 17408 at 3 bits, in TFLOP/s against the tensor peak.
The timed region (K steps) is repeated and its median reported.

Other workloads print the same line for their own shapes and metric:
--workload linear512 | sweep (--m, --shape) | moe (--m, --halves, --shared)
| prefill (TFLOP/s; --shape, --fp8) | encode (weights/s); --norm adds the
MLP's input RMSNorm, --rounding e4m3 the EXLR8 codebook rounding, --fp8 the
prefill on FP8 tensor cores (E4M3 weights, per-token E4M3 activations).
--impl reference times the CPU oracle on a bounded sample of the same workload.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gemm_trellis_tile_gb300 import synthetic as S  # noqa: E402
from gemm_trellis_tile_gb300 import workloads as WL  # noqa: E402

L2_FALLBACK_BYTES = 129 * 1024 * 1024

# One metric string per kind of line, the same in both arms.
METRIC_DECODE = "decode GEMV compressed-weight GB/s vs HBM peak (\u00b5s/layer); prefill TFLOP/s"
METRIC_PREFILL = "prefill TFLOP/s (2*M*in*out per step)"
METRIC_ENCODE = "trellis encode weights/s (Viterbi search, whole tiles)"
BYTES_NOTE = "algorithmic bytes: code words + side vectors + activations"

# The prefill half of the default line: 2048 tokens through 5120 -> 17408 at 3 bits.
PREFILL_DEFAULT = dict(m=2048, shape="5120x17408")

# A prefill region at least this long is compared with the sustained tensor peak.
SUSTAINED_REGION_S = 0.5

# Timed-region repeats: at least this many, and enough for this much device time.
MIN_REPEATS = 5
MAX_REPEATS = 200
REPEAT_SECONDS = 0.25

# DRAM bytes per contraction launch (dram__bytes_read.sum + dram__bytes_write.sum
# from one ncu capture of this kernel, averaged over the step's launches), by
# workload at M=1; None where no capture of the current kernel exists.
GEMV_TRAFFIC_BYTES = {
    "dense gated MLP 5120->17408->5120, gate 2-bit / up 3-bit / down 3-bit, M=1": 44.71e6,
}
# The same for one prefill GEMM launch (the trellis_gemm kernel alone).
PREFILL_TRAFFIC_BYTES = {
    "prefill GEMM 5120x17408 3-bit, M=2048 tokens": 125.26e6,
    "prefill GEMM 5120x17408 3-bit, M=2048 tokens, FP8 tensor cores (E4M3 weights, "
    "per-token E4M3 activations)": 103.69e6,
}


# Instruction mix of the trellis GEMV per decoded weight, by workload at M=1:
# lane-instructions (warp instructions x 32) per weight over the step's
# contraction launches, from one ncu capture of this kernel
# (smsp__inst_executed.sum and smsp__inst_executed_pipe_alu.sum); None where no
# capture of the current kernel exists.
GEMV_ISSUE_MIX = {
    "dense gated MLP 5120->17408->5120, gate 2-bit / up 3-bit / down 3-bit, M=1":
        {"issue": 5.55, "alu": 2.59},
}
# Per SM sub-partition and clock: one warp instruction issued, 16 lanes of the
# integer ALU pipe (a warp instruction holds it for two cycles: ncu's
# sm__pipe_alu_cycles_active / sm__inst_executed_pipe_alu = 2.0 on this kernel).
ISSUE_LANES_PER_CLK = 32
ALU_LANES_PER_CLK = 16
SMSP_PER_SM = 4


def issue_roofline(name, weights_per_s, sms, clocks):
    """The GEMV against the instruction-issue bound of its decode: with I lane-
    instructions per weight (the capture's mix), an SM issues at most
    4 x 32 / I weights per clock, and the ALU pipe allows 4 x 16 / A (A = ALU
    lane-instructions per weight); the bound is the smaller, at the median SM
    clock sampled during the timed region (else the maximum clock)."""
    mix = GEMV_ISSUE_MIX.get(name) if name else None
    if mix is None:
        return None
    peaks, _ = measured_peaks()
    mhz = (clocks or {}).get("sm_mhz") or float(peaks.get("sm_max_mhz", 2070.0))
    f = sms * SMSP_PER_SM * mhz * 1e6
    by_issue = f * ISSUE_LANES_PER_CLK / mix["issue"]
    by_alu = f * ALU_LANES_PER_CLK / mix["alu"]
    peak = min(by_issue, by_alu)
    return {"bound": "alu", "pipe": "issue" if by_issue <= by_alu else "alu",
            "kernel": "trellis_gemv", "achieved": weights_per_s / 1e12, "peak": peak / 1e12,
            "unit": "T weights/s", "frac": weights_per_s / peak,
            "lane_instr_per_weight": mix["issue"], "alu_lane_instr_per_weight": mix["alu"],
            "peak_source": "derived: %d SMs x 4 sub-partitions x %.0f MHz x min(32 issue "
                           "lanes / %.2f, 16 ALU lanes / %.2f) lane-instructions per weight "
                           "(ncu counters of this kernel)" % (sms, mhz, mix["issue"],
                                                              mix["alu"])}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=4000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", default="escha", choices=["escha", "reference"])
    p.add_argument("--workload", default="mlp",
                   choices=["mlp", "linear512", "sweep", "prefill", "moe", "encode"])
    p.add_argument("--m", type=int, default=1, help="tokens per step")
    p.add_argument("--shape", default=None, help="in x out (sweep: default 5120x10240; "
                   "prefill: default 5120x17408)")
    p.add_argument("--norm", action="store_true",
                   help="mlp: input RMSNorm (weight stored as w - 1) fused into the input rotations")
    p.add_argument("--shared", action="store_true",
                   help="moe: add a shared expert (3-bit) that every token uses with weight 1")
    p.add_argument("--halves", action="store_true",
                   help="moe: experts stored by halves of 128 intermediate channels, a width "
                        "per half for gate/up and per expert for down, pointer tables")
    p.add_argument("--rounding", default="fp16", choices=["fp16", "e4m3"],
                   help="codebook rounding: fp16 values, or the EXLR8 E4M3 variant")
    p.add_argument("--fp8", action="store_true",
                   help="prefill: kind::f8f6f4 GEMM on E4M3 weights and per-token E4M3 "
                        "activations (implies --rounding e4m3)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-prefill", action="store_true",
                   help="default line: leave out the prefill half of the metric")
    p.add_argument("--repeats", type=int, default=0,
                   help="repeats of the K-step timed region (median reported); 0 = automatic")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    return p.parse_args()


# ---------------------------------------------------------------- environment

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class Replicas:
    """N independent replicas of the workload, one process per GPU (launched by
    torchrun): each rank builds its own rank-seeded weight sets and inputs, the
    timed region has a barrier on both sides, and its time is the slowest
    rank's.  Nothing is exchanged on the data path.  With world == 1 there is
    no process group and the barriers and reduction do nothing."""

    def __init__(self, rank, world, local, backend="nccl"):
        self.rank, self.world = rank, world
        self.dist = None
        if world > 1:
            import torch.distributed as dist
            if backend == "nccl":
                import torch
                torch.cuda.set_device(local)
            dist.init_process_group(backend)
            self.dist = dist

    def seed(self, base, inst=0):
        """Seed of weight set `inst` on this rank (distinct across ranks and sets)."""
        return base + 7919 * inst + 1000003 * self.rank

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()

    def slowest(self, ms, device):
        """The largest of the ranks' times; every rank gets it."""
        if self.dist is None:
            return ms
        import torch
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def emit(self, line):
        """The job's one JSON line, from rank 0."""
        if self.rank == 0:
            print(json.dumps(line), flush=True)

    def close(self):
        if self.dist is not None:
            self.dist.destroy_process_group()
            self.dist = None


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def repeats_for(first_ms, asked=0):
    """Repeats of a timed region whose first run took `first_ms`."""
    if asked > 0:
        return asked
    want = int(np.ceil(REPEAT_SECONDS * 1e3 / max(first_ms, 1e-3)))
    return max(MIN_REPEATS, min(MAX_REPEATS, want))


def median_region(run, rep, dev, asked=0):
    """Time `run()` (K steps launched on the current stream) between CUDA
    events, a barrier and a synchronize on both sides, repeatedly; returns
    (median ms, repeats, min ms, max ms), each repeat the slowest rank's."""
    import torch

    def once():
        rep.barrier()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        run()
        t1.record()
        torch.cuda.synchronize()
        rep.barrier()
        return rep.slowest(t0.elapsed_time(t1), dev)
    times = [once()]
    for _ in range(repeats_for(times[0], asked) - 1):
        times.append(once())
    return statistics.median(times), len(times), min(times), max(times)


class ClockSampler:
    """nvidia-smi clock/throttle samples taken while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", "escha_clocks_%d_%d.csv" % (os.getpid(), gpu_index))

    def start(self):
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- workloads

def workload_spec(args):
    """Layers of one step as (in, out, bits), a description and the codebook rounding."""
    spec = _workload_spec(args)
    spec["rounding"] = args.rounding
    spec["fp8"] = bool(args.fp8 and spec["kind"] == "prefill")
    if spec["fp8"]:
        spec["rounding"] = "e4m3"
        spec["name"] += ", FP8 tensor cores (E4M3 weights, per-token E4M3 activations)"
        return spec
    if args.rounding == "e4m3":
        spec["name"] += ", E4M3 codebook rounding"
    if args.norm and spec["kind"] == "mlp":
        spec["norm"] = True
        spec["name"] += ", input RMSNorm"
    return spec


def _workload_spec(args):
    if args.workload == "mlp":
        layers = WL.mlp_layers(5120, 17408, (2, 3, 3))
        name = "dense gated MLP 5120->17408->5120, gate 2-bit / up 3-bit / down 3-bit, M=%d" % args.m
        return dict(kind="mlp", layers=layers, name=name, seed=S.seed_for(1))
    if args.workload == "linear512":
        return dict(kind="linear", layers=[(512, 512, 2)], seed=S.seed_for(0),
                    name="single linear 512x512 2-bit, M=%d" % args.m)
    if args.workload == "moe" and args.halves:
        return dict(kind="moe", halves=True, layers=WL.mlp_layers(6144, 2048, (3, 3, 3)),
                    seed=S.seed_for(3, 2),
                    name="routed MoE 256 experts 6144->2048->6144 stored by halves, gate/up "
                         "2/3/4-bit per half, down 2/3/4-bit per expert, top-8, M=%d" % args.m)
    if args.workload == "moe":
        return dict(kind="moe", layers=WL.mlp_layers(6144, 2048, (3, 3, 3)), seed=S.seed_for(3),
                    shared=args.shared,
                    name="routed MoE 256 experts 6144->2048->6144, 2/3/4-bit per expert, top-8, "
                         "M=%d" % args.m + (", plus a 3-bit shared expert" if args.shared else ""))
    if args.workload == "encode":
        k, n = (int(v) for v in (args.shape or "2048x2048").split("x"))
        bits = 2
        return dict(kind="encode", layers=[(k, n, bits)], seed=S.seed_for(5, k),
                    name="trellis encode (Viterbi, tail-biting) of a %dx%d fp32 W_inner "
                         "~N(0, 1.244^2) at %d bits" % (k, n, bits))
    if args.workload == "prefill":
        k, n = (int(v) for v in (args.shape or "5120x17408").split("x"))
        return dict(kind="prefill", layers=[(k, n, 3)], seed=S.seed_for(4, k),
                    name="prefill GEMM %dx%d 3-bit, M=%d tokens" % (k, n, args.m))
    k, n = (int(v) for v in (args.shape or "5120x10240").split("x"))
    return dict(kind="linear", layers=[(k, n, 2)], seed=S.seed_for(2, k),
                name="decode sweep linear %dx%d 2-bit, M=%d" % (k, n, args.m))


def step_bytes(spec, m):
    return sum(WL.layer_bytes(m, i, o, b) for i, o, b in spec["layers"])


def make_instance(spec, seed):
    rng = np.random.default_rng(seed)
    if spec["kind"] == "mlp":
        hidden, inter = spec["layers"][0][0], spec["layers"][0][1]
        bits = tuple(b for _, _, b in spec["layers"])
        return S.make_mlp(rng, hidden, inter, *bits)
    k, n, b = spec["layers"][0]
    return dict(layer=S.make_linear(rng, k, n, b))


def instance_matrices(spec, inst):
    return [inst["gate"], inst["up"], inst["down"]] if spec["kind"] == "mlp" else [inst["layer"]]


# ---------------------------------------------------------------- CPU oracle leg

def oracle_sample_rate(spec, m, seconds, seed=7):
    """Run the CPU oracle on 128-output column blocks of the workload's matrices
    until `seconds` of work; return (GB/s of algorithmic bytes, effective cores,
    sample description)."""
    from oracle import escha_oracle as O
    mats = instance_matrices(spec, make_instance(spec, spec["seed"]))
    rng = np.random.default_rng(seed)
    done_bytes = 0
    blocks = 0
    t0 = time.perf_counter()
    c0 = time.process_time()
    while True:
        lay = mats[blocks % len(mats)]
        k, n = lay["in_features"], lay["out_features"]
        blk = int(rng.integers(n // 128))
        x = S.make_activations(rng, m, k)
        su = O.fold_scales(lay["rin"], lay["s_in"])
        sv = O.fold_scales(lay["rout"], lay["s_out"])
        O.linear_forward_columns(x, lay["code"], lay["bits"], su, sv, [blk],
                                 rounding=spec["rounding"])
        done_bytes += WL.layer_bytes(m, k, 128, lay["bits"])
        blocks += 1
        if time.perf_counter() - t0 >= seconds:
            break
    wall = time.perf_counter() - t0
    cpu = time.process_time() - c0
    return (done_bytes / wall / 1e9, round(cpu / wall, 2),
            "%d column blocks of 128 outputs (full input depth) across the workload's matrices, "
            "%.1f s" % (blocks, wall))


def run_reference_encode(args, spec):
    """--impl reference for the encoder: the oracle's Viterbi search, a bounded
    number of tiles of the same matrix per step."""
    k, n, bits = spec["layers"][0]
    rng = np.random.default_rng(spec["seed"])
    w = (rng.standard_normal((k, n)) * S.CODEBOOK_STD).astype(np.float32)
    steps = args.steps if args.steps != 4000 else 5
    warm = args.warmup if args.warmup != 50 else 3
    budget = 120.0 / max(1, steps + warm)
    for _ in range(warm):
        encode_oracle_rate(w, bits, min(budget, 2.0))
    t0 = time.perf_counter()
    c0 = time.process_time()
    done = 0.0
    for _ in range(steps):
        done += encode_oracle_rate(w, bits, budget)[3]
    wall = time.perf_counter() - t0
    cores = round((time.process_time() - c0) / wall, 2)
    value = done / wall
    line = {"impl": "reference", "metric": METRIC_ENCODE,
            "value": value, "unit": "weights/s", "n_gpus": args.gpus, "steps": steps,
            "warmup": warm, "ms_per_step": 1e3 * wall / steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": spec["name"]},
            "cpu_baseline": {"value": value, "unit": "weights/s", "cores": cores,
                             "kind": "oracle",
                             "sample": "per step: as many whole tiles as %.0f s allow" % budget},
            "e2e": {"value": value, "unit": "weights/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def prefill_oracle_layer(spec):
    """The prefill workload's first weight set, as the GPU leg builds it."""
    k, n, b = spec["layers"][0]
    return S.make_linear(np.random.default_rng(spec["seed"]), k, n, b)


def prefill_oracle_sample(spec, lay, x, rng):
    """The CPU oracle's prefill layer on one sample: the tokens x through one
    128-column output block of the layer (fp16 or FP8 route); returns its flops."""
    from oracle import escha_oracle as O
    k, n, b = spec["layers"][0]
    su = O.fold_scales(lay["rin"], lay["s_in"])
    sv = O.fold_scales(lay["rout"], lay["s_out"])
    blk = [int(rng.integers(n // 128))]
    if spec["fp8"]:
        O.linear_forward_fp8_columns(x, lay["code"], b, su, sv, blk)
    else:
        O.linear_forward_columns(x, lay["code"], b, su, sv, blk, rounding=spec["rounding"])
    return WL.layer_flops(x.shape[0], k, 128)


def prefill_oracle_rate(spec, m, seconds):
    """(TFLOP/s, cores, sample) of the CPU oracle's prefill layer over `seconds`."""
    lay = prefill_oracle_layer(spec)
    rng = np.random.default_rng(spec["seed"] + 29)
    rows = min(m, 256)
    x = S.make_activations(rng, rows, spec["layers"][0][0])
    t0 = time.perf_counter()
    c0 = time.process_time()
    flops, blocks = 0, 0
    while True:
        flops += prefill_oracle_sample(spec, lay, x, rng)
        blocks += 1
        if time.perf_counter() - t0 >= seconds:
            break
    wall = time.perf_counter() - t0
    return (flops / wall / 1e12, round((time.process_time() - c0) / wall, 2),
            "%d tokens through %d random 128-output column blocks (full input depth), %.1f s"
            % (rows, blocks, wall))


def run_reference_prefill(args, spec):
    """--impl reference for the prefill: the oracle's layer on a bounded sample per step."""
    steps = args.steps if args.steps != 4000 else 5
    warm = args.warmup if args.warmup != 50 else 3
    budget = 120.0 / max(1, steps + warm)
    prefill_oracle_rate(spec, args.m, min(budget, 2.0) * warm)
    t0 = time.perf_counter()
    c0 = time.process_time()
    rates = [prefill_oracle_rate(spec, args.m, budget) for _ in range(steps)]
    wall = time.perf_counter() - t0
    cores = round((time.process_time() - c0) / wall, 2)
    value = statistics.mean(r[0] for r in rates)
    line = {"impl": "reference", "metric": METRIC_PREFILL,
            "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": steps,
            "warmup": warm, "ms_per_step": 1e3 * wall / steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": spec["name"]},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": "per step: " + rates[-1][2]},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_reference(args, spec, rank):
    """--impl reference: the CPU oracle, as it stands, on a bounded sample per step."""
    if rank != 0:
        return 0
    if spec["kind"] == "encode":
        return run_reference_encode(args, spec)
    if spec["kind"] == "prefill":
        return run_reference_prefill(args, spec)
    from oracle import escha_oracle as O
    mats = instance_matrices(spec, make_instance(spec, spec["seed"]))
    rng = np.random.default_rng(11)
    budget = 150.0 / max(1, args.steps + args.warmup)   # seconds per step
    probe = mats[0]
    t0 = time.perf_counter()
    O.decode_columns(probe["code"][:8], probe["bits"], np.arange(128), rounding=spec["rounding"])
    per_ktile = max(1e-6, (time.perf_counter() - t0) / 8)
    ktiles = max(8, int(budget / per_ktile) // 8 * 8)

    def one_step(i):
        lay = mats[i % len(mats)]
        k, n, b = lay["in_features"], lay["out_features"], lay["bits"]
        kt = min(ktiles, k // 16)
        blk = int(rng.integers(n // 128))
        kk = kt * 16
        x = S.make_activations(rng, args.m, kk)
        w = O.decode_columns(lay["code"][:kt], b, np.arange(blk * 128, blk * 128 + 128),
                             rounding=spec["rounding"])
        su = O.fold_scales(lay["rin"][:kk], lay["s_in"][:kk])
        y_pre = O.had_blockwise(x * su) @ w.astype(np.float64)
        _ = O.had_blockwise(y_pre) * O.fold_scales(lay["rout"], lay["s_out"])[blk * 128:blk * 128 + 128]
        return WL.layer_bytes(args.m, kk, 128, b)

    for i in range(args.warmup):
        one_step(i)
    t0 = time.perf_counter()
    c0 = time.process_time()
    total = 0
    for i in range(args.steps):
        total += one_step(i)
    wall = time.perf_counter() - t0
    cores = round((time.process_time() - c0) / wall, 2)
    value = total / wall / 1e9
    depth = min(ktiles, max(lay["in_features"] // 16 for lay in mats))
    sample = ("per step: one 128-output column block of one matrix (cycling through the "
              "workload's matrices), %d k-tiles deep" % depth)
    line = {"impl": "reference", "metric": METRIC_DECODE, "value": value,
            "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * wall / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": spec["name"]},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    if spec["kind"] == "mlp" and not args.no_prefill and args.workload == "mlp":
        pspec = prefill_spec(args)
        pv, pcores, psample = prefill_oracle_rate(pspec, PREFILL_DEFAULT["m"], args.cpu_seconds)
        line["prefill"] = {"workload": pspec["name"], "metric": METRIC_PREFILL, "value": pv,
                           "unit": "TFLOP/s", "dtype": "f64",
                           "cpu_baseline": {"value": pv, "unit": "TFLOP/s", "cores": pcores,
                                            "kind": "oracle", "sample": psample}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU leg

def run_moe(args, spec, rank, world, local):
    """Routed experts at decode: GB/s of the algorithmic bytes of each step's
    distinct routed experts (their code words and side vectors, the shared
    hidden vectors, activations), over 64 cycled seeded routings."""
    import torch
    from gemm_trellis_tile_gb300 import build, escha
    rep = Replicas(rank, world, local)
    build.build()
    escha.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    E, hidden, inter, m = 256, 6144, 2048, args.m
    halves = spec.get("halves", False)
    H = inter // 128
    seed = rep.seed(spec["seed"])
    mspec = (S.make_moe_half_spec if halves else S.make_moe_spec)(seed, E, hidden, inter)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)

    def draw(shape):
        return torch.randint(-32768, 32768, shape, dtype=torch.int16, device=dev, generator=gen)
    t = {k: torch.from_numpy(mspec[k]).to(dev) for k in (
        "rin_hidden", "s_in_hidden", "rout_gate", "s_out_gate", "rout_up", "s_out_up",
        "rin_down", "s_in_down", "rout_hidden", "s_out_hidden")}
    sidevec = (t["rin_hidden"], t["s_in_hidden"], t["rout_gate"], t["s_out_gate"], t["rout_up"],
            t["s_out_up"], t["rin_down"], t["s_in_down"], t["rout_hidden"], t["s_out_hidden"])
    if halves:
        # one allocation per half, as a loader that fetches halves one by one would hold them
        codes = []
        for e in range(E):
            bd = int(mspec["down_bits"][e])
            codes.append((
                [draw((hidden // 16, 8, 16 * int(mspec["gate_bits"][e, h]))) for h in range(H)],
                [draw((hidden // 16, 8, 16 * int(mspec["up_bits"][e, h]))) for h in range(H)],
                [draw((8, hidden // 16, 16 * bd)) for _ in range(H)]))
        tabs = [torch.tensor([[c[part][h].data_ptr() for h in range(H)] for c in codes],
                             dtype=torch.int64, device=dev) for part in range(3)]
        bits_t = [torch.from_numpy(np.ascontiguousarray(mspec[k])).to(dev)
                  for k in ("gate_bits", "up_bits", "down_bits")]
        moe = escha.MoEHalves(hidden, inter, *tabs, *bits_t, *sidevec)
    else:
        codes = []
        for e in range(E):
            b = int(mspec["bits"][e])
            shapes = [(hidden // 16, inter // 16, 16 * b)] * 2 + [(inter // 16, hidden // 16, 16 * b)]
            codes.append(tuple(draw(sh) for sh in shapes))
        moe = escha.MoE(hidden, inter, [c[0] for c in codes], [c[1] for c in codes],
                        [c[2] for c in codes], mspec["bits"], *sidevec)
    moe.set_rounding(spec["rounding"])
    shared_keep = None
    if spec.get("shared"):
        sh = S.make_moe_shared_expert(mspec, bits=3)
        shared_keep = {k: torch.from_numpy(v).to(dev) for k, v in sh.items() if k != "bits"}
        t2 = shared_keep
        moe.set_shared_expert(t2["gate"], t2["up"], t2["down"], 3, t2["rout_gate"],
                              t2["s_out_gate"], t2["rout_up"], t2["s_out_up"], t2["rin_down"],
                              t2["s_in_down"])
    rng = np.random.default_rng(spec["seed"] + 29)
    R = 64
    routes = [S.make_routing(rng, m, E, 8) for _ in range(R)]
    ids_d = [torch.from_numpy(r[0]).to(dev) for r in routes]
    w_d = [torch.from_numpy(r[1]).to(dev) for r in routes]

    def route_bytes(ids):
        tot = WL.side_bytes(hidden, 0) + WL.side_bytes(0, hidden) + 2 * m * 2 * hidden
        for e in sorted(set(ids.reshape(-1).tolist())):
            if halves:
                for h in range(H):
                    tot += WL.code_bytes(hidden, 128, int(mspec["gate_bits"][e, h]))
                    tot += WL.code_bytes(hidden, 128, int(mspec["up_bits"][e, h]))
                tot += WL.code_bytes(inter, hidden, int(mspec["down_bits"][e]))
            else:
                b = int(mspec["bits"][e])
                tot += 2 * WL.code_bytes(hidden, inter, b) + WL.code_bytes(inter, hidden, b)
            tot += 3 * 6 * inter
        if spec.get("shared"):
            tot += 2 * WL.code_bytes(hidden, inter, 3) + WL.code_bytes(inter, hidden, 3) + 3 * 6 * inter
        return tot
    rbytes = [route_bytes(r[0]) for r in routes]
    x_host = torch.from_numpy(S.make_activations(rng, m, hidden)).pin_memory()
    x = x_host.to(dev)
    y = torch.empty((m, hidden), dtype=torch.float16, device=dev)

    def step(i):
        moe.gemv(x, ids_d[i % R], w_d[i % R], y)

    for i in range(max(args.warmup, R)):
        step(i)
    torch.cuda.synchronize()
    if moe.check() != 0:
        raise SystemExit("device error flag set during warm-up")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                for i in range(R):
                    fn(i)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        return g

    def timed(g, reps, sampler=None):
        if sampler is not None:
            sampler.start()
        rep.barrier()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(reps):
            g.replay()
        t1.record()
        torch.cuda.synchronize()
        clk = sampler.stop() if sampler is not None else None
        rep.barrier()
        elapsed = t0.elapsed_time(t1)
        elapsed = rep.slowest(elapsed, dev)
        return elapsed, clk

    reps = max(1, args.steps // R)
    steps = reps * R
    g_main = capture(step)
    ms, clocks = timed(g_main, reps, ClockSampler(dev.index if dev.index is not None else 0))

    # Dominant kernel: the two trellis contraction launches of each call
    # (stages 1 and 3), timed as (routing plan and rotation + contractions)
    # minus (routing plan and rotation alone) over the same cycled routings,
    # CUDA events on the launching stream around whole graph replays.
    def stages(ss):
        def fn(i):
            for s in ss:
                moe.gemv(x, ids_d[i % R], w_d[i % R], y, stage=s)
        return fn
    g_k = capture(stages((0, 1, 3)))
    g_p = capture(stages((0,)))
    kp_ms, _ = timed(g_k, reps)
    p_ms, _ = timed(g_p, reps)
    k_ms = kp_ms - p_ms
    k_n = 2 * steps
    per_pass = sum(rbytes)
    gemv_bytes = reps * (per_pass - R * (WL.side_bytes(hidden, 0) + WL.side_bytes(0, hidden)))
    achieved = gemv_bytes / (k_ms / 1e3) / 1e9 if k_ms > 0 else None
    y_host = torch.empty((m, hidden), dtype=torch.float16).pin_memory()
    e_steps = min(steps, 2 * R)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(e_steps):
        x.copy_(x_host, non_blocking=True)
        step(i)
        y_host.copy_(y, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    e_ms = e0.elapsed_time(e1)
    if moe.check() != 0:
        raise SystemExit("device error flag set")
    peaks, src = measured_peaks()
    peak = float(peaks["hbm_gbs"])
    value = world * reps * per_pass / (ms / 1e3) / 1e9
    line = {
        "metric": METRIC_DECODE,
        "value": value, "unit": "GB/s", "n_gpus": world, "steps": steps, "warmup": args.warmup,
        "ms_per_step": ms / steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic (seeded device-generated code "
        "words, 64 cycled uniform top-8 routings)",
        "config": {"workload": spec["name"], "tokens": m, "bytes_per_step": per_pass / R,
                   "bytes": BYTES_NOTE + " of each step's distinct routed experts",
                   "l2": "256 experts, %.1f GB of code words; 64 routings cycled"
                         % (sum(c.numel() * 2 for cc in codes for part in cc
                                for c in (part if isinstance(part, list) else [part])) / 1e9),
                   "timing": "CUDA graph of 64 public API calls, CUDA events"},
        "roofline": {"bound": "hbm", "kernel": "trellis_gemv (MoE jobs)",
                     "launch_us": 1e3 * k_ms / k_n, "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak if achieved else None,
                     "traffic": None, "peak_source": src + " (MEASURED_PEAKS.json hbm_gbs)"},
        "e2e": {"value": e_steps * (per_pass / R) / (e_ms / 1e3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": int(x_host.numel() * 2),
                "d2h_bytes_per_step": int(y_host.numel() * 2)},
        "gpu_launches": 5 * steps,
        "clocks": clocks,
    }
    rep.emit(line)
    rep.close()
    return 0


def prefill_spec(args):
    """The prefill workload of the default line (2048 tokens, 5120 -> 17408, 3-bit)."""
    import argparse as _ap
    pa = _ap.Namespace(**vars(args))
    pa.workload, pa.m, pa.shape, pa.fp8 = "prefill", PREFILL_DEFAULT["m"], PREFILL_DEFAULT["shape"], False
    pa.rounding = "fp16"
    return workload_spec(pa)


def tensor_peak(peaks, src, region_s, steps, fp8):
    """The tensor peak a prefill region is compared with, and its note.  A
    timed region of SUSTAINED_REGION_S or more runs the GEMM back to back
    under the power cap: the sustained bf16 peak; a shorter one: the burst
    peak.  fp16 has the bf16 nominal rate; E4M3 twice it (4.5 : 2.25 PFLOP/s)."""
    key = "bf16_tflops_sustained" if region_s >= SUSTAINED_REGION_S else "bf16_tflops"
    peak = float(peaks[key])
    if fp8:
        return 2.0 * peak, (src + " (MEASURED_PEAKS.json %s x 2, the nominal dense E4M3 : bf16 "
                            "ratio 4.5 : 2.25 PFLOP/s; the %s-step region lasts %.2f s)"
                            % (key, steps, region_s))
    return peak, (src + " (MEASURED_PEAKS.json %s: the %s-step region lasts %.2f s; fp16 has "
                  "the same nominal dense rate)" % (key, steps, region_s))


def measure_prefill(args, spec, rep, dev, m, want_cpu):
    """Prefill GEMM of `spec` at m tokens: TFLOP/s of 2*m*in*out per step (median
    over repeats of the K-step region), its roofline against the tensor peak,
    e2e through the C ABI with host buffers, and the CPU oracle's rate."""
    import torch
    from gemm_trellis_tile_gb300 import build, escha
    build.build()
    escha.load()
    k, n, b = spec["layers"][0]
    n_inst = 4   # rotating weight sets: 4 x code + activations + outputs > L2
    lins = []
    for r in range(n_inst):
        lins.append(escha.Linear.from_arrays(S.make_linear(np.random.default_rng(
            rep.seed(spec["seed"], r)), k, n, b)))
        lins[-1].set_rounding(spec["rounding"])
    rng = np.random.default_rng(spec["seed"] + 17)
    x_host = torch.from_numpy(S.make_activations(rng, m, k)).pin_memory()
    x = x_host.to(dev)
    y = torch.empty((m, n), dtype=torch.float16, device=dev)
    for lin in lins:
        lin.reserve(m)
    fp8 = spec["fp8"]

    def call(lin):
        return lin.gemm_fp8(x, y) if fp8 else lin.gemm(x, y)
    for i in range(max(args.warmup, 3)):
        call(lins[i % n_inst])
    torch.cuda.synchronize()
    for lin in lins:
        if lin.check() != 0:
            raise SystemExit("device error flag set during warm-up")

    def run():
        for i in range(args.steps):
            call(lins[i % n_inst])
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    ms, n_rep, lo, hi = median_region(run, rep, dev, args.repeats)
    clocks = sampler.stop()
    # dominant kernel: the GEMM launches alone, from the handles' own event pairs
    for lin in lins:
        lin.profile(True)
    run()
    torch.cuda.synchronize()
    k_ms, k_n = 0.0, 0
    for lin in lins:
        a, c = lin.collect()
        k_ms += a
        k_n += c
        lin.profile(False)
    flops = WL.layer_flops(m, k, n)
    achieved = flops * k_n / (k_ms / 1e3) / 1e12 if k_ms > 0 else None
    # e2e: host activations in, host result out, through the public call
    y_host = torch.empty((m, n), dtype=torch.float16).pin_memory()
    e_steps = min(args.steps, 20)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(e_steps):
        x.copy_(x_host, non_blocking=True)
        call(lins[i % n_inst])
        y_host.copy_(y, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    e_ms = e0.elapsed_time(e1)
    for lin in lins:
        if lin.check() != 0:
            raise SystemExit("device error flag set")
    peaks, src = measured_peaks()
    peak, peak_note = tensor_peak(peaks, src, ms / 1e3, args.steps, fp8)
    world = rep.world
    out = {
        "workload": spec["name"], "metric": METRIC_PREFILL,
        "value": world * args.steps * flops / (ms / 1e3) / 1e12, "unit": "TFLOP/s",
        "ms_per_step": ms / args.steps, "steps": args.steps,
        "dtype": "e4m3" if fp8 else "f16", "tokens": m,
        "l2": "4 rotating weight sets; activations %.0f MB, output %.0f MB per step"
              % (m * k * 2 / 1e6, m * n * 2 / 1e6),
        "timing": "CUDA events around back-to-back public API calls; median of %d repeats "
                  "of the %d-step region (min %.4f, max %.4f ms per step)"
                  % (n_rep, args.steps, lo / args.steps, hi / args.steps),
        "roofline": {"bound": "tensor", "kernel": "trellis_gemm", "achieved": achieved,
                     "launch_us": 1e3 * k_ms / k_n if k_n else None,
                     "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak if achieved else None,
                     "traffic": PREFILL_TRAFFIC_BYTES.get(spec["name"]),
                     "peak_source": peak_note},
        "e2e": {"value": e_steps * flops / (e_ms / 1e3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(x_host.numel() * 2),
                "d2h_bytes_per_step": int(y_host.numel() * 2)},
        "gpu_launches": prefill_launches(m, k, n, props_sms(dev), fp8) * args.steps,
        "clocks": clocks,
    }
    if want_cpu:
        v, cores, sample = prefill_oracle_rate(spec, m, args.cpu_seconds)
        out["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                               "sample": sample}
    return out


def run_prefill(args, spec, rank, world, local):
    """Prefill GEMM: TFLOP/s of 2*M*in*out per step against the tensor peak."""
    import torch
    rep = Replicas(rank, world, local)
    dev = torch.device("cuda", torch.cuda.current_device())
    p = measure_prefill(args, spec, rep, dev, args.m,
                        want_cpu=(rank == 0 and world == 1 and not args.no_cpu_baseline))
    line = {
        "metric": METRIC_PREFILL, "value": p["value"], "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": p["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": p["dtype"],
        "data": "synthetic (seeded uniform code words)",
        "config": {"workload": spec["name"], "tokens": args.m, "l2": p["l2"],
                   "timing": p["timing"]},
        "roofline": p["roofline"], "e2e": p["e2e"], "gpu_launches": p["gpu_launches"],
        "clocks": p["clocks"],
    }
    if "cpu_baseline" in p:
        line["cpu_baseline"] = p["cpu_baseline"]
    rep.emit(line)
    rep.close()
    return 0


# Trellis edges the encoder evaluates per tile: two passes (free start, then
# the tail-biting constraint) x 256 steps x 2^16 states.  Each edge needs at
# least three rounded fp32 operations (difference, square, path sum).
ENCODE_EDGES_PER_TILE = 2 * 256 * 65536
ENCODE_FP32_OPS_PER_EDGE = 3


def encode_oracle_rate(w, bits, seconds):
    """The CPU oracle's encoder on tiles of w until `seconds`:
    (weights/s, cores, sample, weights encoded)."""
    from oracle import escha_oracle as O
    perm = O.perm_forward()
    kt, nt = w.shape[0] // 16, w.shape[1] // 16
    t0 = time.perf_counter()
    c0 = time.process_time()
    n = 0
    while True:
        i, j = divmod(n % (kt * nt), nt)
        vals = w[16 * i:16 * i + 16, 16 * j:16 * j + 16].reshape(-1)[perm]
        O.viterbi_encode_tile(vals, bits)
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    wall = time.perf_counter() - t0
    return (256 * n / wall, round((time.process_time() - c0) / wall, 2),
            "%d tiles of the same matrix, %.1f s" % (n, wall), 256 * n)


def run_encode(args, spec, rank, world, local):
    """Viterbi trellis encoder: weights encoded per second (whole tiles)."""
    import torch
    from gemm_trellis_tile_gb300 import build, escha
    rep = Replicas(rank, world, local)
    build.build()
    escha.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    k, n, bits = spec["layers"][0]
    rng = np.random.default_rng(rep.seed(spec["seed"]))
    w_host_np = (rng.standard_normal((k, n)) * S.CODEBOOK_STD).astype(np.float32)
    w_host = torch.from_numpy(w_host_np).pin_memory()
    w = w_host.to(dev)
    code = torch.empty((k // 16, n // 16, 16 * bits), dtype=torch.int16, device=dev)
    lib = escha.load()
    stream = torch.cuda.current_stream()

    def step():
        escha.check(lib.escha_trellis_encode(escha._ptr(w), k, n, bits, 0, escha._ptr(code),
                                             None, escha._stream(stream)), "escha_trellis_encode")

    steps = args.steps if args.steps != 4000 else 5
    warm = max(3, args.warmup if args.warmup != 50 else 3)
    for _ in range(warm):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    rep.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(steps):
        step()
    t1.record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    rep.barrier()
    ms = t0.elapsed_time(t1)
    ms = rep.slowest(ms, dev)
    tiles = (k // 16) * (n // 16)
    weights = k * n
    # e2e: host matrix in, host code out, through the C ABI
    code_host = torch.empty(code.shape, dtype=torch.int16).pin_memory()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e_steps = min(steps, 3)
    e0.record()
    for _ in range(e_steps):
        w.copy_(w_host, non_blocking=True)
        step()
        code_host.copy_(code, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    e_ms = e0.elapsed_time(e1)
    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count
    peaks, _ = measured_peaks()
    sm_mhz = float(peaks.get("sm_max_mhz", 2070.0))
    # FP32 pipes: 128 lanes per SM per clock
    peak_edges = sms * 128 * sm_mhz * 1e6 / ENCODE_FP32_OPS_PER_EDGE
    achieved_edges = steps * tiles * ENCODE_EDGES_PER_TILE / (ms / 1e3)
    line = {
        "metric": METRIC_ENCODE,
        "value": world * steps * weights / (ms / 1e3), "unit": "weights/s", "n_gpus": world,
        "steps": steps, "warmup": warm, "ms_per_step": ms / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded "
        "N(0, 1.244^2) fp32 matrix)",
        "config": {"workload": spec["name"], "tiles": tiles,
                   "l2": "input %.0f MB, read once per tile; the search runs in shared memory"
                         % (weights * 4 / 1e6),
                   "timing": "CUDA events around back-to-back public API calls"},
        "roofline": {"bound": "alu", "kernel": "trellis_encode", "achieved": achieved_edges / 1e12,
                     "peak": peak_edges / 1e12, "unit": "T trellis edges/s",
                     "frac": achieved_edges / peak_edges, "traffic": None,
                     "peak_source": "derived: %d SMs x 128 fp32 lanes x %.0f MHz / %d rounded "
                                    "fp32 operations per edge" % (sms, sm_mhz,
                                                                  ENCODE_FP32_OPS_PER_EDGE)},
        "e2e": {"value": e_steps * weights / (e_ms / 1e3), "unit": "weights/s",
                "h2d_bytes_per_step": int(w_host.numel() * 4),
                "d2h_bytes_per_step": int(code_host.numel() * 2)},
        "gpu_launches": steps,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, sample, _ = encode_oracle_rate(w_host_np, bits, args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": "weights/s", "cores": cores,
                                "kind": "oracle", "sample": sample}
    rep.emit(line)
    rep.close()
    return 0


def props_sms(dev):
    import torch
    return torch.cuda.get_device_properties(dev).multi_processor_count


def prefill_launches(m, k, n, sms, fp8=False):
    """Kernels of one prefill call: the input rotation (FP8: rotation and
    quantisation) and the GEMM, which finishes tiles shared between CTAs
    itself.  (The call also clears the shared tiles' arrival counters with a
    cudaMemsetAsync, which is not a kernel of this library.)"""
    return 2


def make_handles(spec, inst):
    from gemm_trellis_tile_gb300 import escha
    if spec["kind"] == "mlp":
        g = escha.Linear.from_arrays(inst["gate"])
        u = escha.Linear.from_arrays(inst["up"])
        d = escha.Linear.from_arrays(inst["down"])
        for h in (g, u, d):
            h.set_rounding(spec["rounding"])
        return escha.MLP(g, u, d), (g, u, d)
    lin = escha.Linear.from_arrays(inst["layer"])
    lin.set_rounding(spec["rounding"])
    return lin, (lin,)


def main():
    args = parse_args()
    rank, world, local = dist_env()
    if args.workload == "prefill" and args.m == 1:
        args.m = 2048
    spec = workload_spec(args)
    if args.impl == "reference":
        return run_reference(args, spec, rank)
    if spec["kind"] == "prefill":
        return run_prefill(args, spec, rank, world, local)
    if spec["kind"] == "moe":
        return run_moe(args, spec, rank, world, local)
    if spec["kind"] == "encode":
        return run_encode(args, spec, rank, world, local)

    import torch
    from gemm_trellis_tile_gb300 import build, escha
    rep = Replicas(rank, world, local)
    build.build()
    escha.load()
    dev = torch.device("cuda", torch.cuda.current_device())
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 0) or L2_FALLBACK_BYTES
    m = args.m
    k_in = spec["layers"][0][0]
    n_out = spec["layers"][-1][1]
    launches_per_step = 5 if spec["kind"] == "mlp" else 3
    gemv_launches_per_step = 2 if spec["kind"] == "mlp" else 1

    # Rotating weight sets, together more than 4x L2, so no step finds its
    # code words in L2 from an earlier step.
    code_per_inst = sum(WL.code_bytes(i, o, b) for i, o, b in spec["layers"])
    n_inst = max(2, int(np.ceil(4.0 * l2 / code_per_inst)))
    handles = []
    for r in range(n_inst):
        inst = make_instance(spec, rep.seed(spec["seed"], r))
        handles.append(make_handles(spec, inst))
        if spec.get("norm"):
            nrng = np.random.default_rng(spec["seed"] + 31 * r)
            handles[-1][0].set_input_norm(
                torch.from_numpy(S.make_norm_weight(nrng, spec["layers"][0][0])).to(dev))
        del inst
    rng = np.random.default_rng(spec["seed"] + 17)
    x_host = torch.from_numpy(S.make_activations(rng, m, k_in)).pin_memory()
    x = x_host.to(dev)
    y = torch.empty((m, n_out), dtype=torch.float16, device=dev)

    def step(i):
        handles[i % n_inst][0].gemv(x, y)

    for i in range(max(args.warmup, n_inst)):
        step(i)
    torch.cuda.synchronize()
    for h, _ in handles:
        if h.check() != 0:
            raise SystemExit("device error flag set during warm-up")

    # CUDA graphs: one graph per pass over the weight sets, plus a remainder.
    # The timed graphs hold the public calls only: an event node between two
    # kernels of a graph costs microseconds and stops the next kernel from
    # starting early, so the dominant kernel is timed in a second region.
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())

    def capture(fn, count):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                for i in range(count):
                    fn(i)
        return g

    def timed_replays(graphs, sampler=None):
        """Median over repeats of the K-step region (replays of `graphs`)."""
        if sampler is not None:
            sampler.start()

        def run():
            for g in graphs:
                g.replay()
        med, n, lo, hi = median_region(run, rep, dev, args.repeats)
        clk = sampler.stop() if sampler is not None else None
        return med, clk, (n, lo, hi)

    per_graph = n_inst
    full, rem = divmod(args.steps, per_graph)
    g_main = capture(step, per_graph)
    g_rem = capture(step, rem) if rem else None
    torch.cuda.synchronize()
    for i in range(3):
        g_main.replay()
    torch.cuda.synchronize()
    ms, clocks, reps_info = timed_replays([g_main] * full + ([g_rem] if g_rem else []),
                                          ClockSampler(dev.index if dev.index is not None else 0))

    # Dominant kernel: the same steps with only the trellis contraction stage(s)
    # of each call (escha_*_gemv_stage), K steps between two CUDA events on the
    # launching stream; the average launch duration is that time over the
    # launches.  The other stages' buffers hold the previous full call's values.
    k_stages = (1, 3) if spec["kind"] == "mlp" else (1,)

    def kstep(i):
        for s in k_stages:
            handles[i % n_inst][0].gemv(x, y, stage=s)

    gk_main = capture(kstep, per_graph)
    gk_rem = capture(kstep, rem) if rem else None
    for i in range(3):
        gk_main.replay()
    torch.cuda.synchronize()
    k_ms, _, _ = timed_replays([gk_main] * full + ([gk_rem] if gk_rem else []))
    k_n = gemv_launches_per_step * args.steps
    k_bytes = WL.gemv_kernel_bytes(m, spec["layers"]) * args.steps
    achieved = k_bytes / (k_ms / 1e3) / 1e9 if k_ms > 0 else None

    # End to end through the C ABI: host input copied in, result copied out.
    y_host = torch.empty((m, n_out), dtype=torch.float16).pin_memory()
    e2e_steps = min(args.steps, 2000)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(e2e_steps):
        x.copy_(x_host, non_blocking=True)
        handles[i % n_inst][0].gemv(x, y)
        y_host.copy_(y, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)

    for h, _ in handles:
        st = h.check()
        if st != 0:
            raise SystemExit("device error flag set: status %d" % st)

    sbytes = step_bytes(spec, m)
    value = world * args.steps * sbytes / (ms / 1e3) / 1e9
    peaks, peak_src = measured_peaks()
    peak = float(peaks["hbm_gbs"])
    k_launch_s = k_ms / 1e3 / k_n
    weights_per_launch = sum(i * o for i, o, _ in spec["layers"]) / gemv_launches_per_step
    line = {
        "metric": METRIC_DECODE,
        "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "us_per_layer": 1e3 * ms / args.steps / len(spec["layers"]),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded uniform code words, N(1,0.1) scales, N(0,1) activations)",
        "config": {"workload": spec["name"], "tokens": m,
                   "bytes_per_step": sbytes, "bytes": BYTES_NOTE,
                   "l2": "%d rotating weight sets, %.0f MB of code words (> 4x L2)"
                         % (n_inst, n_inst * code_per_inst / 1e6),
                   "timing": "CUDA graphs of the public API calls, CUDA events; median of %d "
                             "repeats of the %d-step region (min %.4f, max %.4f ms per step)"
                             % (reps_info[0], args.steps, reps_info[1] / args.steps,
                                reps_info[2] / args.steps)},
        "roofline": {"bound": "hbm", "kernel": "trellis_gemv",
                     "launch_us": 1e3 * k_ms / k_n,
                     "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": (achieved / peak) if achieved else None,
                     "traffic": GEMV_TRAFFIC_BYTES.get(spec["name"]) if m == 1 else None,
                     "peak_source": peak_src + " (MEASURED_PEAKS.json hbm_gbs)"},
        "e2e": {"value": e2e_steps * sbytes / (e2e_ms / 1e3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": int(x_host.numel() * 2),
                "d2h_bytes_per_step": int(y_host.numel() * 2)},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    issue = issue_roofline(spec["name"] if m == 1 else None, weights_per_launch / k_launch_s,
                           props.multi_processor_count, clocks)
    if issue is not None:
        line["roofline_issue"] = issue
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, sample = oracle_sample_rate(spec, m, args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle",
                                "sample": sample}
    if spec["kind"] == "mlp" and not args.no_prefill and args.workload == "mlp":
        pspec = prefill_spec(args)
        line["prefill"] = measure_prefill(args, pspec, rep, dev, PREFILL_DEFAULT["m"],
                                          want_cpu=(rank == 0 and world == 1
                                                    and not args.no_cpu_baseline))
    rep.emit(line)
    rep.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
