"""GPU parity of the dense trellis path against the CPU oracle, through the C ABI.

Decoded weights must match the oracle bit for bit; layer outputs must be within
relative L2 2e-3 of the fp64 oracle (the oracle keeps every intermediate in
fp64; the GPU rounds the rotated activations and the output to fp16 once each).
"""

import numpy as np
import pytest

from gemm_trellis_tile_gb300 import synthetic as S
from oracle import escha_oracle as O
from tests.helpers import (REL_L2_TOL, make_linear_handle, oracle_layer_dict, oracle_linear,
                           worst_rel_l2)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gemm_trellis_tile_gb300 import build, escha
    build.build()
    escha.load()


# ---------------------------------------------------------------- decode

@pytest.mark.parametrize("bits,k,n", [(2, 512, 512), (3, 384, 640), (4, 256, 1280), (2, 2048, 2048),
                                      (3, 1024, 4096), (4, 4096, 1024)])
def test_decode_bit_exact(bits, k, n):
    rng = np.random.default_rng(100 + bits + k)
    layer = S.make_linear(rng, k, n, bits)
    lin, _ = make_linear_handle(layer)
    w_gpu = lin.decode().cpu().numpy().view(np.uint16)
    w_ref = O.decode_matrix(layer["code"], bits).view(np.uint16)
    assert np.array_equal(w_gpu, w_ref)


def test_decode_covers_every_state_value():
    """~1M random states: every one of the 65536 codebook states is exercised."""
    rng = np.random.default_rng(7)
    layer = S.make_linear(rng, 2048, 2048, 4)
    states = O.tile_states(layer["code"].reshape(-1, 64), 4)
    assert np.unique(states).size == 65536
    lin, _ = make_linear_handle(layer)
    w_gpu = lin.decode().cpu().numpy().view(np.uint16)
    assert np.array_equal(w_gpu, O.decode_matrix(layer["code"], 4).view(np.uint16))


# ---------------------------------------------------------------- GEMV

def _gemv_case(layer, ms, seed):
    lin, _ = make_linear_handle(layer)
    w = O.decode_matrix(layer["code"], layer["bits"])
    rng = np.random.default_rng(seed)
    for m in ms:
        x = S.make_activations(rng, m, layer["in_features"])
        y = lin.gemv(torch.from_numpy(x).cuda())
        torch.cuda.synchronize()
        assert lin.check() == 0
        ref = oracle_linear(layer, x, w)
        err = worst_rel_l2(y.cpu().numpy(), ref)
        assert err <= REL_L2_TOL, (m, err)


def test_gemv_single_linear_512():
    """512x512 at 2 bits, every token count 1..16."""
    layer = S.make_linear(np.random.default_rng(S.seed_for(0)), 512, 512, 2)
    _gemv_case(layer, list(range(1, 17)), 1)


@pytest.mark.parametrize("bits,k,n", [(3, 384, 640), (4, 1280, 256), (2, 128, 128), (3, 2048, 1536),
                                      (4, 640, 3840)])
def test_gemv_small_shapes(bits, k, n):
    layer = S.make_linear(np.random.default_rng(200 + bits + k), k, n, bits)
    _gemv_case(layer, [1, 3, 8, 9, 16], 2)


@pytest.mark.parametrize("k,n", [(5120, 10240), (6144, 5120)])
def test_gemv_decode_sweep_full_size(k, n):
    """The decode-sweep shapes at full size, M = 1, 2, 4, 8, 16."""
    layer = S.make_linear(np.random.default_rng(S.seed_for(2, k)), k, n, 2)
    _gemv_case(layer, [1, 2, 4, 8, 16], 3)


def test_gemv_config_from_device_and_nine_entry_layout():
    rng = np.random.default_rng(9)
    layer = S.make_linear(rng, 256, 384, 3)
    layer9 = dict(layer)
    layer9["config"] = np.array([16, 48, 3, 1, 1, 256, 384, 256, 384], dtype=np.int32)
    x = S.make_activations(rng, 2, 256)
    ref = oracle_linear(layer, x)
    for lay, dev in ((layer, True), (layer9, False), (layer9, True)):
        lin, _ = make_linear_handle(lay, config_on_device=dev)
        y = lin.gemv(torch.from_numpy(x).cuda()).cpu().numpy()
        assert worst_rel_l2(y, ref) <= REL_L2_TOL


def test_gemv_repeatable_and_independent_of_previous_call():
    rng = np.random.default_rng(11)
    layer = S.make_linear(rng, 1024, 2048, 3)
    lin, _ = make_linear_handle(layer)
    xa = torch.from_numpy(S.make_activations(rng, 16, 1024)).cuda()
    xb = torch.from_numpy(S.make_activations(rng, 1, 1024)).cuda()
    ya1 = lin.gemv(xa).clone()
    yb = lin.gemv(xb).clone()
    ya2 = lin.gemv(xa).clone()
    assert torch.equal(ya1, ya2)                    # deterministic
    assert torch.equal(yb[0], lin.gemv(xb)[0])


# ---------------------------------------------------------------- MLP

def _mlp_oracle(mlp, x, down_blocks=None):
    g = oracle_layer_dict(mlp["gate"])
    u = oracle_layer_dict(mlp["up"])
    hg = O.linear_forward(x, g["w"], g["su"], g["sv"])
    hu = O.linear_forward(x, u["w"], u["su"], u["sv"])
    h = O.silu(hg) * hu
    d = mlp["down"]
    su, sv = O.fold_scales(d["rin"], d["s_in"]), O.fold_scales(d["rout"], d["s_out"])
    if down_blocks is None:
        return None, O.linear_forward(h, O.decode_matrix(d["code"], d["bits"]), su, sv)
    return O.linear_forward_columns(h, d["code"], d["bits"], su, sv, down_blocks)


def _mlp_handle(mlp):
    from gemm_trellis_tile_gb300 import escha
    gate, kg = make_linear_handle(mlp["gate"])
    up, ku = make_linear_handle(mlp["up"])
    down, kd = make_linear_handle(mlp["down"])
    return escha.MLP(gate, up, down), (gate, up, down, kg, ku, kd)


def test_mlp_small_all_widths():
    rng = np.random.default_rng(21)
    mlp = S.make_mlp(rng, 512, 1536, 2, 3, 4)
    handle, keep = _mlp_handle(mlp)
    for m in (1, 5, 16):
        x = S.make_activations(rng, m, 512)
        y = handle.gemv(torch.from_numpy(x).cuda()).cpu().numpy()
        _, ref = _mlp_oracle(mlp, x)
        assert worst_rel_l2(y, ref) <= REL_L2_TOL, m


def test_mlp_dense_full_size_sampled():
    """The 5120->17408->5120 gated MLP (2/3/3 bits) at M=1 and M=4.

    The oracle decodes gate and up in full (the down input needs every channel)
    and down only for three sampled 128-column blocks, including the last.
    """
    rng = np.random.default_rng(S.seed_for(1))
    mlp = S.make_mlp(rng, 5120, 17408, 2, 3, 3)
    handle, keep = _mlp_handle(mlp)
    blocks = [0, 17, 39]
    for m in (1, 4):
        x = S.make_activations(rng, m, 5120)
        y = handle.gemv(torch.from_numpy(x).cuda()).cpu().numpy()
        cols, ref = _mlp_oracle(mlp, x, blocks)
        assert np.all(np.isfinite(y))
        assert worst_rel_l2(y[:, cols], ref) <= REL_L2_TOL


# ---------------------------------------------------------------- errors and self test

def test_argument_errors_on_gpu():
    from gemm_trellis_tile_gb300 import escha
    rng = np.random.default_rng(31)
    layer = S.make_linear(rng, 256, 256, 2)
    lin, _ = make_linear_handle(layer)
    x = torch.zeros((17, 256), dtype=torch.float16, device="cuda")
    with pytest.raises(escha.EschaError) as e:
        lin.gemv(x)
    assert e.value.status == 1
    buf = torch.zeros(300, dtype=torch.float16, device="cuda")
    with pytest.raises(escha.EschaError):
        lin.gemv(buf[1:257].view(1, 256))   # misaligned
    bad = dict(layer)
    bad["config"] = np.array([16, 5, 1, 1, 256, 256], dtype=np.int32)
    with pytest.raises(escha.EschaError) as e:
        make_linear_handle(bad)
    assert e.value.status == 2


def test_binding_refuses_wrong_widths_before_any_launch():
    """Kernels read whole rows of the layer's width: other shapes stop in the binding."""
    rng = np.random.default_rng(33)
    layer = S.make_linear(rng, 256, 384, 2)
    lin, _ = make_linear_handle(layer)
    for bad in (torch.zeros((2, 128), dtype=torch.float16, device="cuda"),
                torch.zeros((256,), dtype=torch.float16, device="cuda")):
        for call in (lin.gemv, lin.gemm):
            with pytest.raises(ValueError):
                call(bad)
    x = torch.zeros((2, 256), dtype=torch.float16, device="cuda")
    with pytest.raises(ValueError):
        lin.gemv(x, torch.zeros((2, 256), dtype=torch.float16, device="cuda"))   # y width
    with pytest.raises(ValueError):
        lin.gemm_fp8_codes(torch.zeros((2, 128), dtype=torch.uint8, device="cuda"),
                           torch.zeros((2,), dtype=torch.float32, device="cuda"))
    assert lin.check() == 0


def test_bounded_wait_times_out_and_context_survives():
    from gemm_trellis_tile_gb300 import escha
    assert escha.selftest_wait_timeout(20000) == 5
    rng = np.random.default_rng(41)
    layer = S.make_linear(rng, 256, 256, 2)
    lin, _ = make_linear_handle(layer)
    x = S.make_activations(rng, 1, 256)
    y = lin.gemv(torch.from_numpy(x).cuda()).cpu().numpy()
    assert worst_rel_l2(y, oracle_linear(layer, x)) <= REL_L2_TOL
    assert lin.check() == 0


def test_profiler_counts_trellis_launches():
    rng = np.random.default_rng(51)
    layer = S.make_linear(rng, 512, 512, 2)
    lin, _ = make_linear_handle(layer)
    lin.profile(True)
    x = torch.from_numpy(S.make_activations(rng, 1, 512)).cuda()
    for _ in range(3):
        lin.gemv(x)
    ms, n = lin.collect()
    assert n == 3 and ms > 0
    lin.profile(False)
    lin.gemv(x)
    assert lin.collect() == (0.0, 0)


def test_stages_compose_to_the_full_call():
    """Stages 0..N-1 in order give the full call's output bit for bit."""
    from gemm_trellis_tile_gb300 import escha
    rng = np.random.default_rng(61)
    layer = S.make_linear(rng, 768, 1280, 3)
    lin, _ = make_linear_handle(layer)
    mlp = S.make_mlp(rng, 512, 1536, 2, 3, 4)
    handle, keep = _mlp_handle(mlp)
    for m in (1, 11):
        x = S.make_activations(rng, m, 768)
        xt = torch.from_numpy(x).cuda()
        full = lin.gemv(xt)
        ylin = torch.empty_like(full)
        for s in range(escha.Linear.STAGES):
            lin.gemv(xt, ylin, stage=s)
        assert torch.equal(full, ylin)
        assert worst_rel_l2(ylin.cpu().numpy(), oracle_linear(layer, x)) <= REL_L2_TOL
        xm = torch.from_numpy(S.make_activations(rng, m, 512)).cuda()
        full = handle.gemv(xm)
        ymlp = torch.empty_like(full)
        for s in range(escha.MLP.STAGES):
            handle.gemv(xm, ymlp, stage=s)
        assert torch.equal(full, ymlp)
    assert ylin.shape == (11, 1280)
    for bad in (-1, escha.Linear.STAGES):
        with pytest.raises(escha.EschaError) as e:
            lin.gemv(xt, ylin, stage=bad)
        assert e.value.status == 1


_SYNC_DEBUG_SCRIPT = r"""
import hashlib, sys
import numpy as np, torch
sys.path.insert(0, sys.argv[1])
from gemm_trellis_tile_gb300 import escha, synthetic as S
escha.load()
rng = np.random.default_rng(91)
lin = escha.Linear.from_arrays(S.make_linear(rng, 512, 768, 3))
x = torch.from_numpy(S.make_activations(rng, 4, 512)).cuda()
y1 = lin.gemv(x)
y2 = lin.gemm(torch.cat([x] * 80))
torch.cuda.synchronize()
assert lin.check() == 0
h = hashlib.sha256(y1.cpu().numpy().tobytes() + y2.cpu().numpy().tobytes()).hexdigest()
print(h)
"""


def test_sync_debug_mode_gives_the_same_results():
    """ESCHA_SYNC_DEBUG=1 synchronises after every compute call; results are
    bit-identical to a run without it."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    outs = []
    for flag in ("0", "1"):
        env = dict(os.environ, ESCHA_SYNC_DEBUG=flag)
        r = subprocess.run([sys.executable, "-c", _SYNC_DEBUG_SCRIPT, root], env=env,
                           capture_output=True, text=True, timeout=300)
        assert r.returncode == 0, r.stderr[-2000:]
        outs.append(r.stdout.strip().splitlines()[-1])
    assert outs[0] == outs[1]
