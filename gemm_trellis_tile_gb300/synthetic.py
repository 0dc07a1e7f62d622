"""Seeded synthetic inputs for trellis-coded layers.

This module only draws random numbers; it holds none of the method's
arithmetic.  The same arrays feed the CUDA library and the CPU oracle.

Recipe (per layer): code words uniform over int16; rin, rout ~ N(1, 0.1)
rounded to fp16; s_in, s_out ~ U(0.98, 1.02) fp32; activations ~ N(0, 1)
rounded to fp16.  Multi-layer workloads (the gated MLP and the MoE) scale each
matrix's rout by an exact power of two 2^-k, k = round(log2(sqrt(in) * 1.2441)),
so that intermediate activations stay inside the fp16 range; 1.2441 is the
standard deviation of the cb=1 codebook over all 65536 states.
"""

import math
import numpy as np

CODEBOOK_STD = 1.2441


def overflow_guard_shift(in_features):
    """k such that rout * 2^-k keeps a random-code layer's output near unit scale."""
    return int(round(math.log2(math.sqrt(in_features) * CODEBOOK_STD)))


def make_linear(rng, in_features, out_features, bits, guard=False):
    """One trellis-coded linear layer as host numpy arrays."""
    assert in_features % 128 == 0 and out_features % 128 == 0
    code = rng.integers(-32768, 32768, size=(in_features // 16, out_features // 16, 16 * bits),
                        dtype=np.int16)
    rin = rng.normal(1.0, 0.1, in_features).astype(np.float16)
    rout = rng.normal(1.0, 0.1, out_features)
    if guard:
        rout = rout * 2.0 ** (-overflow_guard_shift(in_features))
    rout = rout.astype(np.float16)
    s_in = rng.uniform(0.98, 1.02, in_features).astype(np.float32)
    s_out = rng.uniform(0.98, 1.02, out_features).astype(np.float32)
    config = np.array([16, bits, 1, 1, in_features, out_features], dtype=np.int32)
    return dict(code=code, rin=rin, rout=rout, s_in=s_in, s_out=s_out, config=config,
                bits=bits, in_features=in_features, out_features=out_features)


def make_activations(rng, m, features):
    return rng.normal(0.0, 1.0, (m, features)).astype(np.float16)


def make_activation_rows_mixed(rng, m, features):
    """fp16 rows of N(0, 1) values times a per-row factor e^U(-8, 5), with row 0
    all zeros and row 1 holding a single non-zero value (m >= 3)."""
    x = rng.normal(0.0, 1.0, (m, features)) * np.exp(rng.uniform(-8, 5, size=(m, 1)))
    x[0] = 0.0
    x[1] = 0.0
    x[1, rng.integers(features)] = rng.normal()
    return x.astype(np.float16)


def make_mlp(rng, hidden, inter, bits_gate, bits_up, bits_down):
    """Gated MLP down(silu(gate x) * up x) with the fp16 range guard on every matrix."""
    return dict(gate=make_linear(rng, hidden, inter, bits_gate, guard=True),
                up=make_linear(rng, hidden, inter, bits_up, guard=True),
                down=make_linear(rng, inter, hidden, bits_down, guard=True))


def make_norm_weight(rng, n):
    """An RMSNorm weight as escha stores it (centred on zero: w - 1), fp16."""
    return rng.normal(0.2, 0.3, n).astype(np.float16)


def make_moe_spec(seed, num_experts, hidden, inter, bits_choices=(2, 3, 4)):
    """Routed-expert stack: widths, shared hidden-side vectors and per-expert
    intermediate-side vectors.  Code words are drawn per expert on demand
    (make_moe_expert_codes), so a test can build only the experts it routes to.

    Every expert gets one width b_e drawn uniformly from bits_choices for all
    three of its matrices.  The hidden side (gate/up input, down output) uses
    one shared rin/s_in and one shared rout/s_out; the intermediate side is per
    expert.  rout vectors carry the fp16 range guard of their matrix.
    """
    rng = np.random.default_rng([seed, 0])
    E = num_experts
    bits = rng.choice(np.asarray(bits_choices, dtype=np.int32), size=E).astype(np.int32)
    kg = overflow_guard_shift(hidden)   # gate/up: hidden -> inter
    kd = overflow_guard_shift(inter)    # down: inter -> hidden

    def f16(a):
        return a.astype(np.float16)

    return dict(
        seed=seed, num_experts=E, hidden=hidden, inter=inter, bits=bits,
        rin_hidden=f16(rng.normal(1.0, 0.1, hidden)),
        s_in_hidden=rng.uniform(0.98, 1.02, hidden).astype(np.float32),
        rout_hidden=f16(rng.normal(1.0, 0.1, hidden) * 2.0 ** (-kd)),
        s_out_hidden=rng.uniform(0.98, 1.02, hidden).astype(np.float32),
        rout_gate=f16(rng.normal(1.0, 0.1, (E, inter)) * 2.0 ** (-kg)),
        s_out_gate=rng.uniform(0.98, 1.02, (E, inter)).astype(np.float32),
        rout_up=f16(rng.normal(1.0, 0.1, (E, inter)) * 2.0 ** (-kg)),
        s_out_up=rng.uniform(0.98, 1.02, (E, inter)).astype(np.float32),
        rin_down=f16(rng.normal(1.0, 0.1, (E, inter))),
        s_in_down=rng.uniform(0.98, 1.02, (E, inter)).astype(np.float32),
    )


def make_moe_expert_codes(spec, e):
    """Code words of expert e: (gate, up, down) int16 tensors."""
    rng = np.random.default_rng([spec["seed"], 1, int(e)])
    b = int(spec["bits"][e])
    h, i = spec["hidden"], spec["inter"]
    gate = rng.integers(-32768, 32768, size=(h // 16, i // 16, 16 * b), dtype=np.int16)
    up = rng.integers(-32768, 32768, size=(h // 16, i // 16, 16 * b), dtype=np.int16)
    down = rng.integers(-32768, 32768, size=(i // 16, h // 16, 16 * b), dtype=np.int16)
    return gate, up, down



def make_moe_shared_expert(spec, bits=4):
    """The shared expert of a routed-expert stack: code words and its own
    intermediate-side vectors, drawn like a routed expert's (rout vectors with
    the fp16 range guard)."""
    rng = np.random.default_rng([spec["seed"], 4])
    h, i = spec["hidden"], spec["inter"]
    kg = overflow_guard_shift(h)

    def code(k, n):
        return rng.integers(-32768, 32768, size=(k // 16, n // 16, 16 * bits), dtype=np.int16)
    return dict(
        bits=bits, gate=code(h, i), up=code(h, i), down=code(i, h),
        rout_gate=(rng.normal(1.0, 0.1, i) * 2.0 ** (-kg)).astype(np.float16),
        s_out_gate=rng.uniform(0.98, 1.02, i).astype(np.float32),
        rout_up=(rng.normal(1.0, 0.1, i) * 2.0 ** (-kg)).astype(np.float16),
        s_out_up=rng.uniform(0.98, 1.02, i).astype(np.float32),
        rin_down=rng.normal(1.0, 0.1, i).astype(np.float16),
        s_in_down=rng.uniform(0.98, 1.02, i).astype(np.float32))


def make_moe_half_spec(seed, num_experts, hidden, inter, bits_choices=(2, 3, 4)):
    """Routed-expert stack stored by halves of 128 intermediate channels: the
    side vectors of make_moe_spec, a width per half for gate and for up
    (gate_bits, up_bits [E, inter/128]) and one width per expert for down
    (down_bits [E]), each drawn uniformly from bits_choices."""
    spec = make_moe_spec(seed, num_experts, hidden, inter, bits_choices)
    rng = np.random.default_rng([seed, 2])
    H = inter // 128
    choices = np.asarray(bits_choices, dtype=np.int32)
    spec["gate_bits"] = rng.choice(choices, size=(num_experts, H)).astype(np.int32)
    spec["up_bits"] = rng.choice(choices, size=(num_experts, H)).astype(np.int32)
    spec["down_bits"] = spec.pop("bits")
    spec["halves"] = H
    return spec


def make_moe_expert_half_codes(spec, e):
    """Code words of expert e by halves: lists of H int16 tensors for gate and
    up ([hidden/16, 8, 16*b], output channels 128h..128h+127) and for down
    ([8, hidden/16, 16*b], input channels 128h..128h+127)."""
    rng = np.random.default_rng([spec["seed"], 3, int(e)])
    hid, H = spec["hidden"], spec["halves"]
    bd = int(spec["down_bits"][e])

    def draw(shape):
        return rng.integers(-32768, 32768, size=shape, dtype=np.int16)
    gate = [draw((hid // 16, 8, 16 * int(spec["gate_bits"][e, h]))) for h in range(H)]
    up = [draw((hid // 16, 8, 16 * int(spec["up_bits"][e, h]))) for h in range(H)]
    down = [draw((8, hid // 16, 16 * bd)) for _ in range(H)]
    return gate, up, down


def make_routing(rng, m, num_experts, topk=8):
    """topk distinct experts per token, uniform; weights = softmax of N(0,1) logits."""
    ids = np.stack([rng.choice(num_experts, size=topk, replace=False) for _ in range(m)]).astype(np.int32)
    logits = rng.normal(0.0, 1.0, (m, topk))
    w = np.exp(logits - logits.max(axis=1, keepdims=True))
    w = (w / w.sum(axis=1, keepdims=True)).astype(np.float32)
    return ids, w


# The five workloads, by shape (seed = 1000 + index).
WORKLOADS = {
    0: dict(name="linear 512x512 2-bit", kind="linear", in_features=512, out_features=512, bits=2),
    1: dict(name="dense gated MLP 5120->17408->5120 (gate 2-bit, up 3-bit, down 3-bit)",
            kind="mlp", hidden=5120, inter=17408, bits=(2, 3, 3)),
    2: dict(name="decode sweep: 5120->10240 2-bit and 6144->5120 2-bit",
            kind="sweep", shapes=((5120, 10240, 2), (6144, 5120, 2)), m=(1, 2, 4, 8, 16)),
    3: dict(name="routed MoE: 256 experts, 6144->2048->6144, 2/3/4-bit per expert, top-8",
            kind="moe", experts=256, hidden=6144, inter=2048, topk=8, m=(1, 2, 4, 8)),
    4: dict(name="prefill M=2048: 5120->17408 3-bit and 17408->5120 3-bit",
            kind="prefill", m=2048, shapes=((5120, 17408, 3), (17408, 5120, 3))),
}


def seed_for(workload_index, extra=0):
    return 1000 + workload_index + 100000 * extra
