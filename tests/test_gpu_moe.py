"""GPU parity of the routed-expert path against the CPU oracle, through the C ABI.

Outputs must be within relative L2 2e-3 of the fp64 oracle.  Small shapes are
compared in full against the oracle's moe_forward; the GLM-shaped layer (256
experts, 6144 -> 2048 -> 6144, mixed 2/3/4-bit) is compared on sampled output
blocks of one token, with the oracle decoding that token's experts.
"""

import numpy as np
import pytest

from gemm_trellis_tile_gb300 import synthetic as S
from oracle import escha_oracle as O
from tests.helpers import REL_L2_TOL, worst_rel_l2

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gemm_trellis_tile_gb300 import build, escha
    build.build()
    escha.load()


def _expert_layers(spec, e, codes):
    """Oracle layer dicts (w, su, sv) of expert e with the shared hidden side."""
    g, u, d = codes
    b = int(spec["bits"][e])
    su_h = O.fold_scales(spec["rin_hidden"], spec["s_in_hidden"])
    sv_h = O.fold_scales(spec["rout_hidden"], spec["s_out_hidden"])
    gate = dict(w=O.decode_matrix(g, b), su=su_h,
                sv=O.fold_scales(spec["rout_gate"][e], spec["s_out_gate"][e]))
    up = dict(w=O.decode_matrix(u, b), su=su_h,
              sv=O.fold_scales(spec["rout_up"][e], spec["s_out_up"][e]))
    down = dict(w=O.decode_matrix(d, b), su=O.fold_scales(spec["rin_down"][e], spec["s_in_down"][e]),
                sv=sv_h)
    return gate, up, down


def _run(moe, x, ids, w):
    y = moe.gemv(torch.from_numpy(x).cuda(), torch.from_numpy(ids).cuda(),
                 torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    return y.cpu().numpy()


def _small(seed, E=16, hidden=512, inter=256):
    from gemm_trellis_tile_gb300 import escha
    spec = S.make_moe_spec(seed, E, hidden, inter)
    codes = {e: S.make_moe_expert_codes(spec, e) for e in range(E)}
    moe = escha.MoE.from_arrays(spec, codes)
    experts = [_expert_layers(spec, e, codes[e]) for e in range(E)]
    return spec, moe, experts


@pytest.mark.parametrize("m,topk", [(1, 8), (3, 8), (8, 8), (5, 2), (8, 1)])
def test_moe_small_matches_oracle(m, topk):
    spec, moe, experts = _small(3000)
    rng = np.random.default_rng(3100 + m * 10 + topk)
    x = S.make_activations(rng, m, spec["hidden"])
    ids, w = S.make_routing(rng, m, spec["num_experts"], topk)
    y = _run(moe, x, ids, w)
    assert moe.check() == 0
    ref = O.moe_forward(x, experts, ids, w)
    assert worst_rel_l2(y, ref) <= REL_L2_TOL


def test_moe_repeated_calls_with_different_routing():
    """Routing is read on the device every call; stale job tables must not leak."""
    spec, moe, experts = _small(3001)
    rng = np.random.default_rng(3200)
    for m in (8, 1, 4):
        x = S.make_activations(rng, m, spec["hidden"])
        ids, w = S.make_routing(rng, m, spec["num_experts"], 8)
        y = _run(moe, x, ids, w)
        assert worst_rel_l2(y, O.moe_forward(x, experts, ids, w)) <= REL_L2_TOL


def test_moe_duplicate_ids_are_summed():
    spec, moe, experts = _small(3002)
    rng = np.random.default_rng(3300)
    x = S.make_activations(rng, 2, spec["hidden"])
    ids = np.array([[3, 3, 5, 7], [1, 2, 3, 3]], dtype=np.int32)
    w = np.array([[0.25, 0.5, 0.125, 0.125], [0.1, 0.2, 0.3, 0.4]], dtype=np.float32)
    y = _run(moe, x, ids, w)
    assert worst_rel_l2(y, O.moe_forward(x, experts, ids, w)) <= REL_L2_TOL


def test_moe_out_of_range_id_is_skipped_and_flagged():
    spec, moe, experts = _small(3003)
    rng = np.random.default_rng(3400)
    x = S.make_activations(rng, 1, spec["hidden"])
    ids = np.array([[2, 99, 4, -1]], dtype=np.int32)
    w = np.array([[0.4, 0.3, 0.2, 0.1]], dtype=np.float32)
    y = _run(moe, x, ids, w)
    assert moe.check() == 1                       # ESCHA_ERR_INVALID_ARG, flag cleared
    ref = O.moe_forward(x, experts, np.array([[2, 4]]), np.array([[0.4, 0.2]]))
    assert worst_rel_l2(y, ref) <= REL_L2_TOL
    assert moe.check() == 0


def test_moe_profiler_counts_two_trellis_launches_per_call():
    spec, moe, experts = _small(3004)
    rng = np.random.default_rng(3500)
    x = torch.from_numpy(S.make_activations(rng, 2, spec["hidden"])).cuda()
    ids, w = S.make_routing(rng, 2, spec["num_experts"], 8)
    moe.profile(True)
    for _ in range(3):
        moe.gemv(x, torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda())
    ms, n = moe.collect()
    assert n == 6 and ms > 0
    moe.profile(False)


def test_moe_glm_shape_full_size_sampled():
    """256 experts, 6144 -> 2048 -> 6144, mixed widths, top-8, M = 4.

    Only routed experts get code words; the oracle decodes token 0's eight
    experts (gate and up in full, down on three sampled 128-column blocks).
    """
    from gemm_trellis_tile_gb300 import escha
    spec = S.make_moe_spec(S.seed_for(3), 256, 6144, 2048)
    rng = np.random.default_rng(S.seed_for(3, 1))
    m = 4
    x = S.make_activations(rng, m, 6144)
    ids, w = S.make_routing(rng, m, 256, 8)
    routed = sorted(set(ids.reshape(-1).tolist()))
    codes = {e: S.make_moe_expert_codes(spec, e) for e in routed}
    moe = escha.MoE.from_arrays(spec, codes)
    y = _run(moe, x, ids, w)
    assert moe.check() == 0
    assert np.all(np.isfinite(y))
    blocks = [0, 23, 47]
    cols = np.concatenate([np.arange(b * 128, b * 128 + 128) for b in blocks])
    ref = np.zeros(cols.size)
    su_h = O.fold_scales(spec["rin_hidden"], spec["s_in_hidden"])
    sv_h = O.fold_scales(spec["rout_hidden"], spec["s_out_hidden"])
    for k in range(8):
        e = int(ids[0, k])
        g, u, d = codes[e]
        b = int(spec["bits"][e])
        hg = O.linear_forward(x[:1], O.decode_matrix(g, b), su_h,
                              O.fold_scales(spec["rout_gate"][e], spec["s_out_gate"][e]))
        hu = O.linear_forward(x[:1], O.decode_matrix(u, b), su_h,
                              O.fold_scales(spec["rout_up"][e], spec["s_out_up"][e]))
        h = O.silu(hg) * hu
        _, yd = O.linear_forward_columns(h, d, b, O.fold_scales(spec["rin_down"][e],
                                                                  spec["s_in_down"][e]),
                                         sv_h, blocks)
        ref += float(w[0, k]) * yd[0]
    assert worst_rel_l2(y[0, cols], ref) <= REL_L2_TOL


def test_moe_stages_compose_to_the_full_call():
    from gemm_trellis_tile_gb300 import escha
    spec, moe, experts = _small(3005)
    rng = np.random.default_rng(3600)
    x = torch.from_numpy(S.make_activations(rng, 3, spec["hidden"])).cuda()
    ids, w = S.make_routing(rng, 3, spec["num_experts"], 8)
    ids, w = torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda()
    full = moe.gemv(x, ids, w)
    staged = torch.empty_like(full)
    for s in range(escha.MoE.STAGES):
        moe.gemv(x, ids, w, staged, stage=s)
    assert torch.equal(full, staged)
    with pytest.raises(escha.EschaError) as e:
        moe.gemv(x, ids, w, staged, stage=escha.MoE.STAGES)
    assert e.value.status == 1


def _shared_layers(spec, sh):
    su_h = O.fold_scales(spec["rin_hidden"], spec["s_in_hidden"])
    sv_h = O.fold_scales(spec["rout_hidden"], spec["s_out_hidden"])
    b = sh["bits"]
    return (dict(w=O.decode_matrix(sh["gate"], b), su=su_h,
                 sv=O.fold_scales(sh["rout_gate"], sh["s_out_gate"])),
            dict(w=O.decode_matrix(sh["up"], b), su=su_h,
                 sv=O.fold_scales(sh["rout_up"], sh["s_out_up"])),
            dict(w=O.decode_matrix(sh["down"], b),
                 su=O.fold_scales(sh["rin_down"], sh["s_in_down"]), sv=sv_h))


def _set_shared(moe, sh):
    t = {k: torch.from_numpy(v).cuda() for k, v in sh.items() if k != "bits"}
    moe.set_shared_expert(t["gate"], t["up"], t["down"], sh["bits"], t["rout_gate"],
                          t["s_out_gate"], t["rout_up"], t["s_out_up"], t["rin_down"],
                          t["s_in_down"])
    return t


@pytest.mark.parametrize("m,topk", [(1, 8), (4, 8), (8, 8), (3, 2)])
def test_moe_shared_expert_matches_oracle(m, topk):
    """Routed experts plus the shared expert; at M = 8, top-8 with 64 distinct
    experts the shared expert takes the 65th slot."""
    from gemm_trellis_tile_gb300 import escha
    E = 96 if m == 8 else 16
    spec = S.make_moe_spec(3700 + m, E, 512, 256)
    rng = np.random.default_rng(3710 + m * 10 + topk)
    x = S.make_activations(rng, m, spec["hidden"])
    if m == 8:
        ids = rng.permutation(E)[:64].reshape(8, 8).astype(np.int32)  # 64 distinct experts
        _, w = S.make_routing(rng, m, E, topk)
    else:
        ids, w = S.make_routing(rng, m, E, topk)
    used = sorted(set(ids.reshape(-1).tolist()))
    codes = {e: S.make_moe_expert_codes(spec, e) for e in used}
    moe = escha.MoE.from_arrays(spec, codes)
    sh = S.make_moe_shared_expert(spec)
    keep = _set_shared(moe, sh)
    y = _run(moe, x, ids, w)
    assert moe.check() == 0
    experts = {e: _expert_layers(spec, e, codes[e]) for e in used}
    ref = O.moe_forward_shared(x, experts, ids, w, _shared_layers(spec, sh))
    assert worst_rel_l2(y, ref) <= REL_L2_TOL
    del keep


def test_moe_shared_expert_removed_restores_routed_only():
    spec, moe, experts = _small(3800)
    rng = np.random.default_rng(3801)
    x = torch.from_numpy(S.make_activations(rng, 2, spec["hidden"])).cuda()
    ids, w = S.make_routing(rng, 2, spec["num_experts"], 8)
    ids, w = torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda()
    plain = moe.gemv(x, ids, w)
    keep = _set_shared(moe, S.make_moe_shared_expert(spec, bits=2))
    with_shared = moe.gemv(x, ids, w)
    moe.set_shared_expert(None, None, None, 0, None, None, None, None, None, None)
    again = moe.gemv(x, ids, w)
    torch.cuda.synchronize()
    assert torch.equal(plain, again) and not torch.equal(plain, with_shared)
    del keep
