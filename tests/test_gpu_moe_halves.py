"""GPU parity of the routed-expert path stored by halves (EXLR8 manifest
layout: per-half widths for gate/up, per-expert widths for down, pointer
table re-read every call), through the C ABI, against the CPU oracle.

Outputs must be within relative L2 2e-3 of the fp64 oracle, whose expert
matrices are the halves decoded and put side by side (gate, up) or stacked
(down).
"""

import numpy as np
import pytest

from gemm_trellis_tile_gb300 import synthetic as S
from oracle import escha_oracle as O
from tests.helpers import REL_L2_TOL, rel_l2, worst_rel_l2

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gemm_trellis_tile_gb300 import build, escha
    build.build()
    escha.load()


def _expert(spec, e, codes, rounding="fp16"):
    """Oracle layer dicts (w, su, sv) of expert e from its halves."""
    g, u, d = codes
    su_h = O.fold_scales(spec["rin_hidden"], spec["s_in_hidden"])
    sv_h = O.fold_scales(spec["rout_hidden"], spec["s_out_hidden"])
    gate = dict(w=O.decode_column_halves(g, spec["gate_bits"][e], rounding), su=su_h,
                sv=O.fold_scales(spec["rout_gate"][e], spec["s_out_gate"][e]))
    up = dict(w=O.decode_column_halves(u, spec["up_bits"][e], rounding), su=su_h,
              sv=O.fold_scales(spec["rout_up"][e], spec["s_out_up"][e]))
    down = dict(w=O.decode_row_halves(d, spec["down_bits"][e], rounding),
                su=O.fold_scales(spec["rin_down"][e], spec["s_in_down"][e]), sv=sv_h)
    return gate, up, down


def _run(moe, x, ids, w):
    y = moe.gemv(torch.from_numpy(x).cuda(), torch.from_numpy(ids).cuda(),
                 torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    return y.cpu().numpy()


def _small(seed, E=12, hidden=384, inter=384):
    from gemm_trellis_tile_gb300 import escha
    spec = S.make_moe_half_spec(seed, E, hidden, inter)
    codes = {e: S.make_moe_expert_half_codes(spec, e) for e in range(E)}
    moe = escha.MoEHalves.from_arrays(spec, codes)
    return spec, codes, moe


@pytest.mark.parametrize("m,topk", [(1, 8), (3, 8), (8, 8), (5, 3), (8, 1)])
def test_moe_halves_small_matches_oracle(m, topk):
    spec, codes, moe = _small(5000)
    rng = np.random.default_rng(5100 + 10 * m + topk)
    x = S.make_activations(rng, m, spec["hidden"])
    ids, w = S.make_routing(rng, m, spec["num_experts"], topk)
    y = _run(moe, x, ids, w)
    assert moe.check() == 0
    experts = {e: _expert(spec, e, codes[e]) for e in set(ids.reshape(-1).tolist())}
    ref = O.moe_forward(x, experts, ids, w)
    assert worst_rel_l2(y, ref) <= REL_L2_TOL


def test_moe_halves_with_uniform_widths_equals_whole_matrix_storage():
    """Widths uniform per expert: the halves of each whole code tensor (cut at
    every 8th tile column for gate/up, every 8th tile row for down) given to
    escha_moe_create_halves compute the same layer as the whole tensors given
    to escha_moe_create."""
    from gemm_trellis_tile_gb300 import escha
    E, hidden, inter = 10, 256, 512
    spec = S.make_moe_spec(5200, E, hidden, inter)
    whole = {e: S.make_moe_expert_codes(spec, e) for e in range(E)}
    H = inter // 128
    hspec = dict(spec)
    hspec["halves"] = H
    hspec["gate_bits"] = np.repeat(spec["bits"][:, None], H, axis=1).astype(np.int32)
    hspec["up_bits"] = hspec["gate_bits"].copy()
    hspec["down_bits"] = spec["bits"].copy()
    halves = {e: ([np.ascontiguousarray(g[:, 8 * h:8 * h + 8]) for h in range(H)],
                  [np.ascontiguousarray(u[:, 8 * h:8 * h + 8]) for h in range(H)],
                  [np.ascontiguousarray(d[8 * h:8 * h + 8]) for h in range(H)])
              for e, (g, u, d) in whole.items()}
    a = escha.MoE.from_arrays(spec, whole)
    b = escha.MoEHalves.from_arrays(hspec, halves)
    rng = np.random.default_rng(5201)
    for m in (1, 6):
        x = S.make_activations(rng, m, hidden)
        ids, w = S.make_routing(rng, m, E, 8)
        ya, yb = _run(a, x, ids, w), _run(b, x, ids, w)
        assert a.check() == 0 and b.check() == 0
        experts = {e: _expert(hspec, e, halves[e]) for e in set(ids.reshape(-1).tolist())}
        ref = O.moe_forward(x, experts, ids, w)
        assert worst_rel_l2(yb, ref) <= REL_L2_TOL
        assert rel_l2(yb, ya) <= 2e-4          # the same sums, grouped differently in fp32


def test_moe_halves_table_is_reread_every_call():
    """Writing other pointers and widths into the device tables between calls
    changes the layer without a new handle: point expert 3's halves at expert
    7's code (gate half 1 at a fresh 4-bit code, down at expert 7's halves)."""
    spec, codes, moe = _small(5300)
    rng = np.random.default_rng(5301)
    x = S.make_activations(rng, 2, spec["hidden"])
    ids = np.array([[3, 1, 4, 9], [3, 0, 11, 7]], dtype=np.int32)
    w = np.array([[0.4, 0.3, 0.2, 0.1], [0.25, 0.25, 0.25, 0.25]], dtype=np.float32)
    y0 = _run(moe, x, ids, w)
    assert moe.check() == 0
    ref0 = O.moe_forward(x, {e: _expert(spec, e, codes[e]) for e in range(12)}, ids, w)
    assert worst_rel_l2(y0, ref0) <= REL_L2_TOL

    t = moe.tables
    fresh = rng.integers(-32768, 32768, size=(spec["hidden"] // 16, 8, 64), dtype=np.int16)
    fresh_d = torch.from_numpy(fresh).cuda()
    t["gate_half"][3] = t["gate_half"][7]
    t["gate_bits"][3] = t["gate_bits"][7]
    t["gate_half"][3, 1] = fresh_d.data_ptr()
    t["gate_bits"][3, 1] = 4
    t["down_half"][3] = t["down_half"][7]
    t["down_bits"][3] = t["down_bits"][7]
    torch.cuda.synchronize()
    y1 = _run(moe, x, ids, w)
    assert moe.check() == 0
    spec2 = dict(spec)
    spec2["gate_bits"] = spec["gate_bits"].copy()
    spec2["gate_bits"][3] = spec["gate_bits"][7]
    spec2["gate_bits"][3, 1] = 4
    spec2["down_bits"] = spec["down_bits"].copy()
    spec2["down_bits"][3] = spec["down_bits"][7]
    g7, u7, d7 = codes[7]
    codes2 = dict(codes)
    codes2[3] = ([g7[0], fresh] + list(g7[2:]), codes[3][1], d7)
    ref1 = O.moe_forward(x, {e: _expert(spec2, e, codes2[e]) for e in range(12)}, ids, w)
    assert worst_rel_l2(y1, ref1) <= REL_L2_TOL
    assert rel_l2(y1, y0) > 0.05


@pytest.mark.parametrize("what", ["null_down", "misaligned_gate", "bad_width"])
def test_moe_halves_bad_table_entry_is_flagged_not_read(what):
    """A null or misaligned pointer, or a width outside {2,3,4}, in an entry
    of a routed expert is never dereferenced: a zero code stands in and the
    handle's error flag reports ESCHA_ERR_INVALID_ARG.  Restoring the entry
    restores the layer."""
    spec, codes, moe = _small(5400)
    rng = np.random.default_rng(5401)
    x = S.make_activations(rng, 1, spec["hidden"])
    ids = np.array([[2, 5, 6, 8]], dtype=np.int32)
    w = np.array([[0.4, 0.3, 0.2, 0.1]], dtype=np.float32)
    t = moe.tables
    if what == "null_down":
        saved = t["down_half"][5, 1].clone()
        t["down_half"][5, 1] = 0
        key = "down_half"
    elif what == "misaligned_gate":
        saved = t["gate_half"][6, 0].clone()
        t["gate_half"][6, 0] = saved + 8
        key = "gate_half"
    else:
        saved = t["up_bits"][2, 2].clone()
        t["up_bits"][2, 2] = 5
        key = "up_bits"
    torch.cuda.synchronize()
    y = _run(moe, x, ids, w)
    assert moe.check() == 1
    assert np.all(np.isfinite(y))
    if key == "down_half":
        t[key][5, 1] = saved
    elif key == "gate_half":
        t[key][6, 0] = saved
    else:
        t[key][2, 2] = saved
    torch.cuda.synchronize()
    y = _run(moe, x, ids, w)
    assert moe.check() == 0
    ref = O.moe_forward(x, {e: _expert(spec, e, codes[e]) for e in (2, 5, 6, 8)}, ids, w)
    assert worst_rel_l2(y, ref) <= REL_L2_TOL


def test_moe_halves_e4m3_rounding():
    spec, codes, moe = _small(5500)
    moe.set_rounding("e4m3")
    rng = np.random.default_rng(5501)
    x = S.make_activations(rng, 4, spec["hidden"])
    ids, w = S.make_routing(rng, 4, spec["num_experts"], 8)
    y = _run(moe, x, ids, w)
    assert moe.check() == 0
    experts = {e: _expert(spec, e, codes[e], "e4m3") for e in set(ids.reshape(-1).tolist())}
    assert worst_rel_l2(y, O.moe_forward(x, experts, ids, w)) <= REL_L2_TOL


def test_moe_halves_stages_compose_to_the_full_call():
    from gemm_trellis_tile_gb300 import escha
    spec, codes, moe = _small(5600)
    rng = np.random.default_rng(5601)
    x = torch.from_numpy(S.make_activations(rng, 3, spec["hidden"])).cuda()
    ids, w = S.make_routing(rng, 3, spec["num_experts"], 8)
    ids, w = torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda()
    full = moe.gemv(x, ids, w)
    staged = torch.empty_like(full)
    for s in range(escha.MoE.STAGES):
        moe.gemv(x, ids, w, staged, stage=s)
    assert torch.equal(full, staged)


@pytest.mark.parametrize("m", [1, 8])
def test_moe_halves_glm_shape_full_size_sampled(m):
    """256 experts, 6144 -> 2048 -> 6144, 16 halves per matrix at per-half
    widths, top-8.  Only routed experts get code words; the oracle computes
    token 0 (gate and up in full, down on three sampled 128-column blocks)."""
    from gemm_trellis_tile_gb300 import escha
    spec = S.make_moe_half_spec(S.seed_for(3, 2), 256, 6144, 2048)
    rng = np.random.default_rng(S.seed_for(3, 3) + m)
    x = S.make_activations(rng, m, 6144)
    ids, w = S.make_routing(rng, m, 256, 8)
    routed = sorted(set(ids.reshape(-1).tolist()))
    codes = {e: S.make_moe_expert_half_codes(spec, e) for e in routed}
    moe = escha.MoEHalves.from_arrays(spec, codes)
    y = _run(moe, x, ids, w)
    assert moe.check() == 0
    assert np.all(np.isfinite(y))
    blocks = [0, 23, 47]
    cols = np.concatenate([np.arange(b * 128, b * 128 + 128) for b in blocks])
    ref = np.zeros(cols.size)
    for k in range(8):
        e = int(ids[0, k])
        g, u, d = codes[e]
        su_h = O.fold_scales(spec["rin_hidden"], spec["s_in_hidden"])
        sv_h = O.fold_scales(spec["rout_hidden"], spec["s_out_hidden"])
        hg = O.linear_forward(x[:1], O.decode_column_halves(g, spec["gate_bits"][e]), su_h,
                              O.fold_scales(spec["rout_gate"][e], spec["s_out_gate"][e]))
        hu = O.linear_forward(x[:1], O.decode_column_halves(u, spec["up_bits"][e]), su_h,
                              O.fold_scales(spec["rout_up"][e], spec["s_out_up"][e]))
        h = O.silu(hg) * hu
        wd = np.concatenate([O.decode_columns(c, int(spec["down_bits"][e]), cols) for c in d],
                            axis=0)
        xh = O.had_blockwise(h * O.fold_scales(spec["rin_down"][e], spec["s_in_down"][e]))
        ref += float(w[0, k]) * (O.had_blockwise(xh @ wd.astype(np.float64)) * sv_h[cols])[0]
    assert worst_rel_l2(y[0, cols], ref) <= REL_L2_TOL
