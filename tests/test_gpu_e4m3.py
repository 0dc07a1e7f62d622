"""GPU parity of the EXLR8 E4M3 variant against the CPU oracle, through the C ABI.

With ESCHA_ROUND_E4M3 every codebook value is rounded to FP8 E4M3 (nearest
even, saturating; EXLR8 format page).  Decoded weights must equal the oracle's
E4M3 decode bit for bit; layer outputs (GEMV, GEMM, MoE) must be within
relative L2 2e-3 of the fp64 oracle fed the E4M3 weights.  The rounding moves
weights by 2.7 % RMS, so a path that skipped it would fail by an order of
magnitude.
"""

import numpy as np
import pytest

from gemm_trellis_tile_gb300 import synthetic as S
from oracle import escha_oracle as O
from tests.helpers import (REL_L2_TOL, make_linear_handle, oracle_layer_dict, oracle_linear,
                           rel_l2, worst_rel_l2)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gemm_trellis_tile_gb300 import build, escha
    build.build()
    escha.load()


@pytest.mark.parametrize("bits,k,n", [(2, 512, 512), (3, 384, 640), (4, 256, 1280)])
def test_decode_e4m3_bit_exact(bits, k, n):
    rng = np.random.default_rng(7000 + bits)
    layer = S.make_linear(rng, k, n, bits)
    lin, _ = make_linear_handle(layer)
    lin.set_rounding("e4m3")
    got = lin.decode().cpu().numpy()
    ref = O.decode_matrix(layer["code"], bits, rounding="e4m3")
    assert np.array_equal(got.view(np.uint16), ref.view(np.uint16))
    lin.set_rounding("fp16")
    got = lin.decode().cpu().numpy()
    assert np.array_equal(got.view(np.uint16), O.decode_matrix(layer["code"], bits).view(np.uint16))


@pytest.mark.parametrize("bits,k,n", [(2, 512, 512), (3, 1024, 1536), (4, 768, 640)])
def test_gemv_and_gemm_e4m3_match_oracle(bits, k, n):
    rng = np.random.default_rng(7100 + bits)
    layer = S.make_linear(rng, k, n, bits)
    lin, _ = make_linear_handle(layer)
    lin.set_rounding("e4m3")
    w8 = O.decode_matrix(layer["code"], bits, rounding="e4m3")
    w16 = O.decode_matrix(layer["code"], bits)
    for m in (1, 5, 16):
        x = S.make_activations(rng, m, k)
        xt = torch.from_numpy(x).cuda()
        ref = oracle_linear(layer, x, w8)
        y = lin.gemv(xt).cpu().numpy()
        assert worst_rel_l2(y, ref) <= REL_L2_TOL, m
        # the rounding is visible: the fp16 weights are far outside the tolerance
        assert rel_l2(oracle_linear(layer, x, w16), ref) > 5 * REL_L2_TOL
        yg = lin.gemm(xt).cpu().numpy()
        assert worst_rel_l2(yg, ref) <= REL_L2_TOL, m
    x = S.make_activations(rng, 300, k)
    assert worst_rel_l2(lin.gemm(torch.from_numpy(x).cuda()).cpu().numpy(),
                  oracle_linear(layer, x, w8)) <= REL_L2_TOL


def test_mlp_takes_each_matrix_rounding():
    from gemm_trellis_tile_gb300 import escha
    rng = np.random.default_rng(7200)
    mlp = S.make_mlp(rng, 512, 1536, 2, 3, 4)
    gate, kg = make_linear_handle(mlp["gate"])
    up, ku = make_linear_handle(mlp["up"])
    down, kd = make_linear_handle(mlp["down"])
    for h in (gate, up, down):
        h.set_rounding("e4m3")
    handle = escha.MLP(gate, up, down)
    x = S.make_activations(rng, 3, 512)
    y = handle.gemv(torch.from_numpy(x).cuda()).cpu().numpy()
    ref = O.mlp_forward(x, oracle_layer_dict(mlp["gate"], rounding="e4m3"),
                        oracle_layer_dict(mlp["up"], rounding="e4m3"),
                        oracle_layer_dict(mlp["down"], rounding="e4m3"))
    assert worst_rel_l2(y, ref) <= REL_L2_TOL


def test_moe_e4m3_matches_oracle():
    from gemm_trellis_tile_gb300 import escha
    E, hidden, inter = 16, 512, 256
    spec = S.make_moe_spec(7300, E, hidden, inter)
    codes = {e: S.make_moe_expert_codes(spec, e) for e in range(E)}
    moe = escha.MoE.from_arrays(spec, codes)
    moe.set_rounding("e4m3")
    experts = []
    for e in range(E):
        g, u, d = codes[e]
        b = int(spec["bits"][e])
        su_h = O.fold_scales(spec["rin_hidden"], spec["s_in_hidden"])
        sv_h = O.fold_scales(spec["rout_hidden"], spec["s_out_hidden"])
        experts.append((
            dict(w=O.decode_matrix(g, b, rounding="e4m3"), su=su_h,
                 sv=O.fold_scales(spec["rout_gate"][e], spec["s_out_gate"][e])),
            dict(w=O.decode_matrix(u, b, rounding="e4m3"), su=su_h,
                 sv=O.fold_scales(spec["rout_up"][e], spec["s_out_up"][e])),
            dict(w=O.decode_matrix(d, b, rounding="e4m3"),
                 su=O.fold_scales(spec["rin_down"][e], spec["s_in_down"][e]), sv=sv_h)))
    rng = np.random.default_rng(7301)
    for m in (1, 6):
        x = S.make_activations(rng, m, hidden)
        ids, w = S.make_routing(rng, m, E, 8)
        y = moe.gemv(torch.from_numpy(x).cuda(), torch.from_numpy(ids).cuda(),
                     torch.from_numpy(w).cuda()).cpu().numpy()
        assert moe.check() == 0
        assert worst_rel_l2(y, O.moe_forward(x, experts, ids, w)) <= REL_L2_TOL


def test_set_rounding_rejects_unknown_modes():
    from gemm_trellis_tile_gb300 import escha
    rng = np.random.default_rng(7400)
    lin, _ = make_linear_handle(S.make_linear(rng, 256, 256, 2))
    assert escha.load().escha_linear_set_rounding(lin.handle, 2) == 1
    assert escha.load().escha_linear_set_rounding(lin.handle, -1) == 1
