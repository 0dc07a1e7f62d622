"""GPU parity of the tcgen05 prefill GEMM against the CPU oracle, through the C ABI.

Outputs must be within relative L2 2e-3 of the fp64 oracle.  Small and ragged
shapes (M not a multiple of the 256-row tile, single rows) are compared in
full; the 2048-token prefill shapes are compared on all rows of sampled
128-column blocks.
"""

import numpy as np
import pytest

from gemm_trellis_tile_gb300 import synthetic as S
from oracle import escha_oracle as O
from tests.helpers import (REL_L2_TOL, make_linear_handle, oracle_linear, oracle_scales,
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


@pytest.mark.parametrize("m,k,n,bits", [(256, 128, 128, 2), (300, 512, 384, 3), (1, 256, 256, 4),
                                        (1000, 1024, 640, 2), (517, 2048, 1280, 4),
                                        (64, 384, 256, 3), (64, 17408, 256, 2)])
def test_gemm_matches_oracle(m, k, n, bits):
    """(64, 17408, 256): each of the two tiles is shared by 17 CTAs."""
    rng = np.random.default_rng(5000 + m + k + bits)
    layer = S.make_linear(rng, k, n, bits)
    lin, _ = make_linear_handle(layer)
    x = S.make_activations(rng, m, k)
    y = lin.gemm(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    assert lin.check() == 0
    got = y.cpu().numpy()
    assert np.all(np.isfinite(got))
    assert worst_rel_l2(got, oracle_linear(layer, x)) <= REL_L2_TOL


def test_gemm_is_bit_reproducible_with_shared_tiles():
    """Shared tiles are finished by whichever CTA arrives last, always summing
    the CTAs' partials in CTA order: repeated calls give the same bits."""
    rng = np.random.default_rng(5050)
    layer = S.make_linear(rng, 2048, 1280, 3)
    lin, _ = make_linear_handle(layer)
    x = torch.from_numpy(S.make_activations(rng, 517, 2048)).cuda()
    first = lin.gemm(x).cpu().numpy().view(np.uint16)
    for _ in range(4):
        again = lin.gemm(x).cpu().numpy().view(np.uint16)
        assert np.array_equal(first, again)
    assert lin.check() == 0


def test_gemm_agrees_with_gemv_and_grows_workspace():
    rng = np.random.default_rng(5100)
    layer = S.make_linear(rng, 1024, 1536, 3)
    lin, _ = make_linear_handle(layer)
    w = O.decode_matrix(layer["code"], 3)
    for m in (8, 16, 700, 3):
        x = S.make_activations(rng, m, 1024)
        xt = torch.from_numpy(x).cuda()
        yg = lin.gemm(xt).cpu().numpy()
        ref = oracle_linear(layer, x, w)
        assert worst_rel_l2(yg, ref) <= REL_L2_TOL, m
        if m <= 16:
            yv = lin.gemv(xt).cpu().numpy()
            assert worst_rel_l2(yg, yv) <= REL_L2_TOL
    lin.reserve(4096)
    x = S.make_activations(rng, 5, 1024)
    assert worst_rel_l2(lin.gemm(torch.from_numpy(x).cuda()).cpu().numpy(),
                  oracle_linear(layer, x, w)) <= REL_L2_TOL


@pytest.mark.parametrize("k,n,blocks", [(5120, 17408, [0, 67, 135]), (17408, 5120, [0, 21, 39])])
def test_gemm_prefill_full_size_sampled(k, n, blocks):
    """M = 2048 tokens at 3 bits, both prefill shapes; all rows of sampled blocks."""
    rng = np.random.default_rng(S.seed_for(4, k))
    layer = S.make_linear(rng, k, n, 3)
    lin, _ = make_linear_handle(layer)
    x = S.make_activations(rng, 2048, k)
    y = lin.gemm(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    assert lin.check() == 0
    got = y.cpu().numpy()
    assert np.all(np.isfinite(got))
    su, sv = oracle_scales(layer)
    cols, ref = O.linear_forward_columns(x, layer["code"], 3, su, sv, blocks)
    assert worst_rel_l2(got[:, cols], ref) <= REL_L2_TOL
