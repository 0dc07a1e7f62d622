"""GPU parity of the FP8 prefill (EXLR8 variant) against the CPU oracle, through the C ABI.

The activation quantiser decides integer codes, so its E4M3 codes and fp32
scales must equal the oracle's bit for bit.  The kind::f8f6f4 GEMM's outputs
must be within relative L2 2e-3 of the oracle's FP8 layer (E4M3 activations
and E4M3 weights, contraction and everything after it in fp64), on small,
ragged and split-tile shapes in full and on sampled blocks of the 2048-token
prefill shapes.  The activation rounding moves outputs by about 2-3 % RMS, so
a kernel that skipped it would fail by an order of magnitude.
"""

import numpy as np
import pytest

from gemm_trellis_tile_gb300 import synthetic as S
from oracle import escha_oracle as O
from tests.helpers import REL_L2_TOL, make_linear_handle, oracle_linear, oracle_scales, rel_l2

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gemm_trellis_tile_gb300 import build, escha
    build.build()
    escha.load()


def _e4m3_values(q_u8):
    return q_u8.view(torch.float8_e4m3fn).to(torch.float64).cpu().numpy()


@pytest.mark.parametrize("m,k", [(37, 640), (3, 17408), (5, 128), (1, 5120)])
def test_quantize_rows_bit_exact(m, k):
    from gemm_trellis_tile_gb300 import escha
    rng = np.random.default_rng(9100 + m + k)
    xh = S.make_activation_rows_mixed(rng, m, k) if m >= 3 else S.make_activations(rng, m, k)
    q, d = escha.quantize_e4m3_rows(torch.from_numpy(xh).cuda())
    torch.cuda.synchronize()
    q_ref, d_ref = O.quantize_rows_e4m3(xh)
    assert np.array_equal(_e4m3_values(q), q_ref)
    assert np.array_equal(d.cpu().numpy(), d_ref)


def test_quantize_rows_wide_after_narrow():
    """The quantiser's shared memory grows with K (2K bytes): a wide row (64 KB,
    above the default 48 KB limit) after a narrow one must still launch."""
    from gemm_trellis_tile_gb300 import escha
    rng = np.random.default_rng(9150)
    for k in (32768, 128, 32768):
        xh = S.make_activations(rng, 2, k)
        q, d = escha.quantize_e4m3_rows(torch.from_numpy(xh).cuda())
        torch.cuda.synchronize()
        q_ref, d_ref = O.quantize_rows_e4m3(xh)
        assert np.array_equal(_e4m3_values(q), q_ref), k
        assert np.array_equal(d.cpu().numpy(), d_ref), k


@pytest.mark.parametrize("m,k,n,bits", [(256, 128, 128, 2), (300, 512, 384, 3), (1, 256, 256, 4),
                                        (600, 1920, 1280, 2), (517, 2048, 1280, 4),
                                        (64, 384, 256, 3), (64, 8192, 256, 3)])
def test_gemm_fp8_matches_oracle(m, k, n, bits):
    """(600, 1920, 1280): tiles split between two CTAs; (64, 8192, 256): each
    of the two tiles shared by four."""
    rng = np.random.default_rng(9200 + m + k + bits)
    layer = S.make_linear(rng, k, n, bits)
    lin, _ = make_linear_handle(layer)
    lin.set_rounding("e4m3")
    x = S.make_activations(rng, m, k)
    y = lin.gemm_fp8(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    assert lin.check() == 0
    got = y.cpu().numpy()
    assert np.all(np.isfinite(got))
    w8 = O.decode_matrix(layer["code"], bits, rounding="e4m3")
    su, sv = oracle_scales(layer)
    assert rel_l2(got, O.linear_forward_fp8(x, w8, su, sv)) <= REL_L2_TOL
    # the activations really were rounded: the fp16-activation layer is far off
    assert rel_l2(got, oracle_linear(layer, x, w8)) > 3 * REL_L2_TOL


# One activation code that the two sides round differently moves its row by at
# most one E4M3 step of that code, 2^-3 |q_k|, against the row's |q|: under
# 2^-3 * 448 / |q| (q_k < 448; the largest element always maps to 448 exactly),
# 1.4e-2 for 1024 Gaussian activations.  The kernel's fp32 rotation and the
# oracle's fp64 one round xh to different fp16 neighbours for about one
# activation in 10^5, and only some of those cross an E4M3 rounding boundary.
ROW_TOL_ONE_CODE = 2e-2


def test_gemm_fp8_on_oracle_codes_per_row():
    """The contraction alone, fed the oracle's E4M3 codes of rows that span 13
    orders of magnitude (and a zero row): every row within the tolerance."""
    rng = np.random.default_rng(9300)
    layer = S.make_linear(rng, 1024, 768, 3)
    lin, _ = make_linear_handle(layer)
    lin.set_rounding("e4m3")
    w8 = O.decode_matrix(layer["code"], 3, rounding="e4m3")
    _, sv = oracle_scales(layer)
    for m in (9, 700, 4):
        xh = S.make_activation_rows_mixed(rng, m, 1024)
        q, d = O.quantize_rows_e4m3(xh)
        q8 = torch.from_numpy(q).to(torch.float8_e4m3fn).view(torch.uint8).cuda()
        got = lin.gemm_fp8_codes(q8, torch.from_numpy(d).cuda()).cpu().numpy()
        assert lin.check() == 0
        assert np.all(got[0] == 0)                        # zero row: d = 0
        ref = O.linear_forward_fp8_codes(q, d, w8, sv)
        for r in range(1, m):
            assert rel_l2(got[r], ref[r]) <= REL_L2_TOL, (m, r)


def test_gemm_fp8_mixed_rows_end_to_end_and_workspace_growth():
    rng = np.random.default_rng(9350)
    layer = S.make_linear(rng, 1024, 768, 3)
    lin, _ = make_linear_handle(layer)
    lin.set_rounding("e4m3")
    w8 = O.decode_matrix(layer["code"], 3, rounding="e4m3")
    su, sv = oracle_scales(layer)
    for m in (9, 700, 4):
        x = S.make_activation_rows_mixed(rng, m, 1024)
        got = lin.gemm_fp8(torch.from_numpy(x).cuda()).cpu().numpy()
        assert lin.check() == 0
        assert np.all(got[0] == 0)
        ref = O.linear_forward_fp8(x, w8, su, sv)
        rows = [rel_l2(got[r], ref[r]) for r in range(1, m)]
        assert max(rows) <= ROW_TOL_ONE_CODE, (m, max(rows))
        assert np.median(rows) <= REL_L2_TOL, m


def test_gemm_fp8_requires_the_e4m3_rounding():
    from gemm_trellis_tile_gb300 import escha
    rng = np.random.default_rng(9400)
    layer = S.make_linear(rng, 256, 256, 2)
    lin, _ = make_linear_handle(layer)
    x = torch.from_numpy(S.make_activations(rng, 4, 256)).cuda()
    with pytest.raises(escha.EschaError) as e:
        lin.gemm_fp8(x)
    assert e.value.status == 2


@pytest.mark.parametrize("k,n,blocks", [(5120, 17408, [0, 67, 135]), (17408, 5120, [0, 21, 39])])
def test_gemm_fp8_prefill_full_size_sampled(k, n, blocks):
    """M = 2048 tokens at 3 bits, both prefill shapes; all rows of sampled blocks."""
    rng = np.random.default_rng(S.seed_for(4, k))
    layer = S.make_linear(rng, k, n, 3)
    lin, _ = make_linear_handle(layer)
    lin.set_rounding("e4m3")
    x = S.make_activations(rng, 2048, k)
    y = lin.gemm_fp8(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    assert lin.check() == 0
    got = y.cpu().numpy()
    assert np.all(np.isfinite(got))
    su, sv = oracle_scales(layer)
    cols, ref = O.linear_forward_fp8_columns(x, layer["code"], 3, su, sv, blocks)
    assert rel_l2(got[:, cols], ref) <= REL_L2_TOL
