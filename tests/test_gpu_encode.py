"""GPU trellis encoder (Viterbi search, tail-biting) against the CPU oracle.

The encoder's output is an integer code, so parity is bit for bit: for every
tile the GPU search must pick the same path as the oracle's fp32 search (same
arithmetic, same tie rules), and report the same path cost.  At sizes the
oracle cannot encode in seconds the tests check sampled tiles against the
oracle and properties that hold at any size: the reported cost is the squared
error of the decoded code, and the rate-distortion bound of a Gaussian source
holds with the encoder close to it.
"""

import numpy as np
import pytest

from oracle import escha_oracle as O

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

CODEBOOK_STD = 1.244  # RMS of the cb=1 codebook values: sources at this scale use it fully


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gemm_trellis_tile_gb300 import build, escha
    build.build()
    escha.load()


def _encode(w, bits, rounding="fp16"):
    from gemm_trellis_tile_gb300 import escha
    code, err = escha.trellis_encode(torch.from_numpy(w).cuda(), bits, rounding, sq_err=True)
    torch.cuda.synchronize()
    return code.cpu().numpy(), err.cpu().numpy()


def _tile_values(w, i, j):
    tile = w[16 * i:16 * i + 16, 16 * j:16 * j + 16].reshape(-1)
    return tile[O.perm_forward()]


def _check_tiles(w, bits, rounding, code, err, tiles):
    for i, j in tiles:
        ref, _, total = O.viterbi_encode_tile(_tile_values(w, i, j), bits, rounding)
        assert np.array_equal(code[i, j], ref), (i, j)
        assert np.float32(err[i, j]) == np.float32(total), (i, j, err[i, j], total)


@pytest.mark.parametrize("bits,k,n", [(2, 32, 32), (3, 48, 16), (4, 16, 48)])
def test_encode_matches_oracle_bit_exact(bits, k, n):
    rng = np.random.default_rng(1100 + bits)
    w = (rng.standard_normal((k, n)) * CODEBOOK_STD).astype(np.float32)
    code, err = _encode(w, bits)
    assert code.shape == (k // 16, n // 16, 16 * bits)
    assert np.array_equal(code, O.encode_matrix(w, bits))
    _check_tiles(w, bits, "fp16", code, err, [(i, j) for i in range(k // 16) for j in range(n // 16)])


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_encode_e4m3_matches_oracle_bit_exact(bits):
    rng = np.random.default_rng(1200 + bits)
    w = (rng.standard_normal((32, 16)) * CODEBOOK_STD).astype(np.float32)
    code, err = _encode(w, bits, "e4m3")
    _check_tiles(w, bits, "e4m3", code, err, [(0, 0), (1, 0)])


def test_encode_degenerate_tiles():
    """All-zero tiles (ties everywhere: the lowest-t and lowest-state rules decide),
    a constant tile far outside the codebook's range, and an exactly
    representable tile (a decoded code: cost 0)."""
    rng = np.random.default_rng(1300)
    exact = O.decode_matrix(rng.integers(-32768, 32768, size=(1, 1, 32), dtype=np.int16), 2)
    w = np.zeros((16, 48), dtype=np.float32)
    w[:, 16:32] = 40.0
    w[:, 32:48] = exact.astype(np.float32)
    code, err = _encode(w, 2)
    _check_tiles(w, 2, "fp16", code, err, [(0, 0), (0, 1), (0, 2)])
    assert err[0, 2] == 0.0


def test_encode_large_layer_sampled_and_bounded():
    """A 1024 x 2048 layer (8192 tiles, every SM persistent over many tiles):
    sampled tiles equal the oracle's, each reported cost is the decoded code's
    squared error, and the whole layer sits between the Gaussian bound 2^-R and
    1.2 x of it."""
    bits = 2
    rng = np.random.default_rng(1400)
    w = (rng.standard_normal((1024, 2048)) * CODEBOOK_STD).astype(np.float32)
    code, err = _encode(w, bits)
    kt, nt = 64, 128
    picks = [(0, 0), (kt - 1, nt - 1), (17, 93), (40, 5)]
    _check_tiles(w, bits, "fp16", code, err, picks)
    dec = O.decode_matrix(code, bits).astype(np.float64)
    diff2 = ((dec - w.astype(np.float64)) ** 2).reshape(kt, 16, nt, 16).sum(axis=(1, 3))
    assert np.allclose(err.astype(np.float64), diff2, rtol=1e-4, atol=1e-6)
    rel = np.sqrt(diff2.sum() / np.sum(w.astype(np.float64) ** 2))
    assert 2.0 ** -bits <= rel <= 1.2 * 2.0 ** -bits
