"""Pins of the CPU oracle against what the pages and mathematics fix.

Every check here compares the oracle with something other than itself: a
decoder printed on the pages, a value printed on the pages, a library routine
(torch fp16 arithmetic, scipy's Hadamard), the PTX ISA fragment table, a
closed form, an invariant, or brute force on tiny inputs.
"""

import json
import os

import numpy as np
import pytest
import scipy.linalg
import torch

from oracle import escha_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_constants.json")


def golden(key):
    with open(GOLDEN) as f:
        return json.load(f)[key]["value"]


def random_tiles(rng, n, bits):
    return rng.integers(-32768, 32768, size=(n, 16 * bits), dtype=np.int16)


# ---------------------------------------------------------------- fp16 helpers

def test_numpy_half_decode_matches_torch_all_bit_patterns():
    u16 = np.arange(65536, dtype=np.uint16)
    ours = u16.view(np.float16).astype(np.float64)
    ref = torch.from_numpy(u16.view(np.int16)).view(torch.float16).double().numpy()
    finite = np.isfinite(ref)
    assert np.array_equal(ours[finite], ref[finite])
    assert np.array_equal(np.isnan(ours), np.isnan(ref))


def test_numpy_double_to_half_rounds_correctly():
    """numpy's fp64 -> fp16 is one round-to-nearest-even step.

    Checked against Python's struct 'e' packing (a correctly rounded
    double -> half conversion), including exact ties and values just off a tie.
    torch is only used for fp32 inputs: its fp64 -> fp16 goes through fp32.
    """
    import struct
    rng = np.random.default_rng(1)
    x = rng.normal(0, 2, 50000)
    h = np.arange(0x3000, 0x4400, dtype=np.uint16).view(np.float16).astype(np.float64)
    ties = (h[:-1] + h[1:]) / 2
    x = np.concatenate([x, ties, -ties, np.nextafter(ties, 0), np.nextafter(ties, 10)])
    ours = x.astype(np.float16).view(np.uint16)
    ref = np.array([struct.unpack('<H', struct.pack('<e', v))[0] for v in x], dtype=np.uint16)
    assert np.array_equal(ours, ref)
    x32 = x.astype(np.float32)
    t = torch.from_numpy(x32).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(x32.astype(np.float16).view(np.uint16), t)


# ---------------------------------------------------------------- codebook

def test_codebook_equals_torch_fp16_add_all_states():
    """fp16_lo + fp16_hi as an fp16 addition, checked with torch's CPU half add."""
    states = np.arange(65536)
    lo, hi = O.codebook_halves(states)
    ref = (torch.from_numpy(lo.view(np.int16)).view(torch.float16)
           + torch.from_numpy(hi.view(np.int16)).view(torch.float16))
    ours = O.codebook_value(states)
    assert np.array_equal(ours.view(np.uint16), ref.view(torch.int16).numpy().view(np.uint16))


def test_codebook_state_zero_by_hand():
    # v = 0 -> (0 & mask) ^ 0x3B603B60: both halves 0x3B60 = 2^-1 * (1 + 864/1024)
    half = 0.5 * (1 + 864 / 1024)
    assert O.codebook_value(np.array([0]))[0] == np.float16(2 * half)
    # state 1: v = 0xCBAC1FED -> masked 0x8BAC0FED -> xor -> 0xB0CC348D
    v = ((0xCBAC1FED & 0x8FFF8FFF) ^ 0x3B603B60)
    assert v == 0xB0CC348D
    lo = np.uint16(v & 0xFFFF).view(np.float16).astype(np.float64)
    hi = np.uint16(v >> 16).view(np.float16).astype(np.float64)
    assert O.codebook_value(np.array([1]))[0] == np.float16(lo + hi)


def test_codebook_halves_have_forced_exponent():
    """The mask/xor forces each half's exponent to 12..15: |half| in [0.125, 2)."""
    lo, hi = O.codebook_halves(np.arange(65536))
    for h in (lo, hi):
        a = np.abs(h.astype(np.float64))
        assert a.min() >= 0.125 and a.max() < 2.0


def test_codebook_std_matches_printed_codebook_scale():
    """Std of the decoded values over all states vs EXL3's codebook_scale 1.24371088."""
    vals = O.codebook_value(np.arange(65536)).astype(np.float64)
    scale = golden("codebook_scale")
    assert abs(vals.std() - scale) / scale < 1e-3
    # the page's measured inner-domain std (1.2318) is within 1% as well
    assert abs(vals.std() - golden("inner_domain_std_measured")) / vals.std() < 0.01


def _hand_value(state):
    """Codebook value of one state computed by hand from the printed constants."""
    v = (state * 0xCBAC1FED) & 0xFFFFFFFF
    v = (v & 0x8FFF8FFF) ^ 0x3B603B60
    return np.float16(np.uint16(v & 0xFFFF).view(np.float16).astype(np.float64)
                      + np.uint16(v >> 16).view(np.float16).astype(np.float64))


@pytest.mark.parametrize("mutation", ["mult", "mask", "xor_forced_bits", "xor_free_bits", "nosum"])
def test_codebook_pins_reject_plausible_mistakes(mutation, monkeypatch):
    """Each plausible slip in the codebook fails at least one of the pins above.

    A changed multiplier or a changed XOR in bits the mask lets through only
    permutes the value multiset (the std cannot see it); the by-hand values of
    states 0 and 1 can.  A changed mask, a changed XOR in the forced exponent
    bits, or a dropped half moves the std off the printed codebook scale.
    """
    if mutation == "mult":
        monkeypatch.setattr(O, "MCG_MULT", 0xCBAC1FEB)
    elif mutation == "mask":
        monkeypatch.setattr(O, "MCG_MASK", 0x9FFF9FFF)
    elif mutation == "xor_forced_bits":
        monkeypatch.setattr(O, "MCG_XOR", 0x2B602B60)
    elif mutation == "xor_free_bits":
        monkeypatch.setattr(O, "MCG_XOR", 0x3C603C60)
    states = np.arange(65536)
    if mutation == "nosum":
        lo, _ = O.codebook_halves(states)
        vals = lo.astype(np.float64)
    else:
        vals = O.codebook_value(states).astype(np.float64)
    scale = golden("codebook_scale")
    std_off = abs(vals.std() - scale) / scale > 5e-3
    hand_off = (O.codebook_value(np.array([0]))[0] != _hand_value(0)
                or O.codebook_value(np.array([1]))[0] != _hand_value(1))
    if mutation == "nosum":
        assert std_off
    else:
        assert std_off or hand_off


# ---------------------------------------------------------------- bit layout

def test_words_per_tile_printed():
    printed = golden("code_words_per_tile")
    for b, w in printed.items():
        assert O.words_per_tile(int(b)) == w


def test_stream_model_equals_printed_k2_decoder():
    rng = np.random.default_rng(2)
    tiles = random_tiles(rng, 512, 2)
    assert np.array_equal(O.tile_states(tiles, 2), O.tile_states_k2_printed(tiles))


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_overlap_invariant_including_wrap(bits):
    """State t+1 begins with state t's last 16-bits bits (including 255 -> 0)."""
    rng = np.random.default_rng(3 + bits)
    st = O.tile_states(random_tiles(rng, 256, bits), bits).astype(np.int64)
    nxt = np.roll(st, -1, axis=-1)
    mask = (1 << (16 - bits)) - 1
    assert np.array_equal(st & mask, nxt >> bits)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_single_bit_flip_locality(bits):
    """Flipping stream bit p changes exactly the states whose window covers p, at the right bit."""
    rng = np.random.default_rng(10 + bits)
    n = 256 * bits
    base_bits = rng.integers(0, 2, size=n).astype(np.uint8)
    base = O.tile_states(O.pack_stream_bits(base_bits), bits).astype(np.int64)
    for p in list(range(0, n, 37)) + [0, n - 1, n - 16, 15]:
        flipped_bits = base_bits.copy()
        flipped_bits[p] ^= 1
        st = O.tile_states(O.pack_stream_bits(flipped_bits), bits).astype(np.int64)
        diff = st ^ base
        for s in range(256):
            start = (bits * (s + 1) - 16) % n
            offset = (p - start) % n
            if offset < 16:
                assert diff[s] == 1 << (15 - offset), (p, s)
            else:
                assert diff[s] == 0, (p, s)


def test_k2_word_pairing_by_hand():
    """A lone set bit at the MSB of uint32 word 0 (high int16 of the first pair).

    That is stream bit 0.  At bits=2 state s ends at bit 2s+1, so bit 0 lies in the
    windows of states 0..7 (state 0 ends at bit 1) and wraps for state 255.
    The printed decoder gives the same.
    """
    code = np.zeros((1, 32), dtype=np.uint16)
    code[0, 1] = 0x8000           # word 0 = u16[0] | u16[1] << 16 -> bit 31
    tiles = code.view(np.int16)
    st = O.tile_states(tiles, 2)[0]
    expect = np.zeros(256, dtype=np.int64)
    for s in range(256):
        start = (2 * (s + 1) - 16) % 512
        off = (0 - start) % 512
        if off < 16:
            expect[s] = 1 << (15 - off)
    assert np.array_equal(st, expect)
    assert np.array_equal(O.tile_states_k2_printed(tiles)[0], expect)
    assert expect[0] == 1 << 1 and expect[7] == 1 << 15 and expect[255] == 0


# ---------------------------------------------------------------- permutation

def test_perm_is_bijection():
    perm = O.perm_forward()
    assert sorted(perm.tolist()) == list(range(256))


def test_perm_matches_ptx_m16n8k16_b_fragments():
    """Lane L = 4g + t holds symbols 8L..8L+7 = the B fragments of two m16n8k16 MMAs.

    PTX ISA, mma.m16n8k16 .f16 B fragment: b0 = (B[2t][g], B[2t+1][g]),
    b1 = (B[2t+8][g], B[2t+9][g]); the second MMA covers columns 8..15.
    Tile rows are B's k (input channel), columns its n (output channel).
    """
    perm = O.perm_forward()
    for lane in range(32):
        g, t = lane // 4, lane % 4
        for j in range(8):
            nh, reg, half = j // 4, (j // 2) % 2, j % 2
            k = 2 * t + half + 8 * reg
            n = g + 8 * nh
            assert perm[8 * lane + j] == k * 16 + n


def test_perm_closed_form_row_pairs():
    """[MLX]: r = 8*rh + 2*q + {0,1}; e = r & 1; both rows of a lane pair map to one t."""
    for c in range(16):
        for q in range(4):
            for rh in range(2):
                t = 4 * (4 * (c & 7) + q) + 2 * ((c >> 3) & 1) + rh
                for e in range(2):
                    r = 8 * rh + 2 * q + e
                    assert O.perm_symbol_of(r, c) == 2 * t + e


def test_decode_matrix_tile_placement():
    """code[i, j] lands at W_inner[16i:16i+16, 16j:16j+16], K-tile index major."""
    rng = np.random.default_rng(5)
    code = rng.integers(-32768, 32768, size=(3, 5, 32), dtype=np.int16)
    w = O.decode_matrix(code, 2)
    assert w.shape == (48, 80)
    for i in range(3):
        for j in range(5):
            tile = O.decode_tiles(code[i, j], 2)
            assert np.array_equal(w[16 * i:16 * i + 16, 16 * j:16 * j + 16].view(np.uint16),
                                  tile.view(np.uint16))
    cols = np.array([0, 17, 33, 79])
    assert np.array_equal(O.decode_columns(code, 2, cols).view(np.uint16),
                          w[:, cols].view(np.uint16))


def test_decode_tile_brute_force_single_symbol():
    """Build a tile whose stream makes one state distinctive and find its value by hand."""
    bits = 3
    n = 256 * bits
    rng = np.random.default_rng(6)
    stream = rng.integers(0, 2, size=n).astype(np.uint8)
    tile = O.pack_stream_bits(stream)
    w = O.decode_tiles(tile, bits)
    for s in (0, 1, 77, 255):
        start = bits * (s + 1) - 16
        state = 0
        for i in range(16):
            state = (state << 1) | int(stream[(start + i) % n])
        v = (state * 0xCBAC1FED) & 0xFFFFFFFF
        v = (v & 0x8FFF8FFF) ^ 0x3B603B60
        val = np.float16(np.uint16(v & 0xFFFF).view(np.float16).astype(np.float64)
                         + np.uint16(v >> 16).view(np.float16).astype(np.float64))
        lane, j = s // 8, s % 8
        g, t = lane // 4, lane % 4
        k = 2 * t + (j % 2) + 8 * ((j // 2) % 2)
        c = g + 8 * (j // 4)
        assert w[k, c] == val


# ---------------------------------------------------------------- Hadamard

def test_hadamard_matches_scipy_and_closed_form():
    h = O.sylvester_hadamard(128)
    assert np.array_equal(h, scipy.linalg.hadamard(128).astype(np.float64))
    a = np.arange(128)
    pc = np.vectorize(lambda v: bin(v).count("1"))(a[:, None] & a[None, :])
    assert np.array_equal(h, (-1.0) ** pc)


def test_hadamard_symmetric_orthogonal_self_inverse():
    h = O.had128_matrix()
    assert np.array_equal(h, h.T)
    assert np.allclose(h @ h, np.eye(128), atol=1e-13)
    rng = np.random.default_rng(7)
    x = rng.normal(size=(3, 384))
    assert np.allclose(O.had_blockwise(O.had_blockwise(x)), x, atol=1e-12)
    assert np.allclose(np.linalg.norm(O.had_blockwise(x), axis=1), np.linalg.norm(x, axis=1))
    assert np.allclose(O.had_blockwise(x), x @ O.blockdiag_hadamard(384), atol=1e-12)


def test_hadamard_blocks_are_independent():
    x = np.zeros((1, 256))
    x[0, 130] = 1.0
    y = O.had_blockwise(x)
    assert np.all(y[0, :128] == 0) and np.allclose(np.abs(y[0, 128:]), 1 / np.sqrt(128))


# ---------------------------------------------------------------- layers

def make_small_layer(rng, k, n, bits):
    code = rng.integers(-32768, 32768, size=(k // 16, n // 16, 16 * bits), dtype=np.int16)
    rin = rng.normal(1, 0.1, k).astype(np.float16)
    rout = rng.normal(1, 0.1, n).astype(np.float16)
    s_in = rng.uniform(0.98, 1.02, k).astype(np.float32)
    s_out = rng.uniform(0.98, 1.02, n).astype(np.float32)
    return code, rin, rout, s_in, s_out


@pytest.mark.parametrize("k,n,bits", [(128, 128, 2), (256, 384, 3), (384, 256, 4)])
def test_activation_route_equals_weight_route(k, n, bits):
    rng = np.random.default_rng(8 + bits)
    code, rin, rout, s_in, s_out = make_small_layer(rng, k, n, bits)
    w_inner = O.decode_matrix(code, bits)
    su, sv = O.fold_scales(rin, s_in), O.fold_scales(rout, s_out)
    x = rng.normal(size=(5, k)).astype(np.float16)
    y_act = O.linear_forward(x, w_inner, su, sv)
    y_w = x.astype(np.float64) @ O.reconstruct_weight(w_inner, su, sv)
    assert np.allclose(y_act, y_w, rtol=1e-10, atol=1e-9)


def test_layer_brute_force_loops():
    """Per-element loops on a 128x128 layer, one token."""
    rng = np.random.default_rng(9)
    code, rin, rout, s_in, s_out = make_small_layer(rng, 128, 128, 2)
    w = O.decode_matrix(code, 2).astype(np.float64)
    su, sv = O.fold_scales(rin, s_in), O.fold_scales(rout, s_out)
    x = rng.normal(size=128)
    H = [[(-1.0) ** bin(a & b).count("1") / np.sqrt(128) for b in range(128)] for a in range(128)]
    xh = [sum(x[a] * su[a] * H[a][k] for a in range(128)) for k in range(128)]
    yp = [sum(xh[k] * w[k, n] for k in range(128)) for n in range(128)]
    y = [sum(yp[b] * H[b][n] for b in range(128)) * sv[n] for n in range(128)]
    assert np.allclose(O.linear_forward(x[None, :], w, su, sv)[0], y, rtol=1e-10, atol=1e-10)


def test_layer_rejects_transposed_weight():
    rng = np.random.default_rng(10)
    code, rin, rout, s_in, s_out = make_small_layer(rng, 128, 128, 2)
    w = O.decode_matrix(code, 2)
    su, sv = O.fold_scales(rin, s_in), O.fold_scales(rout, s_out)
    x = rng.normal(size=(2, 128))
    assert not np.allclose(O.linear_forward(x, w, su, sv), O.linear_forward(x, w.T, su, sv))


def test_linear_forward_columns_matches_full():
    rng = np.random.default_rng(11)
    code, rin, rout, s_in, s_out = make_small_layer(rng, 256, 512, 3)
    su, sv = O.fold_scales(rin, s_in), O.fold_scales(rout, s_out)
    x = rng.normal(size=(3, 256))
    full = O.linear_forward(x, O.decode_matrix(code, 3), su, sv)
    cols, part = O.linear_forward_columns(x, code, 3, su, sv, [1, 3])
    assert np.allclose(full[:, cols], part, rtol=1e-12, atol=1e-12)


def test_moe_single_output_rotation_by_linearity():
    """sum_k w_k had(y_k) sv == had(sum_k w_k y_k) sv: one rotation serves all experts."""
    rng = np.random.default_rng(12)
    ys = rng.normal(size=(8, 256))
    w = rng.random(8)
    sv = rng.uniform(0.5, 1.5, 256)
    a = sum(w[k] * O.had_blockwise(ys[k:k + 1])[0] * sv for k in range(8))
    b = O.had_blockwise((w[:, None] * ys).sum(0, keepdims=True))[0] * sv
    assert np.allclose(a, b, rtol=1e-12, atol=1e-12)


def test_mlp_brute_force_loops_gate_takes_the_silu():
    """down(silu(gate(x)) * up(x)) on a 128 -> 256 -> 128 MLP, two tokens, by
    per-element loops: Hadamard entries from their sign formula, each layer by
    the activation route, SiLU as z / (1 + e^-z) with math.exp.  Gate and up
    are distinct matrices scaled so that their outputs are O(1), where SiLU is
    far from linear; swapping their roles, or another activation, moves the
    result by O(1) relative."""
    import math
    rng = np.random.default_rng(14)

    def layer(k, n, b, scale):
        code, rin, rout, s_in, s_out = make_small_layer(rng, k, n, b)
        return dict(w=O.decode_matrix(code, b).astype(np.float64), su=O.fold_scales(rin, s_in),
                    sv=O.fold_scales(rout, s_out) * scale)
    gate, up, down = layer(128, 256, 2, 1 / 16), layer(128, 256, 3, 1 / 16), layer(256, 128, 4, 1.0)
    x = rng.normal(size=(2, 128))
    H = [[(-1.0) ** bin(a & b).count("1") / math.sqrt(128) for b in range(128)] for a in range(128)]

    def had(v):
        out = [0.0] * len(v)
        for b0 in range(0, len(v), 128):
            for k in range(128):
                out[b0 + k] = sum(v[b0 + a] * H[a][k] for a in range(128))
        return out

    def lin(v, L):
        k_in, n_out = L["w"].shape
        xh = had([v[a] * L["su"][a] for a in range(k_in)])
        yp = [sum(xh[k] * L["w"][k, n] for k in range(k_in)) for n in range(n_out)]
        return [t * L["sv"][n] for n, t in enumerate(had(yp))]

    def mlp_loops(v, first, second):
        g, u = lin(v, first), lin(v, second)
        return lin([g[j] / (1.0 + math.exp(-g[j])) * u[j] for j in range(len(g))], down)

    ours = O.mlp_forward(x, gate, up, down)
    for t in range(2):
        ref = np.array(mlp_loops(list(x[t]), gate, up))
        assert np.allclose(ours[t], ref, rtol=1e-10, atol=1e-10 * np.abs(ref).max())
        swapped = np.array(mlp_loops(list(x[t]), up, gate))
        assert np.linalg.norm(swapped - ref) > 0.1 * np.linalg.norm(ref)
    g = O.linear_forward(x, gate["w"], gate["su"], gate["sv"])
    assert 0.3 < np.std(g) < 3.0           # SiLU acts in its curved range


def test_moe_forward_reduces_to_mlp():
    rng = np.random.default_rng(13)

    def layer(k, n, b):
        code, rin, rout, s_in, s_out = make_small_layer(rng, k, n, b)
        return dict(w=O.decode_matrix(code, b), su=O.fold_scales(rin, s_in),
                    sv=O.fold_scales(rout, s_out))
    experts = [(layer(128, 256, 2), layer(128, 256, 2), layer(256, 128, 2)) for _ in range(3)]
    x = rng.normal(size=(2, 128))
    ids = np.array([[1, 2], [0, 1]])
    wts = np.array([[1.0, 0.0], [0.25, 0.75]])
    y = O.moe_forward(x, experts, ids, wts)
    assert np.allclose(y[0], O.mlp_forward(x[0:1], *experts[1])[0])
    ref1 = 0.25 * O.mlp_forward(x[1:2], *experts[0])[0] + 0.75 * O.mlp_forward(x[1:2], *experts[1])[0]
    assert np.allclose(y[1], ref1)



@pytest.mark.parametrize("bits", [2, 3, 4])
def test_halves_reassemble_the_whole_matrix(bits):
    """EXLR8 halves: gate/up are cut along their output channels, down along its
    input channels, 128 channels (8 tiles) per half.  Cutting one whole code
    tensor at every 8th tile column (row) and decoding the halves one by one
    must give the whole matrix's decode -- a half cut along the wrong axis, or
    halves put back in the wrong order, fails."""
    rng = np.random.default_rng(21 + bits)
    code = rng.integers(-32768, 32768, size=(8, 32, 16 * bits), dtype=np.int16)   # 128 x 512
    whole = O.decode_matrix(code, bits).view(np.uint16)
    cols = [code[:, 8 * h:8 * h + 8] for h in range(4)]
    assert np.array_equal(O.decode_column_halves(cols, [bits] * 4).view(np.uint16), whole)
    assert not np.array_equal(O.decode_column_halves(cols[::-1], [bits] * 4).view(np.uint16), whole)
    code_t = rng.integers(-32768, 32768, size=(32, 8, 16 * bits), dtype=np.int16)  # 512 x 128
    whole_t = O.decode_matrix(code_t, bits).view(np.uint16)
    rows = [code_t[8 * h:8 * h + 8] for h in range(4)]
    assert np.array_equal(O.decode_row_halves(rows, bits).view(np.uint16), whole_t)


def test_mixed_width_halves_place_each_half_by_its_own_width():
    """A half's width changes only its own 128 columns: recoding one half at
    another width leaves every other column of the matrix bit-identical, and a
    single-symbol brute force lands the changed weight in that half's block."""
    rng = np.random.default_rng(25)
    widths = [2, 4, 3]
    halves = [rng.integers(-32768, 32768, size=(4, 8, 16 * b), dtype=np.int16) for b in widths]
    w = O.decode_column_halves(halves, widths).view(np.uint16)
    assert w.shape == (64, 384)
    alt = list(halves)
    alt[1] = rng.integers(-32768, 32768, size=(4, 8, 16 * 2), dtype=np.int16)
    w2 = O.decode_column_halves(alt, [2, 2, 3]).view(np.uint16)
    assert np.array_equal(w2[:, :128], w[:, :128]) and np.array_equal(w2[:, 256:], w[:, 256:])
    # flip one code bit of tile (2, 5) of half 2: only that tile's weights move
    flip = [h.copy() for h in halves]
    flip[2][2, 5, 0] ^= np.int16(1)
    diff = np.nonzero(O.decode_column_halves(flip, widths).view(np.uint16) != w)
    assert diff[0].size > 0
    assert set(diff[0] // 16) == {2} and set(diff[1] // 16) == {2 * 8 + 5}


def test_half_shape_and_byte_accounting_match_the_pages():
    """A half is 128 inner channels x 6144 (about 786k weights), 16 per matrix,
    three matrices per expert (37,748,736 weights); two halves make a
    256-channel fragment whose size at K = 2, 3, 4 is a multiple of 64 KiB
    (32*K bytes per 256-weight tile)."""
    half = golden("half")
    pair = golden("half_pair_alignment")
    hidden, inter = half["hidden"], 2048
    assert inter // half["inner_channels"] == half["halves_per_matrix"]
    weights = half["inner_channels"] * hidden
    assert abs(weights - half["weights_about"]) / half["weights_about"] < 0.01
    assert 3 * half["halves_per_matrix"] * weights == golden("expert_weights")
    for k in (2, 3, 4):
        pair_bytes = (pair["pair_channels"] * hidden // 256) * 32 * k
        assert pair_bytes % pair["align_bytes"] == 0



def test_rms_norm_weight_offset_reproduces_the_pages_table():
    """The Metal page's table: a stored escha norm weight plus 1 gives the base
    weight for the offset tensors (residual at bf16 rounding), and the
    linear-attention gated norm carries no offset.  On a constant input (and
    eps = 0) RMSNorm returns exactly the applied weight."""
    for row in golden("rmsnorm_offset_table"):
        x = np.full((1, 4), 2.5)
        w = np.full(4, row["escha"])
        y = O.rms_norm(x, w, 0.0, stored_minus_one=row["offset"])
        assert np.allclose(y, row["base"], atol=1e-12)
        assert abs(row["escha"] + (1.0 if row["offset"] else 0.0) - row["base"]) < 1e-9
        other = O.rms_norm(x, w, 0.0, stored_minus_one=not row["offset"])
        assert abs(other[0, 0] - row["base"]) > 0.99          # the trap the page describes


def test_rms_norm_closed_forms():
    """x = (3, 4): mean square 12.5; scale invariance; unit RMS for unit weight;
    a zero row stays zero (eps > 0); brute-force loops on a random case."""
    y = O.rms_norm(np.array([[3.0, 4.0]]), np.zeros(2), 0.0)
    assert np.allclose(y, [[3.0 / np.sqrt(12.5), 4.0 / np.sqrt(12.5)]], rtol=1e-15)
    rng = np.random.default_rng(30)
    x = rng.normal(size=(3, 64))
    w = rng.normal(size=64) * 0.1
    assert np.allclose(O.rms_norm(7.0 * x, w, 0.0), O.rms_norm(x, w, 0.0), rtol=1e-12)
    u = O.rms_norm(x, np.zeros(64), 0.0)
    assert np.allclose(np.sqrt(np.mean(u * u, axis=1)), 1.0, rtol=1e-12)
    assert np.array_equal(O.rms_norm(np.zeros((1, 8)), np.zeros(8), 1e-6), np.zeros((1, 8)))
    eps = 1e-3
    ref = np.empty_like(x)
    for i in range(3):
        ms = sum(v * v for v in x[i]) / 64
        for j in range(64):
            ref[i, j] = x[i, j] / np.sqrt(ms + eps) * (w[j] + 1.0)
    assert np.allclose(O.rms_norm(x, w, eps), ref, rtol=1e-13)



def test_moe_shared_expert_is_an_expert_every_token_uses_with_weight_one():
    """Adding the shared expert equals routing it to every token as a ninth
    expert of weight 1 (and a zero shared expert changes nothing)."""
    rng = np.random.default_rng(14)

    def layer(k, n, b):
        code, rin, rout, s_in, s_out = make_small_layer(rng, k, n, b)
        return dict(w=O.decode_matrix(code, b), su=O.fold_scales(rin, s_in),
                    sv=O.fold_scales(rout, s_out))
    experts = [(layer(128, 256, 2), layer(128, 256, 3), layer(256, 128, 2)) for _ in range(4)]
    shared = (layer(128, 256, 4), layer(128, 256, 4), layer(256, 128, 4))
    x = rng.normal(size=(3, 128))
    ids = np.array([[0, 2], [1, 3], [3, 0]])
    wts = rng.random((3, 2))
    y = O.moe_forward_shared(x, experts, ids, wts, shared)
    ids9 = np.concatenate([ids, np.full((3, 1), 4)], axis=1)
    w9 = np.concatenate([wts, np.ones((3, 1))], axis=1)
    assert np.allclose(y, O.moe_forward(x, experts + [shared], ids9, w9), rtol=1e-12)
    zero = tuple(dict(d, w=np.zeros_like(d["w"])) for d in shared)
    assert np.allclose(O.moe_forward_shared(x, experts, ids, wts, zero),
                       O.moe_forward(x, experts, ids, wts), rtol=1e-12, atol=1e-12)


def test_silu_closed_form():
    z = np.array([0.0, 1.0, -1.0, 20.0])
    assert np.allclose(O.silu(z), [0.0, 1 / (1 + np.exp(-1)), -1 / (1 + np.e), 20.0], atol=1e-7)


# ---------------------------------------------------------------- E4M3 rounding (EXLR8)

def _e4m3_table():
    """All finite FP8 E4M3 values, decoded from their bit patterns (bias 7,
    three mantissa bits, exponent field 0 = subnormal, S.1111.111 = NaN)."""
    vals = []
    for code in range(256):
        s, e, m = code >> 7, (code >> 3) & 15, code & 7
        if e == 15 and m == 7:
            continue                                     # NaN
        mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
        vals.append(-mag if s else mag)
    return np.array(sorted(set(vals)))


def test_e4m3_table_extremes():
    t = _e4m3_table()
    assert t.max() == 448.0 and t.min() == -448.0        # 1.75 * 2^8
    assert np.min(t[t > 0]) == 2.0 ** -9                 # smallest subnormal


def test_e4m3_round_matches_torch_float8_on_every_fp16_in_range():
    v = np.arange(65536, dtype=np.uint16).view(np.float16).astype(np.float64)
    v = v[np.isfinite(v) & (np.abs(v) <= 448)]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(O.e4m3_round(v), ref)


def test_e4m3_round_fixes_every_e4m3_value_and_breaks_ties_to_even():
    t = _e4m3_table()
    assert np.array_equal(O.e4m3_round(t), t)
    pos = t[t >= 0]
    mids = (pos[:-1] + pos[1:]) / 2
    got = O.e4m3_round(mids)
    # the tie goes to the neighbour whose mantissa field is even
    for lo_v, hi_v, g in zip(pos[:-1], pos[1:], got):
        def mant(v):
            if v < 2.0 ** -6:
                return int(round(v / 2.0 ** -9))
            return int(round((v / 2.0 ** np.floor(np.log2(v)) - 1) * 8))
        want = lo_v if mant(lo_v) % 2 == 0 else hi_v
        assert g == want, (lo_v, hi_v, g)


def test_e4m3_round_saturates():
    got = O.e4m3_round(np.array([449.0, 464.0, 1e4, -500.0, 65504.0]))
    assert np.array_equal(got, [448.0, 448.0, 448.0, -448.0, 448.0])


def test_e4m3_codebook_rounds_the_fp16_value_and_never_saturates():
    st = np.arange(65536, dtype=np.uint32)
    w = O.codebook_value(st).astype(np.float64)
    w8 = O.codebook_value_e4m3(st).astype(np.float64)
    table = _e4m3_table()
    assert np.all(np.isin(w8, table))
    assert np.abs(w).max() < 4.0                         # far below 448
    # every value is the nearest table entry to the fp16 value
    idx = np.searchsorted(table, w)
    lo = table[np.clip(idx - 1, 0, table.size - 1)]
    hi = table[np.clip(idx, 0, table.size - 1)]
    assert np.all(np.minimum(np.abs(w - lo), np.abs(w - hi)) == np.abs(w - w8))


def test_decode_e4m3_is_rounding_of_decode_fp16():
    rng = np.random.default_rng(77)
    code = rng.integers(-32768, 32768, size=(3, 4, 48), dtype=np.int16)
    w = O.decode_matrix(code, 3).astype(np.float64)
    w8 = O.decode_matrix(code, 3, rounding="e4m3").astype(np.float64)
    ref = torch.from_numpy(w).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(w8, ref)


# ---------------------------------------------------------------- FP8 prefill activations (EXLR8)

def _e4m3_scaled_rows(rng, m, k, exps):
    """Rows whose values are E4M3 values times 2^e (e per row), each row holding
    +-448 * 2^e once: exactly representable in fp16 and in the quantiser."""
    t = _e4m3_table()
    rows = []
    for e in exps:
        r = rng.choice(t, size=k)
        r[rng.integers(k)] = rng.choice([-448.0, 448.0])
        rows.append(r * 2.0 ** e)
    x = np.array(rows).astype(np.float16)
    assert np.array_equal(x.astype(np.float64), np.array(rows))
    return x, np.array(rows)


def test_quantize_rows_is_exact_on_scaled_e4m3_rows():
    """amax = 448 * 2^e makes the scale a power of two: q are the E4M3 values
    and d = 2^e, exactly (a wrong axis, constant or inverse breaks this)."""
    rng = np.random.default_rng(901)
    exps = [-8, -5, -2, 0, -3]
    xh, exact = _e4m3_scaled_rows(rng, len(exps), 384, exps)
    q, d = O.quantize_rows_e4m3(xh)
    assert d.dtype == np.float32
    assert np.array_equal(d.astype(np.float64), 2.0 ** np.array(exps, dtype=np.float64))
    assert np.array_equal(q * d.astype(np.float64)[:, None], exact)


def test_quantize_rows_matches_torch_float8_cast():
    """The rounding step against torch's float8_e4m3fn cast of the same fp32 products."""
    rng = np.random.default_rng(902)
    xh = (rng.standard_normal((7, 640)) * rng.choice([1e-3, 0.1, 3.0, 50.0], size=(7, 1)))
    xh = xh.astype(np.float16)
    q, d = O.quantize_rows_e4m3(xh)
    x32 = torch.from_numpy(xh.astype(np.float32))
    amax = x32.abs().amax(dim=1)
    inv = torch.tensor(448.0, dtype=torch.float32) / amax
    ref = (x32 * inv[:, None]).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(q, ref)
    assert np.array_equal(d, (amax / torch.tensor(448.0, dtype=torch.float32)).numpy())


def test_quantize_rows_range_and_error_bound():
    """|q| <= 448 with 448 reached at each row's largest element; the
    dequantised error is within E4M3's half spacing: 2^-4 relative above 2^-6,
    2^-10 absolute below (times d), plus fp32 rounding of the scale."""
    rng = np.random.default_rng(903)
    xh = (rng.standard_normal((9, 1024)) * np.exp(rng.uniform(-6, 4, size=(9, 1)))).astype(np.float16)
    q, d = O.quantize_rows_e4m3(xh)
    x = xh.astype(np.float64)
    assert np.all(np.abs(q) <= 448.0)
    rows = np.arange(9)
    assert np.all(np.abs(q[rows, np.argmax(np.abs(x), axis=1)]) == 448.0)
    assert np.all(np.isin(q, _e4m3_table()))
    dd = d.astype(np.float64)[:, None]
    err = np.abs(q * dd - x)
    bound = (2.0 ** -4 * np.abs(x) + 2.0 ** -10 * dd) * (1 + 2.0 ** -20)
    assert np.all(err <= bound)
    # the bound is not loose everywhere: rounding really happens
    assert np.max(err / np.maximum(bound, 1e-30)) > 0.5


def test_quantize_rows_zero_row_and_single_element():
    xh = np.zeros((3, 128), dtype=np.float16)
    xh[1, 5] = -0.75
    q, d = O.quantize_rows_e4m3(xh)
    assert d[0] == 0 and d[2] == 0 and np.all(q[0] == 0) and np.all(q[2] == 0)
    assert q[1, 5] == -448.0 and np.count_nonzero(q[1]) == 1
    assert d[1] == np.float32(0.75) / np.float32(448)


def test_linear_fp8_equals_exact_layer_when_activations_are_e4m3():
    """With rotated activations that the quantiser represents exactly, the FP8
    layer is the plain layer definition (had(had(x su) W) sv) on E4M3 weights."""
    rng = np.random.default_rng(904)
    k, n = 256, 384
    code = rng.integers(-32768, 32768, size=(k // 16, n // 16, 48), dtype=np.int16)
    w8 = O.decode_matrix(code, 3, rounding="e4m3").astype(np.float64)
    su = rng.uniform(0.5, 1.5, size=k)
    sv = rng.uniform(0.5, 1.5, size=n)
    _, xh_target = _e4m3_scaled_rows(rng, 4, k, [-6, -3, -1, -4])
    x = O.had_blockwise(xh_target) / su               # had is its own inverse
    assert np.array_equal(O.rotate_in_fp16(x, su).astype(np.float64), xh_target)
    got = O.linear_forward_fp8(x, w8, su, sv)
    ref = O.linear_forward(x, w8, su, sv)
    assert np.max(np.abs(got - ref)) <= 1e-10 * np.max(np.abs(ref))


def test_linear_fp8_differs_from_fp16_layer_by_the_activation_rounding():
    """On Gaussian activations the FP8 layer stays within E4M3's relative
    rounding (RMS at most 2^-4/sqrt(3)) of the fp16 layer, and is not equal to it."""
    rng = np.random.default_rng(905)
    k, n = 512, 256
    code = rng.integers(-32768, 32768, size=(k // 16, n // 16, 32), dtype=np.int16)
    w8 = O.decode_matrix(code, 2, rounding="e4m3").astype(np.float64)
    su = rng.uniform(0.9, 1.1, size=k)
    sv = np.ones(n)
    x = rng.standard_normal((6, k))
    got = O.linear_forward_fp8(x, w8, su, sv)
    xh = O.rotate_in_fp16(x, su).astype(np.float64)
    ref = O.linear_forward(O.had_blockwise(xh), w8, np.ones(k), sv)   # had(had(xh)) = xh
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert 1e-3 < rel < 2.0 ** -4 / np.sqrt(3)


def test_linear_fp8_brute_force_loops():
    """Per-element loops on a 128x128 E4M3 layer, two tokens: the Hadamard from
    its sign formula, fp16 and fp32 roundings through struct (IEEE half and
    single), the E4M3 code by searching the whole table (ties to the even
    mantissa), then explicit sums."""
    import struct

    def f16(v):
        return struct.unpack("e", struct.pack("e", v))[0]

    def f32(v):
        return struct.unpack("f", struct.pack("f", v))[0]

    table = _e4m3_table()

    def even_mantissa(v):
        a = abs(v)
        if a < 2.0 ** -6:
            return int(round(a / 2.0 ** -9)) % 2 == 0
        return int(round((a / 2.0 ** np.floor(np.log2(a)) - 1) * 8)) % 2 == 0

    def e4m3(v):
        dist = np.abs(table - v)
        best = table[dist == dist.min()]
        if best.size == 1:
            return float(best[0])
        return float([t for t in best if even_mantissa(t)][0])

    rng = np.random.default_rng(907)
    k = n = 128
    code = rng.integers(-32768, 32768, size=(k // 16, n // 16, 48), dtype=np.int16)
    w8 = O.decode_matrix(code, 3, rounding="e4m3").astype(np.float64)
    su = rng.uniform(0.5, 1.5, size=k)
    sv = rng.uniform(0.5, 1.5, size=n)
    x = rng.normal(size=(2, k)) * np.array([[0.01], [30.0]])
    H = [[(-1.0) ** bin(a & b).count("1") / np.sqrt(128) for b in range(128)] for a in range(128)]
    ref = []
    for row in x:
        xh = [f16(sum(row[a] * su[a] * H[a][j] for a in range(k))) for j in range(k)]
        amax = max(abs(v) for v in xh)
        inv, d = f32(448.0 / amax), f32(amax / 448.0)
        q = [e4m3(f32(v * inv)) for v in xh]
        yp = [d * sum(q[j] * w8[j, c] for j in range(k)) for c in range(n)]
        ref.append([sum(yp[b] * H[b][c] for b in range(n)) * sv[c] for c in range(n)])
    got = O.linear_forward_fp8(x, w8, su, sv)
    assert np.allclose(got, np.array(ref), rtol=1e-10, atol=1e-12 * np.max(np.abs(ref)))


def test_linear_fp8_columns_match_full_layer():
    rng = np.random.default_rng(906)
    k, n = 256, 512
    code = rng.integers(-32768, 32768, size=(k // 16, n // 16, 64), dtype=np.int16)
    w8 = O.decode_matrix(code, 4, rounding="e4m3").astype(np.float64)
    su = rng.uniform(0.5, 1.5, size=k)
    sv = rng.uniform(0.5, 1.5, size=n)
    x = rng.standard_normal((5, k))
    full = O.linear_forward_fp8(x, w8, su, sv)
    cols, part = O.linear_forward_fp8_columns(x, code, 4, su, sv, [1, 3])
    assert np.array_equal(cols, np.r_[128:256, 384:512])
    assert np.allclose(part, full[:, cols], rtol=0, atol=1e-12 * np.max(np.abs(full)))


# ---------------------------------------------------------------- Viterbi encoder (EXLR8, MLX)

def _decoded(code, bits, rounding="fp16"):
    return O.codebook(O.tile_states(code, bits), rounding).astype(np.float64)


@pytest.mark.parametrize("bits,rounding", [(2, "fp16"), (3, "fp16"), (4, "fp16"), (3, "e4m3")])
def test_encoder_recovers_every_decodable_tile_exactly(bits, rounding):
    """A tile that some code decodes to is encoded with zero error."""
    rng = np.random.default_rng(900 + bits)
    for _ in range(2):
        code = random_tiles(rng, 1, bits)[0]
        vals = _decoded(code, bits, rounding).astype(np.float32)
        enc, states, cost = O.viterbi_encode_tile(vals, bits, rounding)
        assert cost == 0.0
        assert np.array_equal(_decoded(enc, bits, rounding), vals.astype(np.float64))


@pytest.mark.parametrize("bits", [2, 3])
def test_encoder_path_is_circular_and_its_cost_is_the_decoded_error(bits):
    rng = np.random.default_rng(910 + bits)
    vals = (rng.standard_normal(256) * 1.244).astype(np.float32)
    enc, states, cost = O.viterbi_encode_tile(vals, bits)
    # the packed stream reproduces every state, the wrap-around one included
    assert np.array_equal(O.tile_states(enc, bits), states)
    err = np.sum((_decoded(enc, bits) - vals.astype(np.float64)) ** 2)
    assert abs(cost - err) <= 1e-5 * err


@pytest.mark.parametrize("bits", [2, 3])
def test_encoder_path_is_locally_optimal(bits):
    """No change of one symbol's new bits (with the windows it enters) lowers the error."""
    rng = np.random.default_rng(920 + bits)
    vals = (rng.standard_normal(256) * 1.244).astype(np.float64)
    enc, states, _ = O.viterbi_encode_tile(vals.astype(np.float32), bits)
    stream = O.tile_stream_bits(enc).astype(np.uint8)
    base = np.sum((_decoded(enc, bits) - vals) ** 2)
    for i in range(0, 256, 5):
        for alt in range(1, 1 << bits):
            s2 = stream.copy()
            for t in range(bits):
                s2[bits * i + t] ^= (alt >> (bits - 1 - t)) & 1
            code2 = O.pack_stream_bits(s2)
            assert np.sum((_decoded(code2, bits) - vals) ** 2) >= base - 1e-9


@pytest.mark.parametrize("bits", [2, 3])
def test_encoder_sits_near_the_shannon_bound(bits):
    """Gaussian weights coded at R bits each: no code gets the relative
    Frobenius error below 2^-R, and trellis coding comes close ([MLX] puts it a
    few percent above the bound on the model's Hadamard-rotated weights; on 8 random Gaussian tiles this
    encoder lands 9-10 % above the bound at 2 and 3 bits)."""
    rng = np.random.default_rng(930 + bits)
    num, den = 0.0, 0.0
    for _ in range(8):
        vals = (rng.standard_normal(256) * 1.244).astype(np.float32)
        enc, _, _ = O.viterbi_encode_tile(vals, bits)
        num += np.sum((_decoded(enc, bits) - vals.astype(np.float64)) ** 2)
        den += np.sum(vals.astype(np.float64) ** 2)
    rel = np.sqrt(num / den)
    assert 2.0 ** -bits <= rel <= 1.2 * 2.0 ** -bits


def test_encode_matrix_places_tiles_by_the_permutation():
    rng = np.random.default_rng(940)
    code = rng.integers(-32768, 32768, size=(2, 3, 32), dtype=np.int16)
    w = O.decode_matrix(code, 2)
    back = O.encode_matrix(w, 2)
    assert np.array_equal(O.decode_matrix(back, 2), w)
