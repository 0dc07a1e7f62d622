"""Plain CPU oracle for EXL3-style trellis-coded linear layers.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this module:
only the tests, the package smoke check and the benchmark's CPU-baseline leg use
it.  It shares no code with the CUDA library and is deliberately slow and literal:
every step is written the way the source pages define it, in numpy, with fp64
arithmetic except where fp16 rounding is itself part of the definition.

Sources (web pages, cited by title and section):
  [FMT]   "The escha W2 format, recovered and verified" -- sections "Tensor
          mapping", "Reconstruction", "Codebook: cb=1 (MCG), verified",
          "Bit layout: the part that is easy to get wrong", "How each claim
          was verified".
  [MLX]   "Escha-W2 runs on Metal" -- the tensor table, the activation-side
          reconstruction, the three-instruction codebook, the tile packing
          paragraph with the closed-form permutation inverse.
  [EXLR8] the EXLR8 format page -- the shared per-layer rotation ("The sharing
          trick"), the 16x16 tile packing, expert shapes, and the E4M3 rounding
          of every codebook value (round-to-nearest-even, saturating).

Readings taken where the pages are silent or ambiguous (each also listed in the
design notes):
  * Bit stream.  A tile's 16*bits int16 words are paired little-endian into
    8*bits uint32 words; the stream is those words in order, each read from its
    most significant bit down.  State s is the 16 stream bits ending at bit
    bits*(s+1)-1, circularly (tail-biting).  For bits=2 this is exactly the
    decoder printed in [FMT] "Bit layout"; for bits=3 and 4 the pages give no
    decoder, and a constant window offset cannot be seen by the overlap
    invariant, so the bits=3/4 window origin is PARITY UNPINNED.
  * Codebook sum.  "fp16_lo + fp16_hi" is one IEEE fp16 addition, i.e. the
    exact sum rounded once to fp16, round-to-nearest-even.
  * Permutation.  [MLX] prints the inverse map (tile position -> lane pair t
    and half e); the symbol index is s = 2*t + e.  The forward map used for
    placement ("tile[perm] = values", [FMT]) is the inverse of that.
  * Hadamard.  Natural (Sylvester) order, normalised by 1/sqrt(128), applied to
    each consecutive block of 128 channels.
  * Trellis encoder.  [EXLR8] and [MLX] say the encoder picks, per tile, the
    bitstream whose decoded tile has the least squared error, by Viterbi
    search over the 16-bit-state trellis; they do not say how the circular
    (tail-biting) constraint is met.  Reading taken: two Viterbi passes.  Pass
    1 runs with every start state allowed; pass 2 fixes the 16-K bits that the
    last window shares with the first (from pass 1's best end state) and
    allows only start and end states that agree with them, which makes the
    path circular.  The search decides integer codes, so it runs in fp32 with
    each step's error (v - c)^2 and sum rounded separately, ties to the lowest
    index: the precision and order the CUDA encoder uses.
  * E4M3 variant.  [EXLR8] rounds each codebook output to FP8 E4M3; the
    value rounded is the codebook's fp16 value (after its one fp16
    addition), to the nearest E4M3 value, ties to even mantissa, magnitudes
    above 448 clamped to 448 (saturating; E4M3 has no infinities).
  * FP8 prefill.  [EXLR8] says E4M3-exact weights let prefill multiply on FP8
    tensor cores, but not how the activations become FP8.  Reading taken:
    each token's rotated fp16 activations xh are scaled by their largest
    magnitude onto E4M3's range: amax = max|xh|, inv = fl32(448 / amax),
    q = E4M3(fl32(xh * inv)), d = fl32(amax / 448), and the layer computes
    y = had(d * (q @ W_inner)) * sv.  q is an integer decision, so it is taken
    in fp32 with IEEE rounding, the precision of the CUDA quantiser; a zero
    row gives q = 0 and d = 0.
  * Halves.  [EXLR8] stores each expert matrix as 16 "halves" of 128
    intermediate channels (output channels of gate and up, input channels of
    down) with a width per half for gate/up and per expert for down, but does
    not print a half's code layout.  Reading taken: a half is a code tensor of
    its own in the [FMT] "Tensor mapping" layout, i.e. the whole matrix's tile
    columns 8h..8h+7 (gate, up) or tile rows 8h..8h+7 (down).

The fp16 <-> float conversions use numpy's IEEE half type.
"""

import numpy as np

TILE = 16                       # [FMT] "Tensor mapping": 16x16 tiles
SYMBOLS_PER_TILE = TILE * TILE  # 256 trellis states per tile
HAD_BLOCK = 128                 # [FMT] "Reconstruction": Hadamard of size 128

MCG_MULT = 0xCBAC1FED           # [FMT] "Codebook: cb=1 (MCG)"
MCG_MASK = 0x8FFF8FFF
MCG_XOR = 0x3B603B60

SUPPORTED_BITS = (2, 3, 4)


# ----------------------------------------------------------------------------
# Bit stream and trellis states  ([FMT] "Bit layout", [MLX] tile packing)
# ----------------------------------------------------------------------------

def words_per_tile(bits):
    """int16 words per tile: 256 symbols x bits / 16 ([FMT] "Tensor mapping")."""
    return SYMBOLS_PER_TILE * bits // 16


def tile_u32_words(tile_code):
    """Pair the tile's int16 words little-endian into uint32 words.

    tile_code: int16 [..., 16*bits].  Returns uint64 [..., 8*bits] (values < 2^32).
    """
    u16 = np.asarray(tile_code).view(np.uint16).astype(np.uint64)
    return u16[..., 0::2] | (u16[..., 1::2] << np.uint64(16))


def tile_stream_bits(tile_code):
    """The tile's bit stream, one uint8 per bit, words in order, MSB first."""
    w = tile_u32_words(tile_code)
    shifts = np.arange(31, -1, -1, dtype=np.uint64)           # MSB first
    bits = (w[..., :, None] >> shifts) & np.uint64(1)
    return bits.reshape(*w.shape[:-1], -1).astype(np.uint8)


def window_positions(bits):
    """Stream positions of each state's 16-bit window, MSB first: [256, 16].

    State s ends at stream bit bits*(s+1)-1; the stream is circular.
    """
    n = SYMBOLS_PER_TILE * bits
    s = np.arange(SYMBOLS_PER_TILE)[:, None]
    i = np.arange(16)[None, :]
    return (bits * (s + 1) - 16 + i) % n


def tile_states(tile_code, bits):
    """All 256 16-bit trellis states of each tile (stream model): uint32 [..., 256]."""
    assert bits in SUPPORTED_BITS
    stream = tile_stream_bits(tile_code)
    assert stream.shape[-1] == SYMBOLS_PER_TILE * bits
    window = stream[..., window_positions(bits)]              # [..., 256, 16]
    place = (1 << np.arange(15, -1, -1)).astype(np.uint32)      # MSB first
    return (window.astype(np.uint32) * place).sum(axis=-1).astype(np.uint32)


def tile_states_k2_printed(tile_code):
    """bits=2 states by the decoder printed in [FMT] "Bit layout".

    Lane L handles symbols t = 8L .. 8L+7.  It forms a 64-bit value from the
    word pair (i0, i1), shifts it right by 16 when bit 3 of t is clear, and
    takes symbol t+j as the 16 bits that sit 14-2j bits above the bottom.  Independent of the stream
    model above; the two must agree.
    """
    u32 = tile_u32_words(tile_code)
    assert u32.shape[-1] == 16
    out = np.zeros(u32.shape[:-1] + (SYMBOLS_PER_TILE,), dtype=np.uint32)
    for lane in range(32):
        t = 8 * lane
        i1 = t >> 4
        i0 = (i1 + 15) & 15
        b = (u32[..., i0] << np.uint64(32)) | u32[..., i1]
        b = b >> np.uint64(((~t) & 8) << 1)
        for j in range(8):
            out[..., t + j] = ((b >> np.uint64(14 - 2 * j)) & np.uint64(0xFFFF)).astype(np.uint32)
    return out


def pack_stream_bits(stream_bits):
    """Test helper: pack a 256*bits-bit stream (uint8 per bit) into int16 words.

    The inverse of tile_stream_bits: words MSB first, uint32 split into two
    little-endian int16 words.  Used to build tiles from hand-chosen streams.
    """
    stream_bits = np.asarray(stream_bits, dtype=np.uint64)
    nbits = stream_bits.shape[-1]
    assert nbits % 32 == 0
    w = stream_bits.reshape(*stream_bits.shape[:-1], nbits // 32, 32)
    place = np.uint64(1) << np.arange(31, -1, -1, dtype=np.uint64)
    u32 = (w * place).sum(axis=-1).astype(np.uint64)
    lo = (u32 & np.uint64(0xFFFF)).astype(np.uint16)
    hi = (u32 >> np.uint64(16)).astype(np.uint16)
    u16 = np.stack([lo, hi], axis=-1).reshape(*u32.shape[:-1], -1)
    return u16.view(np.int16)


# ----------------------------------------------------------------------------
# Codebook cb=1 ("3INST")  ([FMT] "Codebook: cb=1 (MCG), verified"; [MLX])
# ----------------------------------------------------------------------------

def mcg_word(states):
    """v = state * 0xCBAC1FED (mod 2^32); v = (v & 0x8FFF8FFF) ^ 0x3B603B60."""
    v = (np.asarray(states, dtype=np.uint64) * np.uint64(MCG_MULT)) & np.uint64(0xFFFFFFFF)
    v = (v & np.uint64(MCG_MASK)) ^ np.uint64(MCG_XOR)
    return v


def codebook_halves(states):
    """The two fp16 numbers of the codebook word: (low half, high half), as float16."""
    v = mcg_word(states)
    lo = (v & np.uint64(0xFFFF)).astype(np.uint16).view(np.float16)
    hi = (v >> np.uint64(16)).astype(np.uint16).view(np.float16)
    return lo, hi


def codebook_value(states):
    """fp16_lo + fp16_hi as one fp16 addition: exact sum, rounded once (RNE)."""
    lo, hi = codebook_halves(states)
    exact = lo.astype(np.float64) + hi.astype(np.float64)
    return exact.astype(np.float16)


# ----------------------------------------------------------------------------
# E4M3 rounding of codebook values  ([EXLR8]: each codebook output is rounded
# to FP8 E4M3, nearest even, saturating)
# ----------------------------------------------------------------------------

E4M3_MAX = 448.0        # largest finite FP8 E4M3 value: 1.75 * 2^8
E4M3_MIN_EXP = -6       # exponent of the smallest normal value (bias 7)
E4M3_MANT_BITS = 3


def e4m3_round(x):
    """Nearest FP8 E4M3 value (ties to even mantissa), saturating at +-448.

    The spacing of E4M3 values in the binade [2^e, 2^(e+1)) is 2^(e-3); below
    2^-6 (subnormals) it stays 2^-9.  Rounding |x| / spacing to the nearest
    integer, halves to even, is round-to-nearest-even on the mantissa.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, E4M3_MIN_EXP)
    q = np.exp2(e - E4M3_MANT_BITS)
    r = np.minimum(np.round(a / q) * q, E4M3_MAX)
    return np.copysign(r, x)


def codebook_value_e4m3(states):
    """The codebook's fp16 value rounded to E4M3 (returned as float16, exactly)."""
    return e4m3_round(codebook_value(states).astype(np.float64)).astype(np.float16)


def codebook(states, rounding="fp16"):
    """Weight value of each state: the fp16 codebook value, or its E4M3 rounding."""
    if rounding == "fp16":
        return codebook_value(states)
    if rounding == "e4m3":
        return codebook_value_e4m3(states)
    raise ValueError(rounding)


# ----------------------------------------------------------------------------
# Trellis encoder: Viterbi search  ([EXLR8]: the code of a tile is the trellis
# path of least squared error; [MLX] tail-biting windows)
# ----------------------------------------------------------------------------

def _viterbi_pass(values, bits, cvals, start_ok=None, end_ok=None):
    """One Viterbi pass over the 256 symbols of a tile.

    State s of symbol i is its 16-bit window; the next state is
    ((s << bits) | new bits) & 0xFFFF, so the predecessors of s are
    (s >> bits) | (t << (16 - bits)) for t < 2^bits.  Costs are fp32: each
    step adds (v_i - c(s))^2, the difference, square and sum each rounded.
    Returns (states [256] uint32, total cost).
    """
    nu = 1 << (16 - bits)                                    # predecessor groups
    inf = np.float32(np.inf)
    v = np.asarray(values, dtype=np.float32)
    d = v[0] - cvals
    cost = (d * d).astype(np.float32)
    if start_ok is not None:
        cost = np.where(start_ok, cost, inf).astype(np.float32)
    back = np.empty((SYMBOLS_PER_TILE, nu), dtype=np.uint8)
    succ_group = (np.arange(1 << 16, dtype=np.int64) >> bits)  # u of each state's predecessors
    for i in range(1, SYMBOLS_PER_TILE):
        grid = cost.reshape(1 << bits, nu)                   # [t][u]: state = u + t * nu
        t_best = np.argmin(grid, axis=0)                     # first (lowest t) on ties
        m = grid[t_best, np.arange(nu)]
        back[i] = t_best
        d = v[i] - cvals
        cost = ((d * d).astype(np.float32) + m[succ_group]).astype(np.float32)
    if end_ok is not None:
        cost = np.where(end_ok, cost, inf).astype(np.float32)
    s = int(np.argmin(cost))                                 # lowest state on ties
    total = float(cost[s])
    states = np.empty(SYMBOLS_PER_TILE, dtype=np.uint32)
    states[-1] = s
    for i in range(SYMBOLS_PER_TILE - 1, 0, -1):
        u = s >> bits
        s = u | (int(back[i][u]) << (16 - bits))
        states[i - 1] = s
    return states, total


def viterbi_encode_tile(values, bits, rounding="fp16"):
    """Encode one tile's 256 symbol values (symbol order): tail-biting path.

    Returns (tile code int16 [16*bits], states uint32 [256], squared error).
    """
    cvals = codebook(np.arange(1 << 16, dtype=np.uint32), rounding).astype(np.float32)
    st1, _ = _viterbi_pass(values, bits, cvals)
    mask = (1 << (16 - bits)) - 1
    o = int(st1[-1]) & mask                                  # bits shared by last and first window
    s = np.arange(1 << 16, dtype=np.int64)
    states, total = _viterbi_pass(values, bits, cvals, start_ok=(s >> bits) == o,
                                  end_ok=(s & mask) == o)
    # stream bits K*i .. K*i+K-1 are the low `bits` bits of state i, MSB first
    shift = np.arange(bits - 1, -1, -1, dtype=np.uint32)
    stream = ((states[:, None] >> shift[None, :]) & 1).reshape(-1).astype(np.uint8)
    return pack_stream_bits(stream), states, total


def encode_matrix(w, bits, rounding="fp16"):
    """Code tensor int16 [in/16, out/16, 16*bits] of W_inner [in, out] (tile by tile)."""
    w = np.asarray(w, dtype=np.float32)
    k, n = w.shape
    perm = perm_forward()
    code = np.empty((k // TILE, n // TILE, words_per_tile(bits)), dtype=np.int16)
    for i in range(k // TILE):
        for j in range(n // TILE):
            tile = w[TILE * i:TILE * (i + 1), TILE * j:TILE * (j + 1)].reshape(-1)
            code[i, j], _, _ = viterbi_encode_tile(tile[perm], bits, rounding)
    return code


# ----------------------------------------------------------------------------
# Tensor-core permutation  ([MLX] closed-form inverse; [FMT] "tile[perm] = values")
# ----------------------------------------------------------------------------

def perm_symbol_of(r, c):
    """Closed-form inverse: tile row r (input channel), column c (output) -> symbol s.

    t = 4*(4*(c&7) + q) + 2*((c>>3)&1) + rh with q = (r>>1)&3, rh = r>>3,
    e = r&1, and s = 2*t + e.
    """
    q = (r >> 1) & 3
    rh = r >> 3
    e = r & 1
    t = 4 * (4 * (c & 7) + q) + 2 * ((c >> 3) & 1) + rh
    return 2 * t + e


def perm_forward():
    """perm[s] = flat tile index r*16 + c where symbol s lands (inverse of the above)."""
    perm = np.full(SYMBOLS_PER_TILE, -1, dtype=np.int64)
    for r in range(TILE):
        for c in range(TILE):
            s = perm_symbol_of(r, c)
            perm[s] = r * TILE + c
    return perm


# ----------------------------------------------------------------------------
# Decode: code tensor -> W_inner  ([FMT] "Tensor mapping", "Bit layout")
# ----------------------------------------------------------------------------

def decode_tiles(tile_codes, bits, rounding="fp16"):
    """Decode tiles: int16 [..., 16*bits] -> float16 [..., 16, 16] (row = input channel)."""
    values = codebook(tile_states(tile_codes, bits), rounding)  # [..., 256]
    perm = perm_forward()
    flat = np.empty(values.shape, dtype=np.float16)
    flat[..., perm] = values                                    # tile[perm] = values
    return flat.reshape(*values.shape[:-1], TILE, TILE)


def decode_matrix(code, bits, chunk=4096, rounding="fp16"):
    """W_inner fp16 [in, out] from the code tensor int16 [in/16, out/16, 16*bits].

    code[i, j] holds W_inner[16i:16i+16, 16j:16j+16] (K-tile index major).
    """
    kt, nt, nw = code.shape
    assert nw == words_per_tile(bits)
    flat = code.reshape(kt * nt, nw)
    tiles = np.empty((kt * nt, TILE, TILE), dtype=np.float16)
    for a in range(0, kt * nt, chunk):
        tiles[a:a + chunk] = decode_tiles(flat[a:a + chunk], bits, rounding)
    return tiles.reshape(kt, nt, TILE, TILE).transpose(0, 2, 1, 3).reshape(kt * TILE, nt * TILE)


def decode_columns(code, bits, cols, rounding="fp16"):
    """W_inner[:, cols] (fp16) decoding only the tile columns that hold `cols`."""
    cols = np.asarray(cols)
    kt = code.shape[0]
    out = np.empty((kt * TILE, cols.size), dtype=np.float16)
    for jt in np.unique(cols // TILE):
        tiles = decode_tiles(code[:, jt, :], bits, rounding)    # [kt, 16, 16]
        strip = tiles.reshape(kt * TILE, TILE)
        sel = np.nonzero(cols // TILE == jt)[0]
        out[:, sel] = strip[:, cols[sel] % TILE]
    return out



def decode_column_halves(halves, bits, rounding="fp16"):
    """W_inner [in, 128*H] of a matrix stored by halves along its output side.

    [EXLR8] manifest paragraph: an expert's gate and up matrices are split into
    "halves" of 128 intermediate channels each -- their output channels -- and
    each half is coded at its own width.  halves[h] is the code int16
    [in/16, 8, 16*bits[h]] of output channels 128h .. 128h+127 (a code tensor in
    the [FMT] "Tensor mapping" layout of its own); the matrix is the halves'
    decoded columns side by side.
    """
    return np.concatenate([decode_matrix(c, int(b), rounding=rounding)
                           for c, b in zip(halves, bits)], axis=1)


def decode_row_halves(halves, bits, rounding="fp16"):
    """W_inner [128*H, out] of a matrix stored by halves along its input side.

    [EXLR8] manifest paragraph: down's halves are 128 of its input (intermediate)
    channels, and down has one width per expert (the error feedback of its
    calibrated rounding crosses halves).  halves[h] is the code int16 [8, out/16, 16*bits] of
    input channels 128h .. 128h+127; the matrix is the halves' decoded rows
    stacked in order.
    """
    return np.concatenate([decode_matrix(c, int(bits), rounding=rounding) for c in halves],
                          axis=0)


# ----------------------------------------------------------------------------
# Blockwise Hadamard-128  ([FMT] "Reconstruction"; [EXLR8] rotation)
# ----------------------------------------------------------------------------

def sylvester_hadamard(n):
    """Unnormalised Sylvester Hadamard matrix of order n (power of 2), natural order."""
    h = np.ones((1, 1))
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    assert h.shape[0] == n
    return h


def had128_matrix():
    """H_128 / sqrt(128): symmetric and orthogonal."""
    return sylvester_hadamard(HAD_BLOCK) / np.sqrt(HAD_BLOCK)


def had_blockwise(x):
    """Apply H_128/sqrt(128) to each consecutive 128-block of the last axis (fp64)."""
    x = np.asarray(x, dtype=np.float64)
    n = x.shape[-1]
    assert n % HAD_BLOCK == 0
    xb = x.reshape(*x.shape[:-1], n // HAD_BLOCK, HAD_BLOCK)
    return (xb @ had128_matrix()).reshape(x.shape)


def blockdiag_hadamard(n):
    """Dense block-diagonal matrix diag(H128, ..., H128)/sqrt(128) of order n."""
    h = had128_matrix()
    out = np.zeros((n, n))
    for b in range(0, n, HAD_BLOCK):
        out[b:b + HAD_BLOCK, b:b + HAD_BLOCK] = h
    return out


# ----------------------------------------------------------------------------
# Layers  ([MLX] activation-side reconstruction; [FMT] "Reconstruction")
# ----------------------------------------------------------------------------

def fold_scales(r, s):
    """su = rin * s_in  or  sv = rout * s_out, in fp64 ([MLX])."""
    return np.asarray(r).astype(np.float64) * np.asarray(s).astype(np.float64)


def linear_forward(x, w_inner, su, sv):
    """y = had(had(x * su) @ W_inner) * sv, fp64 throughout.

    x: [M, in] (any float dtype); w_inner: [in, out]; su: [in]; sv: [out].
    """
    x = np.asarray(x).astype(np.float64)
    xh = had_blockwise(x * su)
    y_pre = xh @ np.asarray(w_inner).astype(np.float64)
    return had_blockwise(y_pre) * sv


def linear_forward_columns(x, code, bits, su, sv, blocks, rounding="fp16"):
    """Output columns of the 128-blocks `blocks` only (decodes just those columns)."""
    x = np.asarray(x).astype(np.float64)
    xh = had_blockwise(x * su)
    cols = np.concatenate([np.arange(b * HAD_BLOCK, (b + 1) * HAD_BLOCK) for b in blocks])
    w = decode_columns(code, bits, cols, rounding).astype(np.float64)
    y_pre = xh @ w
    y = had_blockwise(y_pre) * sv[cols]
    return cols, y


def reconstruct_weight(w_inner, su, sv):
    """Weight-side route ([FMT] "Reconstruction"): W [in, out] such that y = x @ W.

    W = had_l(W_inner); W *= su[:, None]; W = had_r(W); W *= sv[None, :].
    """
    k, n = w_inner.shape
    w = blockdiag_hadamard(k) @ np.asarray(w_inner).astype(np.float64)
    w = w * np.asarray(su)[:, None]
    w = w @ blockdiag_hadamard(n)
    return w * np.asarray(sv)[None, :]


# ----------------------------------------------------------------------------
# FP8 prefill  ([EXLR8]: decoded weights are exact E4M3 values, so prefill can
# multiply them on FP8 tensor cores; the activation scaling is the reading in
# the header)
# ----------------------------------------------------------------------------

def rotate_in_fp16(x, su):
    """xh = fp16(had128(x * su)): the rotated activations, rounded once to fp16."""
    return had_blockwise(np.asarray(x).astype(np.float64) * su).astype(np.float16)


def quantize_rows_e4m3(xh):
    """Per-token E4M3 quantisation of fp16 activations: (q, d) with xh ~ q * d.

    xh: [M, K] fp16.  Per row: amax = max|xh|, inv = fl32(448 / amax),
    q = E4M3(fl32(xh * inv)) (nearest even, saturating), d = fl32(amax / 448);
    a row of zeros gives q = 0, d = 0.  Returns q [M, K] float64 (each an E4M3
    value, exactly) and d [M] float32.
    """
    xh32 = np.asarray(xh, dtype=np.float16).astype(np.float32)
    amax = np.max(np.abs(xh32), axis=1)
    nz = amax > 0
    inv = np.zeros_like(amax)
    d = np.zeros_like(amax)
    inv[nz] = np.float32(E4M3_MAX) / amax[nz]
    d[nz] = amax[nz] / np.float32(E4M3_MAX)
    prod = xh32 * inv[:, None]            # fp32 products, one rounding each
    q = e4m3_round(prod.astype(np.float64))
    return q, d


def linear_forward_fp8(x, w_inner, su, sv):
    """FP8 prefill layer: y = had(d * (q @ W_inner)) * sv, (q, d) = quantised xh.

    W_inner must hold E4M3 values (the EXLR8 rounding); the contraction of the
    two E4M3 operands and everything after it is fp64.
    """
    q, d = quantize_rows_e4m3(rotate_in_fp16(x, su))
    return linear_forward_fp8_codes(q, d, w_inner, sv)


def linear_forward_fp8_codes(q, d, w_inner, sv):
    """The FP8 layer after quantisation: y = had(d * (q @ W_inner)) * sv, fp64.

    q: [M, K] E4M3 activation values; d: [M] their per-row scales.
    """
    y_pre = (np.asarray(q, dtype=np.float64) @ np.asarray(w_inner).astype(np.float64))
    y_pre = y_pre * np.asarray(d).astype(np.float64)[:, None]
    return had_blockwise(y_pre) * sv


def linear_forward_fp8_columns(x, code, bits, su, sv, blocks):
    """Output columns of the 128-blocks `blocks` of linear_forward_fp8 (E4M3 weights)."""
    q, d = quantize_rows_e4m3(rotate_in_fp16(x, su))
    cols = np.concatenate([np.arange(b * HAD_BLOCK, (b + 1) * HAD_BLOCK) for b in blocks])
    w = decode_columns(code, bits, cols, "e4m3").astype(np.float64)
    y_pre = (q @ w) * d.astype(np.float64)[:, None]
    return cols, had_blockwise(y_pre) * sv[cols]


def rms_norm(x, w_stored, eps, stored_minus_one=True):
    """RMSNorm of each row of x: x / sqrt(mean(x^2) + eps) * w, fp64.

    "Escha-W2 runs on Metal", model-loading paragraph: the checkpoint keeps
    RMSNorm weights minus one (w - 1), so the weight applied is stored + 1 --
    except the gated norms inside the linear-attention block, which are
    stored as they are (stored_minus_one=False).
    """
    x = np.asarray(x).astype(np.float64)
    w = np.asarray(w_stored).astype(np.float64) + (1.0 if stored_minus_one else 0.0)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * w


def silu(z):
    return z / (1.0 + np.exp(-z))


def mlp_forward(x, gate, up, down):
    """down(silu(gate(x)) * up(x)); each layer is a dict(w=W_inner, su=, sv=)."""
    g = linear_forward(x, gate["w"], gate["su"], gate["sv"])
    u = linear_forward(x, up["w"], up["su"], up["sv"])
    return linear_forward(silu(g) * u, down["w"], down["su"], down["sv"])


def moe_forward(x, experts, ids, weights):
    """sum_k w[m,k] * mlp_{ids[m,k]}(x[m]) per token ([EXLR8] routed experts).

    experts[e] = (gate, up, down) layer dicts; gate/up share the hidden-side su
    and down shares the hidden-side sv across experts ("The sharing trick").
    """
    x = np.asarray(x).astype(np.float64)
    m, hidden = x.shape
    y = np.zeros((m, hidden))
    for t in range(m):
        for k in range(ids.shape[1]):
            gate, up, down = experts[int(ids[t, k])]
            y[t] += float(weights[t, k]) * mlp_forward(x[t:t + 1], gate, up, down)[0]
    return y


def moe_forward_shared(x, experts, ids, weights, shared):
    """Routed experts plus the shared expert, which every token uses with
    weight 1 ([EXLR8] "The sharing trick": the hidden-side rotation is shared
    by all routed experts and the shared expert).  shared = (gate, up, down)."""
    return moe_forward(x, experts, ids, weights) + mlp_forward(x, *shared)
