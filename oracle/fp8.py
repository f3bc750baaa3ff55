"""FP8 (e4m3) inputs with block scales for the forward: the quantiser, the
dequantised values and the attention of those values.

TEST INFRASTRUCTURE ONLY (see the package docstring): the library never
imports this module.

Sources:
  * "Flash Attention V3技术解析" (mlqm.cn), section 1.3 ("低精度计算的工程实践"):
    FP8 products need the contracted dimension contiguous in memory, so the
    P V product reads V transposed; quantisation is block-wise.
  * the same page, section 3.2 ("精度控制策略"): every block computes its own
    scale factor from the largest magnitude in the block and is divided by
    it before rounding.
  * "4.3 FlashAttention-2与FlashAttention-3演进", FlashAttention-3 section 2:
    FP8 inputs halve data movement and multiply work; the softmax statistics
    stay in higher precision.

Readings where the pages leave a step open (also listed in the design notes):
  * Format: e4m3 ("fn": no infinities, 0x7F and 0xFF are NaN, largest finite
    value 448), the FP8 form with the longer mantissa. The page's block
    scale divides max|block| by 127 and rounds to an integer, which is the
    int8 recipe; for e4m3 the matching constant is 448 and the rounding is to
    the nearest e4m3 value, ties to even, with values past 448 held at 448.
    scale = max|block| / 448 in fp32 (1 for an all-zero block), and the
    stored code is e4m3(x / scale) with the division in fp32.
  * Blocks: the page's blocks are 64 x 64. A scale that changed along d would
    not factor out of S = Q K^T, so Q and K get one scale per block of 64
    rows spanning every column. P V contracts over keys, so V's scales run
    along d instead: one per channel (column) of each key/value head, over
    all its keys; it multiplies column c of the output.
  * V is stored transposed, [B, Hkv, d, NP] with NP = N rounded up to 128 and
    zero codes past N, the K-contiguous layout the page asks for.
  * P is rounded to e4m3 for the P V product; the row sum l uses the
    unrounded values. The pages fix nothing more, so the tolerance below
    assumes only what any such scheme must satisfy: each probability is taken
    relative to a reference no larger than the row's true running maximum
    (so P' >= P), multiplied by a power of two >= 1, and rounded to the
    nearest e4m3 value without reaching 448. It holds for every choice of
    reference lag and power of two; the constants in it come from the e4m3
    and bf16 formats alone.

What the CUDA path must match: the quantiser bit for bit (an integer
encoding decided in fp32 on both sides), and the attention of the dequantised
inputs within the per-element bound `p_rounding_bound` states, with a mean
error within `p_rounding_expected` (the only approximation is the rounding of
P, plus bf16 output rounding).

Pins (tests/test_oracle_fp8.py): the decoder against the format's table of all
256 codes written out from the definition, the encoder against a brute-force
nearest-value search over that table with ties to the even code, known tie
and saturation cases, and the dequantised attention against the dense oracle.
"""
import numpy as np

from .attention import forward

E4M3_MAX = 448.0
ROW_BLOCK = 64            # rows per Q / K scale block
KEY_PAD = 128             # V^T rows are padded to a multiple of this many keys
# Rounding constants of the formats (round to nearest):
E4M3_REL = 2.0 ** -4      # e4m3 keeps 3 fraction bits: a normal value moves by at most 2^-4 of itself
E4M3_SUB_HALF = 2.0 ** -10  # half the e4m3 subnormal step 2^-9
BF16_REL = 2.0 ** -8      # bf16 keeps 7 fraction bits: at most 2^-8 of the value
# Largest |beta| (see error_bias) of a correct result: twice bf16's relative
# rounding bound. Rounding to nearest is unbiased to first order; the second
# order (probabilities are denser at the low end of each rounding interval)
# leaves about 1e-3 on the workloads here.
BIAS_MAX = 2.0 * BF16_REL


def e4m3_decode(codes):
    """float64 values of e4m3 codes (uint8). Sign bit 7, exponent bits 6..3
    (bias 7), mantissa bits 2..0; exponent 0 is subnormal (m/8 * 2^-6);
    0x7F and 0xFF are NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    val = sign * mag
    return np.where((c & 0x7F) == 0x7F, np.nan, val)


def e4m3_encode(x):
    """uint8 e4m3 codes of float32 values: round to nearest, ties to even,
    magnitudes past 448 held at 448 (finite inputs only)."""
    a64 = np.asarray(x, dtype=np.float32).astype(np.float64)
    if not np.isfinite(a64).all():
        raise ValueError("finite inputs only")
    neg = np.signbit(a64)
    a = np.abs(a64)
    _, ex = np.frexp(a)                        # a = f * 2^ex, f in [0.5, 1): floor(log2 a) = ex - 1
    normal = a >= 2.0 ** -6
    step = np.where(normal, np.ldexp(1.0, np.where(normal, ex - 1 - 3, 0)), 2.0 ** -9)
    val = np.round(a / step) * step            # exact power-of-two scaling; numpy rounds halves to even
    val = np.minimum(val, E4M3_MAX)
    # encode the rounded magnitude (it may have carried into the next binade)
    _, ev = np.frexp(val)
    is_norm = val >= 2.0 ** -6
    E = np.where(is_norm, ev - 1 + 7, 0).astype(np.int64)
    M = np.where(is_norm, (val / np.ldexp(1.0, np.where(is_norm, ev - 1, 0)) - 1.0) * 8.0, val / 2.0 ** -9)
    code = (E << 3) | np.rint(M).astype(np.int64)
    code = np.where(neg, code | 0x80, code)                 # the sign survives, zero included
    return code.astype(np.uint8)


def _scale_of(amax32):
    """fp32 scale = amax / 448 (1 where the block is all zero)."""
    amax32 = np.asarray(amax32, dtype=np.float32)
    s = (amax32 / np.float32(E4M3_MAX)).astype(np.float32)
    return np.where(amax32 > 0, s, np.float32(1.0)).astype(np.float32)


def quantize_rows(x):
    """Q or K [..., N, d] (values exactly representable in fp32, e.g. bf16)
    -> (codes uint8 [..., N, d], scales float32 [..., ceil(N / 64)])."""
    x32 = np.asarray(x, dtype=np.float32)
    *lead, N, d = x32.shape
    nb = (N + ROW_BLOCK - 1) // ROW_BLOCK
    pad = nb * ROW_BLOCK - N
    xp = np.concatenate([x32, np.zeros((*lead, pad, d), np.float32)], axis=-2) if pad else x32
    blocks = xp.reshape(*lead, nb, ROW_BLOCK, d)
    scales = _scale_of(np.abs(blocks).max(axis=(-1, -2)))
    q = (blocks / scales[..., None, None]).astype(np.float32)
    codes = e4m3_encode(q).reshape(*lead, nb * ROW_BLOCK, d)[..., :N, :]
    return np.ascontiguousarray(codes), scales


def quantize_v_transposed(v):
    """V [..., N, d] -> (codes uint8 [..., d, NP], scales float32 [..., d]):
    column c of the head scaled by max_j |V[j, c]| / 448 and stored as row c
    of V^T, zero codes for keys N..NP-1 (NP = N rounded up to 128)."""
    v32 = np.asarray(v, dtype=np.float32)
    *lead, N, d = v32.shape
    NP = (N + KEY_PAD - 1) // KEY_PAD * KEY_PAD
    scales = _scale_of(np.abs(v32).max(axis=-2))             # [..., d]
    q = (v32 / scales[..., None, :]).astype(np.float32)
    codes = np.zeros((*lead, d, NP), np.uint8)
    codes[..., :, :N] = np.swapaxes(e4m3_encode(q), -1, -2)
    return codes, scales


def dequantize_rows(codes, scales):
    """[..., N, d] float64 values of row-block codes."""
    *lead, N, d = codes.shape
    blk = np.repeat(np.asarray(scales, np.float64), ROW_BLOCK, axis=-1)[..., :N]
    return e4m3_decode(codes) * blk[..., :, None]


def dequantize_v_transposed(codes_t, scales, N):
    """[..., N, d] float64 values of transposed V codes (padding dropped)."""
    vt = e4m3_decode(codes_t[..., :, :N]) * np.asarray(scales, np.float64)[..., :, None]
    return np.swapaxes(vt, -1, -2)


def forward_fp8(q_codes, q_scales, k_codes, k_scales, vt_codes, v_scales, causal, scale):
    """Exact (fp64) attention of the dequantised inputs: (O, LSE) with the
    shapes of `attention.forward`."""
    N = q_codes.shape[-2]
    q = dequantize_rows(q_codes, q_scales)
    k = dequantize_rows(k_codes, k_scales)
    v = dequantize_v_transposed(vt_codes, v_scales, k_codes.shape[-2])
    assert q.shape[-2] == N
    return forward(q, k, v, causal, scale)


def _p_terms(q, k, v, causal, scale, rows):
    """Per head: (w = P / l [R, Nk], visible [R, Nk], l [R, 1], V) for the
    query rows `rows` (all when None), P_j = exp(s_j - max s) in true units."""
    B, Hq, N, d = q.shape
    G = Hq // k.shape[1]
    for b in range(B):
        for h in range(Hq):
            r = np.arange(N) if rows is None else np.asarray(rows[b, h])
            kh, vh = k[b, h // G], v[b, h // G]
            s = (q[b, h, r] @ kh.T) * scale
            off = kh.shape[0] - N                      # keys Nk vs queries N: bottom-right causal
            visible = np.ones(s.shape, bool) if not causal else (np.arange(kh.shape[0])[None, :] <= r[:, None] + off)
            s = np.where(visible, s, -np.inf)
            mx = s.max(axis=1, keepdims=True)
            seen = np.isfinite(mx)                     # rows that see no key: O = 0 exactly
            p = np.where(seen, np.exp(s - np.where(seen, mx, 0.0)), 0.0)
            l = np.where(seen, p.sum(axis=1, keepdims=True), 1.0)
            yield b, h, p / l, visible, l, vh


def p_rounding_bound(q, k, v, causal, scale, o_ref, rows=None):
    """Per-element bound on |O_fp8 - O| for dequantised inputs q, k, v
    (float64) and the exact O (o_ref: [B, Hq, N, d], or [B, Hq, R, d] for
    the query rows `rows` [B, Hq, R]).

    Let P_j = exp(s_j - max s), l = sum_j P_j (>= 1) and w_j = P_j / l. The
    kernel rounds P'_j 2^k to e4m3, where P'_j = P_j 2^t >= P_j is relative to
    a reference that trails the true max by t >= 0 and k >= 0; it divides by
    the unrounded sum, which scales by the same 2^t. A normal e4m3 result
    moves by at most 2^-4 of itself; a subnormal one by at most 2^-10 in units
    of P' 2^k, which is at most 2^-10 in units of P. Hence
      |dO_c| <= 2^-4 sum_j w_j |V_jc| + 2^-10 sum_(visible j) |V_jc| / l,
    plus the bf16 rounding of the result (at most 2^-8 of it) and 1e-6."""
    out = np.empty_like(o_ref, dtype=np.float64)
    for b, h, w, visible, l, vh in _p_terms(q, k, v, causal, scale, rows):
        av = np.abs(vh)
        out[b, h] = (E4M3_REL * (w @ av) + E4M3_SUB_HALF * ((visible @ av) / l)
                     + BF16_REL * np.abs(o_ref[b, h]) + 1e-6)
    return out


def p_rounding_expected(q, k, v, causal, scale, o_ref, rows=None):
    """Per-element upper bound on the EXPECTED |O_fp8 - O| (same arguments as
    `p_rounding_bound`), for a mean-error gate.

    Model: each rounding error is uniform over its rounding interval and
    independent of the others. A normal e4m3 value then has a relative error
    of mean square at most (2^-4)^2 / 3, a subnormal one an absolute error (in
    P units) of mean square at most (2^-10)^2 / 3. With the weights above,
      E[dO_c^2] <= (2^-8 / 3) sum_j w_j^2 V_jc^2 + (2^-20 / 3) sum_(visible j) V_jc^2 / l^2,
    and E|dO_c| <= sqrt(E[dO_c^2]) (Jensen). The bf16 rounding of the result
    adds at most a quarter of its step, 2^-9 |O_c|, on average."""
    out = np.empty_like(o_ref, dtype=np.float64)
    for b, h, w, visible, l, vh in _p_terms(q, k, v, causal, scale, rows):
        v2 = vh * vh
        var = (E4M3_REL ** 2 / 3.0) * ((w * w) @ v2) + (E4M3_SUB_HALF ** 2 / 3.0) * ((visible @ v2) / (l * l))
        out[b, h] = np.sqrt(var) + 0.5 * BF16_REL * np.abs(o_ref[b, h])
    return out


def error_bias(err, o_ref):
    """Least-squares coefficient beta of err ~ beta * O: round to nearest is
    unbiased to first order, so a correct result has |beta| near 0, while an
    output scaled by (1 + e) has beta = e."""
    den = float((o_ref * o_ref).sum())
    return float((err * o_ref).sum() / den) if den > 0 else 0.0
