"""Pins for the FP8 part of the oracle (oracle/fp8.py), on the CPU.

The e4m3 decoder is checked against values the format's definition fixes and
against torch's float8_e4m3fn type (an independent library conversion); the
encoder against a brute-force nearest-value search over all finite codes with
ties to the even code, against torch for in-range values, and on hand-made
tie and saturation cases; the quantisers against their defining properties;
the rounding bound against a direct emulation of rounded probabilities."""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8


def test_decode_fixed_values():
    d = fp8.e4m3_decode
    assert d(0x00) == 0.0 and np.signbit(d(0x80))
    assert d(0x01) == 2.0 ** -9 and d(0x07) == 7 * 2.0 ** -9      # subnormals: m/8 * 2^-6
    assert d(0x08) == 2.0 ** -6                                    # smallest normal
    assert d(0x38) == 1.0 and d(0x3C) == 1.5 and d(0x40) == 2.0
    assert d(0x77) == 240.0 and d(0x78) == 256.0 and d(0x7E) == 448.0
    assert np.isnan(d(0x7F)) and np.isnan(d(0xFF)) and d(0xFE) == -448.0


def test_decode_matches_torch_and_is_monotone():
    codes = np.arange(256, dtype=np.uint8)
    ours = fp8.e4m3_decode(codes)
    theirs = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    assert np.array_equal(np.isnan(ours), np.isnan(theirs))
    fin = ~np.isnan(ours)
    assert np.array_equal(ours[fin], theirs[fin])
    pos = ours[:0x7F]
    assert (np.diff(pos) > 0).all()                                  # 0x00..0x7E strictly increasing


def brute_force_encode(x):
    """Nearest finite e4m3 value by exhaustive search; ties to the even code;
    past 448 held at 448; the sign kept (zero included)."""
    codes = np.arange(0x7F, dtype=np.uint8)                         # 0 .. 448
    vals = fp8.e4m3_decode(codes)
    out = np.empty(x.shape, np.uint8)
    for i, xi in enumerate(np.asarray(x, np.float64).ravel()):
        a = min(abs(xi), 448.0)
        dist = np.abs(vals - a)
        best = np.flatnonzero(dist == dist.min())
        c = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        out.ravel()[i] = c | (0x80 if np.signbit(xi) else 0)
    return out


def test_encode_matches_brute_force():
    rng = np.random.default_rng(5)
    x = np.concatenate([
        rng.normal(0, 1, 3000), rng.normal(0, 100, 2000), rng.uniform(-600, 600, 1000),
        rng.uniform(-2.0 ** -5, 2.0 ** -5, 2000),                   # subnormal range
        fp8.e4m3_decode(np.arange(0x7F)) * rng.choice([-1, 1], 0x7F),  # exact codes
        [0.0, -0.0, 1e-30, -1e-30],
    ]).astype(np.float32)
    mids = (fp8.e4m3_decode(np.arange(1, 0x7F)) + fp8.e4m3_decode(np.arange(0, 0x7E))) / 2
    x = np.concatenate([x, mids.astype(np.float32), -mids.astype(np.float32)])   # every tie
    assert np.array_equal(fp8.e4m3_encode(x), brute_force_encode(x))


def test_encode_matches_torch_in_range():
    rng = np.random.default_rng(6)
    x = np.concatenate([rng.normal(0, 30, 20000), rng.uniform(-463, 463, 5000),
                        rng.uniform(-0.05, 0.05, 5000)]).astype(np.float32)
    theirs = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.e4m3_encode(x), theirs)


def test_encode_ties_and_saturation():
    e = fp8.e4m3_encode
    x = np.array([1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -10, 464.0, 465.0, 500.0, 1e6, -1e6, -0.0],
                 np.float32)
    assert list(e(x)) == [0x38, 0x3A, 0x00, 0x02, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x80]
    with pytest.raises(ValueError):
        e(np.array([np.inf], np.float32))


@pytest.mark.parametrize("d", [16, 96, 128])
def test_quantize_rows_properties(d):
    rng = np.random.default_rng(7 + d)
    x = torch.from_numpy(rng.normal(0, 2, (2, 3, 200, d)).astype(np.float32)).to(torch.bfloat16).float().numpy()
    x[0, 0, 64:128] = 0.0                                            # an all-zero block
    codes, scales = fp8.quantize_rows(x)
    assert codes.shape == x.shape and scales.shape == (2, 3, 4)
    assert scales[0, 0, 1] == 1.0 and (codes[0, 0, 64:128] == 0).all()
    # each block's largest magnitude lands on +-448 and its scale is amax / 448 in fp32
    for b, h, blk in [(0, 1, 0), (1, 2, 3), (1, 0, 2)]:
        rows = x[b, h, 64 * blk:64 * blk + 64]
        amax = np.float32(np.abs(rows).max())
        assert scales[b, h, blk] == np.float32(amax / np.float32(448.0))
        i = np.unravel_index(np.abs(rows).argmax(), rows.shape)
        assert codes[b, h, 64 * blk + i[0], i[1]] in (0x7E, 0xFE)
    deq = fp8.dequantize_rows(codes, scales)
    # rounding error at most half a step: 2^-4 relative for normals, 2^-10 * scale below
    blk_scale = np.repeat(scales.astype(np.float64), 64, axis=-1)[..., :200, None]
    err = np.abs(deq - x)
    assert (err <= np.maximum(2.0 ** -4 * np.abs(x), 2.0 ** -10 * blk_scale) * (1 + 1e-6)).all()


@pytest.mark.parametrize("d", [16, 48, 128, 224])
def test_quantize_v_transposed_layout(d):
    rng = np.random.default_rng(8 + d)
    v = rng.normal(0, 1, (1, 2, 150, d)).astype(np.float32)
    codes, scales = fp8.quantize_v_transposed(v)
    assert codes.shape == (1, 2, d, 256) and scales.shape == (1, 2, d)
    assert (codes[..., 150:] == 0).all()
    # column c of V is row c of V^T, quantised with its own scale
    c = min(17, d - 1)
    s = np.float32(np.abs(v[0, 1, :, c]).max() / np.float32(448.0))
    assert scales[0, 1, c] == s
    assert np.array_equal(codes[0, 1, c, :150], fp8.e4m3_encode((v[0, 1, :, c] / s).astype(np.float32)))
    back = fp8.dequantize_v_transposed(codes, scales, 150)
    assert back.shape == v.shape
    assert np.abs(back - v).max() <= 2.0 ** -4 * np.abs(v).max()


def test_forward_fp8_is_dense_oracle_of_dequantised_inputs():
    rng = np.random.default_rng(9)
    q, k, v = (torch.from_numpy(rng.normal(0, 1, (1, 2, 130, 128)).astype(np.float32)).to(torch.bfloat16).float()
               .numpy() for _ in range(3))
    qc, qs = fp8.quantize_rows(q)
    kc, ks = fp8.quantize_rows(k)
    vc, vs = fp8.quantize_v_transposed(v)
    o, lse = fp8.forward_fp8(qc, qs, kc, ks, vc, vs, True, 128 ** -0.5)
    o2, lse2 = oracle.forward(fp8.dequantize_rows(qc, qs), fp8.dequantize_rows(kc, ks),
                              fp8.dequantize_v_transposed(vc, vs, 130), True, 128 ** -0.5)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
    # and close to the unquantised attention (a loose sanity bar, not a pin)
    o3, _ = oracle.forward(q.astype(np.float64), k.astype(np.float64), v.astype(np.float64), True, 128 ** -0.5)
    assert np.abs(o - o3).mean() < 0.05


def _emulate_rounded_p(q, k, v, causal, scale, pow2, max_lag, seed):
    """Attention with P rounded the way any admissible kernel may round it:
    P' = exp(s - m') relative to a reference m' that trails the row's true
    max by a random t in [0, max_lag] (log2 units, a different t per row),
    multiplied by 2^pow2, rounded to e4m3, divided back, and normalised by the
    unrounded sum; then the bf16 rounding of the result."""
    rng = np.random.default_rng(seed)
    N = q.shape[2]
    s = (q[0, 0] @ k[0, 0].T) * scale
    if causal:
        s = np.where(np.arange(k.shape[2])[None, :] <= np.arange(N)[:, None] + (k.shape[2] - N), s, -np.inf)
    lag = rng.uniform(0, max_lag, (N, 1)) * np.log(2.0)
    p_stale = np.exp(s - s.max(axis=1, keepdims=True) + lag)
    assert (p_stale * 2.0 ** pow2).max() < 448
    p_r = fp8.e4m3_decode(fp8.e4m3_encode((p_stale * 2.0 ** pow2).astype(np.float32))) / 2.0 ** pow2
    o = (p_r @ v[0, 0]) / p_stale.sum(axis=1, keepdims=True)
    return torch.from_numpy(o).to(torch.bfloat16).double().numpy()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("pow2,max_lag,q_mult", [(0, 0.0, 1.0), (4, 4.0, 1.0), (8, 0.5, 2.0), (2, 6.0, 4.0)])
def test_p_rounding_bound_covers_rounded_probabilities(causal, pow2, max_lag, q_mult):
    """The per-element bound holds, and the mean error stays within the
    expected-error bound with the bias coefficient near 0, for every
    admissible choice of scaling and reference lag (emulated directly); an
    output scaled by 1.03 breaks the mean or the bias gate."""
    rng = np.random.default_rng(10 + causal + pow2)
    N, d = 400, 128
    q = rng.normal(0, 1, (1, 1, N, d)) * q_mult
    k = rng.normal(0, 1, (1, 1, N, d))
    v = rng.normal(0, 1, (1, 1, N, d))
    scale = d ** -0.5
    o, _ = oracle.forward(q, k, v, causal, scale)
    o_emul = _emulate_rounded_p(q, k, v, causal, scale, pow2, max_lag, seed=pow2)
    err = o_emul - o[0, 0]
    bound = fp8.p_rounding_bound(q, k, v, causal, scale, o)[0, 0]
    expected = fp8.p_rounding_expected(q, k, v, causal, scale, o)[0, 0]
    assert (np.abs(err) <= bound).all()
    assert np.abs(err).max() > 1e-4                   # the rounding is visible, so the check bites
    assert np.abs(err).mean() <= expected.mean()
    assert np.abs(err).mean() >= 0.2 * expected.mean()   # and the expectation is not vacuous
    assert abs(fp8.error_bias(err, o[0, 0])) <= fp8.BIAS_MAX
    bad = o_emul * 1.03 - o[0, 0]
    assert np.abs(bad).mean() > expected.mean() or abs(fp8.error_bias(bad, o[0, 0])) > fp8.BIAS_MAX
    # and the bound of a subset of rows is the same as the full one there
    rows = np.array([[[0, 7, 150, 399]]])
    sub = fp8.p_rounding_bound(q, k, v, causal, scale, o[:, :, rows[0, 0]], rows=rows)
    assert np.allclose(sub[0, 0], bound[rows[0, 0]], rtol=1e-12, atol=0)
    sub_e = fp8.p_rounding_expected(q, k, v, causal, scale, o[:, :, rows[0, 0]], rows=rows)
    assert np.allclose(sub_e[0, 0], expected[rows[0, 0]], rtol=1e-12, atol=0)


def test_p_rounding_bound_breaks_on_a_planted_mistake():
    """Rounding P to 2 fraction bits instead of 3 (one bit lost) exceeds the
    per-element bound somewhere: the bound is tight enough to see it."""
    rng = np.random.default_rng(5)
    N, d = 400, 128
    q, k, v = (rng.normal(0, 1, (1, 1, N, d)) for _ in range(3))
    scale = d ** -0.5
    o, _ = oracle.forward(q, k, v, False, scale)
    s = (q[0, 0] @ k[0, 0].T) * scale
    p = np.exp(s - s.max(axis=1, keepdims=True))
    m, e = np.frexp(p)
    p2 = np.ldexp(np.round(m * 8) / 8, e)               # 3 significant bits: 2 fraction bits
    o_bad = (p2 @ v[0, 0]) / p.sum(axis=1, keepdims=True)
    bound = fp8.p_rounding_bound(q, k, v, False, scale, o)[0, 0]
    expected = fp8.p_rounding_expected(q, k, v, False, scale, o)[0, 0]
    assert (np.abs(o_bad - o[0, 0]) > bound).any() or np.abs(o_bad - o[0, 0]).mean() > expected.mean()
