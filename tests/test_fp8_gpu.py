"""FP8 (e4m3, block-scaled) forward through the C ABI against the oracle.

The quantisers are integer (byte) work decided in fp32 on both sides, so their
codes and scales must match oracle/fp8.py bit for bit. The attention must
match the exact attention of the dequantised inputs within the bounds the
rounding of P to e4m3 allows, derived in oracle/fp8.py from the e4m3 and bf16
formats alone: per element (p_rounding_bound), on average over the compared
elements (p_rounding_expected), and without a component along O itself
(error_bias); and the LSE within the dense path's 1e-3 (it uses unrounded
probabilities)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8 as ofp8
import exact_attention_79_gb300 as pkg
from exact_attention_79_gb300 import configs, inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def quantized(t):
    g = {n: x.to(DEV) for n, x in t.items()}
    return pkg.quantize_fp8(g["q"], g["k"], g["v"])


def oracle_quant(t):
    f = {n: inputs.to_f64(x) for n, x in t.items()}
    qc, qs = ofp8.quantize_rows(f["q"])
    kc, ks = ofp8.quantize_rows(f["k"])
    vc, vs = ofp8.quantize_v_transposed(f["v"])
    return qc, qs, kc, ks, vc, vs


@pytest.mark.parametrize("B,Hq,Hkv,N", [(1, 2, 2, 128), (2, 3, 1, 333), (1, 4, 2, 1000), (1, 1, 1, 64), (1, 1, 1, 1)])
def test_fp8_quantisers_bit_exact(fa, B, Hq, Hkv, N):
    t = inputs.make_inputs(B, Hq, Hkv, N, 128, "bf16", seed=N + Hq)
    t["q"][:, :, : min(N, 64)] = 0                                   # an all-zero block: scale 1, codes 0
    got = [x.cpu().numpy() for x in quantized(t)]
    fa.check_device_status()
    ref = oracle_quant(t)
    for name, a, r in zip(("q8", "q_scale", "k8", "k_scale", "vt8", "v_scale"), got, ref):
        assert a.shape == r.shape, name
        assert np.array_equal(a.view(np.uint32) if a.dtype == np.float32 else a,
                              r.view(np.uint32) if r.dtype == np.float32 else r), name


# The mean and bias gates are statistical: applied when at least this many
# elements are compared, so that one unlucky rounding cannot decide them.
STAT_MIN_ELEMENTS = 16384


def check_errors(err, bound, expected, ro):
    """err = O_gpu - O_oracle on the compared elements; bound, expected from
    oracle.fp8 for the same elements; ro the oracle's O there."""
    a = np.abs(err)
    assert (a <= bound).all(), (float(a.max()), float((a - bound).max()))
    if err.size >= STAT_MIN_ELEMENTS:
        assert a.mean() <= expected.mean(), (float(a.mean()), float(expected.mean()))
        assert abs(ofp8.error_bias(err, ro)) <= ofp8.BIAS_MAX, ofp8.error_bias(err, ro)
    return float(a.max()), float(a.mean()), float(expected.mean())


def check_against_bound(o, lse, q8, qs, k8, ks, vt8, vs, causal, scale):
    deq_q = ofp8.dequantize_rows(q8, qs)
    deq_k = ofp8.dequantize_rows(k8, ks)
    deq_v = ofp8.dequantize_v_transposed(vt8, vs, k8.shape[-2])
    ro, rl = oracle.forward(deq_q, deq_k, deq_v, causal, scale)
    bound = ofp8.p_rounding_bound(deq_q, deq_k, deq_v, causal, scale, ro)
    expected = ofp8.p_rounding_expected(deq_q, deq_k, deq_v, causal, scale, ro)
    res = check_errors(o - ro, bound, expected, ro)
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(lse), fin)
    assert np.abs(lse[fin] - rl[fin]).max() <= configs.TOL_LSE_MAX
    return res


def check_sampled_rows(o, lse, deq, causal, scale, rows):
    """o, lse: the full GPU outputs (numpy); deq: dequantised q, k, v."""
    B, H = rows.shape[:2]
    ro, rl = oracle.forward_rows(*deq, causal, scale, rows)
    bound = ofp8.p_rounding_bound(*deq, causal, scale, ro, rows=rows)
    expected = ofp8.p_rounding_expected(*deq, causal, scale, ro, rows=rows)
    bi, hi = np.arange(B)[:, None, None], np.arange(H)[None, :, None]
    res = check_errors(o[bi, hi, rows] - ro, bound, expected, ro)
    assert np.abs(lse[bi, hi, rows] - rl).max() <= configs.TOL_LSE_MAX
    return res


@pytest.mark.parametrize("B,Hq,Hkv,N", [(1, 2, 2, 128), (2, 4, 2, 333), (1, 2, 1, 1000)])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_within_rounding_bound(fa, B, Hq, Hkv, N, causal):
    t = inputs.make_inputs(B, Hq, Hkv, N, 128, "bf16", seed=7 * N + causal)
    q8, qs, k8, ks, vt8, vs = quantized(t)
    o, lse = pkg.fwd_fp8(q8, qs, k8, ks, vt8, vs, causal=causal)
    fa.check_device_status()
    host = [x.cpu().numpy() for x in (q8, qs, k8, ks, vt8, vs)]
    print(check_against_bound(o.float().cpu().numpy(), lse.cpu().numpy(), *host, causal, 128 ** -0.5))


def test_fp8_forward_rescales_and_sharp_logits(fa):
    """Keys growing along the sequence and Q x 4: the running max rises often
    by more than 2^4 several times, rescaling the accumulator, and the softmax
    is sharp."""
    N = 1300
    t = inputs.make_inputs(1, 2, 2, N, 128, "bf16", seed=77, q_mult=4.0)
    t["k"] = (t["k"].float() * torch.linspace(0.3, 3.0, N).view(1, 1, N, 1)).to(torch.bfloat16)
    q8, qs, k8, ks, vt8, vs = quantized(t)
    host = [x.cpu().numpy() for x in (q8, qs, k8, ks, vt8, vs)]
    for causal in (True, False):
        o, lse = pkg.fwd_fp8(q8, qs, k8, ks, vt8, vs, causal=causal)
        fa.check_device_status()
        check_against_bound(o.float().cpu().numpy(), lse.cpu().numpy(), *host, causal, 128 ** -0.5)


def test_fp8_forward_full_size_sampled_rows(fa):
    """16 heads, N = 8192, causal (the bench's FP8 workload): the oracle
    computes 256 seeded query rows per head of the dequantised attention and
    the bounds for those rows; max, mean and bias gates."""
    w = configs.WORKLOADS["fp8_h16_n8192_d128_causal_fwd"]
    t = inputs.make_workload_inputs(w)
    q8, qs, k8, ks, vt8, vs = quantized(t)
    o, lse = pkg.fwd_fp8(q8, qs, k8, ks, vt8, vs, causal=True)
    fa.check_device_status()
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    host = [x.cpu().numpy() for x in (q8, qs, k8, ks, vt8, vs)]
    deq = (ofp8.dequantize_rows(host[0], host[1]), ofp8.dequantize_rows(host[2], host[3]),
           ofp8.dequantize_v_transposed(host[4], host[5], w.N))
    rows = inputs.sample_rows(w.B, w.Hq, w.N, 256, seed=4)
    print(check_sampled_rows(o, lse, deq, True, w.scale, rows))


@pytest.mark.parametrize("N,causal", [(333, True), (1000, False)])
def test_fp8_head_dim_64(fa, N, causal):
    """d = 64 runs in the d = 128 kernel: Q, K and V^T read zeros past d,
    V's scales exist only for the 64 columns and the store clips."""
    t = inputs.make_inputs(2, 4, 2, N, 64, "bf16", seed=N + 64)
    q8, qs, k8, ks, vt8, vs = quantized(t)
    host = [x.cpu().numpy() for x in (q8, qs, k8, ks, vt8, vs)]
    assert all(np.array_equal(a, r) for a, r in zip(host, oracle_quant(t)))
    o, lse = pkg.fwd_fp8(q8, qs, k8, ks, vt8, vs, causal=causal)
    fa.check_device_status()
    check_against_bound(o.float().cpu().numpy(), lse.cpu().numpy(), *host, causal, 64 ** -0.5)


@pytest.mark.parametrize("d", [24, 40, 136])
def test_fp8_refuses_other_head_dims(fa, d):
    x = torch.zeros(1, 1, 128, d, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(pkg.FAError):
        pkg.quantize_fp8(x, x, x)
    fa.check_device_status()


@pytest.mark.parametrize("N,causal", [(1, True), (1, False), (64, True), (129, False)])
def test_fp8_forward_degenerate_sizes(fa, N, causal):
    """One query, one 64-row scale block, a ragged second key tile."""
    t = inputs.make_inputs(1, 2, 1, N, 128, "bf16", seed=N + 5)
    q8, qs, k8, ks, vt8, vs = quantized(t)
    o, lse = pkg.fwd_fp8(q8, qs, k8, ks, vt8, vs, causal=causal)
    fa.check_device_status()
    host = [x.cpu().numpy() for x in (q8, qs, k8, ks, vt8, vs)]
    check_against_bound(o.float().cpu().numpy(), lse.cpu().numpy(), *host, causal, 128 ** -0.5)


def test_fp8_forward_long_sequence_sampled_rows(fa):
    """N = 65536 (512 key tiles per causal row at the end), 4 heads: the
    eight-slot ring wraps over a hundred times; 64 seeded rows per head."""
    B, H, N, d = 1, 4, 65536, 128
    t = inputs.make_inputs(B, H, H, N, d, "bf16", seed=65536)
    q8, qs, k8, ks, vt8, vs = quantized(t)
    o, lse = pkg.fwd_fp8(q8, qs, k8, ks, vt8, vs, causal=True)
    fa.check_device_status()
    host = [x.cpu().numpy() for x in (q8, qs, k8, ks, vt8, vs)]
    deq = (ofp8.dequantize_rows(host[0], host[1]), ofp8.dequantize_rows(host[2], host[3]),
           ofp8.dequantize_v_transposed(host[4], host[5], N))
    rows = inputs.sample_rows(B, H, N, 64, seed=6)
    print(check_sampled_rows(o.float().cpu().numpy(), lse.cpu().numpy(), deq, True, d ** -0.5, rows))


@pytest.mark.parametrize("Nq,Nk,causal", [(200, 700, True), (500, 130, True), (1, 777, True), (300, 1000, False),
                                          (1000, 1000, True)])
def test_fp8_forward_kv_lengths(fa, Nq, Nk, causal):
    """Queries are the last Nq of Nk positions (fa_fwd_fp8_kv, bottom-right
    causal); with Nq > Nk the first rows see nothing: O = 0, LSE = -inf.
    Equal lengths through the same path agree bit for bit with fa_fwd_fp8."""
    B, Hq, Hkv, d = 1, 4, 2, 128
    t = inputs.make_inputs(B, Hq, Hkv, Nq, d, "bf16", seed=Nq + 3 * Nk, Nk=Nk)
    q8, qs, k8, ks, vt8, vs = quantized(t)
    host = [x.cpu().numpy() for x in (q8, qs, k8, ks, vt8, vs)]
    ref = oracle_quant(t)
    assert all(np.array_equal(a, r) for a, r in zip(host, ref))
    o, lse = pkg.fwd_fp8(q8, qs, k8, ks, vt8, vs, causal=causal)
    fa.check_device_status()
    o_np, lse_np = o.float().cpu().numpy(), lse.cpu().numpy()
    check_against_bound(o_np, lse_np, *host, causal, d ** -0.5)
    if Nq == Nk:
        lib = pkg.load()
        o2 = torch.empty_like(o)
        l2 = torch.empty_like(lse)
        P = pkg._ptr
        assert lib.fa_fwd_fp8_kv(P(q8), P(qs), P(k8), P(ks), P(vt8), P(vs), P(o2), P(l2), B, Hq, Hkv, Nq, Nk, d,
                                 int(causal), d ** -0.5, pkg._stream(q8)) == 0
        fa.check_device_status()
        assert torch.equal(o, o2) and torch.equal(lse, l2)


# ---- d = 192 and 256: the one-tile-per-CTA kernel (csrc/fa_fwd_fp8_wide.cu)

@pytest.mark.parametrize("d,B,Hq,Hkv,N", [(256, 1, 2, 2, 128), (192, 2, 3, 1, 333), (256, 1, 2, 1, 1000)])
def test_fp8_wide_quantisers_bit_exact(fa, d, B, Hq, Hkv, N):
    t = inputs.make_inputs(B, Hq, Hkv, N, d, "bf16", seed=N + d)
    got = [x.cpu().numpy() for x in quantized(t)]
    fa.check_device_status()
    for name, a, r in zip(("q8", "q_scale", "k8", "k_scale", "vt8", "v_scale"), got, oracle_quant(t)):
        assert a.shape == r.shape, name
        assert np.array_equal(a.view(np.uint32) if a.dtype == np.float32 else a,
                              r.view(np.uint32) if r.dtype == np.float32 else r), name


@pytest.mark.parametrize("d", [192, 256])
@pytest.mark.parametrize("B,Hq,Hkv,N", [(1, 2, 2, 128), (2, 4, 2, 333), (1, 2, 1, 1000)])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_wide_forward_within_rounding_bound(fa, d, B, Hq, Hkv, N, causal):
    """Six-slot ring (wraps after three key tiles at N = 333 and 1000), the
    last 64-column box of d = 192 past d, ragged key and query tails."""
    t = inputs.make_inputs(B, Hq, Hkv, N, d, "bf16", seed=11 * N + d + causal)
    q8, qs, k8, ks, vt8, vs = quantized(t)
    o, lse = pkg.fwd_fp8(q8, qs, k8, ks, vt8, vs, causal=causal)
    fa.check_device_status()
    host = [x.cpu().numpy() for x in (q8, qs, k8, ks, vt8, vs)]
    print(check_against_bound(o.float().cpu().numpy(), lse.cpu().numpy(), *host, causal, d ** -0.5))


def test_fp8_wide_forward_rescales_and_sharp_logits(fa):
    N, d = 1300, 256
    t = inputs.make_inputs(1, 2, 2, N, d, "bf16", seed=78, q_mult=4.0)
    t["k"] = (t["k"].float() * torch.linspace(0.3, 3.0, N).view(1, 1, N, 1)).to(torch.bfloat16)
    q8, qs, k8, ks, vt8, vs = quantized(t)
    host = [x.cpu().numpy() for x in (q8, qs, k8, ks, vt8, vs)]
    for causal in (True, False):
        o, lse = pkg.fwd_fp8(q8, qs, k8, ks, vt8, vs, causal=causal)
        fa.check_device_status()
        check_against_bound(o.float().cpu().numpy(), lse.cpu().numpy(), *host, causal, d ** -0.5)


@pytest.mark.parametrize("Nq,Nk,causal,d", [(200, 700, True, 256), (500, 130, True, 192), (1, 777, True, 256),
                                            (1, 1, False, 192), (300, 1000, False, 256)])
def test_fp8_wide_forward_kv_lengths_and_degenerate(fa, Nq, Nk, causal, d):
    t = inputs.make_inputs(1, 4, 2, Nq, d, "bf16", seed=Nq + 5 * Nk + d, Nk=Nk)
    q8, qs, k8, ks, vt8, vs = quantized(t)
    o, lse = pkg.fwd_fp8(q8, qs, k8, ks, vt8, vs, causal=causal)
    fa.check_device_status()
    host = [x.cpu().numpy() for x in (q8, qs, k8, ks, vt8, vs)]
    check_against_bound(o.float().cpu().numpy(), lse.cpu().numpy(), *host, causal, d ** -0.5)


def test_fp8_wide_forward_full_size_sampled_rows(fa):
    """16 heads, N = 8192, d = 256, causal (the bench's d = 256 FP8
    workload): 256 seeded rows per head against the oracle; max, mean and
    bias gates."""
    w = configs.WORKLOADS["fp8_h16_n8192_d256_causal_fwd"]
    t = inputs.make_workload_inputs(w)
    q8, qs, k8, ks, vt8, vs = quantized(t)
    o, lse = pkg.fwd_fp8(q8, qs, k8, ks, vt8, vs, causal=True)
    fa.check_device_status()
    host = [x.cpu().numpy() for x in (q8, qs, k8, ks, vt8, vs)]
    deq = (ofp8.dequantize_rows(host[0], host[1]), ofp8.dequantize_rows(host[2], host[3]),
           ofp8.dequantize_v_transposed(host[4], host[5], w.N))
    rows = inputs.sample_rows(w.B, w.Hq, w.N, 256, seed=9)
    print(check_sampled_rows(o.float().cpu().numpy(), lse.cpu().numpy(), deq, True, w.scale, rows))


# ---- head dimensions between the built ones: multiples of 16, zero-filled in the next kernel up

@pytest.mark.parametrize("d,N", [(16, 200), (48, 333), (96, 129), (160, 300), (224, 1000)])
def test_fp8_ragged_head_dim_quantisers_bit_exact(fa, d, N):
    """The V quantiser's last 64-column pass holds d % 64 columns."""
    t = inputs.make_inputs(2, 2, 1, N, d, "bf16", seed=3 * N + d)
    got = [x.cpu().numpy() for x in quantized(t)]
    fa.check_device_status()
    for name, a, r in zip(("q8", "q_scale", "k8", "k_scale", "vt8", "v_scale"), got, oracle_quant(t)):
        assert a.shape == r.shape, name
        assert np.array_equal(a.view(np.uint32) if a.dtype == np.float32 else a,
                              r.view(np.uint32) if r.dtype == np.float32 else r), name


@pytest.mark.parametrize("d", [32, 96, 160, 224])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_ragged_head_dim_forward_within_rounding_bound(fa, d, causal):
    t = inputs.make_inputs(1, 4, 2, 700, d, "bf16", seed=17 * d + causal)
    q8, qs, k8, ks, vt8, vs = quantized(t)
    o, lse = pkg.fwd_fp8(q8, qs, k8, ks, vt8, vs, causal=causal)
    fa.check_device_status()
    host = [x.cpu().numpy() for x in (q8, qs, k8, ks, vt8, vs)]
    check_against_bound(o.float().cpu().numpy(), lse.cpu().numpy(), *host, causal, d ** -0.5)
