"""Forward parity: the CUDA forward (through the C ABI) against the
double-precision oracle on the same seeded, rounded inputs.

Bar: max|dO| <= 2e-2, mean|dO| <= 2e-3, max|dLSE| <= 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_79_gb300 import configs, inputs

pytestmark = pytest.mark.gpu


def run_fwd(fa, t, causal, scale):
    dev = torch.device("cuda:0")
    q, k, v = (t[n].to(dev) for n in ("q", "k", "v"))
    o, lse = fa.fwd(q, k, v, causal=causal, scale=scale)
    fa.check_device_status()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def check_fwd(o, lse, ro, rl, label=""):
    err = np.abs(o - ro)
    lerr = np.abs(lse - rl)
    assert np.isfinite(o).all() and np.isfinite(lse).all(), label
    assert err.max() <= configs.TOL_O_MAX, (label, "max", err.max())
    assert err.mean() <= configs.TOL_O_MEAN, (label, "mean", err.mean())
    assert lerr.max() <= configs.TOL_LSE_MAX, (label, "lse", lerr.max())
    return err.max(), err.mean(), lerr.max()


EDGE = [
    # B, Hq, Hkv, N, d, causal, dtype
    (1, 1, 1, 1, 64, False, "bf16"),
    (1, 1, 1, 1, 128, True, "bf16"),
    (1, 2, 1, 127, 128, True, "bf16"),
    (1, 2, 2, 128, 64, False, "bf16"),
    (1, 2, 2, 128, 128, True, "bf16"),
    (2, 4, 2, 129, 128, True, "bf16"),
    (1, 8, 1, 257, 128, True, "bf16"),
    (1, 2, 2, 300, 64, False, "bf16"),
    (1, 2, 2, 300, 64, True, "bf16"),
    (1, 4, 4, 384, 128, False, "bf16"),
    (1, 2, 1, 1000, 128, True, "bf16"),
    (1, 3, 3, 640, 128, False, "bf16"),
    (1, 1, 1, 128, 64, False, "fp32"),
    (1, 2, 1, 200, 64, True, "fp32"),
    (1, 2, 2, 513, 64, False, "fp32"),
]


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal,dtype", EDGE)
def test_fwd_edge_sizes(fa, B, Hq, Hkv, N, d, causal, dtype):
    scale = d ** -0.5
    t = inputs.make_inputs(B, Hq, Hkv, N, d, dtype, seed=N + d)
    o, lse = run_fwd(fa, t, causal, scale)
    f = {k: inputs.to_f64(v) for k, v in t.items()}
    ro, rl = oracle.forward(f["q"], f["k"], f["v"], causal, scale)
    check_fwd(o, lse, ro, rl, (B, Hq, Hkv, N, d, causal, dtype))


@pytest.mark.parametrize("name", ["fp32_h1_n128_d64", "bf16_b4_h16_n2048_d64", "bf16_b4_h16_n2048_d64_q4"])
def test_fwd_workload_full(fa, name):
    w = configs.WORKLOADS[name]
    t = inputs.make_workload_inputs(w)
    o, lse = run_fwd(fa, t, w.causal, w.scale)
    f = {k: inputs.to_f64(v) for k, v in t.items()}
    ro, rl = oracle.forward(f["q"], f["k"], f["v"], w.causal, w.scale)
    print(name, check_fwd(o, lse, ro, rl, name))


@pytest.mark.parametrize("name", ["bf16_gqa_b2_h64kv8_n4096_d128_causal", "bf16_h8_n65536_d128_causal_fwdbwd"])
def test_fwd_workload_sampled_rows(fa, name):
    """Full-size launch; the oracle computes 256 seeded query rows per head."""
    w = configs.WORKLOADS[name]
    t = inputs.make_workload_inputs(w, with_grad=False)
    o, lse = run_fwd(fa, t, w.causal, w.scale)
    rows = inputs.sample_rows(w.B, w.Hq, w.N, 256, seed=1)
    f = {k: inputs.to_f64(v) for k, v in t.items()}
    ro, rl = oracle.forward_rows(f["q"], f["k"], f["v"], w.causal, w.scale, rows)
    bi = np.arange(w.B)[:, None, None]
    hi = np.arange(w.Hq)[None, :, None]
    print(name, check_fwd(o[bi, hi, rows], lse[bi, hi, rows], ro, rl, name))
    assert np.isfinite(o).all() and np.isfinite(lse).all()


def test_fwd_longest_sequence_sampled_rows(fa):
    """N = 131072, the longest sequence a block mask can describe (1024 query
    tiles): the dense causal forward with two query heads on one KV head, and
    the block-sparse forward with a local window of 8 key tiles. 128 seeded
    query rows per head, the first and the last row among them, against the
    oracle."""
    B, Hq, Hkv, N, d = 1, 2, 1, 131072, 128
    scale = d ** -0.5
    t = inputs.make_inputs(B, Hq, Hkv, N, d, "bf16", seed=131072)
    f = {k: inputs.to_f64(v) for k, v in t.items()}
    inner = inputs.sample_rows(B, Hq, N - 2, 126, seed=4) + 1          # rows 1 .. N-2
    ends = np.broadcast_to(np.array([0, N - 1]), (B, Hq, 2))
    rows = np.sort(np.concatenate([inner, ends], axis=2), axis=2)
    bi = np.arange(B)[:, None, None]
    hi = np.arange(Hq)[None, :, None]

    o, lse = run_fwd(fa, t, True, scale)
    ro, rl = oracle.forward_rows(f["q"], f["k"], f["v"], True, scale, rows)
    print("dense", check_fwd(o[bi, hi, rows], lse[bi, hi, rows], ro, rl, "dense N=131072"))

    T = N // 128
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    m = ((j <= i) & (j > i - 8))[None, None]
    dev = torch.device("cuda:0")
    q, k, v = (t[n].to(dev) for n in ("q", "k", "v"))
    os_, ls_ = fa.fwd(q, k, v, causal=True, scale=scale, block_mask=torch.from_numpy(m.astype(np.uint8)).to(dev))
    fa.check_device_status()
    os_, ls_ = os_.float().cpu().numpy(), ls_.cpu().numpy()
    ro, rl = oracle.forward_rows(f["q"], f["k"], f["v"], True, scale, rows, block_mask=m)
    print("local window", check_fwd(os_[bi, hi, rows], ls_[bi, hi, rows], ro, rl, "block-sparse N=131072"))


def test_fwd_n8192_full(fa):
    w = configs.WORKLOADS["bf16_h16_n8192_d128_causal_fwdbwd"]
    t = inputs.make_workload_inputs(w, with_grad=False)
    o, lse = run_fwd(fa, t, w.causal, w.scale)
    f = {k: inputs.to_f64(v) for k, v in t.items()}
    ro, rl = oracle.forward(f["q"], f["k"], f["v"], w.causal, w.scale)
    print(w.name, check_fwd(o, lse, ro, rl, w.name))


def test_fwd_deterministic_and_guard_bands(fa):
    """Two runs give identical bits; rows past N and memory around the output
    are never written."""
    B, Hq, Hkv, N, d = 1, 4, 2, 333, 128
    t = inputs.make_inputs(B, Hq, Hkv, N, d, "bf16", seed=5)
    dev = torch.device("cuda:0")
    q, k, v = (t[n].to(dev) for n in ("q", "k", "v"))
    pad = 4096
    n = B * Hq * N * d
    canary = torch.full((n + 2 * pad,), -12345.0, dtype=torch.bfloat16, device=dev)
    o = canary[pad:pad + n].view(B, Hq, N, d)
    lse_buf = torch.full((B * Hq * N + 2 * 64,), -777.0, dtype=torch.float32, device=dev)
    lse = lse_buf[64:64 + B * Hq * N].view(B, Hq, N)
    fa.fwd(q, k, v, causal=True, out=o, lse=lse)
    o2, l2 = fa.fwd(q, k, v, causal=True)
    fa.check_device_status()
    assert torch.equal(o, o2) and torch.equal(lse, l2)
    assert bool((canary[:pad] == -12345.0).all()) and bool((canary[pad + n:] == -12345.0).all())
    assert bool((lse_buf[:64] == -777.0).all()) and bool((lse_buf[64 + B * Hq * N:] == -777.0).all())


def test_fwd_rejects_bad_arguments(fa):
    import ctypes
    lib = fa.load()
    dev = torch.device("cuda:0")
    x = torch.zeros(1, 2, 128, 64, dtype=torch.bfloat16, device=dev)
    lse = torch.zeros(1, 2, 128, dtype=torch.float32, device=dev)
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    s = ctypes.c_void_p(0)
    assert lib.fa_fwd(None, P(x), P(x), P(x), P(lse), 1, 2, 2, 128, 64, 0, 0.125, s) == 1
    assert lib.fa_fwd(P(x), P(x), P(x), P(x), P(lse), 1, 2, 2, 128, 100, 0, 0.125, s) == 1
    assert lib.fa_fwd(P(x), P(x), P(x), P(x), P(lse), 1, 2, 3, 128, 64, 0, 0.125, s) == 1
    assert lib.fa_fwd(P(x), P(x), P(x), P(x), P(lse), 1, 2, 2, 0, 64, 0, 0.125, s) == 1
    assert lib.fa_fwd(P(x), P(x), P(x), P(x), P(lse), 1, 2, 2, 128, 64, 0, float("nan"), s) == 1
    mis = ctypes.c_void_p(x.data_ptr() + 2)
    assert lib.fa_fwd(mis, P(x), P(x), P(x), P(lse), 1, 2, 2, 100, 64, 0, 0.125, s) == 1
    xf = torch.zeros(1, 1, 128, 128, dtype=torch.float32, device=dev)
    assert lib.fa_fwd_f32(P(xf), P(xf), P(xf), P(xf), P(lse), 1, 1, 1, 128, 128, 0, 0.1, s) == 2
    fa.check_device_status()


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal", [(1, 1, 1, 1, 64, False), (1, 1, 1, 1, 128, True),
                                                  (1, 2, 1, 300, 64, True), (2, 4, 2, 520, 128, False)])
def test_fwd_repeated_calls_identical(fa, B, Hq, Hkv, N, d, causal):
    """Ten launches on the same inputs, output buffers reused by the caching
    allocator: every launch gives the same bits, and those match the oracle.
    Catches reads of undefined registers or shared memory that depend on what
    an earlier launch left behind."""
    scale = d ** -0.5
    t = inputs.make_inputs(B, Hq, Hkv, N, d, "bf16", seed=31 + N, with_grad=False)
    dev = torch.device("cuda:0")
    q, k, v = (t[n].to(dev) for n in ("q", "k", "v"))
    runs = []
    for _ in range(10):
        o, lse = fa.fwd(q, k, v, causal=causal, scale=scale)
        runs.append((o.clone(), lse.clone()))
        del o, lse
    fa.check_device_status()
    for o, lse in runs[1:]:
        assert torch.equal(o, runs[0][0]) and torch.equal(lse, runs[0][1])
    f = {n: inputs.to_f64(t[n]) for n in ("q", "k", "v")}
    ro, rl = oracle.forward(f["q"], f["k"], f["v"], causal, scale)
    check_fwd(runs[0][0].float().cpu().numpy(), runs[0][1].cpu().numpy(), ro, rl, "repeated")
