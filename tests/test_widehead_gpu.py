"""Head dimensions 136..256 (multiples of 8) in the forward: the wide-head
kernel (one 128-row query tile per CTA, K and V staged in 32 KB pieces),
d in (128, 192] running in the 192 build and (192, 256] in the 256 build with
the columns past d read as zeros and never written. The CUDA path through the
C ABI against the double-precision oracle on the same rounded inputs; bars as
for the dense path. The backward has no kernel above d = 128 and says so."""
import numpy as np
import pytest
import torch

import oracle
import exact_attention_79_gb300 as pkg
from exact_attention_79_gb300 import configs, inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def check_fwd(o, lse, ro, rl):
    o = o.float().cpu().numpy() if torch.is_tensor(o) else o
    lse = lse.cpu().numpy() if torch.is_tensor(lse) else lse
    fin = np.isfinite(rl)
    err = np.abs(o - ro)
    assert err.max() <= configs.TOL_O_MAX, err.max()
    assert err.mean() <= configs.TOL_O_MEAN, err.mean()
    assert np.array_equal(np.isfinite(lse), fin)
    if fin.any():
        assert np.abs(lse[fin] - rl[fin]).max() <= configs.TOL_LSE_MAX
    assert (lse[~fin] == -np.inf).all() and (o[~fin] == 0).all()
    return float(err.max())


def run_guarded(fa, g, causal, scale):
    """Forward into a buffer with guard bands: nothing outside O may change."""
    B, Hq, N, d = g["q"].shape
    pad = 1024
    total = B * Hq * N * d
    buf = torch.full((total + 2 * pad,), -7.0, dtype=torch.bfloat16, device=DEV)
    o = buf[pad:pad + total].view(B, Hq, N, d)
    o, lse = fa.fwd(g["q"], g["k"], g["v"], causal=causal, scale=scale, out=o)
    fa.check_device_status()
    assert bool((buf[:pad] == -7.0).all()) and bool((buf[pad + total:] == -7.0).all())
    return o, lse


@pytest.mark.parametrize("d", [136, 192, 200, 248, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_wide_fwd_ragged_gqa(fa, d, causal):
    B, Hq, Hkv, N = 2, 4, 2, 333            # three query tiles, the last one ragged
    scale = d ** -0.5
    t = inputs.make_inputs(B, Hq, Hkv, N, d, "bf16", seed=d + (1 if causal else 0))
    g = {n: x.to(DEV) for n, x in t.items()}
    o, lse = run_guarded(fa, g, causal, scale)
    f = {n: inputs.to_f64(x) for n, x in t.items()}
    ro, rl = oracle.forward(f["q"], f["k"], f["v"], causal, scale)
    check_fwd(o, lse, ro, rl)


@pytest.mark.parametrize("d", [192, 256])
def test_wide_fwd_many_tiles_and_rescale(fa, d):
    """Twelve key tiles (the 5-slot ring wraps several times) with keys that
    grow along the sequence, so the running max of most rows rises by more
    than 2^8 several times and the accumulator rescale runs."""
    B, Hq, Hkv, N = 1, 2, 1, 1500
    scale = d ** -0.5
    t = inputs.make_inputs(B, Hq, Hkv, N, d, "bf16", seed=40 + d)
    growth = torch.linspace(0.5, 4.0, N).view(1, 1, N, 1)
    t["k"] = (t["k"].float() * growth).to(torch.bfloat16)
    g = {n: x.to(DEV) for n, x in t.items()}
    f = {n: inputs.to_f64(x) for n, x in t.items()}
    for causal in (True, False):
        o, lse = run_guarded(fa, g, causal, scale)
        ro, rl = oracle.forward(f["q"], f["k"], f["v"], causal, scale)
        check_fwd(o, lse, ro, rl)


@pytest.mark.parametrize("Nq,Nk,causal", [(200, 700, True), (500, 130, True), (1, 777, True), (300, 1000, False)])
def test_wide_fwd_kv_lengths(fa, Nq, Nk, causal):
    """Queries are the last Nq of Nk positions (bottom-right causal); with more
    queries than keys the first rows see nothing: O = 0, LSE = -inf."""
    B, Hq, Hkv, d = 1, 2, 2, 256
    scale = d ** -0.5
    t = inputs.make_inputs(B, Hq, Hkv, Nq, d, "bf16", seed=Nq + Nk, Nk=Nk)
    g = {n: x.to(DEV) for n, x in t.items()}
    o, lse = run_guarded(fa, g, causal, scale)
    f = {n: inputs.to_f64(x) for n, x in t.items()}
    ro, rl = oracle.forward(f["q"], f["k"], f["v"], causal, scale)
    check_fwd(o, lse, ro, rl)


def test_wide_fwd_workload_sampled_rows(fa):
    """The d = 256 workload at full size (16 heads, N = 8192, causal); the
    oracle computes 256 seeded query rows per head."""
    w = configs.WORKLOADS["bf16_h16_n8192_d256_causal_fwd"]
    t = inputs.make_workload_inputs(w, with_grad=False)
    g = {n: x.to(DEV) for n, x in t.items()}
    o, lse = fa.fwd(g["q"], g["k"], g["v"], causal=w.causal, scale=w.scale)
    fa.check_device_status()
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    rows = inputs.sample_rows(w.B, w.Hq, w.N, 256, seed=3)
    f = {n: inputs.to_f64(x) for n, x in t.items()}
    ro, rl = oracle.forward_rows(f["q"], f["k"], f["v"], w.causal, w.scale, rows)
    bi = np.arange(w.B)[:, None, None]
    hi = np.arange(w.Hq)[None, :, None]
    check_fwd(o[bi, hi, rows], lse[bi, hi, rows], ro, rl)


def test_wide_fwd_repeated_calls_identical(fa):
    t = inputs.make_inputs(1, 4, 4, 1000, 256, "bf16", seed=9)
    g = {n: x.to(DEV) for n, x in t.items()}
    o1, l1 = fa.fwd(g["q"], g["k"], g["v"], causal=True)
    for _ in range(5):
        o2, l2 = fa.fwd(g["q"], g["k"], g["v"], causal=True)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
    fa.check_device_status()


def test_wide_block_mask_refused(fa):
    q = torch.zeros(1, 2, 256, 256, dtype=torch.bfloat16, device=DEV)
    lse = torch.zeros(1, 2, 256, dtype=torch.float32, device=DEV)
    with pytest.raises(pkg.FAError):
        fa.fwd(q, q, q, causal=True, block_mask=torch.ones(1, 1, 2, 2, dtype=torch.bool, device=DEV))
    with pytest.raises(pkg.FAError):
        fa.bwd(q, q, q, q, lse, q, block_mask=torch.ones(1, 1, 2, 2, dtype=torch.bool, device=DEV))
    fa.check_device_status()


def test_wide_fwd_long_sequence_sampled_rows(fa):
    """d = 256, N = 32768, 4 heads, causal: 256 key tiles for the last rows,
    the ring wraps about two hundred times and all four heads fit one head
    group; 64 seeded rows per head against the oracle."""
    B, H, N, d = 1, 4, 32768, 256
    t = inputs.make_inputs(B, H, H, N, d, "bf16", seed=32768)
    g = {n: x.to(DEV) for n, x in t.items()}
    o, lse = fa.fwd(g["q"], g["k"], g["v"], causal=True)
    fa.check_device_status()
    rows = inputs.sample_rows(B, H, N, 64, seed=7)
    f = {n: inputs.to_f64(x) for n, x in t.items()}
    ro, rl = oracle.forward_rows(f["q"], f["k"], f["v"], True, d ** -0.5, rows)
    bi, hi = np.arange(B)[:, None, None], np.arange(H)[None, :, None]
    check_fwd(o[bi, hi, rows], lse[bi, hi, rows], ro, rl)
