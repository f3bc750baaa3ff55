"""The backward at head dimensions 136..256 (csrc/fa_bwd_wide.cu: dV, dK and
dQ in three passes over 128-row steps, no atomics) through fa_bwd,
fa_bwd_kv, fa_bwd_deterministic and fa_bwd_noalloc, against the
double-precision oracle on the same rounded inputs: gradients within the
relative Frobenius bound, bit-identical from run to run and across the entry
points that share the path."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from exact_attention_79_gb300 import configs, inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def rel_fro(got, ref):
    den = np.linalg.norm(ref)
    if den == 0.0:
        return float(np.abs(got).max()) if got.size else 0.0
    return float(np.linalg.norm(got - ref) / den)


def check_grads(got, ref):
    errs = {n: rel_fro(g.float().cpu().numpy(), r) for n, g, r in zip(("dq", "dk", "dv"), got, ref)}
    assert all(np.isfinite(g.float().cpu().numpy()).all() for g in got)
    assert max(errs.values()) <= configs.TOL_GRAD_REL_FRO, errs
    return errs


CASES = [
    # B, Hq, Hkv, Nq, Nk, d, causal
    (1, 2, 2, 128, 128, 256, True),
    (1, 2, 2, 64, 64, 256, False),       # half a 128-row step, half a key tile
    (2, 4, 2, 333, 333, 256, True),      # ragged rows and keys, GQA
    (1, 2, 1, 700, 700, 192, False),     # d = 192 in the 256 build
    (1, 3, 3, 300, 300, 136, True),
    (1, 8, 2, 1000, 1000, 248, True),
    (1, 2, 2, 300, 1000, 256, True),     # queries at the end of longer keys
    (1, 2, 2, 500, 200, 256, True),      # more queries than keys: the first rows see nothing
    (1, 2, 2, 1, 777, 256, True),        # one decoding query
    (1, 1, 1, 1, 1, 256, False),
]


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal", CASES)
def test_wide_backward_matches_oracle(fa, B, Hq, Hkv, Nq, Nk, d, causal):
    scale = d ** -0.5
    t = inputs.make_inputs(B, Hq, Hkv, Nq, d, "bf16", seed=Nq + 5 * Nk + d, with_grad=True, Nk=Nk)
    g = {n: x.to(DEV) for n, x in t.items()}
    o, lse = fa.fwd(g["q"], g["k"], g["v"], causal=causal, scale=scale)
    a = fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal=causal, scale=scale)
    b = fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal=causal, scale=scale)
    fa.check_device_status()
    for x, y in zip(a, b):
        assert torch.equal(x, y)                 # no atomics: every output bit reproducible
    f = {n: inputs.to_f64(x) for n, x in t.items()}
    _, _, rdq, rdk, rdv = oracle.backward(f["q"], f["k"], f["v"], f["do"], causal, scale)
    print(check_grads(a, (rdq, rdk, rdv)))
    if Nq == Nk:
        c = fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal=causal, scale=scale, deterministic=True)
        fa.check_device_status()
        for x, y in zip(a, c):
            assert torch.equal(x, y)             # the same three passes


def test_wide_backward_full_size_sampled_rows(fa):
    """16 heads, N = 8192, d = 256, causal (the size the d = 256 forward is
    measured at): 256 seeded query rows (dQ) and 256 key rows (dK, dV) per
    head against the oracle, which computes LSE and D of every row itself."""
    B, H, N, d = 1, 16, 8192, 256
    scale = d ** -0.5
    t = inputs.make_inputs(B, H, H, N, d, "bf16", seed=8256, with_grad=True)
    g = {n: x.to(DEV) for n, x in t.items()}
    o, lse = fa.fwd(g["q"], g["k"], g["v"], causal=True, scale=scale)
    dq, dk, dv = fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal=True, scale=scale)
    fa.check_device_status()
    f = {n: inputs.to_f64(x) for n, x in t.items()}
    qr = inputs.sample_rows(B, H, N, 256, seed=1)
    kr = inputs.sample_rows(B, H, N, 256, seed=2)
    rl, rD = oracle.row_statistics(f["q"], f["k"], f["v"], f["do"], True, scale)
    rdq, rdk, rdv = oracle.backward_rows(f["q"], f["k"], f["v"], f["do"], True, scale, qr, kr, rl, rD)
    bi, hi = np.arange(B)[:, None, None], np.arange(H)[None, :, None]
    dq, dk, dv = (x.float().cpu().numpy() for x in (dq, dk, dv))
    assert all(np.isfinite(x).all() for x in (dq, dk, dv))
    errs = {"dq": rel_fro(dq[bi, hi, qr], rdq), "dk": rel_fro(dk[bi, hi, kr], rdk), "dv": rel_fro(dv[bi, hi, kr], rdv)}
    print(errs)
    assert max(errs.values()) <= configs.TOL_GRAD_REL_FRO, errs


def test_wide_backward_ragged_head_groups(fa):
    """3 heads at N = 24576, d = 256, causal: the passes walk heads in groups
    whose streamed operands fit in 64 MB of L2, here groups of 2 and 1 in
    every pass. 128 seeded query rows (dQ) and 128 key rows (dK, dV) per head
    against the oracle."""
    B, H, N, d = 1, 3, 24576, 256
    scale = d ** -0.5
    t = inputs.make_inputs(B, H, H, N, d, "bf16", seed=8257, with_grad=True)
    g = {n: x.to(DEV) for n, x in t.items()}
    o, lse = fa.fwd(g["q"], g["k"], g["v"], causal=True, scale=scale)
    dq, dk, dv = fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal=True, scale=scale)
    fa.check_device_status()
    f = {n: inputs.to_f64(x) for n, x in t.items()}
    qr = inputs.sample_rows(B, H, N, 128, seed=3)
    kr = inputs.sample_rows(B, H, N, 128, seed=4)
    rl, rD = oracle.row_statistics(f["q"], f["k"], f["v"], f["do"], True, scale)
    rdq, rdk, rdv = oracle.backward_rows(f["q"], f["k"], f["v"], f["do"], True, scale, qr, kr, rl, rD)
    bi, hi = np.arange(B)[:, None, None], np.arange(H)[None, :, None]
    dq, dk, dv = (x.float().cpu().numpy() for x in (dq, dk, dv))
    assert all(np.isfinite(x).all() for x in (dq, dk, dv))
    errs = {"dq": rel_fro(dq[bi, hi, qr], rdq), "dk": rel_fro(dk[bi, hi, kr], rdk), "dv": rel_fro(dv[bi, hi, kr], rdv)}
    print(errs)
    assert max(errs.values()) <= configs.TOL_GRAD_REL_FRO, errs


def test_wide_backward_noalloc_matches_fa_bwd(fa):
    lib = fa.load()
    B, Hq, Hkv, N, d = 1, 4, 2, 600, 256
    t = inputs.make_inputs(B, Hq, Hkv, N, d, "bf16", seed=31, with_grad=True)
    q, k, v, do = (t[n].to(DEV) for n in ("q", "k", "v", "do"))
    o, lse = fa.fwd(q, k, v, causal=True)
    ref = fa.bwd(q, k, v, o, lse, do, causal=True)
    got = [torch.full_like(x, float("nan")) for x in ref]
    P = lambda x: ctypes.c_void_p(x.data_ptr())  # noqa: E731
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.fa_bwd_noalloc(P(q), P(k), P(v), P(o), P(lse), P(do), P(got[0]), P(got[1]), P(got[2]),
                              B, Hq, Hkv, N, d, 1, d ** -0.5, s) == 0
    fa.check_device_status()
    for x, y in zip(got, ref):
        assert torch.equal(x, y)
