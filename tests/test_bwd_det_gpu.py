"""The deterministic backward (fa_bwd_deterministic): parity with the
double-precision oracle, bit-identical results on repeated runs, and
agreement with fa_bwd.

Bar: relative Frobenius error <= 1e-2 per gradient tensor.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from exact_attention_79_gb300 import configs, inputs

pytestmark = pytest.mark.gpu


def rel_fro(got, ref):
    den = np.linalg.norm(ref)
    if den == 0.0:
        return float(np.abs(got).max()) if got.size else 0.0
    return float(np.linalg.norm(got - ref) / den)


def fwd_bwd(fa, t, causal, scale, deterministic=True):
    dev = torch.device("cuda:0")
    g = {k: v.to(dev) for k, v in t.items()}
    o, lse = fa.fwd(g["q"], g["k"], g["v"], causal=causal, scale=scale)
    grads = fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal=causal, scale=scale, deterministic=deterministic)
    fa.check_device_status()
    return g, o, lse, grads


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal", [
    (1, 1, 1, 1, 128, True),
    (1, 2, 1, 127, 128, True),
    (2, 4, 2, 129, 128, True),
    (1, 8, 1, 257, 128, True),
    (1, 2, 2, 300, 64, False),
    (1, 2, 2, 300, 64, True),
    (1, 3, 3, 640, 128, False),
    (1, 2, 1, 1000, 128, True),
])
def test_det_bwd_edge_sizes(fa, B, Hq, Hkv, N, d, causal):
    scale = d ** -0.5
    t = inputs.make_inputs(B, Hq, Hkv, N, d, "bf16", seed=300 + N, with_grad=True)
    _, _, _, grads = fwd_bwd(fa, t, causal, scale)
    f = {k: inputs.to_f64(v) for k, v in t.items()}
    _, _, rdq, rdk, rdv = oracle.backward(f["q"], f["k"], f["v"], f["do"], causal, scale)
    errs = {n: rel_fro(g.float().cpu().numpy(), r) for n, g, r in zip(("dq", "dk", "dv"), grads, (rdq, rdk, rdv))}
    assert max(errs.values()) <= configs.TOL_GRAD_REL_FRO, errs


def test_det_bwd_n8192_full(fa):
    w = configs.WORKLOADS["bf16_h16_n8192_d128_causal_fwdbwd"]
    t = inputs.make_workload_inputs(w)
    _, _, _, grads = fwd_bwd(fa, t, w.causal, w.scale)
    f = {k: inputs.to_f64(v) for k, v in t.items()}
    _, _, rdq, rdk, rdv = oracle.backward(f["q"], f["k"], f["v"], f["do"], w.causal, w.scale)
    errs = {n: rel_fro(g.float().cpu().numpy(), r) for n, g, r in zip(("dq", "dk", "dv"), grads, (rdq, rdk, rdv))}
    print(w.name, errs)
    assert max(errs.values()) <= configs.TOL_GRAD_REL_FRO, errs


def test_det_bwd_is_bit_reproducible_and_matches_fa_bwd(fa):
    B, Hq, Hkv, N, d = 2, 8, 2, 900, 128
    t = inputs.make_inputs(B, Hq, Hkv, N, d, "bf16", seed=31, with_grad=True)
    g, o, lse, a = fwd_bwd(fa, t, True, d ** -0.5)
    b = fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal=True, deterministic=True)
    ref = fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal=True)
    fa.check_device_status()
    for x, y, r in zip(a, b, ref):
        assert torch.equal(x, y)
        assert rel_fro(x.float().cpu().numpy(), r.float().cpu().numpy()) < 5e-3


def test_det_bwd_workspace_needs_only_lse_and_d(fa):
    lib = fa.load()
    B, Hq, Hkv, N, d = 1, 2, 2, 256, 64
    small = 2 * B * Hq * 256 * 4
    dev = torch.device("cuda:0")
    t = inputs.make_inputs(B, Hq, Hkv, N, d, "bf16", seed=5, with_grad=True)
    q, k, v, do = (t[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = fa.fwd(q, k, v, causal=False)
    # the workspace is the head of a larger buffer whose tail is a canary: the
    # call may write only the `small` bytes it was given
    arena = torch.full((small + (1 << 20),), 0xA5, dtype=torch.uint8, device=dev)
    ws = arena[:small]
    out = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
    P = lambda x: ctypes.c_void_p(x.data_ptr())  # noqa: E731
    args = [P(q), P(k), P(v), P(o), P(lse), P(do), P(out[0]), P(out[1]), P(out[2]), P(ws)]
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.fa_bwd_deterministic(*args, small, B, Hq, Hkv, N, d, 0, 0.125, s) == 0
    assert lib.fa_bwd_deterministic(*args, small - 256, B, Hq, Hkv, N, d, 0, 0.125, s) == 6
    fa.check_device_status()
    assert bool((arena[small:] == 0xA5).all()), "wrote past the end of the workspace"
    ref = fa.bwd(q, k, v, o, lse, do, causal=False, scale=0.125)
    for x, r in zip(out, ref):
        assert rel_fro(x.float().cpu().numpy(), r.float().cpu().numpy()) < 5e-3
