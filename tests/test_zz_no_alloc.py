"""fa_bwd_noalloc, the backward for callers that cannot allocate device
memory at call time (for example a plugin that only receives fixed buffers
from its host framework): its scratch is a fixed 32 MiB array owned by the
library instead of a caller-provided workspace.

It must give what fa_bwd gives (dK and dV bit for bit, dQ up to the order
of its fp32 reductions) on two calls in a row (the second call must not be
disturbed by what the first left in the shared array), must match the
oracle, and must refuse a problem whose scratch would not fit, without
launching anything. This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from exact_attention_79_gb300 import configs, inputs

pytestmark = pytest.mark.gpu

SCRATCH_LIMIT = 32 << 20


def rel_fro(got, ref):
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / den) if den > 0 else float(np.abs(got).max())


def test_noalloc_matches_fa_bwd_twice(fa):
    """Two calls in a row with different inputs: dK and dV bit-equal to
    fa_bwd's (both are accumulated in a fixed order), dQ equal up to the order
    of its fp32 reductions, and the first call's gradients within the
    tolerances of the double-precision oracle."""
    lib = fa.load()
    B, Hq, Hkv, N, d = 1, 8, 2, 1000, 128
    scale = d ** -0.5
    assert fa.bwd_workspace_bytes(B, Hq, Hkv, N, d) <= SCRATCH_LIMIT
    dev = torch.device("cuda:0")
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call, seed in enumerate((21, 22)):
        t = inputs.make_inputs(B, Hq, Hkv, N, d, "bf16", seed=seed, with_grad=True)
        q, k, v, do = (t[n].to(dev) for n in ("q", "k", "v", "do"))
        o, lse = fa.fwd(q, k, v, causal=True)
        ref = fa.bwd(q, k, v, o, lse, do, causal=True)
        got = [torch.full_like(x, float("nan")) for x in ref]
        rc = lib.fa_bwd_noalloc(P(q), P(k), P(v), P(o), P(lse), P(do), P(got[0]), P(got[1]), P(got[2]),
                                B, Hq, Hkv, N, d, 1, scale, stream)
        assert rc == 0, (call, rc)
        fa.check_device_status()
        assert torch.equal(got[1], ref[1]) and torch.equal(got[2], ref[2]), call
        g, r = got[0].float().cpu().numpy(), ref[0].float().cpu().numpy()
        assert np.isfinite(g).all(), call
        assert rel_fro(g, r) <= 1e-3, (call, rel_fro(g, r))
        if call == 0:
            f = {n: inputs.to_f64(x) for n, x in t.items()}
            _, _, rdq, rdk, rdv = oracle.backward(f["q"], f["k"], f["v"], f["do"], True, scale)
            for name, x, rx in zip(("dq", "dk", "dv"), got, (rdq, rdk, rdv)):
                e = rel_fro(x.float().cpu().numpy(), rx)
                assert e <= configs.TOL_GRAD_REL_FRO, (name, e)


def test_noalloc_refuses_problems_beyond_its_scratch(fa):
    lib = fa.load()
    B, Hq, Hkv, N, d = 1, 16, 16, 8192, 128
    assert fa.bwd_workspace_bytes(B, Hq, Hkv, N, d) > SCRATCH_LIMIT
    dev = torch.device("cuda:0")
    x = torch.zeros(16, dtype=torch.bfloat16, device=dev)     # never touched: refused before any launch
    lse = torch.zeros(16, dtype=torch.float32, device=dev)
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = lib.fa_bwd_noalloc(P(x), P(x), P(x), P(x), P(lse), P(x), P(x), P(x), P(x),
                            B, Hq, Hkv, N, d, 1, d ** -0.5, None)
    assert rc == 6       # FA_ERR_WORKSPACE
    fa.check_device_status()
