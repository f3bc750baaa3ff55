"""fa_bwd_noalloc, the backward for callers that cannot allocate device
memory at call time (for example a plugin that only receives fixed buffers
from its host framework): its scratch is a fixed 32 MiB array owned by the
library instead of a caller-provided workspace.

It must give what fa_bwd gives, on two calls in a row (the second call must
not be disturbed by what the first left in the shared array), and must refuse
a problem whose scratch would not fit, without launching anything. This file
is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from exact_attention_79_gb300 import configs, inputs

pytestmark = pytest.mark.gpu

SCRATCH_LIMIT = 32 << 20


def rel_fro(got, ref):
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / den) if den > 0 else float(np.abs(got).max())


def test_noalloc_matches_fa_bwd_twice(fa):
    lib = fa.load()
    B, Hq, Hkv, N, d = 1, 8, 2, 1000, 128
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
                                B, Hq, Hkv, N, d, 1, d ** -0.5, stream)
        assert rc == 0, (call, rc)
        fa.check_device_status()
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            g, r = g.float().cpu().numpy(), r.float().cpu().numpy()
            assert np.isfinite(g).all(), (call, name)
            assert rel_fro(g, r) <= configs.TOL_GRAD_REL_FRO, (call, name, rel_fro(g, r))


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
