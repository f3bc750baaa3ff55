"""Head dimensions other than 64 and 128 (multiples of 8 up to 128): they run
in the kernels built for the next size up, with the columns past d read as
zeros and never written. The CUDA path through the C ABI against the
double-precision oracle; bars as for the dense path."""
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


@pytest.mark.parametrize("d", [8, 32, 48, 72, 80, 96, 112])
@pytest.mark.parametrize("causal", [False, True])
def test_headdim_fwd_bwd(fa, d, causal):
    B, Hq, Hkv, N = 1, 4, 2, 333
    scale = d ** -0.5
    t = inputs.make_inputs(B, Hq, Hkv, N, d, "bf16", seed=d + 2, with_grad=True)
    dev = torch.device("cuda:0")
    g = {n: x.to(dev) for n, x in t.items()}
    # guard bands around the outputs: nothing past d may be written
    pad = 512
    buf = torch.full((B * Hq * N * d + 2 * pad,), -7.0, dtype=torch.bfloat16, device=dev)
    o = buf[pad:pad + B * Hq * N * d].view(B, Hq, N, d)
    o, lse = fa.fwd(g["q"], g["k"], g["v"], causal=causal, scale=scale, out=o)
    dq, dk, dv = fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal=causal, scale=scale)
    fa.check_device_status()
    assert bool((buf[:pad] == -7.0).all()) and bool((buf[pad + B * Hq * N * d:] == -7.0).all())
    f = {n: inputs.to_f64(x) for n, x in t.items()}
    ro, rl, rdq, rdk, rdv = oracle.backward(f["q"], f["k"], f["v"], f["do"], causal, scale)
    err = np.abs(o.float().cpu().numpy() - ro)
    assert err.max() <= configs.TOL_O_MAX and err.mean() <= configs.TOL_O_MEAN
    assert np.abs(lse.cpu().numpy() - rl).max() <= configs.TOL_LSE_MAX
    errs = {n: rel_fro(a.float().cpu().numpy(), r) for n, a, r in zip(("dq", "dk", "dv"), (dq, dk, dv), (rdq, rdk, rdv))}
    assert max(errs.values()) <= configs.TOL_GRAD_REL_FRO, errs


@pytest.mark.parametrize("d", [16, 40, 96, 120])
def test_headdim_deterministic(fa, d):
    """The bit-reproducible backward at other head dims: the same next-size-up
    kernels; against the oracle and bit-identical across two runs."""
    B, Hq, Hkv, N = 1, 4, 2, 300
    scale = d ** -0.5
    t = inputs.make_inputs(B, Hq, Hkv, N, d, "bf16", seed=3 * d, with_grad=True)
    dev = torch.device("cuda:0")
    g = {n: x.to(dev) for n, x in t.items()}
    o, lse = fa.fwd(g["q"], g["k"], g["v"], causal=True, scale=scale)
    r1 = fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal=True, scale=scale, deterministic=True)
    r2 = fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal=True, scale=scale, deterministic=True)
    fa.check_device_status()
    assert all(torch.equal(a, b) for a, b in zip(r1, r2))
    f = {n: inputs.to_f64(x) for n, x in t.items()}
    _, _, rdq, rdk, rdv = oracle.backward(f["q"], f["k"], f["v"], f["do"], True, scale)
    errs = {n: rel_fro(a.float().cpu().numpy(), r) for n, a, r in zip(("dq", "dk", "dv"), r1, (rdq, rdk, rdv))}
    assert max(errs.values()) <= configs.TOL_GRAD_REL_FRO, errs
