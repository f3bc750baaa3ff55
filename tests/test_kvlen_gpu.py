"""Queries and keys of different lengths (fa_fwd_kv, fa_bwd_kv): the queries
are the last Nq of Nk positions, so under the causal rule key j is visible to
query i iff j <= i + (Nk - Nq). The CUDA path through the C ABI against the
double-precision oracle on the same rounded inputs; bars as for the dense
path (rows that see no key must give exactly O = 0 and LSE = -inf)."""
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


CASES = [
    # B, Hq, Hkv, Nq, Nk, d, causal
    (1, 2, 2, 128, 1024, 128, True),     # a chunk at the end of a longer sequence
    (1, 4, 2, 300, 1000, 128, True),     # ragged on both sides, offset not a tile multiple
    (2, 2, 1, 1, 777, 128, True),        # one decoding query
    (1, 2, 2, 500, 200, 128, True),      # more queries than keys: the first 300 rows see nothing
    (1, 2, 2, 300, 1000, 64, False),
    (1, 3, 3, 700, 129, 64, True),
    (1, 2, 2, 1000, 1000, 128, True),    # equal lengths through the same entry points
]


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal", CASES)
def test_kvlen_fwd_bwd(fa, B, Hq, Hkv, Nq, Nk, d, causal):
    scale = d ** -0.5
    t = inputs.make_inputs(B, Hq, Hkv, Nq, d, "bf16", seed=Nq + 7 * Nk, with_grad=True, Nk=Nk)
    dev = torch.device("cuda:0")
    g = {n: x.to(dev) for n, x in t.items()}
    o, lse = fa.fwd(g["q"], g["k"], g["v"], causal=causal, scale=scale)
    dq, dk, dv = fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal=causal, scale=scale)
    fa.check_device_status()
    f = {n: inputs.to_f64(x) for n, x in t.items()}
    ro, rl, rdq, rdk, rdv = oracle.backward(f["q"], f["k"], f["v"], f["do"], causal, scale)
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    seen = np.isfinite(rl)
    assert np.all(o[~seen] == 0) and np.all(np.isneginf(lse[~seen]))
    err = np.abs(o - ro)
    assert err.max() <= configs.TOL_O_MAX and err.mean() <= configs.TOL_O_MEAN
    assert np.abs(lse[seen] - rl[seen]).max() <= configs.TOL_LSE_MAX
    got = [x.float().cpu().numpy() for x in (dq, dk, dv)]
    assert all(np.isfinite(x).all() for x in got)
    errs = {n: rel_fro(a, r) for n, a, r in zip(("dq", "dk", "dv"), got, (rdq, rdk, rdv))}
    assert max(errs.values()) <= configs.TOL_GRAD_REL_FRO, errs


def test_kvlen_equal_lengths_match_fa_fwd(fa):
    """Nq == Nk through fa_fwd_kv gives fa_fwd's bits."""
    B, Hq, Hkv, N, d = 1, 4, 2, 600, 128
    t = inputs.make_inputs(B, Hq, Hkv, N, d, "bf16", seed=3, with_grad=False)
    dev = torch.device("cuda:0")
    q, k, v = (t[n].to(dev) for n in ("q", "k", "v"))
    lib = fa.load()
    import ctypes
    P = lambda x: ctypes.c_void_p(x.data_ptr())  # noqa: E731
    o1, l1 = torch.empty_like(q), torch.empty(B, Hq, N, dtype=torch.float32, device=dev)
    assert lib.fa_fwd_kv(P(q), P(k), P(v), P(o1), P(l1), B, Hq, Hkv, N, N, d, 1, d ** -0.5, None) == 0
    o2, l2 = fa.fwd(q, k, v, causal=True)
    fa.check_device_status()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_kvlen_chunked_prefill_workload_sampled_rows(fa):
    """The unequal-length bench workload at full size (GQA 32/8 heads, 4096
    queries at the end of 32768 keys, causal): 256 seeded query rows per head
    of O, LSE and dQ, and 256 seeded key rows per KV head of dK and dV,
    against the oracle (which computes LSE and D of every query row itself);
    two backward launches give bit-identical dK and dV."""
    w = configs.WORKLOADS["bf16_gqa_h32kv8_nq4096_nk32768_d128_causal_fwdbwd"]
    t = inputs.make_workload_inputs(w)
    dev = torch.device("cuda:0")
    g = {n: x.to(dev) for n, x in t.items()}
    o, lse = fa.fwd(g["q"], g["k"], g["v"], causal=True, scale=w.scale)
    a = fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal=True, scale=w.scale)
    b = fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal=True, scale=w.scale)
    fa.check_device_status()
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    rows = inputs.sample_rows(w.B, w.Hq, w.N, 256, seed=1)
    krows = inputs.sample_rows(w.B, w.Hkv, w.Nk, 256, seed=2)
    f = {n: inputs.to_f64(t[n]) for n in ("q", "k", "v", "do")}
    ro, rl = oracle.forward_rows(f["q"], f["k"], f["v"], True, w.scale, rows)
    bi = np.arange(w.B)[:, None, None]
    hi = np.arange(w.Hq)[None, :, None]
    hk = np.arange(w.Hkv)[None, :, None]
    og = o.float().cpu().numpy()[bi, hi, rows]
    lg = lse.cpu().numpy()[bi, hi, rows]
    err = np.abs(og - ro)
    assert err.max() <= configs.TOL_O_MAX and err.mean() <= configs.TOL_O_MEAN
    assert np.abs(lg - rl).max() <= configs.TOL_LSE_MAX
    rl_all, rD_all = oracle.row_statistics(f["q"], f["k"], f["v"], f["do"], True, w.scale)
    assert np.abs(lse.cpu().numpy() - rl_all).max() <= configs.TOL_LSE_MAX
    rdq, rdk, rdv = oracle.backward_rows(f["q"], f["k"], f["v"], f["do"], True, w.scale, rows, krows, rl_all, rD_all)
    dq, dk, dv = (x.float().cpu().numpy() for x in a)
    assert all(np.isfinite(x).all() for x in (dq, dk, dv))
    errs = {"dq": rel_fro(dq[bi, hi, rows], rdq), "dk": rel_fro(dk[bi, hk, krows], rdk),
            "dv": rel_fro(dv[bi, hk, krows], rdv)}
    print(w.name, errs)
    assert max(errs.values()) <= configs.TOL_GRAD_REL_FRO, errs
