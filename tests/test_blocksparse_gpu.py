"""Block-sparse attention (masks over 128 x 128 tiles): the CUDA path through
the C ABI against the double-precision oracle with the same block mask.

Bars as for the dense path: forward max|dO| <= 2e-2, mean|dO| <= 2e-3,
max|dLSE| <= 1e-3 on rows that see a key (rows that see none must give
exactly O = 0 and LSE = -inf); gradients relative Frobenius error <= 1e-2.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_79_gb300 import configs, inputs

pytestmark = pytest.mark.gpu


def block_mask(B, Hq, N, density, seed, empty_tiles=()):
    """Seeded random block mask [B, Hq, T, T] (numpy bool). Tiles listed in
    empty_tiles as (b, h, i) see no key tile at all."""
    T = (N + 127) // 128
    rng = np.random.Generator(np.random.PCG64(seed))
    m = rng.random((B, Hq, T, T)) < density
    for b, h, i in empty_tiles:
        m[b, h, i, :] = False
    return m


def run_fwd(fa, t, causal, scale, mask_np, broadcast_heads=False):
    dev = torch.device("cuda:0")
    q, k, v = (t[n].to(dev) for n in ("q", "k", "v"))
    mt = torch.tensor(mask_np[:, :1] if broadcast_heads else mask_np, dtype=torch.uint8, device=dev)
    o, lse = fa.fwd(q, k, v, causal=causal, scale=scale, block_mask=mt)
    fa.check_device_status()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def check_fwd(o, lse, ro, rl):
    seen = np.isfinite(rl)
    assert np.all(o[~seen] == 0) and np.all(np.isneginf(lse[~seen]))
    assert np.isfinite(o).all() and np.isfinite(lse[seen]).all()
    err = np.abs(o - ro)
    assert err.max() <= configs.TOL_O_MAX and err.mean() <= configs.TOL_O_MEAN, (err.max(), err.mean())
    assert np.abs(lse[seen] - rl[seen]).max() <= configs.TOL_LSE_MAX


CASES = [
    # B, Hq, Hkv, N, d, causal, density, empty (b, h, i) tiles
    (1, 2, 2, 300, 128, False, 0.5, ((0, 1, 1),)),
    (1, 2, 2, 300, 128, True, 0.5, ()),
    (2, 4, 2, 1000, 128, True, 0.4, ((1, 3, 2), (0, 0, 0))),
    (1, 4, 1, 1000, 64, False, 0.3, ((0, 2, 5),)),
    (1, 2, 2, 129, 64, True, 0.7, ()),
    (1, 3, 3, 1536, 128, False, 0.25, ((0, 0, 0), (0, 0, 1))),
]


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal,density,empty", CASES)
def test_blocksparse_fwd(fa, B, Hq, Hkv, N, d, causal, density, empty):
    scale = d ** -0.5
    t = inputs.make_inputs(B, Hq, Hkv, N, d, "bf16", seed=N + 3, with_grad=False)
    m = block_mask(B, Hq, N, density, seed=N, empty_tiles=empty)
    o, lse = run_fwd(fa, t, causal, scale, m)
    f = {n: inputs.to_f64(t[n]) for n in ("q", "k", "v")}
    ro, rl = oracle.forward(f["q"], f["k"], f["v"], causal, scale, block_mask=m)
    check_fwd(o, lse, ro, rl)


def test_blocksparse_fwd_broadcast_over_heads(fa):
    B, Hq, Hkv, N, d = 2, 4, 4, 700, 128
    t = inputs.make_inputs(B, Hq, Hkv, N, d, "bf16", seed=11, with_grad=False)
    m = block_mask(B, 1, N, 0.5, seed=12)
    o, lse = run_fwd(fa, t, True, d ** -0.5, m, broadcast_heads=True)
    f = {n: inputs.to_f64(t[n]) for n in ("q", "k", "v")}
    ro, rl = oracle.forward(f["q"], f["k"], f["v"], True, d ** -0.5, block_mask=m)
    check_fwd(o, lse, ro, rl)


@pytest.mark.parametrize("causal", [False, True])
def test_blocksparse_all_ones_equals_dense(fa, causal):
    """With every tile visible the block-sparse kernel computes exactly what the
    dense one does: same bits."""
    B, Hq, Hkv, N, d = 1, 4, 2, 1000, 128
    t = inputs.make_inputs(B, Hq, Hkv, N, d, "bf16", seed=13, with_grad=False)
    dev = torch.device("cuda:0")
    q, k, v = (t[n].to(dev) for n in ("q", "k", "v"))
    T = (N + 127) // 128
    ones = torch.ones(1, 1, T, T, dtype=torch.uint8, device=dev)
    o1, l1 = fa.fwd(q, k, v, causal=causal, block_mask=ones)
    o2, l2 = fa.fwd(q, k, v, causal=causal)
    fa.check_device_status()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_blocksparse_rejects_bad_masks(fa):
    dev = torch.device("cuda:0")
    q = torch.zeros(1, 2, 256, 64, dtype=torch.bfloat16, device=dev)
    with pytest.raises(ValueError):
        fa.fwd(q, q, q, block_mask=torch.ones(1, 2, 3, 3, dtype=torch.uint8, device=dev))
    with pytest.raises(ValueError):
        fa.fwd(q, q, q, block_mask=torch.ones(1, 2, 2, 2, dtype=torch.int32, device=dev))
    lib = fa.load()
    import ctypes
    P = lambda x: ctypes.c_void_p(x.data_ptr())  # noqa: E731
    lse = torch.zeros(1, 2, 256, dtype=torch.float32, device=dev)
    assert lib.fa_fwd_blocksparse(P(q), P(q), P(q), P(q), P(lse), None, 0, 0, 1, 2, 2, 256, 64, 0, 0.125, None) == 1
    m = torch.ones(1, 1, 2, 2, dtype=torch.uint8, device=dev)
    assert lib.fa_fwd_blocksparse(P(q), P(q), P(q), P(q), P(lse), P(m), -1, 0, 1, 2, 2, 256, 64, 0, 0.125, None) == 1
    fa.check_device_status()


def rel_fro(got, ref):
    den = np.linalg.norm(ref)
    if den == 0.0:
        return float(np.abs(got).max()) if got.size else 0.0
    return float(np.linalg.norm(got - ref) / den)


BWD_CASES = [
    # B, Hq, Hkv, N, d, causal, density, empty (b, h, i) query tiles
    (1, 2, 2, 300, 128, False, 0.5, ((0, 1, 1),)),
    (1, 2, 2, 300, 128, True, 0.6, ()),
    (2, 4, 2, 1000, 128, True, 0.4, ((1, 3, 2),)),
    (1, 4, 1, 1000, 64, False, 0.3, ((0, 2, 5),)),
    (1, 2, 2, 1536, 128, False, 0.15, ()),
]


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal,density,empty", BWD_CASES)
def test_blocksparse_bwd(fa, B, Hq, Hkv, N, d, causal, density, empty):
    scale = d ** -0.5
    t = inputs.make_inputs(B, Hq, Hkv, N, d, "bf16", seed=N + 5, with_grad=True)
    m = block_mask(B, Hq, N, density, seed=N + 1, empty_tiles=empty)
    dev = torch.device("cuda:0")
    g = {n: x.to(dev) for n, x in t.items()}
    mt = torch.tensor(m, dtype=torch.uint8, device=dev)
    o, lse = fa.fwd(g["q"], g["k"], g["v"], causal=causal, scale=scale, block_mask=mt)
    dq, dk, dv = fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal=causal, scale=scale, block_mask=mt)
    fa.check_device_status()
    f = {n: inputs.to_f64(x) for n, x in t.items()}
    ro, rl, rdq, rdk, rdv = oracle.backward(f["q"], f["k"], f["v"], f["do"], causal, scale, block_mask=m)
    check_fwd(o.float().cpu().numpy(), lse.cpu().numpy(), ro, rl)
    got = [x.float().cpu().numpy() for x in (dq, dk, dv)]
    assert all(np.isfinite(x).all() for x in got)
    errs = {n: rel_fro(a, r) for n, a, r in zip(("dq", "dk", "dv"), got, (rdq, rdk, rdv))}
    assert max(errs.values()) <= configs.TOL_GRAD_REL_FRO, errs


def test_blocksparse_bwd_key_tile_seen_by_nobody(fa):
    """A key tile no query tile sees gets dK = dV = 0 exactly (its dK/dV
    block has no step at all)."""
    B, Hq, Hkv, N, d = 1, 2, 1, 512, 128
    t = inputs.make_inputs(B, Hq, Hkv, N, d, "bf16", seed=21, with_grad=True)
    m = np.ones((B, Hq, 4, 4), dtype=bool)
    m[:, :, :, 2] = False                           # key tile 2 hidden from every query tile
    dev = torch.device("cuda:0")
    g = {n: x.to(dev) for n, x in t.items()}
    mt = torch.tensor(m, dtype=torch.uint8, device=dev)
    o, lse = fa.fwd(g["q"], g["k"], g["v"], block_mask=mt)
    dq, dk, dv = fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], block_mask=mt)
    fa.check_device_status()
    assert bool((dk[:, :, 256:384] == 0).all()) and bool((dv[:, :, 256:384] == 0).all())
    f = {n: inputs.to_f64(x) for n, x in t.items()}
    _, _, rdq, rdk, rdv = oracle.backward(f["q"], f["k"], f["v"], f["do"], False, d ** -0.5, block_mask=m)
    for a, r in zip((dq, dk, dv), (rdq, rdk, rdv)):
        assert rel_fro(a.float().cpu().numpy(), r) <= configs.TOL_GRAD_REL_FRO


def test_blocksparse_bwd_all_ones_equals_dense_dkdv(fa):
    """With every tile visible the block-sparse backward visits the same steps
    in the same order: dK and dV bit-identical to fa_bwd (dQ equal up to the
    order of its fp32 reductions)."""
    B, Hq, Hkv, N, d = 1, 4, 2, 700, 128
    t = inputs.make_inputs(B, Hq, Hkv, N, d, "bf16", seed=23, with_grad=True)
    dev = torch.device("cuda:0")
    g = {n: x.to(dev) for n, x in t.items()}
    T = (N + 127) // 128
    ones = torch.ones(1, 1, T, T, dtype=torch.uint8, device=dev)
    o, lse = fa.fwd(g["q"], g["k"], g["v"], causal=True)
    a = fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal=True, block_mask=ones)
    b = fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal=True)
    fa.check_device_status()
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    assert float((a[0].float() - b[0].float()).abs().max()) < 1e-2


def test_blocksparse_local_window_workload_sampled_rows(fa):
    """The block-sparse bench workload at full size (16 heads, N = 32768, a
    causal window of 16 key tiles, the mask broadcast over heads as bench.py
    passes it): 256 seeded query rows per head against the oracle."""
    w = configs.WORKLOADS["bf16_h16_n32768_d128_local16_fwdbwd"]
    t = inputs.make_workload_inputs(w, with_grad=False)
    m = w.block_mask()
    dev = torch.device("cuda:0")
    q, k, v = (t[n].to(dev) for n in ("q", "k", "v"))
    mt = torch.tensor(m, dtype=torch.uint8, device=dev)
    o, lse = fa.fwd(q, k, v, causal=True, scale=w.scale, block_mask=mt)
    fa.check_device_status()
    rows = inputs.sample_rows(w.B, w.Hq, w.N, 256, seed=1)
    f = {n: inputs.to_f64(t[n]) for n in ("q", "k", "v")}
    ro, rl = oracle.forward_rows(f["q"], f["k"], f["v"], True, w.scale, rows, block_mask=m)
    bi = np.arange(w.B)[:, None, None]
    hi = np.arange(w.Hq)[None, :, None]
    check_fwd(o.float().cpu().numpy()[bi, hi, rows], lse.cpu().numpy()[bi, hi, rows], ro, rl)


def test_blocksparse_local_window_workload_bwd_sampled_rows(fa):
    """The same workload's backward at full size: 256 seeded query rows per
    head of dQ and 256 seeded key rows per head of dK and dV against the
    oracle (LSE and D of every query row from the oracle itself, under the
    same block mask); two launches give bit-identical dK and dV. Key tiles are
    visited by at most 16 query tiles, so every dK/dV block has a short, varied
    step list."""
    w = configs.WORKLOADS["bf16_h16_n32768_d128_local16_fwdbwd"]
    t = inputs.make_workload_inputs(w, with_grad=True)
    dev = torch.device("cuda:0")
    g = {n: x.to(dev) for n, x in t.items()}
    m = w.block_mask()
    mt = torch.tensor(m, dtype=torch.uint8, device=dev)
    o, lse = fa.fwd(g["q"], g["k"], g["v"], causal=True, scale=w.scale, block_mask=mt)
    a = fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal=True, scale=w.scale, block_mask=mt)
    b = fa.bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal=True, scale=w.scale, block_mask=mt)
    fa.check_device_status()
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    assert float((a[0].float() - b[0].float()).abs().max()) < 1e-2
    f = {n: inputs.to_f64(t[n]) for n in ("q", "k", "v", "do")}
    rl_all, rD_all = oracle.row_statistics(f["q"], f["k"], f["v"], f["do"], True, w.scale, block_mask=m)
    assert np.abs(lse.cpu().numpy() - rl_all).max() <= configs.TOL_LSE_MAX
    rows = inputs.sample_rows(w.B, w.Hq, w.N, 256, seed=1)
    krows = inputs.sample_rows(w.B, w.Hkv, w.N, 256, seed=2)
    rdq, rdk, rdv = oracle.backward_rows(f["q"], f["k"], f["v"], f["do"], True, w.scale, rows, krows, rl_all, rD_all,
                                         block_mask=m)
    dq, dk, dv = (x.float().cpu().numpy() for x in a)
    assert all(np.isfinite(x).all() for x in (dq, dk, dv))
    bi = np.arange(w.B)[:, None, None]
    hi = np.arange(w.Hq)[None, :, None]
    hk = np.arange(w.Hkv)[None, :, None]
    errs = {"dq": rel_fro(dq[bi, hi, rows], rdq), "dk": rel_fro(dk[bi, hk, krows], rdk),
            "dv": rel_fro(dv[bi, hk, krows], rdv)}
    print(w.name, errs)
    assert max(errs.values()) <= configs.TOL_GRAD_REL_FRO, errs
