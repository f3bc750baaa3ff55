"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no attention arithmetic: it only draws numbers and rounds
them to the storage type. Both the CUDA path and the oracle read its output.

Recipe: numpy's PCG64 generator (bit-identical on x86 and Arm), seed given per
call (0 by default), standard normal float32 drawn in the order Q, K, V, dO
with shapes Q, dO [B,Hq,N,d] and K, V [B,Hkv,N,d]. Q is multiplied by the
workload's q_mult (a power of two, so exact) before rounding. bf16 workloads
round each value to nearest-even bfloat16. Sampled row indices use separate
generators (seed 1 for query rows, seed 2 for key rows), one draw without
replacement per head in head order.
"""
import numpy as np
import torch

_TORCH_DTYPE = {"bf16": torch.bfloat16, "fp32": torch.float32}


def _normal(rng, shape):
    return rng.standard_normal(size=shape, dtype=np.float32)


def make_inputs(B, Hq, Hkv, N, d, dtype="bf16", seed=0, q_mult=1.0, with_grad=False, Nk=None):
    """Return a dict of CPU torch tensors q, k, v (and do when with_grad) in the
    storage dtype ("bf16" or "fp32"). Nk: positions of k and v (default N)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    tdt = _TORCH_DTYPE[dtype]
    Nk = N if Nk is None else Nk
    q = _normal(rng, (B, Hq, N, d))
    if q_mult != 1.0:
        q *= np.float32(q_mult)
    out = {"q": torch.from_numpy(q).to(tdt)}
    out["k"] = torch.from_numpy(_normal(rng, (B, Hkv, Nk, d))).to(tdt)
    out["v"] = torch.from_numpy(_normal(rng, (B, Hkv, Nk, d))).to(tdt)
    if with_grad:
        out["do"] = torch.from_numpy(_normal(rng, (B, Hq, N, d))).to(tdt)
    return out


def make_workload_inputs(w, seed=0, with_grad=None):
    """Inputs for a configs.Workload."""
    if with_grad is None:
        with_grad = w.backward
    storage = "bf16" if w.dtype == "fp8e4m3" else w.dtype      # fp8 inputs start as bf16 and are quantised
    return make_inputs(w.B, w.Hq, w.Hkv, w.N, w.d, storage, seed, w.q_mult, with_grad, Nk=(w.Nk or None))


def sample_rows(B, H, N, count, seed):
    """[B, H, count] distinct row indices per head, sorted per head."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = np.empty((B, H, min(count, N)), dtype=np.int64)
    for b in range(B):
        for h in range(H):
            out[b, h] = np.sort(rng.choice(N, size=out.shape[2], replace=False))
    return out


def to_f64(t):
    """Exact upcast of a CPU torch tensor to a float64 numpy array."""
    return t.to(torch.float64).numpy()
