"""The worked example in tests/golden/two_keys.txt: one head, two query rows,
two keys, d = 8, integer inputs (exact in bf16), scale 1/2.

The stored outputs were written by tests/golden/make_golden.py from the
oracle. Here they are pinned to mathematics that shares nothing with the
oracle's code: the softmax rows and logsumexps in closed form (logits 0, 1
and 0, 2), the causal first row equal to V_0, and the gradients by central
differences of <O, dO> computed with scalar math. The GPU test runs the CUDA
forward and backward on the same inputs through the C ABI.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "two_keys.txt")


def load():
    rows = {}
    scale = None
    with open(GOLDEN) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            name, *vals = line.split()
            if name == "scale":
                scale = float(vals[0])
                continue
            rows.setdefault(name, []).append([float(x) for x in vals])
    g = {n: np.asarray(r) for n, r in rows.items()}
    for n in list(g):
        if n.endswith(".lse"):
            g[n] = g[n].reshape(-1)
    return scale, g


def attention_by_hand(q, k, v, scale, causal):
    """O and LSE with scalar math: for each row, the visible logits, their
    largest, the exponentials, the sum, the weighted values."""
    n, d = len(q), len(q[0])
    o = [[0.0] * d for _ in range(n)]
    lse = [0.0] * n
    for i in range(n):
        keys = range(i + 1) if causal else range(len(k))
        s = [scale * sum(q[i][c] * k[j][c] for c in range(d)) for j in keys]
        m = max(s)
        w = [math.exp(x - m) for x in s]
        tot = sum(w)
        lse[i] = m + math.log(tot)
        for j, wj in zip(keys, w):
            for c in range(d):
                o[i][c] += wj / tot * v[j][c]
    return o, lse


def test_softmax_rows_in_closed_form():
    scale, g = load()
    e = math.e
    p0 = [1 / (1 + e), e / (1 + e)]                 # query 0: logits 0 and 1
    p1 = [1 / (1 + e * e), e * e / (1 + e * e)]     # query 1: logits 0 and 2
    v = g["v"]
    np.testing.assert_allclose(g["full.o"][0], p0[0] * v[0] + p0[1] * v[1], rtol=0, atol=1e-14)
    np.testing.assert_allclose(g["full.o"][1], p1[0] * v[0] + p1[1] * v[1], rtol=0, atol=1e-14)
    np.testing.assert_allclose(g["full.lse"], [math.log(1 + e), math.log(1 + e * e)], rtol=0, atol=1e-14)
    # causal: query 0 sees key 0 only, query 1 both
    np.testing.assert_array_equal(g["causal.o"][0], v[0])
    assert g["causal.lse"][0] == 0.0
    np.testing.assert_allclose(g["causal.o"][1], g["full.o"][1], rtol=0, atol=1e-15)
    assert scale == 0.5


@pytest.mark.parametrize("causal", [False, True])
def test_stored_values_by_scalar_math(causal):
    scale, g = load()
    tag = "causal" if causal else "full"
    o, lse = attention_by_hand(g["q"].tolist(), g["k"].tolist(), g["v"].tolist(), scale, causal)
    np.testing.assert_allclose(g[f"{tag}.o"], o, rtol=0, atol=1e-13)
    np.testing.assert_allclose(g[f"{tag}.lse"], lse, rtol=0, atol=1e-13)

    # gradients of L = <O, dO> by central differences, each input entry in turn
    do = g["do"]

    def loss(q, k, v):
        oo, _ = attention_by_hand(q, k, v, scale, causal)
        return float((np.asarray(oo) * do).sum())

    h = 1e-6
    base = {"q": g["q"], "k": g["k"], "v": g["v"]}
    for name in ("q", "k", "v"):
        grad = np.zeros_like(base[name])
        for idx in np.ndindex(grad.shape):
            args = {n: a.copy() for n, a in base.items()}
            args[name][idx] += h
            up = loss(args["q"].tolist(), args["k"].tolist(), args["v"].tolist())
            args[name][idx] -= 2 * h
            dn = loss(args["q"].tolist(), args["k"].tolist(), args["v"].tolist())
            grad[idx] = (up - dn) / (2 * h)
        np.testing.assert_allclose(g[f"{tag}.d{name}"], grad, rtol=0, atol=2e-8, err_msg=f"{tag} d{name}")


def test_oracle_reproduces_the_file():
    scale, g = load()
    q, k, v, do = (g[n].reshape(1, 1, 2, 8) for n in ("q", "k", "v", "do"))
    for causal in (False, True):
        tag = "causal" if causal else "full"
        o, lse, dq, dk, dv = oracle.backward(q, k, v, do, causal, scale)
        for name, a in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
            np.testing.assert_array_equal(a[0, 0], g[f"{tag}.{name}"], err_msg=f"{tag}.{name}")


@pytest.mark.gpu
@pytest.mark.parametrize("causal", [False, True])
def test_cuda_path_on_the_worked_example(fa, causal):
    """bf16 inputs are exact. O carries two bf16 roundings: P before P V and
    O itself at the end (each at most 2^-9 relative); LSE is fp32; the
    gradients carry the rounding of P, dS and the stored O to bf16."""
    scale, g = load()
    tag = "causal" if causal else "full"
    dev = torch.device("cuda:0")
    q, k, v, do = (torch.tensor(g[n], dtype=torch.bfloat16, device=dev).reshape(1, 1, 2, 8)
                   for n in ("q", "k", "v", "do"))
    o, lse = fa.fwd(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = fa.bwd(q, k, v, o, lse, do, causal=causal, scale=scale)
    fa.check_device_status()
    ref_o = g[f"{tag}.o"]
    got_o = o.float().cpu().numpy()[0, 0]
    assert np.all(np.abs(got_o - ref_o) <= 2.0 ** -7 * np.abs(ref_o) + 1e-6), (got_o, ref_o)
    np.testing.assert_allclose(lse.cpu().numpy()[0, 0], g[f"{tag}.lse"], rtol=0, atol=1e-5)
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        got = t.float().cpu().numpy()[0, 0]
        ref = g[f"{tag}.{name}"]
        np.testing.assert_allclose(got, ref, rtol=0, atol=2e-2 * max(1.0, np.abs(ref).max()), err_msg=name)
