"""Pins for the double-precision oracle, checked against things other than
itself: torch's float64 scaled-dot-product attention and autograd (an
independent library routine for the same quantity), a pure-Python brute force
on tiny inputs, closed forms, invariants and central finite differences.

No GPU needed.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as oa


def rand_qkv(B, Hq, Hkv, N, d, seed, with_do=False, q_scale=1.0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, Hq, N, d)) * q_scale
    k = rng.standard_normal((B, Hkv, N, d))
    v = rng.standard_normal((B, Hkv, N, d))
    if with_do:
        return q, k, v, rng.standard_normal((B, Hq, N, d))
    return q, k, v


# ---------------------------------------------------------------- library routine

def torch_sdpa(q, k, v, causal, scale):
    """torch's float64 CPU attention (math path) with K/V heads expanded to the
    query heads, h -> h // G."""
    G = q.shape[1] // k.shape[1]
    qt = torch.from_numpy(q)
    kt = torch.from_numpy(k).repeat_interleave(G, dim=1)
    vt = torch.from_numpy(v).repeat_interleave(G, dim=1)
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=causal, scale=scale)


CASES = [
    # B, Hq, Hkv, N, d, causal
    (1, 1, 1, 1, 4, False),
    (1, 1, 1, 1, 4, True),
    (2, 4, 2, 7, 8, False),
    (2, 4, 2, 7, 8, True),
    (1, 8, 1, 33, 16, True),
    (1, 3, 3, 130, 16, False),
    (2, 2, 1, 129, 32, True),
]


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal", CASES)
def test_forward_matches_torch_sdpa(B, Hq, Hkv, N, d, causal):
    q, k, v = rand_qkv(B, Hq, Hkv, N, d, seed=N * 7 + d)
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle.forward(q, k, v, causal, scale)
    o_t = torch_sdpa(q, k, v, causal, scale).numpy()
    np.testing.assert_allclose(o, o_t, rtol=0, atol=1e-12)


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal", CASES)
def test_backward_matches_torch_autograd(B, Hq, Hkv, N, d, causal):
    q, k, v, do = rand_qkv(B, Hq, Hkv, N, d, seed=N * 11 + d, with_do=True)
    scale = 0.37
    o, lse, dq, dk, dv = oracle.backward(q, k, v, do, causal, scale)
    qt = torch.from_numpy(q).requires_grad_()
    kt = torch.from_numpy(k).requires_grad_()
    vt = torch.from_numpy(v).requires_grad_()
    G = Hq // Hkv
    ot = torch.nn.functional.scaled_dot_product_attention(
        qt, kt.repeat_interleave(G, 1), vt.repeat_interleave(G, 1), is_causal=causal, scale=scale)
    ot.backward(torch.from_numpy(do))
    np.testing.assert_allclose(o, ot.detach().numpy(), atol=1e-12, rtol=0)
    np.testing.assert_allclose(dq, qt.grad.numpy(), atol=1e-11, rtol=0)
    np.testing.assert_allclose(dk, kt.grad.numpy(), atol=1e-11, rtol=0)
    np.testing.assert_allclose(dv, vt.grad.numpy(), atol=1e-11, rtol=0)


# ---------------------------------------------------------------- pure-Python brute force

def brute_force(q, k, v, do, causal, scale):
    """Scalar loops, no numpy arithmetic: softmax row by row, then the chain
    rule element by element."""
    B, Hq, N, d = q.shape
    G = Hq // k.shape[1]
    o = [[[[0.0] * d for _ in range(N)] for _ in range(Hq)] for _ in range(B)]
    lse = [[[0.0] * N for _ in range(Hq)] for _ in range(B)]
    dq = [[[[0.0] * d for _ in range(N)] for _ in range(Hq)] for _ in range(B)]
    dk = [[[[0.0] * d for _ in range(N)] for _ in range(k.shape[1])] for _ in range(B)]
    dv = [[[[0.0] * d for _ in range(N)] for _ in range(k.shape[1])] for _ in range(B)]
    for b in range(B):
        for h in range(Hq):
            g = h // G
            for i in range(N):
                keys = [j for j in range(N) if (not causal or j <= i)]
                s = {j: scale * sum(float(q[b, h, i, c]) * float(k[b, g, j, c]) for c in range(d)) for j in keys}
                mx = max(s.values())
                tot = sum(math.exp(s[j] - mx) for j in keys)
                lse[b][h][i] = mx + math.log(tot)
                p = {j: math.exp(s[j] - lse[b][h][i]) for j in keys}
                for c in range(d):
                    o[b][h][i][c] = sum(p[j] * float(v[b, g, j, c]) for j in keys)
                Di = sum(float(do[b, h, i, c]) * o[b][h][i][c] for c in range(d))
                for j in keys:
                    dp = sum(float(do[b, h, i, c]) * float(v[b, g, j, c]) for c in range(d))
                    ds = p[j] * (dp - Di)
                    for c in range(d):
                        dq[b][h][i][c] += scale * ds * float(k[b, g, j, c])
                        dk[b][g][j][c] += scale * ds * float(q[b, h, i, c])
                        dv[b][g][j][c] += p[j] * float(do[b, h, i, c])
    return [np.array(x) for x in (o, lse, dq, dk, dv)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv,N,d", [(1, 1, 1, 3), (2, 1, 5, 3), (4, 2, 6, 4)])
def test_against_brute_force(causal, Hq, Hkv, N, d):
    q, k, v, do = rand_qkv(1, Hq, Hkv, N, d, seed=3 + N, with_do=True, q_scale=2.0)
    ref = brute_force(q, k, v, do, causal, 0.61)
    got = oracle.backward(q, k, v, do, causal, 0.61)
    for r, g in zip(ref, got):
        np.testing.assert_allclose(g, r, atol=1e-12, rtol=0)


# ---------------------------------------------------------------- finite differences

@pytest.mark.parametrize("causal", [False, True])
def test_gradients_by_finite_differences(causal):
    q, k, v, do = rand_qkv(1, 2, 1, 6, 3, seed=5, with_do=True)
    scale = 0.8
    _, _, dq, dk, dv = oracle.backward(q, k, v, do, causal, scale)

    def loss(qq, kk, vv):
        o, _ = oracle.forward(qq, kk, vv, causal, scale)
        return float((o * do).sum())

    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}; args_p[name] = xp
            args_m = {"q": q, "k": k, "v": v}; args_m[name] = xm
            num[idx] = (loss(args_p["q"], args_p["k"], args_p["v"]) - loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * h)
        np.testing.assert_allclose(g, num, atol=1e-7, rtol=1e-6, err_msg=name)


# ---------------------------------------------------------------- closed forms

def test_single_key_gives_that_value_row():
    q, k, v = rand_qkv(2, 4, 2, 1, 8, seed=9)
    o, lse = oracle.forward(q, k, v, False, 0.3)
    G = 2
    for h in range(4):
        np.testing.assert_allclose(o[:, h, 0], v[:, h // G, 0], atol=1e-15)
        np.testing.assert_allclose(lse[:, h, 0], 0.3 * (q[:, h, 0] * k[:, h // G, 0]).sum(-1), atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_is_uniform_average(causal):
    N = 23
    _, k, v = rand_qkv(1, 2, 2, N, 5, seed=4)
    q = np.zeros((1, 2, N, 5))
    o, lse = oracle.forward(q, k, v, causal, 1.0)
    if causal:
        ref = np.cumsum(v, axis=2) / np.arange(1, N + 1)[None, None, :, None]
        ref_lse = np.log(np.arange(1, N + 1))[None, None, :].repeat(2, 1)
    else:
        ref = np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape)
        ref_lse = np.full((1, 2, N), math.log(N))
    np.testing.assert_allclose(o, ref, atol=1e-14)
    np.testing.assert_allclose(lse, ref_lse, atol=1e-14)
    # dV for Q = 0 and dO: every visible query spreads dO_i uniformly over its keys
    do = np.random.default_rng(1).standard_normal(q.shape)
    _, _, _, _, dv = oracle.backward(q, k, v, do, causal, 1.0)
    ref_dv = np.zeros_like(v)
    for i in range(N):
        cnt = i + 1 if causal else N
        ref_dv[:, :, :cnt] += do[:, :, i:i + 1] / cnt
    np.testing.assert_allclose(dv, ref_dv, atol=1e-13)


def test_constant_value_rows():
    q, k, _ = rand_qkv(1, 3, 3, 17, 6, seed=2, q_scale=3.0)
    vrow = np.random.default_rng(0).standard_normal(6)
    v = np.broadcast_to(vrow, (1, 3, 17, 6)).copy()
    for causal in (False, True):
        o, _ = oracle.forward(q, k, v, causal, 0.5)
        np.testing.assert_allclose(o, np.broadcast_to(vrow, o.shape), atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_identity_values_expose_softmax_rows(causal):
    """With V = I (d = N) the output row is the probability row itself: it is
    non-negative, sums to 1, is zero above the diagonal when causal, and
    P_ij = exp(S_ij - LSE_i)."""
    N = 9
    rng = np.random.default_rng(8)
    q = rng.standard_normal((1, 1, N, N)) * 2
    k = rng.standard_normal((1, 1, N, N))
    v = np.eye(N)[None, None]
    o, lse = oracle.forward(q, k, v, causal, 0.7)
    P = o[0, 0]
    assert (P >= 0).all()
    np.testing.assert_allclose(P.sum(axis=1), 1.0, atol=1e-14)
    if causal:
        assert np.all(np.triu(P, 1) == 0)
    S = 0.7 * q[0, 0] @ k[0, 0].T
    mask = np.tril(np.ones((N, N), bool)) if causal else np.ones((N, N), bool)
    np.testing.assert_allclose(P[mask], np.exp(S - lse[0, 0][:, None])[mask], atol=1e-14)


def test_one_hot_dominant_logit_selects_value_row():
    N, d = 8, 8
    k = np.eye(N)[None, None, :, :d]          # orthonormal keys
    v = np.random.default_rng(3).standard_normal((1, 1, N, d))
    q = np.zeros((1, 1, N, d))
    target = [5, 0, 7, 2, 2, 1, 6, 3]
    for i, j in enumerate(target):
        q[0, 0, i] = 30.0 * k[0, 0, j]
    o, lse = oracle.forward(q, k, v, False, 1.0)
    for i, j in enumerate(target):
        np.testing.assert_allclose(o[0, 0, i], v[0, 0, j], atol=1e-11)
        np.testing.assert_allclose(lse[0, 0, i], 30.0, atol=1e-11)


def test_key_permutation_invariance_non_causal():
    q, k, v, do = rand_qkv(1, 2, 1, 31, 8, seed=12, with_do=True)
    perm = np.random.default_rng(5).permutation(31)
    o1, l1, dq1, dk1, dv1 = oracle.backward(q, k, v, do, False, 0.35)
    o2, l2, dq2, dk2, dv2 = oracle.backward(q, k[:, :, perm], v[:, :, perm], do, False, 0.35)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)
    np.testing.assert_allclose(dq1, dq2, atol=1e-13)
    np.testing.assert_allclose(dk1[:, :, perm], dk2, atol=1e-13)
    np.testing.assert_allclose(dv1[:, :, perm], dv2, atol=1e-13)


def test_causal_first_row_and_last_row():
    """Row 0 sees only key 0; the last row sees every key, so it equals the
    non-causal result."""
    q, k, v = rand_qkv(1, 2, 2, 14, 4, seed=21)
    oc, lc = oracle.forward(q, k, v, True, 0.5)
    on, ln = oracle.forward(q, k, v, False, 0.5)
    np.testing.assert_allclose(oc[:, :, 0], v[:, :, 0], atol=1e-15)
    np.testing.assert_allclose(oc[:, :, -1], on[:, :, -1], atol=1e-14)
    np.testing.assert_allclose(lc[:, :, -1], ln[:, :, -1], atol=1e-14)


def test_gqa_equals_mha_with_replicated_kv():
    q, k, v, do = rand_qkv(2, 6, 2, 19, 8, seed=17, with_do=True)
    G = 3
    kr = np.repeat(k, G, axis=1)
    vr = np.repeat(v, G, axis=1)
    for causal in (False, True):
        g = oracle.backward(q, k, v, do, causal, 0.4)
        m = oracle.backward(q, kr, vr, do, causal, 0.4)
        for a, b in zip(g[:3], m[:3]):
            np.testing.assert_allclose(a, b, atol=1e-13)
        np.testing.assert_allclose(g[3], m[3].reshape(2, 2, G, 19, 8).sum(2), atol=1e-12)
        np.testing.assert_allclose(g[4], m[4].reshape(2, 2, G, 19, 8).sum(2), atol=1e-12)


def test_scale_acts_on_logits_only():
    q, k, v = rand_qkv(1, 1, 1, 12, 4, seed=30)
    o1, l1 = oracle.forward(q, k, v, True, 0.25)
    o2, l2 = oracle.forward(q * 0.25, k, v, True, 1.0)
    np.testing.assert_allclose(o1, o2, atol=1e-14)
    np.testing.assert_allclose(l1, l2, atol=1e-14)


# ---------------------------------------------------------------- sampled-row modes

@pytest.mark.parametrize("causal", [False, True])
def test_row_modes_equal_full_computation(causal):
    B, Hq, Hkv, N, d = 1, 4, 2, 97, 8
    q, k, v, do = rand_qkv(B, Hq, Hkv, N, d, seed=40, with_do=True)
    s = 0.3
    o, lse, dq, dk, dv = oracle.backward(q, k, v, do, causal, s)
    rng = np.random.default_rng(0)
    qr = np.stack([np.stack([np.sort(rng.choice(N, 11, replace=False)) for _ in range(Hq)])])
    kr = np.stack([np.stack([np.sort(rng.choice(N, 13, replace=False)) for _ in range(Hkv)])])
    o_r, lse_r = oracle.forward_rows(q, k, v, causal, s, qr)
    for h in range(Hq):
        np.testing.assert_allclose(o_r[0, h], o[0, h, qr[0, h]], atol=1e-13)
        np.testing.assert_allclose(lse_r[0, h], lse[0, h, qr[0, h]], atol=1e-13)
    lse_s, D_s = oracle.row_statistics(q, k, v, do, causal, s, block=16, threads=2)
    np.testing.assert_allclose(lse_s, lse, atol=1e-13)
    np.testing.assert_allclose(D_s, (do * o).sum(-1), atol=1e-13)
    dq_r, dk_r, dv_r = oracle.backward_rows(q, k, v, do, causal, s, qr, kr, lse_s, D_s)
    for h in range(Hq):
        np.testing.assert_allclose(dq_r[0, h], dq[0, h, qr[0, h]], atol=1e-12)
    for g in range(Hkv):
        np.testing.assert_allclose(dk_r[0, g], dk[0, g, kr[0, g]], atol=1e-12)
        np.testing.assert_allclose(dv_r[0, g], dv[0, g, kr[0, g]], atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_query_row_slabs_sum_to_full_backward(causal):
    B, Hq, Hkv, N, d = 1, 4, 2, 50, 8
    q, k, v, do = rand_qkv(B, Hq, Hkv, N, d, seed=44, with_do=True)
    o, lse, dq, dk, dv = oracle.backward(q, k, v, do, causal, 0.3)
    dk_sum = np.zeros_like(dk)
    dv_sum = np.zeros_like(dv)
    for h in range(Hq):
        for rows in (np.arange(0, 17), np.arange(17, 40), np.arange(40, 50)):
            o_r, l_r, D_r, dq_r, dk_p, dv_p = oracle.backward_query_rows(q, k, v, do, causal, 0.3, 0, h, rows)
            np.testing.assert_allclose(o_r, o[0, h, rows], atol=1e-13)
            np.testing.assert_allclose(l_r, lse[0, h, rows], atol=1e-13)
            np.testing.assert_allclose(D_r, (do[0, h, rows] * o[0, h, rows]).sum(-1), atol=1e-13)
            np.testing.assert_allclose(dq_r, dq[0, h, rows], atol=1e-12)
            dk_sum[0, h // 2] += dk_p
            dv_sum[0, h // 2] += dv_p
    np.testing.assert_allclose(dk_sum, dk, atol=1e-12)
    np.testing.assert_allclose(dv_sum, dv, atol=1e-12)


# ---------------------------------------------------------------- the pages' tiled algorithm

@pytest.mark.parametrize("deferred", [False, True])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,block", [(1, 4), (13, 4), (64, 16), (130, 64)])
def test_tiled_online_softmax_equals_definition(deferred, causal, N, block):
    q, k, v = rand_qkv(1, 4, 2, N, 8, seed=N, q_scale=4.0)
    o, lse = oracle.forward(q, k, v, causal, 0.35)
    ot, lt = oracle.tiled_forward(q, k, v, causal, 0.35, block=block, deferred=deferred)
    np.testing.assert_allclose(ot, o, atol=1e-12)
    np.testing.assert_allclose(lt, lse, atol=1e-12)


# ---------------------------------------------------------------- the pins catch planted mistakes

def _planted(monkeypatch, kind):
    real_scores = oa._scores
    real_softmax = oa._softmax_rows
    if kind == "drop_scale":
        monkeypatch.setattr(oa, "_scores", lambda qh, kh, s, c, r, bm=None, off=0: real_scores(qh, kh, 1.0, c, r, bm,
                                                                                               off))
    elif kind == "block_mask_transposed":
        monkeypatch.setattr(oa, "_scores", lambda qh, kh, s, c, r, bm=None, off=0: real_scores(
            qh, kh, s, c, r, None if bm is None else np.swapaxes(bm, 0, 1), off))
    elif kind == "causal_top_left":
        monkeypatch.setattr(oa, "_scores", lambda qh, kh, s, c, r, bm=None, off=0: real_scores(qh, kh, s, c, r, bm, 0))
    elif kind == "mask_strict":
        def f(qh, kh, s, causal, r, bm=None, off=0):
            out = s * (qh @ kh.T)
            if causal:
                out = np.where(np.arange(kh.shape[0])[None, :] < r[:, None], out, -np.inf)
                out[:, 0] = np.where(r == 0, s * (qh @ kh[0]), out[:, 0])
            return out
        monkeypatch.setattr(oa, "_scores", f)
    elif kind == "lse_log2":
        def g(s):
            p, lse = real_softmax(s)
            return p, lse / math.log(2)
        monkeypatch.setattr(oa, "_softmax_rows", g)
    elif kind == "no_max_shift":
        def g(s):
            m = s.max(axis=1)
            e = np.exp(s - m[:, None])
            lse = np.log(e.sum(axis=1))          # forgets to add the max back
            return np.exp(s - m[:, None] - lse[:, None]), lse
        monkeypatch.setattr(oa, "_softmax_rows", g)


@pytest.mark.parametrize("kind", ["drop_scale", "mask_strict", "lse_log2", "no_max_shift", "block_mask_transposed",
                                  "causal_top_left"])
def test_pins_fail_on_planted_mistakes(monkeypatch, kind):
    """Each planted mistake must break at least one of the pins above."""
    _planted(monkeypatch, kind)
    failures = 0
    checks = [
        lambda: test_forward_matches_torch_sdpa(2, 4, 2, 7, 8, True),
        lambda: test_against_brute_force(True, 2, 1, 5, 3),
        lambda: test_single_key_gives_that_value_row(),
        lambda: test_zero_query_is_uniform_average(True),
        lambda: test_block_mask_matches_torch_sdpa(False),
        lambda: test_kv_length_matches_torch_sdpa(200, 300, True),
    ]
    for c in checks:
        try:
            c()
        except AssertionError:
            failures += 1
    assert failures >= 1, kind


def test_transposed_operand_would_be_caught():
    """Using K^T Q (scores transposed) instead of Q K^T differs from torch."""
    q, k, v = rand_qkv(1, 1, 1, 6, 6, seed=77)
    o_t = torch_sdpa(q, k, v, True, 0.5).numpy()
    s_wrong = 0.5 * (k[0, 0] @ q[0, 0].T)
    s_wrong = np.where(np.tril(np.ones((6, 6), bool)), s_wrong, -np.inf)
    p = np.exp(s_wrong - s_wrong.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    assert np.abs(p @ v[0, 0] - o_t[0, 0]).max() > 1e-3
    o, _ = oracle.forward(q, k, v, True, 0.5)
    np.testing.assert_allclose(o, o_t, atol=1e-12)


# ---------------------------------------------------------------- block masks
def _block_mask(B, Hq, n, density, seed):
    """Random block mask with the diagonal block always on, so every query row
    sees at least one key (its own) and torch's masked softmax stays finite."""
    rng = np.random.Generator(np.random.PCG64(seed))
    m = rng.random((B, Hq, n, n)) < density
    m[..., np.arange(n), np.arange(n)] = True
    return m


def _expand(block_mask, N):
    bm = np.repeat(np.repeat(block_mask, oa.BLOCK, axis=-2), oa.BLOCK, axis=-1)
    return bm[..., :N, :N]


@pytest.mark.parametrize("causal", [False, True])
def test_block_mask_all_ones_is_dense(causal):
    """An all-true block mask changes nothing, bit for bit."""
    q, k, v, do = rand_qkv(1, 2, 1, 300, 8, seed=41, with_do=True)
    n = 3
    ones = np.ones((1, 2, n, n), dtype=bool)
    a = oa.backward(q, k, v, do, causal, 0.3)
    b = oa.backward(q, k, v, do, causal, 0.3, block_mask=ones)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("causal", [False, True])
def test_block_mask_matches_torch_sdpa(causal):
    """Forward and gradients against torch float64 scaled_dot_product_attention
    with the same mask expanded to elements (AND the causal mask), an
    independent library routine; rows of 300 keys span three blocks, the last
    one ragged, and the mask is not symmetric."""
    B, Hq, Hkv, N, d = 1, 4, 2, 300, 8
    q, k, v, do = rand_qkv(B, Hq, Hkv, N, d, seed=43, with_do=True)
    bm = _block_mask(B, Hq, 3, 0.5, seed=44)
    assert not np.array_equal(bm, np.swapaxes(bm, -1, -2))
    o, lse, dq, dk, dv = oa.backward(q, k, v, do, causal, 0.25, block_mask=bm)
    allowed = _expand(bm, N)
    if causal:
        allowed = allowed & np.tril(np.ones((N, N), dtype=bool))
    G = Hq // Hkv
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    kk = tk.repeat_interleave(G, dim=1)
    vv = tv.repeat_interleave(G, dim=1)
    to = torch.nn.functional.scaled_dot_product_attention(tq, kk, vv, attn_mask=torch.tensor(allowed), scale=0.25)
    to.backward(torch.tensor(do))
    s = 0.25 * torch.einsum("bhid,bhjd->bhij", tq.detach(), kk.detach())
    s = s.masked_fill(~torch.tensor(allowed), float("-inf"))
    tlse = torch.logsumexp(s, dim=-1)
    np.testing.assert_allclose(o, to.detach().numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, tlse.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-9, atol=1e-11)


def test_block_mask_empty_rows():
    """A query block with no visible key block: its rows give O = 0,
    LSE = -inf and dQ = 0, and they add nothing to dK, dV; so dK, dV equal
    those of the unmasked problem with those rows' dO set to zero (then
    dP = 0, D = 0 and dS = 0 for them)."""
    B, Hq, Hkv, N, d = 1, 2, 2, 384, 8
    q, k, v, do = rand_qkv(B, Hq, Hkv, N, d, seed=45, with_do=True)
    bm = np.ones((B, Hq, 3, 3), dtype=bool)
    bm[:, 0, 1, :] = False                      # head 0, query block 1 sees nothing
    o, lse, dq, dk, dv = oa.backward(q, k, v, do, False, 0.3, block_mask=bm)
    rows = slice(128, 256)
    assert np.all(o[:, 0, rows] == 0) and np.all(np.isneginf(lse[:, 0, rows])) and np.all(dq[:, 0, rows] == 0)
    do0 = do.copy()
    do0[:, 0, rows] = 0
    _, _, dq_ref, dk_ref, dv_ref = oa.backward(q, k, v, do0, False, 0.3)
    np.testing.assert_allclose(dk, dk_ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dv, dv_ref, rtol=1e-12, atol=1e-13)
    other = [r for r in range(N) if not 128 <= r < 256]
    np.testing.assert_allclose(dq[:, 0, other], dq_ref[:, 0, other], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dq[:, 1], dq_ref[:, 1], rtol=1e-12, atol=1e-13)


def test_block_mask_rows_mode_matches_full():
    """forward_rows with a block mask gives the same rows as forward."""
    B, Hq, Hkv, N, d = 1, 2, 1, 300, 8
    q, k, v = rand_qkv(B, Hq, Hkv, N, d, seed=47)
    bm = _block_mask(B, Hq, 3, 0.5, seed=48)
    o, lse = oa.forward(q, k, v, True, 0.2, block_mask=bm)
    rows = np.array([[[0, 5, 130, 299]] * Hq])
    ro, rl = oa.forward_rows(q, k, v, True, 0.2, rows, block_mask=bm)
    for h in range(Hq):
        np.testing.assert_array_equal(ro[0, h], o[0, h, rows[0, h]])
        np.testing.assert_array_equal(rl[0, h], lse[0, h, rows[0, h]])


# ---------------------------------------------------------------- Nq != Nk
@pytest.mark.parametrize("Nq,Nk,causal", [(200, 300, True), (200, 300, False), (300, 200, True), (1, 257, True)])
def test_kv_length_matches_torch_sdpa(Nq, Nk, causal):
    """Queries as the last Nq of Nk positions (bottom-right causal): forward,
    LSE and gradients against torch float64 scaled_dot_product_attention with
    the explicit element mask j <= i + Nk - Nq. Rows that see no key (Nq > Nk)
    are compared to the oracle's convention O = 0, LSE = -inf, dQ = 0."""
    B, Hq, Hkv, d = 1, 4, 2, 8
    rng = np.random.default_rng(Nq * 1000 + Nk)
    q = rng.standard_normal((B, Hq, Nq, d))
    k = rng.standard_normal((B, Hkv, Nk, d))
    v = rng.standard_normal((B, Hkv, Nk, d))
    do = rng.standard_normal((B, Hq, Nq, d))
    o, lse, dq, dk, dv = oa.backward(q, k, v, do, causal, 0.3)
    allowed = np.ones((Nq, Nk), dtype=bool)
    if causal:
        allowed = np.arange(Nk)[None, :] <= np.arange(Nq)[:, None] + (Nk - Nq)
    seen = allowed.any(axis=1)
    G = Hq // Hkv
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    kk = tk.repeat_interleave(G, dim=1)
    vv = tv.repeat_interleave(G, dim=1)
    am = torch.tensor(allowed)
    am_safe = am | torch.tensor(~seen)[:, None]          # keep torch finite on rows that see nothing
    to = torch.nn.functional.scaled_dot_product_attention(tq, kk, vv, attn_mask=am_safe, scale=0.3)
    to = to * torch.tensor(seen, dtype=to.dtype)[:, None]
    to.backward(torch.tensor(do))
    np.testing.assert_allclose(o, to.detach().numpy(), rtol=1e-10, atol=1e-12)
    s = 0.3 * torch.einsum("bhid,bhjd->bhij", tq.detach(), kk.detach()).masked_fill(~am, float("-inf"))
    tl = torch.logsumexp(s, dim=-1).numpy()
    np.testing.assert_allclose(lse[..., seen], tl[..., seen], rtol=1e-10, atol=1e-12)
    assert np.all(np.isneginf(lse[..., ~seen])) and np.all(dq[:, :, ~seen] == 0)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-9, atol=1e-11)


def test_single_query_decoding_sees_every_key():
    """One query at the end of Nk keys, causal, sees all of them: the same as
    the non-causal result (a closed form of the bottom-right rule)."""
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 2, 1, 8))
    k = rng.standard_normal((1, 2, 77, 8))
    v = rng.standard_normal((1, 2, 77, 8))
    a = oa.forward(q, k, v, True, 0.5)
    b = oa.forward(q, k, v, False, 0.5)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_kv_length_rows_mode_matches_full():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((1, 2, 150, 8))
    k = rng.standard_normal((1, 1, 400, 8))
    v = rng.standard_normal((1, 1, 400, 8))
    o, lse = oa.forward(q, k, v, True, 0.4)
    rows = np.array([[[0, 7, 149]] * 2])
    ro, rl = oa.forward_rows(q, k, v, True, 0.4, rows)
    for h in range(2):
        np.testing.assert_array_equal(ro[0, h], o[0, h, rows[0, h]])
        np.testing.assert_array_equal(rl[0, h], lse[0, h, rows[0, h]])


# ---------------------------------------------------------------- row modes with Nq != Nk and block masks
@pytest.mark.parametrize("Nq,Nk,causal", [(150, 400, True), (300, 130, True), (1, 257, True), (120, 333, False)])
def test_kv_length_row_statistics_and_backward_rows_match_full(Nq, Nk, causal):
    """The sampled-row modes with keys longer (or shorter) than queries equal
    the full `backward`, itself pinned against torch above; rows that see no
    key (Nq > Nk, causal) have LSE = -inf, D = 0 and dQ = 0."""
    B, Hq, Hkv, d = 1, 4, 2, 8
    rng = np.random.default_rng(Nq * 31 + Nk)
    q = rng.standard_normal((B, Hq, Nq, d))
    k = rng.standard_normal((B, Hkv, Nk, d))
    v = rng.standard_normal((B, Hkv, Nk, d))
    do = rng.standard_normal((B, Hq, Nq, d))
    o, lse, dq, dk, dv = oa.backward(q, k, v, do, causal, 0.35)
    lse_s, D_s = oa.row_statistics(q, k, v, do, causal, 0.35, block=64, threads=2)
    seen = np.isfinite(lse)
    assert np.array_equal(np.isfinite(lse_s), seen)
    np.testing.assert_allclose(lse_s[seen], lse[seen], atol=1e-13)
    np.testing.assert_allclose(D_s, (do * o).sum(-1), atol=1e-13)
    assert np.all(D_s[~seen] == 0)
    qr = np.stack([np.stack([np.sort(rng.choice(Nq, min(Nq, 9), replace=False)) for _ in range(Hq)])])
    kr = np.stack([np.stack([np.sort(rng.choice(Nk, 11, replace=False)) for _ in range(Hkv)])])
    if Nq > Nk and causal:
        qr[0, 0, 0] = 0                        # a row that sees no key
    dq_r, dk_r, dv_r = oa.backward_rows(q, k, v, do, causal, 0.35, qr, kr, lse_s, D_s)
    for h in range(Hq):
        np.testing.assert_allclose(dq_r[0, h], dq[0, h, qr[0, h]], atol=1e-12)
    for g in range(Hkv):
        np.testing.assert_allclose(dk_r[0, g], dk[0, g, kr[0, g]], atol=1e-12)
        np.testing.assert_allclose(dv_r[0, g], dv[0, g, kr[0, g]], atol=1e-12)
    if Nq > Nk and causal:
        assert np.all(dq_r[0, 0, 0] == 0)


@pytest.mark.parametrize("causal", [False, True])
def test_block_mask_row_statistics_and_backward_rows_match_full(causal):
    """The same for a block mask (pinned against torch above), including a
    query tile that sees no key tile and a local-window mask whose slabs span
    several tiles."""
    B, Hq, Hkv, N, d = 1, 4, 2, 520, 8
    q, k, v, do = rand_qkv(B, Hq, Hkv, N, d, seed=61, with_do=True)
    T = 5
    bm = _block_mask(B, Hq, T, 0.6, seed=62)
    bm[:, 1, 2, :] = False                     # head 1, query tile 2 sees nothing
    i, j = np.arange(T)[:, None], np.arange(T)[None, :]
    bm[:, 3] = (j <= i) & (j > i - 2)          # head 3: a window of two tiles
    o, lse, dq, dk, dv = oa.backward(q, k, v, do, causal, 0.3, block_mask=bm)
    lse_s, D_s = oa.row_statistics(q, k, v, do, causal, 0.3, block=200, threads=2, block_mask=bm)
    seen = np.isfinite(lse)
    assert (~seen).any() and np.array_equal(np.isfinite(lse_s), seen)
    np.testing.assert_allclose(lse_s[seen], lse[seen], atol=1e-13)
    np.testing.assert_allclose(D_s, (do * o).sum(-1), atol=1e-13)
    rng = np.random.default_rng(63)
    qr = np.stack([np.stack([np.sort(rng.choice(N, 12, replace=False)) for _ in range(Hq)])])
    qr[0, 1, 0] = 300                          # head 1, inside the empty query tile
    qr[0, 1] = np.sort(qr[0, 1])
    kr = np.stack([np.stack([np.sort(rng.choice(N, 14, replace=False)) for _ in range(Hkv)])])
    dq_r, dk_r, dv_r = oa.backward_rows(q, k, v, do, causal, 0.3, qr, kr, lse_s, D_s, block_mask=bm)
    for h in range(Hq):
        np.testing.assert_allclose(dq_r[0, h], dq[0, h, qr[0, h]], atol=1e-12)
    for g in range(Hkv):
        np.testing.assert_allclose(dk_r[0, g], dk[0, g, kr[0, g]], atol=1e-12)
        np.testing.assert_allclose(dv_r[0, g], dv[0, g, kr[0, g]], atol=1e-12)
