"""fa_fwd_pair: the forward computed by clusters of two CTAs with tcgen05
cta_group::2 products (csrc/fa_fwd_pair.cu), through the C ABI.

It must match the double-precision oracle within the forward's tolerances and
give fa_fwd_kv's bits (every row's products and softmax are the same
operations in the same order), including clusters whose second query tile
pair is partly or wholly past the last row, tiles that see no key, ragged
key tails and head dimensions below 128. Unsupported forms are refused before
any launch. A stalled issuer times out and the context stays usable."""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from exact_attention_79_gb300 import configs, inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def P(t):
    return ctypes.c_void_p(t.data_ptr())


def run_pair(lib, q, k, v, causal, scale):
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, Hq, Nq), float("nan"), dtype=torch.float32, device=DEV)
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.fa_fwd_pair(P(q), P(k), P(v), P(o), P(lse), B, Hq, Hkv, Nq, Nk, d, int(causal), scale, s)
    return rc, o, lse


def run_kv(lib, q, k, v, causal, scale):
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=DEV)
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.fa_fwd_kv(P(q), P(k), P(v), P(o), P(lse), B, Hq, Hkv, Nq, Nk, d, int(causal), scale, s) == 0
    return o, lse


CASES = [
    # B, Hq, Hkv, Nq, Nk, d, causal
    (1, 2, 2, 128, 128, 128, True),      # one query tile: the cluster's other three are absent
    (1, 2, 1, 640, 640, 128, True),      # five tiles: the second cluster holds one
    (2, 4, 2, 333, 333, 128, False),     # ragged rows and keys
    (1, 8, 1, 1000, 1000, 128, True),    # GQA, eight tiles, ragged last
    (1, 4, 2, 300, 1000, 128, True),     # queries at the end of longer keys
    (1, 2, 2, 500, 200, 128, True),      # more queries than keys: the first rows see nothing
    (1, 3, 3, 700, 700, 96, True),       # d below 128: zero-filled columns
    (2, 2, 2, 1, 777, 128, True),        # one decoding query
    (1, 2, 2, 1, 1, 128, False),
]


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal", CASES)
def test_pair_forward_matches_oracle_and_fa_fwd_kv(fa, B, Hq, Hkv, Nq, Nk, d, causal):
    lib = fa.load()
    scale = d ** -0.5
    t = inputs.make_inputs(B, Hq, Hkv, Nq, d, "bf16", seed=Nq + 3 * Nk + d, Nk=Nk)
    q, k, v = (t[n].to(DEV) for n in ("q", "k", "v"))
    rc, o, lse = run_pair(lib, q, k, v, causal, scale)
    assert rc == 0, rc
    fa.check_device_status()
    o2, lse2 = run_kv(lib, q, k, v, causal, scale)
    fa.check_device_status()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    f = {n: inputs.to_f64(t[n]) for n in ("q", "k", "v")}
    ro, rl = oracle.forward(f["q"], f["k"], f["v"], causal, scale)
    on, ln = o.float().cpu().numpy(), lse.cpu().numpy()
    seen = np.isfinite(rl)
    assert np.all(on[~seen] == 0) and np.all(np.isneginf(ln[~seen]))
    err = np.abs(on - ro)
    assert err.max() <= configs.TOL_O_MAX and err.mean() <= configs.TOL_O_MEAN
    assert np.abs(ln[seen] - rl[seen]).max() <= configs.TOL_LSE_MAX


@pytest.mark.parametrize("name", ["bf16_h16_n8192_d128_causal_fwdbwd", "bf16_gqa_b2_h64kv8_n4096_d128_causal"])
def test_pair_forward_full_size(fa, name):
    """The benchmark workloads: fa_fwd's bits, and 256 seeded rows per head
    against the oracle."""
    lib = fa.load()
    w = configs.WORKLOADS[name]
    t = inputs.make_workload_inputs(w, with_grad=False)
    q, k, v = (t[n].to(DEV) for n in ("q", "k", "v"))
    rc, o, lse = run_pair(lib, q, k, v, w.causal, w.scale)
    assert rc == 0
    o2, lse2 = fa.fwd(q, k, v, causal=w.causal, scale=w.scale)
    fa.check_device_status()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    rows = inputs.sample_rows(w.B, w.Hq, w.N, 256, seed=1)
    f = {n: inputs.to_f64(t[n]) for n in ("q", "k", "v")}
    ro, rl = oracle.forward_rows(f["q"], f["k"], f["v"], w.causal, w.scale, rows)
    bi, hi = np.arange(w.B)[:, None, None], np.arange(w.Hq)[None, :, None]
    err = np.abs(o.float().cpu().numpy()[bi, hi, rows] - ro)
    assert err.max() <= configs.TOL_O_MAX and err.mean() <= configs.TOL_O_MEAN
    assert np.abs(lse.cpu().numpy()[bi, hi, rows] - rl).max() <= configs.TOL_LSE_MAX


@pytest.mark.parametrize("d", [64, 136, 256])
def test_pair_forward_refuses_other_head_dims(fa, d):
    lib = fa.load()
    x = torch.zeros(1, 1, 128, d, dtype=torch.bfloat16, device=DEV)
    rc, _, _ = run_pair(lib, x, x, x, True, 0.1)
    assert rc == 2        # FA_ERR_UNSUPPORTED, nothing launched
    fa.check_device_status()


CHILD = r'''
import ctypes, os, sys, time
sys.path.insert(0, ROOT)
import torch
import exact_attention_79_gb300 as fa
from exact_attention_79_gb300 import inputs
lib = fa.load()
dev = torch.device("cuda:0")
t = inputs.make_inputs(1, 2, 2, 600, 128, "bf16", seed=5)
q, k, v = (t[n].to(dev) for n in ("q", "k", "v"))
s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
P = lambda x: ctypes.c_void_p(x.data_ptr())
def call():
    o = torch.empty_like(q)
    l = torch.empty(1, 2, 600, dtype=torch.float32, device=dev)
    assert lib.fa_fwd_pair(P(q), P(k), P(v), P(o), P(l), 1, 2, 2, 600, 600, 128, 1, 128 ** -0.5, s) == 0
    return o, l
ref = call()
assert lib.fa_device_status(s) == 0
os.environ["FA_TEST_STALL"] = "1"
t0 = time.time()
call()
assert lib.fa_device_status(s) == 5 and time.time() - t0 >= 0.25
os.environ["FA_TEST_STALL"] = "0"
again = call()
assert lib.fa_device_status(s) == 0
assert torch.equal(again[0], ref[0]) and torch.equal(again[1], ref[1])
print("pair-timeout-ok")
'''


def test_pair_forward_timeout_path():
    """FA_TEST_STALL: the even CTA's issuer waits on a barrier nothing arrives
    on; both CTAs of every cluster unwind, the call reports FA_ERR_TIMEOUT and
    the next call gives the same bits as before."""
    env = dict(os.environ, FA_WAIT_LIMIT_MS="300", FA_TEST_STALL="0")
    r = subprocess.run([sys.executable, "-c", "ROOT = %r\n" % ROOT + CHILD], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and "pair-timeout-ok" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]
