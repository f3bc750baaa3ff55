"""Failure detection on the GPU without any fault: with FA_TEST_STALL=1 the
tensor-core issuer (of the forward kernels: d <= 128, wide-head, FP8 at d = 128
and 256; of the backward's dK/dV pass; and of the three passes of the
backward above d = 128) first waits on a barrier nothing arrives on, so its
bounded wait (FA_WAIT_LIMIT_MS, here 300 ms) runs out; every other role of
the block sees the abort flag and unwinds, the block stores nothing and the
call reports FA_ERR_TIMEOUT through fa_device_status. The next call on the
same context must be correct, and a stall on one stream must not be reported
to a call on another.  Runs in a child process because the wait
limit is read once per process."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import ctypes, os, sys, time
sys.path.insert(0, ROOT)
import numpy as np, torch
import exact_attention_79_gb300 as fa
import oracle
from exact_attention_79_gb300 import configs, inputs
lib = fa.load()
dev = torch.device("cuda:0")
stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
t = inputs.make_inputs(1, 2, 2, 300, 128, "bf16", seed=1, with_grad=True)
g = {n: x.to(dev) for n, x in t.items()}
f = {n: inputs.to_f64(x) for n, x in t.items()}
ro, rl, rdq, rdk, rdv = oracle.backward(f["q"], f["k"], f["v"], f["do"], True, 128 ** -0.5)

def run(stall, what):
    os.environ["FA_TEST_STALL"] = "1" if stall else "0"
    t0 = time.time()
    if what == "fwd":
        out = fa.fwd(g["q"], g["k"], g["v"], causal=True)
    else:
        out = fa.bwd(g["q"], g["k"], g["v"], o_ok, lse_ok, g["do"], causal=True)
    code = lib.fa_device_status(stream)
    return out, code, time.time() - t0

out, code, dt = run(True, "fwd")
assert code == 5 and dt >= 0.25, (code, dt)                      # FA_ERR_TIMEOUT after the 300 ms limit
(o_ok, lse_ok), code, _ = run(False, "fwd")
assert code == 0
assert np.abs(o_ok.float().cpu().numpy() - ro).max() <= configs.TOL_O_MAX
out, code, dt = run(True, "bwd")
assert code == 5 and dt >= 0.25, (code, dt)
(dq, dk, dv), code, _ = run(False, "bwd")
assert code == 0
for a, r in zip((dq, dk, dv), (rdq, rdk, rdv)):
    a = a.float().cpu().numpy()
    assert np.linalg.norm(a - r) / np.linalg.norm(r) <= configs.TOL_GRAD_REL_FRO

# the wide-head forward (d = 256) and the FP8 forwards (d = 128, 256) take the same path
tw = inputs.make_inputs(1, 2, 2, 300, 256, "bf16", seed=2)
gw = {n: x.to(dev) for n, x in tw.items()}
q8, qs, k8, ks, vt8, vs = fa.quantize_fp8(g["q"], g["k"], g["v"])
w8 = fa.quantize_fp8(gw["q"], gw["k"], gw["v"])
os.environ["FA_TEST_STALL"] = "0"
refs = {"wide": fa.fwd(gw["q"], gw["k"], gw["v"], causal=True),
        "fp8": fa.fwd_fp8(q8, qs, k8, ks, vt8, vs, causal=True),
        "fp8_wide": fa.fwd_fp8(*w8, causal=True)}
assert lib.fa_device_status(stream) == 0
for name, call in (("wide", lambda: fa.fwd(gw["q"], gw["k"], gw["v"], causal=True)),
                   ("fp8", lambda: fa.fwd_fp8(q8, qs, k8, ks, vt8, vs, causal=True)),
                   ("fp8_wide", lambda: fa.fwd_fp8(*w8, causal=True))):
    os.environ["FA_TEST_STALL"] = "1"
    t0 = time.time()
    call()
    code = lib.fa_device_status(stream)
    assert code == 5 and time.time() - t0 >= 0.25, (name, code)
    os.environ["FA_TEST_STALL"] = "0"
    again = call()
    assert lib.fa_device_status(stream) == 0, name
    ref = refs[name]
    assert torch.equal(again[0], ref[0]) and torch.equal(again[1], ref[1]), name
# the backward above d = 128 (three passes, each issuer stalls) takes the same path
tb = inputs.make_inputs(1, 2, 2, 300, 256, "bf16", seed=3, with_grad=True)
gb = {n: x.to(dev) for n, x in tb.items()}
os.environ["FA_TEST_STALL"] = "0"
ob, lb = fa.fwd(gb["q"], gb["k"], gb["v"], causal=True)
ref_b = fa.bwd(gb["q"], gb["k"], gb["v"], ob, lb, gb["do"], causal=True)
assert lib.fa_device_status(stream) == 0
os.environ["FA_TEST_STALL"] = "1"
t0 = time.time()
fa.bwd(gb["q"], gb["k"], gb["v"], ob, lb, gb["do"], causal=True)
assert lib.fa_device_status(stream) == 5 and time.time() - t0 >= 0.25
os.environ["FA_TEST_STALL"] = "0"
again_b = fa.bwd(gb["q"], gb["k"], gb["v"], ob, lb, gb["do"], causal=True)
assert lib.fa_device_status(stream) == 0
assert all(torch.equal(x, y) for x, y in zip(again_b, ref_b))

# status words are per stream: a stall on one stream is reported to that
# stream only, while a call on another stream, overlapping it, reports FA_OK
sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
ha, hb = ctypes.c_void_p(sa.cuda_stream), ctypes.c_void_p(sb.cuda_stream)
torch.cuda.synchronize()
os.environ["FA_TEST_STALL"] = "1"
with torch.cuda.stream(sa):
    fa.fwd(g["q"], g["k"], g["v"], causal=True)
os.environ["FA_TEST_STALL"] = "0"
with torch.cuda.stream(sb):
    o_b, lse_b = fa.fwd(g["q"], g["k"], g["v"], causal=True)
t0 = time.time()
assert lib.fa_device_status(hb) == 0
assert torch.equal(o_b, o_ok) and torch.equal(lse_b, lse_ok)
assert lib.fa_device_status(ha) == 5
assert lib.fa_device_status(ha) == 0             # read and cleared
assert lib.fa_device_status(stream) == 0
print("timeout-path-ok")
'''


def test_bounded_wait_runs_out_and_context_stays_usable():
    env = dict(os.environ, FA_WAIT_LIMIT_MS="300", FA_TEST_STALL="0")
    r = subprocess.run([sys.executable, "-c", "ROOT = %r\n" % ROOT + CHILD], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0 and "timeout-path-ok" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]
