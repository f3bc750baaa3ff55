"""Independent calls at the same time: two host threads, each on its own CUDA
stream, run forward + deterministic backward on different problems (and the
forward at d = 256 on a third stream) while the others run. Each result has
the bits of the same call made alone, and every stream reports FA_OK.
The library keeps no state shared between calls beyond the per-stream status
words and the clock accumulator, which the results never read."""
import threading

import pytest
import torch

from exact_attention_79_gb300 import inputs

pytestmark = pytest.mark.gpu

PROBLEMS = [
    # B, Hq, Hkv, N, d, causal, backward
    (1, 8, 2, 2000, 128, True, True),
    (2, 4, 4, 777, 64, False, True),
    (1, 4, 1, 1500, 256, True, False),
]


def _run(fa, t, causal, backward, stream):
    with torch.cuda.stream(stream):
        o, lse = fa.fwd(t["q"], t["k"], t["v"], causal=causal)
        outs = [o, lse]
        if backward:
            outs += list(fa.bwd(t["q"], t["k"], t["v"], o, lse, t["do"], causal=causal, deterministic=True))
    return outs


def test_concurrent_streams_and_threads_match_solo_runs(fa):
    dev = torch.device("cuda:0")
    data = []
    for n, (B, Hq, Hkv, N, d, causal, backward) in enumerate(PROBLEMS):
        t = inputs.make_inputs(B, Hq, Hkv, N, d, "bf16", seed=900 + n, with_grad=True)
        data.append(({k: v.to(dev) for k, v in t.items()}, causal, backward))

    solo = []
    for t, causal, backward in data:
        solo.append([x.clone() for x in _run(fa, t, causal, backward, torch.cuda.current_stream())])
        torch.cuda.synchronize()
    fa.check_device_status()

    streams = [torch.cuda.Stream() for _ in data]
    results = [None] * len(data)
    errors = []

    def worker(n):
        try:
            for _ in range(3):                      # overlap several rounds of each problem
                t, causal, backward = data[n]
                results[n] = _run(fa, t, causal, backward, streams[n])
        except Exception as e:                      # reported below, in the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(n,)) for n in range(len(data))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for n, s in enumerate(streams):
        fa.check_device_status(s.cuda_stream)
        for got, want in zip(results[n], solo[n]):
            assert torch.equal(got, want), n
