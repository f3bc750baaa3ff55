"""The library's calls inside a CUDA graph: fa_fwd and fa_bwd_deterministic
captured once on a stream and replayed, with new contents in the same input
buffers between replays, give the bits of the same calls made directly.

The calls are capturable: every launch parameter (tensor maps included) is
passed by value, the library allocates nothing during a call, and the
per-device set-up it does once (architecture check, status-word address) is
done by an ordinary call before the capture. The workspace comes from
torch's allocator, which serves a capture from the graph's own pool.
"""
import pytest
import torch

from exact_attention_79_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d,causal", [(128, True), (64, False), (256, True)])
def test_graph_replay_matches_direct_calls(fa, d, causal):
    B, Hq, Hkv, N = 1, 4, 2, 1000
    dev = torch.device("cuda:0")
    first = {k: v.to(dev) for k, v in inputs.make_inputs(B, Hq, Hkv, N, d, "bf16", seed=71, with_grad=True).items()}
    second = {k: v.to(dev) for k, v in inputs.make_inputs(B, Hq, Hkv, N, d, "bf16", seed=72, with_grad=True).items()}

    def step(t):
        o, lse = fa.fwd(t["q"], t["k"], t["v"], causal=causal)
        dq, dk, dv = fa.bwd(t["q"], t["k"], t["v"], o, lse, t["do"], causal=causal, deterministic=True)
        return o, lse, dq, dk, dv

    # direct calls (these also do the library's one-time set-up on this device)
    want_first = [x.clone() for x in step(first)]
    want_second = [x.clone() for x in step(second)]
    torch.cuda.synchronize()
    fa.check_device_status()

    static = {k: v.clone() for k, v in first.items()}
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(static)                     # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        outs = step(static)

    for src, want in ((first, want_first), (second, want_second), (first, want_first)):
        for k in static:
            static[k].copy_(src[k])
        graph.replay()
        torch.cuda.synchronize()
        for name, got, ref in zip(("o", "lse", "dq", "dk", "dv"), outs, want):
            assert torch.equal(got, ref), name
    fa.check_device_status()
