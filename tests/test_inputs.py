"""The seeded input generator: deterministic, correctly shaped, rounded to
the storage type."""
import numpy as np
import torch

from exact_attention_79_gb300 import configs, inputs


def test_deterministic_and_shaped():
    a = inputs.make_inputs(2, 4, 2, 33, 16, "bf16", seed=0, with_grad=True)
    b = inputs.make_inputs(2, 4, 2, 33, 16, "bf16", seed=0, with_grad=True)
    for key in ("q", "k", "v", "do"):
        assert torch.equal(a[key], b[key])
        assert a[key].dtype == torch.bfloat16
    assert a["q"].shape == (2, 4, 33, 16) and a["do"].shape == (2, 4, 33, 16)
    assert a["k"].shape == (2, 2, 33, 16) and a["v"].shape == (2, 2, 33, 16)
    c = inputs.make_inputs(2, 4, 2, 33, 16, "bf16", seed=1)
    assert not torch.equal(a["q"], c["q"])


def test_q_multiplier_is_exact_power_of_two():
    a = inputs.make_inputs(1, 2, 2, 40, 8, "bf16", seed=3)
    b = inputs.make_inputs(1, 2, 2, 40, 8, "bf16", seed=3, q_mult=4.0)
    assert torch.equal(a["q"].float() * 4, b["q"].float())
    assert torch.equal(a["k"], b["k"])


def test_fp32_workload_and_standard_normal():
    w = configs.WORKLOADS["fp32_h1_n128_d64"]
    t = inputs.make_workload_inputs(w)
    assert t["q"].dtype == torch.float32 and "do" not in t
    big = inputs.make_inputs(1, 1, 1, 4096, 64, "fp32", seed=0)["q"].numpy()
    assert abs(big.mean()) < 0.01 and abs(big.std() - 1) < 0.01


def test_sampled_rows_distinct_sorted():
    r = inputs.sample_rows(1, 8, 65536, 256, seed=1)
    assert r.shape == (1, 8, 256)
    for h in range(8):
        assert np.all(np.diff(r[0, h]) > 0) and r[0, h].min() >= 0 and r[0, h].max() < 65536


def test_flop_counts():
    w = configs.WORKLOADS["bf16_h16_n8192_d128_causal_fwdbwd"]
    assert w.flops_fwd == 4 * 16 * 8192 ** 2 * 128 / 2
    assert w.flops_bwd == 2.5 * w.flops_fwd
