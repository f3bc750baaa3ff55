"""The N > 1 path of bench.py on CPU: replicas share no data, so the only
cross-rank logic is the max-over-ranks timing and the whole-job value; two
gloo ranks on 127.0.0.1 exercise it. The reference arm's non-zero ranks
must exit without doing work."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out_path):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [120.0, 250.0][rank]                 # rank 1 is the slow replica
    slowest = bench.max_over_ranks(local_ms, world)
    value = bench.whole_job_tflops(world, 1e12, 10, slowest)
    dist.barrier()
    with open(f"{out_path}.{rank}", "w") as f:
        json.dump({"slowest": slowest, "value": value}, f)
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_replica(tmp_path):
    port = _free_port()
    out = str(tmp_path / "r")
    mp.start_processes(_rank, args=(2, port, out), nprocs=2, start_method="spawn", join=True)
    res = [json.load(open(f"{out}.{r}")) for r in range(2)]
    assert res[0] == res[1]
    assert res[0]["slowest"] == 250.0
    # 2 replicas x 10 steps x 1 TFLOP over 0.25 s
    assert abs(res[0]["value"] - 80.0) < 1e-9


def test_single_rank_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_tflops(1, 2e12, 4, 1000.0) == 8.0


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_exp_roofline_and_percentiles_arithmetic():
    """The exponential ceiling counts one ex2 per visible (query, key) pair,
    flops_fwd / (4 d) of them (4 d floating-point operations per pair); the
    step spread is nearest-rank."""
    sys.path.insert(0, ROOT)
    import bench
    from exact_attention_79_gb300 import configs
    w = configs.WORKLOADS["bf16_h16_n8192_d128_causal_fwdbwd"]
    r = bench.exp_roofline(w, 8.0, 152, 2000.0, 0.5, "fwd_kernel")
    exps = w.flops_fwd / (4 * 128)
    assert abs(r["exps_per_launch"] - exps) < 1e-6 * exps
    assert abs(r["peak"] - 8.0 * 152 * 2000e6 / 1e9) < 1e-9
    assert abs(r["achieved"] - exps / 0.5e-3 / 1e9) < 1e-6 * r["achieved"]
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-12
    assert bench.exp_roofline(w, 8.0, 152, None, 0.5, "fwd_kernel") is None
    p = bench.percentiles([5.0, 1.0, 3.0, 2.0, 4.0, 6.0, 7.0, 8.0, 9.0, 10.0, 11.0])
    assert p == {"p10": 2.0, "p50": 6.0, "p90": 10.0}
    assert bench.percentiles([]) is None


def test_reference_arm_line_on_cpu():
    """Rank 0 of the reference arm runs the oracle on the host and prints one
    JSON line with the contract's keys; its e2e moves no bytes."""
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["config"]["workload"] == "bf16_h16_n8192_d128_causal_fwdbwd"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["e2e"]["value"] == line["value"]


def test_clock_summary_rules():
    """Fewer than three nvidia-smi samples inside the timed window are never
    reported as the timed clock; the kernels' own clock wins when given; any
    throttle reason seen during the run is listed."""
    sys.path.insert(0, ROOT)
    import bench
    cs = bench.ClockSampler.__new__(bench.ClockSampler)
    row = lambda mhz, slow="Not Active", cap="Not Active": ["ts", str(mhz), "2070", "900", "0x0", slow, "Not Active",
                                                           "Not Active", cap]
    cs.rows = [(0.5, row(2070)), (1.5, row(1900, cap="Active")), (2.5, row(1950)), (9.0, row(2070))]
    out = cs.summary(1.0, 2.0)                      # one sample inside
    assert out["in_window"] == 1 and "smi_sm_mhz_in_window" not in out and out["sm_mhz"] is None
    assert out["reasons"] == ["sw_power_cap"] and out["sm_max_mhz"] == 2070.0
    out = cs.summary(1.0, 2.0, kernel_mhz=1923.0)
    assert out["sm_mhz"] == 1923.0 and "timed kernels" in out["sm_mhz_source"]
    cs.rows += [(1.6, row(1910)), (1.7, row(1920, slow="Active"))]
    out = cs.summary(1.0, 2.0)                      # three inside
    assert out["smi_sm_mhz_in_window"] == 1910.0 and out["sm_mhz"] == 1910.0
    assert out["reasons"] == ["hw_slowdown", "sw_power_cap"]
