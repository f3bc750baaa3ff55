#!/usr/bin/env python3
"""Attention throughput on GB300: forward + backward TFLOP/s (bf16, d=128).

One step = one pass of the whole path over one batch: fa_fwd, then the three
backward phases (fa_bwd_preprocess, fa_bwd_dkdv, fa_bwd_dq), all through the
C ABI. FLOPs are counted as 4 B Hq N^2 d for the forward (halved when causal)
and 2.5x that for the backward. Prints one JSON line. A workload without a
backward (configs.Workload.backward false) times the forward call alone.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl native|reference]

--impl reference times the double-precision CPU oracle on the host cores on
the same workload and metric, each step a bounded slab of query rows.
Multi-GPU (torchrun): independent replicas, one per rank; value = all ranks'
FLOPs over the slowest rank's time.
"""
import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "bf16_h16_n8192_d128_causal_fwdbwd"
METRIC = "attention TFLOPS fwd+bwd (bf16, d=128) and % of GB300 dense BF16 peak"
FALLBACK_PEAK_TFLOPS = 1900.0     # used only when MEASURED_PEAKS.json is absent
L2_FLUSH_BYTES = 256 << 20


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--e2e-sets", type=int, default=3, help="device buffer sets the end-to-end pipeline rotates over")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="budget of the oracle CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--bwd", choices=["fused", "deterministic"], default="fused",
                    help="backward timed: fa_bwd's three phases (default) or fa_bwd_deterministic")
    ap.add_argument("--fwd", choices=["single", "pair"], default="single",
                    help="dense bf16 forward timed: fa_fwd (default) or fa_fwd_pair (CTA pairs, cta_group::2)")
    return ap.parse_args()


def metric_for(w):
    if w.backward:
        return METRIC
    peak = "FP8" if w.dtype == "fp8e4m3" else "BF16"
    return f"attention TFLOPS fwd ({w.dtype}, d={w.d}) and % of GB300 dense {peak} peak"


def peak_tflops(dtype="bf16"):
    """Dense tensor peak for the workload's arithmetic: the measured bf16 burst
    figure; e4m3 takes it times the nominal fp8 : bf16 dense ratio (4.5 : 2.25)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            peak, src = float(json.load(f)["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    except Exception:
        peak, src = FALLBACK_PEAK_TFLOPS, "fallback 1.9 PFLOP/s (MEASURED_PEAKS.json absent)"
    if dtype == "fp8e4m3":
        return 2.0 * peak, src + " x 2 (nominal e4m3 / bf16 dense ratio)"
    return peak, src


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.rows = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_id), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1, kernel_mhz=None):
        """Clock record of the timed region. nvidia-smi samples every 50 ms,
        so a short timed region holds few samples: its median SM clock is
        reported only from samples inside the window (at least 3), else under
        smi_sm_mhz_out_of_window. sm_mhz is the clock the timed kernels
        measured themselves (fa_sm_clock_mhz) when available. Throttle
        reasons are those seen in any sample of the run."""
        inside = [r for t, r in self.rows if t0 <= t <= t1 and len(r) >= 9]
        every = [r for _, r in self.rows if len(r) >= 9]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        def median_sm(rows):
            sm = sorted(v for v in (num(r[1]) for r in rows) if v is not None)
            return sm[len(sm) // 2] if sm else None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in every for i in range(4) if r[5 + i].lower().startswith("active")})
        mx = [v for v in (num(r[2]) for r in every) if v is not None]
        out = {"sm_max_mhz": max(mx) if mx else None, "reasons": reasons if every else ["unavailable"],
               "samples": len(every), "in_window": len(inside)}
        if len(inside) >= 3:
            out["smi_sm_mhz_in_window"] = median_sm(inside)
        else:
            out["smi_sm_mhz_out_of_window"] = median_sm(every)
        if kernel_mhz:
            out["sm_mhz"] = kernel_mhz
            out["sm_mhz_source"] = "timed kernels themselves (fa_sm_clock_mhz: SM cycles / ns over every CTA)"
        else:
            out["sm_mhz"] = out.get("smi_sm_mhz_in_window")
            out["sm_mhz_source"] = "nvidia-smi samples inside the timed region" if out["sm_mhz"] else None
        return out


def clock_rated_peak(dtype, n_sms, mhz):
    """Dense tensor rate at the given SM clock: 4096 bf16 multiply-adds per
    SM per clock (8192 FLOP; measured for every MMA form the kernels use),
    twice that for e4m3, half for tf32. TFLOP/s, or None without a clock."""
    if not mhz:
        return None
    per_clk = {"fp8e4m3": 16384.0, "fp32": 4096.0}.get(dtype, 8192.0)
    return n_sms * per_clk * mhz * 1e6 / 1e12


# ------------------------------------------------------------------ oracle timing
def oracle_rows_flops(rows, N, d, causal):
    """Algorithmic fwd+bwd FLOPs of the given query rows: 14 d per visible key
    (4 d of them the forward's)."""
    import numpy as np
    keys = (np.asarray(rows) + 1) if causal else np.full(len(rows), N)
    return 14.0 * d * float(keys.sum())


def oracle_slab_runner(w, seed=0):
    """Returns (run(rows) -> flops, np): the oracle's full forward + backward
    arithmetic (the forward alone for a workload without a backward) for a
    slab of query rows of head (0, 0)."""
    import numpy as np
    import oracle
    from exact_attention_79_gb300 import inputs
    t = inputs.make_inputs(1, 1, 1, w.N, w.d, "bf16" if w.dtype == "fp8e4m3" else w.dtype, seed=seed,
                           with_grad=w.backward)
    f = {k: inputs.to_f64(v) for k, v in t.items()}
    if w.dtype == "fp8e4m3":
        # the oracle's attention of the dequantised e4m3 inputs (quantised once, outside the timing)
        from oracle import fp8 as ofp8
        qc, qs = ofp8.quantize_rows(f["q"])
        kc, ks = ofp8.quantize_rows(f["k"])
        vc, vs = ofp8.quantize_v_transposed(f["v"])
        f = {"q": ofp8.dequantize_rows(qc, qs), "k": ofp8.dequantize_rows(kc, ks),
             "v": ofp8.dequantize_v_transposed(vc, vs, w.N)}

    def run(rows):
        if not w.backward:
            oracle.forward_rows(f["q"], f["k"], f["v"], w.causal, w.scale, np.asarray(rows)[None, None])
            return oracle_rows_flops(rows, w.N, w.d, w.causal) * 4.0 / 14.0
        oracle.backward_query_rows(f["q"], f["k"], f["v"], f["do"], w.causal, w.scale, 0, 0, rows)
        return oracle_rows_flops(rows, w.N, w.d, w.causal)
    return run, np


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def cpu_baseline(w, budget_s):
    """The oracle as it stands, on host cores, over seeded random query rows of
    one head until the time budget is spent."""
    run, np = oracle_slab_runner(w)
    rng = np.random.Generator(np.random.PCG64(7))
    flops = 0.0
    nrows = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < budget_s:
        rows = np.sort(rng.choice(w.N, size=min(128, w.N), replace=False))
        flops += run(rows)
        nrows += len(rows)
    dt = time.perf_counter() - t0
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"{nrows} seeded query rows of head 0 (full {'fwd+bwd' if w.backward else 'forward'} "
                      f"arithmetic per row, fp64), {dt:.1f} s"}


def reference_arm(args, w):
    """The oracle timed on the host cores, K steps after W warm-up steps; each
    step a slab of query rows sized so the whole run takes a few minutes."""
    run, np = oracle_slab_runner(w)
    rng = np.random.Generator(np.random.PCG64(11))
    probe_rows = np.sort(rng.choice(w.N, size=min(64, w.N), replace=False))
    t0 = time.perf_counter()
    run(probe_rows)
    per_row = (time.perf_counter() - t0) / len(probe_rows)
    budget = 150.0
    R = int(max(1, min(w.N, budget / max(1, args.steps + args.warmup) / max(per_row, 1e-9))))
    for _ in range(args.warmup):
        run(np.sort(rng.choice(w.N, size=R, replace=False)))
    flops = 0.0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        flops += run(np.sort(rng.choice(w.N, size=R, replace=False)))
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    line = {
        "impl": "reference", "metric": metric_for(w), "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, **{k: v for k, v in w.describe().items() if k != "workload"},
                   "sample_rows_per_step": R},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"{R} seeded query rows of head 0 per step (full "
                                   f"{'fwd+bwd' if w.backward else 'forward'} arithmetic, fp64)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ traffic from a committed ncu summary
def traffic_from_profile(kernel_file, kernel_name, workload):
    """dram bytes per launch from profiles/<kernel>__<workload>.md, if that
    summary was taken on the current kernel source (its sha256 matches)."""
    path = os.path.join(ROOT, "profiles", f"{kernel_name}__{workload}.md")
    src = os.path.join(ROOT, "exact_attention_79_gb300", "csrc", kernel_file)
    try:
        text = open(path).read()
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith(("kernel_source_sha256", "dram_bytes_per_launch")):
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha256") != sha:
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------------ exponential ceiling, step spread
def exp_roofline(w, ex2_per_cycle_per_sm, n_sms, sm_mhz, fwd_ms, kernel):
    """The forward kernel against the exponential unit: one ex2 per visible
    (query, key) pair, flops_fwd / (4 d) of them, over the ex2 rate measured
    on this GPU (fa_ex2_throughput) at the SM clock sampled under load. None
    when the clock or the rate is unknown."""
    if not sm_mhz or not ex2_per_cycle_per_sm or ex2_per_cycle_per_sm <= 0 or fwd_ms <= 0:
        return None
    exps = w.flops_fwd / (4.0 * w.d)
    peak = ex2_per_cycle_per_sm * n_sms * sm_mhz * 1e6 / 1e9
    achieved = exps / (fwd_ms / 1e3) / 1e9
    return {"bound": "exp", "achieved": achieved, "peak": peak, "unit": "Gexp/s", "frac": achieved / peak,
            "kernel": kernel, "exps_per_launch": exps, "ex2_per_cycle_per_sm": ex2_per_cycle_per_sm,
            "n_sms": n_sms, "sm_mhz": sm_mhz}


def percentiles(xs):
    """p10, p50, p90 of a list of step times (nearest rank)."""
    v = sorted(xs)
    if not v:
        return None
    pick = lambda q: v[min(len(v) - 1, int(round(q * (len(v) - 1))))]  # noqa: E731
    return {"p10": pick(0.1), "p50": pick(0.5), "p90": pick(0.9)}


# ------------------------------------------------------------------ replicas across ranks
def max_over_ranks(x, world):
    """The largest of every rank's x (one float); x itself on a single rank.
    The replicas share no data; this is the only collective of the bench."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world, flops_per_step, steps, slowest_total_ms):
    """Work of all replicas (each did `steps` steps of `flops_per_step`) over
    the slowest replica's time (weak scaling)."""
    return world * flops_per_step * steps / (slowest_total_ms / 1e3) / 1e12


# ------------------------------------------------------------------ native arm
def native_arm(args, w):
    import ctypes

    import torch
    import torch.distributed as dist

    import exact_attention_79_gb300 as fa
    from exact_attention_79_gb300 import inputs

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lib = fa.load()

    fwd_only = not w.backward
    t = inputs.make_workload_inputs(w, with_grad=not fwd_only)
    q, k, v = (t[n].to(dev) for n in ("q", "k", "v"))
    do = None if fwd_only else t["do"].to(dev)
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.Hq, w.N, dtype=torch.float32, device=dev)
    dq, dk, dv = (None, None, None) if fwd_only else (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    sparse = bool(w.block_window)
    kvlen = bool(w.Nk)
    ws_bytes = (0 if fwd_only else
                int(lib.fa_bwd_blocksparse_workspace_bytes(w.B, w.Hq, w.Hkv, w.N, w.d)) if sparse
                else fa.bwd_workspace_bytes(w.B, w.Hq, w.Hkv, w.N, w.d))
    mask = torch.tensor(w.block_mask(), dtype=torch.uint8, device=dev) if sparse else None
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sptr = ctypes.c_void_p(stream.cuda_stream)
    P = lambda x: ctypes.c_void_p(x.data_ptr())  # noqa: E731
    dims = (w.B, w.Hq, w.Hkv, w.N, w.d)
    causal = int(w.causal)
    scale = float(w.scale)

    def check(name, code):
        if code != 0:
            raise RuntimeError(f"{name} failed with status {code}")

    det = args.bwd == "deterministic"
    if (sparse or kvlen) and det:
        raise SystemExit("the deterministic backward has no block-sparse or unequal-length form")
    if fwd_only and (sparse or kvlen or det):
        raise SystemExit("forward-only workloads are dense with equal lengths")
    fwd_name = "fa_fwd" if w.dtype == "bf16" else "fa_fwd_f32"
    pair_fwd = args.fwd == "pair"
    if pair_fwd and (w.dtype != "bf16" or not 64 < w.d <= 128 or sparse or kvlen):
        raise SystemExit("fa_fwd_pair: dense bf16 workloads with 64 < d <= 128 only")
    fp8 = w.dtype == "fp8e4m3"
    if fp8:
        # e4m3 codes and scales, resident before the timed region
        q8, qs, k8, ks, vt8, vs = fa.quantize_fp8(q, k, v)
        torch.cuda.synchronize(dev)

    class Bufs:
        """Device tensors of one step of the path."""

    main = Bufs()
    main.__dict__.update(q=q, k=k, v=v, do=do, o=o, lse=lse, dq=dq, dk=dk, dv=dv)
    if fp8:
        main.__dict__.update(q8=q8, qs=qs, k8=k8, ks=ks, vt8=vt8, vs=vs)

    def run(b, sp, mark, quantize=False):
        """The path's library calls for one step on buffers b and stream sp;
        mark(i) is called at the points the per-kernel events sit (0 before
        the forward, 1 after it, 2-4 after the three backward phases)."""
        def marks(first):
            for i in range(first, 5):
                mark(i)
        if fp8:
            if quantize:
                # the user's whole job from bf16 inputs: quantise, then attention
                check("fa_fp8_quantize_rows", lib.fa_fp8_quantize_rows(P(b.q), P(b.q8), P(b.qs), w.B * w.Hq, w.N,
                                                                       w.d, sp))
                check("fa_fp8_quantize_rows", lib.fa_fp8_quantize_rows(P(b.k), P(b.k8), P(b.ks), w.B * w.Hkv, w.N,
                                                                       w.d, sp))
                check("fa_fp8_quantize_v", lib.fa_fp8_quantize_v(P(b.v), P(b.vt8), P(b.vs), w.B * w.Hkv, w.N, w.d,
                                                                 sp))
            mark(0)
            check("fa_fwd_fp8", lib.fa_fwd_fp8(P(b.q8), P(b.qs), P(b.k8), P(b.ks), P(b.vt8), P(b.vs), P(b.o),
                                               P(b.lse), *dims, causal, scale, sp))
            return marks(1)
        if fwd_only:
            mark(0)
            if pair_fwd:
                check("fa_fwd_pair", lib.fa_fwd_pair(P(b.q), P(b.k), P(b.v), P(b.o), P(b.lse), w.B, w.Hq, w.Hkv, w.N,
                                                     w.N, w.d, causal, scale, sp))
            else:
                check(fwd_name, getattr(lib, fwd_name)(P(b.q), P(b.k), P(b.v), P(b.o), P(b.lse), *dims, causal, scale,
                                                       sp))
            return marks(1)
        if kvlen:
            # queries are the last N of Nk positions (fa_fwd_kv / fa_bwd_kv)
            mark(0)
            check("fa_fwd_kv", lib.fa_fwd_kv(P(b.q), P(b.k), P(b.v), P(b.o), P(b.lse), w.B, w.Hq, w.Hkv, w.N, w.Nk,
                                             w.d, causal, scale, sp))
            mark(1)
            check("fa_bwd_kv", lib.fa_bwd_kv(P(b.q), P(b.k), P(b.v), P(b.o), P(b.lse), P(b.do), P(b.dq), P(b.dk),
                                             P(b.dv), P(ws), ws_bytes, w.B, w.Hq, w.Hkv, w.N, w.Nk, w.d, causal,
                                             scale, sp))
            return marks(2)
        if sparse:
            # the broadcast mask: byte strides 0 over batch and heads
            mark(0)
            check("fa_fwd_blocksparse", lib.fa_fwd_blocksparse(P(b.q), P(b.k), P(b.v), P(b.o), P(b.lse), P(mask), 0, 0,
                                                               *dims, causal, scale, sp))
            mark(1)
            check("fa_bwd_blocksparse", lib.fa_bwd_blocksparse(P(b.q), P(b.k), P(b.v), P(b.o), P(b.lse), P(b.do),
                                                               P(b.dq), P(b.dk), P(b.dv), P(ws), ws_bytes, P(mask), 0,
                                                               0, *dims, causal, scale, sp))
            return marks(2)
        mark(0)
        if pair_fwd:
            check("fa_fwd_pair", lib.fa_fwd_pair(P(b.q), P(b.k), P(b.v), P(b.o), P(b.lse), w.B, w.Hq, w.Hkv, w.N, w.N,
                                                 w.d, causal, scale, sp))
        else:
            check("fa_fwd", lib.fa_fwd(P(b.q), P(b.k), P(b.v), P(b.o), P(b.lse), *dims, causal, scale, sp))
        mark(1)
        if det or w.d > 128:
            # one call: preprocess, then the dK/dV and dQ passes (no atomics); above
            # d = 128 fa_bwd itself runs the three passes (dV, dK, dQ)
            check("fa_bwd_deterministic", (lib.fa_bwd_deterministic if det else lib.fa_bwd)(P(b.q), P(b.k), P(b.v), P(b.o), P(b.lse), P(b.do),
                                                                   P(b.dq), P(b.dk), P(b.dv), P(ws), ws_bytes, *dims,
                                                                   causal, scale, sp))
            return marks(2)
        check("fa_bwd_preprocess", lib.fa_bwd_preprocess(P(b.o), P(b.lse), P(b.do), P(ws), ws_bytes, *dims, sp))
        mark(2)
        check("fa_bwd_dkdv", lib.fa_bwd_dkdv(P(b.q), P(b.k), P(b.v), P(b.do), P(b.dk), P(b.dv), P(ws), ws_bytes,
                                             *dims, causal, scale, sp))
        mark(3)
        check("fa_bwd_dq", lib.fa_bwd_dq(P(b.dq), P(ws), ws_bytes, *dims, scale, sp))
        mark(4)

    def step(ev):
        run(main, sptr, lambda i: ev[i].record(stream))

    def new_events():
        return [torch.cuda.Event(enable_timing=True) for _ in range(5)]

    for _ in range(args.warmup):
        flush.zero_()
        step(new_events())
    fa.check_device_status(stream.cuda_stream)
    # the exponential unit's rate on this GPU (a half-millisecond probe, before the timed region)
    ex2_rate = fa.ex2_throughput(stream.cuda_stream)

    gpu_id = os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local] if world > 1 or \
        "CUDA_VISIBLE_DEVICES" in os.environ else str(local)
    sampler = ClockSampler(gpu_id)
    time.sleep(0.3)
    events = [new_events() for _ in range(args.steps)]
    fa.sm_clock_mhz(stream.cuda_stream)          # reset the kernels' clock sums
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.time()
    for i in range(args.steps):
        flush.zero_()             # L2 flush between steps (outside the events)
        step(events[i])
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    t1 = time.time()
    kernel_mhz = fa.sm_clock_mhz(stream.cuda_stream)
    time.sleep(0.2)
    sampler.stop()
    fa.check_device_status(stream.cuda_stream)

    seg = [[events[i][j].elapsed_time(events[i][j + 1]) for j in range(4)] for i in range(args.steps)]
    step_ms = [events[i][0].elapsed_time(events[i][4]) for i in range(args.steps)]
    total_ms = max_over_ranks(sum(step_ms), world)
    flops_step = w.flops_fwd + (0.0 if fwd_only else w.flops_bwd)
    value = whole_job_tflops(world, flops_step, args.steps, total_ms)
    mean = [sum(s[j] for s in seg) / args.steps for j in range(4)]
    if fp8:
        fwd_kernel = "fwd_fp8_wide_kernel" if w.d > 128 else "fwd_fp8_kernel"
        fwd_src = "fa_fwd_fp8_wide.cu" if w.d > 128 else "fa_fwd_fp8.cu"
    elif pair_fwd:
        fwd_kernel, fwd_src = "fwd_pair_kernel", "fa_fwd_pair.cu"
    else:
        fwd_kernel = "fwd_wide_kernel" if w.d > 128 else "fwd_kernel"
        fwd_src = "fa_fwd_wide.cu" if w.d > 128 else "fa_fwd.cu"
    names = [fwd_kernel, "bwd_pre_kernel", "bwd_dkdv_kernel", "bwd_dq_kernel"]
    if fwd_only:
        names = [fwd_kernel, "-", "-", "-"]
    if det:
        names = ["fwd_kernel", "bwd_deterministic (preprocess + det_dkdv_kernel + det_dq_kernel)", "-", "-"]
    elif w.backward and w.d > 128:
        names = [fwd_kernel, "bwd_wide (preprocess + wide_dv_kernel, wide_dk_kernel, wide_dq_kernel)", "-", "-"]
    if sparse:
        names = ["fwd_kernel (block-sparse)", "bwd_blocksparse (preprocess + block list + dkdv + dq convert)", "-", "-"]
    if kvlen:
        names = ["fwd_kernel (Nq != Nk)", "bwd_kv (preprocess + dkdv + dq convert)", "-", "-"]
    peak, peak_src = peak_tflops(w.dtype)
    # dominant kernel of the step and its tensor roofline
    one_call_bwd = det or sparse or kvlen or (w.backward and w.d > 128)
    dom = 0 if mean[0] >= max(mean[1], mean[2]) else (1 if one_call_bwd else 2)
    dom_flops = w.flops_fwd if dom == 0 else w.flops_bwd
    achieved = dom_flops / (mean[dom] / 1e3) / 1e12
    traffic = None if (one_call_bwd and dom != 0) else traffic_from_profile(
        fwd_src if dom == 0 else "fa_bwd.cu", names[dom], w.name)
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": traffic, "kernel": names[dom], "peak_source": peak_src,
                "algorithmic_flops_per_launch": dom_flops}

    # ---- end to end: pinned host inputs -> device, the path, results -> host,
    # every step. Steps are pipelined the way a user would drive the library:
    # the copy in of step i+1 and the copy out of step i-1 run on their own
    # streams while step i computes, over NSETS sets of device buffers (with
    # two, step i's compute must wait for step i-2's results to leave, which
    # ties the compute stream to the copy-out stream; three leave it a step
    # of slack).
    e2e = None
    if args.e2e_steps > 0:
        names_in = ("q", "k", "v") if fwd_only else ("q", "k", "v", "do")
        names_out = ("o", "lse") if fwd_only else ("o", "lse", "dq", "dk", "dv")
        host_in = [getattr(main, n).cpu().pin_memory() for n in names_in]
        nsets = args.e2e_sets
        host_out = [[torch.empty(getattr(main, n).shape, dtype=getattr(main, n).dtype).pin_memory()
                     for n in names_out] for _ in range(nsets)]
        h2d = sum(x.numel() * x.element_size() for x in host_in)
        d2h = sum(x.numel() * x.element_size() for x in host_out[0])
        sets = [main] + [Bufs() for _ in range(nsets - 1)]
        for extra in sets[1:]:
            for n in names_in + names_out:
                setattr(extra, n, torch.empty_like(getattr(main, n)))
            if fp8:
                for n in ("q8", "qs", "k8", "ks", "vt8", "vs"):
                    setattr(extra, n, torch.empty_like(getattr(main, n)))
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        s_comp = stream
        done_in = [torch.cuda.Event() for _ in range(nsets)]
        done_comp = [torch.cuda.Event() for _ in range(nsets)]
        done_out = [torch.cuda.Event() for _ in range(nsets)]
        started = [False] * nsets

        def e2e_step(i):
            x = i % nsets
            b = sets[x]
            with torch.cuda.stream(s_in):
                if started[x]:
                    s_in.wait_event(done_comp[x])       # step i-nsets has finished reading set x
                for n, src in zip(names_in, host_in):
                    getattr(b, n).copy_(src, non_blocking=True)
                done_in[x].record(s_in)
            s_comp.wait_event(done_in[x])
            if started[x]:
                s_comp.wait_event(done_out[x])          # step i-nsets's results have left set x
            run(b, s_comp.cuda_stream, lambda _i: None, quantize=True)
            done_comp[x].record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done_comp[x])
                for n, dst in zip(names_out, host_out[x]):
                    dst.copy_(getattr(b, n), non_blocking=True)
                done_out[x].record(s_out)
            started[x] = True

        for i in range(2 * nsets):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s_in)
        for i in range(args.e2e_steps):
            e2e_step(i)
        for x in range(nsets):
            s_out.wait_event(done_out[x])
        z.record(s_out)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(a.elapsed_time(z) / args.e2e_steps, world)
        fa.check_device_status(stream.cuda_stream)
        e2e = {"value": world * flops_step / (e2e_ms / 1e3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "pipelining": f"copy in, compute, copy out on three streams over {nsets} device buffer sets"}

    if rank != 0:
        return
    clocks = sampler.summary(t0, t1, kernel_mhz)
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    rated = clock_rated_peak(w.dtype, n_sms, clocks.get("sm_mhz"))
    if rated:
        roofline["clock_rated_peak"] = rated
        roofline["frac_of_clock_rated"] = roofline["achieved"] / rated
        roofline["clock_rated_note"] = (f"{n_sms} SMs x dense tensor FLOP per SM clock x the SM clock the timed "
                                        "kernels measured")
    line = {
        "metric": metric_for(w), "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, **{kk: vv for kk, vv in w.describe().items() if kk != "workload"},
                   "l2": "flushed between steps (256 MiB write, outside the timed events)",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "bwd_variant": "none" if fwd_only else args.bwd,
                   "fwd_variant": args.fwd},
        "frac_of_peak": value / world / peak,
        "fwd_tflops": w.flops_fwd / (mean[0] / 1e3) / 1e12,
        "fwd_frac_of_peak": w.flops_fwd / (mean[0] / 1e3) / 1e12 / peak,
        "fwd_frac_of_clock_rated": (w.flops_fwd / (mean[0] / 1e3) / 1e12 / rated) if rated else None,
        "bwd_tflops": None if fwd_only else w.flops_bwd / (sum(mean[1:]) / 1e3) / 1e12,
        "kernel_ms": {n: m for n, m in zip(names, mean) if n != "-"},
        "roofline": roofline,
        "exp_roofline": exp_roofline(w, ex2_rate, n_sms, clocks.get("sm_mhz"), mean[0], names[0]),
        "step_ms_percentiles": percentiles(step_ms),
        "e2e": e2e,
        # fwd, preprocess, [block list], dK/dV, dQ convert
        "gpu_launches": (1 if (fwd_only or fp8) else 5 if (sparse or (w.backward and w.d > 128)) else
                         3 if det else 4) * args.steps,
        "clocks": clocks,
        "wall_s_timed_region": t1 - t0,
    }
    if world == 1 and not args.no_cpu_baseline and not sparse and not kvlen:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    from exact_attention_79_gb300 import configs
    w = configs.WORKLOADS[args.workload]
    if args.impl == "reference":
        if int(os.environ.get("RANK", "0")) != 0:
            return
        reference_arm(args, w)
        return
    native_arm(args, w)


if __name__ == "__main__":
    main()
