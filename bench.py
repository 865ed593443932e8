#!/usr/bin/env python3
"""Benchmark of the future-attention-mass / pruned-cache hot path on GB300.

One step = one pass of the whole path over the Qwen3-4B-shaped layer
(32 query / 8 KV heads, head_dim 128, S = 8192, bf16, w = 128, 25 % budget,
4 sinks + 128 recent): row LSE -> future-attention mass -> selection on F ->
compaction -> one-token decode over the pruned cache.  Inputs are resident in
HBM before the timed region; L2 is flushed (a 512 MiB write, then a 256 MiB read) before every
timed step.  `value` is the algorithmic TFLOP/s of the two QK^T passes over
the whole step time.  A second measured object, `decode`, is the pruned-cache
decode of the Qwen2.5-1.5B-shaped decode-eviction workload (28 layers,
12/2 heads, fp16, T = 120000 cache pruned to 4096) in GB/s, with every budget
(512 / 1024 / 2048 / 4096) reported; `long_context` times the two passes at
the Llama-3.1-8B-shaped 32 layers x S = 32768 and the Qwen3-8B-shaped
S = 131072 workloads.

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload (the reference arm of this tier: there is no upstream code).
Multi-GPU (torchrun): every rank runs its own independent layer (weak
scaling, no data-path collective); timings are max-reduced over ranks.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import kvp_inputs  # noqa: E402

METRIC = "future-attn-mass TFLOP/s (% bf16 peak); pruned-cache decode HBM GB/s (% peak)"
L2_BYTES = 129 * 1000 * 1000           # L2 of the GB300: 129 MB
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM traffic of one launch of the dominant kernel from an ncu capture, valid only while the
# kernel source is unchanged (sha256 of the .cu file at capture time).
NCU_TRAFFIC = {
    # ncu --set full of the mass pass (mass_tc_persistent_kernel) and the row LSE pass
    # (attn_tc_kernel<0>) on the benchmark layer (S = 8192; the kernel source hashed below),
    # DRAM bytes read + written per launch
    "future_attn_mass": {"sha": "5b69551d3fb6cae3", "bytes": 115430144 + 3844096},
    "lse_pass": {"sha": "5b69551d3fb6cae3", "bytes": 83915008 + 2474752},
}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def rank_workload(w, rank):
    """The independent layer a rank processes under weak scaling (its own seed)."""
    return w.scaled(seed=w.seed + 100 * rank)


def reduce_max(value, world_size, device=None):
    """Max over ranks of a per-rank time (the slowest rank sets the step time)."""
    if world_size <= 1:
        return float(value)
    import torch.distributed as dist
    t = torch.tensor([float(value)], device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank, world_size, ms_per_step):
    """Whole-job throughput: the work of all ranks over the (max-reduced) step time."""
    return flops_per_rank * world_size / (ms_per_step / 1e3) / 1e12


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock, power and throttle reasons, kept with host timestamps so
    that only the samples taken inside the timed region are summarised."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index, period_ms=20):
        self.gpu, self.period = gpu_index, period_ms
        self.proc, self.rows, self.thread = None, [], None
        self.windows = []

    def __enter__(self):
        import threading
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return self

        def reader():
            for line in self.proc.stdout:
                self.rows.append((time.time(), line.strip()))
        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()
        time.sleep(0.2)
        return self

    def mark(self, t0, t1):
        self.windows.append((t0, t1))

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread is not None:
                self.thread.join(timeout=2)

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}

        def inside(ts, slack):
            return any(a - slack <= ts <= b + slack for a, b in self.windows)
        picked, how = [], "inside the timed region"
        for slack in (0.0, 0.05, 0.2):
            picked = [r for ts, r in self.rows if inside(ts, slack)]
            if picked:
                if slack:
                    how = f"within {int(slack * 1e3)} ms of the timed region"
                break
        sms, mx, reasons = [], None, set()
        for r in picked:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 7:
                continue
            try:
                sms.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(self.NAMES, f[3:7]):
                if v == "Active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sms) if sms else None, "sm_max_mhz": mx,
                "samples": len(sms), "window": how, "reasons": sorted(reasons)}


class L2Flush:
    """Evicts L2 between timed steps: writes 512 MiB (4x the 129 MB L2), then reads another
    256 MiB so the dirty lines of the write are written back during the flush and the next
    timed kernel starts from a clean, cold L2.  Then the GPU idles for ~100 us (a clock-count
    delay kernel that touches no memory), so that the host has enqueued the timed launches
    before the first of them can start: the events then bracket device work, not the Python
    binding's and the launch path's host latency (the e2e leg keeps that latency in)."""

    HEAD_START_CYCLES = 200_000

    def __init__(self, dev):
        self.w = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.ones(64 << 20, dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.sum()
        torch.cuda._sleep(self.HEAD_START_CYCLES)


def capture_graph(fn, dev):
    """fn's launches captured into one CUDA graph (after a warm-up call of fn outside capture),
    or None when capture fails."""
    try:
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(dev)
        s.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(s):
            fn()
        torch.cuda.current_stream(dev).wait_stream(s)
        torch.cuda.synchronize(dev)
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize(dev)
        g.replay()
        torch.cuda.synchronize(dev)
        return g
    except Exception:                      # noqa: BLE001 -- any capture problem: no graph
        torch.cuda.synchronize(dev)
        return None


def file_sha(path):
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def oracle_sample_time(w, seconds_hint=None):
    """The fp64 oracle on one query head of the workload's layer (LSE over all rows + F over
    all keys): returns (flops, seconds, cores, description)."""
    import oracle
    x = kvp_inputs.make_prefill_layer(w, 0, device="cpu")
    q = x["q"][:1]
    k = x["k"][:1]
    scale = w.head_dim ** -0.5
    t0 = time.perf_counter()
    lse = oracle.row_lse(q, k, scale)
    oracle.future_attn_mass(q, k, lse, scale, w.window)
    dt = time.perf_counter() - t0
    S, ww = w.seq_len, max(w.seq_len - w.window, 0)
    flops = 2.0 * w.head_dim * (S * (S + 1) // 2 + ww * (ww + 1) // 2)
    desc = (f"one query head (of {w.h_q}) of the {w.name} layer: full causal row LSE and future "
            f"mass over all {S} keys, fp64 numpy")
    return flops, dt, os.cpu_count(), desc


def oracle_eviction_time(n_layers=4):
    """The oracle's selection, compaction and decode on the Qwen2.5-1.5B decode-eviction shapes at
    b = 4096, fp64 numpy on the host cores: selection over all 56 rows x 120000 seeded scores;
    compaction and decode of `n_layers` layers (2 rows each) with 4096 kept rows per row gathered
    from a cache of 8192 tokens per row (the gather and the decode scale with the kept rows, not
    with T).  Rates are per the rows each part ran on."""
    import numpy as np
    import oracle
    w = kvp_inputs.QWEN25_15B_DECODE
    R, T, D, b = w.rows, w.seq_len, w.head_dim, max(w.decode_budgets)
    scores = kvp_inputs.make_scores(R, T, seed=7).numpy()
    t0 = time.perf_counter()
    oracle.select_topk(scores, [b] * R, w.n_sink, w.n_recent, b_max=b)
    t_sel = time.perf_counter() - t0
    x = kvp_inputs.make_decode_cache(w, seq_len=2 * b)
    Rs = n_layers * w.h_kv
    rng = np.random.default_rng(0)
    idx = np.stack([np.sort(rng.choice(2 * b, b, replace=False)) for _ in range(Rs)])
    cnt = np.full(Rs, b)
    k16 = x["k"][:Rs].view(torch.int16).numpy()
    v16 = x["v"][:Rs].view(torch.int16).numpy()
    t0 = time.perf_counter()
    kc, vc = oracle.compact_kv(k16, v16, idx, cnt)
    t_cmp = time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle.decode_attn(x["q"][:n_layers], kc.view(np.float16), vc.view(np.float16), cnt, D ** -0.5)
    t_dec = time.perf_counter() - t0
    kv_bytes = 2 * Rs * b * D * 2
    return {"workload": w.name, "budget": b,
            "select_topk": {"seconds": t_sel, "GB/s": R * T * 4 / t_sel / 1e9, "rows": R},
            "compact_kv": {"seconds": t_cmp, "GB/s": 2 * kv_bytes / t_cmp / 1e9, "rows": Rs},
            "decode_attn": {"seconds": t_dec, "GB/s": kv_bytes / t_dec / 1e9, "rows": Rs},
            "sample": f"selection of all {R} rows; compaction and decode of {n_layers} layers "
                      f"({Rs} rows), 4096 kept rows each gathered from an 8192-token cache"}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    w = kvp_inputs.QWEN3_4B_LAYER
    for _ in range(args.warmup):
        oracle_sample_time(w)
    times = []
    flops = 0.0
    desc = ""
    cores = os.cpu_count()
    for _ in range(args.steps):
        flops, dt, cores, desc = oracle_sample_time(w)
        times.append(dt)
    ms = 1e3 * sum(times) / len(times)
    value = flops / (ms / 1e3) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "seq_len": w.seq_len, "h_q": w.h_q, "h_kv": w.h_kv,
                   "head_dim": w.head_dim, "window": w.window, "sample": "one query head"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_kvp(args):
    import learned_kv_cache_gb300 as kvp
    from learned_kv_cache_gb300.pipeline import PrefillPrunePlan

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    kvp.load()
    peaks, peak_src = load_peaks()
    w = kvp_inputs.QWEN3_4B_LAYER
    R, S, D = w.rows, w.seq_len, w.head_dim
    x = kvp_inputs.make_prefill_layer(rank_workload(w, rank), 0, device=dev)
    x = {k: v.unsqueeze(0).contiguous() for k, v in x.items()}
    plan = PrefillPrunePlan(1, w.h_q, w.h_kv, S, D, x["q"].dtype, w.window, w.n_sink, w.n_recent,
                            w.budget, device=dev)
    budgets = torch.full((R,), w.budget, dtype=torch.int32, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()

    def step(marks=None):
        R_ = R

        def mark(i):
            if marks is not None:
                marks[i].record(stream)
        mark(0)
        kvp.kvp_lse_pass(x["q"], x["k"], lse=plan.lse)
        mark(1)
        kvp.kvp_future_attn_mass(x["q"], x["k"], plan.lse, w.window, F=plan.F, workspace=plan.fam_ws)
        mark(2)
        kvp.kvp_select_topk(plan.F.view(R_, S), budgets, w.n_sink, w.n_recent, w.budget,
                            idx=plan.idx, count=plan.count)
        mark(3)
        kvp.kvp_compact_kv(x["k"].view(R_, S, D), x["v"].view(R_, S, D), plan.idx, plan.count,
                           k_out=plan.kc, v_out=plan.vc)
        mark(4)
        kvp.kvp_decode_attn(x["dq"], plan.kc, plan.vc, plan.count, out=plan.out,
                            workspace=plan.dec_ws)
        mark(5)

    # the clock sampler starts first so that the GPU does not idle (and clock down) between the
    # warm-up steps and the timed ones
    clk = ClockSampler(local).__enter__()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    kvp.kvp_check_device_status()

    K = args.steps
    # The timed steps carry an event at their start and end only: events between the stages would
    # sit between kernels that otherwise start under their predecessor's tail (selection ->
    # compaction -> decode use programmatic dependent launch).  The per-stage breakdown comes from
    # a second run of K steps with an event between every two stages.
    ends = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    barrier()
    torch.cuda.synchronize(dev)
    launches0 = kvp.kvp_launch_count()
    t0 = time.time()
    t_wall = time.perf_counter()
    for s in range(K):
        flush()                            # evict L2 (not timed: outside the events)
        ends[s][0].record(stream)
        step()
        ends[s][1].record(stream)
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall
    clk.mark(t0, time.time())
    launches = kvp.kvp_launch_count() - launches0
    barrier()
    kvp.kvp_check_device_status()
    step_ms = [a.elapsed_time(b) for a, b in ends]
    ms = reduce_max(sum(step_ms) / K, ws, dev)
    marks = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
    for s in range(K):
        flush()
        step(marks[s])
    torch.cuda.synchronize(dev)
    kvp.kvp_check_device_status()
    stage_names = ["lse_pass", "future_attn_mass", "select_topk", "compact_kv", "decode_attn"]
    per_stage = {n: [] for n in stage_names}
    for m in marks:
        for i, n in enumerate(stage_names):
            per_stage[n].append(m[i].elapsed_time(m[i + 1]))
    staged_ms = sum(m[0].elapsed_time(m[5]) for m in marks) / K
    lse_flops = 2.0 * D * w.h_q * (S * (S + 1) // 2)
    ww = S - w.window
    fam_flops = 2.0 * D * w.h_q * (ww * (ww + 1) // 2)
    flops = lse_flops + fam_flops
    value = whole_job_tflops(flops, ws, ms)
    stage_mean = {n: sum(v) / K for n, v in per_stage.items()}

    # dominant kernel roofline
    dom = "future_attn_mass" if stage_mean["future_attn_mass"] >= stage_mean["lse_pass"] else "lse_pass"
    dom_flops = fam_flops if dom == "future_attn_mass" else lse_flops
    achieved = dom_flops / (stage_mean[dom] / 1e3) / 1e12
    peak = float(peaks["bf16_tflops"])
    traffic = None
    tc_src = os.path.join(ROOT, "learned_kv_cache_gb300", "csrc", "attn_mass_tc.cu")
    simt_src = os.path.join(ROOT, "learned_kv_cache_gb300", "csrc", "attn_mass_simt.cu")
    rec = NCU_TRAFFIC.get(dom)
    if rec and rec.get("sha") in (file_sha(tc_src), file_sha(simt_src)):
        traffic = rec["bytes"]
    roofline = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                "peak_source": f"{peak_src} bf16_tflops (burst)"}

    # pruned-cache decode on the decode-eviction workload (HBM bound), every budget
    decode = decode_eviction_measure(kvp, dev, K, args.warmup, flush, peaks, ws)

    # the two passes at the long-context workloads (32 layers x 32768; 131072)
    long_context = long_context_measure(kvp, dev, args.warmup, peaks)

    # NEXT rows: KVpop target epilogue and the steady-state ring-cache decode step
    next_rows = {
        "kvpop_target": target_measure(kvp, x, plan, w, K, args.warmup, flush, peak, stream, dev),
        "ring_decode_step": ring_step_measure(kvp, dev, K, args.warmup, flush, peaks),
        "kvpop_sparse_lse": sparse_lse_measure(kvp, x, w, K, args.warmup, flush, peak, stream, dev),
        "chunked_prefill_compress": chunked_measure(kvp, dev, args.warmup, flush, peaks),
        "kvp_eviction_auc": rank_auc_measure(kvp, dev, args.warmup, min(K, 20), flush, peaks),
    }

    # end to end through the public API with host buffers
    e2e = e2e_measure(kvp, x, plan, budgets, w, K, args.warmup, stream, flops, ws, dev)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        f_c, t_c, cores, desc = oracle_sample_time(w)
        cpu = {"value": f_c / t_c / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": desc, "seconds": t_c, "nproc": os.cpu_count()}
        t_1 = oracle_one_thread_time(w)
        if t_1 is not None:
            cpu["one_thread"] = {"value": f_c / t_1 / 1e12, "unit": "TFLOP/s", "seconds": t_1, "cores": 1}
        # the long-context passes at the oracle's measured rate (not run: hours of CPU time)
        cpu["extrapolated"] = {lw.name: {"flops": lf, "seconds": lf / (f_c / t_c),
                                         "note": "extrapolated from the sample's flop rate"}
                               for lw, lf in ((kvp_inputs.LLAMA31_8B_32L, long_context_flops(kvp_inputs.LLAMA31_8B_32L)),
                                              (kvp_inputs.QWEN3_8B_131K, long_context_flops(kvp_inputs.QWEN3_8B_131K)))}
        cpu["decode_eviction"] = oracle_eviction_time()
    clk.__exit__(None, None, None)
    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "global_batch": ws, "seq_len": S, "h_q": w.h_q,
                   "h_kv": w.h_kv, "head_dim": D, "window": w.window, "budget": w.budget,
                   "n_sink": w.n_sink, "n_recent": w.n_recent,
                   "l2": "flushed before every timed step (512 MiB write + 256 MiB read)",
                   "parallelism": f"replicas: one independent layer per GPU x{ws}"},
        "frac_of_bf16_peak": value / peak,
        "stages_ms": stage_mean,
        "stages_note": "from a second run of the same steps with an event between every two "
                       f"stages (its step: {staged_ms:.4f} ms); the timed steps carry start and end "
                       "events only",
        "roofline": roofline,
        "decode": decode,
        "long_context": long_context,
        "next_rows": next_rows,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": int(launches),
        "clocks": clocks,
        "wall_s_timed_region": t_wall,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def decode_eviction_measure(kvp, dev, K, W, flush, peaks, ws):
    """Qwen2.5-1.5B decode eviction at T = 120000: control decode with key mass, select to the
    budget, compact, pruned decode, at each of the blog's budgets (512 / 1024 / 2048 / 4096).
    The pruned decode's HBM GB/s in a decode loop (back-to-back launches, inputs larger than L2)
    is the reported figure, with the one-launch figure (L2 flushed) and the decode's share of the
    select -> compact -> decode chain beside it; the headline is the largest budget."""
    w = kvp_inputs.QWEN25_15B_DECODE
    x = kvp_inputs.make_decode_cache(w, device=dev)
    per_budget = {}
    for b in w.decode_budgets:
        per_budget[str(b)] = _decode_eviction_budget(kvp, dev, K, W, flush, peaks, w, x, b)
    head = dict(per_budget[str(max(w.decode_budgets))])
    head["budgets"] = {b: {key: r[key] for key in ("value", "frac", "ms", "bytes")} | {
        "isolated_frac": r["isolated"]["frac"],
        "in_chain_frac": r["eviction_step_chain"]["decode_in_chain_frac"],
        "select_topk_ms": r["other_stages"]["select_topk"]["ms"],
        "compact_kv_ms": r["other_stages"]["compact_kv"]["ms"],
        "decode_in_chain_ms": r["eviction_step_chain"]["decode_in_chain_ms"],
        "select_compact_decode_chain_ms": r["eviction_step_chain"]["select_compact_decode_ms"]}
        for b, r in per_budget.items()}
    return head


def _decode_eviction_budget(kvp, dev, K, W, flush, peaks, w, x, b):
    R, T, D = w.rows, w.seq_len, w.head_dim
    full_len = torch.full((R,), T, dtype=torch.int32, device=dev)
    mass = torch.empty(R, T, device=dev)
    budgets = torch.full((R,), b, dtype=torch.int32, device=dev)
    idx = torch.empty(R, b, dtype=torch.int32, device=dev)
    cnt = torch.empty(R, dtype=torch.int32, device=dev)
    kc = torch.empty(R, b, D, dtype=x["k"].dtype, device=dev)
    vc = torch.empty_like(kc)
    out_full = torch.empty(w.n_layers, w.h_q, D, device=dev)
    out = torch.empty_like(out_full)
    ws_full = torch.empty(kvp.kvp_decode_attn_workspace_size(w.n_layers, w.h_q, w.h_kv, D, T, True),
                          dtype=torch.uint8, device=dev)
    ws_pr = torch.empty(kvp.kvp_decode_attn_workspace_size(w.n_layers, w.h_q, w.h_kv, D, b, False),
                        dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        kvp.kvp_decode_attn(x["q"], x["k"], x["v"], full_len, out=out_full, key_mass=mass,
                            workspace=ws_full)
        if ev:
            ev[1].record(stream)
        kvp.kvp_select_topk(mass, budgets, w.n_sink, w.n_recent, b, idx=idx, count=cnt)
        if ev:
            ev[2].record(stream)
        kvp.kvp_compact_kv(x["k"], x["v"], idx, cnt, k_out=kc, v_out=vc)
        if ev:
            ev[3].record(stream)
        flush()
        if ev:
            ev[4].record(stream)
        kvp.kvp_decode_attn(x["q"], kc, vc, cnt, out=out, workspace=ws_pr)
        if ev:
            ev[5].record(stream)

    for _ in range(W):
        step()
    torch.cuda.synchronize(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
    for s in range(K):
        flush()
        step(evs[s])
    torch.cuda.synchronize(dev)
    kvp.kvp_check_device_status()
    t_full = sum(e[0].elapsed_time(e[1]) for e in evs) / K
    t_sel = sum(e[1].elapsed_time(e[2]) for e in evs) / K
    t_cmp = sum(e[2].elapsed_time(e[3]) for e in evs) / K
    t_dec = sum(e[4].elapsed_time(e[5]) for e in evs) / K
    elt = x["k"].element_size()
    dec_bytes = 2 * R * b * D * elt + x["q"].numel() * elt + out.numel() * 4
    full_bytes = 2 * R * T * D * elt + mass.numel() * 4
    cmp_bytes = 4 * R * b * D * elt + R * b * 4
    sel_bytes = R * T * 4 + R * b * 4
    hbm = float(peaks["hbm_gbs"])
    gbs = dec_bytes / (t_dec / 1e3) / 1e9

    # The eviction step as one stream: select -> compact -> pruned decode with nothing between the
    # launches (each kernel starts while the one before finishes: programmatic dependent launch),
    # L2 flushed before the selection; and the same chain without the decode.  Their difference is
    # the decode's cost inside the step (it reads the cache compaction has just written).
    def chain(with_decode):
        ts = []
        for _ in range(K):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            kvp.kvp_select_topk(mass, budgets, w.n_sink, w.n_recent, b, idx=idx, count=cnt)
            kvp.kvp_compact_kv(x["k"], x["v"], idx, cnt, k_out=kc, v_out=vc)
            if with_decode:
                kvp.kvp_decode_attn(x["q"], kc, vc, cnt, out=out, workspace=ws_pr)
            e1.record(stream)
            ts.append((e0, e1))
        torch.cuda.synchronize(dev)
        return sum(a.elapsed_time(z) for a, z in ts) / K

    t_chain = chain(True)
    t_chain0 = chain(False)

    # A decode loop: launches back to back (as successive decode steps run), each over its own
    # copy of the pruned cache, the copies rotated so that everything read since a copy's last
    # use is more than 2.5x L2: every launch reads its cache from HBM.  The average launch
    # duration leaves out the per-measurement event and launch overhead (~4 us, an empty kernel
    # times 4-6 us this way) that the isolated figure carries.
    cache_bytes = 2 * R * b * D * elt
    n_c = max(3, -(-int(2.5 * L2_BYTES) // cache_bytes) + 1)
    copies = [(kc.clone(), vc.clone()) for _ in range(n_c)]
    n_launch = max(30, 3 * n_c)

    def loop():
        for i in range(n_launch):
            ck, cv = copies[i % n_c]
            kvp.kvp_decode_attn(x["q"], ck, cv, cnt, out=out, workspace=ws_pr)

    loop()
    graph = capture_graph(loop, dev)       # the same loop as one CUDA graph, when capture works

    def timed(run):
        t = 0.0
        for _ in range(3):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            run()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            t += e0.elapsed_time(e1) / n_launch / 3
        return t

    t_loop = timed(loop)
    t_graph = timed(graph.replay) if graph is not None else None
    del copies, graph
    kvp.kvp_check_device_status()
    gbs_loop = dec_bytes / (t_loop / 1e3) / 1e9
    gbs_chain = dec_bytes / ((t_chain - t_chain0) / 1e3) / 1e9
    return {
        "workload": w.name, "budget": b, "metric": "pruned-cache decode HBM GB/s",
        "value": gbs_loop, "unit": "GB/s", "frac": gbs_loop / hbm, "peak": hbm,
        "ms": t_loop, "bytes": dec_bytes,
        "timing": f"decode loop: {n_launch} launches back to back over {n_c} rotated copies of the "
                  f"pruned cache ({n_c * cache_bytes / 1e6:.0f} MB > L2), average per launch",
        "graph_replay": None if t_graph is None else {
            "ms": t_graph, "value": dec_bytes / (t_graph / 1e3) / 1e9,
            "frac": dec_bytes / (t_graph / 1e3) / 1e9 / hbm, "note": "the same loop captured as one CUDA graph"},
        "isolated": {"value": gbs, "frac": gbs / hbm, "ms": t_dec,
                     "l2": "flushed before the one timed launch"},
        "eviction_step_chain": {"select_compact_decode_ms": t_chain, "select_compact_ms": t_chain0,
                                "decode_in_chain_ms": t_chain - t_chain0,
                                "decode_in_chain_GB/s": gbs_chain, "decode_in_chain_frac": gbs_chain / hbm,
                                "l2": "flushed before the selection only"},
        "other_stages": {
            "full_cache_decode_with_key_mass": {"ms": t_full, "GB/s": full_bytes / (t_full / 1e3) / 1e9},
            "select_topk": {"ms": t_sel, "GB/s": sel_bytes / (t_sel / 1e3) / 1e9},
            "compact_kv": {"ms": t_cmp, "GB/s": cmp_bytes / (t_cmp / 1e3) / 1e9},
        },
    }


def long_context_flops(w):
    """A1 + A2 flops of a long-context workload: 2*D*H_q*[S(S+1)/2 + (S-w)(S-w+1)/2] per layer."""
    S, ww = w.seq_len, max(w.seq_len - w.window, 0)
    return w.n_layers * 2.0 * w.head_dim * w.h_q * (S * (S + 1) // 2 + ww * (ww + 1) // 2)


def long_context_measure(kvp, dev, W, peaks, K=3):
    """The two passes at the long-context workloads, each pass timed with CUDA events:
    Llama-3.1-8B-shaped 32 layers x S = 32768 (one launch per pass over all 32 layers,
    2.81e14 flop) and the Qwen3-8B-shaped layer at S = 131072 (1.405e14 flop).  Their inputs
    (8 GiB and 1 GiB of Q) are far larger than L2.  A pass runs for tens to hundreds of
    milliseconds, so the fraction is also given against the sustained bf16 peak."""
    res = {}
    stream = torch.cuda.current_stream(dev)
    for w in (kvp_inputs.LLAMA31_8B_32L, kvp_inputs.QWEN3_8B_131K):
        x = kvp_inputs.make_prefill(w, device=dev)
        q, k = x["q"], x["k"]
        del x
        B, S, D = w.n_layers, w.seq_len, w.head_dim
        lse = torch.empty(B, w.h_q, S, device=dev)
        F = torch.empty(B, w.h_kv, S, device=dev)
        fws = torch.empty(kvp.kvp_future_attn_mass_workspace_size(q.dtype, B, w.h_q, w.h_kv, S, D, w.window),
                          dtype=torch.uint8, device=dev)
        for _ in range(W):
            kvp.kvp_lse_pass(q, k, lse=lse)
            kvp.kvp_future_attn_mass(q, k, lse, w.window, F=F, workspace=fws)
        torch.cuda.synchronize(dev)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
        for e in evs:
            e[0].record(stream)
            kvp.kvp_lse_pass(q, k, lse=lse)
            e[1].record(stream)
            kvp.kvp_future_attn_mass(q, k, lse, w.window, F=F, workspace=fws)
            e[2].record(stream)
        torch.cuda.synchronize(dev)
        kvp.kvp_check_device_status()
        t_lse = sum(e[0].elapsed_time(e[1]) for e in evs) / K
        t_fam = sum(e[1].elapsed_time(e[2]) for e in evs) / K
        ww = S - w.window
        f_lse = 2.0 * D * w.h_q * B * (S * (S + 1) // 2)
        f_fam = 2.0 * D * w.h_q * B * (ww * (ww + 1) // 2)
        tf = (f_lse + f_fam) / ((t_lse + t_fam) / 1e3) / 1e12
        res[w.name] = {
            "flops": f_lse + f_fam, "ms": t_lse + t_fam, "value": tf, "unit": "TFLOP/s",
            "frac_burst": tf / float(peaks["bf16_tflops"]),
            "frac_sustained": tf / float(peaks["bf16_tflops_sustained"]),
            "lse_pass": {"ms": t_lse, "TFLOP/s": f_lse / (t_lse / 1e3) / 1e12},
            "future_attn_mass": {"ms": t_fam, "TFLOP/s": f_fam / (t_fam / 1e3) / 1e12},
            "steps": K, "l2": "inputs larger than L2"}
        del q, k, lse, F, fws
        torch.cuda.empty_cache()
    return res


def oracle_one_thread_time(w):
    """The same oracle sample as oracle_sample_time, timed in a fresh process restricted to one
    thread (one BLAS thread; numpy's elementwise loops are single-threaded anyway)."""
    import numpy as np
    x = kvp_inputs.make_prefill_layer(w, 0, device="cpu")
    with tempfile.TemporaryDirectory(prefix="kvp_bench_") as d:
        np.save(os.path.join(d, "q.npy"), x["q"][:1].to(torch.float64).numpy())
        np.save(os.path.join(d, "k.npy"), x["k"][:1].to(torch.float64).numpy())
        code = ("import sys, time, numpy as np\n"
                f"sys.path.insert(0, {ROOT!r})\n"
                "import oracle\n"
                f"q = np.load({os.path.join(d, 'q.npy')!r}); k = np.load({os.path.join(d, 'k.npy')!r})\n"
                f"s = {w.head_dim ** -0.5!r}\n"
                "t = time.perf_counter()\n"
                "l = oracle.row_lse(q, k, s)\n"
                f"oracle.future_attn_mass(q, k, l, s, {w.window})\n"
                "print(time.perf_counter() - t)\n")
        env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
        res = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                             timeout=900)
        if res.returncode != 0:
            return None
        return float(res.stdout.strip().splitlines()[-1])


def target_measure(kvp, x, plan, w, K, W, flush, peak, stream, dev):
    """KVpop target on the same layer: per-query-head future mass through the tensor-core pass
    plus the count-normalise / log / group-max epilogue, timed alone with L2 flushed."""
    R, S = w.h_q, w.seq_len
    tgt = torch.empty(1, w.h_kv, S, device=dev)
    ws = torch.empty(kvp.kvp_future_attn_target_workspace_size(x["q"].dtype, 1, w.h_q, w.h_kv, S,
                                                               w.head_dim, w.window),
                     dtype=torch.uint8, device=dev)

    def run():
        kvp.kvp_future_attn_target(x["q"], x["k"], plan.lse, w.window, target=tgt,
                                   want=("target",), workspace=ws)

    for _ in range(W):
        run()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    for e0, e1 in evs:
        flush()
        e0.record(stream)
        run()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    kvp.kvp_check_device_status()
    ms = sum(a.elapsed_time(b) for a, b in evs) / K
    ww = S - w.window
    flops = 2.0 * w.head_dim * R * (ww * (ww + 1) // 2)
    tf = flops / (ms / 1e3) / 1e12
    return {"metric": "KVpop target pass TFLOP/s", "value": tf, "unit": "TFLOP/s",
            "frac": tf / peak, "ms": ms, "flops": flops, "aggregate": "max_log",
            "l2": "flushed before every launch"}


def sparse_lse_measure(kvp, x, w, K, W, flush, peak, stream, dev):
    """KVpop's running top-k sparse attention on the same layer: the cutoffs from seeded static
    ranks (long-range budget k = budget - sinks - window), then the sparse row LSE (rank-ordered
    key stream where it is shorter).  Its TFLOP/s counts the causal pairs, so skipped tiles show
    up as a rate above the dense pass's."""
    S, D = w.seq_len, w.head_dim
    k_lr = w.budget - w.n_sink - w.window
    ranks = kvp_inputs.make_static_ranks(w.h_kv, S, seed=3, device=dev)
    tau = torch.empty_like(ranks)
    lse = torch.empty(1, w.h_q, S, device=dev)
    sws = torch.empty(max(1, kvp.kvp_sparse_lse_workspace_size(x["q"].dtype, 1, w.h_q, w.h_kv, S, D)),
                      dtype=torch.uint8, device=dev)

    def run(ev=None):
        if ev:
            ev[0].record(stream)
        kvp.kvp_topk_cutoffs(ranks, w.n_sink, w.window, k_lr, tau=tau)
        if ev:
            ev[1].record(stream)
        kvp.kvp_sparse_lse_pass(x["q"], x["k"], ranks, tau, w.n_sink, w.window, lse=lse, workspace=sws)
        if ev:
            ev[2].record(stream)

    for _ in range(W):
        run()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    for e in evs:
        flush()
        run(e)
    torch.cuda.synchronize(dev)
    kvp.kvp_check_device_status()
    t_cut = sum(e[0].elapsed_time(e[1]) for e in evs) / K
    t_lse = sum(e[1].elapsed_time(e[2]) for e in evs) / K
    flops = 2.0 * D * w.h_q * (S * (S + 1) // 2)
    tf = flops / (t_lse / 1e3) / 1e12
    return {"metric": "sparse row LSE TFLOP/s (causal pairs)", "value": tf, "unit": "TFLOP/s",
            "frac": tf / peak, "sparse_lse_ms": t_lse, "cutoffs_us": t_cut * 1e3,
            "k_long_range": k_lr, "l2": "flushed before every pair of launches"}


def chunked_measure(kvp, dev, W, flush, peaks, chunk=8192):
    """Chunked prefill-compress on the Qwen2.5-1.5B cache shapes (56 rows, 120000 tokens, budget
    4096, per-token static scores): the whole loop of compress steps, each timed with L2
    flushed; reports the loop's time and the HBM rate of its K/V movement."""
    w = kvp_inputs.QWEN25_15B_DECODE
    x = kvp_inputs.make_decode_cache(w, device=dev)
    R, T, D = w.rows, w.seq_len, w.head_dim
    b = max(w.decode_budgets)
    scores = kvp_inputs.make_scores(R, T, seed=7, device=dev)
    chunks = [(p0, min(T, p0 + chunk)) for p0 in range(0, T, chunk)]
    ck = [x["k"][:, a:e].contiguous() for a, e in chunks]
    cv = [x["v"][:, a:e].contiguous() for a, e in chunks]
    cs = [scores[:, a:e].contiguous() for a, e in chunks]
    del x
    bufs = [{"k": torch.empty(R, b, D, dtype=ck[0].dtype, device=dev),
             "v": torch.empty(R, b, D, dtype=ck[0].dtype, device=dev),
             "score": torch.empty(R, b, device=dev),
             "pos": torch.empty(R, b, dtype=torch.int32, device=dev)} for _ in range(2)]
    idx = torch.empty(R, b, dtype=torch.int32, device=dev)
    cnt = torch.empty(R, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def loop(evs=None):
        cache, n = None, 0
        for i, (a, e) in enumerate(chunks):
            if evs:
                flush()
                evs[i][0].record(stream)
            out = bufs[i % 2]
            kvp.kvp_chunk_compress(cache, n, ck[i], cv[i], cs[i], a, b, w.n_sink, w.n_recent, out,
                                   idx=idx, count=cnt)
            if evs:
                evs[i][1].record(stream)
            cache, n = out, min(max(b, w.n_sink + w.n_recent), n + (e - a))

    for _ in range(W):
        loop()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in chunks]
    loop(evs)
    torch.cuda.synchronize(dev)
    kvp.kvp_check_device_status()
    step_ms = [a.elapsed_time(e) for a, e in evs]
    elt = ck[0].element_size()
    moved, n = 0, 0
    for a, e in chunks:
        kept = min(max(b, w.n_sink + w.n_recent), n + (e - a))
        moved += 2 * (2 * R * kept * D * elt) + R * (n + e - a) * 4 + R * kept * 12
        n = kept
    gbs = moved / (sum(step_ms) / 1e3) / 1e9
    hbm = float(peaks["hbm_gbs"])
    return {"metric": "chunked prefill-compress HBM GB/s", "value": gbs, "unit": "GB/s",
            "frac": gbs / hbm, "peak": hbm, "loop_ms": sum(step_ms), "steps": len(chunks),
            "chunk": chunk, "budget": b, "mean_step_us": sum(step_ms) / len(chunks) * 1e3,
            "l2": "flushed before every step"}


def rank_auc_measure(kvp, dev, W, K, flush, peaks, M=16):
    """Qwen3-8B 131k shapes (8 KV heads x 131072 tokens): static ranks from scores (the ranking
    sort) and the eviction-cost AUC of M rankings per head, each timed with L2 flushed."""
    w = kvp_inputs.QWEN3_8B_131K
    R, T = w.h_kv, w.seq_len
    s = kvp_inputs.make_scores(R, T, seed=21, device=dev)
    ranks = torch.empty(R, T, dtype=torch.int32, device=dev)
    ws = torch.empty(int(kvp.load().kvp_rank_rows_workspace_size(R, T)), dtype=torch.uint8, device=dev)
    F = torch.rand(R, T, generator=torch.Generator(device=dev).manual_seed(4), device=dev)
    many = torch.stack([torch.randperm(T, device=dev) for _ in range(R * M)]).view(R, M, T).to(torch.int32)
    auc = torch.empty(R, M, dtype=torch.float64, device=dev)
    aws = torch.empty(int(kvp.load().kvp_eviction_auc_workspace_size(R, M, T)), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(W):
        kvp.kvp_rank_rows(s, ranks=ranks, workspace=ws)
        kvp.kvp_eviction_auc(F, many, auc=auc, workspace=aws)
    t_rank, t_auc = [], []
    for _ in range(K):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        flush()
        e[0].record(stream)
        kvp.kvp_rank_rows(s, ranks=ranks, workspace=ws)
        e[1].record(stream)
        flush()
        e[2].record(stream)
        kvp.kvp_eviction_auc(F, many, auc=auc, workspace=aws)
        e[3].record(stream)
        torch.cuda.synchronize(dev)
        t_rank.append(e[0].elapsed_time(e[1]))
        t_auc.append(e[2].elapsed_time(e[3]))
    kvp.kvp_check_device_status()
    ms_r, ms_a = sum(t_rank) / K, sum(t_auc) / K
    rank_bytes = 4 * (2 * R * T * 8) + R * T * 8          # four passes of (key, index) read+write, scores, ranks
    auc_bytes = R * M * T * 4 + R * T * 4
    hbm = float(peaks["hbm_gbs"])
    return {"metric": "eviction-cost AUC HBM GB/s", "value": auc_bytes / (ms_a / 1e3) / 1e9, "unit": "GB/s",
            "frac": auc_bytes / (ms_a / 1e3) / 1e9 / hbm, "auc_ms": ms_a, "rankings": M,
            "rank_rows_ms": ms_r, "rank_rows_GB/s": rank_bytes / (ms_r / 1e3) / 1e9,
            "rows": R, "T": T, "l2": "flushed before every launch"}


def ring_step_measure(kvp, dev, K, W, flush, peaks, cap=4096):
    """Steady-state decode with a static cache of `cap` slots per row on the Qwen2.5-1.5B decode
    workload: per token, insert the new key/value in place (evicting the lowest accumulated
    score outside sinks and the recent window) and decode over the cache while accumulating
    each slot's attention.  L2 is flushed before every token step."""
    w = kvp_inputs.QWEN25_15B_DECODE
    x = kvp_inputs.make_decode_cache(w, device=dev)
    R, T, D = w.rows, w.seq_len, w.head_dim
    kc = x["k"][:, :cap].contiguous()
    vc = x["v"][:, :cap].contiguous()
    del x["k"], x["v"]
    pos = torch.arange(cap, dtype=torch.int32, device=dev).repeat(R, 1).contiguous()
    score = torch.rand(R, cap, generator=torch.Generator(device=dev).manual_seed(5), device=dev)
    fill = torch.full((R,), cap, dtype=torch.int32, device=dev)
    g = torch.Generator(device=dev).manual_seed(6)
    steps = W + K
    new_k = torch.randn(steps, R, D, generator=g, device=dev).to(kc.dtype)
    new_v = torch.randn(steps, R, D, generator=g, device=dev).to(kc.dtype)
    out = torch.empty(w.n_layers, w.h_q, D, device=dev)
    slot = torch.empty(R, dtype=torch.int32, device=dev)
    ws = torch.empty(kvp.kvp_decode_attn_workspace_size(w.n_layers, w.h_q, w.h_kv, D, cap, True),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(t):
        kvp.kvp_ring_insert(kc, vc, pos, score, fill, new_k[t], new_v[t], cap + t, w.n_sink,
                            w.n_recent, out_slot=slot)
        kvp.kvp_decode_attn(x["q"], kc, vc, fill, out=out, key_mass=score, accumulate=True,
                            workspace=ws)

    for t in range(W):
        step(t)
    torch.cuda.synchronize(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    for i, e in enumerate(evs):
        flush()
        e[0].record(stream)
        kvp.kvp_ring_insert(kc, vc, pos, score, fill, new_k[W + i], new_v[W + i], cap + W + i,
                            w.n_sink, w.n_recent, out_slot=slot)
        e[1].record(stream)
        kvp.kvp_decode_attn(x["q"], kc, vc, fill, out=out, key_mass=score, accumulate=True,
                            workspace=ws)
        e[2].record(stream)
    torch.cuda.synchronize(dev)
    kvp.kvp_check_device_status()
    t_ins = sum(e[0].elapsed_time(e[1]) for e in evs) / K
    t_dec = sum(e[1].elapsed_time(e[2]) for e in evs) / K
    elt = kc.element_size()
    ins_bytes = R * cap * 8 + 2 * R * D * elt * 2
    dec_bytes = 2 * R * cap * D * elt + x["q"].numel() * elt + out.numel() * 4 + R * cap * 8
    hbm = float(peaks["hbm_gbs"])
    gbs = (ins_bytes + dec_bytes) / ((t_ins + t_dec) / 1e3) / 1e9

    # The token loop as it runs in serving: token steps back to back, round-robin over n_c
    # independent ring caches (sequences) whose total is more than 2.5x L2, so every step reads
    # its cache from HBM; the average per token leaves out the per-measurement event overhead.
    state_bytes = 2 * R * cap * D * elt + R * cap * 8
    n_c = max(3, -(-int(2.5 * L2_BYTES) // state_bytes) + 1)
    seqs = [(kc.clone(), vc.clone(), pos.clone(), score.clone(), fill.clone()) for _ in range(n_c)]
    n_tok = max(30, 3 * n_c)
    nk = torch.randn(n_tok, R, D, generator=g, device=dev).to(kc.dtype)
    nv = torch.randn(n_tok, R, D, generator=g, device=dev).to(kc.dtype)

    def tokens(t0):
        for i in range(n_tok):
            ck, cv, cp, cs, cf = seqs[i % n_c]
            kvp.kvp_ring_insert(ck, cv, cp, cs, cf, nk[i], nv[i], t0 + i // n_c, w.n_sink,
                                w.n_recent, out_slot=slot)
            kvp.kvp_decode_attn(x["q"], ck, cv, cf, out=out, key_mass=cs, accumulate=True,
                                workspace=ws)

    tokens(cap + steps)
    t_loop = 0.0
    for rep in range(3):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        tokens(cap + steps + (rep + 1) * n_tok)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        t_loop += e0.elapsed_time(e1) / n_tok / 3
    del seqs
    kvp.kvp_check_device_status()
    gbs_loop = (ins_bytes + dec_bytes) / (t_loop / 1e3) / 1e9
    return {"metric": "ring-cache decode step HBM GB/s", "value": gbs_loop, "unit": "GB/s",
            "frac": gbs_loop / hbm, "peak": hbm, "cap": cap, "us_per_token": t_loop * 1e3,
            "bytes": ins_bytes + dec_bytes,
            "timing": f"token loop: {n_tok} token steps back to back, round-robin over {n_c} ring "
                      f"caches ({n_c * state_bytes / 1e6:.0f} MB > L2), average per token",
            "isolated": {"value": gbs, "frac": gbs / hbm, "us_per_token": (t_ins + t_dec) * 1e3,
                         "ring_insert_us": t_ins * 1e3, "decode_with_key_mass_us": t_dec * 1e3,
                         "l2": "flushed before every token step, each launch timed"}}


def e2e_measure(kvp, x, plan, budgets, w, K, W, stream, flops, ws, dev):
    """Whole step through the public API from pinned host buffers
    (PrefillPrunePlan.run_from_host): H2D of Q/K/V and the decode query in four KV-head slices,
    overlapped with the slices' LSE and mass passes, then selection, compaction, decode and the
    D2H of F, the kept indices/counts and the decode output."""
    host = {k: v.cpu().pin_memory() for k, v in x.items()}
    outs = {"F": plan.F, "idx": plan.idx, "count": plan.count, "out": plan.out}
    host_out = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in outs.items()}
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out.values())

    def step():
        plan.run_from_host(host["q"], host["k"], host["v"], host["dq"], budgets, host_out, stream=stream)

    for _ in range(W):
        step()
    torch.cuda.synchronize(dev)
    if ws > 1:                             # every rank starts the timed loop together
        import torch.distributed as dist
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    kvp.kvp_check_device_status()
    ms = reduce_max(e0.elapsed_time(e1) / K, ws, dev)     # the slowest rank sets the time
    return {"value": flops * ws / (ms / 1e3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "overlap": "H2D in four KV-head slices on a copy stream; each slice's LSE pass starts when it lands, its mass pass on a second compute stream"}


def run_ncu_case(args):
    """A fixed case for profiler captures: `--steps` launches of one stage, no timing.
    lse / fam / sparse (cutoffs + sparse LSE) / cutoffs: one Qwen3-4B-shaped layer at --seq-len
    (default 32768: Q = 256 MiB, larger than L2); decode / select / compact / ring / chunked: the
    Qwen2.5-1.5B decode-eviction shapes (T = 120000, 28 layers x 2 KV heads, budget 4096; ring: a
    full static cache of 4096 slots per row, one insert plus one decode with accumulated key mass
    per step; chunked: two compress steps of 8192-token chunks per step, the second onto the
    cache); auc: eviction AUC of 16 random rankings per row, 8 rows x 131072."""
    import learned_kv_cache_gb300 as kvp
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    kvp.load()
    case = args.ncu_case
    if case == "cutoffs":
        w = kvp_inputs.QWEN3_4B_LAYER.scaled(seq_len=args.seq_len)
        k_lr = w.budget - w.n_sink - w.window
        ranks = kvp_inputs.make_static_ranks(w.h_kv, w.seq_len, seed=3, device=dev)
        tau = kvp.kvp_topk_cutoffs(ranks, w.n_sink, w.window, k_lr)
        for _ in range(args.steps):
            kvp.kvp_topk_cutoffs(ranks, w.n_sink, w.window, k_lr, tau=tau)
    elif case == "auc":
        w = kvp_inputs.QWEN3_8B_131K
        R, T, M = w.h_kv, w.seq_len, 16
        F = torch.rand(R, T, generator=torch.Generator(device=dev).manual_seed(4), device=dev)
        many = torch.stack([torch.randperm(T, device=dev) for _ in range(R * M)]).view(R, M, T).to(torch.int32)
        for _ in range(args.steps):
            kvp.kvp_eviction_auc(F, many)
    elif case in ("lse", "fam", "sparse"):
        w = kvp_inputs.QWEN3_4B_LAYER.scaled(seq_len=args.seq_len)
        x = kvp_inputs.make_prefill_layer(w, 0, device=dev)
        q, k = x["q"][None].contiguous(), x["k"][None].contiguous()
        lse = kvp.kvp_lse_pass(q, k)
        F = kvp.kvp_future_attn_mass(q, k, lse, w.window)
        if case == "sparse":
            k_lr = w.budget - w.n_sink - w.window
            ranks = kvp_inputs.make_static_ranks(w.h_kv, w.seq_len, seed=3, device=dev)
            tau = kvp.kvp_topk_cutoffs(ranks, w.n_sink, w.window, k_lr)
        for _ in range(args.steps):
            if case == "lse":
                kvp.kvp_lse_pass(q, k, lse=lse)
            elif case == "fam":
                kvp.kvp_future_attn_mass(q, k, lse, w.window, F=F)
            else:
                kvp.kvp_topk_cutoffs(ranks, w.n_sink, w.window, k_lr, tau=tau)
                kvp.kvp_sparse_lse_pass(q, k, ranks, tau, w.n_sink, w.window, lse=lse)
    else:
        w = kvp_inputs.QWEN25_15B_DECODE
        R, T, D, b = w.rows, w.seq_len, w.head_dim, max(w.decode_budgets)
        gen = torch.Generator(device=dev).manual_seed(0)
        if case == "decode":
            q = torch.randn(w.n_layers, w.h_q, D, generator=gen, device=dev).half()
            kc = torch.randn(R, b, D, generator=gen, device=dev).half()
            vc = torch.randn(R, b, D, generator=gen, device=dev).half()
            lens = torch.full((R,), b, dtype=torch.int32, device=dev)
            for _ in range(args.steps):
                kvp.kvp_decode_attn(q, kc, vc, lens)
        elif case == "select":
            scores = torch.rand(R, T, generator=gen, device=dev)
            budgets = torch.full((R,), b, dtype=torch.int32, device=dev)
            for _ in range(args.steps):
                kvp.kvp_select_topk(scores, budgets, w.n_sink, w.n_recent, b)
        elif case == "compact":
            k = torch.randn(R, T, D, generator=gen, device=dev).half()
            v = torch.randn(R, T, D, generator=gen, device=dev).half()
            idx = torch.sort(torch.randperm(T, device=dev)[:b]).values.to(torch.int32)
            idx = idx[None].repeat(R, 1).contiguous()
            cnt = torch.full((R,), b, dtype=torch.int32, device=dev)
            for _ in range(args.steps):
                kvp.kvp_compact_kv(k, v, idx, cnt)
        elif case == "ring":
            # static cache of `b` slots per row, full: insert + decode with accumulated key mass
            q = torch.randn(w.n_layers, w.h_q, D, generator=gen, device=dev).half()
            kc = torch.randn(R, b, D, generator=gen, device=dev).half()
            vc = torch.randn(R, b, D, generator=gen, device=dev).half()
            pos = torch.arange(b, dtype=torch.int32, device=dev).repeat(R, 1).contiguous()
            score = torch.rand(R, b, generator=gen, device=dev)
            fill = torch.full((R,), b, dtype=torch.int32, device=dev)
            nk = torch.randn(R, D, generator=gen, device=dev).half()
            for t in range(args.steps):
                kvp.kvp_ring_insert(kc, vc, pos, score, fill, nk, nk, b + t, w.n_sink, w.n_recent)
                kvp.kvp_decode_attn(q, kc, vc, fill, key_mass=score, accumulate=True)
        elif case == "chunked":
            # two compress steps per step: the first 8192-token chunk, then the next onto the cache
            x = kvp_inputs.make_decode_cache(w, device=dev)
            scores = kvp_inputs.make_scores(R, 2 * 8192, seed=7, device=dev)
            ck = [x["k"][:, a:a + 8192].contiguous() for a in (0, 8192)]
            cv = [x["v"][:, a:a + 8192].contiguous() for a in (0, 8192)]
            cs = [scores[:, a:a + 8192].contiguous() for a in (0, 8192)]
            del x
            torch.cuda.empty_cache()           # keep the profiled process's device memory small
            bufs = [{"k": torch.empty(R, b, D, dtype=ck[0].dtype, device=dev),
                     "v": torch.empty(R, b, D, dtype=ck[0].dtype, device=dev),
                     "score": torch.empty(R, b, device=dev),
                     "pos": torch.empty(R, b, dtype=torch.int32, device=dev)} for _ in range(2)]
            for _ in range(args.steps):
                kvp.kvp_chunk_compress(None, 0, ck[0], cv[0], cs[0], 0, b, w.n_sink, w.n_recent, bufs[0])
                kvp.kvp_chunk_compress(bufs[0], min(8192, max(b, w.n_sink + w.n_recent)), ck[1], cv[1], cs[1],
                                       8192, b, w.n_sink, w.n_recent, bufs[1])
        else:
            raise SystemExit(f"unknown --ncu-case {case}")
    torch.cuda.synchronize(dev)
    kvp.kvp_check_device_status()
    print(f"ncu case {case}: {args.steps} launches ok", flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="kvp", choices=["kvp", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ncu-case", default=None,
                    help="profiler case: lse | fam | sparse | cutoffs | decode | select | compact | ring | "
                         "chunked | auc (no JSON line)")
    ap.add_argument("--seq-len", type=int, default=32768)
    args = ap.parse_args()
    if args.ncu_case:
        return run_ncu_case(args)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_kvp(args)


if __name__ == "__main__":
    sys.exit(main())
