"""Throughput of the fused indexer -> Top-K -> sparse-attention decode chain on one GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

A step is one call of the fused chain (dsa_decode / dsa_prefill through the C ABI) over one batch
of seeded synthetic inputs already resident in HBM.  The default workload is the batch-8 decode at
L = 32768 (bf16 indexer 64 x 128, K = 2048, 16 heads over a 576-wide latent row).  Steps rotate
over several independent input sets whose total size is several times the 129 MB L2, so every
step reads its caches from HBM.  By default six independent batches are in flight (consecutive
steps on six streams, each input set always on the same stream); the same steps one batch at a time
are reported as `serial`.  Rank 0 prints one JSON line.

--impl reference times the oracle (plain fp64 CPU code) on the host cores on the same workload.
Under torchrun every rank runs an independent replica (no data-path collective); the barrier and
the max over ranks only frame the timing.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "indexer+TopK+sparse-attn queries/s; achieved HBM GB/s vs ~8 TB/s roofline"
NOMINAL_HBM_GBS = 8000.0
L2_BYTES = 129 * 1024 * 1024
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------------------------------------
# algorithmic bytes (what the method must move; scratch and the index round trip excluded)


def idx_elem_bytes(wl):
    return 2 if wl.idx_dtype == "bf16" else 1


def bytes_per_query(wl, n_visible=None):
    """Compulsory HBM bytes for one query: the indexer keys (+E8M0 scales) of every visible
    position, the query-side indexer inputs, the K gathered KV rows (+scales) and q + out."""
    n = wl.L if n_visible is None else n_visible
    e = idx_elem_bytes(wl)
    k_idx = n * wl.d_idx * e + (n * wl.d_idx // 32 if wl.idx_dtype == "mxfp8" else 0)
    q_side = wl.H_idx * wl.d_idx * e + (wl.H_idx * wl.d_idx // 32 if wl.idx_dtype == "mxfp8" else 0) + wl.H_idx * 4
    kv_e = 2 if wl.kv_dtype == "bf16" else 1
    rows = min(wl.K, n)
    if wl.separate_v:
        kv = rows * (wl.D_qk + wl.D_v) * kv_e
    else:
        n_scales = {"fp8": 1, "fp8_t128": -(-wl.D_qk // 128)}.get(wl.kv_dtype, 0)
        kv = rows * wl.D_qk * kv_e + rows * 4 * n_scales
    q_out = wl.H * wl.D_qk * 2 + wl.H * wl.D_v * 2
    return k_idx + q_side + kv + q_out


def step_bytes(wl):
    """Compulsory HBM bytes of one step (all queries; each query's own visible length)."""
    if wl.lengths:
        return sum(bytes_per_query(wl, n) for n in wl.lengths)
    return bytes_per_query(wl) * wl.T


def index_score_bytes(wl, T):
    """Compulsory bytes of one index-score launch over T decode queries: keys (+scales) read,
    query-side inputs read, fp32 scores written (visible positions only)."""
    e = idx_elem_bytes(wl)
    total = 0
    for t in range(T):
        n = wl.lengths[t] if wl.lengths else wl.L
        per_q = n * wl.d_idx * e + wl.H_idx * wl.d_idx * e + wl.H_idx * 4 + n * 4
        if wl.idx_dtype == "mxfp8":
            per_q += n * wl.d_idx // 32 + wl.H_idx * wl.d_idx // 32
        total += per_q
    return total


# ------------------------------------------------------------------------------------------------
# helpers


def measured_hbm_peak():
    try:
        with open(PEAKS_FILE) as f:
            v = json.load(f).get("hbm_gbs")
        if v:
            return float(v), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_peak():
    try:
        with open(PEAKS_FILE) as f:
            v = json.load(f).get("bf16_tflops")
        if v:
            return float(v), "measured (burst)"
    except (OSError, ValueError):
        pass
    return 1900.0, "fallback"


def index_score_flops(wl):
    """Algorithmic FLOPs of one index-score launch: 2 * H_idx * d_idx per visible (query,
    position) pair (the ReLU / weighting epilogue is not counted)."""
    pairs = 0
    for t in range(wl.T):
        pairs += (min(wl.L, wl.q_pos0 + t % wl.q_per_seq + 1) if wl.q_pos0 >= 0 else wl.L)
    return 2 * wl.H_idx * wl.d_idx * pairs


def kernel_source_hash():
    path = os.path.join(ROOT, "top_sparse_attention_gb300", "csrc", "index_score.cu")
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(workload):
    """DRAM bytes per index-score launch from the committed ncu summary, if it was taken on the
    current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", f"index_score_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_hash = re.search(r"source_sha256_16:\s*([0-9a-f]{16})", text)
    m_val = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    if not m_hash or not m_val or m_hash.group(1) != kernel_source_hash():
        return None
    return int(m_val.group(1))


class ClockSampler:
    """nvidia-smi clock/throttle samples taken while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.samples = []
        self._stop = threading.Event()
        self._t = None

    def _run(self):
        while not self._stop.is_set():
            try:
                out = subprocess.run(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                      "--format=csv,noheader,nounits"], capture_output=True, text=True,
                                     timeout=5).stdout.strip()
                if out:
                    self.samples.append([x.strip() for x in out.split(",")])
            except (OSError, subprocess.SubprocessError):
                return
            self._stop.wait(0.05)

    def __enter__(self):
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self._t:
            self._t.join(timeout=10)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(s[0]) for s in self.samples if s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in self.samples for i in range(4) if s[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.samples)}


def blas_threads():
    """Threads numpy's BLAS uses (what the oracle's matmuls run on)."""
    try:
        import ctypes

        for line in open("/proc/self/maps"):
            if "openblas" in line.lower():
                lib = ctypes.CDLL(line.split()[-1])
                for fn in ("openblas_get_num_threads64_", "scipy_openblas_get_num_threads64_",
                           "openblas_get_num_threads"):
                    if hasattr(lib, fn):
                        return int(getattr(lib, fn)())
    except OSError:
        pass
    return os.cpu_count()


def cpu_oracle_rate(wl, cpu_inputs, budget_s):
    """Oracle queries/s on the host: whole chain (scores, full-sort Top-K, attention) for the
    queries of one input set, repeated until `budget_s` seconds of work are done."""
    import numpy as np  # noqa: F401

    import oracle

    a = synth.to_numpy_bits(cpu_inputs)
    ch = oracle.Chain(a, L=wl.L, K=wl.K, q_per_seq=wl.q_per_seq, q_pos0=wl.q_pos0,
                      idx_dtype=wl.idx_dtype, kv_dtype=wl.kv_dtype, sm_scale=wl.sm_scale)
    n = 0
    t0 = time.perf_counter()
    while True:
        oracle.chain_query(ch, n % wl.T, wl.D_v)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s and n >= 1:
            break
    return n / el, n, el


# ------------------------------------------------------------------------------------------------
# arms


def rank_seed_offset(rank, i):
    """Seed offset of input set i on rank `rank`: every replica draws its own batches."""
    return rank * 100 + i


def max_over_ranks(ms, world, device):
    """The slowest rank's per-step time: the job is as fast as its slowest replica."""
    if world <= 1:
        return ms
    import torch.distributed as dist

    t = torch.tensor([ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


GRAPH_MAX_STEPS = 240  # steps held by one captured graph (a multiple of the input-set count is used)


def capture_steps(first, count, stream, streams, enqueue, events=None):
    """One CUDA graph holding steps first .. first+count-1: step i is enqueued by enqueue(i, st)
    on streams[i % len(streams)], all forked from and joined back into `stream`.  Everything the
    steps read stays owned by the caller (a graph keeps raw pointers only).  `events` = (start,
    end) timing events recorded as the graph's first and last nodes (external events)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        if events is not None:
            events[0].record(stream)
        fork = torch.cuda.Event()
        fork.record(stream)
        for st in streams:
            if st is not stream:
                st.wait_event(fork)
        for i in range(first, first + count):
            st = streams[i % len(streams)]
            with torch.cuda.stream(st):
                enqueue(i, st)
        for st in streams:
            if st is not stream:
                stream.wait_stream(st)
        if events is not None:
            events[1].record(stream)
    return g


def step_plan(steps, n_sets):
    """(period, full periods, tail): `steps` steps as replays of one graph of `period` steps (a
    multiple of n_sets, so every replay starts at input set 0) plus one graph of the `tail` steps
    left over.  Up to GRAPH_MAX_STEPS steps form a single graph of exactly `steps` steps."""
    if steps <= GRAPH_MAX_STEPS:
        return steps, 1, 0
    period = max(n_sets, GRAPH_MAX_STEPS // n_sets * n_sets)
    return period, steps // period, steps % period


def timed_steps(steps, n_sets, stream, streams, enqueue, barrier, graphs=True, clocks=None):
    """Device milliseconds per step for exactly `steps` steps, step i enqueued by enqueue(i, st)
    on streams[i % len(streams)].  With graphs, the steps are replayed from CUDA graphs of up to
    GRAPH_MAX_STEPS steps each (captured and replayed before timing), so the host launches a
    handful of graphs and the figure does not depend on the host's launch rate; CUDA events on
    `stream` bracket the region, with a barrier and a device synchronisation on both sides.
    `clocks` (a ClockSampler) samples the GPU clocks while the timed region runs."""
    import contextlib

    sampling = clocks if clocks is not None else contextlib.nullcontext()
    if graphs:
        period, full, tail = step_plan(steps, n_sets)
        single = full == 1 and not tail
        # a single graph carries its own timing events as its first and last nodes, so the figure
        # is the device time of exactly its steps (without the host's graph-launch latency, which
        # a few-step window would not amortise); several graphs are timed around their replays
        ev0 = torch.cuda.Event(enable_timing=True, external=single)
        ev1 = torch.cuda.Event(enable_timing=True, external=single)
        g_period = capture_steps(0, period, stream, streams, enqueue, events=(ev0, ev1) if single else None)
        g_tail = capture_steps(full * period, tail, stream, streams, enqueue) if tail else None
        with torch.cuda.stream(stream):  # untimed replays: every node has run, the graph is resident
            for _ in range(3 if single else 1):
                g_period.replay()
            if g_tail is not None:
                g_tail.replay()
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        with sampling, torch.cuda.stream(stream):
            if not single:
                ev0.record(stream)
            for _ in range(full):
                g_period.replay()
            if g_tail is not None:
                g_tail.replay()
            if not single:
                ev1.record(stream)
            torch.cuda.synchronize()
    else:
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        sampling.__enter__()
        ev0.record(stream)
        for st in streams:
            if st is not stream:
                st.wait_event(ev0)
        for i in range(steps):
            st = streams[i % len(streams)]
            with torch.cuda.stream(st):
                enqueue(i, st)
        for st in streams:
            if st is not stream:
                stream.wait_stream(st)
        ev1.record(stream)
        torch.cuda.synchronize()
        sampling.__exit__(None, None, None)
    barrier()
    return ev0.elapsed_time(ev1) / steps


def input_sets(args, wl):
    """(input sets rotated over, batches in flight) of the timed region: enough sets that their
    compulsory bytes exceed L2 three times over (3 to 8), rounded up to a multiple of the batches in
    flight so that set j always runs on stream j % inflight."""
    n_sets = max(3, min(8, -(-3 * L2_BYTES // max(step_bytes(wl), 1))))
    if args.sets:
        n_sets = args.sets
    inflight = max(1, args.inflight)
    return -(-n_sets // inflight) * inflight, inflight


def run_config(args, wl):
    """The line's `config`: the workload and how the GPU arm runs it.  Both arms print this same
    object, so the two lines describe one configuration."""
    n_sets, inflight = input_sets(args, wl)
    return {"workload": wl.name, "batch": wl.T, "L": wl.L, "K": wl.K, "H_idx": wl.H_idx,
            "d_idx": wl.d_idx, "idx_dtype": wl.idx_dtype, "H": wl.H, "D_qk": wl.D_qk,
            "D_v": wl.D_v, "kv_dtype": wl.kv_dtype, "cuda_graph": not args.no_graph,
            "batches_in_flight": inflight,
            "l2": f"rotating {n_sets} input sets, {n_sets * step_bytes(wl) / 1e6:.0f} MB compulsory bytes > 129 MB L2"}


def run_reference(args, wl):
    """The oracle as it stands, on the host cores: each step is one query of the workload through
    the whole chain (fp64 scores, full-sort Top-K, exact attention)."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle

    cpu = synth.make_inputs(wl)
    a = synth.to_numpy_bits(cpu)
    ch = oracle.Chain(a, L=wl.L, K=wl.K, q_per_seq=wl.q_per_seq, q_pos0=wl.q_pos0,
                      idx_dtype=wl.idx_dtype, kv_dtype=wl.kv_dtype, sm_scale=wl.sm_scale)
    for i in range(args.warmup):
        oracle.chain_query(ch, i % wl.T, wl.D_v)
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle.chain_query(ch, i % wl.T, wl.D_v)
    el = time.perf_counter() - t0
    rate = args.steps / el
    cores = blas_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": "queries/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "config": run_config(args, wl),
        "cpu_baseline": {"value": rate, "unit": "queries/s", "cores": cores, "kind": "oracle",
                         "sample": f"one query of {wl.name} per step, {args.steps} steps "
                                   f"(fp64 numpy oracle, BLAS threads={cores})"},
        "e2e": {"value": rate, "unit": "queries/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, wl):
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    import top_sparse_attention_gb300 as dsa
    from top_sparse_attention_gb300 import build as _build

    _build.build()

    # input sets: each rank draws its own (seed offset by rank) and rotates over R of them
    per_step = step_bytes(wl)
    n_sets, inflight = input_sets(args, wl)
    cpu_sets = [synth.make_inputs(wl, seed_offset=rank_seed_offset(rank, i)) for i in range(n_sets)]
    dev_sets = [{k: (v.to(dev) if v is not None else None) for k, v in s.items()} for s in cpu_sets]
    calls = [dsa.call_from_tensors(s, K=wl.K, sm_scale=wl.sm_scale, q_per_seq=wl.q_per_seq,
                                   q_pos0=wl.q_pos0) for s in dev_sets]
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()

    # warm-up (also the first call of every set outside any graph capture)
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, n_sets)):
            calls[i % n_sets](stream)
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()

    # with inflight > 1, consecutive steps (independent batches) go to different streams so that
    # one batch's selection and attention overlap the next batch's scoring
    streams = [stream] + [torch.cuda.Stream(device=dev) for _ in range(inflight - 1)]

    def enqueue(i, st):
        calls[i % n_sets](st)

    clocks = ClockSampler(dev.index)
    ms = timed_steps(args.steps, n_sets, stream, streams, enqueue, barrier, graphs=not args.no_graph,
                     clocks=clocks)
    ms = max_over_ranks(ms, world, dev)
    # the same steps one batch at a time (one stream), reported beside the headline
    serial = None
    if inflight > 1:
        ms_serial = timed_steps(args.steps, n_sets, stream, [stream], enqueue, barrier,
                                graphs=not args.no_graph)
        ms_serial = max_over_ranks(ms_serial, world, dev)
        serial = {"value": wl.T * world / (ms_serial * 1e-3), "unit": "queries/s",
                  "ms_per_step": ms_serial, "steps": args.steps, "batches_in_flight": 1}
    err = dsa.dsa_get_device_error(stream)
    queries = wl.T * world
    value = queries / (ms * 1e-3)
    # kernels per step as the library plans them (index score, Top-K kernels, attention and the
    # combine kernel when K is split over CTAs, per slice of queries)
    launches_per_step = calls[0].launches

    # ---- per-kernel durations (component entry points, same kernels and launch shapes), events
    # on the launching stream over `reps` launches each
    if args.attn_kernel != "auto":  # the fused chain keeps the library's choice either way
        from top_sparse_attention_gb300 import _native as N
        dsa.dsa_set_attn_kernel(N.DSA_ATTN_TCGEN05)
    kern = kernel_times(dsa, wl, dev_sets, stream, reps=max(5, min(200, args.steps)))
    if args.attn_kernel != "auto":
        dsa.dsa_set_attn_kernel(N.DSA_ATTN_AUTO)
    if wl.q_pos0 < 0:
        peak, peak_kind = measured_hbm_peak()
        a_bytes = index_score_bytes(wl, wl.T)
        achieved = a_bytes / (kern["index_score_us"] * 1e-6) / 1e9
        roofline = {"bound": "hbm", "kernel": "index_score", "achieved": achieved, "peak": peak,
                    "unit": "GB/s", "frac": achieved / peak, "peak_kind": peak_kind,
                    "algorithmic_bytes": a_bytes, "traffic": profiled_traffic(wl.name)}
    else:
        peak, peak_kind = measured_bf16_peak()
        flops = index_score_flops(wl)
        achieved = flops / (kern["index_score_us"] * 1e-6) / 1e12
        roofline = {"bound": "tensor", "kernel": "index_score", "achieved": achieved, "peak": peak,
                    "unit": "TFLOP/s", "frac": achieved / peak, "peak_kind": peak_kind,
                    "algorithmic_flops": flops, "traffic": profiled_traffic(wl.name)}

    # ---- end to end through the C ABI with host buffers (pinned), copies inside the timed region
    e2e = end_to_end(dsa, wl, cpu_sets, dev_sets, stream, steps=args.steps, inflight=inflight)

    line = None
    if rank == 0:
        chain_gbs = per_step * world / (ms * 1e-3) / 1e9
        cpu_base = None
        if world == 1 and not args.no_cpu_baseline:
            rate, n, el = cpu_oracle_rate(wl, cpu_sets[0], args.cpu_seconds)
            cores = blas_threads()
            cpu_base = {"value": rate, "unit": "queries/s", "cores": cores, "kind": "oracle",
                        "sample": f"{n} queries of {wl.name} in {el:.1f} s (fp64 numpy oracle, BLAS threads={cores})"}
        line = {
            "metric": METRIC, "value": value, "unit": "queries/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if wl.idx_dtype == "bf16" else "fp8(e4m3)+bf16",
            "data": "synthetic (seeded N(0,1) inputs, U(0,1) head weights)",
            "config": run_config(args, wl),
            "hbm_gbs": chain_gbs, "hbm_frac_of_8tbs": chain_gbs / NOMINAL_HBM_GBS,
            "hbm_frac_of_measured": chain_gbs / peak,
            "roofline": roofline,
            "kernels_us": kern,
            "kernels_note": "each component entry timed alone (CUDA graph of launches, rotating input sets); "
                            "the index score on every resident slot, as dsa_index_score runs it"
                            + ("; attention on the tensor-memory kernel" if args.attn_kernel != "auto" else ""),
            "next_rows": ({"quant_append": quant_append_time(dsa, wl, stream),
                           "paged_chain": paged_chain_time(dsa, wl, dev_sets, stream)} if wl.q_pos0 < 0 else {}),
            "serial": serial,
            "cpu_baseline": cpu_base,
            "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks.summary(),
            "device_error": err,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def kernel_times(dsa, wl, dev_sets, stream, reps):
    """Average device time of each step's kernel(s), launched alone through the component entry
    points on the same inputs, rotating over the input sets (so the keys come from DRAM).  Each
    component's `reps` launches are captured in one CUDA graph and timed with CUDA events on the
    launching stream around its replay, so the figure is device time without host launch gaps.
    The index score runs here as dsa_index_score does, on every resident slot; inside the fused
    chain a short decode launch takes one CTA per SM (see index_score.cu), which is slower alone
    and faster with batches in flight."""
    n = len(dev_sets)
    L = wl.L
    dev = dev_sets[0]["q"].device
    scores = [torch.empty(wl.T, dsa.ld_scores_for(L), dtype=torch.float32, device=dev) for s in dev_sets]
    idx = [torch.empty(wl.T, wl.K, dtype=torch.int32, device=dev) for s in dev_sets]
    from top_sparse_attention_gb300 import _native

    topk_ws = torch.zeros(max(16, _native.lib.dsa_topk_workspace_size(wl.T, L, wl.K)), dtype=torch.uint8, device=dev)
    attn_ws_bytes = _native.lib.dsa_sparse_attn_workspace_size(wl.T, wl.H, wl.K, wl.D_v)
    attn_ws = torch.zeros(max(16, attn_ws_bytes), dtype=torch.uint8, device=dev) if attn_ws_bytes else None
    out = {}

    def timed(fn):
        with torch.cuda.stream(stream):
            for i in range(3):
                fn(i % n)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(reps):
                fn(i % n)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g.replay()
            torch.cuda.synchronize()
            e0.record(stream)
            g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / reps

    def score(i):
        s = dev_sets[i]
        dsa.dsa_index_score(s["q_idx"], s["w"], s["k_idx"], q_idx_sf=s["q_idx_sf"], k_idx_sf=s["k_idx_sf"],
                            q_per_seq=wl.q_per_seq, q_pos0=wl.q_pos0, n_valid=s["n_valid"], scores=scores[i],
                            stream=stream)

    def topk(i):
        dsa.dsa_topk(scores[i], wl.K, L=L, q_per_seq=wl.q_per_seq, q_pos0=wl.q_pos0,
                     n_valid=dev_sets[i]["n_valid"], idx=idx[i], ws=topk_ws, stream=stream)

    outs = [torch.empty(wl.T, wl.H, wl.D_v, dtype=torch.bfloat16, device=s["q"].device) for s in dev_sets]
    lses = [torch.empty(wl.T, wl.H, dtype=torch.float32, device=s["q"].device) for s in dev_sets]
    def attn(i):
        s = dev_sets[i]
        dsa.dsa_sparse_attn(s["q"], s["kv"], idx[i], sm_scale=wl.sm_scale, kv_v=s["kv_v"], kv_scale=s["kv_scale"],
                            D_v=wl.D_v, q_per_seq=wl.q_per_seq, out=outs[i], lse=lses[i], ws=attn_ws,
                            stream=stream)

    out["index_score_us"] = timed(score)
    out["topk_us"] = timed(topk)
    out["sparse_attn_us"] = timed(attn)
    return out


def quant_append_time(dsa, wl, stream, rows=65536, reps=20):
    """The cache writer (the row of the method just before the chain): one chunk of `rows` new
    tokens, bf16 indexer-key rows (d_idx) to MXFP8 and bf16 latent rows (D_qk) to FP8, written
    into caches of `rows` rows.  Two source sets rotate (their bytes exceed L2); timed like the
    kernels (CUDA graph replay, events on the launching stream).  Bytes: the bf16 sources read
    plus the codes and scales written."""
    dev = torch.device("cuda", torch.cuda.current_device())
    g = torch.Generator(device=dev).manual_seed(7)
    k_src = [torch.randn(rows, wl.d_idx, device=dev, generator=g).to(torch.bfloat16) for _ in range(2)]
    v_src = [torch.randn(rows, wl.D_qk, device=dev, generator=g).to(torch.bfloat16) for _ in range(2)]
    k_codes = torch.empty(rows, wl.d_idx, dtype=torch.uint8, device=dev)
    k_sf = torch.empty(rows, wl.d_idx // 32, dtype=torch.uint8, device=dev)
    v_codes = torch.empty(rows, wl.D_qk, dtype=torch.uint8, device=dev)
    v_scale = torch.empty(rows, dtype=torch.float32, device=dev)
    dst = torch.arange(rows, dtype=torch.int64, device=dev)

    def mx(i):
        dsa.dsa_quantize_mxfp8(k_src[i], codes=k_codes, sf=k_sf, dst_rows=dst, stream=stream)

    def fp8(i):
        dsa.dsa_quantize_fp8_rows(v_src[i], codes=v_codes, scales=v_scale, dst_rows=dst, stream=stream)

    def step(i):
        mx(i)
        fp8(i)

    def timed(fn):
        with torch.cuda.stream(stream):
            for i in range(3):
                fn(i % 2)
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for i in range(reps):
                fn(i % 2)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            gr.replay()
            torch.cuda.synchronize()
            e0.record(stream)
            gr.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / reps

    us = timed(step)
    nbytes = rows * (2 * wl.d_idx + 2 * wl.D_qk + wl.d_idx + wl.d_idx // 32 + wl.D_qk + 4 + 8)
    peak, kind = measured_hbm_peak()
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"rows": rows, "us": us, "mxfp8_us": timed(mx), "fp8_rows_us": timed(fp8), "bytes": nbytes,
            "achieved_gbs": gbs, "peak_gbs": peak, "frac": gbs / peak, "peak_kind": kind,
            "launches_per_chunk": 2}


def paged_chain_time(dsa, wl, dev_sets, stream, block_size=64, steps=500, max_sets=3):
    """The fused chain over paged caches (the N2 row of the scope table): each input set's caches
    copied into pools of `block_size`-position blocks in a random order and read through a block
    table.  One batch at a time, CUDA-graph replay rotating over the sets; compare with `serial`
    (the same chain over contiguous caches)."""
    if wl.q_pos0 >= 0:
        return None
    dev = dev_sets[0]["q"].device
    per_seq = -(-wl.L // block_size)
    n_seq = wl.n_seq
    n_blocks = n_seq * per_seq + 7
    sets = dev_sets[:max_sets]
    g = torch.Generator().manual_seed(17)
    calls, graphs = [], []
    for s in sets:
        table = torch.randperm(n_blocks, generator=g)[: n_seq * per_seq].to(torch.int32).reshape(n_seq, per_seq)
        flat = table.reshape(-1).to(dev).long()
        pools = {}
        for key in ("k_idx", "k_idx_sf", "kv", "kv_v", "kv_scale"):
            c = s[key]
            if c is None:
                pools[key] = None
                continue
            rest = tuple(c.shape[2:])
            pad = per_seq * block_size - wl.L
            if pad:
                c = torch.cat([c, torch.zeros((n_seq, pad) + rest, dtype=c.dtype, device=dev)], dim=1)
            pool = torch.zeros((n_blocks, block_size) + rest, dtype=c.dtype, device=dev)
            pool[flat] = c.reshape((n_seq * per_seq, block_size) + rest)
            pools[key] = pool.reshape((n_blocks * block_size,) + rest)
        call = dsa.DsaCall(q_idx=s["q_idx"], w=s["w"], k_idx=pools["k_idx"], q=s["q"], kv=pools["kv"], K=wl.K,
                           sm_scale=wl.sm_scale, q_idx_sf=s["q_idx_sf"], k_idx_sf=pools["k_idx_sf"],
                           kv_scale=pools["kv_scale"], kv_v=pools["kv_v"], D_v=wl.D_v, q_per_seq=wl.q_per_seq,
                           q_pos0=wl.q_pos0, n_valid=s["n_valid"], block_table=table.to(dev),
                           block_size=block_size, L=wl.L)
        call._pools = pools  # keep the pools alive with the call
        calls.append(call)
    with torch.cuda.stream(stream):
        for c in calls:
            c(stream)
    torch.cuda.synchronize()
    for c in calls:
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            c(stream)
        graphs.append(gr)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for i in range(3):
            graphs[i % len(graphs)].replay()
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(steps):
            graphs[i % len(graphs)].replay()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return {"block_size": block_size, "ms_per_step": ms, "value": wl.T / (ms * 1e-3), "unit": "queries/s",
            "batches_in_flight": 1, "steps": steps}


def end_to_end(dsa, wl, cpu_sets, dev_sets, stream, steps, inflight=1):
    """queries/s through the C ABI with each step's query-side inputs (q, q_idx (+scales), w)
    copied from pinned host memory and its outputs (out, lse) read back, inside the timed region.
    The caches are device-resident state, as in decode, rotating over the same input sets as the
    device timing (their bytes exceed L2).  Inputs sit in one pinned host buffer and one device
    buffer per set, outputs likewise, so a step is one host-to-device copy, the fused call
    (dsa_decode) and one device-to-host copy.  Copies run on their own streams so that
    neighbouring steps' copies overlap the calls, as a serving loop would run them; with
    inflight > 1 consecutive steps' calls run on different streams, as in the device timing.
    Exactly `steps` steps are timed, replayed from the same graph plan as the device timing
    (step_plan); the figure is the larger of the event time and the host's wall time."""
    keys_in = [k for k in ("q", "q_idx", "q_idx_sf", "w") if cpu_sets[0][k] is not None]

    def packed(tensors, device, pinned):
        offs, off = {}, 0
        for k, t in tensors.items():
            nb = t.numel() * t.element_size()
            offs[k] = (off, nb, t.dtype, t.shape)
            off += (nb + 255) // 256 * 256
        buf = torch.empty(off, dtype=torch.uint8, device=device)
        if pinned:
            buf = buf.pin_memory()
        views = {k: buf[o:o + nb].view(dt).view(sh) for k, (o, nb, dt, sh) in offs.items()}
        return buf, views

    dev0 = dev_sets[0]["q"].device
    out_like = {"out": torch.empty(wl.T, wl.H, wl.D_v, dtype=torch.bfloat16),
                "lse": torch.empty(wl.T, wl.H, dtype=torch.float32)}
    sets = []
    for cpu, dev in zip(cpu_sets, dev_sets):
        hin, hv = packed({k: cpu[k] for k in keys_in}, "cpu", True)
        din, dv = packed({k: cpu[k] for k in keys_in}, dev0, False)
        for k in keys_in:
            hv[k].copy_(cpu[k])
        hout, hov = packed(out_like, "cpu", True)
        dout, dov = packed(out_like, dev0, False)
        tensors = dict(dev)
        tensors.update(dv)
        call = dsa.call_from_tensors(tensors, K=wl.K, sm_scale=wl.sm_scale, q_per_seq=wl.q_per_seq,
                                     q_pos0=wl.q_pos0, out=dov["out"], lse=dov["lse"])
        with torch.cuda.stream(stream):
            din.copy_(hin, non_blocking=True)
            for _ in range(2):
                call(stream)
        torch.cuda.synchronize()
        # the tuple keeps every buffer the captured graphs point at (the call owns its workspace):
        # a graph holds raw pointers, and each capture empties torch's allocator cache
        sets.append((hin, din, hout, dout, call))
    h2d, d2h = sets[0][0].numel(), sets[0][2].numel()
    n = len(sets)
    s_in, s_out = torch.cuda.Stream(device=dev0), torch.cuda.Stream(device=dev0)
    comp = [torch.cuda.Stream(device=dev0) for _ in range(inflight)]

    def capture(first, count):
        """Steps first .. first+count-1 in one graph: step i's input copy on s_in, its call on
        comp[i % inflight], its output copy on s_out.  A set's input copy waits for the set's
        previous call (which read those inputs) and its call for the set's previous output copy
        (which read those outputs)."""
        ev_in, ev_call, ev_out = {}, {}, {}
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fork = torch.cuda.Event()
            fork.record(stream)
            for st in [s_in, s_out] + comp:
                st.wait_event(fork)
            for i in range(first, first + count):
                hin, din, hout, dout, call = sets[i % n]
                sc = comp[i % inflight]
                prev = i - n if i - n >= first else None
                if prev is not None:
                    s_in.wait_event(ev_call[prev])
                with torch.cuda.stream(s_in):
                    din.copy_(hin, non_blocking=True)
                ev_in[i] = torch.cuda.Event()
                ev_in[i].record(s_in)
                sc.wait_event(ev_in[i])
                if prev is not None:
                    sc.wait_event(ev_out[prev])
                call(sc)
                ev_call[i] = torch.cuda.Event()
                ev_call[i].record(sc)
                s_out.wait_event(ev_call[i])
                with torch.cuda.stream(s_out):
                    hout.copy_(dout, non_blocking=True)
                ev_out[i] = torch.cuda.Event()
                ev_out[i].record(s_out)
            for st in [s_in, s_out] + comp:
                stream.wait_stream(st)
        return g

    period, full, tail = step_plan(steps, n)
    g_period = capture(0, period)
    g_tail = capture(full * period, tail) if tail else None
    with torch.cuda.stream(stream):
        g_period.replay()
        if g_tail is not None:
            g_tail.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(full):
            g_period.replay()
        if g_tail is not None:
            g_tail.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    ms = max(e0.elapsed_time(e1), wall * 1e3) / steps
    return {"value": wl.T / (ms * 1e-3), "unit": "queries/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": steps,
            "copies_per_step": {"h2d": 1, "d2h": 1}, "batches_in_flight": inflight,
            "pipelined": "copies of adjacent steps overlap the calls"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--inflight", type=int, default=6,
                    help="independent batches in flight (consecutive steps on different streams)")
    ap.add_argument("--steps", type=int, default=20000)  # ~1 s of decode steps: clock samples
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode_b8_l32k_bf16", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--sets", type=int, default=0, help="input sets to rotate over (0 = auto)")
    ap.add_argument("--no-graph", action="store_true", help="launch through the C ABI each step, no CUDA graph")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--attn-kernel", default="auto", choices=["auto", "tcgen05"],
                    help="attention kernel for the component timings of calls on their own (dsa_set_attn_kernel)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    wl = synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, wl)
    return run_ours(args, wl)


if __name__ == "__main__":
    sys.exit(main())
