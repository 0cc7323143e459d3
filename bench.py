"""Benchmark of the Key-Key block selector hot path on one GB300 (or N replicas).

One step = pool every block of the workload's paged K cache into v_b, then one
decode step of the selector for every request (kk_select_step: anchor, scores,
top-K). The headline workload is the largest that fits one GPU: the 7B-like
long context, 32 requests x 131072 tokens (120 GB of bf16 K in shuffled pages),
pooled with head-variance weights (kk_pool_blocks_weighted), W32 K64. The same
JSON line carries one sub-record per other workload ("workloads"): the 0.5B-like
tiny cache (L2 flushed and warm), the 7B-like cache, the shared pool scored as
one tensor-core product (and its three-level hierarchy), and the 1M-token write
path at block sizes 16 and 128 with coarse means, each with its own roofline
fraction.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 7b-long]
    python bench.py --impl reference   # the fp64 CPU oracle on a bounded sample

Under torchrun (N > 1) each rank runs the headline workload on its own GPU
with its own requests (weak scaling, no collective on the data path); the step
time is the maximum over ranks. Sub-records are measured at N = 1 only.
"""
from __future__ import annotations

import argparse
import concurrent.futures
import dataclasses
import hashlib
import json
import multiprocessing
import os
import re
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "K-pool HBM GB/s (vs ~8 TB/s); blocks scored/s; score+top-K µs/step"
WORKLOADS = {
    "pool": None,  # shared pool of pre-pooled v_b, see run_pool_gpu
    "tiny": synth.tiny_05b,
    "7b": synth.qwen7b,
    "7b-long": synth.qwen7b_long,
    "write16": lambda: synth.write_stress(16),
    "write128": lambda: synth.write_stress(128),
}
WORKLOAD_NAMES = {
    "pool": "shared pool: 256 anchors x 65536 pooled bf16 v_b (D128), 4096 owned blocks per anchor, K128",
    "tiny": "0.5B-like paged K: L24 H2 D64 bs16 fp32, 1 x 4096 tokens, W8 K16, unweighted",
    "7b": "7B-like paged K: L28 H4 D128 bs128 bf16, 8 x 32768 tokens, W16 K32",
    "7b-long": ("7B-like long context: L28 H4 D128 bs128 bf16, 32 x 131072 tokens (120 GB), head-variance "
                "weighted, shuffled pages, W32 K64"),
    "write16": "write path: 2^20 tokens of 7B geometry at block size 16, + coarse means over 64 and 512 blocks",
    "write128": "write path: 2^20 tokens of 7B geometry at block size 128, + coarse means over 64 and 512 blocks",
}
DEFAULT_WORKLOAD = "7b-long"
# sources whose ncu traffic figures are committed under profiles/ (a changed
# source makes the figure stale, and the line then reports traffic null)
PROFILE_SRC = {
    "7b": ["kv_cache_block_gb300/csrc/kk_pool_tma.cu", "kv_cache_block_gb300/csrc/kk_tcgen05.cuh",
           "kv_cache_block_gb300/csrc/kk_device.cuh"],
    "7b-long": ["kv_cache_block_gb300/csrc/kk_pool_tma.cu", "kv_cache_block_gb300/csrc/kk_pool.cu",
                "kv_cache_block_gb300/csrc/kk_tcgen05.cuh", "kv_cache_block_gb300/csrc/kk_device.cuh"],
}
PROFILE_FILE = {"7b": "pool_kernel_7b.md", "7b-long": "weighted_pool_7b_long.md"}
L2_FLUSH_BYTES = 256 << 20  # twice the 129 MB L2
E2E_RING_BYTES = 4 << 30    # pinned staging ring for caches too large to hold on the host


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def rank_spec(spec, rank: int):
    """The shard of one rank under weak scaling: the workload's geometry and
    sizes, with requests of its own (every input drawn from a seed offset by
    the rank). Rank 0 keeps the workload's own seed."""
    return spec if rank == 0 else dataclasses.replace(spec, seed=spec.seed + 7919 * rank)


def max_over_ranks(x: float, device=None) -> float:
    """The maximum of ``x`` over the ranks of the default process group (``x``
    itself without one)."""
    import torch
    import torch.distributed as dist

    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_value(units_per_rank: float, steps: int, world: int, max_ms: float) -> float:
    """Whole-job throughput: every rank processed ``units_per_rank`` per step;
    the job took the slowest rank's ``max_ms`` for ``steps`` steps."""
    return world * units_per_rank * steps / (max_ms * 1e-3)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def source_hash(paths) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per pool call of ``workload`` from the committed ncu summary,
    if it was taken on the current kernel sources; else None."""
    if workload not in PROFILE_FILE:
        return None
    path = os.path.join(ROOT, "profiles", PROFILE_FILE[workload])
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    m_h = re.search(r"pool_source_hash:\s*([0-9a-f]+)", text)
    if not m_b or not m_h or m_h.group(1) != source_hash(PROFILE_SRC[workload]):
        return None
    return float(m_b.group(1))


def step_bytes(spec) -> int:
    """Algorithmic bytes of one selector step (anchor, scores, top-K) over
    every request: the W' = min(W, T) anchor token rows of every (layer, head)
    read once, plus every candidate's float32 v_b row; the top-K adds none
    (it is fused with the scores)."""
    w_rows = sum(min(spec.W, int(t)) for t in spec.seq_lens)
    return w_rows * spec.L * spec.H * spec.D * spec.elem_bytes + spec.total_blocks * spec.D * 4


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform

    return platform.processor() or platform.machine()


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 50 ms. The sampler
    is started (first sample seen) before the caller's timed region; only the
    samples taken inside the window passed to ``window`` are summarised."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 50

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []  # (perf_counter seconds, csv line)
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.PERIOD_MS)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            deadline = time.perf_counter() + 5.0
            while not self.lines and time.perf_counter() < deadline and self.proc.poll() is None:
                time.sleep(0.01)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def window(self, t0: float, t1: float):
        self.t0, self.t1 = t0, t1

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(2.0 * self.PERIOD_MS / 1e3)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        return summarize_clocks(self.lines, self.t0, self.t1)


def summarize_clocks(lines, t0=None, t1=None):
    """Median SM clock, max clock and throttle reasons of the samples taken in
    [t0, t1] (all samples when no window is given). When the window is shorter
    than the sampling period and holds none, the first sample after it is
    used and ``in_window`` says so."""
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    parsed = []
    for t, line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) != 6:
            continue
        try:
            sm, mx = float(parts[0]), float(parts[1])
        except ValueError:
            continue
        parsed.append((t, sm, mx, [n for n, v in zip(names, parts[2:]) if v.lower() == "active"]))
    in_window = True
    sel = parsed
    if t0 is not None and t1 is not None:
        sel = [x for x in parsed if t0 <= x[0] <= t1]
        if not sel:
            in_window = False
            sel = [x for x in parsed if x[0] > t1][:1]
    if not sel:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
    reasons = sorted({n for x in sel for n in x[3]})
    return {"sm_mhz": statistics.median(x[1] for x in sel), "sm_max_mhz": max(x[2] for x in sel),
            "reasons": reasons, "samples": len(sel), "in_window": in_window}


# --------------------------------------------------------------------------
# CPU oracle leg: a bounded sample of the workload on every host core
# --------------------------------------------------------------------------

_SAMPLE = None  # per worker process: (kc view, sample spec)


def _sample_spec(spec, blocks: int):
    """One request of ``blocks`` full blocks with the workload's geometry,
    noise and weighting (its Keys are the workload's first request's first
    blocks when copied from the device)."""
    return synth.CacheSpec(name=spec.name + "-sample", L=spec.L, H=spec.H, D=spec.D, bs=spec.bs, dtype=spec.dtype,
                           seq_lens=[spec.bs * blocks], num_topics=spec.num_topics, scale=spec.scale, W=spec.W,
                           K=spec.K, seed=spec.seed, sigma_range=spec.sigma_range, weighted=spec.weighted)


def _oracle_worker_init(path: str, spec_args: dict):
    global _SAMPLE
    sub = synth.CacheSpec(**spec_args)
    flat = np.load(path)
    _SAMPLE = (synth.view_paged(flat, sub), sub)


def _oracle_worker_run(budget_s: float):
    """The oracle as it stands on this worker's copy of the sample request:
    (for weighted workloads) the request's head-variance weights, then every
    block pooled, repeated for ``budget_s`` seconds; then one selector step.
    Returns (bytes of K pooled, seconds)."""
    from oracle import kk_oracle as ko

    kc, sub = _SAMPLE
    T = int(sub.seq_lens[0])
    per_pass = T * sub.L * sub.H * sub.D * sub.elem_bytes
    t0 = time.perf_counter()
    done = 0
    while True:
        w = ko.head_variance_weights(kc, sub.pages, T, sub.bs) if sub.weighted else None
        vb = ko.pool_blocks(kc, sub.pages, sub.n_valid, None if w is None else [w],
                            None if w is None else [0] * len(sub.pages))
        done += per_pass
        if time.perf_counter() - t0 >= budget_s:
            break
    va = ko.anchor(kc, sub.pages, T, sub.bs, sub.W, None if w is None else w)
    vb_table = np.zeros((sub.num_pages, sub.D))
    vb_table[sub.pages] = vb
    ko.score_topk(vb_table, sub.pages, va, sub.K)
    return done, time.perf_counter() - t0


class OracleSampler:
    """A pool of spawned worker processes (one per host core), each holding a
    copy of one sample request of the workload; ``step`` runs the oracle on
    every worker for a bounded time and returns GB/s of K pooled."""

    def __init__(self, spec, flat: np.ndarray, sub, workers: int = 0):
        self.cores = workers or host_cores()
        self.tmp = tempfile.TemporaryDirectory(prefix="kk_oracle_")
        path = os.path.join(self.tmp.name, "sample.npy")
        np.save(path, flat)
        args = {f.name: getattr(sub, f.name) for f in dataclasses.fields(sub)}
        # spawned (never forked after CUDA is initialised); a worker that
        # fails to start breaks the pool and raises instead of being respawned
        self.pool = concurrent.futures.ProcessPoolExecutor(
            self.cores, mp_context=multiprocessing.get_context("spawn"), initializer=_oracle_worker_init,
            initargs=(path, args))
        self.sub = sub
        self.step(0.0)  # start every worker (spawn, load the sample) outside the timed steps
        self.desc = (f"every one of {self.cores} host cores ({cpu_model()}) runs the fp64 numpy oracle as it stands "
                     f"on its own copy of one request of {len(sub.pages)} full blocks of the workload's geometry "
                     f"({'head-variance weights over the request, then ' if sub.weighted else ''}every block pooled, "
                     f"repeated for the time budget; then one selector step)")

    def step(self, budget_s: float):
        t0 = time.perf_counter()
        res = list(self.pool.map(_oracle_worker_run, [budget_s] * self.cores, timeout=budget_s * 20 + 120))
        wall = time.perf_counter() - t0
        done = sum(b for b, _ in res)
        return done / wall / 1e9, wall

    def close(self):
        self.pool.shutdown(wait=True, cancel_futures=True)
        self.tmp.cleanup()


def sample_from_numpy(spec, blocks: int = 4):
    sub = _sample_spec(spec, blocks)
    return synth.gen_paged_numpy(sub), sub


def sample_from_device(spec, storage, blocks: int = 4):
    """The first ``blocks`` blocks of the workload's first request, copied back
    from the device cache into a one-request sample laid out as the workload."""
    import torch

    sub = _sample_spec(spec, blocks)
    L, P, H, bs, D = spec.shape
    pages = torch.as_tensor(np.asarray(spec.pages_of(0)[:blocks], dtype=np.int64), device=storage.device)
    sL, sP, sH, sT = spec.strides()
    view = storage.as_strided((L, P, H, bs, D), (sL, sP, sH, sT, 1))
    blk = view.index_select(1, pages).contiguous().cpu().numpy()  # [L][blocks][H][bs][D]
    if spec.dtype == "bf16":
        blk = blk.view(np.uint16)
    flat = np.empty(sub.storage_elems(), dtype=blk.dtype)
    synth.view_paged(flat, sub)[...] = blk[:, : sub.num_pages]
    return flat, sub


# --------------------------------------------------------------------------
# GPU timing helpers
# --------------------------------------------------------------------------


def graph_time_us(fn, dev, stream, reps: int = 20, replays: int = 10):
    """Microseconds per call of `fn` captured `reps` times in one CUDA graph,
    replayed `replays` times (None if capture fails)."""
    import torch

    try:
        g = torch.cuda.CUDAGraph()
        s2 = torch.cuda.Stream(dev)
        s2.wait_stream(stream)
        with torch.cuda.stream(s2):
            fn()
            with torch.cuda.graph(g, stream=s2):
                for _ in range(reps):
                    fn()
        torch.cuda.synchronize(dev)
        g.replay()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(replays):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) * 1e3 / (reps * replays)
    except Exception as exc:  # noqa: BLE001
        print(f"cuda graph capture failed: {exc}", file=sys.stderr)
        return None


def b2b_us(fn, dev, stream, n: int = 200, warm: int = 5):
    """Microseconds per call of ``fn`` issued back to back ``n`` times."""
    import torch

    for _ in range(warm):
        fn()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        fn()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) * 1e3 / n


class L2Flush:
    """Evicts L2 between timed calls by reading a buffer twice its size. A
    read leaves clean lines behind; a flush that wrote the buffer would leave
    L2 full of dirty lines, and the timed call would pay for writing them back
    (about 129 MB, some 19 us of HBM write time)."""

    def __init__(self, dev):
        import torch

        self.buf = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def __call__(self):
        self.buf.sum()


def per_call_ms(fn, dev, stream, n: int, warm: int, flush=None):
    """CUDA-event time of each of ``n`` calls of ``fn``; with ``flush`` (an
    L2Flush) L2 is evicted before every call, outside the timed interval."""
    import torch

    for _ in range(warm):
        fn()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for i in range(n):
        if flush is not None:
            flush()
        ev[i][0].record(stream)
        fn()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    return [a.elapsed_time(b) for a, b in ev]


class PagedRun:
    """A synthetic paged workload on the device with its pool and select calls."""

    def __init__(self, spec, dev):
        import torch

        from kv_cache_block_gb300 import kk

        self.kk, self.spec, self.dev = kk, spec, dev
        self.storage = synth.gen_paged_cuda(spec, device=dev)
        i32 = lambda a: torch.as_tensor(np.ascontiguousarray(a), dtype=torch.int32, device=dev)  # noqa: E731
        self.pages, self.offsets = i32(spec.pages), i32(spec.offsets)
        self.seq_lens, self.n_valid = i32(spec.seq_lens), i32(spec.n_valid)
        self.desc = kk.kcache_desc(self.storage, kk.KK_F32 if spec.dtype == "f32" else kk.KK_BF16, spec.L, spec.H,
                                   spec.D, spec.bs, spec.num_pages, spec.strides())
        self.bt = kk.BlockTable(self.pages, self.offsets, self.seq_lens, max(spec.nb))
        self.vb = torch.zeros((spec.num_pages, spec.D), device=dev)
        self.idx = torch.zeros((spec.R, spec.K), dtype=torch.int32, device=dev)
        self.top = torch.zeros((spec.R, spec.K), device=dev)
        self.head_w = torch.zeros((spec.R, spec.L * spec.H), device=dev) if spec.weighted else None
        self.ws = None
        if spec.weighted:
            self.ws = torch.empty(kk.kk_head_variance_workspace_bytes(self.desc, spec.total_blocks, spec.R),
                                  dtype=torch.uint8, device=dev)
        # kernels launched by one pool call (the weighted pool: slice sums,
        # variances, weights, combine)
        self.pool_launches = 4 if spec.weighted else 1
        # the workspace that lets very long requests split over several clusters
        nws = kk.kk_select_step_workspace_bytes(spec.R, max(spec.nb), spec.K)
        self.step_ws = torch.zeros(nws, dtype=torch.uint8, device=dev) if nws else None  # zeroed once
        # the anchor ring of the last W tokens (filled from the cache once the
        # cache is written; kept by kk_append_tokens in the decode step)
        self.ring = kk.AnchorRing(spec.R, spec.W, spec.D, device=dev)

    def fill_ring(self):
        self.kk.kk_anchor_ring_fill(self.desc, self.bt, self.ring, head_w=self.head_w)

    def pool(self):
        sp = self.spec
        if sp.weighted:
            self.kk.kk_pool_blocks_weighted(self.desc, self.bt, sp.total_blocks, self.head_w, self.vb, self.ws)
        else:
            self.kk.kk_pool_blocks(self.desc, self.pages, self.n_valid, self.vb)

    def select(self):
        sp = self.spec
        self.kk.kk_select_step(self.desc, self.bt, sp.W, self.vb, sp.K, self.idx, self.top, head_w=self.head_w,
                               workspace=self.step_ws)

    def select_ring(self):
        sp = self.spec
        self.kk.kk_select_step(self.desc, self.bt, sp.W, self.vb, sp.K, self.idx, self.top, head_w=self.head_w,
                               ring=self.ring, workspace=self.step_ws)


def select_record(run, dev, stream, peak_gbs: float, ring: bool = False):
    """Latency of one selector step over all requests (anchor, scores, top-K
    in one launch), back to back and as a CUDA graph, with its roofline
    fraction against the step's algorithmic bytes (the anchor's token rows
    and every candidate's v_b row read once). With ``ring`` the anchor comes
    from the anchor ring (W rows of D floats a request) instead of the
    token rows; the fraction keeps the same algorithmic bytes."""
    sp = run.spec
    fn = run.select_ring if ring else run.select
    if ring:
        run.fill_ring()
    b2b = b2b_us(fn, dev, stream)
    graph = graph_time_us(fn, dev, stream)
    nbytes = step_bytes(sp)
    frac = lambda us: None if us is None else nbytes / (us * 1e-6) / 1e9 / peak_gbs  # noqa: E731
    return {"us_back_to_back": b2b, "us_cuda_graph": graph, "algorithmic_bytes": nbytes,
            "roofline_frac_back_to_back": frac(b2b), "roofline_frac_cuda_graph": frac(graph),
            "blocks_scored_per_s_cuda_graph": None if graph is None else sp.total_blocks / (graph * 1e-6),
            "anchor": "anchor ring (kk_append_tokens / kk_anchor_ring_fill)" if ring else "K cache token rows"}


def pool_record(run, dev, stream, peak_gbs: float, steps: int, warmup: int, flush=None):
    ms = per_call_ms(run.pool, dev, stream, steps, warmup, flush)
    med = statistics.median(ms)
    gbs = run.spec.k_bytes() / (med * 1e-3) / 1e9
    return {"us": med * 1e3, "gbs": gbs, "frac": gbs / peak_gbs, "calls": steps}


# --------------------------------------------------------------------------
# headline workload
# --------------------------------------------------------------------------


def run_main(args, spec, rank, world, local_rank, peak_gbs):
    import torch

    from kv_cache_block_gb300 import kk

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    run = PagedRun(spec, dev)
    stream = torch.cuda.current_stream(dev)

    for _ in range(max(args.warmup, 3)):
        run.pool()
        run.select()
    torch.cuda.synchronize(dev)
    if kk.kk_device_error() != 0:
        raise RuntimeError("device error during warm-up")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local_rank) as clocks:
        t_start = time.perf_counter()
        for i in range(args.steps):
            ev[i][0].record(stream)
            run.pool()
            ev[i][1].record(stream)
            run.select()
            ev[i][2].record(stream)
        torch.cuda.synchronize(dev)
        t_end = time.perf_counter()
        clocks.window(t_start, t_end)
    if world > 1:
        torch.distributed.barrier()
    pool_ms = [a.elapsed_time(b) for a, b, _ in ev]
    sel_ms = [b.elapsed_time(c) for _, b, c in ev]
    total_ms = max_over_ranks(ev[0][0].elapsed_time(ev[-1][2]), dev)
    if kk.kk_device_error() != 0:
        raise RuntimeError("device error during the timed region")
    out = {"pool_ms": statistics.mean(pool_ms), "select_ms": statistics.mean(sel_ms), "total_ms": total_ms,
           "wall_s": t_end - t_start, "clocks": clocks.summary(),
           "launches": (run.pool_launches + 1) * args.steps}
    if rank == 0:
        out.update(main_extras(args, run, dev, stream, peak_gbs))
    return out, run


def main_extras(args, run, dev, stream, peak_gbs):
    """The selector step's latency on its own (one launch, back to back and
    as a CUDA graph; as two launches), the stability-filtered step, the
    hierarchical selection and a whole decode step with the write side."""
    import torch

    from kv_cache_block_gb300 import kk

    sp = run.spec
    out = {"select": select_record(run, dev, stream, peak_gbs),
           "select_ring": select_record(run, dev, stream, peak_gbs, ring=True)}
    va = torch.zeros((sp.R, sp.D), device=dev)

    def anchor_then_score():
        kk.kk_anchor(run.desc, run.bt, sp.W, va, head_w=run.head_w)
        kk.kk_score_topk(run.vb, run.bt, va, sp.K, run.idx, top_scores=run.top)

    out["two_launch_us"] = graph_time_us(anchor_then_score, dev, stream)
    hist = torch.zeros(sp.total_blocks, dtype=torch.int32, device=dev)
    stab = torch.zeros(sp.total_blocks, device=dev)

    def select_stable(ring=None):
        kk.kk_select_step_stable(run.desc, run.bt, sp.W, run.vb, sp.K, 20, 0.5, hist, run.idx, stab=stab,
                                 top_scores=run.top, head_w=run.head_w, ring=ring, workspace=run.step_ws)

    out["stable_us"] = b2b_us(select_stable, dev, stream)
    out["hier"] = hier_record(run, dev, stream)
    out["decode_step_us"] = decode_step_us(run, dev, stream)
    if kk.kk_device_error() != 0:
        raise RuntimeError("device error in the selector legs")
    return out


def hier_record(run, dev, stream):
    """Hierarchical Grid -> Chunk -> Page selection (64 blocks a Chunk, 8
    Chunks a Grid, 50 / 20 / 10 %; coarse levels built once, at write time)
    against the flat selection (kk_score_topk) on the same anchors, back to
    back and as CUDA graphs."""
    import torch

    from kv_cache_block_gb300 import kk

    sp = run.spec
    va = torch.zeros((sp.R, sp.D), device=dev)
    kk.kk_anchor(run.desc, run.bt, sp.W, va, head_w=run.head_w)
    c_max = -(-max(sp.nb) // 64)
    g_max = -(-c_max // 8)
    chunk_reps = torch.zeros((sp.R, c_max, sp.D), device=dev)
    grid_reps = torch.zeros((sp.R, g_max, sp.D), device=dev)
    kk.kk_hier_reps(run.vb, run.bt, 64, 8, chunk_reps, grid_reps)
    h_idx = torch.zeros((sp.R, sp.K), dtype=torch.int32, device=dev)
    f_idx = torch.zeros((sp.R, sp.K), dtype=torch.int32, device=dev)
    h_kept = torch.zeros(sp.R, dtype=torch.int32, device=dev)

    def hier_select():
        kk.kk_hier_select(run.vb, run.bt, chunk_reps, grid_reps, va, 64, 8, (500, 200, 100), h_idx, kept=h_kept,
                          workspace=run.step_ws)

    def flat_select():
        kk.kk_score_topk(run.vb, run.bt, va, sp.K, f_idx, workspace=run.step_ws)

    out = {"hier_us_back_to_back": b2b_us(hier_select, dev, stream),
           "hier_us_cuda_graph": graph_time_us(hier_select, dev, stream),
           "flat_us_back_to_back": b2b_us(flat_select, dev, stream),
           "flat_us_cuda_graph": graph_time_us(flat_select, dev, stream),
           "blocks_kept": int(h_kept.sum().item()), "blocks": sp.total_blocks}
    if kk.kk_device_error() != 0:
        raise RuntimeError("device error in the hierarchy leg")
    return out


def decode_step_us(run, dev, stream):
    """One whole decode step as a CUDA graph: each request's new token
    written into its block with v_b and the anchor ring kept current
    (kk_append_tokens), the stability-filtered selection with the anchor from
    the ring (kk_select_step_stable) and the table of selected pages
    (kk_compact_table); as three launches and as the one fused launch
    (kk_step_options k_new and sel_pages). The token is written at position
    seq_len - 1 (its block exists in this fixed-size cache)."""
    import torch

    from kv_cache_block_gb300 import kk

    sp = run.spec
    k_new = torch.randn((sp.R, sp.L, sp.H, sp.D), device=dev)
    k_new = k_new.to(torch.bfloat16).view(torch.int16) if sp.dtype == "bf16" else k_new
    block_sum = torch.zeros((sp.num_pages, sp.D), device=dev)
    sel_pages = torch.zeros((sp.R, sp.K), dtype=torch.int32, device=dev)
    sel_count = torch.zeros(sp.R, dtype=torch.int32, device=dev)
    hist = torch.zeros(sp.total_blocks, dtype=torch.int32, device=dev)
    stab = torch.zeros(sp.total_blocks, device=dev)

    def decode_step():
        kk.kk_append_tokens(run.desc, run.bt, k_new, block_sum, run.vb, head_w=run.head_w, ring=run.ring)
        kk.kk_select_step_stable(run.desc, run.bt, sp.W, run.vb, sp.K, 20, 0.5, hist, run.idx, stab=stab,
                                 top_scores=run.top, head_w=run.head_w, ring=run.ring, workspace=run.step_ws)
        kk.kk_compact_table(run.idx, run.bt, sel_pages, sel_count=sel_count)

    def decode_step_fused():
        kk.kk_select_step_stable(run.desc, run.bt, sp.W, run.vb, sp.K, 20, 0.5, hist, run.idx, stab=stab,
                                 top_scores=run.top, head_w=run.head_w, ring=run.ring, workspace=run.step_ws,
                                 append=(k_new, block_sum), compact=(sel_pages, None, sel_count))

    run.fill_ring()
    return {"three_launches": graph_time_us(decode_step, dev, stream),
            "fused": graph_time_us(decode_step_fused, dev, stream)}


def e2e_leg(args, run, dev, stream):
    """The step end to end through the public API with host buffers: every
    step copies the whole K cache host -> device, pools it, runs the selector
    and reads v_b, the head weights and the top-K back to pinned host memory.
    A cache larger than E2E_RING_BYTES is streamed from a pinned staging ring
    of that size holding the cache's first bytes (the host keeps no full copy
    of a 120 GB cache); each step still copies every byte of K. This leg runs
    last: afterwards the device cache holds the ring's bytes tiled."""
    import torch

    sp = run.spec
    flat = run.storage.view(torch.uint8)
    nbytes = flat.numel()
    ring = min(nbytes, E2E_RING_BYTES)
    host = torch.empty(ring, dtype=torch.uint8, pin_memory=True)
    host.copy_(flat[:ring])
    pinned = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)  # noqa: E731
    outs = [(run.vb, pinned(run.vb)), (run.idx, pinned(run.idx)), (run.top, pinned(run.top))]
    if run.head_w is not None:
        outs.append((run.head_w, pinned(run.head_w)))
    steps = max(1, min(args.steps, args.e2e_steps))
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        for off in range(0, nbytes, ring):
            n = min(ring, nbytes - off)
            flat[off:off + n].copy_(host[:n], non_blocking=True)
        run.pool()
        run.select()
        for d, h in outs:
            h.copy_(d, non_blocking=True)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    ms = t0.elapsed_time(t1) / steps
    d2h = sum(d.numel() * d.element_size() for d, _ in outs)
    src = ("pinned host copy of the whole cache" if ring == nbytes else
           f"{ring / 2**30:.0f} GiB pinned staging ring holding the cache's first bytes, copied "
           f"{nbytes / ring:.1f} times per step")
    return {"value": sp.k_bytes() / (ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": nbytes,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": steps, "h2d_source": src}


# --------------------------------------------------------------------------
# sub-records: the other workloads
# --------------------------------------------------------------------------


def record_paged(name, dev, stream, peak_gbs, steps, warmup, flush, coarse=False):
    """Pool GB/s (L2 flushed before every call when the cache fits in L2,
    plus the warm figure) and the selector step of one paged workload."""
    import torch

    from kv_cache_block_gb300 import kk

    spec = WORKLOADS[name]()
    run = PagedRun(spec, dev)
    rec = {"workload": WORKLOAD_NAMES[name], "k_bytes": spec.k_bytes(), "blocks": spec.total_blocks,
           "requests": spec.R, "dtype": spec.dtype}
    fits_l2 = spec.k_bytes() < L2_FLUSH_BYTES
    rec["pool"] = pool_record(run, dev, stream, peak_gbs, steps, warmup, flush if fits_l2 else None)
    rec["pool"]["l2"] = "flushed (256 MB read) before every call" if fits_l2 else "inputs larger than L2"
    rec["pool"]["kernel"] = "kk_pool_blocks" + (" (4 launches)" if spec.weighted else "")
    if fits_l2:
        warm = pool_record(run, dev, stream, peak_gbs, steps, warmup, None)
        warm["l2"] = "warm: back to back, the 50 MB cache stays in the 129 MB L2 (a frac above 1 is L2 bandwidth)"
        rec["pool_warm_l2"] = warm
    rec["select"] = select_record(run, dev, stream, peak_gbs)
    rec["select_ring"] = select_record(run, dev, stream, peak_gbs, ring=True)
    rec["decode_step_us_cuda_graph"] = decode_step_us(run, dev, stream)
    if spec.total_blocks >= 2048:
        rec["hier_select"] = hier_record(run, dev, stream)
    if coarse:
        for group in (64, 512):
            out = torch.zeros((spec.R, -(-max(spec.nb) // group), spec.D), device=dev)
            us = statistics.median(per_call_ms(lambda: kk.kk_coarse_means(run.vb, run.bt, group, out), dev,
                                               stream, 20, 3, flush)) * 1e3
            nbytes = spec.total_blocks * spec.D * 4 + out.numel() * 4
            rec[f"coarse_means_{group}"] = {"us": us, "gbs": nbytes / (us * 1e-6) / 1e9,
                                            "frac": nbytes / (us * 1e-6) / 1e9 / peak_gbs,
                                            "l2": "flushed (256 MB read) before every call"}
    if kk.kk_device_error() != 0:
        raise RuntimeError(f"device error in workload {name}")
    del run
    torch.cuda.empty_cache()
    return rec


def run_pool_gpu(dev, warmup: int, steps: int, peaks):
    """Shared-pool scoring: kk_score_pool_batched over the whole pool, L2
    flushed (256 MB read) before every timed call; only the call is timed.
    Then the pool as documents through the three-level selection."""
    import torch

    from kv_cache_block_gb300 import kk

    v_spec, a_spec, mask, K = synth.shared_pool()
    V = synth.gen_rows_cuda(v_spec, device=dev)
    A = synth.gen_rows_cuda(a_spec, device=dev)
    R, N = A.shape[0], V.shape[0]
    Mt = torch.from_numpy(mask.view(np.int32)).to(dev)
    ws = torch.empty(kk.kk_score_pool_batched_workspace_bytes(R, N, K), dtype=torch.uint8, device=dev)
    idx = torch.zeros((R, K), dtype=torch.int32, device=dev)
    top = torch.zeros((R, K), device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    call = lambda: kk.kk_score_pool_batched(A, V, Mt, K, idx, top, ws)  # noqa: E731
    with ClockSampler(dev.index or 0) as clocks:
        t_start = time.perf_counter()
        ms = per_call_ms(call, dev, stream, steps, warmup, flush)
        clocks.window(t_start, time.perf_counter())
    if kk.kk_device_error() != 0:
        raise RuntimeError("device error in the shared-pool leg")
    warm_ms = b2b_us(call, dev, stream, 50) * 1e-3
    owned = int(np.unpackbits(mask.view(np.uint8)).sum())
    in_bytes = A.numel() * 2 + V.numel() * 2 + mask.nbytes
    hier = run_pool_hier(kk, dev, flush, warmup, min(steps, 100), peaks)
    med = statistics.median(ms)
    flops = 2.0 * R * N * 128
    tflops = flops / (med * 1e-3) / 1e12
    nbytes = in_bytes + idx.numel() * 8
    return {"workload": WORKLOAD_NAMES["pool"], "us": med * 1e3, "us_warm_l2": warm_ms * 1e3,
            "l2": "flushed (256 MB read) before every timed call", "blocks_scored_per_s": owned / (med * 1e-3),
            "tensor": {"flops": flops, "tflops": tflops, "peak_tflops": float(peaks["bf16_tflops"]),
                       "frac": tflops / float(peaks["bf16_tflops"])},
            "hbm": {"bytes": nbytes, "gbs": nbytes / (med * 1e-3) / 1e9,
                    "frac": nbytes / (med * 1e-3) / 1e9 / float(peaks["hbm_gbs"])},
            "roofline_us": max(flops / (float(peaks["bf16_tflops"]) * 1e12), nbytes / (float(peaks["hbm_gbs"]) * 1e9))
            * 1e6,
            "kernel": "kk_score_pool_batched (tcgen05 GEMM + select, timed together)",
            "clocks": clocks.summary(), "hier": hier, "calls": steps}


def run_pool_hier(kk, dev, flush, warmup: int, steps: int, peaks):
    """The shared pool as documents, Grid -> Chunk -> block in one product
    (kk_hier_select_pool), L2 flushed before every timed call;
    kk_hier_pool_reps (write time) timed the same way."""
    import torch

    v_spec, a_spec, mask, K = synth.shared_pool_hier()
    R, N, cp, gc, pm = a_spec.N, v_spec.N, 64, 8, (500, 200, 100)
    H = kk.kk_hier_pool_coarse_rows(N, cp, gc)
    M = torch.zeros((H + N, 128), dtype=torch.int16, device=dev)
    M[H:] = synth.gen_rows_cuda(v_spec, device=dev)
    A = synth.gen_rows_cuda(a_spec, device=dev)
    mt = torch.from_numpy(mask.view(np.int32)).to(dev)
    ws = torch.empty(kk.kk_hier_select_pool_workspace_bytes(R, N, cp, gc), dtype=torch.uint8, device=dev)
    idx = torch.zeros((R, K), dtype=torch.int32, device=dev)
    top = torch.zeros((R, K), device=dev)
    kept = torch.zeros(R, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    reps_us = statistics.median(per_call_ms(lambda: kk.kk_hier_pool_reps(M, N, cp, gc), dev, stream, steps, warmup,
                                            flush)) * 1e3
    sel_us = statistics.median(per_call_ms(
        lambda: kk.kk_hier_select_pool(A, M, mt, N, cp, gc, pm, idx, top, kept, ws), dev, stream, steps, warmup,
        flush)) * 1e3
    if kk.kk_device_error() != 0:
        raise RuntimeError("device error in the hierarchical shared-pool leg")
    flops = 2.0 * R * (H + N) * 128
    return {"select_us": sel_us, "reps_us": reps_us, "rows": H + N, "blocks_kept_mean": float(kept.float().mean()),
            "tflops": flops / (sel_us * 1e-6) / 1e12, "frac": flops / (sel_us * 1e-6) / 1e12 / float(peaks["bf16_tflops"])}


def sub_records(args, dev, peaks):
    import torch

    stream = torch.cuda.current_stream(dev)
    peak = float(peaks["hbm_gbs"])
    flush = L2Flush(dev)
    recs = {}
    steps, warm = max(args.steps, 10), max(args.warmup, 3)
    recs["tiny"] = record_paged("tiny", dev, stream, peak, max(steps, 50), warm, flush)
    recs["7b"] = record_paged("7b", dev, stream, peak, steps, warm, flush)
    recs["pool"] = run_pool_gpu(dev, warm, max(steps, 50), peaks)
    recs["write16"] = record_paged("write16", dev, stream, peak, steps, warm, flush, coarse=True)
    recs["write128"] = record_paged("write128", dev, stream, peak, steps, warm, flush, coarse=True)
    return recs


# --------------------------------------------------------------------------
# entry
# --------------------------------------------------------------------------


def run_reference(args, spec, cfg, rank):
    """The CPU oracle as it stands on every host core, each step a bounded
    sample of the workload (one request of 4 blocks per core)."""
    if rank != 0:
        return
    flat, sub = sample_from_numpy(spec)
    sampler = OracleSampler(spec, flat, sub)
    budget = min(args.cpu_budget, 120.0 / max(1, args.steps + args.warmup))
    try:
        t_all = time.perf_counter()
        for _ in range(args.warmup):
            sampler.step(budget)
        vals = [sampler.step(budget) for _ in range(args.steps)]
    finally:
        sampler.close()
    value = statistics.mean(v for v, _ in vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(dt for _, dt in vals),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": cfg,
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": sampler.cores, "kind": "oracle",
                             "cpu_model": cpu_model(), "sample": sampler.desc + f"; {budget:.1f} s a step"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": time.perf_counter() - t_all}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for the CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-subrecords", action="store_true", help="only the headline workload")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--requests", type=int, default=0, help="override the number of requests (profiling runs)")
    args = ap.parse_args()
    rank, world, local_rank = dist_env()
    peaks, peak_kind = measured_peaks()
    if args.workload == "pool":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the CPU oracle leg covers the paged workloads"}))
            return
        import torch

        torch.cuda.set_device(local_rank)
        res = run_pool_gpu(torch.device("cuda", local_rank), max(args.warmup, 3), args.steps, peaks)
        line = {"metric": METRIC, "value": res["blocks_scored_per_s"], "unit": "blocks scored/s", "n_gpus": 1,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["us"] * 1e-3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic", "config": {"workload": WORKLOAD_NAMES["pool"], "l2": res["l2"]},
                "roofline": {"bound": "tensor", "achieved": res["tensor"]["tflops"],
                             "peak": res["tensor"]["peak_tflops"], "unit": "TFLOP/s", "frac": res["tensor"]["frac"],
                             "traffic": None, "kernel": res["kernel"], "peak_source": peak_kind},
                "pool": res, "clocks": res["clocks"], "gpu_launches": 2 * args.steps, "e2e": None}
        print(json.dumps(line))
        return
    spec = WORKLOADS[args.workload]()
    if args.requests:
        spec = dataclasses.replace(spec, seq_lens=spec.seq_lens[:1] * args.requests)
    cfg = {"workload": WORKLOAD_NAMES[args.workload], "requests": spec.R, "blocks": spec.total_blocks,
           "k_bytes": spec.k_bytes(), "l2": "inputs larger than L2 (no flush needed)" if spec.k_bytes() > L2_FLUSH_BYTES
           else "inputs fit in L2 (warm)"}
    if args.impl == "reference":
        run_reference(args, spec, cfg, rank)
        return

    peak = float(peaks["hbm_gbs"])
    res, run = run_main(args, rank_spec(spec, rank), rank, world, local_rank, peak)
    if rank != 0:
        return
    kb = spec.k_bytes()
    value = weak_value(kb, args.steps, world, res["total_ms"]) / 1e9
    achieved = kb / (res["pool_ms"] * 1e-3) / 1e9
    sel = res["select"]
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": res["total_ms"] / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": spec.dtype, "data": "synthetic", "config": cfg,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": profiled_traffic(args.workload) if not args.requests else None,
                     "kernel": "kk_pool_blocks" + (
                         "_weighted (4 launches: slice sums, variances, weights, combine; timed together)"
                         if spec.weighted else ""),
                     "algorithmic_bytes": kb, "peak_source": peak_kind},
        "blocks_scored_per_s": spec.total_blocks / (res["select_ms"] * 1e-3),
        "score_topk_us_per_step": res["select_ms"] * 1e3,
        "score_topk_us_back_to_back": sel["us_back_to_back"], "score_topk_us_cuda_graph": sel["us_cuda_graph"],
        "score_topk_roofline": {"bound": "hbm", "algorithmic_bytes": sel["algorithmic_bytes"], "peak": peak,
                                "frac_in_step": step_bytes(spec) / (res["select_ms"] * 1e-3) / 1e9 / peak,
                                "frac_back_to_back": sel["roofline_frac_back_to_back"],
                                "frac_cuda_graph": sel["roofline_frac_cuda_graph"]},
        "score_topk_ring": res["select_ring"],
        "anchor_then_score_topk_us_cuda_graph": res["two_launch_us"],
        "score_topk_stable_us_back_to_back": res["stable_us"],
        "decode_step_us_cuda_graph": res["decode_step_us"],
        "hier_select": res["hier"],
        "pool_ms_per_step": res["pool_ms"], "clocks": res["clocks"], "gpu_launches": res["launches"],
        "e2e": None,
    }
    if not args.no_cpu_baseline:
        # the sample is copied back before the end-to-end leg rewrites the cache
        flat, sub = sample_from_device(spec, run.storage)
        sampler = OracleSampler(spec, flat, sub)
        try:
            v, dt = sampler.step(args.cpu_budget)
        finally:
            sampler.close()
        line["cpu_baseline"] = {"value": v, "unit": "GB/s", "cores": sampler.cores, "kind": "oracle",
                                "cpu_model": cpu_model(), "sample": sampler.desc, "seconds": dt}
    if not args.no_e2e:
        import torch

        line["e2e"] = e2e_leg(args, run, torch.device("cuda", local_rank), torch.cuda.current_stream())
    del run
    if world == 1 and not args.no_subrecords:
        import torch

        torch.cuda.empty_cache()
        line["workloads"] = sub_records(args, torch.device("cuda", local_rank), peaks)
    print(json.dumps(line))


if __name__ == "__main__":
    main()
