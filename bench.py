"""Benchmark of one paged GQA decode step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                    [--impl ours|reference] [--partition-tokens T] [--compute mma|simt]

One "step" = the whole hot path over one batch: split kernel (phase 1) +
merge kernel (phase 2), through the C ABI.  Prints ONE JSON line (rank 0).

metric  : K/V-read HBM GB/s = unique K/V bytes a step must read / step time
          (unit GB/s, higher is better); us per step and tokens/s ride along.
value   : device-timed with CUDA events on the launching stream, inputs
          resident in HBM; K steps between barrier + synchronize, max over ranks.
e2e     : the same metric through the host-buffer calls: every step copies
          q, the block table and the lengths from pinned host memory, attends,
          and writes the output and the step's status word back to pinned
          host memory.  value: the asynchronous call (pa_decode_host_async /
          pa_decode_multi_host_async) with two buffer sets on alternating
          staging slots, steps issued back to back, one synchronisation at the
          end; sync_*: the synchronous call, which waits for every step.
roofline: the split kernel alone (CUDA events around phase 1 in the same timed
          loop) against the measured HBM copy bandwidth.
cpu_baseline / --impl reference: the float64 oracle on the host cores, on a
          bounded sample of the same workload (cpu_baseline: all cores, plus a
          one-core figure).
repeats : the K-step region repeated for about --repeat-s seconds (spread);
          the clocks are sampled every 20 ms over the loaded window.
per_config: with the default workload, the other configurations the metric
          is quoted on (the tiny page example, Qwen2-style GQA, long context
          with the default split and with 512-token partitions, prefix
          sharing, the serving mix with 8 query tokens per sequence), each
          with device and end-to-end time per step, the split kernel's
          fraction of the HBM peak, the recorded ncu traffic ratio
          and an oracle parity sample.  A workload that fits in L2 is timed
          two ways: one step at a time with L2 flushed before each (events
          around every step), and as the decode of consecutive layers of a
          model (layer_steps: enough copies of the inputs to exceed L2,
          attended in turn back to back).
N > 1   : independent replicas (the path has no exchange step), one per GPU,
          scaling "weak".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "serving_mix_b256_g4_d128"
METRIC = "paged GQA decode: K/V-read HBM GB/s (% of GB300 peak); µs per decode step"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


SPLIT_SOURCES = ("pa_split.cuh", "pa_ptx.cuh", "pa_kernels.cuh", "pa_sched.cuh", "pa_cluster.cuh")


def source_hash() -> str:
    """Hash of the sources of a step's first kernel (the split kernel or the
    cluster kernel): recorded ncu traffic is tied to it."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_gqa_decode_pa_gb300", "csrc")
    names = sorted(f for f in os.listdir(csrc)
                   if f in SPLIT_SOURCES or (f.startswith(("pa_split_", "pa_cluster_"))
                                             and f.endswith(".cu")))
    for f in names:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, opts_key: str):
    """dram bytes per split-kernel launch from a committed ncu summary, if it
    was taken on the current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(f"{workload}|{opts_key}")
    if not e or e.get("source_hash") != source_hash():
        return None
    return float(e["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 20 ms (a read-only
    query; no GPU setting is touched)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 20

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.PERIOD_MS), "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), line.strip()))

    def mark_begin(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)

    def window(self, t0, t1):
        """Median SM clock, max clock and active throttle reasons of the
        samples taken between t0 and t1 (wall clock)."""
        if self.proc is None:
            return None
        inside = [r for (t, r) in self.rows if t0 <= t <= t1]
        if not inside and self.rows:
            inside = [min(self.rows, key=lambda x: abs(x[0] - t1))[1]]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in inside:
            parts = [x.strip() for x in r.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "sm_mhz_min": min(sm), "reasons": sorted(reasons), "samples": len(sm),
                "period_ms": self.PERIOD_MS}


def max_over_ranks(values, device="cpu"):
    """Element-wise max of per-rank timings over all ranks (a no-op when
    torch.distributed is not initialised)."""
    import torch

    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_gbs(bytes_per_rank_step: int, world: int, ms_per_step: float) -> float:
    """All ranks' bytes of one step divided by the slowest rank's step time."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


def make_room_for_next_token(w):
    """Map a fresh physical block (appended to the pool) wherever a
    sequence's next position has none, as a serving engine would before a
    fused append step."""
    bs = w.block_size
    if int(w.cache_seqlens.max()) // bs >= w.block_table.shape[1]:
        # a full row: widen every row by one unmapped column
        w.block_table = np.pad(w.block_table, ((0, 0), (0, 1)), constant_values=-1)
        w.max_blocks_per_seq += 1
    table = w.block_table
    extra = 0
    for b in range(w.B):
        col = int(w.cache_seqlens[b]) // bs
        if table[b, col] < 0:
            table[b, col] = w.num_blocks + extra
            extra += 1
    if extra:
        pad = np.zeros((extra,) + w.k_cache.shape[1:], dtype=np.uint16)
        w.k_cache = np.concatenate([w.k_cache, pad])
        w.v_cache = np.concatenate([w.v_cache, pad])
        w.num_blocks += extra


def make_workload(name, query_tokens=0, group=0):
    """The named workload; query_tokens > 0 gives every sequence that many
    query tokens (its last positions, causal); group > 0 sets G query heads
    per kv head over the same cache."""
    from paged_gqa_decode_pa_gb300 import workloads as wl

    w = wl.make(name)
    if query_tokens > 0:
        w = wl.with_query_tokens(w, np.full(w.B, query_tokens), seed=w.seed + 2000,
                                 name=f"{w.name}+q{query_tokens}")
    if group > 0:
        w = wl.with_group(w, group, seed=w.seed + 3000, name=f"{w.name}+G{group}")
    return w


def query_rows(w) -> int:
    """Output rows of a step: B, or the packed query rows."""
    return w.B if w.cu_q is None else int(w.q.shape[0])


def row_sequences(w) -> np.ndarray:
    """The sequence each output row belongs to (-1: none)."""
    if w.cu_q is None:
        return np.arange(w.B)
    seq = np.full(query_rows(w), -1, dtype=np.int64)
    for b in range(w.B):
        seq[w.cu_q[b]:w.cu_q[b + 1]] = b
    return seq


def oracle_outputs(w, pairs, n_threads: int = 0):
    """The oracle's outputs for (row, head) pairs of the workload."""
    import oracle

    if w.cu_q is None:
        return oracle.decode(w.q, w.k_cache, w.v_cache, w.block_table, w.cache_seqlens,
                             w.scale, w.dtype, pairs=pairs, n_threads=n_threads)
    return oracle.decode_multi(w.q, w.cu_q, w.causal, w.k_cache, w.v_cache, w.block_table,
                               w.cache_seqlens, w.scale, w.dtype, pairs=pairs,
                               n_threads=n_threads)


def metric_bytes_of_pairs(w, pairs) -> float:
    """The share of the step's metric bytes (unique K/V bytes) that the
    outputs in `pairs` account for: the H * n_q outputs of a sequence with
    n_q query rows share its K/V rows (output (row, h) owns 1/(G n_q) of kv
    head h // G), scaled so that all outputs add up to exactly the step's
    unique K/V bytes (shared prefix blocks counted once)."""
    seq = row_sequences(w)
    nq = np.ones(w.B) if w.cu_q is None else np.maximum(np.diff(w.cu_q), 1)
    lens = w.cache_seqlens.astype(np.float64)
    per_row = np.where(seq >= 0, lens[seq] * w.d * 4 / w.G / nq[seq], 0.0)
    total = float(per_row.sum()) * w.H
    return float(per_row[pairs[:, 0]].sum()) * (w.kv_bytes() / total) if total else 0.0


def oracle_sample(w, budget_s: float, seed: int = 0, n_threads: int = 0):
    """Time the oracle on a bounded sample of (b, h) outputs of the workload,
    repeated until about `budget_s` seconds of work have been timed.
    n_threads = 0: all host cores (OpenMP); 1: one core.

    Returns (GB/s in the metric's unit, seconds, pairs, threads, passes)."""
    import oracle

    oracle.build()
    threads = oracle.max_threads() if n_threads <= 0 else n_threads
    rng = np.random.default_rng(seed)
    order = rng.permutation(query_rows(w) * w.H)
    pairs_all = np.stack([order // w.H, order % w.H], axis=1).astype(np.int32)

    def run(pairs):
        t = time.perf_counter()
        oracle_outputs(w, pairs, n_threads)
        return time.perf_counter() - t

    # calibrate on a few outputs, then size the sample for the budget
    n = min(len(pairs_all), max(threads, 8))
    while True:
        pairs = pairs_all[:n]
        dt = run(pairs)
        if dt >= 0.25 * budget_s or n >= len(pairs_all):
            break
        grow = max(2.0, min(16.0, 0.5 * budget_s / max(dt, 1e-3)))
        n = min(len(pairs_all), int(n * grow))
    # the whole workload fits the budget several times over: time repeated passes
    passes = max(1, int(budget_s / max(dt, 1e-3)))
    if passes > 1:
        dt = sum(run(pairs) for _ in range(passes))
    nbytes = metric_bytes_of_pairs(w, pairs) * passes
    return nbytes / dt / 1e9, dt, pairs, threads, passes


def run_reference(args, rank, world):
    """The oracle timed on the host cores (rank 0 only)."""
    if rank != 0:
        return
    w = make_workload(args.config, args.query_tokens, args.group)
    per_step = max(0.05, min(1.0, 90.0 / max(1, args.steps + args.warmup)))
    gbs, dt, pairs, threads, _ = oracle_sample(w, per_step)
    for _ in range(args.warmup):
        oracle_outputs(w, pairs)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle_outputs(w, pairs)
    el = time.perf_counter() - t
    toks = int(w.cache_seqlens[row_sequences(w)[pairs[:, 0]]].astype(np.int64).sum())
    value = metric_bytes_of_pairs(w, pairs) * args.steps / el / 1e9
    sample = (f"{len(pairs)} of {query_rows(w) * w.H} (query row, head) outputs per step, "
              f"{toks} cached tokens")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, args), "gpu_launches": 0,
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(w, args):
    return {"workload": w.name, "B": w.B, "H": w.H, "Hkv": w.Hkv, "d": w.d,
            "block_size": w.block_size, "max_blocks_per_seq": w.max_blocks_per_seq,
            "num_blocks": w.num_blocks, "dtype": w.dtype,
            "mean_seqlen": round(float(np.mean(w.cache_seqlens)), 1),
            "max_seqlen": int(np.max(w.cache_seqlens)),
            "partition_tokens": args.partition_tokens, "compute": args.compute,
            "stages": args.stages, "graph": bool(args.graph),
            "fused_append": bool(args.fused_append),
            "query_rows_per_step": query_rows(w), "causal": bool(w.causal) if w.cu_q is not None else None,
            "kv_bytes_per_step": w.kv_bytes(),
            "l2": ("inputs larger than L2" if w.kv_bytes() > 2 * L2_BYTES
                   else "L2 flushed between timed steps"),
            "parallelism": f"replicas x{args.gpus}"}


class Stepper:
    """One workload resident on the device, with the calls of one decode step
    bound through the C ABI: the step itself (both phases), the two phases
    apart, and the end-to-end host-buffer step."""

    def __init__(self, w, opt_kw, dev, fused_append=False, graph=False, warmup=3):
        import torch

        import paged_gqa_decode_pa_gb300 as pg

        self.pg, self.w, self.dev = pg, w, dev
        if fused_append:
            make_room_for_next_token(w)
        self.q, self.k, self.v, self.t, self.sl = w.torch_tensors(dev)
        q, k, t = self.q, self.k, self.t
        self.multi = w.cu_q is not None
        if self.multi and fused_append:
            raise SystemExit("--fused-append is a one-token-per-sequence step")
        self.out = torch.empty(tuple(q.shape), dtype=torch.float32, device=dev)
        self.opt_kw = opt_kw
        self.opts = pg.options(**opt_kw)
        self.opts_split = pg.options(**opt_kw, phase=pg.PA_PHASE_SPLIT)
        self.opts_merge = pg.options(**opt_kw, phase=pg.PA_PHASE_MERGE)
        if self.multi:
            self.cu = torch.from_numpy(w.cu_q).to(dev)
            self.ws = pg.alloc_workspace_multi(pg.shape_multi(q, k, t), w.max_q, self.opts, dev)
        else:
            self.cu = None
            self.ws = pg.alloc_workspace(pg.shape_of(q, k, t), self.opts, dev)
        self.stream = torch.cuda.current_stream(dev)
        # the step's calls, bound once (per-call Python checks would make the
        # small steps host-bound)
        if self.multi:
            self.bound = {ph: pg.bind_decode_multi(q, self.cu, w.max_q, w.causal, self.k, self.v,
                                                   t, self.sl, w.scale, self.out, self.ws, o,
                                                   self.stream)
                          for ph, o in ((0, self.opts), (1, self.opts_split),
                                        (2, self.opts_merge))}
        else:
            self.bound = {ph: pg.bind_decode(q, self.k, self.v, t, self.sl, w.scale, self.out,
                                             self.ws, o, self.stream)
                          for ph, o in ((0, self.opts), (1, self.opts_split),
                                        (2, self.opts_merge))}
        self.kv_bytes = w.kv_bytes()
        self.flush = self.kv_bytes <= 2 * L2_BYTES
        self.scratch = (torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
                        if self.flush else None)
        for _ in range(warmup):
            self.flush_l2()
            self.attend(self.opts)
        self.attend(self.opts_split)
        self.attend(self.opts_merge)
        torch.cuda.synchronize()
        if pg.pa_read_status(self.ws) != 0:
            raise RuntimeError("device status bits set during warm-up")
        self.decode_step = lambda: self.attend(self.opts)
        if fused_append:
            # each step writes a new K/V row at position len and attends over
            # len + 1 tokens (the lengths are not advanced, so every step
            # rewrites the same slots)
            gen = torch.Generator(device=dev).manual_seed(1)
            self.kn = torch.randn((w.B, w.Hkv, w.d), generator=gen, device=dev).to(k.dtype)
            self.vn = torch.randn((w.B, w.Hkv, w.d), generator=gen, device=dev).to(k.dtype)
            self.kv_bytes += w.B * w.Hkv * w.d * 2 * 2  # the appended rows
            self.decode_step = pg.bind_decode_append(
                self.q, self.kn, self.vn, self.k, self.v, self.t, self.sl, w.scale, self.out,
                self.ws, self.opts, self.stream)
        self.graph = None
        if graph:
            # one decode step captured once and replayed (host launch cost
            # removed); the captured call is bound to the capture stream
            self.graph = torch.cuda.CUDAGraph()
            cap = torch.cuda.Stream(dev)
            cap.wait_stream(self.stream)
            if fused_append:
                cap_step = pg.bind_decode_append(self.q, self.kn, self.vn, self.k, self.v, self.t,
                                                 self.sl, w.scale, self.out, self.ws, self.opts,
                                                 cap)
            elif self.multi:
                cap_step = pg.bind_decode_multi(q, self.cu, w.max_q, w.causal, self.k, self.v, t,
                                                self.sl, w.scale, self.out, self.ws, self.opts, cap)
            else:
                cap_step = pg.bind_decode(q, self.k, self.v, t, self.sl, w.scale, self.out,
                                          self.ws, self.opts, cap)
            with torch.cuda.stream(cap):
                cap_step()
            cap.synchronize()
            with torch.cuda.graph(self.graph, stream=cap):
                cap_step()
            for _ in range(warmup):
                self.graph.replay()
            torch.cuda.synchronize()

    def flush_l2(self):
        if self.flush:
            self.scratch.fill_(1.0)

    def attend(self, o):
        """One step of the path through the C ABI (o selects the phases)."""
        self.bound[o.phase]()

    def steps(self, K):
        """K decode steps; device ms per step.  With the L2 flushed between
        steps each step is bracketed by its own events (the flush stays
        outside); otherwise only the first and the last, so that consecutive
        steps stay back to back on the stream (the split kernel is a
        programmatic dependent of the previous merge, and an event in between
        would serialise them)."""
        import torch

        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
        for i in range(K):
            self.flush_l2()
            if self.flush or i == 0:
                ev[i][0].record(self.stream)
            if self.graph is not None:
                self.graph.replay()
            else:
                self.decode_step()
            if self.flush or i == K - 1:
                ev[i][1].record(self.stream)
        torch.cuda.synchronize()
        if self.flush:
            return float(sum(ev[i][0].elapsed_time(ev[i][1]) for i in range(K))) / K
        return ev[0][0].elapsed_time(ev[K - 1][1]) / K

    def phases(self, K):
        """K steps as two phase calls with an event between them: the split
        kernel's and the merge kernel's own average durations (ms)."""
        import torch

        ev3 = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
        torch.cuda.synchronize()
        for i in range(K):
            self.flush_l2()
            ev3[i][0].record(self.stream)
            self.attend(self.opts_split)
            ev3[i][1].record(self.stream)
            self.attend(self.opts_merge)
            ev3[i][2].record(self.stream)
        torch.cuda.synchronize()
        split_ms = [ev3[i][0].elapsed_time(ev3[i][1]) for i in range(K)]
        merge_ms = [ev3[i][1].elapsed_time(ev3[i][2]) for i in range(K)]
        if self.pg.pa_read_status(self.ws) != 0:
            raise RuntimeError("device status bits set during the timed steps")
        return float(np.mean(split_ms)), float(np.mean(merge_ms))

    def e2e(self, K):
        """End to end through the library's host-buffer entry points: every
        step moves q, the block table and the lengths (and the query
        offsets) from pinned host memory into the workspace's staging, runs
        both phases with the output written to pinned host memory, and
        publishes the step's status word there too.

        async: the serving-loop form -- two buffer sets, one per staging
        slot, and a bound call each (pa_decode_host_async); steps are issued
        back to back and the host synchronises only after the last one, so
        step i + 1's staging overlaps step i's kernels.  sync: one
        pa_decode_host call per step, which waits for the stream before it
        returns.  Returns (async ms per step, sync ms per step, h2d bytes,
        d2h bytes)."""
        import torch

        pg, w = self.pg, self.w
        q, k, v, t, sl, out, dev, stream = (self.q, self.k, self.v, self.t, self.sl, self.out,
                                            self.dev, self.stream)
        Ke = max(3, min(K, 200))
        shape = pg.shape_multi(q, k, t) if self.multi else pg.shape_of(q, k, t)
        sets = []
        for _ in range(2):
            parts = [x.cpu().contiguous().pin_memory() for x in (q, t, sl)]
            if self.multi:
                parts.append(self.cu.cpu().contiguous().pin_memory())
            sets.append((parts, torch.empty(out.shape, dtype=out.dtype).pin_memory()))
        h2d = sum(x.numel() * x.element_size() for x in sets[0][0])
        d2h = sets[0][1].numel() * 4 + 4  # the output and the step's status word
        if self.multi:
            ws_a = pg.alloc_workspace_multi_host_async(shape, w.max_q, q.shape[0], self.opts, dev)
            ws_s = pg.alloc_workspace_multi_host(shape, w.max_q, q.shape[0], self.opts, dev)
            calls = [pg.bind_decode_multi_host_async(p[0], p[3], w.max_q, w.causal, k, v, p[1],
                                                     p[2], w.scale, o, ws_a, s, self.opts,
                                                     stream)
                     for s, (p, o) in enumerate(sets)]
            sync = pg.bind_decode_multi_host(sets[0][0][0], sets[0][0][3], w.max_q, w.causal, k,
                                             v, sets[0][0][1], sets[0][0][2], w.scale,
                                             sets[0][1], ws_s, self.opts, stream)
        else:
            ws_a = pg.alloc_workspace_host_async(shape, self.opts, dev)
            ws_s = pg.alloc_workspace_host(shape, self.opts, dev)
            calls = [pg.bind_decode_host_async(p[0], k, v, p[1], p[2], w.scale, o, ws_a, s,
                                               self.opts, stream)
                     for s, (p, o) in enumerate(sets)]
            sync = pg.bind_decode_host(sets[0][0][0], k, v, sets[0][0][1], sets[0][0][2],
                                       w.scale, sets[0][1], ws_s, self.opts, stream)

        def timed(run_step):
            for i in range(2):
                run_step(i)
            torch.cuda.synchronize()
            if self.flush:
                # L2 flushed before every step, outside its events
                ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)]
                      for _ in range(Ke)]
                for i in range(Ke):
                    self.flush_l2()
                    ev[i][0].record(stream)
                    run_step(i)
                    ev[i][1].record(stream)
                torch.cuda.synchronize()
                return float(sum(ev[i][0].elapsed_time(ev[i][1]) for i in range(Ke))) / Ke
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(Ke):
                run_step(i)
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / Ke

        status = [0]

        def step_sync(i):
            status[0] |= sync()

        ms_sync = timed(step_sync)
        ms_async = timed(lambda i: calls[i % 2]())
        status[0] |= calls[0].status() | calls[1].status()
        if status[0] != 0:
            raise RuntimeError(f"device status bits {status[0]:#x} during the end-to-end steps")
        for _, o in sets:
            if not torch.equal(o, out.cpu()):
                raise RuntimeError("the end-to-end output differs from the device-buffer output")
        return ms_async, ms_sync, h2d, d2h

    def parity(self, n, seed=0):
        """The last output against the oracle on n sampled (row, head) outputs
        (all of them when the step has at most n)."""
        w = self.w
        total = query_rows(w) * w.H
        order = np.random.default_rng(seed).permutation(total)[:min(n, total)]
        pairs = np.stack([order // w.H, order % w.H], axis=1).astype(np.int32)
        ref = oracle_outputs(w, pairs)
        got = self.out.cpu().numpy().astype(np.float64)[pairs[:, 0], pairs[:, 1]]
        err = np.abs(got - ref)
        return {"pairs": int(len(pairs)), "max_abs_err": float(err.max()),
                "mean_abs_err": float(err.mean()), "tolerance": [2e-3, 2e-4]}


def opts_key(kw) -> str:
    return f"part={kw['partition_tokens']},compute={kw['compute']},stages={kw['stages']}"


# The other configurations the metric is quoted on, measured in the same run
# as the headline (one GPU): (entry name, workload, partition_tokens, query
# tokens per sequence).
PER_CONFIG = [
    ("p5_example", "p5_example", 0, 0),
    ("qwen2_b8_g7_d64", "qwen2_b8_g7_d64", 0, 0),
    ("long_ctx_100k_g6_d256", "long_ctx_100k_g6_d256", 0, 0),
    ("long_ctx_100k_g6_d256_part512", "long_ctx_100k_g6_d256", 512, 0),
    ("prefix_share_b64_g8_d128", "prefix_share_b64_g8_d128", 0, 0),
    ("serving_mix_b256_q8_g4_d128", "serving_mix_b256_g4_d128", 0, 8),
]


def per_config_entries(spec: str, default_run: bool):
    """The PER_CONFIG entries --per-config selects."""
    if spec == "none" or (spec == "auto" and not default_run):
        return []
    if spec in ("auto", "all"):
        return list(PER_CONFIG)
    names = [x for x in spec.split(",") if x]
    known = {e[0]: e for e in PER_CONFIG}
    bad = [x for x in names if x not in known]
    if bad:
        raise SystemExit(f"--per-config: unknown entries {bad}; choose from {sorted(known)}")
    return [known[x] for x in names]


MAX_LAYERS = 128


def layer_steps(w, kw, dev, steps, warmup):
    """A step of a small workload as it runs inside a model: the decode of
    consecutive layers, each over its own cache.  L copies of the inputs
    (at least 24, and together more than 2.5x L2, so a copy's K/V rows are
    gone from L2 before its next turn and no flush is needed) are attended in
    turn, back to back on one stream, with events around the whole run.
    Returns (L, device ms per step, MB of K/V over the copies), or None when
    that would need more than MAX_LAYERS copies."""
    import torch

    import paged_gqa_decode_pa_gb300 as pg

    L = max(24, math.ceil(2.5 * L2_BYTES / w.kv_bytes()))
    if L > MAX_LAYERS:
        return None
    opts = pg.options(**kw)
    stream = torch.cuda.current_stream(dev)
    calls, outs, wss = [], [], []
    for _ in range(L):
        q, k, v, t, sl = w.torch_tensors(dev)
        out = torch.empty((w.B, w.H, w.d), dtype=torch.float32, device=dev)
        ws = pg.alloc_workspace(pg.shape_of(q, k, t), opts, dev)
        calls.append(pg.bind_decode(q, k, v, t, sl, w.scale, out, ws, opts, stream))
        outs.append(out)
        wss.append(ws)
    for _ in range(max(warmup, 3)):
        for c in calls:
            c()
    torch.cuda.synchronize()
    reps = max(2, math.ceil(steps / L))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        for c in calls:
            c()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / (reps * L)
    if any(pg.pa_read_status(x) != 0 for x in wss):
        raise RuntimeError("device status bits set during the layer steps")
    if not all(torch.equal(outs[0], o) for o in outs[1:]):
        raise RuntimeError("the layers' outputs differ on identical inputs")
    return L, ms, L * w.kv_bytes() / 1e6


def per_config_entry(name, part, args, dev, peak, query_tokens=0):
    """One configuration at a glance: device and end-to-end time per step,
    the split kernel's fraction of the HBM peak, the recorded ncu traffic
    ratio (when taken on the current kernel sources) and the parity sample."""
    import torch

    w = make_workload(name, query_tokens)
    kw = dict(partition_tokens=part, compute=args.compute, stages=args.stages)
    st = Stepper(w, kw, dev, warmup=args.warmup)
    K = max(args.steps, 20)
    ms = st.steps(K)
    split_ms, merge_ms = st.phases(K)
    e2e_ms, e2e_sync_ms, _, _ = st.e2e(K)
    par = st.parity(256)
    traffic = recorded_traffic(w.name, opts_key(kw))
    kvb = st.kv_bytes
    flushed = st.flush
    layers = None
    if flushed:
        del st
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        lr = layer_steps(w, kw, dev, K, args.warmup)
        if lr is not None:
            n, lms, mb = lr
            if kvb / (lms * 1e-3) / 1e9 > 2 * peak:
                raise RuntimeError("implausible layer-step timing")
            layers = {"layers": n, "us_per_step": round(lms * 1e3, 3),
                      "gbs": round(kvb / (lms * 1e-3) / 1e9, 2),
                      "step_frac": round(kvb / (lms * 1e-3) / 1e9 / peak, 4),
                      "l2": f"{n} copies of the inputs ({mb:.0f} MB of K/V) attended in turn, "
                            f"back to back; no flush"}
    entry = {"workload": w.name, "partition_tokens": part, "query_tokens": query_tokens,
             "steps": K,
             "us_per_step": round(ms * 1e3, 3), "gbs": round(kvb / (ms * 1e-3) / 1e9, 2),
             "split_us": round(split_ms * 1e3, 3), "merge_us": round(merge_ms * 1e3, 3),
             "frac": round(kvb / (split_ms * 1e-3) / 1e9 / peak, 4),
             "step_frac": round(kvb / (ms * 1e-3) / 1e9 / peak, 4),
             "e2e_us": round(e2e_ms * 1e3, 3), "e2e_sync_us": round(e2e_sync_ms * 1e3, 3),
             "kv_bytes_per_step": kvb,
             "traffic_ratio": round(traffic / kvb, 4) if traffic else None,
             "l2": ("inputs larger than L2" if not flushed
                    else "L2 flushed between timed steps"),
             "max_abs_err": par["max_abs_err"], "mean_abs_err": par["mean_abs_err"],
             "parity_outputs": par["pairs"], "layer_steps": layers}
    if not flushed:
        del st
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return entry


def run_ours(args, rank, world, local_rank):
    import torch

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = make_workload(args.config, args.query_tokens, args.group)
    opt_kw = dict(partition_tokens=args.partition_tokens, compute=args.compute,
                  stages=args.stages)
    st = Stepper(w, opt_kw, dev, fused_append=args.fused_append, graph=args.graph,
                 warmup=args.warmup)
    q = st.q
    kv_bytes = st.kv_bytes
    K = args.steps
    # the library's own kernels per step (split + merge, or one cluster kernel)
    import paged_gqa_decode_pa_gb300 as pg

    plan = pg.pa_launch_plan(pg.shape_multi(st.q, st.k, st.t) if st.multi
                             else pg.shape_of(st.q, st.k, st.t), st.opts,
                             w.max_q if st.multi else 0)
    kernels_per_step = 2 if args.fused_append else plan["kernels"]
    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)
    sampler = ClockSampler(f"GPU-{uuid}" if uuid is not None else str(local_rank))
    sampler.start()
    time.sleep(0.3)

    # ---- timed region 1 (the value): K decode steps through pa_decode
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_load0 = time.time()
    ms_value = st.steps(K)
    if world > 1:
        torch.distributed.barrier()
    # ---- the same K-step region repeated (run-to-run spread; a longer
    # loaded window for the clock samples)
    reps = []
    t_rep = time.time()
    while len(reps) < 3 or (time.time() - t_rep < args.repeat_s and len(reps) < 200):
        reps.append(st.steps(K))
    # ---- timed region 2 (the roofline): the split kernel's own duration
    split_ms, merge_ms = st.phases(K)
    t_load1 = time.time()
    clocks = sampler.window(t_load0, t_load1)
    # ---- e2e: host buffers, transfers inside the timed region
    if world > 1:
        torch.distributed.barrier()
    e2e_ms, e2e_sync_ms, h2d, d2h = st.e2e(K)

    # ---- max over ranks
    total_ms = ms_value * K
    total_ms, e2e_ms, e2e_sync_ms, split_avg_ms, merge_avg_ms = max_over_ranks(
        [total_ms, e2e_ms, e2e_sync_ms, split_ms, merge_ms], dev)
    peak, peak_kind = peaks()
    cpu = None
    parity = None
    per_config = None
    if rank == 0 and world == 1:
        if args.cpu_baseline_s > 0:
            gbs, dt, pairs, threads, passes = oracle_sample(w, args.cpu_baseline_s)
            toks = int(w.cache_seqlens[row_sequences(w)[pairs[:, 0]]].astype(np.int64).sum())
            gbs1, dt1, pairs1, _, passes1 = oracle_sample(w, args.cpu_baseline_s / 2,
                                                          n_threads=1)
            toks1 = int(w.cache_seqlens[row_sequences(w)[pairs1[:, 0]]].astype(np.int64).sum())
            cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                   "sample": f"{len(pairs)} of {query_rows(w) * w.H} (query row, head) outputs, "
                             f"{toks} cached tokens, {passes} pass(es), {dt:.1f} s; GB/s counts "
                             f"each output's share (1/G of its kv head, split over its "
                             f"sequence's query rows) of the step's unique K/V bytes",
                   "one_core": {"value": round(gbs1, 4), "unit": "GB/s", "cores": 1,
                                "sample": f"{len(pairs1)} outputs, {toks1} cached tokens, "
                                          f"{passes1} pass(es), {dt1:.1f} s"}}
        parity = st.parity(256)
        default_run = (args.config == DEFAULT_WORKLOAD and args.compute in ("mma", "auto")
                       and not (args.query_tokens or args.group or args.fused_append
                                or args.graph or args.partition_tokens or args.stages))
        chosen = per_config_entries(args.per_config, default_run)
        if chosen:
            del st
            torch.cuda.synchronize()
            torch.cuda.empty_cache()
            per_config = {}
            for entry, name, part, nq in chosen:
                t0 = time.time()
                per_config[entry] = per_config_entry(name, part, args, dev, peak, nq)
                per_config[entry]["clocks"] = sampler.window(t0, time.time())
    sampler.stop()
    if rank != 0:
        return
    ms_per_step = total_ms / K
    value = whole_job_gbs(kv_bytes, world, ms_per_step)
    peak_gbs = peaks()[0]
    if value > 2 * world * peak_gbs or kv_bytes / (split_avg_ms * 1e-3) / 1e9 > 2 * peak_gbs:
        # far above the copy bandwidth: the timed region did not do the work
        raise RuntimeError(f"implausible timing: {value:.0f} GB/s against a {peak_gbs:.0f} GB/s peak")
    e2e_value = whole_job_gbs(kv_bytes, world, e2e_ms)
    achieved = kv_bytes / (split_avg_ms * 1e-3) / 1e9
    traffic = recorded_traffic(w.name, opts_key(opt_kw))
    rep_us = sorted(r * 1e3 for r in reps)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "us_per_step": round(ms_per_step * 1e3, 2),
        "tokens_per_s": round(world * int(q.shape[0]) / (ms_per_step * 1e-3), 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic", "config": workload_config(w, args),
        "gpu_launches": kernels_per_step * K,
        "roofline": {"bound": "hbm", "kernel": "pa_split_kernel",
                     "achieved": round(achieved, 2), "peak": peak, "peak_kind": peak_kind,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic,
                     "algorithmic_bytes_per_launch": kv_bytes,
                     "avg_launch_us": round(split_avg_ms * 1e3, 3),
                     "merge_avg_launch_us": round(merge_avg_ms * 1e3, 3)},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "us_per_step": round(e2e_ms * 1e3, 2),
                "mode": "pa_decode_host_async, two pinned buffer sets alternating staging slots, "
                        "one host synchronisation after the last step",
                "sync_us_per_step": round(e2e_sync_ms * 1e3, 2),
                "sync_value": round(whole_job_gbs(kv_bytes, world, e2e_sync_ms), 2)},
        "repeats": {"n": len(rep_us), "steps_each": K,
                    "us_per_step_min": round(rep_us[0], 2),
                    "us_per_step_median": round(statistics.median(rep_us), 2),
                    "us_per_step_max": round(rep_us[-1], 2)},
        "clocks": clocks,
        "cpu_baseline": cpu,
        "parity_vs_oracle": parity,
        "per_config": per_config,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--partition-tokens", type=int, default=0)
    ap.add_argument("--compute", default="mma", choices=["mma", "simt", "tc", "auto"])
    ap.add_argument("--stages", type=int, default=0, help="pipeline stages (0 = library choice)")
    ap.add_argument("--query-tokens", type=int, default=0,
                    help="query tokens per sequence (0 = the workload's own: one in decode)")
    ap.add_argument("--group", type=int, default=0,
                    help="G query heads per kv head over the same cache (0 = the workload's)")
    ap.add_argument("--fused-append", action="store_true",
                    help="time pa_decode_append (write the new token, attend over len+1)")
    ap.add_argument("--graph", action="store_true",
                    help="replay one captured CUDA graph of pa_decode per step")
    ap.add_argument("--cpu-baseline-s", type=float, default=10.0,
                    help="seconds of oracle work for the cpu_baseline sample on all host "
                         "cores (0 = skip); the one-core sample takes half as long")
    ap.add_argument("--per-config", default="auto",
                    help="also measure the other configurations: auto (when the headline "
                         "workload runs with the default options), all, none, or a "
                         "comma-separated list of entry names")
    ap.add_argument("--repeat-s", type=float, default=0.3,
                    help="seconds of repeated K-step regions after the timed one (spread)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    import __graft_entry__

    __graft_entry__.build()
    if world > 1:
        import torch

        torch.distributed.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch

            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
