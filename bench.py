#!/usr/bin/env python
"""Benchmark: cascade attention over a shared-prefix paged KV cache on GB300.

Workload (default): the decode batch of "vLLM Cascade Attention：用法、场景与原理解析"
§五 — N=64 requests sharing a P=4096-token prefix, each with S=128 private tokens
(the last one is the single query), 32 query heads, 8 KV heads, head_dim 128, bf16,
block size 16, shuffled physical blocks.  Synthetic N(0,1) data, seeded.

One step = the host planner (cascade_plan on the block table) + the device path it
picks (cascade_attn here: a prefix kernel and a suffix kernel that run concurrently
and finish the LSE merge themselves) for one batch.
Inputs stay resident in HBM; L2 is kept cold by rotating over several copies of the
KV cache and queries (more bytes than 2x L2 touched between reuses).  Device steps
are replayed from a CUDA graph of one round of copies; the planner runs on the host
every step while the GPU executes.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle instead
(bounded row samples of the same batch).  Under torchrun every rank runs its own
batch (weak scaling, no collective on the data path); value = all ranks' queries /
the slowest rank's time.
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attn queries/s + HBM GB/s (% of roofline), decode N=64 P=4096 S=128"
UNIT = "queries/s"
L2_BYTES = 129 * 1024 * 1024
KERNEL_SOURCES = {
    "decode_cascade_kernel": ["decode_cascade.cu", "prefix_body.cuh", "common.cuh", "merge.cuh",
                              "kernels.cuh"],
    "prefix_attn_kernel": ["prefix_attn.cu", "prefix_body.cuh", "common.cuh", "merge.cuh"],
    "paged_attn_kernel": ["paged_attn.cu", "common.cuh", "merge.cuh"],
    "paged_tc_kernel": ["paged_tc.cu", "prefix_body.cuh", "common.cuh", "merge.cuh",
                        "kernels.cuh"],
    "merge_slots_kernel": ["combine.cu", "merge.cuh", "common.cuh", "kernels.cuh"],
}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode",
                    help="decode (N=64 P=4096 S=128), tiny, chunked, long")
    ap.add_argument("--copies", type=int, default=0, help="input copies (0: enough for 2x L2)")
    ap.add_argument("--quick", action="store_true",
                    help="device timing only (no e2e, flat comparison or CPU baseline)")
    ap.add_argument("--sweep", action="store_true",
                    help="N x P decode sweep: cascade vs flat at every point, one line each")
    ap.add_argument("--fp8", action="store_true",
                    help="FP8 (E4M3) KV cache: bf16 vs FP8 cascade and flat, one line per "
                         "workload")
    ap.add_argument("--levels", action="store_true",
                    help="tree-shaped decode batches: flat vs two-level vs multi-level "
                         "cascade, one line each")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    return ap.parse_args(argv)


# ----------------------------------------------------------------- distributed --
class Dist:
    """Rank bookkeeping; a process group only when launched with WORLD_SIZE > 1."""

    def __init__(self, backend=None):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend=backend or "nccl")
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x: float) -> float:
        return self._reduce(x, "max")

    def sum(self, x: float) -> float:
        return self._reduce(x, "sum")

    def _reduce(self, x, op):
        if self.pg is None:
            return float(x)
        import torch
        dev = "cuda" if self.pg.get_backend() == "nccl" else "cpu"
        t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX if op == "max" else self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


def aggregate(dist: Dist, queries_local: float, elapsed_s_local: float):
    """Whole-job throughput: every rank's queries over the slowest rank's time."""
    total = dist.sum(queries_local)
    slowest = dist.max(elapsed_s_local)
    return total / slowest if slowest > 0 else 0.0, slowest


# ---------------------------------------------------------------------- clocks --
class ClockSampler:
    """nvidia-smi samples (every 200 ms) kept with their wall-clock timestamps."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(gpu_index), "-lms", "200"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        inside = [l for (t, l) in self.lines if t0 <= t <= t1 + 0.25]
        window = "timed region"
        if not inside:  # region shorter than one sample period: nearest samples
            near = sorted(self.lines, key=lambda x: min(abs(x[0] - t0), abs(x[0] - t1)))
            inside = [l for (_, l) in near[:3]]
            window = "nearest samples (timed region shorter than the 200 ms period)"
        sm, smax, power, reasons = [], [], [], set()
        for l in inside:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "window": "no samples"}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons),
                "samples": len(sm), "window": window}


# ------------------------------------------------------------------- workloads --
def make_batch(name: str, rank: int):
    from shared_prefix_paged_gb300 import workloads
    if name == "decode":
        return workloads.decode_batch(seed=1002 + 7919 * rank)
    if name == "tiny":
        return workloads.tiny_decode(seed=1001 + 7919 * rank)
    if name == "chunked":
        return workloads.chunked_prefill(seed=1003 + 7919 * rank)
    if name == "long":
        return workloads.long_prefix(seed=1004 + 7919 * rank)
    raise SystemExit(f"unknown workload {name}")


def kernel_source_sha(kernel: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "shared_prefix_paged_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path, encoding="utf-8") as f:
            table = json.load(f)
    except (OSError, ValueError):
        return None
    e = table.get(f"{kernel}@{workload}")
    if not e or e.get("source_sha") != kernel_source_sha(kernel):
        return None
    return e.get("bytes_per_launch")


class DeviceRun:
    """Device copies of one batch and the CUDA graphs that replay its steps."""

    def __init__(self, b, copies: int, device):
        import torch
        from shared_prefix_paged_gb300 import csp
        self.b, self.dev, self.R = b, device, copies
        self.q = [b.q.to(device) for _ in range(copies)]
        self.k = [b.k_cache.to(device) for _ in range(copies)]
        self.v = [b.v_cache.to(device) for _ in range(copies)]
        self.bt = torch.from_numpy(b.block_table).to(device)
        self.cu = torch.from_numpy(b.cu_seqlens_q).to(device)
        self.sl = torch.from_numpy(b.seq_lens).to(device)
        self.out = [torch.empty_like(self.q[0]) for _ in range(copies)]
        self.lse = [torch.empty((b.total_q, b.num_q_heads), dtype=torch.float32, device=device)
                    for _ in range(copies)]
        lib = csp.load()
        # host planner with pre-made ctypes arguments
        self._bt_h = np.ascontiguousarray(b.block_table, dtype=np.int32)
        self._sl_h = np.ascontiguousarray(b.seq_lens, dtype=np.int32)
        self._nc_h = np.ascontiguousarray(b.num_computed_tokens, dtype=np.int32)
        self._cpl = ctypes.c_int32(0)
        self._use = ctypes.c_int32(0)
        self._plan_fn = lib.cascade_plan
        self._plan_args = (ctypes.c_void_p(self._bt_h.ctypes.data), self._bt_h.shape[1],
                           b.num_reqs, ctypes.c_void_p(self._sl_h.ctypes.data),
                           ctypes.c_void_p(self._nc_h.ctypes.data), b.block_size,
                           b.num_q_heads, b.num_kv_heads, b.head_dim, 0, csp.MODE_AUTO,
                           ctypes.byref(self._cpl), ctypes.byref(self._use))
        self.plan()
        self.cpl, self.use_cascade = int(self._cpl.value), bool(self._use.value)
        need = max(csp.workspace_size(b.num_reqs, b.total_q, b.max_seqlen_q, b.max_seqlen_k,
                                      c, b.num_q_heads, b.num_kv_heads, b.head_dim)
                   for c in (0, self.cpl))
        self.ws = csp.alloc_workspace(need, device)
        self.schedule, self.prefix_ranges = csp.cascade_schedule(
            b.num_reqs, b.total_q, b.max_seqlen_q, b.max_seqlen_k, self.cpl, b.num_q_heads,
            b.num_kv_heads, b.head_dim) if self.use_cascade else (csp.SCHEDULE_TWO_KERNELS, 0)
        self.single = self.schedule == csp.SCHEDULE_SINGLE
        # the suffix (or flat) kernel: tcgen05 once a request has more than 16 packed
        # rows (query, head-in-group) per KV head, the warp-MMA kernel below that
        self.suffix_kernel = ("paged_tc_kernel"
                              if b.max_seqlen_q * (b.num_q_heads // b.num_kv_heads) > 16
                              else "paged_attn_kernel")
        # the two-kernel schedule's suffix (either kernel) leaves the merge to a third one
        self.merge_after = self.use_cascade and not self.single and self.cpl > 0

    def setup_levels(self, max_levels: int):
        """The multi-level plan of the batch and its workspace."""
        import torch
        from shared_prefix_paged_gb300 import csp
        b = self.b
        self.segs, self.start = csp.cascade_plan_levels(
            b.block_table, b.seq_lens, b.num_computed_tokens, block_size=b.block_size,
            max_levels=max_levels)
        self.start_dev = torch.from_numpy(self.start).to(self.dev)
        self.max_suffix = int((b.seq_lens - self.start).max())
        self.ws_levels = csp.alloc_workspace(csp.workspace_size_levels(
            b.num_reqs, b.total_q, b.max_seqlen_q, b.max_seqlen_k, self.segs, self.max_suffix,
            b.num_q_heads, b.num_kv_heads, b.head_dim), self.dev)

    def plan(self):
        st = self._plan_fn(*self._plan_args)
        if st != 0:
            raise RuntimeError(f"cascade_plan failed: {st}")

    def step(self, i: int, path: str, events=None):
        from shared_prefix_paged_gb300 import csp
        b = self.b
        common = dict(max_seqlen_q=b.max_seqlen_q, max_seqlen_k=b.max_seqlen_k,
                      softmax_scale=b.scale, out=self.out[i], lse=self.lse[i], workspace=self.ws)
        if path == "levels":
            csp.cascade_attn_levels(self.q[i], self.k[i], self.v[i], self.bt, self.cu, self.sl,
                                    segments=self.segs, suffix_start=self.start_dev,
                                    max_suffix_len=self.max_suffix,
                                    **dict(common, workspace=self.ws_levels))
        elif path == "cascade":
            csp.cascade_attn(self.q[i], self.k[i], self.v[i], self.bt, self.cu, self.sl,
                             common_prefix_len=self.cpl, phase_events=events, **common)
        else:
            csp.paged_attn(self.q[i], self.k[i], self.v[i], self.bt, self.cu, self.sl, **common)

    def graph(self, path: str, n_steps: int, events=None):
        import torch
        s = torch.cuda.Stream(self.dev)
        s.wait_stream(torch.cuda.current_stream(self.dev))
        with torch.cuda.stream(s):
            for i in range(n_steps):
                self.step(i % self.R, path, events[i] if events else None)
        torch.cuda.current_stream(self.dev).wait_stream(s)
        torch.cuda.synchronize(self.dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n_steps):
                self.step(i % self.R, path, events[i] if events else None)
        return g


def time_graph_steps(run: DeviceRun, path: str, steps: int, warmup: int, dist: Dist,
                     with_planner=True, clocks=None):
    """Replay `steps` device steps from graphs; returns (elapsed_s, host_s, t0, t1).

    With the planner, the host plans one graph's worth of steps ahead: the plans of the
    first R steps run before the timed region, and after each replay is queued the host
    plans the next R steps while the GPU runs it (the last round plans steps that never
    run).  The timed region thus holds exactly `steps` planner calls and `steps` device
    steps, and the GPU never waits for the host at its start."""
    import torch
    R = run.R
    g = run.graph(path, R)
    tail = steps % R
    g_tail = run.graph(path, tail) if tail else None
    for _ in range(max(1, math.ceil(warmup / R))):
        g.replay()
    torch.cuda.synchronize(run.dev)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    rounds = [R] * (steps // R) + ([tail] if tail else [])
    if with_planner:
        for _ in range(rounds[0]):       # the first round's plans
            run.plan()
    dist.barrier()
    torch.cuda.synchronize(run.dev)
    t0 = time.time()
    h0 = time.perf_counter()
    start.record()
    for k, n in enumerate(rounds):
        (g if n == R else g_tail).replay()
        if with_planner:
            # the next round's plans (after the last round: as many as the first
            # round's, which ran before the region, so every step has one)
            for _ in range(rounds[k + 1] if k + 1 < len(rounds) else rounds[0]):
                run.plan()
    end.record()
    h1 = time.perf_counter()
    torch.cuda.synchronize(run.dev)
    t1 = time.time()
    dist.barrier()
    return start.elapsed_time(end) / 1e3, h1 - h0, t0, t1


def phase_times(run: DeviceRun, rounds: int = 16, batches: int = 3):
    """Average device time of each kernel of a cascade step, from CUDA events recorded
    by cascade_attn_timed between its kernels on the launching stream (with events
    between them the two kernels run back to back instead of overlapping).  A GPU sleep
    queued first lets the host enqueue every step before the GPU reaches them, so the
    steps run back to back with no host gaps inside the event intervals."""
    import torch
    R = run.R
    n_steps = R * rounds
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_steps)]
    for evs in events:       # torch creates the CUDA event on its first record
        for ev in evs:
            ev.record()
    for i in range(R):       # warm
        run.step(i, "cascade")
    torch.cuda.synchronize(run.dev)
    acc = np.zeros(3)
    n = 0
    for _ in range(batches):
        torch.cuda._sleep(50_000_000)   # ~25 ms of GPU time while the host enqueues
        for i in range(n_steps):
            run.step(i % R, "cascade", events[i])
        torch.cuda.synchronize(run.dev)
        for ev in events:
            acc += [ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2]),
                    ev[2].elapsed_time(ev[3])]
            n += 1
    ms = acc / n
    if run.single:
        # one kernel: events 0 and 1 bracket it, event 2 follows immediately
        return {"decode_cascade_kernel": ms[0] * 1e3, "launches_averaged": n}
    out = {"prefix_attn_kernel": ms[0] * 1e3, run.suffix_kernel: ms[1] * 1e3}
    if run.merge_after:
        out["merge_slots_kernel"] = ms[2] * 1e3
    out["launches_averaged"] = n
    return out


def e2e_steps(run: DeviceRun, steps: int):
    """End-to-end steps through the C ABI with host buffers: `cascade_step_host` (one
    call per step) copies the step's q, block table, cu_seqlens and seq_lens from
    pinned host memory to the device, plans on the host, runs the attention call,
    copies out and lse back to pinned host memory and waits.  The KV caches stay
    resident (R copies, rotated as in the device timing).  Returns the rate, the bytes
    copied each way per step and the step count."""
    import torch
    from shared_prefix_paged_gb300 import csp
    b = run.b
    dev = run.dev
    pin = lambda t: t.contiguous().pin_memory()
    q_h = pin(b.q)
    bt_h = pin(torch.from_numpy(np.ascontiguousarray(b.block_table)))
    cu_h = pin(torch.from_numpy(b.cu_seqlens_q))
    sl_h = pin(torch.from_numpy(b.seq_lens))
    nc_h = pin(torch.from_numpy(b.num_computed_tokens))
    out_h = torch.empty(b.q.shape, dtype=torch.bfloat16).pin_memory()
    lse_h = torch.empty((b.total_q, b.num_q_heads), dtype=torch.float32).pin_memory()
    need = max(csp.step_scratch_size(b.cu_seqlens_q, b.seq_lens, b.block_table.shape[1], c,
                                     b.num_q_heads, b.num_kv_heads, b.head_dim)
               for c in (0, run.cpl))
    scratch = csp.alloc_workspace(need, dev)
    calls = [csp.HostStep(q_h, bt_h, cu_h, sl_h, nc_h, run.k[i], run.v[i],
                          softmax_scale=b.scale, out=out_h, lse=lse_h, scratch=scratch)
             for i in range(run.R)]
    h2d = sum(t.numel() * t.element_size() for t in (q_h, bt_h, cu_h, sl_h))
    d2h = out_h.numel() * 2 + lse_h.numel() * 4
    for i in range(5):
        calls[i % run.R]()
    t0 = time.perf_counter()
    for s in range(steps):
        calls[s % run.R]()
    el = time.perf_counter() - t0
    return b.total_q * steps / el, h2d, d2h, steps


def e2e_breakdown(run: DeviceRun, steps: int):
    """The same step's parts issued one by one from Python, for a breakdown: one H2D
    copy of the step's inputs (packed in one pinned buffer), the host planner
    (csp.Planner), the attention call (csp.PreparedCall), one D2H copy of out and lse,
    then the host waits; host parts by perf_counter, device parts by CUDA events on the
    stream.  Returns the average time of each part."""
    import torch
    from shared_prefix_paged_gb300 import csp
    b = run.b
    dev = run.dev
    parts = [("q", b.q.view(torch.int16).reshape(-1)),
             ("bt", torch.from_numpy(np.ascontiguousarray(b.block_table)).reshape(-1)),
             ("cu", torch.from_numpy(b.cu_seqlens_q)),
             ("sl", torch.from_numpy(b.seq_lens))]
    sizes = [t.numel() * t.element_size() for _, t in parts]
    offs = np.cumsum([0] + [(n + 255) // 256 * 256 for n in sizes])
    in_h = torch.empty(int(offs[-1]), dtype=torch.uint8).pin_memory()
    for (name, t), o, n in zip(parts, offs, sizes):
        in_h[o:o + n].copy_(t.contiguous().view(torch.uint8))
    in_d = torch.empty(int(offs[-1]), dtype=torch.uint8, device=dev)
    q_d = in_d[offs[0]:offs[0] + sizes[0]].view(torch.bfloat16).view(b.q.shape)
    bt_d = in_d[offs[1]:offs[1] + sizes[1]].view(torch.int32).view(b.block_table.shape)
    cu_d = in_d[offs[2]:offs[2] + sizes[2]].view(torch.int32)
    sl_d = in_d[offs[3]:offs[3] + sizes[3]].view(torch.int32)
    o_bytes = b.q.numel() * 2
    l_bytes = b.total_q * b.num_q_heads * 4
    res_d = torch.empty(o_bytes + l_bytes, dtype=torch.uint8, device=dev)
    res_h = torch.empty(o_bytes + l_bytes, dtype=torch.uint8).pin_memory()
    out_d = res_d[:o_bytes].view(torch.bfloat16).view(b.q.shape)
    lse_d = res_d[o_bytes:].view(torch.float32).view(b.total_q, b.num_q_heads)
    stream = torch.cuda.current_stream(dev)
    planner = csp.Planner(b.block_table, b.seq_lens, b.num_computed_tokens,
                          block_size=b.block_size, num_q_heads=b.num_q_heads,
                          num_kv_heads=b.num_kv_heads, head_dim=b.head_dim)
    calls = [csp.PreparedCall(q_d, run.k[i], run.v[i], bt_d, cu_d, sl_d,
                              max_seqlen_q=b.max_seqlen_q, max_seqlen_k=b.max_seqlen_k,
                              softmax_scale=b.scale, out=out_d, lse=lse_d, workspace=run.ws,
                              stream=stream) for i in range(run.R)]
    h2d = int(sum(sizes))
    d2h = o_bytes + l_bytes
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    acc = np.zeros(6)

    def one(i, timed):
        h0 = time.perf_counter()
        if timed:
            ev[0].record(stream)
        in_d.copy_(in_h, non_blocking=True)
        if timed:
            ev[1].record(stream)
        h1 = time.perf_counter()
        cpl, use = planner()
        h2 = time.perf_counter()
        calls[i](cpl, use)
        h3 = time.perf_counter()
        if timed:
            ev[2].record(stream)
        res_h.copy_(res_d, non_blocking=True)
        if timed:
            ev[3].record(stream)
        stream.synchronize()
        h4 = time.perf_counter()
        return np.array([h1 - h0, h2 - h1, h3 - h2, h4 - h3, 0.0, 0.0])

    for i in range(5):
        one(i % run.R, False)
    t0 = time.perf_counter()
    for s in range(steps):
        one(s % run.R, False)
    el = time.perf_counter() - t0
    # the breakdown, from separate instrumented steps (events add host work)
    n_bd = min(steps, 500)
    dev_ms = np.zeros(3)
    for s in range(n_bd):
        acc += one(s % run.R, True)
        dev_ms += [ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2]),
                   ev[2].elapsed_time(ev[3])]
    acc /= n_bd
    dev_ms /= n_bd
    breakdown = {"host_h2d_issue_us": round(acc[0] * 1e6, 2),
                 "host_planner_us": round(acc[1] * 1e6, 2),
                 "host_attention_call_us": round(acc[2] * 1e6, 2),
                 "host_d2h_issue_and_wait_us": round(acc[3] * 1e6, 2),
                 "device_h2d_us": round(dev_ms[0] * 1e3, 2),
                 "device_plan_to_kernel_end_us": round(dev_ms[1] * 1e3, 2),
                 "device_d2h_us": round(dev_ms[2] * 1e3, 2),
                 "step_us": round(el / steps * 1e6, 2)}
    return breakdown


def cpu_oracle_rate(b, seconds: float, rng_seed=0):
    """The oracle as it stands on this host's cores: rows (token, head) sampled from the
    batch, as many as fill about `seconds`; returns (queries/s, threads, rows)."""
    import oracle
    threads = os.cpu_count() or 1
    rng = np.random.default_rng(rng_seed)
    total = b.total_q * b.num_q_heads

    def run_rows(n):
        flat = rng.choice(total, size=n, replace=n > total)
        rows = np.stack([flat // b.num_q_heads, flat % b.num_q_heads], 1).astype(np.int32)
        t0 = time.perf_counter()
        oracle.attention(b.q, b.k_cache, b.v_cache, b.block_table, b.cu_seqlens_q, b.seq_lens,
                         b.scale, rows=rows, n_threads=threads)
        return time.perf_counter() - t0

    n = max(threads, 16)
    el = run_rows(n)
    # grow the sample until one run fills about `seconds` (thread start-up dominates
    # small probes, so estimate from the previous run each time)
    while el < 0.7 * seconds and n < 400 * total:
        n = int(min(400 * total, max(2 * n, n * seconds / max(el, 1e-6))))
        el = run_rows(n)
    return (n / b.num_q_heads) / el, threads, n


def roofline_entry(kernel, us, b, run, peaks, workload):
    """Algorithmic bytes (and flops) per launch of a kernel of the cascade step."""
    from shared_prefix_paged_gb300 import accounting
    rows = b.total_q * b.num_q_heads
    kvtok = accounting.kv_bytes_per_token(b.num_kv_heads, b.head_dim)
    q_bytes = rows * b.head_dim * 2
    cpl = run.cpl
    if kernel == "decode_cascade_kernel":
        # the whole step in one launch: KV once, q read, out + lse written
        bytes_ = accounting.cascade_min_bytes(b, cpl)
        flops = None
    elif kernel == "merge_slots_kernel":
        # every row: its slots read (the prefix ranges and one suffix split), out + lse
        # written
        n_slots = run.prefix_ranges + 1
        bytes_ = rows * (n_slots * (b.head_dim * 2 + 4) + b.head_dim * 2 + 4)
        flops = None
    elif kernel == "prefix_attn_kernel":
        # prefix KV once, q, and one partial per row (bf16 O, fp32 LSE)
        bytes_ = cpl * kvtok + q_bytes + rows * (b.head_dim * 2 + 4)
        flops = accounting.prefix_flops(b.total_q, b.num_q_heads, b.head_dim, cpl)
    else:
        # each request's KV after the prefix, q, and the final bf16 output + LSE
        bytes_ = (int((b.seq_lens.astype(np.int64) - cpl).sum()) * kvtok + q_bytes +
                  rows * (b.head_dim * 2 + 4))
        flops = None
    gbs = bytes_ / (us * 1e-6) / 1e9
    hbm_frac = gbs / peaks["hbm_gbs"]
    entry = {"kernel": kernel, "bound": "hbm", "achieved": round(gbs, 1),
             "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(hbm_frac, 4),
             "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json hbm_gbs)",
             "algorithmic_bytes_per_launch": int(bytes_), "us_per_launch": round(us, 3),
             "traffic": committed_traffic(kernel, workload)}
    if flops:
        tf = flops / (us * 1e-6) / 1e12
        tfrac = tf / peaks["bf16_tflops"]
        entry["tensor"] = {"achieved": round(tf, 1), "peak": peaks["bf16_tflops"],
                           "unit": "TFLOP/s", "frac": round(tfrac, 4),
                           "flops_per_launch": int(flops)}
        if tfrac > hbm_frac:
            entry.update(bound="tensor", achieved=round(tf, 1), peak=peaks["bf16_tflops"],
                         unit="TFLOP/s", frac=round(tfrac, 4),
                         peak_source=f"{peaks['source']} (MEASURED_PEAKS.json bf16_tflops, "
                                     "burst)")
    return entry


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json"), encoding="utf-8") as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def default_copies(b):
    """Copies of q and the KV pool so that > 2x L2 is touched between reuses of one."""
    per_copy = (b.k_cache.numel() + b.v_cache.numel() + b.q.numel()) * 2
    return int(min(8, max(2, math.ceil(2 * L2_BYTES / max(per_copy, 1)) + 1)))


# ------------------------------------------------------------------------ arms --
def run_ours(args, dist: Dist):
    import torch
    from shared_prefix_paged_gb300 import accounting, csp
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(dist.local_rank)
    device = torch.device("cuda", dist.local_rank)
    csp.load()
    b = make_batch(args.workload, dist.rank)
    R = args.copies or default_copies(b)
    run = DeviceRun(b, R, device)
    path = "cascade" if run.use_cascade else "flat"
    peaks = load_peaks()
    K, W = args.steps, max(3, args.warmup)

    clocks = ClockSampler(dist.local_rank) if dist.rank == 0 else None
    time.sleep(0.5 if clocks else 0.0)
    elapsed, host_s, t0, t1 = time_graph_steps(run, path, K, W, dist)
    if clocks:
        clocks.stop()
    qps, slowest = aggregate(dist, b.total_q * K, elapsed)
    us_call = elapsed / K * 1e6
    min_bytes = accounting.cascade_min_bytes(b, run.cpl if path == "cascade" else 0)
    kv_bytes = (accounting.cascade_kv_tokens(b.seq_lens, run.cpl) if path == "cascade"
                else accounting.flat_kv_tokens(b.seq_lens)) * accounting.kv_bytes_per_token(
                    b.num_kv_heads, b.head_dim)
    result = {
        "metric": METRIC, "value": round(qps, 1), "unit": UNIT, "n_gpus": dist.world,
        "steps": K, "warmup": W, "ms_per_step": round(slowest / K * 1e3, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 Q/K/V, shuffled physical blocks)",
        "config": {
            "workload": b.name, "num_reqs": b.num_reqs, "total_q": b.total_q,
            "common_prefix_len": run.cpl, "q_heads": b.num_q_heads, "kv_heads": b.num_kv_heads,
            "head_dim": b.head_dim, "block_size": b.block_size, "path": path,
            "schedule": ("single kernel" if run.single else "prefix + suffix kernels")
                        if path == "cascade" else "flat", "prefix_ranges": run.prefix_ranges,
            "l2": f"inputs larger than L2: {R} rotating copies of q and the KV cache",
            "step": "host cascade_plan + device path replayed from a CUDA graph of "
                    f"{R} steps (the host plans the next {R} steps while the GPU runs "
                    "these)", "parallelism": f"replicas x{dist.world}"},
        "us_per_call": round(us_call, 3),
        "kv_gbs": round(kv_bytes / (us_call * 1e-6) / 1e9, 1),
        "min_bytes_per_call": int(min_bytes),
        "hbm_frac_of_measured": round(min_bytes / (us_call * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
        "hbm_frac_of_8tbs": round(min_bytes / (us_call * 1e-6) / 1e9 / 8000.0, 4),
        "host_s_in_timed_region": round(host_s, 4),
        "gpu_launches": K * ((3 if run.merge_after else 2)
                             if path == "cascade" and not run.single else 1),
    }
    if clocks:
        result["clocks"] = clocks.summary(t0, t1)

    if path == "cascade":
        ph = phase_times(run)
        kernels = (["decode_cascade_kernel"] if run.single
                   else ["prefix_attn_kernel", run.suffix_kernel] +
                   (["merge_slots_kernel"] if run.merge_after else []))
        if run.single:
            # one launch per step: the launch's average duration over the timed region
            # is the region's event time / K (an isolated launch, timed with events
            # right around it, also carries the launch gap)
            result["isolated_launch_us"] = round(ph["decode_cascade_kernel"], 3)
            ph["decode_cascade_kernel"] = us_call
        entries = {k: roofline_entry(k, ph[k], b, run, peaks, b.name) for k in kernels}
        dominant = max(kernels, key=lambda k: ph[k])
        result["roofline"] = entries[dominant]
        result["phases_us"] = {k: round(ph[k], 3) for k in kernels}
        result["phases_roofline"] = {k: {kk: entries[k][kk] for kk in
                                         ("bound", "achieved", "unit", "frac")}
                                     for k in kernels}
        result["phase_launches_averaged"] = ph["launches_averaged"]

    if not args.quick:
        # the standard (flat) path on the same batch, for the cascade speedup
        fe, _, _, _ = time_graph_steps(run, "flat", max(R, min(K, 2000)), W, dist,
                                       with_planner=False)
        flat_us = fe / max(R, min(K, 2000)) * 1e6
        result["flat"] = {"us_per_call": round(flat_us, 3),
                          "speedup_cascade_over_flat": round(flat_us / us_call, 3),
                          "kv_bytes": int(accounting.flat_kv_tokens(b.seq_lens) *
                                          accounting.kv_bytes_per_token(b.num_kv_heads,
                                                                        b.head_dim))}
        e_qps, h2d, d2h, e_steps = e2e_steps(run, min(K, 3000))
        bd = e2e_breakdown(run, min(K, 500))
        e_total, _ = aggregate(dist, e_qps, 1.0)
        result["e2e"] = {"value": round(e_total, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                         "d2h_bytes_per_step": d2h, "steps": e_steps,
                         "call": "cascade_step_host (C ABI, host buffers): H2D of q, block "
                                 "table, cu_seqlens, seq_lens from pinned memory, host "
                                 "planner, attention call, D2H of out + lse, host waits; "
                                 "KV cache resident",
                         "breakdown_python_parts": bd}
        if dist.rank == 0 and dist.world == 1:
            rate, threads, rows = cpu_oracle_rate(b, args.cpu_seconds)
            result["cpu_baseline"] = {"value": round(rate, 3), "unit": UNIT, "cores": threads,
                                      "kind": "oracle",
                                      "sample": f"{rows} random (token, head) rows of the "
                                                f"same batch, fp64 C oracle, {threads} threads"}
    return result


def run_reference(args, dist: Dist):
    """The CPU oracle as the reference arm: each step a bounded row sample."""
    import oracle
    b = make_batch(args.workload, 0)
    threads = os.cpu_count() or 1
    K, W = args.steps, max(3, args.warmup)
    total = b.total_q * b.num_q_heads
    rng = np.random.default_rng(0)

    def sample(n):
        flat = rng.choice(total, size=n, replace=n > total)
        return np.stack([flat // b.num_q_heads, flat % b.num_q_heads], 1).astype(np.int32)

    n = max(threads, 16)
    while True:   # per-row cost at a sample size where thread start-up is amortised
        t0 = time.perf_counter()
        oracle.attention(b.q, b.k_cache, b.v_cache, b.block_table, b.cu_seqlens_q, b.seq_lens,
                         b.scale, rows=sample(n), n_threads=threads)
        el = time.perf_counter() - t0
        if el > 1.0 or n >= total:
            break
        n = min(total, 4 * n)
    per_row = el / n
    budget = 120.0  # seconds for the whole run
    rows_per_step = int(max(1, min(total, budget / (K + W) / max(per_row, 1e-9))))
    for _ in range(W):
        oracle.attention(b.q, b.k_cache, b.v_cache, b.block_table, b.cu_seqlens_q,
                         b.seq_lens, b.scale, rows=sample(rows_per_step), n_threads=threads)
    t0 = time.perf_counter()
    for _ in range(K):
        oracle.attention(b.q, b.k_cache, b.v_cache, b.block_table, b.cu_seqlens_q,
                         b.seq_lens, b.scale, rows=sample(rows_per_step), n_threads=threads)
    el = time.perf_counter() - t0
    qps = rows_per_step * K / b.num_q_heads / el
    sample_desc = (f"{rows_per_step} random (token, head) rows per step of the same batch, "
                   f"fp64 C oracle, {threads} threads")
    return {"impl": "reference", "metric": METRIC, "value": round(qps, 3), "unit": UNIT,
            "n_gpus": dist.world, "steps": K, "warmup": W,
            "ms_per_step": round(el / K * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": b.name, "num_reqs": b.num_reqs, "total_q": b.total_q,
                       "q_heads": b.num_q_heads, "kv_heads": b.num_kv_heads,
                       "head_dim": b.head_dim, "block_size": b.block_size},
            "cpu_baseline": {"value": round(qps, 3), "unit": UNIT, "cores": threads,
                             "kind": "oracle", "sample": sample_desc},
            "e2e": {"value": round(qps, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def run_sweep(args, dist: Dist):
    """Cascade vs flat at every point of the N x P decode grid (S=128)."""
    import torch
    from shared_prefix_paged_gb300 import accounting, csp, workloads
    torch.cuda.set_device(dist.local_rank)
    device = torch.device("cuda", dist.local_rank)
    for n in workloads.SWEEP_N:
        for p in workloads.SWEEP_P:
            b = workloads.sweep_point(n, p)
            R = args.copies or default_copies(b)
            run = DeviceRun(b, R, device)
            steps = max(R, min(args.steps, 600))
            pc, _ = csp.cascade_plan(b.block_table, b.seq_lens, b.num_computed_tokens,
                                     mode=csp.MODE_PAGE_THRESHOLDS)
            ce, _, _, _ = time_graph_steps(run, "cascade", steps, args.warmup, dist, False)
            fe, _, _, _ = time_graph_steps(run, "flat", steps, args.warmup, dist, False)
            line = {"sweep": True, "N": n, "P": p, "S": 128, "cpl": run.cpl,
                    "cascade_us": round(ce / steps * 1e6, 3), "flat_us": round(fe / steps * 1e6, 3),
                    "speedup": round(fe / ce, 3),
                    "auto_pick": "cascade" if run.use_cascade else "flat",
                    "pages_rule_pick": "cascade" if pc >= 256 and n >= 8 else "flat",
                    "kv_ratio": round(accounting.flat_kv_tokens(b.seq_lens) /
                                      accounting.cascade_kv_tokens(b.seq_lens, run.cpl), 2)}
            if dist.rank == 0:
                print(json.dumps(line), flush=True)
            del run
            torch.cuda.empty_cache()


def run_levels(args, dist: Dist):
    """Flat, two-level and multi-level cascade on tree-shaped decode batches (families of
    requests over one system prompt, each family over its own document)."""
    import torch
    from shared_prefix_paged_gb300 import accounting, csp, workloads
    torch.cuda.set_device(dist.local_rank)
    device = torch.device("cuda", dist.local_rank)
    peaks = load_peaks()
    for fam, per, system, doc in ((8, 16, 2048, 4096), (4, 16, 1024, 8192),
                                  (16, 8, 4096, 2048)):
        b = workloads.tree_families(families=fam, per_family=per, system=system, doc=doc)
        R = args.copies or default_copies(b)
        run = DeviceRun(b, R, device)
        run.setup_levels(max_levels=3)
        steps = max(R, min(args.steps, 2000))
        t = {}
        for path in ("flat", "cascade", "levels"):
            e, _, _, _ = time_graph_steps(run, path, steps, args.warmup, dist, False)
            t[path] = e / steps * 1e6
        lv = accounting.levels_min_bytes(b, run.segs, run.start)
        line = {"levels": True, "workload": b.name, "num_reqs": b.num_reqs,
                "segments": int(run.segs.shape[0]), "cpl": run.cpl,
                "flat_us": round(t["flat"], 3), "cascade_us": round(t["cascade"], 3),
                "levels_us": round(t["levels"], 3),
                "levels_vs_cascade": round(t["cascade"] / t["levels"], 3),
                "levels_vs_flat": round(t["flat"] / t["levels"], 3),
                "kv_tokens": {"flat": accounting.flat_kv_tokens(b.seq_lens),
                              "cascade": accounting.cascade_kv_tokens(b.seq_lens, run.cpl),
                              "levels": accounting.levels_kv_tokens(b.seq_lens, run.segs,
                                                                    run.start)},
                "levels_hbm_frac": round(lv / (t["levels"] * 1e-6) / 1e9 / peaks["hbm_gbs"], 3),
                "peak_source": peaks["source"]}
        if dist.rank == 0:
            print(json.dumps(line), flush=True)
        del run
        torch.cuda.empty_cache()


def run_fp8(args, dist: Dist):
    """bf16 and FP8 (E4M3, per-tensor scales) KV caches on the same batches: cascade and
    the standard path, microseconds per call and minimal bytes / time."""
    import torch
    from shared_prefix_paged_gb300 import accounting, csp
    torch.cuda.set_device(dist.local_rank)
    device = torch.device("cuda", dist.local_rank)
    peaks = load_peaks()
    for name in ("decode", "chunked"):
        b = make_batch(name, dist.rank)
        R = args.copies or default_copies(b)
        run = DeviceRun(b, R, device)
        # scales that map the largest used magnitude just inside E4M3's range (the +-1000
        # poison of unused slots aside); the bytes are drawn on the device
        def amax(t):
            x = t.float().abs()
            return float(x[torch.isfinite(x) & (x < 999.0)].max())
        ks, vs = amax(run.k[0]) / 440.0, amax(run.v[0]) / 440.0
        k8 = [(run.k[i].float() / ks).to(torch.float8_e4m3fn).view(torch.uint8)
              for i in range(R)]
        v8 = [(run.v[i].float() / vs).to(torch.float8_e4m3fn).view(torch.uint8)
              for i in range(R)]
        ws8 = csp.alloc_workspace(csp.workspace_size_fp8kv(
            b.num_reqs, b.total_q, b.max_seqlen_q, b.max_seqlen_k, run.cpl, b.num_q_heads,
            b.num_kv_heads, b.head_dim), device)
        steps = max(R, min(args.steps, 2000))
        t = {}
        for path in ("cascade", "flat"):
            e, _, _, _ = time_graph_steps(run, path, steps, args.warmup, dist, False)
            t["bf16_" + path] = e / steps * 1e6

        class Fp8Run:
            """DeviceRun's graph interface over the E4M3 caches."""
            def __init__(self, cpl):
                self.R, self.dev, self.cpl = R, device, cpl

            def graph(self, path, n, events=None):
                def step(i):
                    csp.attn_fp8kv(run.q[i], k8[i], v8[i], run.bt, run.cu, run.sl,
                                   max_seqlen_q=b.max_seqlen_q, max_seqlen_k=b.max_seqlen_k,
                                   softmax_scale=b.scale, k_scale=ks, v_scale=vs,
                                   common_prefix_len=self.cpl, out=run.out[i], lse=run.lse[i],
                                   workspace=ws8)
                s = torch.cuda.Stream(device)
                s.wait_stream(torch.cuda.current_stream(device))
                with torch.cuda.stream(s):
                    for i in range(n):
                        step(i % R)
                torch.cuda.current_stream(device).wait_stream(s)
                torch.cuda.synchronize(device)
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    for i in range(n):
                        step(i % R)
                return g

        for path, cpl in (("cascade", run.cpl), ("flat", 0)):
            e, _, _, _ = time_graph_steps(Fp8Run(cpl), path, steps, args.warmup, dist, False)
            t["fp8_" + path] = e / steps * 1e6
        kv8 = accounting.cascade_min_bytes(b, run.cpl) - accounting.cascade_kv_tokens(
            b.seq_lens, run.cpl) * accounting.kv_bytes_per_token(b.num_kv_heads, b.head_dim) // 2
        line = {"fp8": True, "workload": b.name, "cpl": run.cpl,
                "k_scale": ks, "v_scale": vs,
                **{k + "_us": round(v, 3) for k, v in t.items()},
                "fp8_cascade_min_bytes": kv8,
                "fp8_cascade_hbm_frac": round(kv8 / (t["fp8_cascade"] * 1e-6) / 1e9 /
                                              peaks["hbm_gbs"], 3),
                "peak_source": peaks["source"]}
        if dist.rank == 0:
            print(json.dumps(line), flush=True)
        del run
        torch.cuda.empty_cache()


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        # rank 0 alone runs the CPU oracle; other ranks exit without work
        if int(os.environ.get("RANK", "0")) != 0:
            return 0
        os.environ["WORLD_SIZE"] = "1"
        print(json.dumps(run_reference(args, Dist())), flush=True)
        return 0
    dist = Dist()
    try:
        if args.sweep:
            run_sweep(args, dist)
            return 0
        if args.levels:
            run_levels(args, dist)
            return 0
        if args.fp8:
            run_fp8(args, dist)
            return 0
        res = run_ours(args, dist)
        if dist.rank == 0:
            print(json.dumps(res), flush=True)
        return 0
    finally:
        dist.close()


if __name__ == "__main__":
    sys.exit(main())
