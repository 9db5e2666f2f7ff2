"""Throughput of the batch-invariant hot path on GB300.

One step = one speculative-verify step of M = 8 tokens through every reduction of the
path, on the pages' shapes:
  1. bi_rmsnorm       x [8, 4096] bf16 (eps 1e-5)
  2. bi_matmul (NK)   [8, 4096] x W[4096, 4096] stored [N, K]  -> q  [8, 32, 128]
  3. bi_kv_append     the block's 8 new K/V tokens (8 KV heads, head_dim 128)
  4. bi_verify_block  1 sequence, causal block of q = 8, Lk = 65540, 32 query heads /
                      8 KV heads, bf16 paged cache (64-token pages, permuted)
  5. bi_matmul (KN)   [8, 4096] x W[4096, 4096] stored [K, N]  -> y  [8, 4096]
All of it is HBM-bound at M = 8, so `value` is the step's algorithmic bytes (every
operand read once, every result written once) divided by the device time of the step:
whole-job GB/s over all ranks.  Inputs are resident in HBM before the timed region; the
step streams ~336 MB (KV cache 268 MB + two 32 MiB weights), more than 2x the 126 MB L2,
so no input survives in L2 from one step to the next.

`python bench.py [--gpus N --steps K --warmup W]` prints one JSON line.
`--impl reference` times the plain CPU oracle on a bounded sample of the same step.
`--sweep` prints extra lines (GEMM M sweep vs cuBLAS, RMSNorm and attention configs).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "invariant GEMM TFLOP/s & decode-attn HBM GB/s at M=1..8, % roofline, 1 GB300"

# step shape
M_TOK = 8
HIDDEN = 4096
HQ, HKV, HEAD_DIM = 32, 8, 128
LK = 65540
EPS = 1e-5
PAGE = 64

SAMPLE_EVERY = 16  # steps between the ones whose calls are individually timed
REPEAT_MIN_S = 1.5  # wall time of repeated K-step measurements (clock samples need it)
REPEAT_MAX = 100000

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def step_bytes() -> dict:
    """Algorithmic bytes of each call of one step."""
    tok = M_TOK * HIDDEN * 2
    kv_tok = M_TOK * HKV * HEAD_DIM * 2
    return {
        "rmsnorm": 2 * tok + HIDDEN * 2,
        "matmul_nk": HIDDEN * HIDDEN * 2 + 2 * tok,
        "kv_append": 2 * 2 * kv_tok,
        "verify_block": LK * HKV * HEAD_DIM * 2 * 2 + 2 * tok + M_TOK * HQ * 4,
        "matmul_kn": HIDDEN * HIDDEN * 2 + 2 * tok,
    }


def step_flops() -> dict:
    return {
        "matmul_nk": 2 * M_TOK * HIDDEN * HIDDEN,
        "matmul_kn": 2 * M_TOK * HIDDEN * HIDDEN,
        # q.k and p.v for every (query, head, visible key)
        "verify_block": sum(4 * HQ * HEAD_DIM * (LK - M_TOK + j + 1) for j in range(M_TOK)),
    }


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_digest(*names) -> str:
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "invariant_bi_matmul_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """dram bytes per launch of the verify kernels, from the committed ncu summary, or
    None once the attention sources differ from the ones profiled."""
    path = os.path.join(ROOT, "profiles", "attn_verify_q8_L65540.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_call:\s*([0-9.eE+]+)", text)
    s = re.search(r"source_digest:\s*([0-9a-f]+)", text)
    if not m or not s:
        return None
    if s.group(1) != source_digest("attention.cu", "attn_common.cuh", "common.cuh"):
        return None
    return float(m.group(1))


# ---------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (200 ms) taken while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ multi-rank glue

def max_over_ranks(value: float, device) -> float:
    """Largest `value` over all ranks (the slowest replica sets the job's time)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_step: float, world: int, seconds_per_step: float) -> float:
    """Whole-job GB/s: every replica streams bytes_per_step per step (weak scaling)."""
    return bytes_per_step * world / seconds_per_step / 1e9


# ------------------------------------------------------------------------ GPU arm

class Step:
    """Device-resident buffers of one verify step and its five C-ABI calls."""

    def __init__(self, dev, seed: int = 5):
        import torch
        import invariant_bi_matmul_gb300 as bi
        from invariant_bi_matmul_gb300 import inputs
        self.torch, self.bi, self.dev = torch, bi, dev
        L = bi.lib()
        self.L = L
        g = inputs.gemm_inputs(M_TOK, HIDDEN, HIDDEN, seed=seed)
        self.x = g.x.to(dev)
        self.gamma = inputs.normal_bf16((HIDDEN,), 1.0, 0.1, seed=seed + 1).to(dev)
        self.w_q = g.w_nk.to(dev)                                       # [N, K]
        self.w_o = inputs.gemm_inputs(1, HIDDEN, HIDDEN, seed=seed + 2).w_kn.to(dev)  # [K, N]
        p = inputs.paged_inputs([LK], [M_TOK], Hq=HQ, Hkv=HKV, D=HEAD_DIM, seed=seed + 3,
                                device=dev)
        self.k_cache, self.v_cache = p.k_cache, p.v_cache
        self.block_table = p.block_table.to(dev)
        self.seq_lens = p.seq_lens.to(dev)
        self.cu_q = p.cu_q.to(dev)
        self.k_new, self.v_new = p.k_new.to(dev), p.v_new.to(dev)
        self.h = torch.empty(M_TOK, HIDDEN, dtype=torch.bfloat16, device=dev)
        self.q = torch.empty(M_TOK, HQ, HEAD_DIM, dtype=torch.bfloat16, device=dev)
        self.o = torch.empty(M_TOK, HQ, HEAD_DIM, dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty(M_TOK, HQ, dtype=torch.float32, device=dev)
        self.y = torch.empty(M_TOK, HIDDEN, dtype=torch.bfloat16, device=dev)
        ws_bytes = bi.attn_workspace_size(M_TOK, HQ, HEAD_DIM, LK)
        self.ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        self.num_pages = self.k_cache.shape[0]
        self.stream = torch.cuda.current_stream(dev).cuda_stream
        self.scale = 1.0 / math.sqrt(HEAD_DIM)

    def calls(self):
        """The five calls as (name, thunk) through the raw C ABI."""
        L, s = self.L, self.stream
        import ctypes
        f = ctypes.c_float
        x, h, q, o, y = (t.data_ptr() for t in (self.x, self.h, self.q, self.o, self.y))
        return [
            ("rmsnorm", lambda: L.bi_rmsnorm(x, HIDDEN, self.gamma.data_ptr(), h, HIDDEN, 0,
                                             M_TOK, HIDDEN, f(EPS), s)),
            ("matmul_nk", lambda: L.bi_matmul(h, HIDDEN, self.w_q.data_ptr(), HIDDEN, 0, q,
                                              HIDDEN, 0, M_TOK, HIDDEN, HIDDEN, s)),
            ("kv_append", lambda: L.bi_kv_append(
                self.k_new.data_ptr(), self.v_new.data_ptr(), self.k_cache.data_ptr(),
                self.v_cache.data_ptr(), self.num_pages, self.block_table.data_ptr(),
                self.block_table.shape[1], self.seq_lens.data_ptr(), self.cu_q.data_ptr(), 1,
                M_TOK, HKV, HEAD_DIM, PAGE, s)),
            ("verify_block", lambda: L.bi_verify_block(
                q, self.k_cache.data_ptr(), self.v_cache.data_ptr(), self.num_pages,
                self.block_table.data_ptr(), self.block_table.shape[1], self.seq_lens.data_ptr(),
                self.cu_q.data_ptr(), 1, M_TOK, M_TOK, LK, HQ, HKV, HEAD_DIM, PAGE, f(self.scale),
                o, self.lse.data_ptr(), self.ws.data_ptr(), self.ws.numel(), s)),
            ("matmul_kn", lambda: L.bi_matmul(o, HIDDEN, self.w_o.data_ptr(), HIDDEN, 1, y,
                                              HIDDEN, 0, M_TOK, HIDDEN, HIDDEN, s)),
        ]

    # rmsnorm, gemm, kv_append, attention (counter reset, partial, merge), gemm
    LAUNCHES_PER_STEP = 7


def run_gpu(args, rank, world, local_rank):
    import torch
    import invariant_bi_matmul_gb300 as bi

    dev = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(dev)
    bi.set_batch_invariant_limit(M_TOK)
    # the weights are fixed for the whole run and no kernel writes them: matmuls may start
    # streaming them while the previous kernel finishes
    bi.set_weight_prefetch(True)
    st = Step(dev)
    calls = st.calls()
    names = [n for n, _ in calls]

    def one_step(events=None):
        for i, (_, fn) in enumerate(calls):
            if events is not None:
                events[i].record()
            rc = fn()
            if rc != 0:
                raise RuntimeError(f"{names[i]} returned {bi.lib().bi_status_string(rc).decode()}: "
                                   f"{bi.lib().bi_last_error_message().decode()}")
        if events is not None:
            events[len(calls)].record()

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    if bi.device_status() != bi.BI_OK:
        raise RuntimeError("device error word set during warm-up")

    # The timed measurement is K steps bracketed by a barrier and a synchronize, timed
    # with CUDA events on the launching stream.  It is repeated (REPEAT_MIN_S of repeats,
    # at least three) so that the clock sampler sees the GPU under this load; the value
    # is the median repeat.  Per-call CUDA events are recorded on every SAMPLE_EVERY-th
    # step of every repeat: an event recorded between two kernels breaks the programmatic
    # dependent-launch overlap between them, so recording one around every call of every
    # step would slow the step it measures.  Those sampled steps give the per-call
    # durations (parts, roofline).
    # Sampled steps sit in the second half of each repeat: a repeat starts after a
    # synchronize, so its first steps run as fast as the host issues them, and the extra
    # event records of a sampled step would then time the host's issue gaps; by half-way
    # the host is far enough ahead that the events time the kernels.
    half = args.steps // 2
    sampled = [k for k in range(half, args.steps) if (k - half) % SAMPLE_EVERY == 0]
    is_sampled = set(sampled)
    dist = world > 1

    def timed_block(rec):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)]
              for _ in sampled] if rec else None
        if dist:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record()
        for k in range(args.steps):
            one_step(ev[(k - half) // SAMPLE_EVERY] if rec and k in is_sampled else None)
        end.record()
        torch.cuda.synchronize()
        if dist:
            torch.distributed.barrier()
        return start.elapsed_time(end), ev

    reps_ms, events = [], []

    def rep():
        ms_rep, ev = timed_block(True)
        reps_ms.append(max_over_ranks(ms_rep, dev))
        events.extend(ev)

    with ClockSampler(local_rank) as clocks:
        t_wall = time.perf_counter()
        for _ in range(3):
            rep()
        per = (time.perf_counter() - t_wall) / 3
        # every rank runs the same number of repeats (the largest any rank asks for)
        more = max_over_ranks(float(max(0, math.ceil((REPEAT_MIN_S - 3 * per) / per))), dev)
        for _ in range(min(int(more), REPEAT_MAX)):
            rep()
    per_call_ms = {n: 0.0 for n in names}
    for evs in events:
        for i, n in enumerate(names):
            per_call_ms[n] += evs[i].elapsed_time(evs[i + 1])
    per_call_ms = {n: v / len(events) for n, v in per_call_ms.items()}
    status = bi.device_status()
    if status != bi.BI_OK:
        raise RuntimeError(f"device error word after the timed region: {status}")
    elapsed_ms = statistics.median(reps_ms)

    e2e = run_e2e(st, args, dist)
    extra = gemm_vs_cublas(st) if rank == 0 else {}
    kern = kernel_table(dev, st) if rank == 0 else {}
    return {"elapsed_ms": elapsed_ms, "reps_ms": reps_ms, "sampled_steps": len(events),
            "per_call_ms": per_call_ms, "clocks": clocks.summary(), "e2e": e2e,
            "cublas": extra, "kernels": kern}


def run_e2e(st: Step, args, dist):
    """Same step through the public Python API with host buffers: one pinned H2D copy of
    the step's inputs (hidden states, new K/V), the five calls, D2H of the result, every
    step; timed on the host clock around the synchronised loop.  Two ways of issuing it:
    `graph` captures the copies and the five calls once in a CUDA graph and replays it
    every step (how a serving loop issues a fixed-shape decode step); `eager` issues every
    copy and call from Python each step."""
    import torch
    import invariant_bi_matmul_gb300 as bi
    dev = st.dev
    # the step's inputs packed in one pinned buffer (hidden states, then new K, then new
    # V), so one host-to-device copy per step brings them all, as a serving loop packs them
    parts = [st.x, st.k_new, st.v_new]
    sizes = [t.numel() * t.element_size() for t in parts]
    hin = torch.empty(sum(sizes), dtype=torch.uint8).pin_memory()
    din = torch.empty(sum(sizes), dtype=torch.uint8, device=dev)
    views_h, views_d, off = [], [], 0
    for t, nb in zip(parts, sizes):
        views_h.append(hin[off:off + nb].view(t.dtype).view(t.shape))
        views_d.append(din[off:off + nb].view(t.dtype).view(t.shape))
        views_h[-1].copy_(t.cpu())
        off += nb
    hx, hk, hv = views_h
    x, kn, vn = views_d
    hy = torch.empty(M_TOK, HIDDEN, dtype=torch.bfloat16).pin_memory()

    def body():
        din.copy_(hin, non_blocking=True)
        bi.rmsnorm(x, st.gamma, EPS, out=st.h)
        bi.matmul(st.h, st.w_q, "nk", out=st.q.view(M_TOK, HIDDEN))
        bi.kv_append(kn, vn, st.k_cache, st.v_cache, st.block_table, st.seq_lens, st.cu_q)
        bi.verify_block(st.q, st.k_cache, st.v_cache, st.block_table, st.seq_lens, st.cu_q,
                        max_q=M_TOK, max_seq_len=LK, scale=st.scale, out=st.o, lse=st.lse,
                        workspace=st.ws)
        bi.matmul(st.o.view(M_TOK, HIDDEN), st.w_o, "kn", out=st.y)
        hy.copy_(st.y, non_blocking=True)

    def eager_step():
        body()
        torch.cuda.current_stream(dev).synchronize()

    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        for _ in range(3):
            body()
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        body()

    def graph_step():
        graph.replay()
        torch.cuda.current_stream(dev).synchronize()

    n = max(10, min(args.steps, 2000))
    out = {}
    for name, step in (("graph", graph_step), ("eager", eager_step)):
        for _ in range(3):
            step()
        if dist:
            torch.distributed.barrier()
        t0 = time.perf_counter()
        for _ in range(n):
            step()
        out[name] = max_over_ranks((time.perf_counter() - t0) / n, dev)
    # the graph's result equals the eager step's (same inputs, same kernels)
    y_eager = hy.clone()
    graph_step()
    if not torch.equal(hy.view(torch.int16), y_eager.view(torch.int16)):
        raise SystemExit("graph replay and eager step disagree")
    del graph
    h2d = hin.numel()
    d2h = hy.numel() * 2
    return {"sec_per_step": out["graph"], "sec_per_step_eager": out["eager"], "h2d": h2d,
            "d2h": d2h, "steps": n}


def gemm_vs_cublas(st: Step):
    """Invariance cost at the step's shape: bi_matmul vs torch.matmul (cuBLAS, free to
    pick split-K) at M = 8, K = N = 4096, L2 evicted before every rep, A/B alternated."""
    import torch
    import invariant_bi_matmul_gb300 as bi
    flush = torch.ones(128 * 1024 * 1024, dtype=torch.float32, device=st.dev)
    out = torch.empty(M_TOK, HIDDEN, dtype=torch.bfloat16, device=st.dev)
    a_t, b_t = [], []
    for rep in range(31):
        for which in (0, 1) if rep % 2 == 0 else (1, 0):
            flush.sum()  # read-based L2 eviction (leaves no dirty lines)
            s = torch.cuda.Event(enable_timing=True)
            e = torch.cuda.Event(enable_timing=True)
            s.record()
            if which == 0:
                bi.matmul(st.h, st.w_q, "nk", out=out)
            else:
                torch.matmul(st.h, st.w_q.t(), out=out)
            e.record()
            torch.cuda.synchronize()
            (a_t if which == 0 else b_t).append(s.elapsed_time(e) * 1e3)
    a, b = statistics.median(a_t[1:]), statistics.median(b_t[1:])
    return {"bi_matmul_us": round(a, 2), "cublas_us": round(b, 2), "ratio": round(a / b, 3)}


def graph_time_us(fns, n=64, reps=7):
    """Per-call device time of n calls (cycling through fns) captured in one CUDA graph
    and replayed, timed with CUDA events around each replay (median of reps): no host
    launch cost between the calls, so kernels shorter than the Python binding's per-call
    cost are timed as the GPU runs them back to back."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for f in fns:  # first calls (function attributes, occupancy queries) uncaptured
            f()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(n):
            fns[i % len(fns)]()
    g.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record()
        g.replay()
        e.record()
        torch.cuda.synchronize()
        ts.append(s.elapsed_time(e) * 1e3 / n)
    del g
    return statistics.median(ts)


def kernel_table(dev, st=None):
    """The metric's per-kernel half, measured in the same run: the invariant GEMM at
    K = N = 4096 for M = 1, 2, 4, 8 (both W layouts; HBM-bound: GB/s and the fraction of
    the measured HBM copy rate) with cuBLAS (torch.matmul, free to split K) at the same
    shapes and layouts, M = 256 and 2048 (TFLOP/s against the measured bf16 burst peak),
    and RMSNorm [2048, 8192].  Each figure is the per-call device time of 64 back-to-back
    calls in one CUDA graph over rotating weight (or input) sets of 256 MB, more than twice
    the L2, so every call reads its operands from HBM; median of 7 replays.  With the
    step's buffers `st`: the step's verify call timed the same way (32 calls; its K/V,
    268 MB, already exceed twice the L2), the same call with 1, 2 and 4 queries, and the
    floor of any call timed with a pair of CUDA events: an empty-sized kernel between two
    events, with the host ahead."""
    import torch
    import invariant_bi_matmul_gb300 as bi
    from invariant_bi_matmul_gb300 import inputs
    peaks, kind = load_peaks()
    hbm, tf = float(peaks["hbm_gbs"]), float(peaks.get("bf16_tflops", 1900.0))
    N = K = 4096
    sets = 256 * 1024 * 1024 // (2 * N * K)
    gi = inputs.gemm_inputs(2048, N, K, seed=2)
    x = gi.x.to(dev)
    wnk = [gi.w_nk.to(dev)]
    wnk += [wnk[0].clone() for _ in range(sets - 1)]
    wkn = [gi.w_kn.to(dev)]
    wkn += [wkn[0].clone() for _ in range(sets - 1)]
    out = {"_how": (f"per-call device time, 64 calls in one CUDA graph over {sets} rotating "
                    "copies of W (256 MB, > 2x L2), median of 7 replays; peaks "
                    f"{kind}: HBM {hbm} GB/s, bf16 {tf} TFLOP/s (burst)")}
    old = bi.get_batch_invariant_limit()
    bi.set_batch_invariant_limit(1 << 40)
    try:
        for M in (1, 2, 4, 8, 256, 2048):
            xm = x[:M].contiguous()
            y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
            fl = 2.0 * M * N * K
            by = 2.0 * N * K + 2.0 * M * K + 2.0 * M * N
            row = {}
            for lay, ws, cub in (("nk", wnk, lambda w: torch.matmul(xm, w.t(), out=y)),
                                 ("kn", wkn, lambda w: torch.matmul(xm, w, out=y))):
                if M > 8 and lay == "kn":
                    continue
                t = graph_time_us([lambda w=w: bi.matmul(xm, w, lay, out=y) for w in ws])
                tc = graph_time_us([lambda w=w: cub(w) for w in ws])
                row[lay] = {"us": round(t, 2), "TFLOP/s": round(fl / t / 1e6, 1),
                            "GB/s": round(by / t / 1e3, 1),
                            "frac_hbm": round(by / t / 1e3 / hbm, 4),
                            "frac_tensor": round(fl / t / 1e6 / tf, 4),
                            "cublas_us": round(tc, 2), "vs_cublas": round(t / tc, 3)}
            row["bound"] = "hbm" if M <= 64 else "tensor"
            out[f"gemm_M{M}"] = row
        xr, g = inputs.rmsnorm_inputs(2048, 8192, seed=3)
        xr, g = xr.to(dev), g.to(dev)
        by = 4.0 * 2048 * 8192 + 2 * 8192
        rs = [(xr.clone(), torch.empty_like(xr)) for _ in range(8)]
        t = graph_time_us([lambda a=a, o=o: bi.rmsnorm(a, g, 1e-5, out=o) for a, o in rs])
        out["rmsnorm_B2048_H8192"] = {"us": round(t, 2), "GB/s": round(by / t / 1e3, 1),
                                      "frac_hbm": round(by / t / 1e3 / hbm, 4), "bound": "hbm"}
        if st is not None:
            t = graph_time_us([lambda: bi.verify_block(
                st.q, st.k_cache, st.v_cache, st.block_table, st.seq_lens, st.cu_q,
                max_q=M_TOK, max_seq_len=LK, scale=st.scale, out=st.o, lse=st.lse,
                workspace=st.ws)], n=32)
            by = step_bytes()["verify_block"]
            out["verify_block"] = {"us": round(t, 2), "GB/s": round(by / t / 1e3, 1),
                                   "frac_hbm": round(by / t / 1e3 / hbm, 4), "bound": "hbm"}
            # the same cache and sequence with blocks of 1, 2 and 4 queries (the last
            # tokens of the sequence), so the line covers decode and every verify width
            for qn in (1, 2, 4):
                cu = torch.tensor([0, qn], dtype=torch.int32, device=dev)
                t = graph_time_us([lambda qn=qn, cu=cu: bi.verify_block(
                    st.q[:qn], st.k_cache, st.v_cache, st.block_table, st.seq_lens, cu,
                    max_q=qn, max_seq_len=LK, scale=st.scale, out=st.o[:qn],
                    lse=st.lse[:qn], workspace=st.ws)], n=32)
                by = LK * HKV * HEAD_DIM * 2 * 2 + qn * HQ * (HEAD_DIM * 2 * 2 + 4)
                out[f"verify_q{qn}"] = {"us": round(t, 2), "GB/s": round(by / t / 1e3, 1),
                                        "frac_hbm": round(by / t / 1e3 / hbm, 4),
                                        "bound": "hbm"}
            tiny = torch.zeros(1, device=dev)
            ts = []
            for _ in range(21):
                torch.cuda._sleep(200000)  # the GPU busy while the host records ahead
                s0 = torch.cuda.Event(enable_timing=True)
                s1 = torch.cuda.Event(enable_timing=True)
                s0.record()
                tiny.add_(1.0)
                s1.record()
                torch.cuda.synchronize()
                ts.append(s0.elapsed_time(s1) * 1e3)
            out["event_pair_floor_us"] = round(statistics.median(ts), 2)
    finally:
        bi.set_batch_invariant_limit(old)
    del wnk, wkn
    torch.cuda.empty_cache()
    return out


# --------------------------------------------------------------------- oracle arm

def cpu_info():
    """(cores this process may run on, CPU model name)."""
    import platform
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    return int(cores or 1), model or platform.processor() or platform.machine()


class OracleStep:
    """The bench step on the CPU oracle, chained as on the GPU: RMSNorm -> NK matmul (q)
    -> KV append -> verify attention on that q -> KN matmul of its output.  Inputs are the
    same seeded recipe as the GPU step (drawn on the CPU).  `run(pool)` computes every
    output of the step; `pool` (a thread pool, or None for one thread) runs independent
    output columns and attention rows concurrently: the oracle's C code releases the GIL,
    and nothing in a column or row depends on another."""

    def __init__(self, threads: int):
        import numpy as np
        from invariant_bi_matmul_gb300 import inputs
        g = inputs.gemm_inputs(M_TOK, HIDDEN, HIDDEN, seed=5)
        p = inputs.paged_inputs([LK], [M_TOK], Hq=HQ, Hkv=HKV, D=HEAD_DIM, seed=8)
        b = inputs.bf16_bits
        self.x = b(g.x)
        self.gamma = b(inputs.normal_bf16((HIDDEN,), 1.0, 0.1, seed=6))
        w_q, w_o = b(g.w_nk), b(inputs.gemm_inputs(1, HIDDEN, HIDDEN, seed=7).w_kn)
        self.kn, self.vn, self.kc, self.vc = b(p.k_new), b(p.v_new), b(p.k_cache), b(p.v_cache)
        self.bt, self.sl, self.cu = p.block_table.numpy(), p.seq_lens.numpy(), p.cu_q.numpy()
        # output-column blocks of both weights, cut once (layout preserved)
        nb = max(1, min(threads * 2, 64))
        edges = [HIDDEN * i // nb for i in range(nb + 1)]
        self.cols = list(zip(edges[:-1], edges[1:]))
        self.wq_blocks = [np.ascontiguousarray(w_q[c0:c1]) for c0, c1 in self.cols]
        self.wo_blocks = [np.ascontiguousarray(w_o[:, c0:c1]) for c0, c1 in self.cols]

    def _matmul(self, xb, blocks, layout, pool):
        import numpy as np
        import oracle
        run = (lambda w: oracle.matmul(xb, w, layout))
        parts = list(pool.map(run, blocks)) if pool else [run(w) for w in blocks]
        return np.concatenate(parts, axis=1)

    def run(self, pool=None):
        import numpy as np
        import oracle
        h = oracle.bf16_round(oracle.rmsnorm(self.x, self.gamma, EPS))
        q = oracle.bf16_round(self._matmul(h, self.wq_blocks, oracle.W_NK, pool))
        q = q.reshape(M_TOK, HQ, HEAD_DIM)
        kc, vc = oracle.kv_append(self.kn, self.vn, self.kc, self.vc, self.bt, self.sl, self.cu,
                                  PAGE)
        rows = [(j, hh) for j in range(M_TOK) for hh in range(HQ)]
        one = (lambda r: oracle.attention_row(q, kc, vc, self.bt, self.sl, self.cu, 0, r[0],
                                              r[1], HQ, 1.0 / math.sqrt(HEAD_DIM))[0])
        o = list(pool.map(one, rows)) if pool else [one(r) for r in rows]
        ob = oracle.bf16_round(np.stack(o).astype(np.float32)).reshape(M_TOK, HIDDEN)
        return self._matmul(ob, self.wo_blocks, oracle.W_KN, pool)

    def sample_single_thread(self, frac: int = 8):
        """A bounded single-thread sample (about 1/frac of the step's arithmetic): all
        RMSNorm rows and KV-append tokens, 1/frac of each matmul's output columns, 1/frac of
        the attention rows; returns (seconds scaled to the full step, description)."""
        import numpy as np
        import oracle
        t0 = time.perf_counter()
        h = oracle.bf16_round(oracle.rmsnorm(self.x, self.gamma, EPS))
        kc, vc = oracle.kv_append(self.kn, self.vn, self.kc, self.vc, self.bt, self.sl, self.cu,
                                  PAGE)
        fixed = time.perf_counter() - t0
        nb = max(1, len(self.cols) // frac)
        t0 = time.perf_counter()
        for w in self.wq_blocks[:nb]:
            oracle.matmul(h, w, oracle.W_NK)
        for w in self.wo_blocks[:nb]:
            oracle.matmul(h, w, oracle.W_KN)
        mm = (time.perf_counter() - t0) * len(self.cols) / nb
        q = np.zeros((M_TOK, HQ, HEAD_DIM), np.uint16)
        rows = [(j, hh) for j in range(M_TOK) for hh in range(HQ)][::frac]
        t0 = time.perf_counter()
        for j, hh in rows:
            oracle.attention_row(q, kc, vc, self.bt, self.sl, self.cu, 0, j, hh, HQ,
                                 1.0 / math.sqrt(HEAD_DIM))
        at = (time.perf_counter() - t0) * (M_TOK * HQ) / len(rows)
        desc = (f"one thread: all {M_TOK} RMSNorm rows and KV-append tokens, {nb} of "
                f"{len(self.cols)} column blocks of each matmul, 1/{frac} of the "
                f"{M_TOK * HQ} attention rows; times scaled to the full step")
        return fixed + mm + at, desc


def oracle_baseline(steps: int, warmup: int):
    """The oracle on every host core for `steps` full steps (after `warmup`), plus a
    bounded single-thread sample: a cpu_baseline object and the per-step seconds."""
    from concurrent.futures import ThreadPoolExecutor
    cores, model = cpu_info()
    st = OracleStep(cores)
    one_s, one_desc = st.sample_single_thread()
    total = sum(step_bytes().values())
    with ThreadPoolExecutor(max_workers=cores) as pool:
        for _ in range(warmup):
            st.run(pool)
        secs = []
        for _ in range(steps):
            t0 = time.perf_counter()
            st.run(pool)
            secs.append(time.perf_counter() - t0)
    sec = statistics.median(secs)
    base = {"value": round(total / sec / 1e9, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle", "cpu_model": model,
            "sample": (f"{steps} full steps (every output of the step, chained as on the GPU) on "
                       f"{cores} threads over independent output columns and attention rows; "
                       f"median step {sec:.3f} s"),
            "single_thread": {"value": round(total / one_s / 1e9, 4), "cores": 1,
                              "sample": one_desc}}
    return base, secs


def run_reference(args, rank, world):
    if rank != 0:
        return
    base, secs = oracle_baseline(args.steps, args.warmup)
    sec = statistics.median(secs)
    value = sum(step_bytes().values()) / sec / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sec * 1e3, 2), "ms_per_step_total": round(sum(secs) * 1e3, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": workload_config(),
        "cpu_baseline": base,
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config():
    return {
        "workload": ("verify step, M=8 tokens: rmsnorm [8,4096] -> matmul NK K=N=4096 -> "
                     "kv_append -> verify attention (1 seq, q=8, Lk=65540, 32 q / 8 kv heads, "
                     "head_dim 128, 64-token pages) -> matmul KN K=N=4096"),
        "M": M_TOK, "K": HIDDEN, "N": HIDDEN, "seq_len": LK, "verify_width": M_TOK,
        "q_heads": HQ, "kv_heads": HKV, "head_dim": HEAD_DIM, "batch_invariant_limit": M_TOK,
        "l2": "inputs larger than L2: ~336 MB streamed per step vs 126 MB L2, no flush",
    }


# ---------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-sample", action="store_true", default=True)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--case", default=None,
                    help="time one call shape instead of the step (for profiling): "
                         "gemm:M:N:K[:kn][:fast], qgemm:M:N:K:format[:kn], "
                         "attn:B:q:Lk[:fast] or prefill:Lk:new")
    ap.add_argument("--case-reps", type=int, default=5)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.case:
        run_case(args.case, args.case_reps)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if args.steps == 2000:
            args.steps = 10
        if args.warmup == 50:
            args.warmup = 3
        run_reference(args, rank, world)
        return

    # The oracle baseline runs before any CUDA work (no fork after CUDA init).
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu, _ = oracle_baseline(steps=3, warmup=1)

    import torch
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device(f"cuda:{local_rank}"))
    res = run_gpu(args, rank, world, local_rank)
    if args.sweep and rank == 0:
        run_sweep()
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank != 0:
        return

    peaks, peak_kind = load_peaks()
    nbytes = step_bytes()
    flops = step_flops()
    total = sum(nbytes.values())
    ms = res["elapsed_ms"] / args.steps
    value = job_throughput(total, world, ms * 1e-3)
    calls_ms = res["per_call_ms"]
    share = {n: round(v / sum(calls_ms.values()), 4) for n, v in calls_ms.items()}
    parts = {"_note": f"per-call CUDA events on every {SAMPLE_EVERY}th step of the second "
                      f"half of each repeat ({res['sampled_steps']} steps over all repeats); "
                      "those steps run without launch overlap between calls, so the parts add "
                      "up to more than ms_per_step"}
    for n, v in calls_ms.items():
        parts[n] = {"us": round(v * 1e3, 2), "GB/s": round(nbytes[n] / (v * 1e-3) / 1e9, 1),
                    "share": share[n]}
        if n in flops:
            parts[n]["TFLOP/s"] = round(flops[n] / (v * 1e-3) / 1e12, 2)
    dom = max(calls_ms, key=calls_ms.get)
    achieved = nbytes[dom] / (calls_ms[dom] * 1e-3) / 1e9
    hbm = float(peaks["hbm_gbs"])
    roof = {"kernel": f"{dom} (split-KV partial + LSE merge)" if dom == "verify_block" else dom,
            "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
            "frac": round(achieved / hbm, 4), "peak_source": f"{peak_kind} hbm_gbs",
            "traffic": recorded_traffic() if dom == "verify_block" else None,
            "algorithmic_bytes": nbytes[dom]}
    kv = res["kernels"].get("verify_block") if dom == "verify_block" else None
    if kv:
        # the same call back to back in a CUDA graph, and the floor that a pair of events
        # adds to any single call: context for the event-timed figure above
        roof["graph_timed"] = {"us": kv["us"], "achieved": kv["GB/s"], "frac": kv["frac_hbm"],
                               "event_pair_floor_us": res["kernels"].get("event_pair_floor_us")}
    e2e = res["e2e"]
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations/KV, N(0,0.02) weights)",
        "config": workload_config(),
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": round(job_throughput(total, world, e2e["sec_per_step"]), 1), "unit": "GB/s",
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "ms_per_step": round(e2e["sec_per_step"] * 1e3, 4),
                "issue": "the step's copies and calls captured once in a CUDA graph, "
                         "replayed and synchronised every step",
                "eager": {"value": round(job_throughput(total, world,
                                                        e2e["sec_per_step_eager"]), 1),
                          "ms_per_step": round(e2e["sec_per_step_eager"] * 1e3, 4),
                          "issue": "every copy and call issued from Python each step"}},
        "gpu_launches": Step.LAUNCHES_PER_STEP * args.steps,
        "gpu_launches_note": "per timed measurement of K steps (every repeat launches as many)",
        "clocks": res["clocks"],
        "timing": {"repeats": len(res["reps_ms"]),
                   "ms_per_step_min": round(min(res["reps_ms"]) / args.steps, 5),
                   "ms_per_step_max": round(max(res["reps_ms"]) / args.steps, 5),
                   "how": f"each repeat times exactly {args.steps} steps (barrier and "
                          "synchronize on both sides, CUDA events on the launching stream); "
                          "value and ms_per_step are the median repeat"},
        "parts": parts,
        "gemm_vs_cublas_m8": res["cublas"],
        "kernels": res["kernels"],
    }
    print(json.dumps(line), flush=True)


def run_case(spec: str, reps: int):
    """One call shape, `reps` times after three warm-up calls, each timed with CUDA events
    (L2 evicted before each): the unit a profiler capture selects with -s 3 -c 1.
    `fast` sets the batch-invariant limit to 0 (the non-invariant configuration), else
    the limit covers the call."""
    import torch
    import invariant_bi_matmul_gb300 as bi
    from invariant_bi_matmul_gb300 import inputs
    parts = spec.split(":")
    fast = "fast" in parts[1:]
    bi.set_batch_invariant_limit(0 if fast else 1 << 40)
    bi.set_weight_prefetch(True)  # fixed weights
    dev = torch.device("cuda:0")
    flush = torch.ones(128 * 1024 * 1024, dtype=torch.float32, device=dev)
    if parts[0] == "gemm":
        M, N, K = (int(v) for v in parts[1:4])
        lay = "kn" if "kn" in parts[4:] else "nk"
        gi = inputs.gemm_inputs(M, N, K, seed=2)
        x = gi.x.to(dev)
        w = (gi.w_kn if lay == "kn" else gi.w_nk).to(dev)
        y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        fn = lambda: bi.matmul(x, w, lay, out=y)  # noqa: E731
        desc = {"case": "gemm", "M": M, "N": N, "K": K, "layout": lay,
                "splits": bi.matmul_splits(M, N, K, lay,
                                           torch.cuda.get_device_properties(dev).multi_processor_count)}
    elif parts[0] == "qgemm":
        M, N, K = (int(v) for v in parts[1:4])
        fmt = parts[4]
        lay = "kn" if "kn" in parts[5:] else "nk"
        gs = {"mxfp4": 32, "nvfp4": 16, "mxfp8": 32, "affine4": 64, "affine8": 32}[fmt]
        wq, sc, bq = (inputs.quant_weights(inputs.Q_NAMES[fmt], N, K, gs, seed=5) if lay == "nk"
                      else inputs.quant_weights(inputs.Q_NAMES[fmt], K, N, gs, seed=5))
        wq, sc = wq.to(dev), sc.to(dev)
        bq = bq.to(dev) if bq is not None else None
        x = inputs.normal_bf16((M, K), seed=2).to(dev)
        y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        fn = lambda: bi.qmatmul(x, wq, sc, fmt, gs, K, biases=bq, out=y, layout=lay, N=N)  # noqa: E731
        desc = {"case": "qgemm", "M": M, "N": N, "K": K, "format": fmt, "layout": lay}
    elif parts[0] == "attn":
        B, q, L = (int(v) for v in parts[1:4])
        p = inputs.paged_inputs([L] * B, [q] * B, Hq=HQ, Hkv=HKV, D=HEAD_DIM, seed=4, device=dev)
        d = {k: getattr(p, k).to(dev) for k in ("q", "k_cache", "v_cache", "block_table",
                                                 "seq_lens", "cu_q")}
        ws = torch.empty(bi.attn_workspace_size(B * q, HQ, HEAD_DIM, L), dtype=torch.uint8,
                         device=dev)
        out = torch.empty(B * q, HQ, HEAD_DIM, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(B * q, HQ, dtype=torch.float32, device=dev)
        fn = lambda: bi.verify_block(d["q"], d["k_cache"], d["v_cache"], d["block_table"],  # noqa: E731
                                     d["seq_lens"], d["cu_q"], max_q=q, max_seq_len=L,
                                     scale=1 / math.sqrt(HEAD_DIM), out=out, lse=lse,
                                     workspace=ws)
        desc = {"case": "attn", "B": B, "q": q, "Lk": L}
    elif parts[0] == "prefill":
        L, qb = (int(v) for v in parts[1:3])  # prompt length, new tokens (the last qb)
        p = inputs.paged_inputs([L], [qb], Hq=HQ, Hkv=HKV, D=HEAD_DIM, seed=5, device=dev)
        d = {k: getattr(p, k).to(dev) for k in ("q", "k_cache", "v_cache", "block_table",
                                                 "seq_lens", "cu_q")}
        ws = torch.empty(bi.attn_workspace_size(qb, HQ, HEAD_DIM, L), dtype=torch.uint8,
                         device=dev)
        out = torch.empty(qb, HQ, HEAD_DIM, dtype=torch.bfloat16, device=dev)
        fn = lambda: bi.prefill_attn(d["q"], d["k_cache"], d["v_cache"], d["block_table"],  # noqa: E731
                                     d["seq_lens"], d["cu_q"], max_q=qb, max_seq_len=L,
                                     scale=1 / math.sqrt(HEAD_DIM), out=out, want_lse=False,
                                     workspace=ws)
        desc = {"case": "prefill", "Lk": L, "new_tokens": qb}
    else:
        raise SystemExit(f"unknown case {spec!r}")
    for _ in range(3):
        fn()
    ts = []
    for _ in range(reps):
        flush.sum()
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record()
        fn()
        s1.record()
        torch.cuda.synchronize()
        ts.append(round(s0.elapsed_time(s1) * 1e3, 2))
    if bi.device_status() != bi.BI_OK:
        raise SystemExit("device error word set")
    desc.update({"fast": fast, "us": ts})
    print(json.dumps(desc), flush=True)


def run_sweep():
    """Extra JSON lines: GEMM over M (both layouts, vs cuBLAS), RMSNorm at hidden 8192,
    attention over the pages' Lk and q, chunked prefill.  Two timings per shape: one call with L2 evicted
    before it (`*_us`, includes the launch), and `steady_*_us`, the per-call time of a
    back-to-back stream over rotating input sets larger than 2x L2 (for attention, one
    set when its K/V already exceed that; otherwise marked warm).  Each GEMM and attention
    shape is timed inside the batch-invariant limit and again with the limit at 0 (the
    non-invariant configuration the library picks: split-K, the chosen chunk length), and
    `invariance_tax` is the invariant time over the fast one, minus 1."""
    import torch
    import invariant_bi_matmul_gb300 as bi
    from invariant_bi_matmul_gb300 import inputs
    peaks, peak_kind = load_peaks()
    dev = torch.device("cuda:0")
    bi.set_weight_prefetch(True)  # every timed weight is fixed
    # evict L2 by READING a buffer 4x its size (a write-based flush would leave dirty lines
    # whose write-back then competes with the timed kernel's reads)
    flush = torch.ones(128 * 1024 * 1024, dtype=torch.float32, device=dev)

    def t_us(fn, reps=21):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(reps):
            flush.sum()
            s = torch.cuda.Event(enable_timing=True)
            e = torch.cuda.Event(enable_timing=True)
            s.record()
            fn()
            e.record()
            torch.cuda.synchronize()
            ts.append(s.elapsed_time(e) * 1e3)
        return statistics.median(ts)

    def steady_us(fns, n=60):
        for f in fns:
            f()
        torch.cuda.synchronize()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record()
        for i in range(n):
            fns[i % len(fns)]()
        e.record()
        torch.cuda.synchronize()
        return s.elapsed_time(e) * 1e3 / n

    graph_us = graph_time_us

    SET_BYTES = 256 * 1024 * 1024  # rotating inputs: more than 2x the 126 MB L2
    INVARIANT, FAST = 1 << 40, 0   # limits: every call inside it / the limit disabled
    sms = torch.cuda.get_device_properties(dev).multi_processor_count

    K = N = 4096
    gi = inputs.gemm_inputs(2048, N, K, seed=2)
    x, wnk, wkn = gi.x.to(dev), gi.w_nk.to(dev), gi.w_kn.to(dev)
    wsets = [wnk] + [wnk.clone() for _ in range(SET_BYTES // (2 * N * K) - 1)]
    for M in (1, 2, 4, 8, 16, 64, 256, 2048):
        xm = x[:M].contiguous()
        y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
        bi.set_batch_invariant_limit(INVARIANT)
        tn = t_us(lambda: bi.matmul(xm, wnk, "nk", out=y))
        tk = t_us(lambda: bi.matmul(xm, wkn, "kn", out=y))
        tc = t_us(lambda: torch.matmul(xm, wnk.t(), out=y))
        tns = steady_us([lambda w=w: bi.matmul(xm, w, "nk", out=y) for w in wsets])
        tcs = steady_us([lambda w=w: torch.matmul(xm, w.t(), out=y) for w in wsets])
        tng = graph_us([lambda w=w: bi.matmul(xm, w, "nk", out=y) for w in wsets])
        tcg = graph_us([lambda w=w: torch.matmul(xm, w.t(), out=y) for w in wsets])
        # the same call outside the limit (split-K where it pays)
        bi.set_batch_invariant_limit(FAST)
        splits = bi.matmul_splits(M, N, K, "nk", sms)
        tf = t_us(lambda: bi.matmul(xm, wnk, "nk", out=y))
        tfs = steady_us([lambda w=w: bi.matmul(xm, w, "nk", out=y) for w in wsets])
        tfg = graph_us([lambda w=w: bi.matmul(xm, w, "nk", out=y) for w in wsets])
        fl = 2 * M * N * K
        by = 2 * N * K + 4 * M * K
        tf_peak = float(peaks.get("bf16_tflops", 1900.0))
        print(json.dumps({"sweep": "gemm", "M": M, "K": K, "N": N, "nk_us": round(tn, 2),
                          "kn_us": round(tk, 2), "cublas_us": round(tc, 2),
                          "nk_vs_cublas": round(tn / tc, 3), "kn_vs_cublas": round(tk / tc, 3),
                          "nk_TFLOP/s": round(fl / tn / 1e6, 1), "nk_GB/s": round(by / tn / 1e3, 1),
                          "nk_frac_hbm": round(by / tn / 1e3 / peaks["hbm_gbs"], 3),
                          "nk_frac_tensor": round(fl / tn / 1e6 / tf_peak, 3),
                          "steady_nk_us": round(tns, 2), "steady_cublas_us": round(tcs, 2),
                          "steady_nk_vs_cublas": round(tns / tcs, 3),
                          "steady_nk_frac_hbm": round(by / tns / 1e3 / peaks["hbm_gbs"], 3),
                          "steady_nk_frac_tensor": round(fl / tns / 1e6 / tf_peak, 3),
                          "fast_splits": splits, "fast_nk_us": round(tf, 2),
                          "steady_fast_nk_us": round(tfs, 2),
                          "invariance_tax": round(tn / tf - 1.0, 3),
                          "steady_invariance_tax": round(tns / tfs - 1.0, 3),
                          "graph_nk_us": round(tng, 2), "graph_fast_nk_us": round(tfg, 2),
                          "graph_cublas_us": round(tcg, 2),
                          "graph_nk_vs_cublas": round(tng / tcg, 3),
                          "graph_fast_vs_cublas": round(tfg / tcg, 3),
                          "graph_invariance_tax": round(tng / tfg - 1.0, 3),
                          "graph_nk_frac_hbm": round(by / tng / 1e3 / peaks["hbm_gbs"], 3),
                          "graph_nk_frac_tensor": round(fl / tng / 1e6 / tf_peak, 3)}),
              flush=True)
    del wsets
    # IEEE binary16 inputs (bi_matmul_ex): the same kernel with f16 operands
    xh, wh = x.to(torch.float16), wnk.to(torch.float16)
    hsets = [wh] + [wh.clone() for _ in range(SET_BYTES // (2 * N * K) - 1)]
    bi.set_batch_invariant_limit(INVARIANT)
    for M in (8, 2048):
        xm = xh[:M].contiguous()
        y = torch.empty(M, N, dtype=torch.float16, device=dev)
        tg = graph_us([lambda w=w: bi.matmul(xm, w, "nk", out=y) for w in hsets])
        tcg = graph_us([lambda w=w: torch.matmul(xm, w.t(), out=y) for w in hsets])
        fl, by = 2 * M * N * K, 2 * N * K + 4 * M * K
        print(json.dumps({"sweep": "gemm_f16", "M": M, "K": K, "N": N, "graph_us": round(tg, 2),
                          "graph_cublas_us": round(tcg, 2),
                          "graph_frac_hbm": round(by / tg / 1e3 / peaks["hbm_gbs"], 3),
                          "graph_frac_tensor": round(fl / tg / 1e6 / float(
                              peaks.get("bf16_tflops", 1900.0)), 3)}), flush=True)
    del hsets, xh, wh
    # quantized W (bi_qmatmul): rotating sets of packed codes larger than L2
    for fmt, gs in (("mxfp4", 32), ("nvfp4", 16), ("mxfp8", 32), ("affine4", 64)):
        q = inputs.Q_NAMES[fmt]
        wq, sc, bq = inputs.quant_weights(q, N, K, gs, seed=5)
        wq, sc = wq.to(dev), sc.to(dev)
        bq = bq.to(dev) if bq is not None else None
        wbytes = wq.numel() + sc.numel() * sc.element_size() + (
            bq.numel() * bq.element_size() if bq is not None else 0)
        qsets = [(wq, sc, bq)] + [(wq.clone(), sc.clone(), None if bq is None else bq.clone())
                                  for _ in range(max(0, min(63, SET_BYTES // wbytes - 1)))]
        for M in (8, 2048):
            xm = x[:M].contiguous()
            y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
            tg = graph_us([lambda a=a, c=c, b=b: bi.qmatmul(xm, a, c, fmt, gs, K, biases=b, out=y)
                           for a, c, b in qsets])
            fl, by = 2 * M * N * K, wbytes + 2 * M * K + 2 * M * N
            print(json.dumps({"sweep": "qmatmul", "format": fmt, "group": gs, "M": M, "K": K,
                              "N": N, "graph_us": round(tg, 2),
                              "graph_frac_hbm": round(by / tg / 1e3 / peaks["hbm_gbs"], 3),
                              "graph_frac_tensor": round(fl / tg / 1e6 / float(
                                  peaks.get("bf16_tflops", 1900.0)), 3)}), flush=True)
        del qsets, wq, sc, bq
    # fp32 inputs (CUDA cores): W 64 MB, one set (larger than L2)
    xf, wf = x.float(), wnk.float()
    for M in (8, 2048):
        xm = xf[:M].contiguous()
        y = torch.empty(M, N, dtype=torch.float32, device=dev)
        tg = graph_us([lambda: bi.matmul(xm, wf, "nk", out=y)], n=8)
        fl, by = 2 * M * N * K, 4 * N * K + 4 * M * K + 4 * M * N
        print(json.dumps({"sweep": "gemm_f32", "M": M, "K": K, "N": N, "graph_us": round(tg, 2),
                          "TFLOP/s": round(fl / tg / 1e6, 2),
                          "graph_frac_hbm": round(by / tg / 1e3 / peaks["hbm_gbs"], 3)}),
              flush=True)
    del xf, wf
    for B in (1, 3, 16, 128, 2048):
        xr, g = inputs.rmsnorm_inputs(B, 8192, seed=3)
        xr, g = xr.to(dev), g.to(dev)
        yr = torch.empty_like(xr)
        t = t_us(lambda: bi.rmsnorm(xr, g, 1e-5, out=yr))
        by = 4 * B * 8192 + 2 * 8192
        nsets = max(2, min(64, -(-SET_BYTES // by)))
        sets = [(xr.clone(), torch.empty_like(xr)) for _ in range(nsets)]
        ts = steady_us([lambda a=a, o=o: bi.rmsnorm(a, g, 1e-5, out=o) for a, o in sets])
        tg = graph_us([lambda a=a, o=o: bi.rmsnorm(a, g, 1e-5, out=o) for a, o in sets])
        del sets
        print(json.dumps({"sweep": "rmsnorm", "B": B, "H": 8192, "us": round(t, 2),
                          "GB/s": round(by / t / 1e3, 1),
                          "frac_hbm": round(by / t / 1e3 / peaks["hbm_gbs"], 3),
                          "steady_us": round(ts, 2), "steady_GB/s": round(by / ts / 1e3, 1),
                          "steady_frac_hbm": round(by / ts / 1e3 / peaks["hbm_gbs"], 3),
                          "steady_sets": nsets, "steady_cold": nsets * by >= SET_BYTES,
                          "graph_us": round(tg, 2),
                          "graph_frac_hbm": round(by / tg / 1e3 / peaks["hbm_gbs"], 3)}),
              flush=True)
    bi.set_batch_invariant_limit(INVARIANT)
    # row-wise log-softmax (fp32 logits rows) and mean (bf16 activation rows)
    for rows, n in ((32, 128256), (2048, 4096)):
        xl = torch.randn(rows, n, device=dev)
        by = 8 * rows * n
        nsets = max(1, min(64, -(-SET_BYTES // by)))
        sets = [(xl.clone(), torch.empty_like(xl)) for _ in range(nsets)]
        t = t_us(lambda: bi.log_softmax(xl, out=sets[0][1]))
        tg = graph_us([lambda a=a, o=o: bi.log_softmax(a, out=o) for a, o in sets])
        del sets
        print(json.dumps({"sweep": "log_softmax", "rows": rows, "n": n, "us": round(t, 2),
                          "graph_us": round(tg, 2), "graph_GB/s": round(by / tg / 1e3, 1),
                          "graph_frac_hbm": round(by / tg / 1e3 / peaks["hbm_gbs"], 3)}),
              flush=True)
    for rows, n in ((2048, 4096), (32, 128256)):
        xm = torch.randn(rows, n, device=dev).to(torch.bfloat16)
        om = torch.empty(rows, device=dev)
        by = 2 * rows * n + 4 * rows
        nsets = max(1, min(64, -(-SET_BYTES // by)))
        sets = [xm.clone() for _ in range(nsets)]
        t = t_us(lambda: bi.mean(xm, out=om))
        tg = graph_us([lambda a=a: bi.mean(a, out=om) for a in sets])
        del sets
        print(json.dumps({"sweep": "mean", "rows": rows, "n": n, "dtype": "bf16",
                          "us": round(t, 2), "graph_us": round(tg, 2),
                          "graph_GB/s": round(by / tg / 1e3, 1),
                          "graph_frac_hbm": round(by / tg / 1e3 / peaks["hbm_gbs"], 3)}),
              flush=True)
    for B, q, L in ((1, 1, 65540), (1, 8, 65540), (1, 8, 16388), (1, 8, 8196), (1, 8, 1028),
                    (8, 1, 65540), (64, 1, 16388), (64, 4, 8196)):
        bi.set_batch_invariant_limit(INVARIANT)
        p = inputs.paged_inputs([L] * B, [q] * B, Hq=HQ, Hkv=HKV, D=HEAD_DIM, seed=4, device=dev)
        d = {k: getattr(p, k).to(dev) for k in ("q", "k_cache", "v_cache", "block_table",
                                                 "seq_lens", "cu_q")}
        # 8x the invariant workspace: every chunk length is open to the fast path
        ws = torch.empty(8 * bi.attn_workspace_size(B * q, HQ, HEAD_DIM, L), dtype=torch.uint8,
                         device=dev)
        out = torch.empty(B * q, HQ, HEAD_DIM, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(B * q, HQ, dtype=torch.float32, device=dev)
        t = t_us(lambda: bi.verify_block(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                         d["seq_lens"], d["cu_q"], max_q=q, max_seq_len=L,
                                         scale=1 / math.sqrt(HEAD_DIM), out=out, lse=lse,
                                         workspace=ws))
        by = B * L * HKV * HEAD_DIM * 2 * 2
        ts = steady_us([lambda: bi.verify_block(d["q"], d["k_cache"], d["v_cache"],
                                                d["block_table"], d["seq_lens"], d["cu_q"],
                                                max_q=q, max_seq_len=L,
                                                scale=1 / math.sqrt(HEAD_DIM), out=out,
                                                lse=lse, workspace=ws)], n=30)
        # device time per call from a CUDA graph, rotating over copies of the caches
        # until the set exceeds 2x L2
        nsets = 1 if by >= SET_BYTES else min(64, -(-SET_BYTES // by))
        caches = [(d["k_cache"], d["v_cache"])] + [
            (d["k_cache"].clone(), d["v_cache"].clone()) for _ in range(nsets - 1)]
        calls = [lambda kc=kc, vc=vc: bi.verify_block(
            d["q"], kc, vc, d["block_table"], d["seq_lens"], d["cu_q"], max_q=q, max_seq_len=L,
            scale=1 / math.sqrt(HEAD_DIM), out=out, lse=lse, workspace=ws) for kc, vc in caches]
        n_graph = max(8, min(64, nsets * 2))
        tg = graph_us(calls, n=n_graph)
        bi.set_batch_invariant_limit(FAST)
        tfg = graph_us(calls, n=n_graph)
        del caches, calls
        chunk = bi.attn_chunk(B, B * q, q, L, HQ, HKV, HEAD_DIM, ws.numel(), sms)
        tf = t_us(lambda: bi.verify_block(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                          d["seq_lens"], d["cu_q"], max_q=q, max_seq_len=L,
                                          scale=1 / math.sqrt(HEAD_DIM), out=out, lse=lse,
                                          workspace=ws))
        tfs = steady_us([lambda: bi.verify_block(d["q"], d["k_cache"], d["v_cache"],
                                                 d["block_table"], d["seq_lens"], d["cu_q"],
                                                 max_q=q, max_seq_len=L,
                                                 scale=1 / math.sqrt(HEAD_DIM), out=out,
                                                 lse=lse, workspace=ws)], n=30)
        print(json.dumps({"sweep": "attention", "B": B, "q": q, "Lk": L, "us": round(t, 2),
                          "GB/s": round(by / t / 1e3, 1),
                          "frac_hbm": round(by / t / 1e3 / peaks["hbm_gbs"], 3),
                          "steady_us": round(ts, 2), "steady_GB/s": round(by / ts / 1e3, 1),
                          "steady_frac_hbm": round(by / ts / 1e3 / peaks["hbm_gbs"], 3),
                          "steady_cold": by >= SET_BYTES, "fast_chunk": chunk,
                          "fast_us": round(tf, 2), "steady_fast_us": round(tfs, 2),
                          "fast_frac_hbm": round(by / tf / 1e3 / peaks["hbm_gbs"], 3),
                          "invariance_tax": round(t / tf - 1.0, 3),
                          "graph_us": round(tg, 2), "graph_fast_us": round(tfg, 2),
                          "graph_sets": nsets,
                          "graph_frac_hbm": round(by / tg / 1e3 / peaks["hbm_gbs"], 3),
                          "graph_fast_frac_hbm": round(by / tfg / 1e3 / peaks["hbm_gbs"], 3),
                          "graph_invariance_tax": round(tg / tfg - 1.0, 3)}), flush=True)
        del p, d, ws
        torch.cuda.empty_cache()

    # chunked prefill (causal): the whole prompt, and 512 new tokens after a cached prefix.
    # Tensor-bound: flops = 4 * D * Hq * sum over queries of (keys seen)
    for L, qb in ((8192, 8192), (8192, 512), (65540, 512)):
        bi.set_batch_invariant_limit(INVARIANT)
        p = inputs.paged_inputs([L], [qb], Hq=HQ, Hkv=HKV, D=HEAD_DIM, seed=5, device=dev)
        d = {k: getattr(p, k).to(dev) for k in ("q", "k_cache", "v_cache", "block_table",
                                                 "seq_lens", "cu_q")}
        ws = torch.empty(bi.attn_workspace_size(qb, HQ, HEAD_DIM, L), dtype=torch.uint8,
                         device=dev)
        out = torch.empty(qb, HQ, HEAD_DIM, dtype=torch.bfloat16, device=dev)
        call = lambda: bi.prefill_attn(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                       d["seq_lens"], d["cu_q"], max_q=qb, max_seq_len=L,
                                       scale=1 / math.sqrt(HEAD_DIM), out=out, want_lse=False,
                                       workspace=ws)
        t = t_us(call)
        tg = graph_us([call], n=4, reps=5)
        seen = float(sum(range(L - qb + 1, L + 1)))
        flops = 4.0 * HEAD_DIM * HQ * seen
        print(json.dumps({"sweep": "prefill", "Lk": L, "new_tokens": qb, "us": round(t, 2),
                          "graph_us": round(tg, 2),
                          "TFLOP/s": round(flops / tg / 1e6, 1),
                          "graph_frac_tensor": round(flops / tg / 1e6 / peaks["bf16_tflops"], 3),
                          "tokens/s": round(qb / tg * 1e6)}), flush=True)
        del p, d, ws, out
        torch.cuda.empty_cache()


if __name__ == "__main__":
    main()
