"""Benchmark of the paged-attention hot path on one GB300 (or N replicas).

A step is one decode step of the decode-batch workload through all 28 layers:
for each layer, the KV write of the 256 new tokens into that layer's pool and
paged decode attention of the 256 queries (256 sequences, context_lens
U[100, 1024], block_size 256, 16 query / 8 KV heads x 128, bf16; every layer
has its own pool, so the 28 pools, about 20 GB, never fit in L2).  Each layer
is one pa_store_decode_paged call (the KV write fused into the decode launch);
the step is captured once in a CUDA graph and replayed.

The JSON line reports:
  value         algorithmic HBM bytes of the step (KV write + decode) / step
                time, GB/s, device-resident inputs, CUDA events;
  tokens_per_s  decode tokens per second (256 per step);
  eager         the same calls launched one by one from Python;
  unfused       the same step with pa_store_kvcache + pa_decode_paged per
                layer, also graph-captured;
  e2e           the same metric through the C ABI with inputs copied from
                pinned host memory and outputs copied back inside the timed
                region;
  roofline      of the fused KV write + decode call (split kernel and merge),
                against the measured HBM copy bandwidth;
  prefill       the varlen-prefill (16384 packed tokens) and prefix+chunk
                workloads: KV write + prefill, TFLOP/s of visible pairs;
  long_decode   the 512-sequence, 4096-context decode, GB/s;
  cpu_baseline  the CPU oracle on a bounded sample of the step's workload.

``--impl reference`` times the CPU oracle alone on a bounded sample of the
same workload, reporting the same metric.
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
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_110_gb300 import workloads as wl  # noqa: E402

METRIC = "paged decode attn HBM GB/s (% of ~8 TB/s); varlen prefill TFLOP/s; tokens/s"
LAYERS = 28
HQ, HKV, D = wl.HQ, wl.HKV, wl.HEAD_DIM
ROW_BYTES = HKV * D * 2  # one token's K (or V) row of one layer

# DRAM traffic per call from ncu captures (dram__bytes_read.sum +
# dram__bytes_write.sum; one-pass metrics, clock control off), valid only
# while the code of the kernel's source file is unchanged (the key hashes the
# file with its comments and whitespace taken out, so that a comment edit
# keeps the capture and any code edit drops it):
#   decode: the split kernel (mean of two launches) + the merge kernel of one
#     pa_store_decode_paged call, decode-batch workload (2 layers, eager pass);
#   prefill: one prefill_tc_kernel launch of the varlen-prefill workload.
NCU_TRAFFIC = {"code_sha256": "b527dbc7cb18d8b9cd31c12ccf83ae5106d8c6842ddc2b4636f2328a155b8b60",
               "bytes_per_call": 587_439_488 + 6_371_968 + 10_270_208,
               "kernel": "decode_split_kernel<2, 0, 0> + decode_merge_kernel"}
NCU_TRAFFIC_PREFILL = {"code_sha256": "5783926236cbd97f4ba27b9a10d83c8eb239572fc08ae3829f819de54f61be4e",
                       "bytes_per_call": 166_617_088 + 33_789_184, "kernel": "prefill_tc_kernel<0>"}


def _code_sha(path):
    """sha256 of a C / CUDA source's code: comments removed (string and
    character literals kept whole), then every run of whitespace made one
    space."""
    with open(path, encoding="utf-8") as f:
        src = f.read()
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return hashlib.sha256(" ".join("".join(out).split()).encode()).hexdigest()


# ----------------------------------------------------------------- distributed


def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max_sum(world, t_max: float, units_sum: float):
    """Max over ranks of the elapsed time, sum over ranks of the work done."""
    if world == 1:
        return t_max, units_sum
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    a = torch.tensor([t_max], dtype=torch.float64, device=dev)
    b = torch.tensor([units_sum], dtype=torch.float64, device=dev)
    dist.all_reduce(a, op=dist.ReduceOp.MAX)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(a.item()), float(b.item())


# ----------------------------------------------------------------- algorithmic counts


def decode_bytes(ctx, block_size, num_heads=HQ, kv_heads=HKV, head_dim=D, kv_elem_bytes=2):
    """K+V rows read + q read + out written + table entries + context_lens."""
    ctx = np.asarray(ctx, dtype=np.int64)
    kv = int(ctx.sum()) * kv_heads * head_dim * kv_elem_bytes * 2
    qo = len(ctx) * num_heads * head_dim * 2 * 2
    tables = int((-(-ctx // block_size)).sum()) * 4 + len(ctx) * 4
    return kv + qo + tables


def store_bytes(num_tokens, kv_heads=HKV, head_dim=D):
    """K and V rows read and written + the slot."""
    return num_tokens * (kv_heads * head_dim * 2 * 2 * 2 + 4)


def prefill_flops(query_lens, context_lens, num_heads=HQ, head_dim=D):
    """4 * d * Hq per visible (query, key) pair (QK^T and PV, 2 flops each)."""
    pairs = 0
    for lq, lk in zip(np.asarray(query_lens, np.int64), np.asarray(context_lens, np.int64)):
        off = lk - lq
        pairs += lq * (off + 1) + lq * (lq - 1) // 2  # sum_{i<lq} (off + i + 1)
    return 4 * head_dim * num_heads * int(pairs)


# ----------------------------------------------------------------- peaks and clocks


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def wait_first(self, timeout=3.0):
        t0 = time.time()
        while self.proc is not None and not self.lines and time.time() - t0 < timeout:
            time.sleep(0.05)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self, t0=None, t1=None):
        """Samples taken between host times t0 and t1 (the timed region)."""
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if (t0 is not None and ts < t0) or (t1 is not None and ts > t1):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- the decode-batch step


class DecodeStep:
    """28 layers of (KV write of the new tokens, paged decode) over distinct
    per-layer pools that share one set of block tables.  With `fused` (the
    default) each layer is one pa_store_decode_paged call; otherwise
    pa_store_kvcache then pa_decode_paged."""

    def __init__(self, device, seed=wl.SEED_BASE + 2, layers=LAYERS, keep_host_layer0=False, fused=True):
        self.fused = fused
        from paged_kv_cache_110_gb300 import binding as pa
        self.pa = pa
        self.dev = device
        self.layers = layers
        ctx = wl.rng(seed + 7).integers(100, 1024, size=256, endpoint=True).astype(np.int32)
        self.ctx = ctx
        self.layout = wl.make_layout(seed, ctx, 256)
        self.B = len(ctx)
        self.max_ctx = int(ctx.max())
        self.k_cache, self.v_cache, self.tokens = [], [], []
        self.host_layer0 = None
        for l in range(layers):
            kc, vc = wl.make_pool(self.layout, ctx - 1, seed + 1000 * (l + 1), device=device)
            if l == 0 and keep_host_layer0:
                self.host_layer0 = (wl.bf16_bits(kc).copy(), wl.bf16_bits(vc).copy())
            self.k_cache.append(kc)
            self.v_cache.append(vc)
            self.tokens.append(wl.new_tokens(seed + 1000 * (l + 1) + 1, self.B, device=device))
        self.slots_np = np.array([self.layout.slots(b, [c - 1])[0] for b, c in enumerate(ctx)], np.int32)
        self.slots = torch.as_tensor(self.slots_np, device=device)
        self.tables = torch.as_tensor(self.layout.block_tables, device=device)
        self.ctx_t = torch.as_tensor(ctx, device=device)
        n = pa.pa_decode_workspace_bytes(self.B, HQ, D, self.max_ctx)
        self.ws = torch.empty(max(n, 256), dtype=torch.uint8, device=device)
        self.out = [torch.empty((self.B, HQ, D), dtype=torch.bfloat16, device=device) for _ in range(layers)]
        self.decode_bytes = decode_bytes(ctx, 256)
        self.store_bytes = store_bytes(self.B)
        self.step_bytes = layers * (self.decode_bytes + self.store_bytes)

    @property
    def call_bytes(self):
        """Algorithmic bytes of the call the events time: the fused KV write +
        decode, or the decode alone."""
        return self.decode_bytes + (self.store_bytes if self.fused else 0)

    def run(self, events=None):
        pa = self.pa
        for l in range(self.layers):
            t = self.tokens[l]
            if not self.fused:
                pa.pa_store_kvcache(t.k, t.v, self.k_cache[l], self.v_cache[l], self.slots)
            if events is not None:
                events.append((torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)))
                events[-1][0].record()
            if self.fused:
                pa.pa_store_decode_paged(t.q, t.k, t.v, self.k_cache[l], self.v_cache[l], self.tables, self.ctx_t,
                                         self.max_ctx, wl.SCALE, self.out[l], self.ws)
            else:
                pa.pa_decode_paged(t.q, self.k_cache[l], self.v_cache[l], self.tables, self.ctx_t, self.max_ctx,
                                   wl.SCALE, self.out[l], self.ws)
            if events is not None:
                events[-1][1].record()

    def launches_per_step(self):
        # per layer: the decode kernel, its merge when the keys are split, and the
        # KV-write kernel unless it is fused into the decode
        return self.layers * ((0 if self.fused else 1) + (2 if self._multi_split() else 1))

    def _multi_split(self):
        # the library uses a merge kernel whenever a workspace is needed
        return self.pa.pa_decode_workspace_bytes(self.B, HQ, D, self.max_ctx) > 0


class E2EStep:
    """The same step with host buffers: pinned host -> device copies of each
    layer's new q/k/v and the step's metadata, the 28 layers, and the outputs
    copied back, all inside the timed region."""

    def __init__(self, step: DecodeStep):
        self.s = step
        self.h_qkv = [t.qkv.cpu().pin_memory() for t in step.tokens]
        self.d_qkv = [torch.empty_like(t.qkv) for t in step.tokens]
        self.h_slots = torch.as_tensor(step.slots_np).pin_memory()
        self.h_tables = torch.as_tensor(step.layout.block_tables).pin_memory()
        self.h_ctx = torch.as_tensor(step.ctx).pin_memory()
        self.h_out = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in step.out]
        a, b = HQ * D, (HQ + HKV) * D
        self.views = [(q[:, :a].view(-1, HQ, D), q[:, a:b].view(-1, HKV, D), q[:, b:].view(-1, HKV, D))
                      for q in self.d_qkv]
        meta = (self.h_tables, self.h_ctx) if step.fused else (self.h_slots, self.h_tables, self.h_ctx)
        self.h2d = sum(t.numel() * t.element_size() for t in self.h_qkv) + \
            sum(t.numel() * t.element_size() for t in meta)
        self.d2h = sum(t.numel() * t.element_size() for t in self.h_out)

    def layer(self, l):
        """Layer l's C-ABI call(s) on the current stream."""
        s, pa = self.s, self.s.pa
        q, k, v = self.views[l]
        if s.fused:
            pa.pa_store_decode_paged(q, k, v, s.k_cache[l], s.v_cache[l], s.tables, s.ctx_t, s.max_ctx, wl.SCALE,
                                     s.out[l], s.ws)
        else:
            pa.pa_store_kvcache(k, v, s.k_cache[l], s.v_cache[l], s.slots)
            pa.pa_decode_paged(q, s.k_cache[l], s.v_cache[l], s.tables, s.ctx_t, s.max_ctx, wl.SCALE, s.out[l],
                               s.ws)

    def run(self):
        s = self.s
        if not s.fused:
            s.slots.copy_(self.h_slots, non_blocking=True)
        s.tables.copy_(self.h_tables, non_blocking=True)
        s.ctx_t.copy_(self.h_ctx, non_blocking=True)
        for l in range(s.layers):
            self.d_qkv[l].copy_(self.h_qkv[l], non_blocking=True)
            self.layer(l)
            self.h_out[l].copy_(s.out[l], non_blocking=True)


class E2EGraphStep:
    """The end-to-end step as a serving engine runs it: the public C-ABI calls
    of one step (pinned host -> device copies of each layer's new q/k/v and the
    metadata, the 28 layers' KV write + decode, every layer's output copied
    back) captured once in a CUDA graph and replayed.  Copies run on their own
    streams so that layer l+1's inputs arrive and layer l's output leaves while
    other layers compute; every copy stays inside each replay."""

    def __init__(self, e: E2EStep):
        self.e = e
        s = e.s
        main = torch.cuda.current_stream()
        h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
        self.graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(main)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(self.graph):
                start = torch.cuda.Event()
                start.record(cap)
                h2d.wait_event(start)
                d2h.wait_event(start)
                ev_in = [torch.cuda.Event() for _ in range(s.layers)]
                ev_out = [torch.cuda.Event() for _ in range(s.layers)]
                with torch.cuda.stream(h2d):
                    if not s.fused:
                        s.slots.copy_(e.h_slots, non_blocking=True)
                    s.tables.copy_(e.h_tables, non_blocking=True)
                    s.ctx_t.copy_(e.h_ctx, non_blocking=True)
                    for l in range(s.layers):
                        e.d_qkv[l].copy_(e.h_qkv[l], non_blocking=True)
                        ev_in[l].record(h2d)
                for l in range(s.layers):
                    cap.wait_event(ev_in[l])
                    e.layer(l)
                    ev_out[l].record(cap)
                with torch.cuda.stream(d2h):
                    for l in range(s.layers):
                        d2h.wait_event(ev_out[l])
                        e.h_out[l].copy_(s.out[l], non_blocking=True)
                done = torch.cuda.Event()
                done.record(d2h)
                cap.wait_event(done)
                h2d_done = torch.cuda.Event()
                h2d_done.record(h2d)
                cap.wait_event(h2d_done)
        main.wait_stream(cap)

    def run(self):
        self.graph.replay()


def time_region(fn, steps, world):
    barrier(world)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(steps):
        fn()
    end.record()
    torch.cuda.synchronize()
    barrier(world)
    return start.elapsed_time(end) / 1e3  # seconds


# ----------------------------------------------------------------- prefill and long decode legs


def flush_l2(buf):
    """Write a buffer larger than L2 (the first half of buf), then read another
    one larger than L2 (the second half): the read evicts the written lines,
    so their write-back to HBM happens here and not inside the next timed
    call, which would otherwise pay for up to an L2's worth of foreign writes."""
    half = buf.numel() // 2
    buf[:half].add_(1)
    buf[half:].max()


def prefill_ws(pa, num_seqs, max_q, max_k, device):
    """The caller-owned workspace a prefill call asks for (at least 256 bytes)."""
    n = pa.pa_prefill_workspace_bytes(num_seqs, int(max_q), int(max_k), HQ, HKV)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def time_prefill(device, steps, warmup, flush, only="all"):
    from paged_kv_cache_110_gb300 import binding as pa
    res = {}
    cases = {}
    if only in ("all", "varlen_16k"):
        cases["varlen_16k"] = [wl.varlen_prefill(device=device)]
    if only in ("all", "prefix_2048_chunked"):
        a, b, _ = wl.prefix_chunk(device=device)
        cases["prefix_2048_chunked"] = [a, b]
    if only in ("all", "chunk_512_over_8k"):
        # one long prompt's chunk: 512 new tokens over 7,680 cached ones (few
        # work items: the key range of each is split over several CTAs)
        cases["chunk_512_over_8k"] = [wl.paged_batch(wl.SEED_BASE + 9, [8192], [512], 256, device=device)]
    for name, calls in cases.items():
        kc, vc = calls[0].k_cache, calls[0].v_cache
        prepared = []
        flops = 0
        for c in calls:
            out = torch.empty(c.tokens.q.shape, dtype=torch.bfloat16, device=device)
            prepared.append((c, out, torch.as_tensor(c.slot_mapping, device=device),
                             torch.as_tensor(c.block_tables, device=device),
                             torch.as_tensor(c.cu_seqlens_q, device=device),
                             torch.as_tensor(c.cu_seqlens_k, device=device)))
            flops += prefill_flops(c.query_lens, c.context_lens)

        wss = [torch.empty(max(pa.pa_prefill_workspace_bytes(c.layout.num_seqs, int(c.query_lens.max()),
                                                              int(c.context_lens.max()), HQ, HKV), 256),
                           dtype=torch.uint8, device=device) for c in calls]

        def run(ev=None):
            for (c, out, sl, bt, cq, ck), ws in zip(prepared, wss):
                pa.pa_store_kvcache(c.tokens.k, c.tokens.v, kc, vc, sl)
                if ev is not None:
                    ev.append((torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)))
                    ev[-1][0].record()
                pa.pa_prefill_paged(c.tokens.q, cq, ck, int(c.query_lens.max()), int(c.context_lens.max()),
                                    c.scale, out, k_cache=kc, v_cache=vc, block_table=bt, workspace=ws)
                if ev is not None:
                    ev[-1][1].record()

        for _ in range(warmup):
            run()
        torch.cuda.synchronize()
        times = []
        for _ in range(steps):
            flush_l2(flush)
            ev = []
            run(ev)
            torch.cuda.synchronize()
            times.append(sum(s.elapsed_time(e) for s, e in ev) / 1e3)
        t = statistics.median(times)
        res[name] = {"tflops": flops / t / 1e12, "ms": t * 1e3, "gflop": flops / 1e9,
                     "query_tokens": int(sum(c.num_tokens for c in calls)), "calls": len(calls)}
    return res


def time_long_decode(device, steps, warmup, flush, seqs=512):
    from paged_kv_cache_110_gb300 import binding as pa
    batch = wl.long_decode(device=device, num_seqs=seqs)
    max_ctx = int(batch.context_lens.max())
    ws = torch.empty(max(pa.pa_decode_workspace_bytes(seqs, HQ, D, max_ctx), 256), dtype=torch.uint8, device=device)
    out = torch.empty((seqs, HQ, D), dtype=torch.bfloat16, device=device)
    bt = torch.as_tensor(batch.block_tables, device=device)
    ctx = torch.as_tensor(batch.context_lens, device=device)
    sl = torch.as_tensor(batch.slot_mapping, device=device)
    pa.pa_store_kvcache(batch.tokens.k, batch.tokens.v, batch.k_cache, batch.v_cache, sl)
    for _ in range(warmup):
        pa.pa_decode_paged(batch.tokens.q, batch.k_cache, batch.v_cache, bt, ctx, max_ctx, batch.scale, out, ws)
    times = []
    for _ in range(steps):
        flush_l2(flush)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        pa.pa_decode_paged(batch.tokens.q, batch.k_cache, batch.v_cache, bt, ctx, max_ctx, batch.scale, out, ws)
        e.record()
        torch.cuda.synchronize()
        times.append(s.elapsed_time(e) / 1e3)
    t = statistics.median(times)
    nbytes = decode_bytes(batch.context_lens, 256)
    del batch
    return {"gbs": nbytes / t / 1e9, "ms": t * 1e3, "bytes": nbytes, "seqs": seqs}


def time_long_decode_fp8(device, steps, warmup, flush, scale=2.0 ** -6, seqs=512):
    """The long-decode workload over fp8 (E4M3) pools: the bf16 pool's history
    and the new tokens quantised by pa_store_kvcache_fp8, then
    pa_decode_paged_fp8 timed with L2 flushed before each call."""
    from paged_kv_cache_110_gb300 import binding as pa
    batch = wl.long_decode(device=device, num_seqs=seqs)
    shape = batch.k_cache.shape
    k8 = torch.empty(shape, dtype=torch.uint8, device=device)
    v8 = torch.empty(shape, dtype=torch.uint8, device=device)
    hist = wl.history_rows(batch.layout, batch.context_lens - 1)
    rows = torch.as_tensor(hist.astype(np.int64), device=device)
    for chunk in torch.split(rows, 1 << 18):
        hk = batch.k_cache.view(-1, HKV, D).index_select(0, chunk)
        hv = batch.v_cache.view(-1, HKV, D).index_select(0, chunk)
        pa.pa_store_kvcache_fp8(hk, hv, scale, scale, k8, v8, chunk.to(torch.int32))
    pa.pa_store_kvcache_fp8(batch.tokens.k, batch.tokens.v, scale, scale, k8, v8,
                            torch.as_tensor(batch.slot_mapping, device=device))
    max_ctx = int(batch.context_lens.max())
    ctx_np = batch.context_lens
    ws = torch.empty(max(pa.pa_decode_workspace_bytes(seqs, HQ, D, max_ctx), 256), dtype=torch.uint8, device=device)
    out = torch.empty((seqs, HQ, D), dtype=torch.bfloat16, device=device)
    bt = torch.as_tensor(batch.block_tables, device=device)
    ctx = torch.as_tensor(ctx_np, device=device)
    q = batch.tokens.q
    del batch
    torch.cuda.empty_cache()

    def run():
        pa.pa_decode_paged_fp8(q, k8, v8, scale, scale, bt, ctx, max_ctx, wl.SCALE, out, ws)

    for _ in range(warmup):
        run()
    times = []
    for _ in range(steps):
        flush_l2(flush)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        run()
        e.record()
        torch.cuda.synchronize()
        times.append(s.elapsed_time(e) / 1e3)
    t = statistics.median(times)
    nbytes = decode_bytes(ctx_np, 256, kv_elem_bytes=1)
    return {"gbs": nbytes / t / 1e9, "ms": t * 1e3, "bytes": nbytes, "seqs": seqs, "kv": "fp8 e4m3, scale 2^-6"}


def time_gqa_decode(device, steps, warmup, flush, peak_gbs):
    """pa_decode_paged on the decode batch's contexts (256 sequences, U[100,
    1024], block_size 256) with larger query groups: 32 and 64 query heads over
    8 KV heads (4 and 8 per KV head, the tensor-core decode kernel) beside the
    16 / 8 of the headline (the CUDA-core kernel).  L2 flushed before each call."""
    from paged_kv_cache_110_gb300 import binding as pa
    res = {}
    ctx = wl.rng(wl.SEED_BASE + 9).integers(100, 1024, size=256, endpoint=True)
    for hq, hkv in ((16, 8), (32, 8), (64, 8)):
        b = wl.paged_batch(wl.SEED_BASE + 70, ctx, np.ones_like(ctx), 256, num_heads=hq, num_kv_heads=hkv,
                           device=device)
        max_ctx = int(ctx.max())
        ws = torch.empty(max(pa.pa_decode_workspace_bytes(256, hq, D, max_ctx), 256), dtype=torch.uint8,
                         device=device)
        out = torch.empty((256, hq, D), dtype=torch.bfloat16, device=device)
        bt, cx = torch.as_tensor(b.block_tables, device=device), torch.as_tensor(b.context_lens, device=device)

        def dec():
            pa.pa_decode_paged(b.tokens.q, b.k_cache, b.v_cache, bt, cx, max_ctx, b.scale, out, ws)

        for _ in range(warmup):
            dec()
        times = []
        for _ in range(steps):
            flush_l2(flush)
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            dec()
            e.record()
            torch.cuda.synchronize()
            times.append(s.elapsed_time(e) / 1e3)
        t = statistics.median(times)
        gbs = decode_bytes(ctx, 256, num_heads=hq, kv_heads=hkv) / t / 1e9
        res[f"{hq}q_{hkv}kv"] = {"us": t * 1e6, "gbs": gbs, "frac": gbs / peak_gbs}
        del b
        torch.cuda.empty_cache()
    return res


def time_block_size_sweep(device, steps, warmup, flush):
    """Decode (the 256-sequence decode batch) and varlen prefill at block sizes
    16..256: the same contexts and lengths, pools and tables rebuilt per size;
    L2 flushed before each timed call."""
    from paged_kv_cache_110_gb300 import binding as pa
    res = {"decode_gbs": {}, "prefill_tflops": {}}
    seed = wl.SEED_BASE + 2
    ctx = wl.rng(seed + 7).integers(100, 1024, size=256, endpoint=True)
    lens = wl.varlen_prefill_lengths()
    for bs in (16, 32, 64, 128, 256):
        b = wl.paged_batch(seed, ctx, np.ones_like(ctx), bs, device=device)
        sl = torch.as_tensor(b.slot_mapping, device=device)
        pa.pa_store_kvcache(b.tokens.k, b.tokens.v, b.k_cache, b.v_cache, sl)
        max_ctx = int(ctx.max())
        ws = torch.empty(max(pa.pa_decode_workspace_bytes(256, HQ, D, max_ctx), 256), dtype=torch.uint8,
                         device=device)
        out = torch.empty((256, HQ, D), dtype=torch.bfloat16, device=device)
        bt, cx = torch.as_tensor(b.block_tables, device=device), torch.as_tensor(b.context_lens, device=device)

        def dec():
            pa.pa_decode_paged(b.tokens.q, b.k_cache, b.v_cache, bt, cx, max_ctx, b.scale, out, ws)

        for _ in range(warmup):
            dec()
        times = []
        for _ in range(steps):
            flush_l2(flush)
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            dec()
            e.record()
            torch.cuda.synchronize()
            times.append(s.elapsed_time(e) / 1e3)
        res["decode_gbs"][bs] = decode_bytes(ctx, bs) / statistics.median(times) / 1e9
        del b
        if bs in (16, 64, 256):
            p = wl.paged_batch(wl.SEED_BASE + 3, lens, lens, bs, device=device)
            pa.pa_store_kvcache(p.tokens.k, p.tokens.v, p.k_cache, p.v_cache,
                                torch.as_tensor(p.slot_mapping, device=device))
            pout = torch.empty(p.tokens.q.shape, dtype=torch.bfloat16, device=device)
            pbt = torch.as_tensor(p.block_tables, device=device)
            cq, ck = (torch.as_tensor(x, device=device) for x in (p.cu_seqlens_q, p.cu_seqlens_k))

            pws = prefill_ws(pa, p.layout.num_seqs, int(lens.max()), int(lens.max()), device)

            def pre():
                pa.pa_prefill_paged(p.tokens.q, cq, ck, int(lens.max()), int(lens.max()), p.scale, pout,
                                    k_cache=p.k_cache, v_cache=p.v_cache, block_table=pbt, workspace=pws)

            for _ in range(warmup):
                pre()
            times = []
            for _ in range(steps):
                flush_l2(flush)
                s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                s.record()
                pre()
                e.record()
                torch.cuda.synchronize()
                times.append(s.elapsed_time(e) / 1e3)
            res["prefill_tflops"][bs] = prefill_flops(lens, lens) / statistics.median(times) / 1e12
            del p
        torch.cuda.empty_cache()
    return res


def rope_store_bytes(num_tokens, hq=HQ, hkv=HKV):
    """Algorithmic bytes of the fused head norm + RoPE + KV write per call: the
    fused QKV row read, Q written, K and V rows written, position and slot read
    (the cos/sin table and the norm weights are shared by all tokens and not
    counted)."""
    row = (hq + 2 * hkv) * D * 2
    return num_tokens * (row + hq * D * 2 + 2 * hkv * D * 2 + 8)


def time_rope_store(device, steps, warmup, flush):
    """The fused head norm + RoPE + KV write on the varlen-prefill batch
    (16,384-token budget, block size 256) and on the 256-token decode batch,
    L2 flushed before each call."""
    from paged_kv_cache_110_gb300 import binding as pa
    cs = pa.pa_rope_cos_sin_table(wl.ROPE_BASE, D, 4096, device=device)
    qw, kw = wl.norm_weights(wl.SEED_BASE + 7, device=device)
    res = {}
    cases = {"varlen_16k": wl.varlen_prefill(device=device), "decode_256": wl.decode_batch(device=device)}
    for name, b in cases.items():
        q_out = torch.empty((b.num_tokens, HQ, D), dtype=torch.bfloat16, device=device)
        pos = torch.as_tensor(b.positions, device=device)
        sl = torch.as_tensor(b.slot_mapping, device=device)

        def run():
            pa.pa_norm_rope_store_kvcache(b.tokens.qkv, HQ, HKV, pos, cs, qw, kw, wl.RMS_EPS, q_out, b.k_cache,
                                          b.v_cache, sl)

        for _ in range(warmup):
            run()
        times = []
        for _ in range(steps):
            flush_l2(flush)
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            run()
            e.record()
            torch.cuda.synchronize()
            times.append(s.elapsed_time(e) / 1e3)
        t = statistics.median(times)
        nbytes = rope_store_bytes(b.num_tokens)
        res[name] = {"gbs": nbytes / t / 1e9, "us": t * 1e6, "bytes": nbytes, "tokens": b.num_tokens}
        del b
    return res


def time_mixed(device, steps, warmup, flush):
    """Mixed step: the 256-sequence decode batch plus one 512-token prefill
    chunk over a 2,048-token cached prefix, as ONE prefill launch (decode rows
    are queries of length 1) against the chunk's prefill launch followed by
    the decode launch; L2 flushed before each timed call."""
    from paged_kv_cache_110_gb300 import binding as pa
    dec = wl.decode_batch(device="cpu")
    ctx = np.concatenate([[2048 + 512], dec.context_lens]).astype(np.int32)
    ql = np.concatenate([[512], dec.query_lens]).astype(np.int32)
    b = wl.paged_batch(wl.SEED_BASE + 8, ctx, ql, 256, device=device)
    kc, vc = b.k_cache, b.v_cache
    pa.pa_store_kvcache(b.tokens.k, b.tokens.v, kc, vc, torch.as_tensor(b.slot_mapping, device=device))
    bt = torch.as_tensor(b.block_tables, device=device)
    cq, ck = (torch.as_tensor(x, device=device) for x in (b.cu_seqlens_q, b.cu_seqlens_k))
    out = torch.empty(b.tokens.q.shape, dtype=torch.bfloat16, device=device)
    # separate launches: the chunk alone, then the 256 decode rows
    cq1 = torch.as_tensor(np.array([0, 512], np.int32), device=device)
    ck1 = torch.as_tensor(np.array([0, 2560], np.int32), device=device)
    q1 = b.tokens.q[:512]
    out1 = torch.empty(q1.shape, dtype=torch.bfloat16, device=device)
    qd = b.tokens.q[512:]
    ctx_d = torch.as_tensor(ctx[1:], device=device)
    max_d = int(ctx[1:].max())
    ws = torch.empty(max(pa.pa_decode_workspace_bytes(256, HQ, D, max_d), 256), dtype=torch.uint8, device=device)
    outd = torch.empty((256, HQ, D), dtype=torch.bfloat16, device=device)

    ws_mixed = prefill_ws(pa, len(ctx), 512, int(ctx.max()), device)
    ws_chunk = prefill_ws(pa, 1, 512, 2560, device)

    def mixed():
        pa.pa_prefill_paged(b.tokens.q, cq, ck, 512, int(ctx.max()), b.scale, out, k_cache=kc, v_cache=vc,
                            block_table=bt, workspace=ws_mixed)

    def separate():
        pa.pa_prefill_paged(q1, cq1, ck1, 512, 2560, b.scale, out1, k_cache=kc, v_cache=vc, block_table=bt[:1],
                            workspace=ws_chunk)
        pa.pa_decode_paged(qd, kc, vc, bt[1:], ctx_d, max_d, b.scale, outd, ws)

    res = {}
    for name, fn in (("one_launch", mixed), ("two_launches", separate)):
        for _ in range(warmup):
            fn()
        times = []
        for _ in range(steps):
            flush_l2(flush)
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            fn()
            e.record()
            torch.cuda.synchronize()
            times.append(s.elapsed_time(e) * 1e3)
        res[name] = {"us": statistics.median(times)}
    res["workload"] = "256 decode rows (context U[100,1024]) + one 512-token chunk over a 2,048-token prefix"
    return res


def time_decode_layer_step(device, steps, warmup, layers=LAYERS):
    """The decode step of the attention layers with the head norm and RoPE of
    the new tokens included (the decode-batch workload, 28 layers, graph-
    captured): per layer either pa_norm_rope_store_decode_paged (one call), or
    pa_norm_rope_store_kvcache followed by pa_decode_paged (two calls)."""
    from paged_kv_cache_110_gb300 import binding as pa
    step = DecodeStep(device, layers=layers)
    cs = pa.pa_rope_cos_sin_table(wl.ROPE_BASE, D, 4096, device=device)
    qw, kw = wl.norm_weights(21, device=device)
    pos = torch.as_tensor((step.ctx - 1).astype(np.int32), device=device)
    q_out = [torch.empty((step.B, HQ, D), dtype=torch.bfloat16, device=device) for _ in range(layers)]

    def fused():
        for l in range(layers):
            pa.pa_norm_rope_store_decode_paged(step.tokens[l].qkv, HQ, HKV, cs, qw, kw, wl.RMS_EPS, step.k_cache[l],
                                               step.v_cache[l], step.tables, step.ctx_t, step.max_ctx, wl.SCALE,
                                               step.out[l], step.ws)

    def two():
        for l in range(layers):
            pa.pa_norm_rope_store_kvcache(step.tokens[l].qkv, HQ, HKV, pos, cs, qw, kw, wl.RMS_EPS, q_out[l],
                                          step.k_cache[l], step.v_cache[l], step.slots)
            pa.pa_decode_paged(q_out[l], step.k_cache[l], step.v_cache[l], step.tables, step.ctx_t, step.max_ctx,
                               wl.SCALE, step.out[l], step.ws)

    res = {}
    for name, fn in (("one_call", fused), ("two_calls", two)):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(g):
                fn()
        torch.cuda.current_stream().wait_stream(side)
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize()
        s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record()
        for _ in range(steps):
            g.replay()
        e0.record()
        torch.cuda.synchronize()
        ms = s0.elapsed_time(e0) / steps
        res[name] = {"ms_per_step": ms, "us_per_layer": ms / layers * 1e3}
        del g
    res["workload"] = ("decode batch x 28 layers (256 seqs, context U[100,1024], block_size 256): head RMSNorm + "
                       "RoPE of q and k, KV write and paged decode per layer, graph-captured")
    return res


def time_step_metadata(device, steps, warmup):
    """Device-built step metadata: the varlen-prefill batch (counts and tables
    of ~20 sequences, 16K tokens expanded) and a 512-sequence decode batch;
    microseconds per call (launch-bound work: no L2 flush)."""
    from paged_kv_cache_110_gb300 import binding as pa
    res = {}
    v = wl.varlen_prefill(device="cpu")
    lens = torch.as_tensor(v.context_lens, device=device)
    zeros = torch.zeros_like(lens)
    vt = torch.as_tensor(v.block_tables, device=device)
    t_tokens = int(v.query_lens.sum())
    rng = wl.rng(wl.SEED_BASE + 5)
    dl = torch.as_tensor(rng.integers(1024, 4096, 512, endpoint=True).astype(np.int32), device=device)
    dt = torch.as_tensor(rng.permutation(512 * 16).astype(np.int32).reshape(512, 16), device=device)
    cases = {
        "prefill_varlen_16k": (lambda: pa.pa_prepare_prefill(lens, zeros, lens, vt, 256, v.layout.num_blocks, t_tokens),
                               {"seqs": int(lens.numel()), "tokens": t_tokens}),
        "decode_512": (lambda: pa.pa_prepare_decode(dl, dt, 256, 512 * 16), {"seqs": 512}),
    }
    reps = 20
    for name, (fn, info) in cases.items():
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        # device time: the calls are captured in a CUDA graph (they are
        # capturable by design) and replayed, so host overhead is excluded
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph):
                for _ in range(reps):
                    fn()
        torch.cuda.current_stream().wait_stream(side)
        for _ in range(warmup):
            graph.replay()
        torch.cuda.synchronize()
        times = []
        for _ in range(steps):
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            graph.replay()
            e.record()
            torch.cuda.synchronize()
            times.append(s.elapsed_time(e) * 1e3 / reps)
        res[name] = dict(info, us=statistics.median(times), timing="CUDA graph of %d calls, per call" % reps)
    return res


# ----------------------------------------------------------------- CPU oracle baseline


def oracle_sample(host_layer0, step_meta, target_s=10.0, max_layers=64):
    """Run the CPU oracle (KV write + decode of the full 256-sequence layer)
    on layer-0 inputs repeatedly for about target_s seconds; returns the
    metric value, cores and a description of the sample."""
    import oracle
    kc0, vc0 = host_layer0
    ctx, tables, slots, tokens = step_meta
    k, v, q = (wl.bf16_bits(t) for t in (tokens.k, tokens.v, tokens.q))
    done = 0
    t0 = time.perf_counter()
    while done < max_layers:
        kc, vc = kc0.copy(), vc0.copy()
        oracle.store_kvcache(k, v, kc, vc, slots)
        oracle.decode(q, kc, vc, tables, ctx, wl.SCALE)
        done += 1
        if time.perf_counter() - t0 >= target_s:
            break
    el = time.perf_counter() - t0
    nbytes = done * (decode_bytes(ctx, 256) + store_bytes(len(ctx)))
    return {"value": nbytes / el / 1e9, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{done} layer(s) of the decode-batch step (KV write + decode of 256 sequences) in {el:.1f} s",
            "seconds": el}


def reference_arm(args, rank, world):
    """The CPU oracle as the reference arm: each step is one layer of the
    decode-batch workload (KV write + decode of all 256 sequences)."""
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    seed = wl.SEED_BASE + 2
    ctx = wl.rng(seed + 7).integers(100, 1024, size=256, endpoint=True).astype(np.int32)
    layout = wl.make_layout(seed, ctx, 256)
    kc, vc = wl.make_pool(layout, ctx - 1, seed + 1000, device="cpu")
    kc0, vc0 = wl.bf16_bits(kc).copy(), wl.bf16_bits(vc).copy()
    toks = wl.new_tokens(seed + 1001, 256, device="cpu")
    slots = np.array([layout.slots(b, [c - 1])[0] for b, c in enumerate(ctx)], np.int32)
    k, v, q = (wl.bf16_bits(t) for t in (toks.k, toks.v, toks.q))

    def one():
        a, b = kc0.copy(), vc0.copy()
        oracle.store_kvcache(k, v, a, b, slots)
        oracle.decode(q, a, b, layout.block_tables, ctx, wl.SCALE)

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    el = time.perf_counter() - t0
    nbytes = args.steps * (decode_bytes(ctx, 256) + store_bytes(256))
    val = nbytes / el / 1e9
    cores = oracle.num_threads()
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "decode batch, one layer per step: 256 seqs, context_lens U[100,1024], "
                                   "block_size 256, 16q/8kv x 128, KV write + paged decode"},
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": f"{args.steps} layer(s) of the decode-batch step on the host cores"},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------- main


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extras", action="store_true", help="skip the prefill / long-decode / CPU legs")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--layers", type=int, default=LAYERS, help="layers per step (28 for the headline number)")
    ap.add_argument("--leg", default="all",
                    choices=["all", "prefill", "long_decode", "rope_store", "metadata", "mixed", "fp8", "gqa",
                             "block_sizes", "decode_layer"],
                    help="run one secondary leg alone (profiling); prints that leg's results only")
    ap.add_argument("--long-seqs", type=int, default=512,
                    help="sequences of the long-decode legs run alone (--leg long_decode / fp8); fewer give the "
                         "small case of the same shape for a profiler capture")
    ap.add_argument("--prefill-case", default="all",
                    choices=["all", "varlen_16k", "prefix_2048_chunked", "chunk_512_over_8k"])
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    rank, world, local = dist_init()
    if args.impl == "reference":
        return reference_arm(args, rank, world)

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    device = torch.device("cuda", local)
    peaks, peak_kind = measured_peaks()
    if args.leg != "all":
        flush = torch.zeros(512 << 20, dtype=torch.uint8, device=device)
        if args.leg == "prefill":
            res = time_prefill(device, max(args.steps, 1), args.warmup, flush, args.prefill_case)
        elif args.leg == "fp8":
            res = time_long_decode_fp8(device, max(args.steps, 1), args.warmup, flush, seqs=args.long_seqs)
            res["frac"] = res["gbs"] / peaks["hbm_gbs"]
        elif args.leg == "block_sizes":
            res = time_block_size_sweep(device, max(args.steps, 1), args.warmup, flush)
        elif args.leg == "gqa":
            res = time_gqa_decode(device, max(args.steps, 1), args.warmup, flush, peaks["hbm_gbs"])
        elif args.leg == "mixed":
            res = time_mixed(device, max(args.steps, 1), args.warmup, flush)
        elif args.leg == "decode_layer":
            res = time_decode_layer_step(device, max(args.steps, 1), args.warmup)
        elif args.leg == "metadata":
            res = time_step_metadata(device, max(args.steps, 1), args.warmup)
        elif args.leg == "rope_store":
            res = time_rope_store(device, max(args.steps, 1), args.warmup, flush)
            for v in res.values():
                v["frac"] = v["gbs"] / peaks["hbm_gbs"]
        else:
            res = time_long_decode(device, max(args.steps, 1), args.warmup, flush, seqs=args.long_seqs)
        if rank == 0:
            print(json.dumps({"leg": args.leg, "results": res}), flush=True)
        return 0

    step = DecodeStep(device, seed=wl.SEED_BASE + 2 + 10000 * rank, layers=args.layers,
                      keep_host_layer0=(rank == 0))
    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()

    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0]) if \
        os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0].isdigit() else local
    # the step captured once in a CUDA graph (how a serving engine runs decode):
    # same buffers, same kernels, no per-launch host work
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph):
            step.run()
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()

    # for comparison: the same step with the KV write as its own launch before
    # each decode (pa_store_kvcache + pa_decode_paged), also graph-captured
    step.fused = False
    graph_unfused = torch.cuda.CUDAGraph()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph_unfused):
            step.run()
    torch.cuda.current_stream().wait_stream(side)
    step.fused = True
    for _ in range(args.warmup):
        graph_unfused.replay()
    torch.cuda.synchronize()

    events = []
    with ClockSampler(gpu_index) as clocks:
        clocks.wait_first()
        h0 = time.time()
        # headline: the graph replayed K times
        g_el = time_region(graph.replay, args.steps, world)
        # beside it: the same kernels launched one by one, with CUDA events
        # around every decode call for the roofline
        elapsed = time_region(lambda: step.run(events), args.steps, world)
        unfused_el = time_region(graph_unfused.replay, args.steps, world)
        h1 = time.time()
        time.sleep(0.3)
    del graph, graph_unfused
    t_max, bytes_all = reduce_max_sum(world, g_el, float(step.step_bytes * args.steps))
    value = bytes_all / t_max / 1e9
    eager_t, eager_bytes = reduce_max_sum(world, elapsed, float(step.step_bytes * args.steps))
    eager_value = eager_bytes / eager_t / 1e9
    unfused_t, unfused_bytes = reduce_max_sum(world, unfused_el, float(step.step_bytes * args.steps))
    # the fused call's time inside the graph the headline replays: the step is
    # exactly `layers` such calls, so the per-call time is the step time / layers
    decode_s = t_max / args.steps / step.layers
    achieved = step.call_bytes / decode_s / 1e9
    eager_call_s = sum(s.elapsed_time(e) for s, e in events) / 1e3 / len(events)

    e2e = E2EStep(step)
    for _ in range(2):
        e2e.run()
    e2e_eager_el = time_region(e2e.run, args.steps, world)
    e2e_eager_t, _ = reduce_max_sum(world, e2e_eager_el, float(step.step_bytes * args.steps))
    e2e_graph = E2EGraphStep(e2e)
    for _ in range(2):
        e2e_graph.run()
    e2e_el = time_region(e2e_graph.run, args.steps, world)
    e2e_t, e2e_bytes = reduce_max_sum(world, e2e_el, float(step.step_bytes * args.steps))
    del e2e_graph

    src = os.path.join(ROOT, "paged_kv_cache_110_gb300", "csrc", "decode_paged.cu")
    traffic = NCU_TRAFFIC["bytes_per_call"] if NCU_TRAFFIC["code_sha256"] == _code_sha(src) else None
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_max / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "decode batch x 28 layers: 256 seqs, context_lens U[100,1024], block_size 256, "
                               "16q/8kv x 128 bf16; per layer KV write of 256 tokens + paged decode "
                               "(one pa_store_decode_paged call)",
                   "layers": step.layers, "seqs": step.B, "sum_context": int(step.ctx.sum()),
                   "l2": "inputs larger than L2: 28 distinct layer pools (%.1f GB)" %
                         (step.layers * 2 * step.layout.num_blocks * 256 * ROW_BYTES / 1e9),
                   "parallelism": f"replicas x{world}"},
        "tokens_per_s": world * step.B * args.steps / t_max,
        "hbm_frac_of_8tbs": value / 8000.0,
        "gpu_launches": args.steps * step.launches_per_step(),
        "timing": "the 28-layer step captured once in a CUDA graph and replayed K times (how a serving engine "
                  "runs decode); the same kernels launched one by one from Python are reported under 'eager'",
        "eager": {"value": eager_value, "unit": "GB/s", "ms_per_step": eager_t / args.steps * 1e3},
        "unfused": {"value": unfused_bytes / unfused_t / 1e9, "unit": "GB/s",
                    "ms_per_step": unfused_t / args.steps * 1e3,
                    "how": "the same step, graph-captured, with pa_store_kvcache and pa_decode_paged per layer"},
        "e2e": {"value": e2e_bytes / e2e_t / 1e9, "unit": "GB/s", "h2d_bytes_per_step": e2e.h2d,
                "d2h_bytes_per_step": e2e.d2h, "ms_per_step": e2e_t / args.steps * 1e3,
                "how": "C-ABI calls of the step with pinned-host copies in and out, captured in a CUDA graph with "
                       "the copies on their own streams; every copy is inside each replay",
                "eager_ms_per_step": e2e_eager_t / args.steps * 1e3},
        "roofline": {"bound": "hbm", "kernel": "pa_store_decode_paged (split-KV kernel with the KV write, merge)",
                     "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "peak_kind": peak_kind,
                     "traffic": traffic, "traffic_kernel": NCU_TRAFFIC["kernel"],
                     "algorithmic_bytes_per_call": step.call_bytes,
                     "us_per_call": decode_s * 1e6,
                     "timing": "per call inside the replayed graph: step time / layers (each layer is one call)",
                     "eager_us_per_call": eager_call_s * 1e6},
        "clocks": clocks.summary(h0, h1 + 0.25),
    }
    if rank == 0 and not args.no_extras:
        flush = torch.zeros(512 << 20, dtype=torch.uint8, device=device)
        host0 = step.host_layer0
        meta = (step.ctx, step.layout.block_tables, step.slots_np, step.tokens[0])
        del step, e2e
        torch.cuda.empty_cache()
        pre = time_prefill(device, max(args.steps, 5), 3, flush)
        for v in pre.values():
            v["frac_of_bf16_peak"] = v["tflops"] / peaks["bf16_tflops"]
            v["tokens_per_s"] = v["query_tokens"] / (v["ms"] / 1e3)
        line["prefill"] = pre
        vp = pre["varlen_16k"]
        line["roofline_prefill"] = {
            "bound": "tensor", "kernel": "prefill_tc_kernel (varlen prefill, 16,384-token budget)",
            "achieved": vp["tflops"], "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": vp["tflops"] / peaks["bf16_tflops"], "peak_kind": f"{peak_kind} bf16 dense (burst)",
            "algorithmic_flops_per_call": vp["gflop"] * 1e9, "us_per_call": vp["ms"] * 1e3,
            "counted": "4 * 128 * 16 FLOP per visible (query, key) pair; masked pairs and padding not counted",
            "traffic": NCU_TRAFFIC_PREFILL["bytes_per_call"] if NCU_TRAFFIC_PREFILL["code_sha256"] == _code_sha(
                os.path.join(ROOT, "paged_kv_cache_110_gb300", "csrc", "prefill_paged.cu")) else None,
            "traffic_unit": "bytes per call (DRAM read + write, ncu)"}
        torch.cuda.empty_cache()
        line["block_sizes"] = time_block_size_sweep(device, 5, 2, flush)
        torch.cuda.empty_cache()
        line["gqa_decode"] = time_gqa_decode(device, 10, 3, flush, peaks["hbm_gbs"])
        torch.cuda.empty_cache()
        ld = time_long_decode(device, max(args.steps, 5), 3, flush)
        ld["frac"] = ld["gbs"] / peaks["hbm_gbs"]
        line["long_decode"] = ld
        torch.cuda.empty_cache()
        rs = time_rope_store(device, max(args.steps, 5), 3, flush)
        for v in rs.values():
            v["frac"] = v["gbs"] / peaks["hbm_gbs"]
        line["norm_rope_store"] = rs
        line["step_metadata"] = time_step_metadata(device, max(args.steps, 5), 3)
        torch.cuda.empty_cache()
        line["decode_layer_step"] = time_decode_layer_step(device, 50, 3)
        torch.cuda.empty_cache()
        line["mixed_step"] = time_mixed(device, max(args.steps, 5), 3, flush)
        torch.cuda.empty_cache()
        l8 = time_long_decode_fp8(device, max(args.steps, 5), 3, flush)
        l8["frac"] = l8["gbs"] / peaks["hbm_gbs"]
        line["long_decode_fp8"] = l8
        import oracle
        oracle.build()
        line["cpu_baseline"] = oracle_sample(host0, meta, target_s=args.cpu_seconds)
        # the same oracle on one core, a shorter sample
        all_cores = oracle.num_threads()
        oracle.set_num_threads(1)
        one = oracle_sample(host0, meta, target_s=min(5.0, args.cpu_seconds), max_layers=8)
        oracle.set_num_threads(all_cores)
        line["cpu_baseline"]["one_core"] = {"value": one["value"], "unit": one["unit"], "cores": 1,
                                            "sample": one["sample"]}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
