"""Benchmark of the paged GQA attention hot path on GB300.

One step = RoPE-and-append of the batch's new tokens into the block arena,
then paged attention of those tokens over the arena (the whole hot path of
pages "Building Kshipra" part 3, sections 1 and 4), on the Llama-3-8B-shaped
decode batch (64 sequences, contexts 512-4096, 32 q / 8 kv heads, head dim
128, fp16, block size 16) unless --workload says otherwise.

metric: decode KV-read GB/s = algorithmic KV bytes (keys and values of every
context token, each read once) / step time.  A secondary object measures the
chunked-prefill workload in TFLOP/s (4 x head_dim x q heads x visible
(query, key) pairs per call).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {kshipra,reference}]
Multi-GPU runs (torchrun) run one independent replica per GPU.
"""

from __future__ import annotations

import argparse
import csv
import io
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

MEASURED_PEAKS = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    try:
        with open(MEASURED_PEAKS) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ work sizes

def decode_kv_bytes(w, seqs=None) -> int:
    """Keys and values of every context token of the chosen sequences."""
    ctx = w.context_lens.astype(np.int64)
    if seqs is not None:
        ctx = ctx[seqs]
    return int(ctx.sum()) * w.num_kv_heads * w.head_dim * 2 * 2


def visible_pairs(w) -> int:
    """Causal (query, key) pairs: a query at position p sees keys 0..p."""
    return int((w.positions.astype(np.int64) + 1).sum())


def attention_flops(w) -> float:
    return 4.0 * w.head_dim * w.num_q_heads * visible_pairs(w)


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples every 200 ms while running (SM clock, reasons)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.text = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.text, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.text, _ = self.proc.communicate()
        return False

    def summary(self):
        rows = list(csv.reader(io.StringIO(self.text)))
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ GPU arm

def _events(torch, n):
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def time_loop(torch, fn, steps, warmup, stream):
    """Milliseconds of `steps` back-to-back calls of fn on `stream`, bracketed
    by one pair of CUDA events (no event between the calls, so consecutive
    kernels may overlap their launch as they would in a serving loop)."""
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            fn()
    torch.cuda.synchronize()
    t0, t1 = _events(torch, 2)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for _ in range(steps):
            fn()
        t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1)


def time_steps(torch, dw, steps, warmup, stream, flush=None, fused=False):
    """Times `steps` whole steps on `stream`: append + attention as two calls,
    or (fused) one kshipra_decode_step call.

    Returns (total_ms, per-step append ms list, per-step attention ms list);
    for a fused step the append list is empty and the attention list holds
    the whole call.  Events bracket each call on the launching stream.  When
    `flush` is given (a byte buffer larger than L2), it is overwritten between
    steps, outside the timed windows.
    """
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            dw.decode_step(stream=stream) if fused else dw.step(stream=stream)
    torch.cuda.synchronize()
    if fused:
        ev = _events(torch, 2 * steps)
        with torch.cuda.stream(stream):
            for i in range(steps):
                if flush is not None:
                    flush.fill_(i & 0xFF)
                ev[2 * i].record(stream)
                dw.decode_step(stream=stream)
                ev[2 * i + 1].record(stream)
        torch.cuda.synchronize()
        att = [ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(steps)]
        total = ev[0].elapsed_time(ev[-1]) if flush is None else sum(att)
        return total, [], att
    ev = _events(torch, 3 * steps)
    t0, t1 = _events(torch, 2)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for i in range(steps):
            if flush is not None:
                flush.fill_(i & 0xFF)
            ev[3 * i].record(stream)
            dw.append_step(stream=stream)
            ev[3 * i + 1].record(stream)
            dw.attention(stream=stream)
            ev[3 * i + 2].record(stream)
        t1.record(stream)
    torch.cuda.synchronize()
    app = [ev[3 * i].elapsed_time(ev[3 * i + 1]) for i in range(steps)]
    att = [ev[3 * i + 1].elapsed_time(ev[3 * i + 2]) for i in range(steps)]
    if flush is None:
        total = t0.elapsed_time(t1)
    else:  # the flushes are not part of the work
        total = sum(ev[3 * i].elapsed_time(ev[3 * i + 2]) for i in range(steps))
    return total, app, att


def time_e2e(torch, dw, steps, stream, fused=False, graph=False):
    """Same step through the public API from pinned host memory: every step
    copies its inputs to the device (all of them packed in one pinned block,
    one copy), runs the step (fused or two calls), copies the output back and
    waits for it.  With graph=True those three are captured once in a CUDA
    graph and each step replays it."""
    names = ("q", "k_new", "v_new", "block_tables", "context_lens", "query_start_loc", "positions")
    offs, sizes, total = {}, {}, 0
    for name in names:
        t = getattr(dw, name)
        sizes[name] = t.numel() * t.element_size()
        offs[name] = total
        total += (sizes[name] + 255) // 256 * 256
    host = torch.empty(total, dtype=torch.uint8, pin_memory=True)
    dev = torch.empty(total, dtype=torch.uint8, device=dw.q.device)
    saved = {}
    for name in names:
        t = getattr(dw, name)
        host[offs[name]:offs[name] + sizes[name]].copy_(t.contiguous().view(torch.uint8).reshape(-1))
        saved[name] = t
        setattr(dw, name, dev[offs[name]:offs[name] + sizes[name]].view(t.dtype).view(t.shape))
    out_host = torch.empty(dw.out.shape, dtype=dw.out.dtype, pin_memory=True)
    h2d = sum(sizes.values())
    d2h = out_host.numel() * out_host.element_size()
    def body(st):
        dev.copy_(host, non_blocking=True)
        dw.decode_step(stream=st) if fused else dw.step(stream=st)
        out_host.copy_(dw.out, non_blocking=True)

    try:
        t0, t1 = _events(torch, 2)
        g = None
        if graph:
            with torch.cuda.stream(stream):
                for _ in range(3):
                    body(stream)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                body(torch.cuda.current_stream())
            torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            t0.record(stream)
            for _ in range(steps):
                if g is not None:
                    g.replay()
                else:
                    body(stream)
                stream.synchronize()  # the caller reads the result every step
            t1.record(stream)
        torch.cuda.synchronize()
    finally:
        for name in names:
            setattr(dw, name, saved[name])
    return t0.elapsed_time(t1), h2d, d2h


def gpu_launches_per_step(w, decode_max_rows=16, fused=False):
    """Kernels one step launches, following the library's host-side choices:
    append; decode unless the lengths rule out a decode-class sequence;
    prefill (head_dim 128: one kernel that plans its own work list when at
    most 128 entries can exist, else a planning kernel first; head_dim 64:
    planning kernel + prefill kernel); a fused decode step of a decode-class
    batch is one launch."""
    G = w.num_q_heads // w.num_kv_heads
    S, T = w.num_seqs, int(w.query_lens.sum())
    max_q = int(w.query_lens.max())
    if fused and max_q * G <= decode_max_rows:
        return 1  # kshipra_decode_step: RoPE-and-append inside the decode kernel
    n = 1  # append (for a fused step with prefill rows: K and V only)
    qd = decode_max_rows // G
    if qd >= 1 and T <= (S - 1) * max_q + qd:
        n += 1  # decode (splits merged in the same kernel)
    if max_q * G > decode_max_rows:
        pair_tokens = 2 * (128 // G)
        max_entries = -(-T // pair_tokens) + S
        n += 1 if (w.head_dim == 128 and max_entries <= 128) else 2
    return n


def measure_blocks(torch, stream, pk):
    """Secondary object: block moves.  Swap-out / swap-in of one sequence's
    blocks (32768 tokens, 8 kv heads, head_dim 128, fp16: 128 MiB of K and V)
    to pinned host memory over the CPU-GPU link, and the copy-on-write copy
    of 1024 blocks inside the arena (HBM, read + write)."""
    import paged_kv_cache_arena_gb300 as K
    nb, hkv, bs, d = 4096, 8, 16, 128
    k = torch.randn((nb, hkv, bs, d), device="cuda", dtype=torch.float16)
    v = torch.randn_like(k)
    seq = torch.randperm(nb, device="cuda")[:2048].to(torch.int32)  # 32768 tokens
    hk = torch.empty((2048, hkv, bs, d), dtype=torch.float16, pin_memory=True)
    hv = torch.empty_like(hk, pin_memory=True)
    nbytes = 2 * hk.numel() * 2

    def timed(fn, reps=10):
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
        torch.cuda.synchronize()
        ev = _events(torch, 2)
        with torch.cuda.stream(stream):
            ev[0].record(stream)
            for _ in range(reps):
                fn()
            ev[1].record(stream)
        torch.cuda.synchronize()
        return ev[0].elapsed_time(ev[1]) / reps

    out_ms = timed(lambda: K.kshipra_blocks_swap_out(hk, hv, k, v, seq, stream=stream))
    in_ms = timed(lambda: K.kshipra_blocks_swap_in(k, v, hk, hv, seq, stream=stream))
    src, dst = seq[:1024].contiguous(), seq[1024:].contiguous()
    copy_ms = timed(lambda: K.kshipra_blocks_copy(k, v, src, dst, stream=stream))
    copy_bytes = 2 * 2 * 1024 * hkv * bs * d * 2  # K and V, read + write
    peak = pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    return {"swap_out": {"bytes": nbytes, "ms": round(out_ms, 4), "gbs": round(nbytes / out_ms / 1e6, 1),
                         "to": "pinned host memory"},
            "swap_in": {"bytes": nbytes, "ms": round(in_ms, 4), "gbs": round(nbytes / in_ms / 1e6, 1),
                        "from": "pinned host memory"},
            "cow_copy": {"blocks": 1024, "ms": round(copy_ms, 4),
                         "roofline": {"bound": "hbm", "achieved": round(copy_bytes / copy_ms / 1e6, 1), "peak": peak,
                                      "unit": "GB/s", "frac": round(copy_bytes / copy_ms / 1e6 / peak, 4)}}}


def measure_prefix_cache():
    """Secondary object: the radix-tree prefix cache on the host.  64 system
    prompts of 512 tokens, each shared by 64 requests with 256 tokens of their
    own (block_size 16: 67,584 cached blocks); times insert (request
    finished), match (a new request: 32 shared blocks, then its own tokens)
    and eviction of every block, leaf by leaf with cascades.  Calls go
    straight to the C ABI with prebuilt arrays."""
    import ctypes
    import random
    import time

    import paged_kv_cache_arena_gb300 as K
    from paged_kv_cache_arena_gb300 import _lib
    lib = _lib.load()
    bs, prompts, per_prompt, own, sys_len = 16, 64, 64, 256, 512
    rnd = random.Random(5)
    nblk = (sys_len + own) // bs
    pool = K.BlockPool(prompts * per_prompt * nblk)
    cache = K.PrefixCache(pool, bs)
    systems = [[rnd.randrange(32000) for _ in range(sys_len)] for _ in range(prompts)]
    arr = lambda xs: (ctypes.c_int32 * len(xs))(*xs)
    reqs = [arr(systems[i % prompts] + [rnd.randrange(32000) for _ in range(own)])
            for i in range(prompts * per_prompt)]
    n = sys_len + own
    blocks = (ctypes.c_int32 * nblk)()
    added = ctypes.c_int(0)
    t_ins = 0.0
    for r in reqs:
        lib.kshipra_block_alloc(pool._h, nblk, blocks)
        t0 = time.perf_counter()
        rc = lib.kshipra_prefix_cache_insert(cache._h, r, n, blocks, nblk, ctypes.byref(added))
        t_ins += time.perf_counter() - t0
        assert rc == 0
        lib.kshipra_block_release(pool._h, blocks, nblk)
    nodes = cache.num_nodes
    probes = [arr(systems[i % prompts] + [rnd.randrange(32000) for _ in range(own)]) for i in range(2000)]
    out, nb, nt = (ctypes.c_int32 * nblk)(), ctypes.c_int(0), ctypes.c_int(0)
    t0 = time.perf_counter()
    for r in probes:
        lib.kshipra_prefix_cache_match(cache._h, r, n, out, nblk, ctypes.byref(nb), ctypes.byref(nt))
        lib.kshipra_block_release(pool._h, out, nb.value)
    t_match = time.perf_counter() - t0
    assert nt.value == sys_len
    freed = ctypes.c_int(0)
    t0 = time.perf_counter()
    total = 0
    while True:
        lib.kshipra_prefix_cache_evict(cache._h, 256, ctypes.byref(freed))
        total += freed.value
        if freed.value < 256:
            break
    t_evict = time.perf_counter() - t0
    assert total == nodes and pool.num_free == pool.num_blocks
    cache.close()
    pool.close()
    return {"nodes": nodes, "block_size": bs, "insert_us": round(t_ins / len(reqs) * 1e6, 2),
            "match_us": round(t_match / len(probes) * 1e6, 2), "tokens_per_request": n,
            "evict_us_per_block": round(t_evict / total * 1e6, 3), "where": "host CPU, through the C ABI"}


def measure_prefill(torch, stream, pk):
    """Secondary object: chunked-prefill attention TFLOP/s (L2 flushed)."""
    from workloads import make_config
    from workloads.device import DeviceWorkload
    w = make_config("chunked-prefill")
    dw = DeviceWorkload(w)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    steps = 50
    total, app, att = time_steps(torch, dw, steps, 5, stream, flush=flush)
    _, _, step = time_steps(torch, dw, steps, 5, stream, flush=flush, fused=True)
    att_ms, step_ms = statistics.mean(att), statistics.mean(step)
    flops = attention_flops(w)
    tflops = flops / (att_ms * 1e-3) / 1e12
    step_tflops = flops / (step_ms * 1e-3) / 1e12
    peak = pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    return {"workload": "chunked-prefill", "metric": "chunked-prefill attention TFLOP/s", "unit": "TFLOP/s",
            "value": round(tflops, 2), "ms_per_call": round(att_ms, 5), "flops_per_call": flops,
            "append_ms_per_call": round(statistics.mean(app), 5),
            "roofline": {"bound": "tensor", "achieved": round(tflops, 2), "peak": peak, "unit": "TFLOP/s",
                         "frac": round(tflops / peak, 4), "traffic": None,
                         "peak_note": "fp16 dense = bf16 dense rate (measured cuBLAS bf16 burst)"},
            "step": {"what": "kshipra_decode_step: K/V append, then the attention kernel rotating q itself "
                             "(started as the append's programmatic dependent)",
                     "ms": round(step_ms, 5), "tflops": round(step_tflops, 2), "frac": round(step_tflops / peak, 4),
                     "two_call_ms": round(statistics.mean(app) + att_ms, 5),
                     "two_call_frac": round(flops / ((statistics.mean(app) + att_ms) * 1e-3) / 1e12 / peak, 4)},
            "l2": "flushed between calls (512 MiB write)"}


def decode_class(w, decode_max_rows=16):
    """Sequences the library sends to the decode kernel (query rows = query
    length x group size at most decode_max_rows); the rest go to prefill."""
    G = w.num_q_heads // w.num_kv_heads
    return np.nonzero(w.query_lens.astype(np.int64) * G <= decode_max_rows)[0]


def measure_workload(torch, stream, pk, name, steps=30):
    """Secondary object for one more config: its attention calls timed back
    to back on the launching stream (the append of its new tokens timed
    beside it, and the whole step through kshipra_decode_step), inputs
    larger than L2.  Decode-class sequences are measured in KV GB/s against
    HBM, prefill-class ones in TFLOP/s against the dense tensor peak; a
    mixed batch runs both kernels in one call, and its fraction is the
    larger of the two ideal times (bytes / HBM peak, flops / tensor peak)
    over the measured call."""
    from workloads import make_config
    from workloads.device import DeviceWorkload
    w = make_config(name)
    dw = DeviceWorkload(w)
    _, app, _ = time_steps(torch, dw, steps, 5, stream)
    # attention calls back to back (inputs larger than L2), one pair of events
    att_ms = time_loop(torch, lambda: dw.attention(stream=stream), steps, 5, stream) / steps
    step_ms = time_loop(torch, lambda: dw.decode_step(stream=stream), steps, 5, stream) / steps
    app_ms = statistics.mean(app)
    dec = decode_class(w)
    pre = np.setdiff1d(np.arange(w.num_seqs), dec)
    kv = decode_kv_bytes(w, dec)
    flops = 0.0
    if len(pre):
        toks = np.concatenate([np.arange(w.query_start_loc[s], w.query_start_loc[s + 1]) for s in pre])
        flops = 4.0 * w.head_dim * w.num_q_heads * float((w.positions[toks].astype(np.int64) + 1).sum())
    bw, tc = pk.get("hbm_gbs"), pk.get("bf16_tflops")
    ideal_ms = max(kv / (bw * 1e9), flops / (tc * 1e12)) * 1e3
    out = {"workload": name, "num_seqs": w.num_seqs, "query_tokens": int(w.num_tokens),
           "dtype": w.dtype, "block_size": w.block_size, "attention_ms_per_call": round(att_ms, 5),
           "append_ms_per_call": round(app_ms, 5), "step_ms": round(step_ms, 5),
           "step": "kshipra_decode_step (one decode launch with the append inside, or a K/V append then "
                   "attention kernels rotating q themselves)",
           "attention": "kshipra_paged_attention (decode kernel; with prefill rows too, head_dim 128, the "
                        "prefill kernel beside it on a side stream)" if flops and len(dec) else
                        "kshipra_paged_attention",
           "tokens_per_s": round(w.num_tokens / (att_ms * 1e-3), 1),
           "decode_seqs": int(len(dec)), "decode_kv_bytes": kv, "prefill_seqs": int(len(pre)),
           "prefill_flops": flops, "l2": "inputs larger than L2 (%.0f MB of KV read per call)" % (kv / 1e6),
           "status": None}
    if flops == 0.0:
        out["roofline"] = {"bound": "hbm", "achieved": round(kv / (att_ms * 1e-3) / 1e9, 1), "peak": bw,
                           "unit": "GB/s", "frac": round(ideal_ms / att_ms, 4), "traffic": None}
    else:
        out["roofline"] = {"bound": "hbm" if kv / (bw * 1e9) >= flops / (tc * 1e12) else "tensor",
                           "achieved_gbs": round(kv / (att_ms * 1e-3) / 1e9, 1),
                           "achieved_tflops": round(flops / (att_ms * 1e-3) / 1e12, 2),
                           "peak_gbs": bw, "peak_tflops": tc, "ideal_ms": round(ideal_ms, 5),
                           "frac": round(ideal_ms / att_ms, 4), "traffic": None,
                           "frac_rule": "max(KV bytes / HBM peak, prefill flops / tensor peak) / call time"}
    del dw
    torch.cuda.empty_cache()
    return out


def workload_config(w, world: int) -> dict:
    """The ``config`` object of the JSON line (the same for both arms)."""
    kv = decode_kv_bytes(w)
    return {"workload": w.name, "num_seqs": w.num_seqs,
            "context_lens": "%d-%d" % (int(w.context_lens.min()), int(w.context_lens.max())),
            "heads": "%dq/%dkv" % (w.num_q_heads, w.num_kv_heads), "head_dim": w.head_dim,
            "block_size": w.block_size, "kv_bytes_per_step": kv,
            "parallelism": "replicas" if world > 1 else "single",
            "l2": "inputs larger than L2 (%.0f MB of KV per step)" % (kv / 1e6)}


# ------------------------------------------------------------------ oracle (CPU)

def oracle_sample(w, budget_s: float = 15.0):
    """Times the float64 oracle on whole sequences of the workload, taking
    sequences in order (starting over after the last) until about
    `budget_s` seconds of CPU work, at least one sequence.  Returns
    (seconds, kv_bytes, flops, sequences timed, threads)."""
    import oracle
    threads = oracle.default_threads()
    qsl = w.query_start_loc
    done, secs, per, nxt = [], 0.0, None, 0
    while secs < budget_s or not done:
        take = 1 if per is None else max(1, min(w.num_seqs, int((budget_s - secs) / max(per, 1e-6))))
        batch = [(nxt + i) % w.num_seqs for i in range(take)]
        nxt = (nxt + take) % w.num_seqs
        toks = np.concatenate([np.arange(qsl[s], qsl[s + 1]) for s in batch]).astype(np.int32)
        t = time.perf_counter()
        oracle.workload_attention(w, tokens=toks, nthreads=threads)
        secs += time.perf_counter() - t
        done += batch
        per = secs / len(done)
        if take == 1 and per is not None and secs >= budget_s:
            break
    kv = decode_kv_bytes(w, np.array(done))
    pairs = int(sum((w.positions[qsl[s]:qsl[s + 1]].astype(np.int64) + 1).sum() for s in done))
    flops = 4.0 * w.head_dim * w.num_q_heads * pairs
    return secs, kv, flops, len(done), threads


REFERENCE_BUDGET_S = 120.0  # seconds of oracle work in a whole reference run


def reference_arm(args, w):
    """The oracle as the reference implementation: each step is a bounded
    sample of the same workload, timed on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    # about REFERENCE_BUDGET_S of oracle work in all, at least one sequence per step
    budget = REFERENCE_BUDGET_S / max(1, args.steps + args.warmup)
    for _ in range(args.warmup):
        oracle_sample(w, budget_s=budget)
    secs = kv = 0.0
    n_seqs = threads = 0
    for _ in range(args.steps):
        s_, kv_, _, n_, threads = oracle_sample(w, budget_s=budget)
        secs += s_
        kv += kv_
        n_seqs = n_
    value = kv / secs / 1e9
    line = {"impl": "reference", "metric": "decode KV-read GB/s", "value": round(value, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, args.gpus),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": "%d sequences per step, taken in order of the %d-sequence workload "
                                       "(all q heads), float64 C oracle" % (n_seqs, w.num_seqs)},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ ranks

def max_over_ranks(torch, dist, x: float, device) -> float:
    """The largest x over all ranks (every rank gets it): the job's timed
    region ends when its slowest replica does."""
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, units_per_rank: float, steps: int, total_ms: float) -> float:
    """Whole-job rate in giga-units per second: every rank processes
    units_per_rank per step (weak scaling), over the max-over-ranks time."""
    return world * units_per_rank * steps / (total_ms * 1e-3) / 1e9


# ------------------------------------------------------------------ main

def gpu_arm(args, w):
    import torch
    import torch.distributed as dist

    import paged_kv_cache_arena_gb300 as K
    from workloads.device import DeviceWorkload

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if world > 1:
            dist.barrier()

    K._lib.load()  # fails loudly when the library is not built
    pk, pk_src = peaks()
    dw = DeviceWorkload(w)
    stream = torch.cuda.Stream()
    kv = decode_kv_bytes(w)
    fused = args.step == "fused"
    try:
        smi_id = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:
        smi_id = str(local)
    barrier()
    torch.cuda.synchronize()
    step_fn = (lambda: dw.decode_step(stream=stream)) if fused else (lambda: dw.step(stream=stream))
    with ClockSampler(smi_id) as clk:
        barrier()
        total_ms = time_loop(torch, step_fn, args.steps, args.warmup, stream)
        barrier()
    clocks = clk.summary()
    own_ms = total_ms
    if world > 1:
        total_ms = max_over_ranks(torch, dist, total_ms, "cuda")
    status = K.kshipra_device_status()
    ms_step = total_ms / args.steps
    value = job_throughput(world, kv, args.steps, total_ms)
    # per-call breakdown (an event around each call), a shorter pass of its own
    _, app, att = time_steps(torch, dw, min(args.steps, 200), 3, stream, fused=fused)
    # the fused step is one launch per step: its average launch duration is
    # the timed loop's time per step; the two-call step's attention call is
    # timed by its own events
    att_ms = own_ms / args.steps if fused else statistics.mean(att)
    achieved = kv / (att_ms * 1e-3) / 1e9
    e2e_steps = min(args.steps, 300)
    e2e_ms, h2d, d2h = time_e2e(torch, dw, e2e_steps, stream, fused=fused)
    e2e_value = world * kv * e2e_steps / (e2e_ms * 1e-3) / 1e9
    e2e_how = "plain launches every step (copy in, step, copy out)"
    e2e_plain = round(e2e_value, 2)
    try:
        g_ms, _, _ = time_e2e(torch, dw, e2e_steps, stream, fused=fused, graph=True)
        e2e_value = world * kv * e2e_steps / (g_ms * 1e-3) / 1e9
        e2e_how = "copy in, step and copy out captured once in a CUDA graph, replayed every step"
        graph_error = None
    except Exception as exc:  # reported; the plain-launch figure stands
        graph_error = str(exc)[:200]
    secondary = None
    blocks = None
    if not args.no_prefill:
        try:
            secondary = measure_prefill(torch, stream, pk)
        except Exception as exc:  # reported, never silently substituted
            secondary = {"workload": "chunked-prefill", "error": str(exc)[:200]}
    workloads = []
    if not args.no_workloads:
        for name in ("mixed", "long-decode"):
            if name == w.name:
                continue
            try:
                r = measure_workload(torch, stream, pk, name)
                r["status"] = K.kshipra_device_status()
            except Exception as exc:  # reported, never silently substituted
                r = {"workload": name, "error": str(exc)[:200]}
            workloads.append(r)
    if rank == 0 and not args.no_blocks:
        try:
            blocks = measure_blocks(torch, stream, pk)
            blocks["prefix_cache"] = measure_prefix_cache()
        except Exception as exc:
            blocks = {"error": str(exc)[:200]}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        secs, kv_s, _, n_s, threads = oracle_sample(w)
        cpu = {"value": round(kv_s / secs / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": "%d sequences (%.1f passes over the %d-sequence workload), all q heads, float64 C "
                         "oracle, %.1f s" % (n_s, n_s / w.num_seqs, w.num_seqs, secs)}
    launches = gpu_launches_per_step(w, fused=fused) * args.steps
    if rank == 0:
        line = {
            "metric": "decode KV-read GB/s", "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f16" if w.dtype == "f16" else "bf16", "data": "synthetic",
            "config": workload_config(w, world),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk.get("hbm_gbs"),
                         "unit": "GB/s", "frac": round(achieved / pk.get("hbm_gbs"), 4),
                         "traffic": None,
                         "traffic_note": "DRAM bytes per launch come from an ncu capture of this kernel, not from "
                                         "this run",
                         "kernel": ("decode step (decode_kernel with RoPE-and-append and split combine inside)"
                                    if fused else "paged attention call (decode_kernel, split combine inside)"),
                         "ms_per_launch": round(att_ms, 5), "peak_source": pk_src},
            "append_ms_per_step": round(statistics.mean(app), 5) if app else 0.0,
            "step": "one kshipra_decode_step launch" if fused else "kshipra_kv_append_rope + kshipra_paged_attention",
            "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "inputs": "packed in one pinned block, one host-to-device copy per step",
                    "how": e2e_how, "plain_launches_value": e2e_plain, "graph_error": graph_error},
            "gpu_launches": launches, "clocks": clocks, "device_status": status,
            "cpu_baseline": cpu, "secondary": secondary, "workloads": workloads, "blocks": blocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["kshipra", "reference"], default="kshipra")
    ap.add_argument("--workload", default="llama-decode", choices=["llama-decode", "long-decode", "mixed"])
    ap.add_argument("--no-prefill", action="store_true", help="skip the chunked-prefill secondary object")
    ap.add_argument("--step", choices=["fused", "two-call"], default="fused",
                    help="a decode step as one kshipra_decode_step launch or as append + attention calls")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-blocks", action="store_true", help="skip the block-move secondary object")
    ap.add_argument("--no-workloads", action="store_true", help="skip the mixed and long-decode objects")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    from workloads import make_config
    w = make_config(args.workload)
    if args.impl == "reference":
        reference_arm(args, w)
    else:
        gpu_arm(args, w)


if __name__ == "__main__":
    main()
