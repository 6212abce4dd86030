"""Benchmark of the int4 KIVI paged cache hot path on GB300.

One step = one decode step of every layer of the workload: for each layer, the
append of one new token per sequence (quantize-on-write + residual flush) and
decode attention of one query per sequence over the quantized history plus the
residual. Default workload: Qwen2.5-7B-like attention at 32k context (28
layers, batch 64, H_q 28, H_kv 4, head_dim 128, fp16, G 32, R 128, page 16).
The per-layer cache (~1.6 GB) is far larger than L2, and layers rotate, so no
L2 flush is needed between steps.

The fill (2048-token chunk appends of every layer) is timed per call too and
reported as `append_chunk`. The default run then measures the other workloads
on caches of their own (tiny, Qwen2.5-1.5B-like, Llama-3.1-8B-like, and the
mixed serving trace with its 3:1 mix of 2048-token chunk appends and 1-token
appends) and reports them under `configs`.

Prints one JSON line (rank 0). `--impl reference` times the oracle (plain C++
on the host cores) on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import s4kv_inputs as inp  # noqa: E402

METRIC = "int4 paged decode-attn HBM GB/s (% of GB300 peak), KV-tokens/s; append ns/token"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def tensor_peak():
    """Dense bf16 TFLOP/s (burst: the attention call is timed alone); the f16
    mma.sync path of the kernels is measured against the same dense rate."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return float(json.load(open(p))["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


# ------------------------------------------------------------- byte counts --
def decode_bytes(lens, H, Hq, R, G=32, P=16, e=2, nq=1, bits=4):
    """Algorithmic bytes of one attention call: packed codes + fp32 metadata of
    the quantized history, residual rows, q, fp32 output, block table, lengths
    (nq query rows and output rows per sequence for a multi-query call)."""
    tot = 0
    for T in lens:
        if bits == 8:   # FP8 pages: one byte per key and value element, a key and a value scale
            tot += H * (T * 256 + 8)
        else:
            Tk = G * (T // G)
            Tv = max(0, T - R)
            rk, rv = T - Tk, T - Tv
            tot += H * (Tk * 16 * bits + (Tk // G) * 1024 + Tv * (16 * bits + 32) + (rk + rv) * 128 * e)
        tot += nq * (Hq * 128 * e + Hq * 128 * 4) + 4 * ((T + P - 1) // P) + 4
    return tot


def attention_flops(lens, Hq, nq=1):
    """2 * 128 multiply-adds for q.k and 2 * 128 for p.v per visible (token,
    query row); query i of a chunk of nq sees T - nq + i + 1 tokens."""
    return sum(Hq * 4 * 128 * sum(T - nq + i + 1 for i in range(nq)) for T in lens)


def append_bytes(lens_before, H, R, G=32, e=2, n=1, bits=4):
    """Algorithmic bytes of appending n tokens per sequence, one at a time in
    effect (a decode step appends one)."""
    tot = 0
    for T0 in lens_before:
        per = 0
        if bits == 8:   # FP8: read the rows and scales, write 128 + 128 code bytes, the length
            tot += H * (n * (2 * 128 * e + 256) + 8 + 8) + 3 * 4 + 4
            continue
        for T1 in range(T0 + 1, T0 + n + 1):
            per += 2 * 128 * e            # read the new k and v rows
            per += 2 * 128 * e            # write them into the rings
            if T1 % G == 0:               # key group complete: read 31 ring rows, write codes + 1 KiB
                per += (G - 1) * 128 * e + G * 16 * bits + 1024
            if T1 > R:                    # oldest value leaves the window: read its row, write codes + 32 B
                per += 128 * e + 16 * bits + 32
        tot += H * per + 3 * 4 + 4        # + cu_new, seq_lens_before, block-table entry
    return tot


def chunk_append_bytes(lens_before, news, H, R, G=32, e=2, bits=4):
    """Algorithmic bytes of one append call that adds news[i] tokens to sequence
    i at once (a chunk): read the new k and v rows, the key-ring rows of a key
    group that mixes old and new tokens and the value-ring rows of tokens that
    leave the window; write codes + metadata of every key group completed and
    every value token quantized, and the rows left in the rings."""
    tot = 0
    for T0, n in zip(lens_before, news):
        if n <= 0:
            continue
        T1 = T0 + n
        if bits == 8:
            tot += H * (n * (2 * 128 * e + 256) + 8 + 8) + 3 * 4 + 4
            continue
        Tk0, Tk1 = G * (T0 // G), G * (T1 // G)
        Tv0, Tv1 = max(0, T0 - R), max(0, T1 - R)
        rd = n * 2 * 128 * e
        if Tk0 < T0 and Tk0 + G <= T1:
            rd += (T0 - Tk0) * 128 * e
        rd += max(0, min(T0, Tv1) - Tv0) * 128 * e
        wr = (Tk1 - Tk0) * (16 * bits + 32) + (Tv1 - Tv0) * (16 * bits + 32)
        wr += (T1 - max(Tk1, T0)) * 128 * e + (T1 - max(T0, Tv1)) * 128 * e
        tot += H * (rd + wr) + 3 * 4 + 4
    return tot


# ------------------------------------------------------------------ clocks --
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            t0 = time.time()
            while not self.lines and time.time() - t0 < 5.0:   # sampler up before timing
                time.sleep(0.01)
            self.skip = len(self.lines)
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lines = self.lines[getattr(self, "skip", 0):] or self.lines[-1:]
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = max(mx, float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------ multi-rank --
def combine_ranks(values):
    """Max over ranks of per-rank timings (the slowest rank sets the job time).

    Runs on whatever process group is initialised: NCCL on the GPU ranks of a
    torchrun launch, gloo in the CPU tests."""
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor(list(values), dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.cpu().tolist()


# --------------------------------------------------------------- our arm --
def fill_cache(cache, w, L, lens0, bt, dev, seed, g, bits=4, chunk=2048):
    """Appends every sequence's first lens0[b] tokens to every layer in ragged
    calls of up to `chunk` tokens per sequence. Returns per-call (start event,
    end event, algorithmic bytes, new tokens)."""
    import numpy as np
    import torch
    B, H, R = len(lens0), w.num_kv_heads, w.residual_v
    tdt = w.torch_dtype
    ev = []
    for layer in range(L):
        outl = inp.outlier_channels(seed, layer, H, 128, w.k_outliers).to(dev)
        scale = torch.ones(H, 128, device=dev)
        for h in range(H):
            scale[h, outl[h]] = w.k_outlier_factor
        done = [0] * B
        while any(d < T for d, T in zip(done, lens0)):
            news = [min(chunk, T - d) for d, T in zip(done, lens0)]
            n = sum(news)
            k = (torch.randn((n, H, 128), generator=g, device=dev) * scale).to(tdt)
            v = torch.randn((n, H, 128), generator=g, device=dev).to(tdt)
            cu = torch.tensor([0] + list(np.cumsum(news)), dtype=torch.int32, device=dev)
            before = torch.tensor(done, dtype=torch.int32, device=dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            cache.append(layer, k, v, cu, before, bt)
            e1.record()
            ev.append((e0, e1, chunk_append_bytes(done, news, H, R, bits=bits), n))
            done = [d + x for d, x in zip(done, news)]
    return ev


def chunk_summary(ev):
    """Totals of timed append calls: GB/s of algorithmic bytes, ns per new token."""
    if not ev:
        return None
    ms = sum(a.elapsed_time(b) for a, b, _, _ in ev)
    byt = sum(x for _, _, x, _ in ev)
    tok = sum(n for _, _, _, n in ev)
    return {"calls": len(ev), "ms": ms, "bytes": byt, "tokens": tok,
            "gbs": byt / (ms * 1e-3) / 1e9, "ns_per_token": ms * 1e6 / tok}



def run_ours(args, rank, world):
    import numpy as np
    import torch

    import int4_kivi_quantized_gb300 as s4

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    w = inp.WORKLOADS[args.workload]
    L = args.layers or w.layers
    B, H, Hq, R = w.batch, w.num_kv_heads, w.num_q_heads, w.residual_v
    seed = 1234 + rank
    nq = args.queries
    lens0 = inp.context_lengths(w, seed).tolist()
    total_steps = args.warmup + 3 * args.steps + 1   # warm-up, timed, end-to-end and fused steps
    cap = [(T + total_steps * nq + 15) // 16 for T in lens0]
    num_pages = sum(cap)
    bt = inp.block_tables("permuted" if w.table == "identity" else w.table, B, cap, num_pages,
                          seed).to(dev)
    cache = s4.KVCache(L, num_pages, H, R, B, w.dtype, device=dev, bits=args.bits)
    if args.impl_variant is not None:
        cache.set_option(s4.S4KV_OPT_DECODE_IMPL, args.impl_variant)
    if args.tail_cost:
        cache.set_option(s4.S4KV_OPT_TAIL_COST, args.tail_cost)
    if args.key_split:
        cache.set_option(s4.S4KV_OPT_KEY_SPLIT, 1)
    if getattr(args, "mq_kernel", 0):
        cache.set_option(s4.S4KV_OPT_MQ_KERNEL, args.mq_kernel)
    tdt = w.torch_dtype

    # fill: prefill chunks of up to 2048 tokens per sequence, every layer; each
    # append call is timed (CUDA events around the call only)
    t_fill = time.time()
    g = inp.gen(seed, dev)
    chunk_ev = fill_cache(cache, w, L, lens0, bt, dev, seed, g, bits=args.bits)
    torch.cuda.synchronize()
    rc, detail = cache.status()
    if rc:
        raise RuntimeError(f"fill failed: {s4.s4kv_strerror(rc)} detail {detail}")
    t_fill = time.time() - t_fill
    chunk_stats = chunk_summary(chunk_ev)

    # per-step inputs (new k/v rows and queries of every layer), resident in HBM
    knew = (torch.randn((L, B * nq, H, 128), generator=g, device=dev)).to(tdt)
    vnew = (torch.randn((L, B * nq, H, 128), generator=g, device=dev)).to(tdt)
    qshape = (L, B, Hq, 128) if nq == 1 else (L, B, nq, Hq, 128)
    q = torch.randn(qshape, generator=g, device=dev).to(tdt)
    out = torch.empty(qshape, dtype=torch.float32, device=dev)
    cu1 = torch.arange(B + 1, dtype=torch.int32, device=dev) * nq
    lens = list(lens0)
    # lengths of every step, precomputed: row i = lengths before step i
    lens_tab_host = (torch.arange(total_steps + 1, dtype=torch.int32)[:, None] * nq +
                     torch.tensor(lens0, dtype=torch.int32)[None]).contiguous()
    lens_tab = lens_tab_host.to(dev)
    lens_tab_host = lens_tab_host.pin_memory()
    step_no = 0
    max_len = max(lens0) + total_steps * nq
    if nq == 1:
        ws, ws_bytes = cache.workspace(B, Hq, max_len)
    else:
        ws_bytes = s4.s4kv_multi_query_workspace_bytes(cache.h, B, nq, Hq, max_len)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    ev_dec = []
    ev_app = []

    def attend(layer, qq, lens_after, o):
        if nq == 1:
            s4.s4kv_decode_attention(cache.h, layer, qq, Hq, bt, bt.shape[1], lens_after, None, B,
                                     0.0, o, s4.S4KV_F32, ws, ws_bytes, max_len, stream)
        else:
            s4.s4kv_multi_query_attention(cache.h, layer, qq, nq, Hq, bt, bt.shape[1], lens_after, None,
                                          B, 0.0, o, s4.S4KV_F32, ws, ws_bytes, max_len, stream)

    def step(record=False):
        nonlocal step_no
        before = lens_tab[step_no]
        after = lens_tab[step_no + 1]
        for layer in range(L):
            if record:
                e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
                e0.record(stream)
            s4.s4kv_append(cache.h, layer, knew[layer], vnew[layer], B * nq, cu1, None, before, bt,
                           bt.shape[1], B, stream)
            if record:
                e1.record(stream)
            attend(layer, q[layer], after, out[layer])
            if record:
                e2.record(stream)
                ev_app.append((e0, e1))
                ev_dec.append((e1, e2))
        step_no += 1

    for _ in range(args.warmup):
        step()
        lens = [x + nq for x in lens]
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    lens_timed = list(lens)
    clock = ClockSampler(dev.index)
    clock.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(args.steps):
        step(record=True)
        lens = [x + nq for x in lens]
    t1.record(stream)
    torch.cuda.synchronize()
    clocks = clock.stop()
    if world > 1:
        torch.distributed.barrier()
    ms = t0.elapsed_time(t1) / args.steps
    dec_ms = [a.elapsed_time(b) for a, b in ev_dec]
    app_ms = [a.elapsed_time(b) for a, b in ev_app]
    rc, detail = cache.status()
    if rc:
        raise RuntimeError(f"timed steps failed: {s4.s4kv_strerror(rc)} detail {detail}")

    # bytes per step (the lengths grow by one each step)
    dec_b = app_b = 0
    kv_tokens = flops = 0
    for s in range(args.steps):
        before = [x + s * nq for x in lens_timed]
        after = [x + nq for x in before]
        dec_b += L * decode_bytes(after, H, Hq, R, nq=nq, bits=args.bits)
        app_b += L * append_bytes(before, H, R, n=nq, bits=args.bits)
        kv_tokens += L * sum(after)
        flops += L * attention_flops(after, Hq, nq)
    dec_b /= args.steps
    app_b /= args.steps
    kv_tokens /= args.steps
    flops /= args.steps

    # end to end through the C ABI with host buffers: H2D of the step's new
    # k/v rows, queries and lengths, D2H of every layer's output
    hk = knew.cpu().pin_memory()
    hv = vnew.cpu().pin_memory()
    hq = q.cpu().pin_memory()
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    dk, dv, dq = torch.empty_like(knew), torch.empty_like(vnew), torch.empty_like(q)
    e2e_t0 = torch.cuda.Event(enable_timing=True)
    e2e_t1 = torch.cuda.Event(enable_timing=True)
    dlens = torch.empty((2, B), dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    e2e_t0.record(stream)
    for s in range(args.steps):
        dk.copy_(hk, non_blocking=True)
        dv.copy_(hv, non_blocking=True)
        dq.copy_(hq, non_blocking=True)
        dlens.copy_(lens_tab_host[step_no:step_no + 2], non_blocking=True)
        step_no += 1
        before = dlens[0]
        after = dlens[1]
        for layer in range(L):
            s4.s4kv_append(cache.h, layer, dk[layer], dv[layer], B * nq, cu1, None, before, bt,
                           bt.shape[1], B, stream)
            attend(layer, dq[layer], after, out[layer])
        hout.copy_(out, non_blocking=True)
    e2e_t1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e2e_t0.elapsed_time(e2e_t1) / args.steps
    rc, detail = cache.status()
    if rc:
        raise RuntimeError(f"e2e steps failed: {s4.s4kv_strerror(rc)} detail {detail}")
    h2d = (knew.numel() + vnew.numel() + q.numel()) * 2 + 2 * B * 4
    d2h = out.numel() * 4

    # the same decode steps through s4kv_decode_step: the append and the
    # attention of a layer in one launch (plus the small combine launch)
    fused_ms = None
    if nq == 1:
        torch.cuda.synchronize()
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for s in range(args.steps):
            after = lens_tab[step_no + 1]
            for layer in range(L):
                s4.s4kv_decode_step(cache.h, layer, knew[layer], vnew[layer], q[layer], Hq, bt, bt.shape[1],
                                    after, None, B, 0.0, out[layer], s4.S4KV_F32, ws, ws_bytes, max_len, stream)
            step_no += 1
        f1.record(stream)
        torch.cuda.synchronize()
        fused_ms = f0.elapsed_time(f1) / args.steps
        rc, detail = cache.status()
        if rc:
            raise RuntimeError(f"fused steps failed: {s4.s4kv_strerror(rc)} detail {detail}")

    stats = dict(ms=ms, e2e_ms=e2e_ms, dec_ms=statistics.mean(dec_ms), app_ms=statistics.mean(app_ms),
                 dec_b=dec_b, app_b=app_b, kv_tokens=kv_tokens, flops=flops, nq=nq, h2d=h2d, d2h=d2h,
                 clocks=clocks, chunk=chunk_stats, fused_ms=fused_ms,
                 fill_s=t_fill, L=L, B=B, lens=lens_timed, ws_bytes=ws_bytes)
    if world > 1:
        stats["ms"], stats["e2e_ms"], stats["dec_ms"], stats["app_ms"] = combine_ranks(
            [ms, e2e_ms, stats["dec_ms"], stats["app_ms"]])
    cache.close()
    return stats


CONFIG_RUNS = {
    # workload: (layers run, timed steps, why that many layers)
    "tiny": (1, 20, "the workload's 1 layer; L2 flushed before every call"),
    "qwen2.5-1.5b": (1, 20, "the workload's 1 layer; L2 flushed before every call"),
    "llama3.1-8b": (4, 64, "4 copies of the workload's layer called in turn, so no call finds its pages in L2"),
    "mixed-trace": (2, 8, "2 of the 32 layers (every layer call is alike; each layer's cache exceeds L2)"),
}


def run_config(name, dev, bits=4, warmup=3, seed=4321):
    """One workload on its own cache: fill by 2048-token chunks,
    then timed steps; every layer call is timed with CUDA events around the
    append and around the decode call. The mixed trace draws, per step and
    slot, a 2048-token chunk append or a 1-token decode append at 3:1 (seeded);
    every slot then gets one decode query over its whole context."""
    import numpy as np
    import torch
    import int4_kivi_quantized_gb300 as s4

    w = inp.WORKLOADS[name]
    L, steps, why = CONFIG_RUNS[name]
    B, H, Hq, R = w.batch, w.num_kv_heads, w.num_q_heads, w.residual_v
    lens0 = inp.context_lengths(w, seed).tolist()
    total = warmup + steps
    rng = np.random.default_rng(seed)
    if w.chunk:
        a_, d_ = w.chunk_ratio
        news_tab = np.where(rng.random((total, B)) < a_ / (a_ + d_), w.chunk, 1)
    else:
        news_tab = np.ones((total, B), dtype=np.int64)
    grow = news_tab.sum(axis=0)
    cap = [(T + int(grow[b]) + 15) // 16 for b, T in enumerate(lens0)]
    num_pages = B * max(cap) if w.table == "identity" else sum(cap)
    bt = inp.block_tables(w.table, B, cap, num_pages, seed).to(dev)
    cache = s4.KVCache(L, num_pages, H, R, B, w.dtype, device=dev, bits=bits)
    g = inp.gen(seed, dev)
    fill_ev = fill_cache(cache, w, L, lens0, bt, dev, seed, g, bits=bits)
    max_len = max(T + int(grow[b]) for b, T in enumerate(lens0))
    ws, ws_bytes = cache.workspace(B, Hq, max_len)
    tdt = w.torch_dtype
    scales = []
    for layer in range(L):
        outl = inp.outlier_channels(seed, layer, H, 128, w.k_outliers).to(dev)
        sc = torch.ones(H, 128, device=dev)
        for h in range(H):
            sc[h, outl[h]] = w.k_outlier_factor
        scales.append(sc)
    q = torch.randn((L, B, Hq, 128), generator=g, device=dev).to(tdt)
    out = torch.empty((L, B, Hq, 128), dtype=torch.float32, device=dev)
    per_call = decode_bytes(lens0, H, Hq, R, bits=bits)
    flush = None
    if per_call * L < 2 * 129e6:
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    # every step's inputs are made before the timed steps, so that the host only
    # issues the library's calls while they run
    lens = list(lens0)
    steps_in = []
    for st in range(total):
        news = [int(x) for x in news_tab[st]]
        n = sum(news)
        after = [a + b for a, b in zip(lens, news)]
        cu = torch.tensor([0] + list(np.cumsum(news)), dtype=torch.int32, device=dev)
        before_t = torch.tensor(lens, dtype=torch.int32, device=dev)
        after_t = torch.tensor(after, dtype=torch.int32, device=dev)
        kv = [((torch.randn((n, H, 128), generator=g, device=dev) * scales[layer]).to(tdt),
               torch.randn((n, H, 128), generator=g, device=dev).to(tdt)) for layer in range(L)]
        steps_in.append((news, n, list(lens), after, cu, before_t, after_t, kv))
        lens = after
    torch.cuda.synchronize()
    rec = []
    stream = torch.cuda.current_stream()
    for st in range(total):
        news, n, lens, after, cu, before_t, after_t, kv = steps_in[st]
        for layer in range(L):
            k, v = kv[layer]
            if flush is not None:
                flush.fill_(st & 255)
            e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            e0.record(stream)
            s4.s4kv_append(cache.h, layer, k, v, n, cu, None, before_t, bt, bt.shape[1], B, stream)
            e1.record(stream)
            s4.s4kv_decode_attention(cache.h, layer, q[layer], Hq, bt, bt.shape[1], after_t, None, B, 0.0,
                                     out[layer], s4.S4KV_F32, ws, ws_bytes, max_len, stream)
            e2.record(stream)
            if st >= warmup:
                rec.append((e0, e1, e2, chunk_append_bytes(lens, news, H, R, bits=bits),
                            decode_bytes(after, H, Hq, R, bits=bits), n, sum(after), max(news) > 1))
    torch.cuda.synchronize()
    del steps_in
    rc, detail = cache.status()
    cache.close()
    if rc:
        raise RuntimeError(f"{name}: {s4.s4kv_strerror(rc)} detail {detail}")
    hbm, _ = peaks()
    dec_ms = sum(b.elapsed_time(c) for _, b, c, *_ in rec)
    dec_b = sum(r[4] for r in rec)
    kv_tok = sum(r[6] for r in rec)
    res = {
        "workload": f"{w.name}: batch {B}, H_q={Hq}, H_kv={H}, context {ctx_text(w)}, R={R}, "
                    f"{w.table} pages, {w.dtype}, {bits}-bit codes",
        "layers_run": f"{L} ({why})",
        "timed_steps": steps,
        "decode_attn_gbs": round(dec_b / (dec_ms * 1e-3) / 1e9, 1),
        "decode_attn_frac": round(dec_b / (dec_ms * 1e-3) / 1e9 / hbm, 4),
        "decode_us_per_call": round(dec_ms * 1e3 / len(rec), 2),
        "decode_bytes_per_call": int(dec_b / len(rec)),
        "kv_tokens_per_s": round(kv_tok / (dec_ms * 1e-3), 1),
    }
    single = [r for r in rec if not r[7]]
    if single:
        ms = sum(a.elapsed_time(b) for a, b, *_ in single)
        res["append_ns_per_token"] = round(ms * 1e6 / sum(r[5] for r in single), 2)
    mixed = [r for r in rec if r[7]]
    if mixed:
        ms = sum(a.elapsed_time(b) for a, b, *_ in mixed)
        byt = sum(r[3] for r in mixed)
        res["append_mixed_step"] = {
            "what": "one ragged call per layer and step: 2048-token chunks and 1-token appends mixed 3:1",
            "gbs": round(byt / (ms * 1e-3) / 1e9, 1), "frac": round(byt / (ms * 1e-3) / 1e9 / hbm, 4),
            "ns_per_token": round(ms * 1e6 / sum(r[5] for r in mixed), 3),
            "us_per_call": round(ms * 1e3 / len(mixed), 2)}
    cs = chunk_summary(fill_ev)
    if cs:
        res["append_chunk_fill"] = {"gbs": round(cs["gbs"], 1), "frac": round(cs["gbs"] / hbm, 4),
                                    "ns_per_token": round(cs["ns_per_token"], 3), "calls": cs["calls"]}
    return res


def ctx_text(w):
    if w.ctx[0] == "fixed":
        return f"{w.ctx[1]}"
    return f"{w.ctx[0]} [{w.ctx[1]}, {w.ctx[2]}]"


def decode_source_digest(csrc):
    """sha256 prefix of the decode kernel's sources (the kernel file and the
    device helpers it includes)."""
    import hashlib
    h = hashlib.sha256()
    for name in ("s4kv_decode.cu", "s4kv_kernels.cuh", "s4kv_common.cuh"):
        h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(workload, bits=4):
    """DRAM bytes per decode launch from the committed ncu summary of this
    workload and page format, if the summary was taken on the current decode
    source."""
    import hashlib
    csrc = os.path.join(ROOT, "int4_kivi_quantized_gb300", "csrc")
    fmt = {4: "", 2: "_2bit", 8: "_fp8"}[bits]
    summ = os.path.join(ROOT, "profiles", f"decode_kernel_{workload}{fmt}.md")
    if not os.path.exists(summ):
        return None
    digest = decode_source_digest(csrc)
    fields = {}
    for ln in open(summ):
        if ln.startswith("- ") and ":" in ln:
            k, v = ln[2:].split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    if fields.get("decode source sha256 prefix") != digest:
        return None
    try:
        return int(fields["traffic bytes per launch"])
    except (KeyError, ValueError):
        return None


def traffic_source(workload, bits=4):
    """Where roofline.traffic comes from: the committed ncu summary and the
    decode-source hash it was taken on (None when the hash no longer matches)."""
    fmt = {4: "", 2: "_2bit", 8: "_fp8"}[bits]
    name = f"profiles/decode_kernel_{workload}{fmt}.md"
    if profiled_traffic(workload, bits) is None:
        return None
    digest = decode_source_digest(os.path.join(ROOT, "int4_kivi_quantized_gb300", "csrc"))
    return (f"{name}: ncu dram__bytes_read.sum + dram__bytes_write.sum of one decode_kernel launch, "
            f"taken on decode sources with sha256 prefix {digest} (the current ones); not measured in this run")


def append_source_digest(csrc):
    import hashlib
    h = hashlib.sha256()
    for name in ("s4kv_append.cu", "s4kv_common.cuh"):
        h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()[:16]


def profiled_append_traffic(workload, bits=4):
    """DRAM bytes per token of a chunk append from the committed ncu summary of
    the append kernel, if it was taken on the current append source."""
    csrc = os.path.join(ROOT, "int4_kivi_quantized_gb300", "csrc")
    fmt = {4: "", 2: "_2bit", 8: "_fp8"}[bits]
    summ = os.path.join(ROOT, "profiles", f"append_kernel_{workload}_chunk{fmt}.md")
    if not os.path.exists(summ):
        return None
    fields = {}
    for ln in open(summ):
        if ln.startswith("- ") and ":" in ln:
            k, v = ln[2:].split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    if fields.get("append source sha256 prefix") != append_source_digest(csrc):
        return None
    try:
        return {"dram_bytes_per_launch": int(fields["traffic bytes per launch"]),
                "algorithmic_bytes_per_launch": int(fields["algorithmic bytes per launch"]),
                "source": f"profiles/append_kernel_{workload}_chunk{fmt}.md (ncu; not measured in this run)"}
    except (KeyError, ValueError):
        return None


def report_ours(args, stats, world, cpu):
    hbm, peak_kind = peaks()
    w = inp.WORKLOADS[args.workload]
    L = stats["L"]
    step_bytes = stats["dec_b"] + stats["app_b"]
    value = world * step_bytes / (stats["ms"] * 1e-3) / 1e9
    e2e_val = world * step_bytes / (stats["e2e_ms"] * 1e-3) / 1e9
    dec_gbs = (stats["dec_b"] / L) / (stats["dec_ms"] * 1e-3) / 1e9
    nq = stats.get("nq", 1)
    bits = getattr(args, "bits", 4)
    if nq == 1:
        what = "1 new token + 1 query per sequence per layer"
        step_txt = "per layer: append 1 token/sequence + decode attention 1 query/sequence"
        kern_txt = "decode call = decode_kernel + merge_kernel (paged decode attention, one layer call); CUDA events around both"
    else:
        what = f"{nq} new tokens + {nq} causal queries per sequence per layer (multi-query)"
        step_txt = (f"per layer: append {nq} tokens/sequence + causal attention of those {nq} queries "
                    f"(s4kv_multi_query_attention)")
        mk = getattr(args, "mq_kernel", 0)
        cols = nq * w.num_q_heads // w.num_kv_heads
        tc = mk == 3 or (mk == 0 and cols >= 49)
        if bits == 8:
            kname = "mqt_kernel<8> (tcgen05)" if tc else "mq_fp8_kernel"
        elif tc:
            kname = "mqt_kernel (tcgen05)"
        elif mk == 2 or (mk == 0 and cols >= 64):
            kname = "mqd_kernel"
        else:
            kname = "mq_kernel"
        kern_txt = f"multi-query call = {kname} + mq_merge_kernel (one layer call); CUDA events around both"
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(stats["ms"], 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("e4m3 codes + fp32 per-head scales" if bits == 8 else f"u{bits} codes + fp32 meta")
                 + "; f16 tensor-core operands, fp32 accumulate",
        "data": "synthetic (seeded N(0,1) K/V, key outlier channels x16, N(0,1) q)",
        "config": {
            "workload": f"{w.name}: {L} layers, batch {w.batch}, H_q={w.num_q_heads}, "
                        f"H_kv={w.num_kv_heads}, head_dim 128, context {ctx_text(w)}, G=32, "
                        f"R={w.residual_v}, page 16, {w.dtype}, "
                        f"{'FP8 E4M3 pages' if bits == 8 else f'{bits}-bit codes'}, {what}",
            "step": step_txt,
            "l2": "inputs larger than L2 (about 1.6 GB of cache per layer call, layers rotate)",
            "parallelism": f"replicas x{world} (sequences shard with no exchange)",
        },
        "decode_attn_gbs": round(dec_gbs, 1),
        "decode_attn_pct_of_peak": round(100 * dec_gbs / hbm, 1),
        "kv_tokens_per_s": round(world * stats["kv_tokens"] / (stats["ms"] * 1e-3), 1),
        "append_ns_per_token": round(stats["app_ms"] * 1e6 / (stats["B"] * nq), 2),
        "append_chunk_gbs": round(stats["chunk"]["gbs"], 1) if stats.get("chunk") else None,
        "append_chunk_ns_per_token": round(stats["chunk"]["ns_per_token"], 3) if stats.get("chunk") else None,
        "append_chunk": ({
            "what": "the fill's appends: one ragged call per layer and chunk, up to 2048 new tokens per "
                    "sequence (a token = one position of one sequence across all kv heads); CUDA events "
                    "around each call; algorithmic bytes = new k/v rows read + codes and metadata written "
                    "+ ring rows read and written",
            "gbs": round(stats["chunk"]["gbs"], 1), "frac": round(stats["chunk"]["gbs"] / hbm, 4),
            "peak": hbm, "ns_per_token": round(stats["chunk"]["ns_per_token"], 3),
            "calls": stats["chunk"]["calls"], "tokens_per_call": int(stats["chunk"]["tokens"] / stats["chunk"]["calls"]),
            "bytes_per_call": int(stats["chunk"]["bytes"] / stats["chunk"]["calls"]),
            "traffic": profiled_append_traffic(args.workload, bits)} if stats.get("chunk") else None),
        "e2e": {"value": round(e2e_val, 1), "unit": "GB/s", "h2d_bytes_per_step": stats["h2d"],
                "d2h_bytes_per_step": stats["d2h"], "ms_per_step": round(stats["e2e_ms"], 4)},
        # per layer call: append_kernel, decode_kernel and merge_kernel
        "gpu_launches": args.steps * L * 3,
        "decode_step_fused": ({
            "what": "the same steps through s4kv_decode_step (append + attention of a layer in one cooperative "
                    "launch, plus the combine launch), against the separate append and decode calls of the "
                    "headline loop; microseconds per layer call, whole-step CUDA events",
            "fused_us_per_layer": round(stats["fused_ms"] * 1e3 / L, 2),
            "separate_us_per_layer": round(stats["ms"] * 1e3 / L, 2),
            "launches_per_layer": {"fused": 2, "separate": 3}} if stats.get("fused_ms") else None),
        "roofline": {
            "bound": "hbm",
            "kernel": kern_txt,
            "achieved": round(dec_gbs, 1),
            "peak": hbm,
            "peak_kind": f"{peak_kind} (copy GB/s)",
            "unit": "GB/s",
            "frac": round(dec_gbs / hbm, 4),
            "traffic": profiled_traffic(args.workload, bits),
            "traffic_source": traffic_source(args.workload, bits),
            "algorithmic_bytes_per_launch": int(stats["dec_b"] / L),
        },
        "clocks": stats["clocks"],
        "fill_s": round(stats["fill_s"], 2),
    }
    if nq > 1:
        tpk, tkind = tensor_peak()
        tfl = (stats["flops"] / L) / (stats["dec_ms"] * 1e-3) / 1e12
        r = line["roofline"]
        r["tensor"] = {"achieved_tflops": round(tfl, 1), "peak_tflops": tpk,
                       "peak_kind": f"{tkind} (dense bf16, burst)", "frac": round(tfl / tpk, 4),
                       "flops_per_launch": int(stats["flops"] / L)}
        if tfl / tpk > r["frac"]:
            r.update(bound="tensor", achieved=round(tfl, 1), peak=tpk, unit="TFLOP/s", frac=round(tfl / tpk, 4),
                     peak_kind=f"{tkind} (dense bf16, burst)")
        r["traffic"] = None
        line["multi_query_tokens"] = nq
    if stats.get("configs"):
        cfgs = dict(stats["configs"])
        cfgs[args.workload] = {
            "workload": line["config"]["workload"], "see": "the headline keys of this line",
            "decode_attn_gbs": line["decode_attn_gbs"], "decode_attn_frac": line["roofline"]["frac"],
            "kv_tokens_per_s": line["kv_tokens_per_s"], "append_ns_per_token": line["append_ns_per_token"],
            "append_chunk_fill": {"gbs": line["append_chunk_gbs"],
                                  "ns_per_token": line["append_chunk_ns_per_token"]}}
        order = ["tiny", "qwen2.5-1.5b", "llama3.1-8b", "qwen2.5-7b-32k", "mixed-trace"]
        line["configs"] = {k: cfgs[k] for k in order if k in cfgs}
    if cpu is not None:
        line["cpu_baseline"] = cpu
    return line


# ------------------------------------------------------------ oracle arm --
def oracle_sample(w, seconds_budget=20.0, max_pairs=None, seed=99):
    """Times the oracle (append every token, then decode attention) on sampled
    (sequence, kv head) pairs of the workload at its full length. Returns
    (GB/s of decode-attention algorithmic bytes, append ns/token, sample text,
    pairs done, seconds)."""
    import numpy as np
    import torch
    import oracle

    T = int(inp.context_lengths(w, seed)[0])
    dt = w.torch_dtype
    done, t_dec, t_app, bytes_dec, toks = 0, 0.0, 0.0, 0, 0
    t_start = time.time()
    while True:
        k, v = inp.kv_rows(seed + done, T, 1, 128, dt,
                           inp.outlier_channels(seed, 0, 1, 128, w.k_outliers), w.k_outlier_factor)
        q = inp.queries(seed + done, 1, w.group, 128, dt)
        s = oracle.Seq(num_kv_heads=1, residual_v=w.residual_v,
                       dtype=oracle.F16 if w.dtype == "fp16" else oracle.BF16)
        kb, vb, qb = inp.to_bits(k), inp.to_bits(v), inp.to_bits(q[0])
        a0 = time.perf_counter()
        s.append(kb, vb)
        a1 = time.perf_counter()
        s.attention(0, qb, 1.0 / math.sqrt(128))
        a2 = time.perf_counter()
        t_app += a1 - a0
        t_dec += a2 - a1
        toks += T
        # one (sequence, kv head) pair's share of a decode call's bytes
        bytes_dec += decode_bytes([T], 1, w.group, w.residual_v)
        done += 1
        if (max_pairs and done >= max_pairs) or time.time() - t_start > seconds_budget:
            break
    sample = (f"{done} (sequence, kv head) pairs of {w.name} at T={T}: oracle append of all T "
              f"tokens, then decode attention for the {w.group} query heads of the pair")
    return bytes_dec / t_dec / 1e9, t_app * 1e9 / toks, sample, done, t_dec + t_app


def cpu_baseline(w):
    gbs, ns_tok, sample, pairs, secs = oracle_sample(w, seconds_budget=15.0)
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": sample, "append_ns_per_token_head": round(ns_tok, 1),
            "cpu": _cpu_name(), "nproc": os.cpu_count()}


def _cpu_name():
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith(("model name", "cpu model")):
                return ln.split(":", 1)[1].strip()
        out = subprocess.run(["lscpu"], capture_output=True, text=True).stdout
        for ln in out.splitlines():
            if ln.startswith("Model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def run_reference(args):
    w = inp.WORKLOADS[args.workload]
    import oracle
    oracle.build()
    # each step: one (sequence, kv head) pair at full length, through the oracle
    for i in range(args.warmup):
        oracle_sample(w, seconds_budget=0.0, max_pairs=1, seed=500 + i)
    t0 = time.time()
    gbs_l, ns_l = [], []
    for i in range(args.steps):
        gbs, ns_tok, sample, _, _ = oracle_sample(w, seconds_budget=0.0, max_pairs=1, seed=900 + i)
        gbs_l.append(gbs)
        ns_l.append(ns_tok)
    wall = time.time() - t0
    value = statistics.mean(gbs_l)
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": args.gpus,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(wall * 1e3 / max(args.steps, 1), 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64 attention over fp32-restored int4 cache",
        "data": "synthetic (seeded N(0,1) K/V, key outlier channels, N(0,1) q)",
        "config": {"workload": f"{w.name} (one (sequence, kv head) pair per step)"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample, "cpu": _cpu_name(), "nproc": os.cpu_count(),
                         "append_ns_per_token_head": round(statistics.mean(ns_l), 1)},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="qwen2.5-7b-32k", choices=sorted(inp.WORKLOADS))
    ap.add_argument("--layers", type=int, default=0, help="override the workload's layer count")
    ap.add_argument("--decode-impl", dest="impl_variant", type=int, default=None,
                    help="0 tensor-core path (default), 1 FFMA path")
    ap.add_argument("--tail-cost", dest="tail_cost", type=int, default=0,
                    help="work-partition weight of a tail chunk (0 = library default)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--configs", default="auto", choices=["auto", "on", "off"],
                    help="also run the other workloads (tiny, qwen2.5-1.5b, llama3.1-8b, mixed-trace) after the "
                         "headline (auto: on the default run)")
    ap.add_argument("--bits", type=int, default=4, choices=[2, 4, 8],
                    help="code width of the pages: 4 (default) or 2 (the pages' own KIVI settings), "
                         "8 = FP8 E4M3 pages with per-head scales")
    ap.add_argument("--key-split", dest="key_split", action="store_true",
                    help="decode key scores keep the low f16 part of q' on wide-scale slices")
    ap.add_argument("--mq-kernel", dest="mq_kernel", type=int, default=0, choices=[0, 1, 2, 3],
                    help="multi-query kernel on 4/2-bit pages: 0 by column count, 1 fold, 2 restore "
                         "(mma.sync), 3 restore (tcgen05)")
    ap.add_argument("--queries", type=int, default=1,
                    help="query tokens per sequence and layer call: 1 = decode (default); 2..16 = "
                         "multi-query causal attention of a chunk")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if args.warmup < 3:
        args.warmup = 3

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    stats = run_ours(args, rank, world)
    run_cfgs = args.configs == "on" or (args.configs == "auto" and world == 1 and args.queries == 1
                                         and args.workload == "qwen2.5-7b-32k" and args.bits == 4
                                         and args.impl_variant is None and not args.layers)
    if run_cfgs:
        import torch
        dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
        stats["configs"] = {name: run_config(name, dev, bits=args.bits) for name in CONFIG_RUNS}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(inp.WORKLOADS[args.workload])
    if rank == 0:
        print(json.dumps(report_ours(args, stats, world, cpu)), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
