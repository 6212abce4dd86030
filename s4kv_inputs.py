"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

This module holds only workload shapes and random-number plumbing: no part of
the quantizer or of attention. The CUDA library and the oracle both receive what
it produces, and neither imports it.

The workloads follow the shapes the method's pages name: head_dim 128, the GQA
head counts of Qwen2.5 and Llama-3 models, keys with a few large-magnitude
("outlier") channels and values without them.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    layers: int
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    ctx: tuple            # ("fixed", T) | ("uniform", lo, hi) | ("loguniform", lo, hi)
    dtype: str            # "fp16" | "bf16"
    group_k: int
    group_v: int
    residual_v: int
    page_size: int
    table: str            # "identity" | "permuted" | "fragmented"
    k_outliers: int       # number of key outlier channels per (layer, kv head)
    k_outlier_factor: float
    steps: int            # decode steps of the workload
    chunk: int = 0        # prefill chunk length (mixed trace)
    chunk_ratio: tuple = (0, 1)   # (chunk appends, decode appends) per mix unit

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def torch_dtype(self):
        return torch.float16 if self.dtype == "fp16" else torch.bfloat16


WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 4, 1, 128, ("fixed", 256), "fp16", 32, 32, 32, 16,
                     "identity", 4, 10.0, 1),
    "qwen2.5-1.5b": Workload("qwen2.5-1.5b", 1, 8, 12, 2, 128, ("uniform", 2048, 4096), "fp16",
                             32, 32, 128, 16, "permuted", 3, 8.0, 1),
    "llama3.1-8b": Workload("llama3.1-8b", 1, 32, 32, 8, 128, ("uniform", 1024, 8192), "bf16",
                            32, 32, 128, 16, "permuted", 3, 8.0, 64),
    "qwen2.5-7b-32k": Workload("qwen2.5-7b-32k", 28, 64, 28, 4, 128, ("fixed", 32768), "fp16",
                               32, 32, 128, 16, "permuted", 1, 16.0, 1),
    "mixed-trace": Workload("mixed-trace", 32, 128, 32, 8, 128, ("loguniform", 256, 65536),
                            "bf16", 32, 32, 128, 16, "fragmented", 3, 8.0, 8, 2048, (3, 1)),
}


def outlier_count(frac: float, head_dim: int = 128) -> int:
    """Outlier channels for a fraction of head_dim, rounded to nearest (2% of 128 -> 3)."""
    return int(math.floor(frac * head_dim + 0.5))


def gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    return g


def mix_seed(*parts: int) -> int:
    """A fixed 63-bit mix of integers (splitmix64 finaliser), for per-unit seeds."""
    x = 0x9E3779B97F4A7C15
    for p in parts:
        x = (x ^ (int(p) & 0xFFFFFFFFFFFFFFFF)) & 0xFFFFFFFFFFFFFFFF
        x = (x + 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF
        z = x
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
        x = z ^ (z >> 31)
    return x & 0x7FFFFFFFFFFFFFFF


def outlier_channels(seed: int, layer: int, num_kv_heads: int, head_dim: int, count: int):
    """[num_kv_heads, count] distinct channel indices per KV head of one layer."""
    g = gen(mix_seed(seed, 0xC4A7, layer))
    return torch.stack([torch.randperm(head_dim, generator=g)[:count]
                        for _ in range(num_kv_heads)]) if count else \
        torch.zeros(num_kv_heads, 0, dtype=torch.long)


def context_lengths(w: Workload, seed: int) -> torch.Tensor:
    g = gen(mix_seed(seed, 0x1E45))
    kind = w.ctx[0]
    if kind == "fixed":
        return torch.full((w.batch,), w.ctx[1], dtype=torch.int32)
    lo, hi = w.ctx[1], w.ctx[2]
    if kind == "uniform":
        return torch.randint(lo, hi + 1, (w.batch,), generator=g, dtype=torch.int64).to(torch.int32)
    if kind == "loguniform":
        u = torch.rand(w.batch, generator=g, dtype=torch.float64)
        t = torch.floor(torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))))
        return t.clamp(lo, hi).to(torch.int32)
    raise ValueError(kind)


def kv_rows(seed: int, n: int, num_kv_heads: int, head_dim: int, dtype, outliers=None,
            factor: float = 1.0, device="cpu"):
    """Seeded K and V rows [n, H_kv, d]: N(0, 1), K outlier channels scaled by `factor`.

    `outliers` is an [H_kv, count] index tensor (or None). Values are drawn in
    fp32 and rounded to the cache dtype by torch's round-to-nearest-even cast.
    """
    g = gen(seed, device)
    k = torch.randn((n, num_kv_heads, head_dim), generator=g, device=device, dtype=torch.float32)
    v = torch.randn((n, num_kv_heads, head_dim), generator=g, device=device, dtype=torch.float32)
    if outliers is not None and outliers.numel():
        scale = torch.ones((num_kv_heads, head_dim), dtype=torch.float32)
        for h in range(num_kv_heads):
            scale[h, outliers[h]] = factor
        k = k * scale.to(device)
    return k.to(dtype), v.to(dtype)


def queries(seed: int, batch: int, num_q_heads: int, head_dim: int, dtype, device="cpu"):
    g = gen(seed, device)
    return torch.randn((batch, num_q_heads, head_dim), generator=g, device=device,
                       dtype=torch.float32).to(dtype)


def block_tables(kind: str, batch: int, pages_per_seq, num_pages: int, seed: int):
    """An int32 [batch, max_pages] block table; every entry a distinct physical page.

    identity   : slot b's logical page j -> b * max_pages + j
    permuted   : logical pages of all slots take a random permutation of the pool
    fragmented : pages come off a shuffled free list as the slots grow one page at
                 a time in turn (interleaved growth)
    """
    pages_per_seq = torch.as_tensor(pages_per_seq, dtype=torch.int64)
    if pages_per_seq.dim() == 0:
        pages_per_seq = pages_per_seq.repeat(batch)
    maxp = int(pages_per_seq.max().item()) if batch else 0
    need = int(pages_per_seq.sum().item())
    if need > num_pages:
        raise ValueError("pool too small for the block table")
    bt = torch.full((batch, max(maxp, 1)), -1, dtype=torch.int32)
    g = gen(mix_seed(seed, 0xB7AB))
    if kind == "identity":
        if batch * maxp > num_pages:
            raise ValueError("pool too small for an identity table")
        for b in range(batch):
            n = int(pages_per_seq[b])
            bt[b, :n] = torch.arange(b * maxp, b * maxp + n, dtype=torch.int32)
    elif kind == "permuted":
        perm = torch.randperm(num_pages, generator=g)[:need].to(torch.int32)
        o = 0
        for b in range(batch):
            n = int(pages_per_seq[b])
            bt[b, :n] = perm[o:o + n]
            o += n
    elif kind == "fragmented":
        free = torch.randperm(num_pages, generator=g).to(torch.int32).tolist()
        fill = [0] * batch
        remaining = True
        while remaining:
            remaining = False
            for b in range(batch):
                if fill[b] < int(pages_per_seq[b]):
                    bt[b, fill[b]] = free.pop()
                    fill[b] += 1
                    remaining = True
    else:
        raise ValueError(kind)
    return bt


def to_bits(t: torch.Tensor):
    """Raw 16-bit patterns of an fp16/bf16 tensor as a numpy uint16 array."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")
