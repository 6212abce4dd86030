"""Parity at the workloads' full sizes, in the configuration bench.py times,
on sampled sequences the oracle can rebuild one by one.

Token rows are generated on the device (torch's seeded generator) and the rows
of the sampled sequences are copied back as they are generated; the oracle
rebuilds those sequences from the copies. Codes, metadata and ring rows are
compared byte for byte, attention within |err| <= 2e-3 + 1e-2 |ref|.
"""
import math

import numpy as np
import pytest
import torch

import int4_kivi_quantized_gb300 as s4
import oracle
import s4kv_inputs as inp
from gpu_util import assert_close

pytestmark = pytest.mark.gpu


class DeviceFill:
    """A multi-layer cache filled with device-generated rows; host copies of the
    rows of `watch` = {(layer, b)} are kept for the oracle."""

    def __init__(self, w, seed, lens, layers, extra_tokens, watch, table=None, bits=4):
        self.w, self.seed, self.layers = w, seed, layers
        self.dev = torch.device("cuda")
        self.B, self.H, self.Hq, self.g = len(lens), w.num_kv_heads, w.num_q_heads, w.group
        self.dtype = w.torch_dtype
        cap = [max((int(L) + extra_tokens + 15) // 16, 1) for L in lens]
        self.num_pages = sum(cap)
        self.bt = inp.block_tables(table or w.table, self.B, cap, self.num_pages, seed)
        self.bt_dev = self.bt.to(self.dev)
        self.bits = bits
        self.cache = s4.KVCache(layers, self.num_pages, self.H, w.residual_v, self.B, w.dtype, bits=bits)
        self.cur = [0] * self.B
        self.watch = set(watch)
        self.hist = {key: [] for key in self.watch}
        self.gen = inp.gen(seed, self.dev)
        self.scale = {}
        for layer in range(layers):
            o = inp.outlier_channels(seed, layer, self.H, 128, w.k_outliers)
            sc = torch.ones(self.H, 128)
            for h in range(self.H):
                sc[h, o[h]] = w.k_outlier_factor
            self.scale[layer] = sc.to(self.dev)

    def append(self, news):
        """One ragged append per layer: news[b] new tokens for sequence b."""
        n = int(sum(news))
        cu = torch.tensor([0] + list(np.cumsum(news)), dtype=torch.int32, device=self.dev)
        before = torch.tensor(self.cur, dtype=torch.int32, device=self.dev)
        offs = np.concatenate([[0], np.cumsum(news)])
        for layer in range(self.layers):
            k = (torch.randn((n, self.H, 128), generator=self.gen, device=self.dev) * self.scale[layer]).to(self.dtype)
            v = torch.randn((n, self.H, 128), generator=self.gen, device=self.dev).to(self.dtype)
            self.cache.append(layer, k, v, cu, before, self.bt_dev)
            for (L, b) in self.watch:
                if L == layer and news[b]:
                    self.hist[(L, b)].append((k[offs[b]:offs[b + 1]].cpu(), v[offs[b]:offs[b + 1]].cpu()))
        self.cur = [c + int(x) for c, x in zip(self.cur, news)]

    def fill(self, lens, chunk=2048):
        lens = [int(x) for x in lens]
        while any(c < L for c, L in zip(self.cur, lens)):
            self.append([min(chunk, L - c) for c, L in zip(self.cur, lens)])

    def oracle_seq(self, layer, b):
        s = oracle.Seq(num_kv_heads=self.H, residual_v=self.w.residual_v,
                       dtype=oracle.F16 if self.w.dtype == "fp16" else oracle.BF16, bits=self.bits)
        for k, v in self.hist[(layer, b)]:
            s.append(inp.to_bits(k), inp.to_bits(v))
        return s

    def decode(self, layer, q):
        seq = torch.tensor(self.cur, dtype=torch.int32, device=self.dev)
        return self.cache.decode(layer, q, self.bt_dev, seq, max(self.cur))

    def check(self, layer, b, q_host, out_row):
        s = self.oracle_seq(layer, b)
        assert s.counts()[0] == self.cur[b]
        # bytes of this sequence's pages and rings
        lay = self.cache.layout
        base = lay.layer_offset + layer * lay.layer_stride
        # this sequence's pages in logical order, against the oracle's image of a
        # table that maps logical page j to image page j
        row = self.bt[b][self.bt[b] >= 0]
        pages, valid = s.page_image(np.arange(row.numel(), dtype=np.int32), row.numel())
        idx = row.to(self.dev).long()
        got = self.cache.pool[base:base + self.num_pages * lay.page_stride].view(
            self.num_pages, self.H, lay.record_bytes)[idx].cpu().numpy()
        assert not ((got ^ pages) & valid).any(), f"page bytes differ (layer {layer}, seq {b})"
        if self.bits != 8:   # FP8 pools have no rings
            self._check_rings(s, base, b)
        self._check_attention(s, layer, b, q_host, out_row)

    def _check_rings(self, s, base, b):
        lay = self.cache.layout
        kr, kv, vr, vv = s.ring_image()
        kring = self.cache.pool[base + lay.kring_offset + b * lay.kring_slot_stride:
                                base + lay.kring_offset + (b + 1) * lay.kring_slot_stride]
        vring = self.cache.pool[base + lay.vring_offset + b * lay.vring_slot_stride:
                                base + lay.vring_offset + (b + 1) * lay.vring_slot_stride]
        kring = kring.view(torch.int16).view(self.H, 32, 128).cpu().numpy().view(np.uint16)
        vring = vring.view(torch.int16).view(self.H, self.w.residual_v, 128).cpu().numpy().view(np.uint16)
        assert np.array_equal(kring[kv.astype(bool)], kr[kv.astype(bool)])
        assert np.array_equal(vring[vv.astype(bool)], vr[vv.astype(bool)])

    def _check_attention(self, s, layer, b, q_host, out_row):
        ref = np.zeros((self.Hq, 128), np.float32)
        qb = inp.to_bits(q_host[b])
        for h in range(self.H):
            ref[h * self.g:(h + 1) * self.g] = s.attention(h, qb[h * self.g:(h + 1) * self.g], 1 / math.sqrt(128))
        assert_close(out_row, ref, f"layer {layer} seq {b} T={self.cur[b]}")


@pytest.mark.parametrize("bits", [4, 8])
def test_qwen25_7b_32k_all_28_layers(bits):
    """28 layers, batch 64, H_q 28, H_kv 4, every context 32768, fp16, 1% key
    outlier channels x16: fill, decode every layer, then two decode steps of
    (append 1 token, decode) per layer; sampled sequences against the oracle.
    4-bit KIVI pages (the bench default) and FP8 E4M3 pages (bench --bits 8,
    unit scales)."""
    w = inp.WORKLOADS["qwen2.5-7b-32k"]
    lens = inp.context_lengths(w, 11).tolist()
    watch = [(0, 0), (0, 37), (13, 5), (27, 63)]
    f = DeviceFill(w, 11, lens, w.layers, 4, watch, bits=bits)
    f.fill(lens)
    rc, d = f.cache.status()
    assert rc == 0, (rc, d)
    for step in range(3):
        if step:
            f.append([1] * f.B)
        q = inp.queries(50 + step, f.B, f.Hq, 128, f.dtype)
        outs = {layer: f.decode(layer, q.cuda()) for layer in range(w.layers)}
        rc, d = f.cache.status()
        assert rc == 0, (rc, d)
        for (layer, b) in watch:
            f.check(layer, b, q, outs[layer][b].cpu().numpy())


def test_mixed_serving_trace_full_batch():
    """Llama-3.1-8B shapes (H_q 32, H_kv 8), batch 128, contexts log-uniform in
    [256, 65536], bf16, fragmented block table; eight steps in which each
    sequence takes a 2048-token chunk append or a 1-token decode append (3:1),
    each followed by decode attention. Two of the 32 layers are filled (every
    call has the full per-layer shape); sampled sequences, including ones whose
    flushes cross page boundaries, are checked at the first and last step."""
    w = inp.WORKLOADS["mixed-trace"]
    lens = inp.context_lengths(w, 21).tolist()
    rng = np.random.default_rng(21)
    plan = [[2048 if rng.random() < 0.75 else 1 for _ in lens] for _ in range(w.steps)]
    extra = [sum(p[b] for p in plan) for b in range(len(lens))]
    short = int(np.argmin(lens))
    long_ = int(np.argmax(lens))
    odd = next(b for b in range(len(lens)) if lens[b] % 16 not in (0, 15) and plan[0][b] == 1)
    watch = [(0, short), (1, long_), (0, odd), (1, 77)]
    f = DeviceFill(w, 21, lens, 2, max(extra), watch, table="fragmented")
    f.fill(lens)
    for step in range(w.steps):
        f.append(plan[step])
        q = inp.queries(80 + step, f.B, f.Hq, 128, f.dtype)
        outs = [f.decode(layer, q.cuda()) for layer in range(2)]
        rc, d = f.cache.status()
        assert rc == 0, (rc, d)
        if step in (0, w.steps - 1):
            for (layer, b) in watch:
                f.check(layer, b, q, outs[layer][b].cpu().numpy())
