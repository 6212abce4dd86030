"""Helpers for the GPU tests: seeded workloads on the device and their oracle twins."""
from __future__ import annotations

import math

import numpy as np
import torch

import int4_kivi_quantized_gb300 as s4
import oracle
import s4kv_inputs as inp

ATOL, RTOL = 2e-3, 1e-2   # |gpu - oracle| <= ATOL + RTOL * |oracle|, elementwise


def within_tol(got: np.ndarray, ref: np.ndarray, extra_abs: float = 0.0):
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    ok = err <= ATOL + extra_abs + RTOL * np.abs(ref)
    return bool(ok.all()), float(err.max()), float((err / np.maximum(np.abs(ref), 1e-30)).max())


def assert_close(got, ref, what="", extra_abs=0.0):
    ok, mabs, mrel = within_tol(np.asarray(got), np.asarray(ref), extra_abs)
    assert ok, f"{what}: max abs err {mabs:.3e} (max rel {mrel:.3e}) exceeds {ATOL} + {RTOL}|ref|"
    return mabs


class Scenario:
    """One layer-set of a workload: sequences appended into a fresh cache.

    Token rows of sequence b in layer L are drawn by s4kv_inputs.kv_rows with
    seed mix_seed(seed, L, b, epoch), so any sequence can be rebuilt on the host.
    """

    def __init__(self, w: inp.Workload, seed: int, lens, layers: int = 1, extra_tokens: int = 0,
                 device="cuda", table: str | None = None, slack_pages: int = 0, bits: int = 4,
                 fp8_scales=None):
        self.w, self.seed, self.dev = w, seed, torch.device(device)
        self.lens = [int(x) for x in lens]
        self.B = len(self.lens)
        self.layers = layers
        self.H, self.Hq, self.g = w.num_kv_heads, w.num_q_heads, w.group
        self.dtype = w.torch_dtype
        cap = [max((L + extra_tokens + 15) // 16, 1) for L in self.lens]
        kind = table or w.table
        if kind == "identity":
            self.num_pages = self.B * max(cap)
        else:
            self.num_pages = sum(cap) + slack_pages
        self.bt = inp.block_tables(kind, self.B, cap, self.num_pages, seed)
        self.bt_dev = self.bt.to(self.dev)
        self.bits = bits
        self.cache = s4.KVCache(layers, self.num_pages, self.H, w.residual_v, self.B, w.dtype,
                                device=self.dev, bits=bits)
        # FP8 pages: per layer (key scales [H], value scales [H]); None keeps 1.0
        self.fp8_scales = fp8_scales
        if fp8_scales is not None:
            for L in range(layers):
                self.cache.set_fp8_scales(L, *fp8_scales[L])
        self.outliers = [inp.outlier_channels(seed, L, self.H, 128, w.k_outliers)
                         for L in range(layers)]
        self.cur = [0] * self.B
        self.hist = {}    # (layer, b) -> list of (k, v) host tensors appended so far

    def rows(self, layer, b, n, epoch):
        return inp.kv_rows(inp.mix_seed(self.seed, layer, b, epoch), n, self.H, 128, self.dtype,
                           self.outliers[layer], self.w.k_outlier_factor)

    def append(self, layer, news, epoch, keep=True):
        """news[b] new tokens for every sequence b (one ragged call)."""
        ks, vs = [], []
        for b, n in enumerate(news):
            k, v = self.rows(layer, b, n, epoch)
            ks.append(k)
            vs.append(v)
            if keep:
                self.hist.setdefault((layer, b), []).append((k, v))
        k = torch.cat(ks).to(self.dev)
        v = torch.cat(vs).to(self.dev)
        cu = torch.tensor([0] + list(np.cumsum(news)), dtype=torch.int32, device=self.dev)
        before = torch.tensor(self.cur, dtype=torch.int32, device=self.dev)
        self.cache.append(layer, k, v, cu, before, self.bt_dev)
        return [c + n for c, n in zip(self.cur, news)]

    def fill(self, keep=True):
        for L in range(self.layers):
            self.append(L, self.lens, 0, keep)
        self.cur = list(self.lens)

    def oracle_seq(self, layer, b):
        s = oracle.Seq(num_kv_heads=self.H, residual_v=self.w.residual_v,
                       dtype=oracle.F16 if self.w.dtype == "fp16" else oracle.BF16, bits=self.bits)
        if self.fp8_scales is not None:
            s.set_fp8_scales(*self.fp8_scales[layer])
        for k, v in self.hist[(layer, b)]:
            s.append(inp.to_bits(k), inp.to_bits(v))
        return s

    def decode(self, layer, q, out_dtype=s4.S4KV_F32):
        seq = torch.tensor(self.cur, dtype=torch.int32, device=self.dev)
        return self.cache.decode(layer, q, self.bt_dev, seq, max(self.cur), out_dtype=out_dtype)

    def oracle_attention(self, layer, b, q_host, oseq=None):
        s = oseq or self.oracle_seq(layer, b)
        out = np.zeros((self.Hq, 128), np.float32)
        qb = inp.to_bits(q_host[b])
        for h in range(self.H):
            out[h * self.g:(h + 1) * self.g] = s.attention(h, qb[h * self.g:(h + 1) * self.g],
                                                           1.0 / math.sqrt(128))
        return out

    def pool_pages(self, layer):
        lay = self.cache.layout
        base = lay.layer_offset + layer * lay.layer_stride
        n = self.num_pages * lay.page_stride
        return self.cache.pool[base:base + n].view(self.num_pages, self.H, lay.record_bytes).cpu().numpy()

    def pool_rings(self, layer):
        lay = self.cache.layout
        base = lay.layer_offset + layer * lay.layer_stride
        kr = self.cache.pool[base + lay.kring_offset: base + lay.kring_offset +
                             self.B * lay.kring_slot_stride]
        vr = self.cache.pool[base + lay.vring_offset: base + lay.vring_offset +
                             self.B * lay.vring_slot_stride]
        kr = kr.view(torch.int16).view(self.B, self.H, 32, 128).cpu().numpy().view(np.uint16)
        vr = vr.view(torch.int16).view(self.B, self.H, self.w.residual_v, 128).cpu().numpy().view(np.uint16)
        return kr, vr

    def check_bytes(self, layer, b, oseq=None):
        """Pages and rings of sequence b equal the oracle's image bit for bit."""
        s = oseq or self.oracle_seq(layer, b)
        pages, valid = s.page_image(self.bt[b].numpy(), self.num_pages)
        got = self.pool_pages(layer)
        diff = (got ^ pages) & valid
        assert not diff.any(), f"page bytes differ at {np.argwhere(diff)[:5]}"
        if self.bits == 8:   # FP8 pools have no rings
            return s
        kr, kv, vr, vv = s.ring_image()
        gk, gv = self.pool_rings(layer)
        assert np.array_equal(gk[b][kv.astype(bool)], kr[kv.astype(bool)]), "key ring differs"
        assert np.array_equal(gv[b][vv.astype(bool)], vr[vv.astype(bool)]), "value ring differs"
        return s
