"""GPU vs oracle parity through the C ABI (bit-exact codes/metadata/rings,
attention within |err| <= 2e-3 + 1e-2 |ref|)."""
import math

import numpy as np
import pytest
import torch

import int4_kivi_quantized_gb300 as s4
import oracle
import s4kv_inputs as inp
from gpu_util import Scenario, assert_close

pytestmark = pytest.mark.gpu


def _q(sc, seed):
    return inp.queries(seed, sc.B, sc.Hq, 128, sc.dtype)


def _check_status(sc):
    rc, detail = sc.cache.status()
    assert rc == 0, (s4.s4kv_strerror(rc), detail)


@pytest.mark.parametrize("impl", [0, 1])
def test_tiny_quantize_then_decode(impl):
    """Tiny workload: T = 256 (8 full key groups, value ring of 32), then a 257th
    token (key residual of 1), each followed by one decode step."""
    w = inp.WORKLOADS["tiny"]
    sc = Scenario(w, 11, [256], extra_tokens=1)
    sc.cache.set_option(s4.S4KV_OPT_DECODE_IMPL, impl)
    sc.fill()
    _check_status(sc)
    oseq = sc.check_bytes(0, 0)
    q = _q(sc, 5)
    out = sc.decode(0, q.cuda())
    _check_status(sc)
    assert_close(out.cpu().numpy()[0], sc.oracle_attention(0, 0, q, oseq), "T=256")
    sc.cur = sc.append(0, [1], 1)
    _check_status(sc)
    oseq = sc.check_bytes(0, 0)
    out = sc.decode(0, q.cuda())
    _check_status(sc)
    assert_close(out.cpu().numpy()[0], sc.oracle_attention(0, 0, q, oseq), "T=257")
    kh, vh = sc.cache.dequant(0, 0, sc.bt_dev[0], 257)
    rk, rv = oseq.dequant(0)
    assert np.array_equal(kh[0].cpu().numpy().view(np.uint32), rk.view(np.uint32))
    assert np.array_equal(vh[0].cpu().numpy().view(np.uint32), rv.view(np.uint32))


def test_append_order_invariance():
    """One chunk, token by token, and random chunks give byte-identical pages
    and rings (the canonical state depends only on the tokens and T)."""
    w = inp.WORKLOADS["qwen2.5-1.5b"]
    T = 300
    k, v = inp.kv_rows(3, T, w.num_kv_heads, 128, torch.float16,
                       inp.outlier_channels(3, 0, w.num_kv_heads, 128, 3), 8.0)
    kd, vd = k.cuda(), v.cuda()
    images = []
    rng = np.random.default_rng(0)
    for mode in ("chunk", "single", "random"):
        cache = s4.KVCache(1, 32, w.num_kv_heads, w.residual_v, 1, "fp16")
        bt = torch.randperm(32, generator=inp.gen(9)).to(torch.int32)[:19][None].cuda()
        if mode == "chunk":
            cuts = [0, T]
        elif mode == "single":
            cuts = list(range(T + 1))
        else:
            cuts = [0]
            while cuts[-1] < T:
                cuts.append(min(T, cuts[-1] + int(rng.integers(1, 70))))
        for a, b in zip(cuts[:-1], cuts[1:]):
            cache.append(0, kd[a:b], vd[a:b], torch.tensor([0, b - a], dtype=torch.int32).cuda(),
                         torch.tensor([a], dtype=torch.int32).cuda(), bt)
        rc, d = cache.status()
        assert rc == 0, (rc, d)
        lay = cache.layout
        images.append((cache.pool[lay.layer_offset:lay.layer_offset + lay.layer_stride].cpu().numpy(), bt))
        cache.close()
    # compare the defined bytes only (the oracle's mask); pages and rings alike
    s = oracle.Seq(num_kv_heads=w.num_kv_heads, residual_v=w.residual_v)
    s.append(inp.to_bits(k), inp.to_bits(v))
    bt = images[0][1][0].cpu().numpy()
    pages, valid = s.page_image(bt, 32)
    n = 32 * w.num_kv_heads * 3072
    for img, _ in images:
        got = img[:n].reshape(32, w.num_kv_heads, 3072)
        assert not ((got ^ pages) & valid).any()
    a0 = images[0][0]
    for img, _ in images[1:]:
        got = img[:n].reshape(32, w.num_kv_heads, 3072)
        assert np.array_equal(got & valid, a0[:n].reshape(32, w.num_kv_heads, 3072) & valid)


def test_physical_page_permutation_gives_identical_output():
    w = inp.WORKLOADS["qwen2.5-1.5b"]
    lens = [700, 1500, 33, 2048]
    outs = []
    for table in ("identity", "permuted", "fragmented"):
        sc = Scenario(w, 21, lens, table=table, slack_pages=5)
        sc.fill()
        q = _q(sc, 4)
        outs.append(sc.decode(0, q.cuda()).cpu().numpy())
        _check_status(sc)
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


@pytest.mark.parametrize("warps", [1, 7, 64, 333, 0])
def test_work_partition_sensitivity(warps):
    """Any number of worker warps (so any cut of the segments into partials)
    gives the same attention within tolerance."""
    w = inp.WORKLOADS["qwen2.5-1.5b"]
    lens = [2048, 2500, 3001, 4096, 1, 31, 160, 129]
    sc = Scenario(w, 31, lens)
    sc.cache.set_option(s4.S4KV_OPT_DECODE_WARPS, warps)
    sc.fill()
    q = _q(sc, 6)
    out = sc.decode(0, q.cuda()).cpu().numpy()
    _check_status(sc)
    for b in range(sc.B):
        assert_close(out[b], sc.oracle_attention(0, b, q), f"seq {b} warps {warps}")


@pytest.mark.parametrize("impl", [0, 1])
def test_qwen15b_workload_full_parity(impl):
    """Qwen2.5-1.5B-like layer: B=8, H_q=12, H_kv=2, T ~ U[2048, 4096], fp16,
    3 outlier key channels x8, permuted pages: every output row, every byte."""
    w = inp.WORKLOADS["qwen2.5-1.5b"]
    lens = inp.context_lengths(w, 2).tolist()
    sc = Scenario(w, 2, lens)
    sc.cache.set_option(s4.S4KV_OPT_DECODE_IMPL, impl)
    sc.fill()
    _check_status(sc)
    q = _q(sc, 3)
    out = sc.decode(0, q.cuda()).cpu().numpy()
    _check_status(sc)
    for b in range(sc.B):
        oseq = sc.check_bytes(0, b) if impl == 0 else None
        assert_close(out[b], sc.oracle_attention(0, b, q, oseq), f"seq {b}")


def test_key_split_option_tightens_the_error_on_wide_scale_channels():
    """Qwen2.5-7B-like heads (one key outlier channel x16 per head): decode with
    S4KV_OPT_KEY_SPLIT = 1 (the default) meets the bar, and its worst error
    against the oracle is no larger than with the split off (0, whose error may
    pass the bar on such channels)."""
    w = inp.WORKLOADS["qwen2.5-7b-32k"]
    sc = Scenario(w, 5, [4101, 2045, 700, 13])
    sc.fill()
    q = _q(sc, 6)
    errs = {}
    for split in (1, 0):
        sc.cache.set_option(s4.S4KV_OPT_KEY_SPLIT, split)
        out = sc.decode(0, q.cuda()).cpu().numpy()
        _check_status(sc)
        worst = 0.0
        for b in range(sc.B):
            ref = sc.oracle_attention(0, b, q)
            if split:
                worst = max(worst, assert_close(out[b], ref, f"split {split} seq {b}"))
            else:
                worst = max(worst, float(np.abs(out[b].astype(np.float64) - ref).max()))
        errs[split] = worst
    sc.cache.set_option(s4.S4KV_OPT_KEY_SPLIT, 1)
    assert errs[1] <= errs[0] * 1.05 + 1e-6, errs


def test_llama8b_workload_decode_steps_bf16():
    """Llama-3.1-8B-like layer, bf16, B=32, H_q=32, H_kv=8, T ~ U[1024, 8192],
    shuffled pages: 64 steps of (append 1 token, decode); the oracle checks
    every sequence at the first and last step and two sequences every 8 steps."""
    w = inp.WORKLOADS["llama3.1-8b"]
    lens = inp.context_lengths(w, 4).tolist()
    sc = Scenario(w, 4, lens, extra_tokens=w.steps)
    sc.fill()
    _check_status(sc)
    for step in range(w.steps):
        sc.cur = sc.append(0, [1] * sc.B, 1 + step)
        q = _q(sc, 100 + step)
        out = sc.decode(0, q.cuda())
        if step in (0, w.steps - 1) or step % 8 == 0:
            _check_status(sc)
            o = out.cpu().numpy()
            check = range(sc.B) if step in (0, w.steps - 1) else (step % sc.B, (7 * step) % sc.B)
            for b in check:
                assert_close(o[b], sc.oracle_attention(0, b, q), f"step {step} seq {b}")
    sc.check_bytes(0, 3)
    sc.check_bytes(0, 17)


def test_bf16_output_dtype():
    w = inp.WORKLOADS["llama3.1-8b"]
    sc = Scenario(w, 8, [1000, 77])
    sc.fill()
    q = _q(sc, 1)
    o32 = sc.decode(0, q.cuda(), out_dtype=s4.S4KV_F32).cpu().float().numpy()
    o16 = sc.decode(0, q.cuda(), out_dtype=s4.S4KV_BF16).cpu().float().numpy()
    assert np.array_equal(torch.from_numpy(o32).to(torch.bfloat16).float().numpy(), o16)


def test_edge_lengths_and_empty_sequences():
    """Lengths 0, 1, G-1, G, G+1, R, R+1, a page boundary and a long one."""
    w = inp.WORKLOADS["qwen2.5-1.5b"]
    lens = [0, 1, 31, 32, 33, 128, 129, 16 * 37, 5000]
    sc = Scenario(w, 41, lens)
    sc.fill()
    q = _q(sc, 2)
    out = sc.decode(0, q.cuda()).cpu().numpy()
    _check_status(sc)
    assert not out[0].any()
    for b in range(1, sc.B):
        assert_close(out[b], sc.oracle_attention(0, b, q), f"len {lens[b]}")
