"""FP8 E4M3 pages (cfg.bits = 8; "4.4 KV Cache 量化", sections 4.1 and 4.2: the
fp8_e4m3 KV type with a scale per attention head): page bytes equal the
oracle's FP8 image bit for bit, the debug restore equals the oracle's restored
cache exactly, and decode attention over the pages matches the oracle within
|err| <= 2e-3 + 1e-2 |ref| (both dtypes, calibrated and unit scales, forced
work partitions, partial last pages)."""
import numpy as np
import pytest
import torch

import int4_kivi_quantized_gb300 as s4
import oracle
import s4kv_inputs as inp
from gpu_util import Scenario, assert_close

pytestmark = pytest.mark.gpu


def _status(sc):
    rc, d = sc.cache.status()
    assert rc == 0, (s4.s4kv_strerror(rc), d)


def _check_all(sc, q, what):
    out = sc.decode(0, q.cuda()).cpu().numpy()
    _status(sc)
    for b in range(sc.B):
        oseq = sc.check_bytes(0, b)
        assert_close(out[b], sc.oracle_attention(0, b, q, oseq), f"{what} seq {b} T={sc.cur[b]}")


@pytest.mark.parametrize("name,seed", [("qwen2.5-1.5b", 61), ("llama3.1-8b", 62)])
def test_fp8_pages_and_decode_match_the_oracle(name, seed):
    """Unit scales (the uncalibrated default); lengths around page and group
    boundaries, so partial last pages (stale bytes masked) are covered."""
    w = inp.WORKLOADS[name]
    lens = inp.context_lengths(w, seed).tolist()[:5] + [1, 15, 16, 17, 31, 32, 33, 160]
    sc = Scenario(w, seed, lens, bits=8)
    sc.fill()
    _status(sc)
    _check_all(sc, inp.queries(seed + 1, sc.B, sc.Hq, 128, sc.dtype), name)


def test_fp8_calibrated_scales_and_saturation():
    """Per-head key/value scales, one head's so small that its largest keys
    saturate at +-448: codes still match the oracle bit for bit, and attention
    over the saturated cache matches the oracle's."""
    w = inp.WORKLOADS["qwen2.5-7b-32k"]   # 4 kv heads, one x16 key outlier channel per head
    ks = [0.05, 0.25, 1.0, 3.0]
    vs = [0.5, 0.01, 2.0, 1.0]
    sc = Scenario(w, 63, [3001, 2048, 77, 5], bits=8, fp8_scales=[(ks, vs)])
    sc.fill()
    _status(sc)
    hist = sc.oracle_seq(0, 0).history(0)
    assert (hist["kcode"] & 0x7F == 0x7E).any(), "the test wants saturated key codes on head 0"
    _check_all(sc, inp.queries(64, sc.B, sc.Hq, 128, sc.dtype), "scaled")


def test_fp8_decode_steps_and_exact_restore():
    """One-token appends (every token lands in its page at once), decode every
    few steps; the debug restore equals value(code) * scale of the oracle."""
    w = inp.WORKLOADS["qwen2.5-1.5b"]
    sc = Scenario(w, 65, [95, 300, 0], extra_tokens=40, bits=8,
                  fp8_scales=[([0.5, 2.0], [1.0, 0.125])])
    sc.fill()
    for step in range(1, 40):
        sc.cur = sc.append(0, [1] * sc.B, step)
        if step % 13 == 0:
            q = inp.queries(200 + step, sc.B, sc.Hq, 128, sc.dtype)
            out = sc.decode(0, q.cuda()).cpu().numpy()
            _status(sc)
            for b in range(sc.B):
                assert_close(out[b], sc.oracle_attention(0, b, q), f"step {step} seq {b}")
    for b in range(sc.B):
        s = sc.check_bytes(0, b)
        kh, vh = sc.cache.dequant(0, b, sc.bt_dev[b], sc.cur[b])
        _status(sc)
        for h in range(sc.H):
            ok, ov = s.dequant(h)
            assert np.array_equal(kh[h].cpu().numpy().view(np.uint32), ok.view(np.uint32))
            assert np.array_equal(vh[h].cpu().numpy().view(np.uint32), ov.view(np.uint32))


def test_fp8_append_order_invariance():
    """One chunk, token by token, and random chunks give the same page bytes."""
    w = inp.WORKLOADS["qwen2.5-1.5b"]
    T = 300
    k, v = inp.kv_rows(7, T, w.num_kv_heads, 128, torch.float16,
                       inp.outlier_channels(7, 0, w.num_kv_heads, 128, 3), 8.0)
    kd, vd = k.cuda(), v.cuda()
    rng = np.random.default_rng(1)
    bt = torch.randperm(32, generator=inp.gen(9)).to(torch.int32)[:19][None].cuda()
    s = oracle.Seq(num_kv_heads=w.num_kv_heads, bits=8)
    s.append(inp.to_bits(k), inp.to_bits(v))
    pages, valid = s.page_image(bt[0].cpu().numpy(), 32)
    for mode in ("chunk", "single", "random"):
        cache = s4.KVCache(1, 32, w.num_kv_heads, w.residual_v, 1, "fp16", bits=8)
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
        assert lay.record_bytes == 4096
        got = cache.pool[lay.layer_offset:lay.layer_offset + 32 * lay.page_stride].cpu().numpy()
        got = got.reshape(32, w.num_kv_heads, 4096)
        assert not ((got ^ pages) & valid).any(), mode
        cache.close()


@pytest.mark.parametrize("warps", [1, 7, 333, 0])
def test_fp8_work_partition_sensitivity(warps):
    w = inp.WORKLOADS["llama3.1-8b"]
    sc = Scenario(w, 66, [4101, 700, 13, 2048, 1, 4000], bits=8)
    sc.fill()
    sc.cache.set_option(s4.S4KV_OPT_DECODE_WARPS, warps)
    q = inp.queries(67, sc.B, sc.Hq, 128, sc.dtype)
    out = sc.decode(0, q.cuda()).cpu().numpy()
    _status(sc)
    for b in range(sc.B):
        assert_close(out[b], sc.oracle_attention(0, b, q), f"warps {warps} seq {b}")


def test_fp8_bounded_wait_gives_up_and_the_next_call_is_clean():
    w = inp.WORKLOADS["qwen2.5-1.5b"]
    sc = Scenario(w, 68, [3000, 2500, 4000], bits=8)
    sc.fill()
    sc.cache.set_option(s4.S4KV_OPT_WAIT_NS, 0)
    q = inp.queries(69, sc.B, sc.Hq, 128, sc.dtype)
    sc.decode(0, q.cuda())
    rc, detail = sc.cache.status()
    assert rc == s4.S4KV_ERR_DEVICE_TIMEOUT and detail == s4.S4KV_DEV_TIMEOUT
    sc.cache.set_option(s4.S4KV_OPT_WAIT_NS, 1_000_000_000)
    out = sc.decode(0, q.cuda()).cpu().numpy()
    _status(sc)
    for b in range(sc.B):
        assert_close(out[b], sc.oracle_attention(0, b, q), f"seq {b}")


def test_fp8_refusals():
    """The FFMA path reads KIVI records only; scales must be finite and
    positive, and a KIVI pool has none."""
    w = inp.WORKLOADS["qwen2.5-1.5b"]
    sc = Scenario(w, 70, [100, 40], bits=8)
    sc.fill()
    sc.cache.set_option(s4.S4KV_OPT_DECODE_IMPL, 1)
    with pytest.raises(s4.S4KVError) as e:
        sc.decode(0, inp.queries(1, sc.B, sc.Hq, 128, sc.dtype).cuda())
    assert e.value.code == s4.S4KV_ERR_UNSUPPORTED
    sc.cache.set_option(s4.S4KV_OPT_DECODE_IMPL, 0)
    for bad in ([0.0, 1.0], [1.0, -2.0], [float("nan"), 1.0], [float("inf"), 1.0]):
        with pytest.raises(s4.S4KVError) as e:
            sc.cache.set_fp8_scales(0, bad, [1.0, 1.0])
        assert e.value.code == s4.S4KV_ERR_INVALID_ARG, bad
    kivi = s4.KVCache(1, 8, 2, 32, 1, "fp16")
    with pytest.raises(s4.S4KVError) as e:
        kivi.set_fp8_scales(0, [1.0, 1.0], [1.0, 1.0])
    assert e.value.code == s4.S4KV_ERR_UNSUPPORTED
    kivi.close()
    _status(sc)
