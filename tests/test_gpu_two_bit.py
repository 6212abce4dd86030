"""2-bit KIVI (the pages' own setting: four codes per byte, levels 0..3, same
grouping and residual policy): pages and rings equal the oracle's 2-bit image
bit for bit, and attention over them matches the oracle within
|err| <= 2e-3 + 1e-2 |ref|, for decode (both dtypes, forced work partitions)
and for multi-query chunks."""
import math

import numpy as np
import pytest
import torch

import int4_kivi_quantized_gb300 as s4
import s4kv_inputs as inp
from gpu_util import Scenario, assert_close

pytestmark = pytest.mark.gpu


def _status(sc):
    rc, d = sc.cache.status()
    assert rc == 0, (s4.s4kv_strerror(rc), d)


@pytest.mark.parametrize("name,seed", [("qwen2.5-1.5b", 31), ("llama3.1-8b", 32)])
def test_two_bit_pages_and_decode_match_the_oracle(name, seed):
    w = inp.WORKLOADS[name]
    lens = inp.context_lengths(w, seed).tolist()[:6] + [1, 31, 33, 160]
    sc = Scenario(w, seed, lens, bits=2)
    sc.fill()
    _status(sc)
    q = inp.queries(seed + 1, sc.B, sc.Hq, 128, sc.dtype)
    out = sc.decode(0, q.cuda()).cpu().numpy()
    _status(sc)
    for b in range(sc.B):
        oseq = sc.check_bytes(0, b)
        assert_close(out[b], sc.oracle_attention(0, b, q, oseq), f"{name} seq {b} T={sc.cur[b]}")


def test_two_bit_decode_steps_and_dequant():
    """One-token appends across key-group flushes and value-window evictions,
    each followed by decode; the debug restore equals the oracle's exactly."""
    w = inp.WORKLOADS["qwen2.5-1.5b"]
    sc = Scenario(w, 33, [95, 300, 130], extra_tokens=40, bits=2)
    sc.fill()
    for step in range(1, 40):
        sc.cur = sc.append(0, [1] * sc.B, step)
        if step % 13 == 0:
            q = inp.queries(100 + step, sc.B, sc.Hq, 128, sc.dtype)
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
            assert np.array_equal(kh[h].cpu().numpy(), ok) and np.array_equal(vh[h].cpu().numpy(), ov)


@pytest.mark.parametrize("warps", [1, 7, 0])
def test_two_bit_work_partition_and_key_split(warps):
    w = inp.WORKLOADS["qwen2.5-7b-32k"]
    sc = Scenario(w, 34, [4101, 700, 13], bits=2)
    sc.fill()
    sc.cache.set_option(s4.S4KV_OPT_DECODE_WARPS, warps)
    q = inp.queries(35, sc.B, sc.Hq, 128, sc.dtype)
    for split in (0, 1):
        sc.cache.set_option(s4.S4KV_OPT_KEY_SPLIT, split)
        out = sc.decode(0, q.cuda()).cpu().numpy()
        _status(sc)
        for b in range(sc.B):
            assert_close(out[b], sc.oracle_attention(0, b, q), f"warps {warps} split {split} seq {b}")


@pytest.mark.parametrize("kernel", [2, 3])
def test_two_bit_multi_query_wide(kernel):
    """96 columns (nq 16, GQA group 6): each key group restored once per team,
    for mma.sync (2) or tcgen05 (3)."""
    w = inp.WORKLOADS["qwen2.5-1.5b"]
    sc = Scenario(w, 39, [1500, 290, 40], bits=2)
    sc.cache.set_option(s4.S4KV_OPT_MQ_KERNEL, kernel)
    sc.fill()
    nq = 16
    q = torch.stack([inp.queries(39 * 100 + i, sc.B, sc.Hq, 128, sc.dtype) for i in range(nq)], dim=1)
    seq = torch.tensor(sc.cur, dtype=torch.int32, device="cuda")
    out = sc.cache.multi_query(0, q.cuda(), sc.bt_dev, seq, max(sc.cur)).cpu().numpy()
    _status(sc)
    for b in range(sc.B):
        s = sc.oracle_seq(0, b)
        qb = inp.to_bits(q[b])
        for h in range(sc.H):
            ref = s.attention_causal(h, qb[:, h * sc.g:(h + 1) * sc.g], 1 / math.sqrt(128))
            assert_close(out[b, :, h * sc.g:(h + 1) * sc.g], ref, f"seq {b} head {h}")


def test_two_bit_multi_query():
    w = inp.WORKLOADS["llama3.1-8b"]
    sc = Scenario(w, 36, [2000, 515, 70], bits=2)
    sc.fill()
    nq = 8
    q = torch.stack([inp.queries(37 * 100 + i, sc.B, sc.Hq, 128, sc.dtype) for i in range(nq)], dim=1)
    seq = torch.tensor(sc.cur, dtype=torch.int32, device="cuda")
    out = sc.cache.multi_query(0, q.cuda(), sc.bt_dev, seq, max(sc.cur)).cpu().numpy()
    _status(sc)
    for b in range(sc.B):
        s = sc.oracle_seq(0, b)
        qb = inp.to_bits(q[b])
        for h in range(sc.H):
            ref = s.attention_causal(h, qb[:, h * sc.g:(h + 1) * sc.g], 1 / math.sqrt(128))
            assert_close(out[b, :, h * sc.g:(h + 1) * sc.g], ref, f"seq {b} head {h}")


def test_two_bit_ffma_path_is_refused():
    w = inp.WORKLOADS["qwen2.5-1.5b"]
    sc = Scenario(w, 38, [100], bits=2)
    sc.fill()
    sc.cache.set_option(s4.S4KV_OPT_DECODE_IMPL, 1)
    with pytest.raises(s4.S4KVError) as e:
        sc.decode(0, inp.queries(1, sc.B, sc.Hq, 128, sc.dtype).cuda())
    assert e.value.code == s4.S4KV_ERR_UNSUPPORTED
