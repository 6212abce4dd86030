"""Multi-query attention: the last nq tokens of every sequence attend causally
over the cache after they were appended (query i sees tokens 0 .. T - nq + i).
Every output row is compared with the oracle's causal rows, elementwise within
|err| <= 2e-3 + 1e-2 |ref|, across column counts nq * g from 6 to 96, both
cache dtypes, chunks that cross a key-group boundary, and forced work
partitions; on 4-bit KIVI pages with each multi-query kernel (scales folded
into 8 columns a warp; a group restored once per team for mma.sync on 16
columns a warp; the restored group fed to tcgen05 with tensor-memory
accumulators) and on FP8 E4M3 pages with per-head scales (mma.sync on 16
columns a warp; each group's codes widened once for tcgen05).
"""
import dataclasses
import math

import numpy as np
import pytest
import torch

import int4_kivi_quantized_gb300 as s4
import s4kv_inputs as inp
from gpu_util import Scenario, assert_close

pytestmark = pytest.mark.gpu


def _queries(seed, B, nq, Hq, dtype):
    return torch.stack([inp.queries(seed * 100 + i, B, Hq, 128, dtype) for i in range(nq)], dim=1)


def _check(sc, q, out, what):
    nq = q.shape[1]
    for b in range(sc.B):
        s = sc.oracle_seq(0, b)
        qb = inp.to_bits(q[b])                       # [nq, Hq, 128]
        for h in range(sc.H):
            ref = s.attention_causal(h, qb[:, h * sc.g:(h + 1) * sc.g], 1 / math.sqrt(128))
            assert_close(out[b, :, h * sc.g:(h + 1) * sc.g], ref, f"{what} seq {b} head {h} T={sc.cur[b]}")


def _run(sc, q, max_seq_len=None):
    seq = torch.tensor(sc.cur, dtype=torch.int32, device="cuda")
    out = sc.cache.multi_query(0, q.cuda(), sc.bt_dev, seq, max_seq_len or max(sc.cur))
    rc, d = sc.cache.status()
    return out.cpu().numpy(), rc, d


FP8_SCALES = {2: ([0.5, 2.0], [1.0, 0.25]), 4: ([1.0, 0.5, 0.25, 2.0], [1.0, 2.0, 0.5, 1.0]),
              8: ([1.0, 0.5, 0.25, 2.0, 1.0, 0.125, 1.5, 1.0], [1.0, 2.0, 0.5, 1.0, 0.75, 1.0, 1.0, 4.0])}


def _scenario(w, seed, lens, bits, kernel=0):
    """A cache of 4-bit KIVI pages, or of FP8 pages with per-head scales; kernel:
    the S4KV_OPT_MQ_KERNEL choice."""
    scales = [FP8_SCALES[w.num_kv_heads]] if bits == 8 else None
    sc = Scenario(w, seed, lens, bits=bits, fp8_scales=scales)
    sc.cache.set_option(s4.S4KV_OPT_MQ_KERNEL, kernel)
    return sc


# (page bits, multi-query kernel): automatic, and each kernel of each page format
# forced at every width
KERNELS = [(4, 0), (4, 1), (4, 2), (4, 3), (8, 0), (8, 1), (8, 3)]


@pytest.mark.parametrize("bits,kernel", KERNELS)
@pytest.mark.parametrize("name,nq,lens", [
    ("qwen2.5-1.5b", 2, [300, 1057, 64, 95, 2]),         # 12 columns, team of 2
    ("qwen2.5-1.5b", 5, [777, 3000, 33, 160, 5]),        # 30 columns, team of 4
    ("qwen2.5-1.5b", 16, [1000, 2600, 129, 48, 16]),     # 96 columns, team of 12
    ("llama3.1-8b", 3, [1500, 4097, 200, 31]),           # bf16, 12 columns
    ("llama3.1-8b", 8, [2000, 515, 1029, 70]),           # bf16, 32 columns
])
def test_multi_query_matches_oracle_causal_rows(name, nq, lens, bits, kernel):
    w = inp.WORKLOADS[name]
    sc = _scenario(w, 41 + nq, lens, bits, kernel)
    sc.fill()
    q = _queries(7 + nq, sc.B, nq, sc.Hq, sc.dtype)
    out, rc, d = _run(sc, q)
    assert rc == 0, (s4.s4kv_strerror(rc), d)
    _check(sc, q, out, f"{name} nq={nq}")


@pytest.mark.parametrize("bits,kernel", KERNELS)
def test_multi_query_qwen7b_shapes_thirteen_queries(bits, kernel):
    """g = 7, nq = 13: 91 columns; chunks that end just after and just before a
    key-group boundary."""
    w = inp.WORKLOADS["qwen2.5-7b-32k"]
    sc = _scenario(w, 5, [4096 + 5, 2048 - 3, 700, 13], bits, kernel)
    sc.fill()
    q = _queries(3, sc.B, 13, sc.Hq, sc.dtype)
    out, rc, d = _run(sc, q)
    assert rc == 0, (s4.s4kv_strerror(rc), d)
    _check(sc, q, out, "qwen7b nq=13")


# Widths of the tcgen05 kernel's warp roles: 64 columns (two softmax warps, the
# other two restore; the Llama-3.1-8B shapes at nq = 16) and 96, the widest call,
# with g = 8 heads per kv head (three softmax warps, seven restoring warps).
G8 = dataclasses.replace(inp.WORKLOADS["qwen2.5-1.5b"], name="g8", num_q_heads=16)


@pytest.mark.parametrize("bits,kernel", [(4, 0), (4, 3), (2, 3), (8, 0), (8, 3)])
@pytest.mark.parametrize("w,nq,lens", [
    pytest.param(inp.WORKLOADS["llama3.1-8b"], 16, [2000, 515, 1029, 70], id="llama-64cols"),   # bf16
    pytest.param(G8, 12, [1500, 700, 333, 12], id="g8-96cols"),                                 # fp16
])
def test_multi_query_full_widths(w, nq, lens, bits, kernel):
    sc = _scenario(w, 29 + nq, lens, bits, kernel)
    sc.fill()
    q = _queries(11, sc.B, nq, sc.Hq, sc.dtype)
    out, rc, d = _run(sc, q)
    assert rc == 0, (s4.s4kv_strerror(rc), d)
    _check(sc, q, out, f"{w.name} nq={nq}")


def test_single_query_chunk_equals_decode_attention():
    w = inp.WORKLOADS["llama3.1-8b"]
    sc = Scenario(w, 9, [1234, 4000, 77])
    sc.fill()
    q = _queries(2, sc.B, 1, sc.Hq, sc.dtype)
    out, rc, d = _run(sc, q)
    assert rc == 0, (s4.s4kv_strerror(rc), d)
    dec = sc.decode(0, q[:, 0].cuda()).cpu().numpy()
    assert_close(out[:, 0], dec, "nq=1 vs decode")
    _check(sc, q, out, "nq=1")


@pytest.mark.parametrize("bits,nq,kernel", [(4, 6, 0), (4, 11, 0), (4, 6, 3), (8, 6, 1), (8, 6, 3)])   # 36 / 66 columns
@pytest.mark.parametrize("teams", [1, 7, 64])
def test_multi_query_work_partition_does_not_change_the_result(teams, bits, nq, kernel):
    """Few teams split every segment across many slices (merge of many
    partials); the result must not depend on the split."""
    w = inp.WORKLOADS["qwen2.5-1.5b"]
    sc = _scenario(w, 13, [2222, 900, 45], bits, kernel)
    sc.fill()
    sc.cache.set_option(s4.S4KV_OPT_DECODE_WARPS, teams)
    q = _queries(4, sc.B, nq, sc.Hq, sc.dtype)
    out, rc, d = _run(sc, q)
    sc.cache.set_option(s4.S4KV_OPT_DECODE_WARPS, 0)
    assert rc == 0, (s4.s4kv_strerror(rc), d)
    _check(sc, q, out, f"teams={teams}")


@pytest.mark.parametrize("bits", [4, 8])
def test_chunk_longer_than_a_sequence_is_reported(bits):
    w = inp.WORKLOADS["qwen2.5-1.5b"]
    sc = _scenario(w, 17, [500, 3], bits)
    sc.fill()
    q = _queries(5, sc.B, 4, sc.Hq, sc.dtype)
    out, rc, d = _run(sc, q)
    assert rc == s4.S4KV_ERR_DEVICE and d == s4.S4KV_DEV_BAD_LENGTH
    assert not out[1].any()                          # T < nq: zero rows
    s = sc.oracle_seq(0, 0)
    qb = inp.to_bits(q[0])
    for h in range(sc.H):
        ref = s.attention_causal(h, qb[:, h * sc.g:(h + 1) * sc.g], 1 / math.sqrt(128))
        assert_close(out[0, :, h * sc.g:(h + 1) * sc.g], ref, "valid sequence beside a short one")


def test_multi_query_argument_errors():
    w = inp.WORKLOADS["qwen2.5-1.5b"]
    sc = Scenario(w, 19, [300])
    sc.fill()
    with pytest.raises(s4.S4KVError) as e:
        s4.s4kv_multi_query_workspace_bytes(sc.cache.h, 1, 17, sc.Hq, 300)      # nq > 16
    assert e.value.code == s4.S4KV_ERR_INVALID_ARG
    with pytest.raises(s4.S4KVError) as e:
        s4.s4kv_multi_query_workspace_bytes(sc.cache.h, 1, 0, sc.Hq, 300)
    assert e.value.code == s4.S4KV_ERR_INVALID_ARG


@pytest.mark.parametrize("bits,kernel", [(4, 1), (4, 2), (4, 3), (8, 1), (8, 3)])
def test_multi_query_bounded_wait_gives_up_and_the_next_call_is_clean(bits, kernel):
    """A wait limit of 0 makes each multi-query kernel's first wait run out: the
    call reports the timeout (its copies drained, tensor memory freed), and the
    next call with the normal limit matches the oracle."""
    w = inp.WORKLOADS["qwen2.5-1.5b"]
    sc = _scenario(w, 23, [1800, 700, 90], bits, kernel)
    sc.fill()
    q = _queries(6, sc.B, 11, sc.Hq, sc.dtype)      # 66 columns
    sc.cache.set_option(s4.S4KV_OPT_WAIT_NS, 0)
    _, rc, d = _run(sc, q)
    assert rc == s4.S4KV_ERR_DEVICE_TIMEOUT and d == s4.S4KV_DEV_TIMEOUT, (rc, d)
    sc.cache.set_option(s4.S4KV_OPT_WAIT_NS, 1_000_000_000)
    out, rc, d = _run(sc, q)
    assert rc == 0, (s4.s4kv_strerror(rc), d)
    _check(sc, q, out, f"after timeout, kernel {kernel}")
