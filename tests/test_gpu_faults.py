"""Failure detection without a GPU fault.

Bad caller data (a block-table entry outside the pool, a length that disagrees
with the cache, a slot out of range, malformed cu_new) is made on the host and
handed to the kernels, which check it before any access and report it through
the status word. The bounded-wait path is exercised by setting the wait limit
to 0, so the first mbarrier wait gives up at once; the copies already in flight
are drained, the status reads TIMEOUT, and the next call works normally.
"""
import numpy as np
import pytest
import torch

import int4_kivi_quantized_gb300 as s4
import s4kv_inputs as inp
from gpu_util import Scenario, assert_close

pytestmark = pytest.mark.gpu


def _small(seed=7, lens=(300, 1000, 77)):
    w = inp.WORKLOADS["qwen2.5-1.5b"]
    sc = Scenario(w, seed, list(lens), slack_pages=4)
    sc.fill()
    rc, d = sc.cache.status()
    assert rc == 0, (rc, d)
    return sc


def _good_decode_matches_oracle(sc, seed=1):
    q = inp.queries(seed, sc.B, sc.Hq, 128, sc.dtype)
    out = sc.decode(0, q.cuda()).cpu().numpy()
    rc, d = sc.cache.status()
    assert rc == 0, (rc, d)
    for b in range(sc.B):
        assert_close(out[b], sc.oracle_attention(0, b, q), f"seq {b}")


def test_block_table_entry_outside_the_pool_is_reported():
    sc = _small()
    bad = sc.bt_dev.clone()
    bad[1, 3] = sc.num_pages + 5
    q = inp.queries(1, sc.B, sc.Hq, 128, sc.dtype).cuda()
    seq = torch.tensor(sc.cur, dtype=torch.int32, device="cuda")
    sc.cache.decode(0, q, bad, seq, max(sc.cur))
    rc, detail = sc.cache.status()
    assert rc == s4.S4KV_ERR_DEVICE and detail == s4.S4KV_DEV_BAD_PAGE
    bad[1, 3] = -2
    sc.cache.decode(0, q, bad, seq, max(sc.cur))
    rc, detail = sc.cache.status()
    assert rc == s4.S4KV_ERR_DEVICE and detail == s4.S4KV_DEV_BAD_PAGE
    _good_decode_matches_oracle(sc)   # status cleared, cache intact


def test_length_that_disagrees_with_the_cache_is_reported():
    sc = _small()
    q = inp.queries(2, sc.B, sc.Hq, 128, sc.dtype).cuda()
    seq = torch.tensor([sc.cur[0], sc.cur[1] - 1, sc.cur[2]], dtype=torch.int32, device="cuda")
    out = sc.cache.decode(0, q, sc.bt_dev, seq, max(sc.cur))
    rc, detail = sc.cache.status()
    assert rc == s4.S4KV_ERR_DEVICE and detail == s4.S4KV_DEV_BAD_LENGTH
    assert not out[1].any()          # the mismatched sequence's rows stay zero
    # append with a wrong seq_lens_before is reported too
    k, v = inp.kv_rows(3, 1, sc.H, 128, sc.dtype)
    sc.cache.append(0, k.cuda(), v.cuda(), torch.tensor([0, 1], dtype=torch.int32, device="cuda"),
                    torch.tensor([sc.cur[0] + 3], dtype=torch.int32, device="cuda"), sc.bt_dev[:1])
    rc, detail = sc.cache.status()
    assert rc == s4.S4KV_ERR_DEVICE and detail == s4.S4KV_DEV_BAD_LENGTH
    # a longer sequence than max_seq_len is refused
    seq = torch.tensor(sc.cur, dtype=torch.int32, device="cuda")
    sc.cache.decode(0, q, sc.bt_dev, seq, max(sc.cur) - 1)
    rc, detail = sc.cache.status()
    assert rc == s4.S4KV_ERR_DEVICE and detail == s4.S4KV_DEV_BAD_LENGTH


def test_slot_out_of_range_and_malformed_cu_new_are_reported():
    sc = _small()
    k, v = inp.kv_rows(4, 2, sc.H, 128, sc.dtype)
    kd, vd = k.cuda(), v.cuda()
    slots = torch.tensor([sc.B + 3], dtype=torch.int32, device="cuda")
    s4.s4kv_append(sc.cache.h, 0, kd, vd, 2, torch.tensor([0, 2], dtype=torch.int32, device="cuda"),
                   slots, torch.tensor([0], dtype=torch.int32, device="cuda"), sc.bt_dev,
                   sc.bt_dev.shape[1], 1)
    rc, detail = sc.cache.status()
    assert rc == s4.S4KV_ERR_DEVICE and detail == s4.S4KV_DEV_BAD_SLOT
    # cu_new total disagrees with num_new_tokens: nothing is read or written
    before = sc.cache.pool.clone()
    s4.s4kv_append(sc.cache.h, 0, kd, vd, 2, torch.tensor([0, 5], dtype=torch.int32, device="cuda"),
                   None, torch.tensor([sc.cur[0]], dtype=torch.int32, device="cuda"), sc.bt_dev,
                   sc.bt_dev.shape[1], 1)
    rc, detail = sc.cache.status()
    assert rc == s4.S4KV_ERR_DEVICE and detail == s4.S4KV_DEV_BAD_CU
    lay = sc.cache.layout
    assert torch.equal(before[lay.layer_offset:], sc.cache.pool[lay.layer_offset:])
    _good_decode_matches_oracle(sc)


def test_bounded_wait_gives_up_and_the_next_call_is_clean():
    sc = _small(lens=(3000, 2500, 4000))
    sc.cache.set_option(s4.S4KV_OPT_WAIT_NS, 0)
    q = inp.queries(5, sc.B, sc.Hq, 128, sc.dtype).cuda()
    seq = torch.tensor(sc.cur, dtype=torch.int32, device="cuda")
    sc.cache.decode(0, q, sc.bt_dev, seq, max(sc.cur))
    rc, detail = sc.cache.status()
    assert rc == s4.S4KV_ERR_DEVICE_TIMEOUT and detail == s4.S4KV_DEV_TIMEOUT
    sc.cache.set_option(s4.S4KV_OPT_WAIT_NS, 1_000_000_000)
    _good_decode_matches_oracle(sc, seed=5)   # nothing from the aborted call carries over


def test_host_side_argument_errors_launch_nothing():
    sc = _small()
    q = inp.queries(1, sc.B, sc.Hq, 128, sc.dtype).cuda()
    seq = torch.tensor(sc.cur, dtype=torch.int32, device="cuda")
    out = torch.empty((sc.B, sc.Hq, 128), dtype=torch.float32, device="cuda")
    ws, nbytes = sc.cache.workspace(sc.B, sc.Hq, max(sc.cur))
    bt = sc.bt_dev
    def call(**kw):
        args = dict(h=sc.cache.h, layer=0, q=q, num_q_heads=sc.Hq, block_table=bt, bt_stride=bt.shape[1],
                    seq_lens=seq, slot_ids=None, B=sc.B, sm_scale=0.0, out=out, out_dtype=s4.S4KV_F32,
                    workspace=ws, ws_bytes=nbytes, max_seq_len=max(sc.cur))
        args.update(kw)
        s4.s4kv_decode_attention(**args)
    with pytest.raises(s4.S4KVError) as e:
        call(q=q.data_ptr() + 2)                       # misaligned
    assert e.value.code == s4.S4KV_ERR_INVALID_ARG
    with pytest.raises(s4.S4KVError) as e:
        call(layer=1)                                  # no such layer
    assert e.value.code == s4.S4KV_ERR_INVALID_ARG
    with pytest.raises(s4.S4KVError) as e:
        call(num_q_heads=sc.H * 9)                     # GQA group 9 > 8
    assert e.value.code == s4.S4KV_ERR_UNSUPPORTED
    with pytest.raises(s4.S4KVError) as e:
        call(out_dtype=s4.S4KV_BF16)                   # not the cache dtype
    assert e.value.code == s4.S4KV_ERR_INVALID_ARG
    with pytest.raises(s4.S4KVError) as e:
        call(ws_bytes=nbytes - 16)
    assert e.value.code == s4.S4KV_ERR_WORKSPACE_TOO_SMALL
    with pytest.raises(s4.S4KVError) as e:
        call(seq_lens=None)
    assert e.value.code == s4.S4KV_ERR_INVALID_ARG
    rc, d = sc.cache.status()
    assert rc == 0
    _good_decode_matches_oracle(sc)


def test_dequant_debug_reports_a_length_mismatch():
    sc = _small()
    kh, vh = sc.cache.dequant(0, 0, sc.bt_dev[0], sc.cur[0] - 1)
    rc, detail = sc.cache.status()
    assert rc == s4.S4KV_ERR_DEVICE and detail == s4.S4KV_DEV_BAD_LENGTH
