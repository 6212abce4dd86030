"""s4kv_decode_step: the append of one token per sequence and decode attention
in one cooperative launch. Against the two separate calls (s4kv_append, then
s4kv_decode_attention) on twin caches fed the same rows: the pages and rings
are bit-identical and so is the output (the attention phase is the same code on
the same state); sampled rows also match the oracle. The steps cross key-group
boundaries (a group completed by the new token is quantized in the launch) and
push value tokens out of the window.
"""
import numpy as np
import pytest
import torch

import int4_kivi_quantized_gb300 as s4
import s4kv_inputs as inp
from gpu_util import Scenario, assert_close

pytestmark = pytest.mark.gpu


def _pool_state(sc):
    lay = sc.cache.layout
    base = lay.layer_offset
    return sc.cache.pool[base:base + lay.layer_stride].cpu().numpy()


def _step_rows(sc, step):
    g = inp.gen(9000 + step)
    k = torch.randn((sc.B, sc.H, 128), generator=g).to(sc.dtype)
    v = torch.randn((sc.B, sc.H, 128), generator=g).to(sc.dtype)
    q = torch.randn((sc.B, sc.Hq, 128), generator=g).to(sc.dtype)
    return k, v, q


def _run_twins(name, lens, steps, bits=4, seed=5, extra=None):
    w = inp.WORKLOADS[name]
    a = Scenario(w, seed, lens, extra_tokens=steps, bits=bits)
    b = Scenario(w, seed, lens, extra_tokens=steps, bits=bits)
    a.fill()
    b.fill()
    for sc in (a, b):
        rc, d = sc.cache.status()
        assert rc == 0, (rc, d)
    ws, ws_bytes = b.cache.workspace(b.B, b.Hq, max(lens) + steps)
    for step in range(steps):
        k, v, q = _step_rows(a, step)
        kd, vd, qd = k.cuda(), v.cuda(), q.cuda()
        before = torch.tensor(a.cur, dtype=torch.int32, device="cuda")
        after = before + 1
        cu = torch.arange(a.B + 1, dtype=torch.int32, device="cuda")
        a.cache.append(0, kd, vd, cu, before, a.bt_dev)
        out_a = a.cache.decode(0, qd, a.bt_dev, after, max(a.cur) + 1)
        out_b = torch.full_like(out_a, float("nan"))
        s4.s4kv_decode_step(b.cache.h, 0, kd, vd, qd, b.Hq, b.bt_dev, b.bt_dev.shape[1], after, None, b.B, 0.0,
                            out_b, s4.S4KV_F32, ws, ws_bytes, max(b.cur) + 1)
        for sc in (a, b):
            for i in range(sc.B):
                sc.hist[(0, i)].append((k[i:i + 1], v[i:i + 1]))
            sc.cur = [x + 1 for x in sc.cur]
        rc, d = b.cache.status()
        assert rc == 0, (s4.s4kv_strerror(rc), d)
        assert torch.equal(out_a, out_b), f"step {step}: output differs from append + decode"
        if extra is not None:
            extra(step, a, b, q, out_b)
    # every defined byte of the two pools agrees (rings and pages), and the
    # pages and rings are the oracle's
    pa, pb = _pool_state(a), _pool_state(b)
    for i in range(a.B):
        oseq = b.check_bytes(0, i)
        a.check_bytes(0, i, oseq)
    return a, b, pa, pb


def test_decode_step_matches_append_then_decode_fp16():
    # Qwen2.5-1.5B-like shapes; lengths chosen so that the steps complete key
    # groups (31, 63 -> 32, 64) and push values out of the window (R = 128)
    lens = [31, 63, 129, 300, 1000, 2047, 5, 128]
    a, b, _, _ = _run_twins("qwen2.5-1.5b", lens, steps=40)
    q = inp.queries(77, b.B, b.Hq, 128, b.dtype)
    out = b.decode(0, q.cuda()).cpu().numpy()
    for i in (0, 3, 7):
        assert_close(out[i], b.oracle_attention(0, i, q), f"seq {i}")


def test_decode_step_matches_append_then_decode_bf16_llama():
    w = inp.WORKLOADS["llama3.1-8b"]
    lens = inp.context_lengths(w, 3).tolist()[:6] + [95, 160]
    _run_twins("llama3.1-8b", lens, steps=33)


@pytest.mark.parametrize("bits", [2, 8])
def test_decode_step_other_page_formats(bits):
    lens = [31, 250, 777, 1]
    _run_twins("qwen2.5-1.5b", lens, steps=34, bits=bits)


def test_decode_step_tiny_window():
    # R = 32: a value token leaves the window at every step once T > 32
    _run_twins("tiny", [255], steps=40)


def test_decode_step_reports_a_wrong_length_and_a_timeout():
    w = inp.WORKLOADS["qwen2.5-1.5b"]
    sc = Scenario(w, 13, [100, 40], extra_tokens=4)
    sc.fill()
    ws, ws_bytes = sc.cache.workspace(sc.B, sc.Hq, 200)
    k, v, q = (t.cuda() for t in _step_rows(sc, 0))
    out = torch.empty((sc.B, sc.Hq, 128), dtype=torch.float32, device="cuda")
    bad = torch.tensor([102, 41], dtype=torch.int32, device="cuda")     # sequence 0 would skip a token
    s4.s4kv_decode_step(sc.cache.h, 0, k, v, q, sc.Hq, sc.bt_dev, sc.bt_dev.shape[1], bad, None, sc.B, 0.0, out,
                        s4.S4KV_F32, ws, ws_bytes, 200)
    rc, d = sc.cache.status()
    assert rc == s4.S4KV_ERR_DEVICE and d == s4.S4KV_DEV_BAD_LENGTH
    # the barrier's wait limit at 0: the first CTAs give up at once; the status
    # reads TIMEOUT and a later call works
    sc2 = Scenario(w, 14, [100, 40], extra_tokens=4)
    sc2.fill()
    sc2.cache.set_option(s4.S4KV_OPT_WAIT_NS, 0)
    after = torch.tensor([101, 41], dtype=torch.int32, device="cuda")
    s4.s4kv_decode_step(sc2.cache.h, 0, k, v, q, sc2.Hq, sc2.bt_dev, sc2.bt_dev.shape[1], after, None, sc2.B, 0.0,
                        out, s4.S4KV_F32, ws, ws_bytes, 200)
    rc, d = sc2.cache.status()
    assert rc == s4.S4KV_ERR_DEVICE_TIMEOUT
    sc2.cache.set_option(s4.S4KV_OPT_WAIT_NS, 1_000_000_000)
    after2 = after + 1
    k2, v2, q2 = (t.cuda() for t in _step_rows(sc2, 1))
    s4.s4kv_decode_step(sc2.cache.h, 0, k2, v2, q2, sc2.Hq, sc2.bt_dev, sc2.bt_dev.shape[1], after2, None, sc2.B,
                        0.0, out, s4.S4KV_F32, ws, ws_bytes, 200)
    rc, d = sc2.cache.status()
    assert rc == 0, (s4.s4kv_strerror(rc), d)
    assert torch.isfinite(out).all()
