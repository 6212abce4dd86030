"""s4kv_decode_attention_noalloc: the decode entry point for callers that cannot
allocate device memory at call time (for example while a CUDA graph is being
captured, or under a fixed memory pool). It uses the library's built-in device
scratch array instead of a caller workspace; its output must match the
workspace entry point's within the parity tolerance, on consecutive calls
(the shared array keeps the previous call's contents).

Named to be collected last, so a run that stops at the first failure has run
every other test before this one.
"""
import ctypes

import numpy as np
import pytest
import torch

import int4_kivi_quantized_gb300 as s4
import s4kv_inputs as inp
from gpu_util import Scenario, assert_close

pytestmark = pytest.mark.gpu


def _noalloc(sc, q, out_dtype=s4.S4KV_F32):
    B, Hq, _ = q.shape
    dt = torch.float32 if out_dtype == s4.S4KV_F32 else sc.dtype
    out = torch.full((B, Hq, 128), float("nan"), dtype=dt, device=q.device)
    seq = torch.tensor(sc.cur, dtype=torch.int32, device=q.device)
    s4.s4kv_decode_attention_noalloc(sc.cache.h, 0, q, Hq, sc.bt_dev, sc.bt_dev.shape[1], seq, None,
                                     B, 0.0, out, out_dtype, max(sc.cur))
    return out


@pytest.mark.parametrize("name,seed", [("qwen2.5-1.5b", 3), ("llama3.1-8b", 5)])
def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(name, seed):
    w = inp.WORKLOADS[name]
    lens = inp.context_lengths(w, seed).tolist()[:8]
    sc = Scenario(w, seed, lens)
    sc.fill()
    for call in range(2):
        q = inp.queries(seed * 10 + call, sc.B, sc.Hq, 128, sc.dtype).cuda()
        ref = sc.decode(0, q).cpu().numpy()
        got = _noalloc(sc, q).cpu().numpy()
        rc, detail = sc.cache.status()
        assert rc == 0, (s4.s4kv_strerror(rc), detail)
        assert np.isfinite(got).all()
        assert_close(got, ref, f"{name} call {call}")


def test_noalloc_after_a_larger_call_on_another_cache():
    """Stale scratch: a call with many sequences and long contexts (many split
    segments, many partials) is followed by calls with fewer, shorter, other
    sequences on another cache, then by the large one again. Each output is
    compared with the workspace entry point's (bit for bit: the same kernels
    on the same partition) and with the oracle on sampled rows."""
    big_w = inp.WORKLOADS["llama3.1-8b"]
    big = Scenario(big_w, 41, inp.context_lengths(big_w, 41).tolist())          # 32 sequences
    big.fill()
    small_w = inp.WORKLOADS["qwen2.5-1.5b"]
    small = Scenario(small_w, 43, [37, 1500, 160, 4096, 1])
    small.fill()
    plan = [(big, 0), (small, 1), (small, 2), (big, 3)]
    for sc, k in plan:
        q = inp.queries(700 + k, sc.B, sc.Hq, 128, sc.dtype)
        ref = sc.decode(0, q.cuda()).cpu().numpy()
        got = _noalloc(sc, q.cuda()).cpu().numpy()
        rc, detail = sc.cache.status()
        assert rc == 0, (s4.s4kv_strerror(rc), detail)
        assert np.array_equal(got, ref), f"call {k}: differs from the workspace entry point"
        for b in (0, sc.B - 1):
            assert_close(got[b], sc.oracle_attention(0, b, q), f"call {k} seq {b}")


def test_noalloc_rejects_a_call_whose_scratch_exceeds_the_array():
    """A call that would need more than S4KV_NOALLOC_SCRATCH_BYTES returns
    S4KV_ERR_WORKSPACE_TOO_SMALL and launches nothing: the output buffer keeps
    its contents."""
    limit = 16 << 20
    w = inp.WORKLOADS["llama3.1-8b"]
    sc = Scenario(w, 47, [64, 65])
    sc.fill()
    # the FFMA decode path keeps more partials per SM; find a shape beyond the limit
    sc.cache.set_option(s4.S4KV_OPT_DECODE_IMPL, 1)
    Hq = 64   # 8 query heads per kv head
    need = s4.s4kv_decode_workspace_bytes(sc.cache.h, 4096, Hq, 128)
    if need <= limit:
        pytest.skip(f"no decode shape needs more than the scratch array here ({need} bytes)")
    q = torch.zeros((4096, Hq, 128), dtype=sc.dtype, device="cuda")
    out = torch.full((4096, Hq, 128), 7.0, dtype=torch.float32, device="cuda")
    seq = torch.zeros(4096, dtype=torch.int32, device="cuda")
    bt = torch.zeros((4096, 8), dtype=torch.int32, device="cuda")
    L = s4._lib
    rc = L.s4kv_decode_attention_noalloc(sc.cache.h, 0, ctypes.c_void_p(q.data_ptr()), Hq,
                                         ctypes.c_void_p(bt.data_ptr()), 8, ctypes.c_void_p(seq.data_ptr()),
                                         None, 4096, ctypes.c_float(0.0), ctypes.c_void_p(out.data_ptr()),
                                         s4.S4KV_F32, 128, None)
    assert rc == s4.S4KV_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
    rc, detail = sc.cache.status()
    assert rc == 0
