"""s4kv_decode_attention_noalloc: the decode entry point for callers that cannot
allocate device memory at call time (for example while a CUDA graph is being
captured, or under a fixed memory pool). It uses the library's built-in device
scratch array instead of a caller workspace; its output must match the
workspace entry point's within the parity tolerance, on consecutive calls
(the shared array keeps the previous call's contents).

Named to be collected last, so a run that stops at the first failure has run
every other test before this one.
"""
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
