"""A decode step (for every layer: append one token per sequence, then decode
attention with the merge kernel launched as a programmatic dependent; or the
same through s4kv_decode_step, a cooperative launch plus the merge launch)
captured in one CUDA graph: replaying it leaves the same cache bytes and the
same outputs, bit for bit, as running the same calls eagerly from the same state.
The calls allocate nothing and take an explicit stream, so they can be
captured once the first eager call has set each kernel's shared-memory limit."""
import pytest
import torch

import int4_kivi_quantized_gb300 as s4
import s4kv_inputs as inp
from gpu_util import Scenario

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("bits", [4, 2, 8])
def test_graph_replay_equals_eager_step(bits, fused):
    """fused: each layer's step through s4kv_decode_step (a cooperative launch and
    the merge launch) instead of s4kv_append + s4kv_decode_attention."""
    w = inp.WORKLOADS["llama3.1-8b"]
    lens = inp.context_lengths(w, 61).tolist()[:12]
    sc = Scenario(w, 61, lens, layers=2, extra_tokens=4, bits=bits)
    sc.fill(keep=False)
    dev = torch.device("cuda")
    B, H, Hq, L = sc.B, sc.H, sc.Hq, 2
    g = torch.Generator(device=dev).manual_seed(5)
    knew = torch.randn((L, B, H, 128), generator=g, device=dev).to(sc.dtype)
    vnew = torch.randn((L, B, H, 128), generator=g, device=dev).to(sc.dtype)
    q = torch.randn((L, B, Hq, 128), generator=g, device=dev).to(sc.dtype)
    out = torch.zeros((L, B, Hq, 128), dtype=torch.float32, device=dev)
    cu = torch.arange(B + 1, dtype=torch.int32, device=dev)
    before = torch.tensor(sc.cur, dtype=torch.int32, device=dev)
    after = before + 1
    max_len = max(sc.cur) + 1
    nbytes = s4.s4kv_decode_workspace_bytes(sc.cache.h, B, Hq, max_len)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    bt = sc.bt_dev

    def step(stream):
        for layer in range(L):
            if fused:
                s4.s4kv_decode_step(sc.cache.h, layer, knew[layer], vnew[layer], q[layer], Hq, bt, bt.shape[1],
                                    after, None, B, 0.0, out[layer], s4.S4KV_F32, ws, nbytes, max_len, stream)
                continue
            s4.s4kv_append(sc.cache.h, layer, knew[layer], vnew[layer], B, cu, None, before, bt, bt.shape[1], B,
                           stream)
            s4.s4kv_decode_attention(sc.cache.h, layer, q[layer], Hq, bt, bt.shape[1], after, None, B, 0.0,
                                     out[layer], s4.S4KV_F32, ws, nbytes, max_len, stream)

    snapshot = sc.cache.pool.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(side)                                   # eager (also sets the kernels' smem limits)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    rc, d = sc.cache.status()
    assert rc == 0, (s4.s4kv_strerror(rc), d)
    eager_out = out.clone()
    eager_pool = sc.cache.pool.clone()

    sc.cache.pool.copy_(snapshot)
    out.zero_()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(torch.cuda.current_stream())
    graph.replay()
    torch.cuda.synchronize()
    rc, d = sc.cache.status()
    assert rc == 0, (s4.s4kv_strerror(rc), d)
    assert torch.equal(out, eager_out)
    lay = sc.cache.layout
    assert torch.equal(sc.cache.pool[lay.lens_offset:], eager_pool[lay.lens_offset:])
