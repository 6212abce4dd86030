"""Quantizer ties through the append kernels (bit-exact against the oracle).

The code of x is rne(fl(fl(x - min) / s)). Rows are built so that many
quotients are exact half-integers (min 0, max 15 * 2^e, so s = 2^e and
x = (k + 1/2) 2^e) or lie within a few units in the last place of one. On
these, a code computed any way other than the IEEE division followed by a
half-to-even rounding (a reciprocal multiply, a rounding of the unrounded
quotient, a rounding that sends halves up) gives other codes. Whole new
32-token tiles (one chunk) and token-by-token appends both go through the
check, for 4- and 2-bit codes and both input formats.
"""
import numpy as np
import pytest
import torch

import int4_kivi_quantized_gb300 as s4
import oracle
import s4kv_inputs as inp

pytestmark = pytest.mark.gpu


def _tie_rows(T, H, bits, dtype, seed):
    """K rows whose channels (over each 32-token group) and V rows whose
    32-channel groups (per token) hold min 0, max levels * 2^e and values at
    or next to (k + 1/2) 2^e."""
    levels = (1 << bits) - 1
    rng = np.random.default_rng(seed)
    tdt = torch.float16 if dtype == "fp16" else torch.bfloat16

    def near_half(shape, e):
        k = rng.integers(0, levels, shape)
        x = (k + 0.5) * 2.0 ** e
        t = torch.from_numpy(x.astype(np.float32)).to(tdt)
        bits16 = t.view(torch.int16).numpy().astype(np.int32)
        step = rng.choice([-1, 0, 0, 0, 1], size=shape)            # mostly exact ties, some 1 ulp off
        return torch.from_numpy((bits16 + step).astype(np.int16)).view(tdt).float().numpy()

    k = np.empty((T, H, 128), np.float32)
    for g0 in range(0, T, 32):
        n = min(32, T - g0)
        for h in range(H):
            e = rng.integers(-6, 4, 128)
            blk = near_half((n, 128), 0)
            blk = blk * (2.0 ** e)[None, :]
            blk[0] = 0.0
            if n > 1:
                blk[1] = levels * 2.0 ** e
            k[g0:g0 + n, h] = blk
    v = np.empty((T, H, 4, 32), np.float32)
    for t in range(T):
        for h in range(H):
            e = rng.integers(-6, 4, 4)
            grp = near_half((4, 32), 0) * (2.0 ** e)[:, None]
            grp[:, 0] = 0.0
            grp[:, 1] = levels * 2.0 ** e
            v[t, h] = grp
    v = v.reshape(T, H, 128)
    return torch.from_numpy(k).to(tdt), torch.from_numpy(v).to(tdt)


@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("mode", ["chunk", "tokens"])
def test_tie_heavy_rows_give_the_oracle_pages(bits, dtype, mode):
    T, H, R = 200, 2, 32
    k, v = _tie_rows(T, H, bits, dtype, 10 * bits + (dtype == "bf16"))
    cache = s4.KVCache(1, 16, H, R, 1, dtype, bits=bits)
    bt = torch.randperm(16, generator=inp.gen(3)).to(torch.int32)[:13][None].cuda()
    kd, vd = k.cuda(), v.cuda()
    cuts = [0, T] if mode == "chunk" else list(range(T + 1))
    for a, b in zip(cuts[:-1], cuts[1:]):
        cache.append(0, kd[a:b], vd[a:b], torch.tensor([0, b - a], dtype=torch.int32).cuda(),
                     torch.tensor([a], dtype=torch.int32).cuda(), bt)
    rc, d = cache.status()
    assert rc == 0, (rc, d)
    s = oracle.Seq(num_kv_heads=H, residual_v=R, dtype=oracle.F16 if dtype == "fp16" else oracle.BF16,
                   bits=bits)
    s.append(inp.to_bits(k), inp.to_bits(v))
    pages, valid = s.page_image(bt[0].cpu().numpy(), 16)
    lay = cache.layout
    got = cache.pool[lay.layer_offset:lay.layer_offset + 16 * lay.page_stride].view(16, H, lay.record_bytes)
    got = got.cpu().numpy()
    diff = (got ^ pages) & valid
    assert not diff.any(), f"page bytes differ at {np.argwhere(diff)[:5]}"
    # the rows really are tie-heavy: many key quotients land exactly on a half-integer
    hist = s.history(0)
    Tk = hist["kscale"].shape[0] * 32
    x = k[:Tk, 0].float().numpy().reshape(-1, 32, 128)
    t = (x - hist["kmin"][:, None, :]) / hist["kscale"][:, None, :]
    assert np.mean(t - np.floor(t) == 0.5) > 0.3
    cache.close()
