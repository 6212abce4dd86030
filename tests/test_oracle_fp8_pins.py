"""Pins of the oracle's FP8 E4M3 page mode (bits = 8) against things outside it:
torch's float8_e4m3fn conversions (an independent implementation of the same
format), closed forms of the format ("4.4 KV Cache 量化", sections 4.1 and 4.2:
the fp8_e4m3 KV type with a per-attention-head scale), a float64 softmax over
the restored cache, and an inverse reader of the stated record layout."""
import math

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _f16_bits(a):
    return np.ascontiguousarray(a, np.float16).view(np.uint16)


def _torch_e4m3(x: np.ndarray) -> np.ndarray:
    """float32 -> e4m3 code bytes through torch (round to nearest even)."""
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def _torch_e4m3_value(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn)
    return t.float().numpy()


def test_decode_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ref = _torch_e4m3_value(codes)
    got = np.array([oracle.e4m3_decode(c) for c in codes], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2   # 0x7f and 0xff
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_decode_closed_forms():
    assert oracle.e4m3_decode(0x7E) == 448.0          # 1.75 * 2^8, the largest finite
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9       # smallest subnormal
    assert oracle.e4m3_decode(0x08) == 2.0 ** -6       # smallest normal
    assert oracle.e4m3_decode(0x38) == 1.0             # exponent field 7 = bias
    assert math.copysign(1.0, oracle.e4m3_decode(0x80)) == -1.0


def test_every_finite_value_encodes_to_its_own_code():
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c, hex(c)


def test_midpoints_go_to_the_even_code():
    """Halfway between two neighbouring magnitudes the even mantissa wins; just
    off the midpoint the nearer one wins."""
    for c in range(0, 0x7E):
        lo, hi = oracle.e4m3_decode(c), oracle.e4m3_decode(c + 1)
        mid = np.float32((lo + hi) / 2)            # exact: both are short dyadic numbers
        assert float(mid) == (lo + hi) / 2
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(mid) == even, hex(c)
        assert oracle.e4m3_encode(-mid) == 0x80 | even
        below = np.nextafter(mid, np.float32(0))
        above = np.nextafter(mid, np.float32(np.inf))
        assert oracle.e4m3_encode(below) == c and oracle.e4m3_encode(above) == c + 1


def test_encode_matches_torch_on_random_values_below_448():
    rng = np.random.default_rng(3)
    mag = np.exp2(rng.uniform(-14, math.log2(447.9), 200000)).astype(np.float32)
    x = (mag * rng.choice([-1, 1], mag.size)).astype(np.float32)
    got = np.array([oracle.e4m3_encode(v) for v in x[:20000]], np.uint8)
    assert np.array_equal(got, _torch_e4m3(x[:20000]))


def test_saturation_signed_zero_and_nan():
    assert oracle.e4m3_encode(448.0) == 0x7E
    assert oracle.e4m3_encode(463.9) == 0x7E and oracle.e4m3_encode(1e30) == 0x7E
    assert oracle.e4m3_encode(float("inf")) == 0x7E and oracle.e4m3_encode(float("-inf")) == 0xFE
    assert oracle.e4m3_encode(-1000.0) == 0xFE
    assert oracle.e4m3_encode(0.0) == 0x00 and oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(-1e-30) == 0x80                 # underflow keeps the sign
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00             # tie between 0 and 2^-9: even (0)
    assert oracle.e4m3_encode(3 * 2.0 ** -10) == 0x02         # tie between 1 and 2 (x 2^-9): even
    assert oracle.e4m3_encode(float("nan")) & 0x7F == 0x7F


def _fp8_seq(T, H, seed, kscale, vscale, dtype=np.float16):
    rng = np.random.default_rng(seed)
    k = (rng.normal(size=(T, H, 128)) * 4).astype(dtype)
    v = rng.normal(size=(T, H, 128)).astype(dtype)
    s = oracle.Seq(num_kv_heads=H, bits=8)
    s.set_fp8_scales(kscale, vscale)
    s.append(_f16_bits(k), _f16_bits(v))
    return s, k, v


def test_fp8_sequence_restores_through_torch_rounding():
    """Every token is stored at once (no residual), as e4m3(x / scale) with the
    division rounded to float32 first; restored as value(code) * scale."""
    H, T = 3, 77
    ks = np.array([1.0, 0.015625, 3.5], np.float32)
    vs = np.array([1.0, 0.01, 2.0], np.float32)
    s, k, v = _fp8_seq(T, H, 9, ks, vs)
    assert s.counts() == (T, T, T, 0, 0)
    for h in range(H):
        kq = k[:, h].astype(np.float32) / ks[h]
        vq = v[:, h].astype(np.float32) / vs[h]
        hist = s.history(h)
        kh, vh = s.dequant(h)
        for x, code, restored, sc in ((kq, hist["kcode"], kh, ks[h]), (vq, hist["vcode"], vh, vs[h])):
            # torch's cast is not saturating (NaN from 480 up): compare below 448,
            # and check the saturated code above it
            inside = np.abs(x) < 448
            ref = _torch_e4m3(np.where(inside, x, 0))
            assert np.array_equal(code[inside], ref[inside])
            assert np.array_equal(code[~inside], np.where(x[~inside] > 0, 0x7E, 0xFE).astype(np.uint8))
            want = np.where(inside, _torch_e4m3_value(ref), np.sign(x) * 448).astype(np.float32) * sc
            assert np.array_equal(restored, want)
    # head 1's keys exceed 448 / 64 = 7 somewhere: those saturate
    assert (s.history(1)["kcode"] & 0x7F == 0x7E).any()


def test_fp8_attention_is_float64_softmax_over_the_restored_cache():
    H, T, g = 2, 130, 4
    s, k, v = _fp8_seq(T, H, 10, np.array([0.5, 1.0], np.float32), np.array([1.0, 0.25], np.float32))
    rng = np.random.default_rng(11)
    q = rng.normal(size=(g, 128)).astype(np.float16)
    for h in range(H):
        kh, vh = s.dequant(h)
        out = s.attention(h, _f16_bits(q), 1 / math.sqrt(128))
        z = (q.astype(np.float64) @ kh.astype(np.float64).T) * float(np.float32(1 / math.sqrt(128)))
        p = np.exp(z - z.max(axis=-1, keepdims=True))
        ref = (p / p.sum(axis=-1, keepdims=True)) @ vh.astype(np.float64)
        np.testing.assert_allclose(out, ref, rtol=1e-6, atol=1e-7)
        # E4M3 keeps 3 mantissa bits: the restored cache is within 2^-4 relative of
        # the input wherever nothing saturates or underflows
        ok = np.abs(k[:, h].astype(np.float32)) > 0.1
        rel = np.abs(kh[ok] - k[:, h][ok]) / np.abs(k[:, h][ok])
        assert rel.max() <= 2.0 ** -4 + 1e-7


def _read_fp8_record(rec):
    """Inverse of the stated FP8 record layout: every byte offset is decoded to
    the (token, channel) it holds. Keys [0, 2048): word (kp, L) at kp*512 + 16L,
    L = 4a + b; its bytes 8u .. 8u+7 hold slice kk = 2kp + u, byte
    8u + 4(j div 2) + 2 hi + (j mod 2) is token a + 8 hi of channel 32b + 4kk + j.
    Values [2048, 4096): same words; bytes 8u .. 8u+7 hold channel tile
    mt = 2kp + u; byte 8u + 4w + 2 up + r is channel 16mt + a + 8up of token
    2b + r + 8w."""
    kc = np.full((16, 128), -1, np.int32)
    vc = np.full((16, 128), -1, np.int32)
    for half, out in ((0, kc), (1, vc)):
        for off in range(2048):
            kp, rem = divmod(off, 512)
            L, byte = divmod(rem, 16)
            a, b = divmod(L, 4)
            u, inner = divmod(byte, 8)
            hi4, lo2 = divmod(inner, 4)
            mid, low = divmod(lo2, 2)
            if half == 0:
                tok, ch = a + 8 * mid, 32 * b + 4 * (2 * kp + u) + 2 * hi4 + low
            else:
                tok, ch = 2 * b + low + 8 * hi4, 16 * (2 * kp + u) + a + 8 * mid
            assert out[tok, ch] == -1, "two bytes claim one element"
            out[tok, ch] = rec[2048 * half + off]
    return kc, vc


def test_fp8_page_image_round_trips_through_the_stated_format():
    H, T = 2, 53
    s, _, _ = _fp8_seq(T, H, 12, np.ones(H, np.float32), np.ones(H, np.float32))
    npages = 9
    bt = np.random.default_rng(4).permutation(npages)[:4].astype(np.int32)
    pages, valid = s.page_image(bt, npages)
    assert pages.shape == (npages, H, 4096)
    for h in range(H):
        hist = s.history(h)
        for lp in range(4):
            kc, vc = _read_fp8_record(pages[bt[lp], h])
            n = min(16, T - 16 * lp)
            assert np.array_equal(kc[:n], hist["kcode"][16 * lp:16 * lp + n])
            assert np.array_equal(vc[:n], hist["vcode"][16 * lp:16 * lp + n])
    # one key byte and one value byte per element of every stored token
    assert (valid == 0xFF).sum() == H * T * 256 and ((valid != 0) & (valid != 0xFF)).sum() == 0
    unused = sorted(set(range(npages)) - set(bt.tolist()))
    assert not valid[unused].any()
