"""Pins of the oracle against facts fixed outside it (CPU only).

Each test checks the oracle against something other than a retyping of its own
formula: values the method's pages print, hand-derived fixtures, closed forms,
textbook routines (numpy's IEEE conversions, a float64 softmax) and brute force.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import s4kv_inputs as inp

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f16_bits(a):
    return np.asarray(a, np.float16).view(np.uint16)


# ---------------------------------------------------------------- widening --
def test_widen_fp16_matches_ieee_for_every_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.widen(bits, oracle.F16)
    ref = bits.view(np.float16).astype(np.float32)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite].view(np.uint32), ref[finite].view(np.uint32))
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))


def test_widen_bf16_matches_torch_for_every_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.widen(bits, oracle.BF16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite].view(np.uint32), ref[finite].view(np.uint32))
    assert np.array_equal(np.isnan(got), np.isnan(ref))


# --------------------------------------------------------------- quantizer --
def test_integer_ramp_is_exact():
    x = np.arange(16, dtype=np.float32)
    codes, s, mn = oracle.quantize_group(x)
    assert s == 1.0 and mn == 0.0
    assert codes.tolist() == list(range(16))
    for c, v in zip(codes, x):
        assert oracle.dequant(c, s, mn) == v


def test_constant_group_round_trips_exactly():
    for v in [0.0, -3.25, 1e-3, 7.0, -0.0]:
        x = np.full(32, v, np.float32)
        codes, s, mn = oracle.quantize_group(x)
        assert s == 0.0 and not codes.any()
        assert oracle.dequant(0, s, mn) == np.float32(v)


def test_two_valued_group_hits_both_ends():
    rng = np.random.default_rng(1)
    for _ in range(200):
        a, b = sorted(rng.normal(size=2).astype(np.float32))
        if a == b:
            continue
        x = rng.choice([a, b], size=32).astype(np.float32)
        x[0], x[1] = a, b
        codes, s, mn = oracle.quantize_group(x)
        assert set(codes.tolist()) <= {0, 15}
        assert codes[0] == 0 and codes[1] == 15
        assert oracle.dequant(0, s, mn) == a
        assert abs(float(oracle.dequant(15, s, mn)) - float(b)) <= 4 * np.spacing(np.float32(abs(b) + abs(a)))


def test_ties_go_to_the_even_code():
    # min 0, max 15 -> scale 1; (x - min) / s lands exactly on .5
    x = np.array([0, 15, 0.5, 1.5, 2.5, 3.5, 14.5, 13.5], np.float32)
    codes, s, mn = oracle.quantize_group(x)
    assert s == 1.0
    assert codes.tolist() == [0, 15, 0, 2, 2, 4, 14, 14]


def test_negative_zero_never_reaches_the_metadata():
    x = np.array([-0.0, 0.0, 1.5, -0.0], np.float32)
    codes, s, mn = oracle.quantize_group(x)
    assert np.float32(mn).view(np.uint32) == 0
    x = np.array([-0.0, -0.0], np.float32)
    codes, s, mn = oracle.quantize_group(x)
    assert np.float32(mn).view(np.uint32) == 0 and s == 0


def test_brute_force_nearest_level_and_error_bound():
    """Codes are the nearest of the 16 levels mn + c*s (checked in float64 by
    enumeration), and |x - x^| <= s/2 + 2 ulp(max |x|)."""
    rng = np.random.default_rng(7)
    for trial in range(3000):
        n = int(rng.integers(1, 33))
        scale = 10.0 ** rng.uniform(-3, 3)
        x = (rng.normal(size=n) * scale).astype(np.float16).astype(np.float32)
        codes, s, mn = oracle.quantize_group(x)
        assert mn == x.min() + np.float32(0)
        if s == 0:
            assert not codes.any()
            continue
        levels = float(mn) + np.arange(16) * float(s)
        for xi, c in zip(x, codes):
            dist = np.abs(float(xi) - levels)
            best = np.min(dist)
            # a different choice is allowed only at a (near) tie, where the fp32
            # quotient decides: then c must be within one level of the argmin
            if dist[c] > best:
                assert dist[c] - best <= 1e-5 * float(s) + 4 * np.spacing(np.float32(abs(xi) + abs(mn)))
            xh = oracle.dequant(c, s, mn)
            ulp = float(np.spacing(np.float32(np.max(np.abs(x)))))
            assert abs(float(xh) - float(xi)) <= float(s) / 2 + 2 * ulp


def test_key_outlier_channel_does_not_widen_other_channels():
    """Per-channel key groups: scaling one channel x10 leaves every other
    channel's (scale, min) bit-identical (section 3.1: the large channel is
    isolated by the vertical grouping)."""
    rng = np.random.default_rng(3)
    k = rng.normal(size=(32, 1, 128)).astype(np.float16)
    v = rng.normal(size=(32, 1, 128)).astype(np.float16)
    a = oracle.Seq(residual_v=0)
    a.append(_f16_bits(k), _f16_bits(v))
    k2 = k.copy()
    k2[:, :, 17] *= np.float16(10)
    b = oracle.Seq(residual_v=0)
    b.append(_f16_bits(k2), _f16_bits(v))
    ha, hb = a.history(0), b.history(0)
    others = [c for c in range(128) if c != 17]
    assert np.array_equal(ha["kscale"][:, others].view(np.uint32), hb["kscale"][:, others].view(np.uint32))
    assert np.array_equal(ha["kmin"][:, others].view(np.uint32), hb["kmin"][:, others].view(np.uint32))
    assert hb["kscale"][0, 17] > 5 * ha["kscale"][0, 17]


def test_value_outlier_only_touches_its_own_channel_group():
    rng = np.random.default_rng(4)
    k = rng.normal(size=(1, 1, 128)).astype(np.float16)
    v = rng.normal(size=(1, 1, 128)).astype(np.float16)
    v2 = v.copy()
    v2[0, 0, 40] = np.float16(30.0)  # channel 40 -> value group 1
    a, b = oracle.Seq(residual_v=0), oracle.Seq(residual_v=0)
    a.append(_f16_bits(k), _f16_bits(v))
    b.append(_f16_bits(k), _f16_bits(v2))
    ha, hb = a.history(0), b.history(0)
    for g in (0, 2, 3):
        assert ha["vscale"][0, g] == hb["vscale"][0, g] and ha["vmin"][0, g] == hb["vmin"][0, g]
    assert hb["vscale"][0, 1] > ha["vscale"][0, 1]


# ----------------------------------------------------------- state machine --
def test_figure_toy_g4_r4_matches_hand_derivation():
    g = json.load(open(os.path.join(GOLDEN, "kivi_figure_g4_r4.json")))
    s = oracle.Seq(head_dim=g["head_dim"], num_kv_heads=1, group_k=g["group_k"],
                   group_v=g["group_v"], residual_v=g["residual_v"], bits=g["bits"])
    k = _f16_bits(np.array(g["k"], np.float32)[:, None, :])
    v = _f16_bits(np.array(g["v"], np.float32)[:, None, :])
    s.append(k, v)
    e = g["expect"]
    assert s.counts() == (e["T"], e["Tk"], e["Tv"], e["k_residual_rows"], e["v_residual_rows"])
    h = s.history(0)
    assert h["kcode"].tolist() == e["kcode"]
    assert np.array_equal(h["kmin"], np.array(e["kmin"], np.float32))
    assert np.array_equal(h["kscale"], np.array(e["kscale"], np.float32))
    assert h["vcode"].tolist() == e["vcode"]
    assert np.array_equal(h["vmin"], np.array(e["vmin"], np.float32))
    assert np.array_equal(h["vscale"], np.array(e["vscale"], np.float32))
    # the residual rows are the newest tokens, untouched
    kh, vh = s.dequant(0)
    assert np.array_equal(kh[8:], np.array(g["k"], np.float32)[8:])
    assert np.array_equal(vh[6:], np.array(g["v"], np.float32)[6:])
    # restored history: code * scale + min
    assert np.array_equal(vh[3], np.full(4, -1, np.float32))
    assert np.array_equal(vh[5], np.array([0, 1.0, 0, 1.5], np.float32))


@pytest.mark.parametrize("G,R", [(32, 128), (32, 32), (4, 4), (16, 0), (32, 5)])
def test_canonical_state_closed_form(G, R):
    """After T tokens: Tk = G*floor(T/G) keys and Tv = max(0, T-R) values are
    quantized, the key residual holds T mod G < G rows and the value residual
    min(T, R). The history equals quantizing the full token matrix directly,
    group by group, whatever the chunking of the appends."""
    rng = np.random.default_rng(G * 1000 + R)
    T = 150
    H = 2
    k = rng.normal(size=(T, H, 128)).astype(np.float16)
    v = rng.normal(size=(T, H, 128)).astype(np.float16)
    s1 = oracle.Seq(num_kv_heads=H, group_k=G, residual_v=R)
    s2 = oracle.Seq(num_kv_heads=H, group_k=G, residual_v=R)
    s1.append(_f16_bits(k), _f16_bits(v))
    o = 0
    while o < T:
        n = int(rng.integers(1, 40))
        s2.append(_f16_bits(k[o:o + n]), _f16_bits(v[o:o + n]))
        o += n
    Tk, Tv = G * (T // G), max(0, T - R)
    assert s1.counts() == (T, Tk, Tv, T % G, min(T, R))
    for h in range(H):
        h1, h2 = s1.history(h), s2.history(h)
        for key in h1:
            assert np.array_equal(h1[key], h2[key]), key
        kf = k[:, h, :].astype(np.float32)
        vf = v[:, h, :].astype(np.float32)
        for grp in range(Tk // G):
            for c in (0, 5, 127):
                codes, sc, mn = oracle.quantize_group(kf[grp * G:(grp + 1) * G, c])
                assert np.array_equal(h1["kcode"][grp * G:(grp + 1) * G, c], codes)
                assert h1["kscale"][grp, c] == sc and h1["kmin"][grp, c] == mn
        for t in range(0, Tv, 7):
            for gv in range(4):
                codes, sc, mn = oracle.quantize_group(vf[t, gv * 32:(gv + 1) * 32])
                assert np.array_equal(h1["vcode"][t, gv * 32:(gv + 1) * 32], codes)
                assert h1["vscale"][t, gv] == sc and h1["vmin"][t, gv] == mn


# ---------------------------------------------------------------- attention --
def _np_attention(q, kh, vh, sm_scale):
    z = (q.astype(np.float64) @ kh.astype(np.float64).T) * float(np.float32(sm_scale))
    z -= z.max(axis=-1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=-1, keepdims=True)
    return p @ vh.astype(np.float64)


def test_attention_unquantized_case_is_textbook():
    """T <= min(R, G-1): nothing is quantized, so the result is plain attention
    over the raw inputs (section 2's P = softmax(QK^T/sqrt d), output PV)."""
    rng = np.random.default_rng(11)
    T, g = 20, 4
    k = rng.normal(size=(T, 1, 128)).astype(np.float16)
    v = rng.normal(size=(T, 1, 128)).astype(np.float16)
    q = rng.normal(size=(g, 128)).astype(np.float16)
    s = oracle.Seq(residual_v=32)
    s.append(_f16_bits(k), _f16_bits(v))
    assert s.counts()[1:3] == (0, 0)
    out = s.attention(0, _f16_bits(q), 1 / math.sqrt(128))
    ref = _np_attention(q.astype(np.float32), k[:, 0].astype(np.float32), v[:, 0].astype(np.float32),
                        1 / math.sqrt(128))
    np.testing.assert_allclose(out, ref, rtol=1e-6, atol=1e-7)


def test_attention_matches_float64_two_pass_softmax_on_dequantized_cache():
    rng = np.random.default_rng(12)
    T, g = 300, 7
    k = (rng.normal(size=(T, 1, 128)) * 3).astype(np.float16)
    v = rng.normal(size=(T, 1, 128)).astype(np.float16)
    q = rng.normal(size=(g, 128)).astype(np.float16)
    s = oracle.Seq(residual_v=128)
    s.append(_f16_bits(k), _f16_bits(v))
    kh, vh = s.dequant(0)
    out = s.attention(0, _f16_bits(q), 0.1)
    ref = _np_attention(q.astype(np.float32), kh, vh, 0.1)
    np.testing.assert_allclose(out, ref, rtol=1e-6, atol=1e-7)
    # the quantized history is really used: raw keys give a different answer
    raw = _np_attention(q.astype(np.float32), k[:, 0].astype(np.float32), v[:, 0].astype(np.float32), 0.1)
    assert np.max(np.abs(raw - out)) > 1e-4


def test_attention_special_cases():
    rng = np.random.default_rng(13)
    # T = 1: the output is the single value row
    s = oracle.Seq(residual_v=0)
    k = rng.normal(size=(1, 1, 128)).astype(np.float16)
    v = rng.normal(size=(1, 1, 128)).astype(np.float16)
    s.append(_f16_bits(k), _f16_bits(v))
    kh, vh = s.dequant(0)
    out = s.attention(0, _f16_bits(rng.normal(size=(2, 128)).astype(np.float16)), 0.3)
    assert np.array_equal(out[0], vh[0]) and np.array_equal(out[1], vh[0])
    # q = 0: uniform weights, the mean of the restored values
    T = 100
    s = oracle.Seq(residual_v=16)
    k = rng.normal(size=(T, 1, 128)).astype(np.float16)
    v = rng.normal(size=(T, 1, 128)).astype(np.float16)
    s.append(_f16_bits(k), _f16_bits(v))
    kh, vh = s.dequant(0)
    out = s.attention(0, _f16_bits(np.zeros((1, 128), np.float16)), 0.1)
    np.testing.assert_allclose(out[0], vh.astype(np.float64).mean(0), rtol=1e-6, atol=1e-7)
    # all keys equal: uniform weights again, whatever q is
    s = oracle.Seq(residual_v=8)
    kc = np.repeat(rng.normal(size=(1, 1, 128)).astype(np.float16), 64, axis=0)
    v = rng.normal(size=(64, 1, 128)).astype(np.float16)
    s.append(_f16_bits(kc), _f16_bits(v))
    kh, vh = s.dequant(0)
    assert np.all(kh == kh[0])
    out = s.attention(0, _f16_bits(rng.normal(size=(3, 128)).astype(np.float16)), 0.2)
    for j in range(3):
        np.testing.assert_allclose(out[j], vh.astype(np.float64).mean(0), rtol=1e-6, atol=1e-7)
    # T = 0: zeros
    s = oracle.Seq()
    out = s.attention(0, _f16_bits(np.ones((2, 128), np.float16)), 0.1)
    assert not out.any()


# ------------------------------------------------------------------ memory --
# ------------------------------------------------- causal multi-query rows --
def _np_causal(q, kh, vh, sm_scale):
    """Textbook causal attention in float64: q [nq, g, d]; query i sees the
    first T - nq + i + 1 rows of kh, vh."""
    nq, g, _ = q.shape
    T = kh.shape[0]
    out = np.zeros(q.shape, np.float64)
    for i in range(nq):
        n = T - nq + i + 1
        z = float(np.float32(sm_scale)) * (q[i].astype(np.float64) @ kh[:n].astype(np.float64).T)
        z -= z.max(axis=1, keepdims=True)
        p = np.exp(z)
        out[i] = (p @ vh[:n].astype(np.float64)) / p.sum(axis=1, keepdims=True)
    return out


def test_causal_rows_unquantized_case_is_textbook():
    """Nothing quantized (T < G, T <= R): the chunk's rows are plain causal
    attention over the raw inputs."""
    rng = np.random.default_rng(21)
    T, nq, g = 25, 6, 3
    k = rng.normal(size=(T, 1, 128)).astype(np.float16)
    v = rng.normal(size=(T, 1, 128)).astype(np.float16)
    q = rng.normal(size=(nq, g, 128)).astype(np.float16)
    s = oracle.Seq(residual_v=32)
    s.append(_f16_bits(k), _f16_bits(v))
    assert s.counts()[1:3] == (0, 0)
    out = s.attention_causal(0, _f16_bits(q), 1 / math.sqrt(128))
    ref = _np_causal(q.astype(np.float32), k[:, 0].astype(np.float32), v[:, 0].astype(np.float32),
                     1 / math.sqrt(128))
    np.testing.assert_allclose(out, ref, rtol=1e-6, atol=1e-7)


def test_causal_single_query_is_decode_attention():
    rng = np.random.default_rng(22)
    T, g = 333, 4
    k = (rng.normal(size=(T, 1, 128)) * 2).astype(np.float16)
    v = rng.normal(size=(T, 1, 128)).astype(np.float16)
    q = rng.normal(size=(1, g, 128)).astype(np.float16)
    s = oracle.Seq(residual_v=64)
    s.append(_f16_bits(k), _f16_bits(v))
    np.testing.assert_array_equal(s.attention_causal(0, _f16_bits(q), 0.1)[0], s.attention(0, _f16_bits(q[0]), 0.1))


def test_causal_rows_ignore_tokens_after_their_position():
    """Changing only the last token (still in both rings, so no quantization
    group sees it) leaves every earlier query's row bit-identical and changes
    the last row."""
    rng = np.random.default_rng(23)
    T, nq, g = 301, 5, 2
    k = rng.normal(size=(T, 1, 128)).astype(np.float16)
    v = rng.normal(size=(T, 1, 128)).astype(np.float16)
    q = rng.normal(size=(nq, g, 128)).astype(np.float16)
    k2, v2 = k.copy(), v.copy()
    k2[-1] *= -3
    v2[-1] += 5
    a, b = oracle.Seq(residual_v=128), oracle.Seq(residual_v=128)
    a.append(_f16_bits(k), _f16_bits(v))
    b.append(_f16_bits(k2), _f16_bits(v2))
    assert T % 32 != 0   # the last key is in the key ring
    oa = a.attention_causal(0, _f16_bits(q), 0.09)
    ob = b.attention_causal(0, _f16_bits(q), 0.09)
    np.testing.assert_array_equal(oa[:-1], ob[:-1])
    assert np.abs(oa[-1] - ob[-1]).max() > 1e-3


def test_causal_rows_match_masked_float64_softmax_on_dequantized_cache():
    rng = np.random.default_rng(24)
    T, nq, g = 700, 16, 4
    k = (rng.normal(size=(T, 1, 128)) * 3).astype(np.float16)
    v = rng.normal(size=(T, 1, 128)).astype(np.float16)
    q = rng.normal(size=(nq, g, 128)).astype(np.float16)
    s = oracle.Seq(residual_v=128)
    s.append(_f16_bits(k), _f16_bits(v))
    kh, vh = s.dequant(0)
    out = s.attention_causal(0, _f16_bits(q), 1 / math.sqrt(128))
    ref = _np_causal(q.astype(np.float32), kh, vh, 1 / math.sqrt(128))
    np.testing.assert_allclose(out, ref, rtol=2e-6, atol=2e-7)
    with pytest.raises(ValueError):
        s.attention_causal(0, _f16_bits(np.zeros((T + 1, g, 128), np.float16)), 0.1)


def test_memory_formula_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "mkv_formula.json")))
    for c in g["cases"]:
        got = oracle.mkv_bytes(g["L"], g["B"], g["T"], g["H_kv"], g["d"], c["bits"] / 8)
        assert got == c["bytes"]
    assert g["cases"][0]["bytes"] == 4 * 2 ** 30


# -------------------------------------------------------------- page image --
def _read_page_image(pages, bt, T, Tk, Tv, H):
    """Reads codes and metadata back from a page image, following the byte
    format stated in include/s4kv.h (independent of the oracle's writer)."""
    kc = np.zeros((H, Tk, 128), np.uint8)
    ks = np.zeros((H, Tk // 32, 128), np.float32)
    km = np.zeros((H, Tk // 32, 128), np.float32)
    vc = np.zeros((H, Tv, 128), np.uint8)
    vs = np.zeros((H, Tv, 4), np.float32)
    vm = np.zeros((H, Tv, 4), np.float32)
    for h in range(H):
        for t in range(Tk):
            rec = pages[bt[t // 16], h]
            tau = t % 16
            for c in range(128):
                lane = 4 * (tau % 8) + c // 32
                kk = (c % 32) // 4
                byte = {0: 0, 1: 2, 2: 1, 3: 3}[c % 4]
                b = rec[(kk // 4) * 512 + lane * 16 + (kk % 4) * 4 + byte]
                kc[h, t, c] = (b >> 4) if tau >= 8 else (b & 15)
        for grp in range(Tk // 32):
            for c in range(128):
                rec = pages[bt[2 * grp + c // 64], h]
                cl = c % 64
                off = 1024 + (2 * ((cl % 32) // 4) + cl // 32) * 16 + 4 * (cl % 4)
                ks[h, grp, c] = rec[off:off + 4].view(np.float32)[0]
                km[h, grp, c] = rec[off + 256:off + 260].view(np.float32)[0]
        for t in range(Tv):
            rec = pages[bt[t // 16], h]
            tau = t % 16
            b_ = (tau % 8) // 2
            byte = {(0, 0): 0, (1, 0): 1, (0, 1): 2, (1, 1): 3}[(tau // 8, tau % 2)]
            for c in range(128):
                lane = 4 * (c % 8) + b_
                mt = c // 16
                bb = rec[1536 + (mt // 4) * 512 + lane * 16 + (mt % 4) * 4 + byte]
                vc[h, t, c] = (bb >> 4) if (c % 16) >= 8 else (bb & 15)
            e = tau % 2 + 2 * (tau // 8)
            for k in range(4):
                o1 = 2560 + ((2 * k) * 4 + b_) * 16 + 4 * e
                o2 = 2560 + ((2 * k + 1) * 4 + b_) * 16 + 4 * e
                vs[h, t, k] = rec[o1:o1 + 4].view(np.float32)[0]
                vm[h, t, k] = rec[o2:o2 + 4].view(np.float32)[0]
    return kc, ks, km, vc, vs, vm


def test_page_image_round_trips_through_the_stated_format():
    rng = np.random.default_rng(21)
    H, T = 2, 77
    k = rng.normal(size=(T, H, 128)).astype(np.float16)
    v = rng.normal(size=(T, H, 128)).astype(np.float16)
    s = oracle.Seq(num_kv_heads=H, residual_v=20)
    s.append(_f16_bits(k), _f16_bits(v))
    _, Tk, Tv, _, _ = s.counts()
    npages = 12
    bt = rng.permutation(npages)[:5].astype(np.int32)
    pages, valid = s.page_image(bt, npages)
    kc, ks, km, vc, vs, vm = _read_page_image(pages, bt, T, Tk, Tv, H)
    for h in range(H):
        hist = s.history(h)
        assert np.array_equal(kc[h], hist["kcode"])
        assert np.array_equal(ks[h], hist["kscale"]) and np.array_equal(km[h], hist["kmin"])
        assert np.array_equal(vc[h], hist["vcode"])
        assert np.array_equal(vs[h], hist["vscale"]) and np.array_equal(vm[h], hist["vmin"])
    # defined bytes: 64 code bytes per key token, 1 KiB of key metadata per group,
    # 64 code bytes + 32 metadata bytes per value token
    ones = np.unpackbits(valid).sum() // 8
    assert ones == H * (Tk * 64 + (Tk // 32) * 1024 + Tv * 96)
    # pages outside the table are untouched
    unused = sorted(set(range(npages)) - set(bt.tolist()))
    assert not valid[unused].any()


def _read_page_image_2bit(pages, bt, Tk, Tv, H):
    """Reads codes and metadata back from a 2-bit page image (2048-byte records),
    following the byte format stated in include/s4kv.h."""
    kc = np.zeros((H, Tk, 128), np.uint8)
    ks = np.zeros((H, Tk // 32, 128), np.float32)
    km = np.zeros((H, Tk // 32, 128), np.float32)
    vc = np.zeros((H, Tv, 128), np.uint8)
    vs = np.zeros((H, Tv, 4), np.float32)
    vm = np.zeros((H, Tv, 4), np.float32)
    for h in range(H):
        for t in range(Tk):
            rec = pages[bt[t // 16], h]
            tau = t % 16
            for c in range(128):
                kk = (c % 32) // 4
                byte = {0: 0, 1: 2, 2: 1, 3: 3}[c % 4]
                b = rec[(4 * (tau % 8) + c // 32) * 16 + (kk // 2) * 4 + byte]
                pos = 2 * (kk % 2) + (tau // 8)
                kc[h, t, c] = (b >> (2 * pos)) & 3
        for grp in range(Tk // 32):
            for c in range(128):
                rec = pages[bt[2 * grp + c // 64], h]
                cl = c % 64
                off = 512 + (2 * ((cl % 32) // 4) + cl // 32) * 16 + 4 * (cl % 4)
                ks[h, grp, c] = rec[off:off + 4].view(np.float32)[0]
                km[h, grp, c] = rec[off + 256:off + 260].view(np.float32)[0]
        for t in range(Tv):
            rec = pages[bt[t // 16], h]
            tau = t % 16
            b_ = (tau % 8) // 2
            byte = {(0, 0): 0, (1, 0): 1, (0, 1): 2, (1, 1): 3}[(tau // 8, tau % 2)]
            for c in range(128):
                bb = rec[1024 + (4 * (c % 8) + b_) * 16 + (c // 32) * 4 + byte]
                vc[h, t, c] = (bb >> (2 * ((c % 32) // 8))) & 3
            e = tau % 2 + 2 * (tau // 8)
            for k in range(4):
                o1 = 1536 + ((2 * k) * 4 + b_) * 16 + 4 * e
                o2 = 1536 + ((2 * k + 1) * 4 + b_) * 16 + 4 * e
                vs[h, t, k] = rec[o1:o1 + 4].view(np.float32)[0]
                vm[h, t, k] = rec[o2:o2 + 4].view(np.float32)[0]
    return kc, ks, km, vc, vs, vm


def test_page_image_2bit_round_trips_through_the_stated_format():
    rng = np.random.default_rng(25)
    H, T = 2, 93
    k = rng.normal(size=(T, H, 128)).astype(np.float16)
    v = rng.normal(size=(T, H, 128)).astype(np.float16)
    s = oracle.Seq(num_kv_heads=H, residual_v=20, bits=2)
    s.append(_f16_bits(k), _f16_bits(v))
    _, Tk, Tv, _, _ = s.counts()
    npages = 14
    bt = rng.permutation(npages)[:6].astype(np.int32)
    pages, valid = s.page_image(bt, npages)
    assert pages.shape[-1] == 2048
    kc, ks, km, vc, vs, vm = _read_page_image_2bit(pages, bt, Tk, Tv, H)
    for h in range(H):
        hist = s.history(h)
        assert hist["kcode"].max() == 3 and hist["vcode"].max() == 3
        assert np.array_equal(kc[h], hist["kcode"])
        assert np.array_equal(ks[h], hist["kscale"]) and np.array_equal(km[h], hist["kmin"])
        assert np.array_equal(vc[h], hist["vcode"])
        assert np.array_equal(vs[h], hist["vscale"]) and np.array_equal(vm[h], hist["vmin"])
    # 32 code bytes per key token, 1 KiB of key metadata per group, 32 code
    # bytes + 32 metadata bytes per value token
    ones = np.unpackbits(valid).sum() // 8
    assert ones == H * (Tk * 32 + (Tk // 32) * 1024 + Tv * 64)
    unused = sorted(set(range(npages)) - set(bt.tolist()))
    assert not valid[unused].any()


def test_ring_image_positions():
    rng = np.random.default_rng(22)
    T, R = 45, 10
    k = rng.normal(size=(T, 1, 128)).astype(np.float16)
    v = rng.normal(size=(T, 1, 128)).astype(np.float16)
    s = oracle.Seq(residual_v=R)
    s.append(_f16_bits(k), _f16_bits(v))
    kr, kv, vr, vv = s.ring_image()
    kb, vb = _f16_bits(k), _f16_bits(v)
    assert kv[0].sum() == T % 32 and vv[0].sum() == R
    for t in range(32 * (T // 32), T):
        assert np.array_equal(kr[0, t % 32], kb[t, 0])
    for t in range(T - R, T):
        assert np.array_equal(vr[0, t % R], vb[t, 0])


def test_inputs_are_seeded_and_shaped():
    w = inp.WORKLOADS["qwen2.5-1.5b"]
    assert inp.outlier_count(0.02) == 3 and inp.outlier_count(0.01) == 1
    o = inp.outlier_channels(5, 0, w.num_kv_heads, 128, 3)
    k1, v1 = inp.kv_rows(9, 40, 2, 128, torch.float16, o, 8.0)
    k2, v2 = inp.kv_rows(9, 40, 2, 128, torch.float16, o, 8.0)
    assert torch.equal(k1, k2) and torch.equal(v1, v2)
    sd = k1.float().std(dim=(0,))
    for h in range(2):
        others = [c for c in range(128) if c not in o[h].tolist()]
        assert sd[h, o[h]].min() > 3 * sd[h, others].mean()
    lens = inp.context_lengths(w, 1)
    assert lens.min() >= 2048 and lens.max() <= 4096
    bt = inp.block_tables("fragmented", 4, [3, 5, 1, 2], 64, 1)
    used = bt[bt >= 0]
    assert used.numel() == 11 and used.unique().numel() == 11


def test_dequant_is_one_rounding_of_the_exact_value():
    """x^ = code * scale + min rounded once (a fused multiply-add): checked on
    cases where float64 holds code*scale + min exactly, so rounding that float64
    to float32 is the single correct rounding."""
    from fractions import Fraction
    rng = np.random.default_rng(5)
    hits = diffs = 0
    for _ in range(20000):
        c = int(rng.integers(0, 16))
        s = np.float32(rng.uniform(0, 1) * 10.0 ** rng.uniform(-2, 1))
        mn = np.float32(rng.normal() * 10.0 ** rng.uniform(-2, 1))
        exact = Fraction(c) * Fraction(float(s)) + Fraction(float(mn))
        f64 = float(c) * float(s) + float(mn)
        if Fraction(f64) != exact:
            continue
        hits += 1
        want = np.float32(f64)
        got = oracle.dequant(c, s, mn)
        assert got.view(np.uint32) == want.view(np.uint32)
        if np.float32(np.float32(c) * s) + mn != want:
            diffs += 1
    assert hits > 10000
    assert diffs > 0   # some cases separate one rounding from two
