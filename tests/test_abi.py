"""The C ABI on the CPU: symbols, fail-fast validation, the memory ledger and
the pool layout (no device calls)."""
import ctypes
import json
import os
import re

import pytest

import int4_kivi_quantized_gb300 as s4

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "s4kv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(s4kv_[a-z_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(s4.LIB_PATH)
    names = _declared()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n


def test_fail_fast_on_unsupported_shapes():
    ok = s4.make_config(2, 64, 4, 128, 8)
    s4.s4kv_cache_bytes(ok)
    bad = [dict(head_dim=64), dict(head_dim=256), dict(page_size=32), dict(group_k=16),
           dict(group_v=64)]
    for kw in bad:
        with pytest.raises(s4.S4KVError) as e:
            s4.s4kv_cache_bytes(s4.make_config(2, 64, 4, 128, 8, **kw))
        assert e.value.code == s4.S4KV_ERR_UNSUPPORTED, kw
    for kw in [dict(dtype=7), dict(residual_v=0), dict(residual_v=2000)]:
        cfg = s4.make_config(2, 64, 4, kw.pop("residual_v", 128), 8, **kw)
        with pytest.raises(s4.S4KVError) as e:
            s4.s4kv_cache_bytes(cfg)
        assert e.value.code == s4.S4KV_ERR_UNSUPPORTED
    with pytest.raises(s4.S4KVError) as e:
        s4.s4kv_cache_bytes(s4.make_config(0, 64, 4, 128, 8))
    assert e.value.code == s4.S4KV_ERR_INVALID_ARG


def test_create_rejects_bad_pools_without_touching_the_device():
    cfg = s4.make_config(1, 16, 1, 32, 1)
    with pytest.raises(s4.S4KVError) as e:
        s4.s4kv_cache_create(cfg, None, 1 << 20)
    assert e.value.code == s4.S4KV_ERR_INVALID_ARG
    with pytest.raises(s4.S4KVError) as e:
        s4.s4kv_cache_create(cfg, 0x1000_0010, 1 << 20)   # not 256-byte aligned
    assert e.value.code == s4.S4KV_ERR_INVALID_ARG
    need, _ = s4.s4kv_cache_bytes(cfg)
    with pytest.raises(s4.S4KVError) as e:
        s4.s4kv_cache_create(cfg, 0x1000_0000, need - 1)
    assert e.value.code == s4.S4KV_ERR_POOL_TOO_SMALL


def test_memory_ledger_matches_the_worked_example():
    """M_KV = 2 L B T H_KV d b: 4 GiB at 16 bits for L=32, H_KV=8, d=128,
    T=32768 (section 1 of the KV-cache quantization page); the int4 codes are a
    quarter of that; fp32 scale+min add 8 bytes per key group-channel and per
    value token-group."""
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "mkv_formula.json")))
    cfg = s4.make_config(g["L"], 1, g["H_kv"], 128, 1)
    r = s4.s4kv_kv_bytes(cfg, g["B"], g["T"])
    assert r["fp16_equiv_bytes"] == g["cases"][0]["bytes"] == 4 * 2 ** 30
    assert r["code_bytes"] == 2 ** 30
    k_meta = (32768 // 32) * 128 * 8
    v_meta = (32768 - 128) * 4 * 8
    assert r["meta_bytes"] == 32 * 8 * (k_meta + v_meta)
    assert r["paged_bytes"] == 32 * 8 * 2048 * 3072
    assert r["residual_bytes"] == 32 * 8 * (32 + 128) * 128 * 2
    # density against fp16: codes 0.25x, codes + metadata 0.375x (192 of 512 bytes)
    _, per = s4.s4kv_cache_bytes(cfg)
    assert per == 192
    assert r["paged_bytes"] / r["fp16_equiv_bytes"] == 0.375


def test_two_bit_configuration_ledger_and_layout():
    """2-bit codes (the pages' own KIVI setting): the code bytes are the worked
    example's 0.5 GiB, records shrink to 2048 bytes (128 bytes per token·head),
    metadata is unchanged; any other code width is refused."""
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "mkv_formula.json")))
    cfg = s4.make_config(g["L"], 1, g["H_kv"], 128, 1, bits=2)
    r = s4.s4kv_kv_bytes(cfg, g["B"], g["T"])
    two = next(c for c in g["cases"] if c["bits"] == 2)
    assert r["code_bytes"] == two["bytes"]
    assert r["paged_bytes"] == 32 * 8 * 2048 * 2048
    _, per = s4.s4kv_cache_bytes(cfg)
    assert per == 128
    lay = s4.make_config(1, 10, 2, 64, 4, bits=2)
    pool, _ = s4.s4kv_cache_bytes(lay)
    four, _ = s4.s4kv_cache_bytes(s4.make_config(1, 10, 2, 64, 4))
    assert four - pool == 10 * 2 * 1024
    for bad in (1, 3, 5, 16):
        with pytest.raises(s4.S4KVError) as e:
            s4.s4kv_cache_bytes(s4.make_config(1, 10, 2, 64, 4, bits=bad))
        assert e.value.code == s4.S4KV_ERR_UNSUPPORTED, bad


def test_fp8_configuration_ledger_and_layout():
    """FP8 E4M3 pages (bits = 8): the code bytes are the worked example's 2 GiB
    at 8 bits, records are 4096 bytes (256 bytes per token·head), there is no
    metadata and no ring, and the pool holds one key and one value scale per
    layer and kv head ahead of the layers."""
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "mkv_formula.json")))
    cfg = s4.make_config(g["L"], 1, g["H_kv"], 128, 1, bits=8)
    r = s4.s4kv_kv_bytes(cfg, g["B"], g["T"])
    eight = next(c for c in g["cases"] if c["bits"] == 8)
    assert r["code_bytes"] == eight["bytes"]
    assert r["paged_bytes"] == eight["bytes"]          # one byte per element, pages exactly full
    assert r["meta_bytes"] == 0 and r["residual_bytes"] == 0
    _, per = s4.s4kv_cache_bytes(cfg)
    assert per == 256
    L, P, H, S = 3, 10, 2, 4
    pool8, _ = s4.s4kv_cache_bytes(s4.make_config(L, P, H, 64, S, bits=8))
    pool4, _ = s4.s4kv_cache_bytes(s4.make_config(L, P, H, 64, S))
    rings = S * H * (32 + 64) * 128 * 2
    # per layer: 1024 more page bytes per (page, head), no rings; plus the scale table
    scale_table = -(-(L * 2 * H * 4) // 256) * 256
    layer4 = -(-(P * H * 3072) // 256) * 256 + rings
    layer8 = -(-(P * H * 4096) // 256) * 256
    assert pool8 - pool4 == L * (layer8 - layer4) + scale_table


def test_capacity_tokens_is_the_largest_pool_within_the_budget():
    """Tokens that fit: the page count is the largest whose pool fits the budget
    (one more page would not), and against a 16-bit cache of the same budget
    (M_KV = 2 L B T H_KV d b with b = 2) the quantized pages hold about 512/192
    (4-bit), 512/128 (2-bit) or 512/256 (FP8: the doubling the pages report for
    vLLM's FP8 cache) times the tokens, less the fixed ring overhead."""
    L, H = 32, 8
    budget = 40 * 2 ** 30
    for bits, per in ((4, 192), (2, 128), (8, 256)):
        cfg = s4.make_config(L, 1, H, 128, 64, bits=bits)
        tokens, pages = s4.s4kv_capacity_tokens(cfg, budget)
        assert tokens == 16 * pages
        fit, _ = s4.s4kv_cache_bytes(s4.make_config(L, pages, H, 128, 64, bits=bits))
        over, _ = s4.s4kv_cache_bytes(s4.make_config(L, pages + 1, H, 128, 64, bits=bits))
        assert fit <= budget < over
        fp16_tokens = budget / (2 * L * H * 128 * 2)
        ratio = tokens / fp16_tokens
        assert 0.95 * (512 / per) < ratio < 512 / per, (bits, ratio)
    cfg = s4.make_config(L, 1, H, 128, 64)
    assert s4.s4kv_capacity_tokens(cfg, 1000) == (0, 0)
    with pytest.raises(s4.S4KVError):
        s4.s4kv_capacity_tokens(cfg, -1.0)


def test_layout_is_aligned_and_disjoint():
    cfg = s4.make_config(3, 100, 4, 128, 16, s4.S4KV_BF16)
    need, _ = s4.s4kv_cache_bytes(cfg)
    # a layout needs a handle; build one against a fake (never dereferenced) address
    # through the size function only: recompute the documented layout here
    assert need % 256 == 0
    lay_fields = [f for f, _ in s4.s4kv_layout._fields_]
    assert "kring_offset" in lay_fields and "vring_offset" in lay_fields
