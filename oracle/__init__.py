"""ctypes front of the s4kv oracle (``oracle/s4kv_oracle.cpp``).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg may import this module; the library package never does, and
this module imports nothing from it. Inputs reach the oracle as numpy arrays of
raw fp16/bf16 bit patterns (uint16), exactly as they reach the CUDA path.

What the oracle computes, and the passages it follows, is stated in the header
comment of ``s4kv_oracle.cpp``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "s4kv_oracle.cpp")
_LIB = os.path.join(_HERE, "liborc.so")
_lock = threading.Lock()
_lib = None

F16, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle with plain IEEE float semantics (no contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["g++", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c++17", "-fPIC",
             "-shared", _SRC, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


class _Cfg(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "head_dim", "num_kv_heads", "group_k", "group_v", "residual_v", "page_size", "dtype",
        "bits")]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            L.orc_widen.restype = ctypes.c_float
            L.orc_widen.argtypes = [ctypes.c_uint16, ctypes.c_int]
            L.orc_widen_array.argtypes = [P, ctypes.c_long, ctypes.c_int, P]
            L.orc_quantize_group.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P,
                                             P, ctypes.c_int]
            L.orc_dequant.restype = ctypes.c_float
            L.orc_dequant.argtypes = [ctypes.c_int, ctypes.c_float, ctypes.c_float]
            L.orc_mkv_bytes.restype = ctypes.c_double
            L.orc_mkv_bytes.argtypes = [ctypes.c_double] * 6
            L.orc_seq_new.restype = P
            L.orc_seq_new.argtypes = [ctypes.POINTER(_Cfg)]
            L.orc_seq_free.argtypes = [P]
            L.orc_seq_append.argtypes = [P, P, P, ctypes.c_long]
            L.orc_seq_counts.argtypes = [P, P]
            L.orc_seq_history.argtypes = [P, ctypes.c_int, P, P, P, P, P, P]
            L.orc_seq_dequant.argtypes = [P, ctypes.c_int, P, P]
            L.orc_attention_row.argtypes = [P, P, P, ctypes.c_long, ctypes.c_int, ctypes.c_float,
                                            P]
            L.orc_seq_attention.argtypes = [P, ctypes.c_int, P, ctypes.c_int, ctypes.c_float, P]
            L.orc_seq_set_fp8_scales.argtypes = [P, P, P]
            L.orc_seq_set_fp8_scales.restype = None
            L.orc_e4m3_encode.argtypes = [ctypes.c_float]
            L.orc_e4m3_encode.restype = ctypes.c_uint8
            L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.orc_e4m3_decode.restype = ctypes.c_float
            L.orc_seq_attention_causal.argtypes = [P, ctypes.c_int, P, ctypes.c_int, ctypes.c_int, ctypes.c_float, P]
            L.orc_seq_attention_causal.restype = ctypes.c_int
            L.orc_seq_page_image.restype = ctypes.c_int
            L.orc_seq_page_image.argtypes = [P, P, ctypes.c_long, P, P]
            L.orc_seq_ring_image.argtypes = [P, P, P, P, P]
            _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


def widen(bits: np.ndarray, dtype: int) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, np.float32)
    lib().orc_widen_array(_p(bits), bits.size, dtype, _p(out))
    return out


def quantize_group(x: np.ndarray, bits: int = 4):
    """Quantize one group (a 1-D float32 array). Returns (codes u8, scale, min)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    codes = np.zeros(x.size, np.uint8)
    s = np.zeros(1, np.float32)
    m = np.zeros(1, np.float32)
    lib().orc_quantize_group(_p(x), x.size, 1, bits, _p(s), _p(m), _p(codes), 1)
    return codes, np.float32(s[0]), np.float32(m[0])


def e4m3_encode(y: float) -> int:
    """FP8 E4M3 code of y: nearest, ties to even, saturating at 448."""
    return int(lib().orc_e4m3_encode(float(y)))


def e4m3_decode(code: int) -> float:
    return float(lib().orc_e4m3_decode(int(code)))


def dequant(code: int, s: float, mn: float) -> np.float32:
    return np.float32(lib().orc_dequant(int(code), float(s), float(mn)))


def mkv_bytes(L, B, T, H, d, b) -> float:
    return lib().orc_mkv_bytes(L, B, T, H, d, b)


def attention_row(q: np.ndarray, khat: np.ndarray, vhat: np.ndarray, sm_scale: float):
    q = np.ascontiguousarray(q, np.float32)
    khat = np.ascontiguousarray(khat, np.float32)
    vhat = np.ascontiguousarray(vhat, np.float32)
    T, d = khat.shape if khat.size else (0, q.size)
    out = np.empty(q.size, np.float32)
    lib().orc_attention_row(_p(q), _p(khat), _p(vhat), T, q.size, float(sm_scale), _p(out))
    return out


class Seq:
    """One sequence's oracle cache state (all KV heads of one layer)."""

    def __init__(self, head_dim=128, num_kv_heads=1, group_k=32, group_v=32, residual_v=128,
                 page_size=16, dtype=F16, bits=4):
        self.cfg = _Cfg(head_dim, num_kv_heads, group_k, group_v, residual_v, page_size, dtype,
                        bits)
        self.h = lib().orc_seq_new(ctypes.byref(self.cfg))
        if not self.h:
            raise ValueError("oracle rejected the configuration")

    def __del__(self):
        if getattr(self, "h", None):
            lib().orc_seq_free(self.h)
            self.h = None

    @property
    def d(self):
        return self.cfg.head_dim

    @property
    def H(self):
        return self.cfg.num_kv_heads

    def append(self, k_bits: np.ndarray, v_bits: np.ndarray):
        """k_bits, v_bits: uint16 [n, H_kv, d] raw rows."""
        k = np.ascontiguousarray(k_bits, np.uint16)
        v = np.ascontiguousarray(v_bits, np.uint16)
        assert k.shape == v.shape and k.shape[1:] == (self.H, self.d)
        lib().orc_seq_append(self.h, _p(k), _p(v), k.shape[0])

    def counts(self):
        """(T, Tk, Tv, key residual rows, value residual rows)."""
        c = np.zeros(5, np.int64)
        lib().orc_seq_counts(self.h, _p(c))
        return tuple(int(x) for x in c)

    def history(self, head: int):
        T, Tk, Tv, _, _ = self.counts()
        d, G, Gv = self.d, self.cfg.group_k, self.cfg.group_v
        kc = np.zeros((Tk, d), np.uint8)
        ks = np.zeros((Tk // G, d), np.float32)
        km = np.zeros((Tk // G, d), np.float32)
        vc = np.zeros((Tv, d), np.uint8)
        vs = np.zeros((Tv, d // Gv), np.float32)
        vm = np.zeros((Tv, d // Gv), np.float32)
        lib().orc_seq_history(self.h, head, _p(kc), _p(ks), _p(km), _p(vc), _p(vs), _p(vm))
        return dict(kcode=kc, kscale=ks, kmin=km, vcode=vc, vscale=vs, vmin=vm)

    def dequant(self, head: int):
        T = self.counts()[0]
        kh = np.zeros((T, self.d), np.float32)
        vh = np.zeros((T, self.d), np.float32)
        lib().orc_seq_dequant(self.h, head, _p(kh), _p(vh))
        return kh, vh

    def attention(self, head: int, q_bits: np.ndarray, sm_scale: float):
        """q_bits: uint16 [g, d] raw query rows of the g heads reading KV head `head`."""
        q = np.ascontiguousarray(q_bits, np.uint16)
        out = np.zeros(q.shape, np.float32)
        lib().orc_seq_attention(self.h, head, _p(q), q.shape[0], float(sm_scale), _p(out))
        return out

    def set_fp8_scales(self, kscale, vscale):
        """Per-head scales of an FP8 (bits = 8) sequence, before its first append."""
        ks = np.ascontiguousarray(kscale, np.float32)
        vs = np.ascontiguousarray(vscale, np.float32)
        lib().orc_seq_set_fp8_scales(self.h, _p(ks), _p(vs))

    def attention_causal(self, head: int, q_bits: np.ndarray, sm_scale: float):
        """q_bits: uint16 [nq, g, d], the raw query rows of the last nq tokens for
        the g heads reading KV head `head`; query i attends to tokens
        0 .. T - nq + i. Returns fp32 [nq, g, d]."""
        q = np.ascontiguousarray(q_bits, np.uint16)
        nq, g = q.shape[0], q.shape[1]
        out = np.zeros(q.shape, np.float32)
        rc = lib().orc_seq_attention_causal(self.h, head, _p(q), nq, g, float(sm_scale), _p(out))
        if rc != 0:
            raise ValueError(f"causal attention needs 1 <= nq <= T (nq={nq})")
        return out

    def page_image(self, block_table_row: np.ndarray, num_pages: int):
        bt = np.ascontiguousarray(block_table_row, np.int32)
        rec = {4: 3072, 2: 2048, 8: 4096}[self.cfg.bits]
        pages = np.zeros((num_pages, self.H, rec), np.uint8)
        valid = np.zeros((num_pages, self.H, rec), np.uint8)
        rc = lib().orc_seq_page_image(self.h, _p(bt), num_pages, _p(pages), _p(valid))
        if rc != 0:
            raise ValueError(f"page image failed ({rc})")
        return pages, valid

    def ring_image(self):
        G, R, d, H = self.cfg.group_k, self.cfg.residual_v, self.d, self.H
        kr = np.zeros((H, G, d), np.uint16)
        kv = np.zeros((H, G), np.uint8)
        vr = np.zeros((H, max(R, 1), d), np.uint16)
        vv = np.zeros((H, max(R, 1)), np.uint8)
        lib().orc_seq_ring_image(self.h, _p(kr), _p(kv), _p(vr), _p(vv))
        return kr, kv, vr, vv
