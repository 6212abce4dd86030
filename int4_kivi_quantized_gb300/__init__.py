"""Python binding of libs4kv.so, the int4 KIVI-style paged KV cache for GB300.

Argument marshalling only: every step of the path runs in the library's CUDA
kernels. Functions carry the C ABI's names (include/s4kv.h); pointer arguments
accept a torch tensor (its data_ptr), an int address or None; `stream` accepts a
torch.cuda.Stream, an int handle or None (the current torch stream).

There is no fallback: if the shared library is missing or fails to load,
importing this package raises.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libs4kv.so")

S4KV_OK = 0
S4KV_ERR_INVALID_ARG = 1
S4KV_ERR_UNSUPPORTED = 2
S4KV_ERR_CUDA = 3
S4KV_ERR_POOL_TOO_SMALL = 4
S4KV_ERR_DEVICE = 5
S4KV_ERR_DEVICE_TIMEOUT = 6
S4KV_ERR_WORKSPACE_TOO_SMALL = 7

S4KV_F16, S4KV_BF16, S4KV_F32 = 0, 1, 2

S4KV_DEV_BAD_PAGE, S4KV_DEV_BAD_LENGTH, S4KV_DEV_BAD_SLOT = 1, 2, 3
S4KV_DEV_BAD_TABLE, S4KV_DEV_BAD_CU, S4KV_DEV_TIMEOUT = 4, 5, 6

S4KV_OPT_DECODE_WARPS, S4KV_OPT_DECODE_IMPL, S4KV_OPT_WAIT_NS, S4KV_OPT_TAIL_COST = 1, 2, 3, 4
S4KV_OPT_KEY_SPLIT = 5
S4KV_OPT_MQ_KERNEL = 6


class S4KVError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {s4kv_strerror(code)} (status {code})")
        self.code = code


class s4kv_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "num_layers", "num_pages", "page_size", "num_kv_heads", "head_dim", "group_k", "group_v",
        "residual_v", "max_slots", "dtype", "bits")]


class s4kv_layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in (
        "pool_bytes", "status_offset", "lens_offset", "layer_offset", "layer_stride", "page_stride",
        "record_bytes", "kcode_offset", "kmeta_offset", "vcode_offset", "vmeta_offset",
        "kring_offset", "kring_slot_stride", "kring_head_stride", "kring_row_stride",
        "vring_offset", "vring_slot_stride", "vring_head_stride", "vring_row_stride", "scale_offset")]


class s4kv_kv_bytes_report(ctypes.Structure):
    _fields_ = [(n, ctypes.c_double) for n in (
        "fp16_equiv_bytes", "code_bytes", "meta_bytes", "residual_bytes", "paged_bytes")]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                          "(or python int4_kivi_quantized_gb300/build.py)")
    L = ctypes.CDLL(LIB_PATH)
    P, I, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    sig = {
        "s4kv_cache_bytes": [ctypes.POINTER(s4kv_config), ctypes.POINTER(SZ), ctypes.POINTER(SZ)],
        "s4kv_cache_create": [ctypes.POINTER(s4kv_config), P, SZ, ctypes.POINTER(P)],
        "s4kv_cache_destroy": [P],
        "s4kv_get_layout": [P, ctypes.POINTER(s4kv_layout)],
        "s4kv_append": [P, I, P, P, I, P, P, P, P, I, I, P],
        "s4kv_decode_workspace_bytes": [P, I, I, I, ctypes.POINTER(SZ)],
        "s4kv_decode_attention": [P, I, P, I, P, I, P, P, I, ctypes.c_float, P, I, P, SZ, I, P],
        "s4kv_decode_attention_noalloc": [P, I, P, I, P, I, P, P, I, ctypes.c_float, P, I, I, P],
        "s4kv_decode_step": [P, I, P, P, P, I, P, I, P, P, I, ctypes.c_float, P, I, P, SZ, I, P],
        "s4kv_multi_query_workspace_bytes": [P, I, I, I, I, ctypes.POINTER(SZ)],
        "s4kv_multi_query_attention": [P, I, P, I, I, P, I, P, P, I, ctypes.c_float, P, I, P, SZ, I, P],
        "s4kv_dequant_debug": [P, I, I, P, I, P, P, P],
        "s4kv_get_status": [P, P, ctypes.POINTER(I)],
        "s4kv_kv_bytes": [ctypes.POINTER(s4kv_config), ctypes.c_double, ctypes.c_double,
                          ctypes.POINTER(s4kv_kv_bytes_report)],
        "s4kv_set_option": [P, I, ctypes.c_longlong],
        "s4kv_capacity_tokens": [ctypes.POINTER(s4kv_config), ctypes.c_double, ctypes.POINTER(ctypes.c_longlong),
                                 ctypes.POINTER(ctypes.c_longlong)],
        "s4kv_set_fp8_scales": [P, I, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_float), P],
    }
    for name, args in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = I
    L.s4kv_strerror.argtypes = [I]
    L.s4kv_strerror.restype = ctypes.c_char_p
    return L


_lib = _load()


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return ctypes.c_void_p(x)
    return ctypes.c_void_p(x.data_ptr())


def _stream(s):
    if s is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(s, int):
        return ctypes.c_void_p(s)
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc: int, what: str):
    if rc != S4KV_OK:
        raise S4KVError(rc, what)


def s4kv_strerror(code: int) -> str:
    return _lib.s4kv_strerror(int(code)).decode()


def make_config(num_layers, num_pages, num_kv_heads, residual_v, max_slots, dtype=S4KV_F16,
                head_dim=128, page_size=16, group_k=32, group_v=32, bits=4) -> s4kv_config:
    return s4kv_config(num_layers, num_pages, page_size, num_kv_heads, head_dim, group_k, group_v,
                       residual_v, max_slots, dtype, bits)


def s4kv_capacity_tokens(cfg: s4kv_config, budget_bytes: float):
    """(tokens, pages) of KV that fit in budget_bytes for this configuration."""
    t, p = ctypes.c_longlong(), ctypes.c_longlong()
    _check(_lib.s4kv_capacity_tokens(ctypes.byref(cfg), float(budget_bytes), ctypes.byref(t), ctypes.byref(p)),
           "s4kv_capacity_tokens")
    return t.value, p.value


def s4kv_cache_bytes(cfg: s4kv_config):
    pool = ctypes.c_size_t()
    per = ctypes.c_size_t()
    _check(_lib.s4kv_cache_bytes(ctypes.byref(cfg), ctypes.byref(pool), ctypes.byref(per)),
           "s4kv_cache_bytes")
    return pool.value, per.value


def s4kv_kv_bytes(cfg: s4kv_config, batch: float, tokens: float) -> dict:
    r = s4kv_kv_bytes_report()
    _check(_lib.s4kv_kv_bytes(ctypes.byref(cfg), float(batch), float(tokens), ctypes.byref(r)),
           "s4kv_kv_bytes")
    return {n: getattr(r, n) for n, _ in r._fields_}


def s4kv_cache_create(cfg: s4kv_config, pool, pool_bytes: int):
    h = ctypes.c_void_p()
    _check(_lib.s4kv_cache_create(ctypes.byref(cfg), _ptr(pool), int(pool_bytes), ctypes.byref(h)),
           "s4kv_cache_create")
    return h


def s4kv_set_fp8_scales(h, layer, k_scale, v_scale, stream=None):
    """FP8 pools: per-kv-head key and value scales of one layer (host sequences)."""
    ks = (ctypes.c_float * len(k_scale))(*[float(x) for x in k_scale])
    vs = (ctypes.c_float * len(v_scale))(*[float(x) for x in v_scale])
    _check(_lib.s4kv_set_fp8_scales(h, int(layer), ks, vs, _stream(stream)), "s4kv_set_fp8_scales")


def s4kv_cache_destroy(h):
    _check(_lib.s4kv_cache_destroy(h), "s4kv_cache_destroy")


def s4kv_get_layout(h) -> s4kv_layout:
    lay = s4kv_layout()
    _check(_lib.s4kv_get_layout(h, ctypes.byref(lay)), "s4kv_get_layout")
    return lay


def s4kv_set_option(h, option: int, value: int):
    _check(_lib.s4kv_set_option(h, int(option), int(value)), "s4kv_set_option")


def s4kv_append(h, layer, k, v, num_new_tokens, cu_new, slot_ids, seq_lens_before, block_table,
                bt_stride, n, stream=None):
    _check(_lib.s4kv_append(h, int(layer), _ptr(k), _ptr(v), int(num_new_tokens), _ptr(cu_new),
                            _ptr(slot_ids), _ptr(seq_lens_before), _ptr(block_table),
                            int(bt_stride), int(n), _stream(stream)), "s4kv_append")


def s4kv_decode_workspace_bytes(h, B, num_q_heads, max_seq_len) -> int:
    out = ctypes.c_size_t()
    _check(_lib.s4kv_decode_workspace_bytes(h, int(B), int(num_q_heads), int(max_seq_len),
                                            ctypes.byref(out)), "s4kv_decode_workspace_bytes")
    return out.value


def s4kv_decode_attention(h, layer, q, num_q_heads, block_table, bt_stride, seq_lens, slot_ids, B,
                          sm_scale, out, out_dtype, workspace, ws_bytes, max_seq_len, stream=None):
    _check(_lib.s4kv_decode_attention(h, int(layer), _ptr(q), int(num_q_heads), _ptr(block_table),
                                      int(bt_stride), _ptr(seq_lens), _ptr(slot_ids), int(B),
                                      float(sm_scale), _ptr(out), int(out_dtype), _ptr(workspace),
                                      int(ws_bytes), int(max_seq_len), _stream(stream)),
           "s4kv_decode_attention")


def s4kv_multi_query_workspace_bytes(h, B, num_q_tokens, num_q_heads, max_seq_len) -> int:
    out = ctypes.c_size_t()
    _check(_lib.s4kv_multi_query_workspace_bytes(h, int(B), int(num_q_tokens), int(num_q_heads),
                                                 int(max_seq_len), ctypes.byref(out)),
           "s4kv_multi_query_workspace_bytes")
    return out.value


def s4kv_multi_query_attention(h, layer, q, num_q_tokens, num_q_heads, block_table, bt_stride, seq_lens,
                               slot_ids, B, sm_scale, out, out_dtype, workspace, ws_bytes, max_seq_len,
                               stream=None):
    _check(_lib.s4kv_multi_query_attention(h, int(layer), _ptr(q), int(num_q_tokens), int(num_q_heads),
                                           _ptr(block_table), int(bt_stride), _ptr(seq_lens), _ptr(slot_ids),
                                           int(B), float(sm_scale), _ptr(out), int(out_dtype), _ptr(workspace),
                                           int(ws_bytes), int(max_seq_len), _stream(stream)),
           "s4kv_multi_query_attention")


def s4kv_decode_step(h, layer, k_new, v_new, q, num_q_heads, block_table, bt_stride, seq_lens, slot_ids, B,
                     sm_scale, out, out_dtype, workspace, ws_bytes, max_seq_len, stream=None):
    """One token appended per sequence and decode attention over the result, in one launch."""
    _check(_lib.s4kv_decode_step(h, int(layer), _ptr(k_new), _ptr(v_new), _ptr(q), int(num_q_heads),
                                 _ptr(block_table), int(bt_stride), _ptr(seq_lens), _ptr(slot_ids), int(B),
                                 float(sm_scale), _ptr(out), int(out_dtype), _ptr(workspace), int(ws_bytes),
                                 int(max_seq_len), _stream(stream)), "s4kv_decode_step")


def s4kv_decode_attention_noalloc(h, layer, q, num_q_heads, block_table, bt_stride, seq_lens, slot_ids,
                                  B, sm_scale, out, out_dtype, max_seq_len, stream=None):
    """Decode attention with the library's built-in device scratch (no workspace)."""
    _check(_lib.s4kv_decode_attention_noalloc(h, int(layer), _ptr(q), int(num_q_heads),
                                              _ptr(block_table), int(bt_stride), _ptr(seq_lens),
                                              _ptr(slot_ids), int(B), float(sm_scale), _ptr(out),
                                              int(out_dtype), int(max_seq_len), _stream(stream)),
           "s4kv_decode_attention_noalloc")


def s4kv_dequant_debug(h, layer, slot, block_table_row, seq_len, out_k, out_v, stream=None):
    _check(_lib.s4kv_dequant_debug(h, int(layer), int(slot), _ptr(block_table_row), int(seq_len),
                                   _ptr(out_k), _ptr(out_v), _stream(stream)), "s4kv_dequant_debug")


def s4kv_get_status(h, stream=None):
    """Returns (status, detail); does not raise on a device-side status."""
    detail = ctypes.c_int(0)
    rc = _lib.s4kv_get_status(h, _stream(stream), ctypes.byref(detail))
    return rc, detail.value


class KVCache:
    """A cache bound to a torch-allocated device pool (torch provides memory only)."""

    def __init__(self, num_layers, num_pages, num_kv_heads, residual_v, max_slots, dtype="fp16",
                 device="cuda", bits=4):
        import torch
        self.dtype = dtype
        self.cdtype = S4KV_F16 if dtype == "fp16" else S4KV_BF16
        self.torch_dtype = torch.float16 if dtype == "fp16" else torch.bfloat16
        self.bits = bits
        self.cfg = make_config(num_layers, num_pages, num_kv_heads, residual_v, max_slots,
                               self.cdtype, bits=bits)
        self.pool_bytes, self.bytes_per_token_head = s4kv_cache_bytes(self.cfg)
        # 256-byte alignment is guaranteed by the caching allocator
        self.pool = torch.empty(self.pool_bytes, dtype=torch.uint8, device=device)
        self.h = s4kv_cache_create(self.cfg, self.pool, self.pool_bytes)
        self.layout = s4kv_get_layout(self.h)
        self.H = num_kv_heads
        self.R = residual_v
        self._ws = None

    def close(self):
        if getattr(self, "h", None):
            s4kv_cache_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_option(self, option, value):
        s4kv_set_option(self.h, option, value)

    def set_fp8_scales(self, layer, k_scale, v_scale, stream=None):
        """FP8 pools (bits=8): key and value scale of every kv head of `layer`."""
        if len(k_scale) != self.H or len(v_scale) != self.H:
            raise ValueError("one key and one value scale per kv head")
        s4kv_set_fp8_scales(self.h, layer, k_scale, v_scale, stream)

    def append(self, layer, k, v, cu_new, seq_lens_before, block_table, slot_ids=None, stream=None):
        n = seq_lens_before.numel()
        s4kv_append(self.h, layer, k, v, k.shape[0], cu_new, slot_ids, seq_lens_before,
                    block_table, block_table.shape[1], n, stream)

    def workspace(self, B, num_q_heads, max_seq_len):
        import torch
        nbytes = s4kv_decode_workspace_bytes(self.h, B, num_q_heads, max_seq_len)
        if self._ws is None or self._ws.numel() < nbytes:
            self._ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=self.pool.device)
        return self._ws, nbytes

    def decode(self, layer, q, block_table, seq_lens, max_seq_len, out=None, out_dtype=S4KV_F32,
               slot_ids=None, sm_scale=0.0, stream=None):
        import torch
        B, Hq, _ = q.shape
        if out is None:
            dt = torch.float32 if out_dtype == S4KV_F32 else self.torch_dtype
            out = torch.empty((B, Hq, 128), dtype=dt, device=q.device)
        ws, nbytes = self.workspace(B, Hq, max_seq_len)
        s4kv_decode_attention(self.h, layer, q, Hq, block_table, block_table.shape[1], seq_lens,
                              slot_ids, B, sm_scale, out, out_dtype, ws, nbytes, max_seq_len, stream)
        return out

    def multi_query(self, layer, q, block_table, seq_lens, max_seq_len, out=None, out_dtype=S4KV_F32,
                    slot_ids=None, sm_scale=0.0, stream=None):
        """Causal attention of the last nq tokens: q [B, nq, H_q, 128] -> out [B, nq, H_q, 128]."""
        import torch
        B, nq, Hq, _ = q.shape
        if out is None:
            dt = torch.float32 if out_dtype == S4KV_F32 else self.torch_dtype
            out = torch.empty((B, nq, Hq, 128), dtype=dt, device=q.device)
        nbytes = s4kv_multi_query_workspace_bytes(self.h, B, nq, Hq, max_seq_len)
        if self._ws is None or self._ws.numel() < nbytes:
            self._ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=self.pool.device)
        s4kv_multi_query_attention(self.h, layer, q, nq, Hq, block_table, block_table.shape[1], seq_lens,
                                   slot_ids, B, sm_scale, out, out_dtype, self._ws, nbytes, max_seq_len, stream)
        return out

    def dequant(self, layer, slot, block_table_row, seq_len, stream=None):
        import torch
        k = torch.empty((self.H, seq_len, 128), dtype=torch.float32, device=self.pool.device)
        v = torch.empty_like(k)
        s4kv_dequant_debug(self.h, layer, slot, block_table_row, seq_len, k, v, stream)
        return k, v

    def status(self, stream=None):
        return s4kv_get_status(self.h, stream)
