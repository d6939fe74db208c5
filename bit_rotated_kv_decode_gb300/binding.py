"""Thin ctypes binding of the C ABI in include/oscar.h (argument marshalling only).

Every computation runs in the CUDA library; this module only converts Python
objects (torch tensors, numpy arrays, ints) into the pointers and sizes the C
functions take, and raises ``OscarError`` on a non-OK status.  Importing it
loads the library and fails loudly if it has not been built.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_float, c_int32, c_int64, c_size_t, c_uint64, c_void_p

import numpy as np

from .build import LIB

OSCAR_OK = 0
OSCAR_ERR_INVALID_ARG = 1
OSCAR_ERR_OUT_OF_PAGES = 2
OSCAR_ERR_STATE = 3
OSCAR_ERR_CUDA = 4
OSCAR_ERR_TIMEOUT = 5
OSCAR_ERR_DEVICE_CHECK = 6
OSCAR_ERR_DRY_RUN = 7
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "OUT_OF_PAGES", 3: "STATE", 4: "CUDA", 5: "TIMEOUT",
                6: "DEVICE_CHECK", 7: "DRY_RUN"}

HEAD_DIM = 128
RECORD_BYTES = 4608
BF16_PAGES_PER_REQUEST = 5


class oscar_cache_config(ctypes.Structure):
    _fields_ = [("num_layers", c_int32), ("num_q_heads", c_int32), ("num_kv_heads", c_int32),
                ("head_dim", c_int32), ("sink_tokens", c_int32), ("recent_tokens", c_int32),
                ("page_tokens", c_int32), ("group_size", c_int32), ("max_requests", c_int32),
                ("max_pages_per_request", c_int32), ("num_int2_pages", c_int64), ("num_bf16_pages", c_int64),
                ("softmax_scale", c_float), ("page_perm_seed", c_uint64)]


class oscar_cache_layout(ctypes.Structure):
    _fields_ = [(name, c_size_t) for name in (
        "total_bytes", "int2_pool_offset", "int2_layer_stride", "int2_page_stride", "int2_record_bytes",
        "bf16_pool_offset", "bf16_layer_stride", "bf16_page_stride", "bf16_record_bytes",
        "rot_k_offset", "rot_v_offset", "rot_kt_offset", "rot_vt_offset", "rot_colnorm_offset",
        "tau_k_offset", "tau_v_offset",
        "hist_pt_offset", "bf16_pt_offset", "error_word_offset", "decode_count_offset", "decode_flag_offset")]


class OscarError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_P = c_void_p
_SIGNATURES = {
    "oscar_version": (c_char_p, []),
    "oscar_cache_device_bytes": (c_size_t, [POINTER(oscar_cache_config)]),
    "oscar_cache_create": (c_int32, [POINTER(oscar_cache_config), _P, c_size_t, _P, _P, POINTER(c_float),
                                     POINTER(c_float), _P, POINTER(_P)]),
    "oscar_cache_destroy": (c_int32, [_P]),
    "oscar_cache_get_layout": (c_int32, [_P, POINTER(oscar_cache_layout)]),
    "oscar_request_open": (c_int32, [_P, _P, POINTER(c_int32)]),
    "oscar_request_fork": (c_int32, [_P, c_int32, c_int64, _P, POINTER(c_int32)]),
    "oscar_request_close": (c_int32, [_P, c_int32]),
    "oscar_request_length": (c_int32, [_P, c_int32, c_int32, POINTER(c_int64), POINTER(c_int64)]),
    "oscar_request_pages": (c_int32, [_P, c_int32, POINTER(c_int32), c_int32, POINTER(c_int32), POINTER(c_int32)]),
    "oscar_cache_free_pages": (c_int32, [_P, POINTER(c_int64), POINTER(c_int64)]),
    "oscar_prefill_quantize": (c_int32, [_P, c_int32, c_int32, _P, _P, c_int64, _P]),
    "oscar_append": (c_int32, [_P, c_int32, c_int32, POINTER(c_int32), _P, _P, _P]),
    "oscar_demote": (c_int32, [_P, c_int32, c_int32, POINTER(c_int32), _P]),
    "oscar_demote_layers": (c_int32, [_P, c_int32, c_int32, c_int32, POINTER(c_int32), _P]),
    "oscar_decode_workspace_bytes": (c_int32, [_P, c_int32, POINTER(c_int32), POINTER(c_size_t)]),
    "oscar_decode_attention": (c_int32, [_P, c_int32, c_int32, POINTER(c_int32), _P, _P, _P, c_size_t, _P]),
    "oscar_decode_attention_noalloc": (c_int32, [_P, c_int32, c_int32, POINTER(c_int32), _P, _P, _P]),
    "oscar_decode_step": (c_int32, [_P, c_int32, c_int32, POINTER(c_int32), _P, _P, _P, _P, _P, c_size_t, _P]),
    "oscar_cache_check": (c_int32, [_P, _P]),
    "oscar_debug_decode_hooks": (c_int32, [_P, ctypes.c_uint32, c_int32]),
    "oscar_last_error": (c_char_p, [_P]),
    "oscar_bf16_decode_workspace_bytes": (c_size_t, [c_int32, POINTER(c_int32), c_int32, c_int32]),
    "oscar_bf16_decode": (c_int32, [_P, c_int64, _P, c_int32, POINTER(c_int32), c_int32, c_int32, c_int32, c_float,
                                    _P, _P, _P, c_size_t, _P]),
}

_lib = None


def load(path: str = LIB) -> ctypes.CDLL:
    """Load the CUDA library (once); raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library {path} is missing: run bit_rotated_kv_decode_gb300.build.build()")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def exported_symbols() -> list[str]:
    return list(_SIGNATURES)


def make_config(num_layers, num_q_heads, num_kv_heads, max_requests, max_pages_per_request, num_int2_pages,
                num_bf16_pages=0, softmax_scale=0.0, page_perm_seed=0, group_size=128) -> oscar_cache_config:
    return oscar_cache_config(num_layers, num_q_heads, num_kv_heads, HEAD_DIM, 64, 256, 64, group_size, max_requests,
                              max_pages_per_request, num_int2_pages, num_bf16_pages, softmax_scale, page_perm_seed)


def _ptr(t) -> int | None:
    """Device address of a dense row-major tensor (the C ABI takes no strides)."""
    if t is None:
        return None
    if not t.is_contiguous():
        raise OscarError(OSCAR_ERR_INVALID_ARG, "tensor must be contiguous (dense row-major)")
    return t.data_ptr()


def _stream_ptr(stream) -> int | None:
    if stream is None:
        import torch
        if not torch.cuda.is_available():
            return None
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


class OscarCache:
    """Owner of one cache handle and its device buffer (a torch uint8 tensor)."""

    def __init__(self, cfg: oscar_cache_config, rot_k=None, rot_v=None, tau_k=None, tau_v=None,
                 device="cuda", stream=None, dry_run: bool = False):
        import torch
        self.lib = load()
        self.cfg = cfg
        self.dry = dry_run
        self.bytes = self.lib.oscar_cache_device_bytes(ctypes.byref(cfg))
        if self.bytes == 0:
            raise OscarError(OSCAR_ERR_INVALID_ARG, "invalid cache configuration")
        lh = cfg.num_layers * cfg.num_kv_heads
        tk = np.ascontiguousarray(np.asarray(tau_k, dtype=np.float32).reshape(lh))
        tv = np.ascontiguousarray(np.asarray(tau_v, dtype=np.float32).reshape(lh))
        self._tau = (tk, tv)
        self.mem = None
        if not dry_run:
            self.mem = torch.empty(self.bytes + 256, dtype=torch.uint8, device=device)
            off = (-self.mem.data_ptr()) % 256
            self.mem = self.mem[off:off + self.bytes]
            assert rot_k.is_cuda and rot_k.dtype == torch.float32 and rot_k.is_contiguous()
            assert rot_v.is_cuda and rot_v.dtype == torch.float32 and rot_v.is_contiguous()
        handle = c_void_p()
        st = self.lib.oscar_cache_create(ctypes.byref(cfg), _ptr(self.mem), self.bytes, _ptr(rot_k), _ptr(rot_v),
                                         tk.ctypes.data_as(POINTER(c_float)), tv.ctypes.data_as(POINTER(c_float)),
                                         None if dry_run else _stream_ptr(stream), ctypes.byref(handle))
        if st != OSCAR_OK:
            raise OscarError(st, "oscar_cache_create failed")
        self.h = handle

    # -- helpers ----------------------------------------------------------------
    def _check(self, st: int, what: str, allow_dry: bool = False) -> None:
        if st == OSCAR_OK or (allow_dry and st == OSCAR_ERR_DRY_RUN and self.dry):
            return
        raise OscarError(st, f"{what}: {self.lib.oscar_last_error(self.h).decode()}")

    def close_handle(self) -> None:
        if getattr(self, "h", None):
            self.lib.oscar_cache_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close_handle()
        except Exception:
            pass

    def layout(self) -> oscar_cache_layout:
        lay = oscar_cache_layout()
        self._check(self.lib.oscar_cache_get_layout(self.h, ctypes.byref(lay)), "layout")
        return lay

    # -- requests -----------------------------------------------------------------
    def open(self, stream=None) -> int:
        r = c_int32()
        self._check(self.lib.oscar_request_open(self.h, None if self.dry else _stream_ptr(stream), ctypes.byref(r)),
                    "open")
        return r.value

    def fork(self, parent: int, prefix_tokens: int, stream=None) -> int:
        r = c_int32()
        self._check(self.lib.oscar_request_fork(self.h, parent, prefix_tokens,
                                                None if self.dry else _stream_ptr(stream), ctypes.byref(r)), "fork")
        return r.value

    def close(self, req: int) -> None:
        self._check(self.lib.oscar_request_close(self.h, req), "close")

    def length(self, req: int, layer: int):
        t, he = c_int64(), c_int64()
        self._check(self.lib.oscar_request_length(self.h, req, layer, ctypes.byref(t), ctypes.byref(he)), "length")
        return t.value, he.value

    def pages(self, req: int):
        n = c_int32()
        bf = (c_int32 * BF16_PAGES_PER_REQUEST)()
        self._check(self.lib.oscar_request_pages(self.h, req, None, 0, ctypes.byref(n), bf), "pages")
        buf = (c_int32 * max(1, n.value))()
        self._check(self.lib.oscar_request_pages(self.h, req, buf, n.value, ctypes.byref(n), bf), "pages")
        return list(buf)[:n.value], list(bf)

    def free_pages(self):
        a, b = c_int64(), c_int64()
        self._check(self.lib.oscar_cache_free_pages(self.h, ctypes.byref(a), ctypes.byref(b)), "free_pages")
        return a.value, b.value

    # -- write path ---------------------------------------------------------------
    def prefill(self, req: int, layer: int, k, v, n_tokens: int | None = None, stream=None) -> None:
        n = int(k.shape[0]) if n_tokens is None else n_tokens
        self._check(self.lib.oscar_prefill_quantize(self.h, req, layer, _ptr(k), _ptr(v), n,
                                                    None if self.dry else _stream_ptr(stream)), "prefill",
                    allow_dry=True)

    @staticmethod
    def _reqs(reqs):
        arr = (c_int32 * len(reqs))(*[int(r) for r in reqs])
        return arr

    def append(self, layer: int, reqs, k, v, stream=None) -> None:
        arr = self._reqs(reqs)
        self._check(self.lib.oscar_append(self.h, layer, len(reqs), arr, _ptr(k), _ptr(v),
                                          None if self.dry else _stream_ptr(stream)), "append", allow_dry=True)

    def demote(self, layer: int, reqs, stream=None) -> None:
        arr = self._reqs(reqs)
        self._check(self.lib.oscar_demote(self.h, layer, len(reqs), arr, None if self.dry else _stream_ptr(stream)),
                    "demote", allow_dry=True)

    def demote_layers(self, layer_begin: int, layer_end: int, reqs, stream=None) -> None:
        arr = self._reqs(reqs)
        self._check(self.lib.oscar_demote_layers(self.h, layer_begin, layer_end, len(reqs), arr,
                                                 None if self.dry else _stream_ptr(stream)),
                    "demote_layers", allow_dry=True)

    # -- decode -------------------------------------------------------------------
    def workspace_bytes(self, reqs) -> int:
        arr = self._reqs(reqs)
        b = c_size_t()
        self._check(self.lib.oscar_decode_workspace_bytes(self.h, len(reqs), arr, ctypes.byref(b)), "workspace")
        return b.value

    def decode(self, layer: int, reqs, q, out, workspace, stream=None) -> None:
        arr = self._reqs(reqs)
        self._check(self.lib.oscar_decode_attention(self.h, layer, len(reqs), arr, _ptr(q), _ptr(out),
                                                    _ptr(workspace), workspace.numel() * workspace.element_size(),
                                                    _stream_ptr(stream)), "decode")

    def step(self, layer: int, reqs, k, v, q, out, workspace, stream=None) -> None:
        """Append k / v of every request, then decode with q (one fused call)."""
        arr = self._reqs(reqs)
        nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        self._check(self.lib.oscar_decode_step(self.h, layer, len(reqs), arr, _ptr(k), _ptr(v), _ptr(q), _ptr(out),
                                               _ptr(workspace), nbytes, None if self.dry else _stream_ptr(stream)),
                    "decode step", allow_dry=True)

    def decode_noalloc(self, layer: int, reqs, q, out, stream=None) -> None:
        """Decode with the library's fixed static scratch (no workspace argument)."""
        arr = self._reqs(reqs)
        self._check(self.lib.oscar_decode_attention_noalloc(self.h, layer, len(reqs), arr, _ptr(q), _ptr(out),
                                                            None if self.dry else _stream_ptr(stream)),
                    "decode (fixed scratch)", allow_dry=True)

    def check(self, stream=None) -> None:
        self._check(self.lib.oscar_cache_check(self.h, None if self.dry else _stream_ptr(stream)), "device check")

    def debug_decode_hooks(self, wait_limit: int = 100000, hold_copy: int = -1) -> None:
        """Failure-detection hooks of this cache's decode launches (tests only)."""
        self._check(self.lib.oscar_debug_decode_hooks(self.h, wait_limit, hold_copy), "decode hooks")

    # -- views of device memory (for tests and inspection) ------------------------
    def int2_pool(self, layer: int):
        lay = self.layout()
        rec = lay.int2_record_bytes          # 4608 (group 128) or 5120 (group 64)
        n = self.cfg.num_int2_pages * self.cfg.num_kv_heads * rec
        base = lay.int2_pool_offset + layer * lay.int2_layer_stride
        return self.mem[base:base + n].view(self.cfg.num_int2_pages, self.cfg.num_kv_heads, rec)

    def bf16_pool(self, layer: int):
        import torch
        lay = self.layout()
        nb = self.cfg.num_bf16_pages or BF16_PAGES_PER_REQUEST * self.cfg.max_requests
        n = nb * lay.bf16_page_stride
        base = lay.bf16_pool_offset + layer * lay.bf16_layer_stride
        return self.mem[base:base + n].view(torch.int16).view(nb, self.cfg.num_kv_heads, 2, 64, HEAD_DIM)

    def device_page_table(self):
        import torch
        lay = self.layout()
        n = self.cfg.max_requests * self.cfg.max_pages_per_request
        return self.mem[lay.hist_pt_offset:lay.hist_pt_offset + 4 * n].view(torch.int32).view(
            self.cfg.max_requests, self.cfg.max_pages_per_request)


def bf16_decode(kv, page_table, lens, q, out, num_kv_heads: int, scale: float = 0.0, workspace=None, stream=None):
    """Uncompressed BF16 paged decode attention (the baseline): kv bf16
    [pages][Hkv][2][64][128], page_table int32 [n][max_pages] (device), lens host
    ints, q bf16 [n][Hq][128], out fp32 [n][Hq][128].  Returns the workspace."""
    lib = load()
    n, hq = q.shape[0], q.shape[1]
    arr = (c_int32 * n)(*[int(x) for x in lens])
    need = lib.oscar_bf16_decode_workspace_bytes(n, arr, hq, num_kv_heads)
    if need == 0:
        raise OscarError(1, "bf16_decode: arguments outside the supported limits")
    if workspace is None or workspace.numel() < need:
        workspace = new_workspace(need)
    st = lib.oscar_bf16_decode(_ptr(kv), kv.shape[0], _ptr(page_table), page_table.shape[1], arr, n, hq,
                               num_kv_heads, float(scale), _ptr(q), _ptr(out), _ptr(workspace), workspace.numel(),
                               _stream_ptr(stream))
    if st != 0:
        raise OscarError(st, "oscar_bf16_decode failed")
    return workspace


def new_workspace(nbytes: int, device="cuda"):
    """Zeroed, 256-byte aligned device workspace of at least nbytes."""
    import torch
    t = torch.zeros(nbytes + 256, dtype=torch.uint8, device=device)
    off = (-t.data_ptr()) % 256
    return t[off:off + nbytes]
