"""Python binding of the GB300 masked multi-head attention decode step.

Argument marshalling only: every entry point of ``include/ftd.h`` is exposed
under the same name and forwards plain integers (device or host addresses)
and sizes to ``_build/libftd.so`` through ctypes.  All decode work runs in
the library's CUDA kernels; there is no CPU path here.  If the library has
not been built, ``load_library`` raises instead of falling back.

``DecodeStep`` is a convenience wrapper for callers holding torch tensors:
it reads ``data_ptr()`` and the current CUDA stream and calls the same ABI.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from ._build import LIB, build_library  # noqa: F401

FTD_OK = 0
FTD_ERR_INVALID_ARG = 1
FTD_ERR_UNSUPPORTED = 2
FTD_ERR_OOM = 3
FTD_ERR_CUDA = 4
FTD_ERR_SEQ_OVERFLOW = 5
FTD_ERR_DEVICE_TIMEOUT = 6
FTD_ERR_BAD_PAGE = 7

FTD_F32, FTD_F16, FTD_BF16, FTD_I8 = 0, 1, 2, 3
FTD_KERNEL_AUTO, FTD_KERNEL_CUDA_CORE = 0, 1
DTYPES = {"f32": FTD_F32, "f16": FTD_F16, "bf16": FTD_BF16, "i8": FTD_I8}

# Symbols include/ftd.h declares; the loader checks each one is exported.
EXPORTS = ("ftd_init", "ftd_cache_ptrs", "ftd_decode_mha", "ftd_decode_mha_current", "ftd_decode_mha_paged",
           "ftd_decode_mha_host", "ftd_get_error", "ftd_destroy", "ftd_status_str", "ftd_last_error",
           "ftd_kernel_launches", "ftd_decode_mha_noalloc", "ftd_debug_stall_next",
           "ftd_debug_late_lengths", "ftd_decode_mha_proj")


class FtdConfig(ctypes.Structure):
    _fields_ = [("max_batch", ctypes.c_int), ("n_q_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("max_len", ctypes.c_int), ("qkv_dtype", ctypes.c_int),
                ("cache_dtype", ctypes.c_int), ("softmax_scale", ctypes.c_float),
                ("out_dtype", ctypes.c_int), ("window", ctypes.c_int), ("page_size", ctypes.c_int),
                ("num_pages", ctypes.c_int), ("q_len", ctypes.c_int), ("kernel", ctypes.c_int),
                ("proj_dim", ctypes.c_int), ("wait_limit_us", ctypes.c_int)]


class FtdError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{ftd_status_str(status)}: {message}")
        self.status = status


_lib: Optional[ctypes.CDLL] = None


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load the built library (``_build/libftd.so``) and declare its signatures."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or LIB
    if not os.path.exists(path):
        raise FileNotFoundError(
            f"{path} is missing: build it with decode_step_masked_gb300.build_library() "
            "(there is no fallback implementation)")
    lib = ctypes.CDLL(path)
    for name in EXPORTS:
        getattr(lib, name)  # AttributeError if a declared symbol is not exported
    P, I = ctypes.c_void_p, ctypes.c_int
    lib.ftd_init.argtypes = [ctypes.POINTER(FtdConfig), P, ctypes.POINTER(P)]
    lib.ftd_init.restype = I
    lib.ftd_cache_ptrs.argtypes = [P, ctypes.POINTER(P), ctypes.POINTER(P), ctypes.POINTER(P)]
    lib.ftd_cache_ptrs.restype = I
    for fn in (lib.ftd_decode_mha, lib.ftd_decode_mha_host):
        fn.argtypes = [P] * 11
        fn.restype = I
    lib.ftd_decode_mha_current.argtypes = [P] * 10
    lib.ftd_decode_mha_current.restype = I
    lib.ftd_decode_mha_paged.argtypes = [P] * 12
    lib.ftd_decode_mha_paged.restype = I
    lib.ftd_decode_mha_proj.argtypes = [P] * 13
    lib.ftd_decode_mha_proj.restype = I
    lib.ftd_get_error.argtypes = [P]
    lib.ftd_get_error.restype = I
    lib.ftd_destroy.argtypes = [P]
    lib.ftd_destroy.restype = None
    lib.ftd_status_str.argtypes = [I]
    lib.ftd_status_str.restype = ctypes.c_char_p
    lib.ftd_last_error.argtypes = []
    lib.ftd_last_error.restype = ctypes.c_char_p
    lib.ftd_kernel_launches.argtypes = []
    lib.ftd_kernel_launches.restype = ctypes.c_uint64
    lib.ftd_decode_mha_noalloc.argtypes = [ctypes.POINTER(FtdConfig)] + [P] * 11
    lib.ftd_decode_mha_noalloc.restype = I
    lib.ftd_debug_stall_next.argtypes = [P, I]
    lib.ftd_debug_stall_next.restype = I
    lib.ftd_debug_late_lengths.argtypes = [P, P, I, I, P]
    lib.ftd_debug_late_lengths.restype = I
    if path == LIB:
        _lib = lib
    return lib


# ------------------------------------------------------------ same-name ABI
def ftd_status_str(status: int) -> str:
    return load_library().ftd_status_str(int(status)).decode()


def ftd_last_error() -> str:
    return load_library().ftd_last_error().decode()


def ftd_kernel_launches() -> int:
    return int(load_library().ftd_kernel_launches())


def ftd_init(cfg: FtdConfig, stream: int = 0):
    """Returns (status, ctx handle as int or None)."""
    h = ctypes.c_void_p()
    st = load_library().ftd_init(ctypes.byref(cfg), ctypes.c_void_p(stream or None), ctypes.byref(h))
    return st, h.value


def ftd_cache_ptrs(ctx: int):
    k, v, s = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_void_p()
    st = load_library().ftd_cache_ptrs(ctypes.c_void_p(ctx), ctypes.byref(k), ctypes.byref(v), ctypes.byref(s))
    return st, k.value, v.value, s.value


def _ptrs(*xs):
    # Addresses go through as Python ints (or None): the argtypes declare them
    # c_void_p, and ctypes converts ints itself, without a wrapper object per
    # argument on the per-step path.
    return xs


def ftd_decode_mha(ctx, q, k_new, v_new, qkv_bias, k_cache, v_cache, seq_lens, scales, out, stream) -> int:
    return load_library().ftd_decode_mha(*_ptrs(ctx, q, k_new, v_new, qkv_bias, k_cache, v_cache, seq_lens,
                                                scales, out, stream))


def ftd_decode_mha_current(q, k_new, v_new, qkv_bias, k_cache, v_cache, seq_lens, scales, out, stream) -> int:
    return load_library().ftd_decode_mha_current(*_ptrs(q, k_new, v_new, qkv_bias, k_cache, v_cache, seq_lens,
                                                        scales, out, stream))


def ftd_decode_mha_paged(ctx, q, k_new, v_new, qkv_bias, k_pages, v_pages, block_table, seq_lens, scales, out,
                         stream) -> int:
    return load_library().ftd_decode_mha_paged(*_ptrs(ctx, q, k_new, v_new, qkv_bias, k_pages, v_pages,
                                                      block_table, seq_lens, scales, out, stream))


def ftd_decode_mha_proj(ctx, q, k_new, v_new, qkv_bias, k_cache, v_cache, seq_lens, scales, out, w_o, y,
                        stream) -> int:
    return load_library().ftd_decode_mha_proj(*_ptrs(ctx, q, k_new, v_new, qkv_bias, k_cache, v_cache, seq_lens,
                                                     scales, out, w_o, y, stream))


def ftd_decode_mha_host(ctx, q, k_new, v_new, qkv_bias, k_cache, v_cache, seq_lens, scales, out,
                        stream) -> int:
    return load_library().ftd_decode_mha_host(*_ptrs(ctx, q, k_new, v_new, qkv_bias, k_cache, v_cache,
                                                     seq_lens, scales, out, stream))


def ftd_decode_mha_noalloc(cfg: FtdConfig, q, k_new, v_new, qkv_bias, k_cache, v_cache, seq_lens, scales, out,
                           device_err, stream) -> int:
    """The decode step without a context: scratch lives in the library's static device array."""
    return load_library().ftd_decode_mha_noalloc(ctypes.byref(cfg), *_ptrs(q, k_new, v_new, qkv_bias, k_cache,
                                                                           v_cache, seq_lens, scales, out,
                                                                           device_err, stream))


def ftd_debug_stall_next(ctx, calls: int) -> int:
    """Test hook: the next ``calls`` decode calls withhold one tile copy (bounded-wait error path)."""
    return load_library().ftd_debug_stall_next(ctypes.c_void_p(ctx), int(calls))


def ftd_debug_late_lengths(src, dst, n: int, delay_us: int, stream) -> int:
    """Test hook: a kernel that lets the next launch start at once and copies n lengths src -> dst late."""
    return load_library().ftd_debug_late_lengths(src, dst, int(n), int(delay_us), stream)


def ftd_get_error(ctx) -> int:
    return load_library().ftd_get_error(ctypes.c_void_p(ctx))


def ftd_destroy(ctx) -> None:
    load_library().ftd_destroy(ctypes.c_void_p(ctx or None))


def check(status: int) -> None:
    if status != FTD_OK:
        raise FtdError(status, ftd_last_error())


# ------------------------------------------------------- torch convenience
def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


class DecodeStep:
    """Owns one library context; calls take torch CUDA tensors (marshalling only)."""

    def __init__(self, max_batch, n_q_heads, n_kv_heads, head_dim, max_len, qkv_dtype="bf16",
                 cache_dtype="bf16", softmax_scale=0.0, stream: Optional[int] = None, out_dtype="f32",
                 window=0, page_size=0, num_pages=0, q_len=1, kernel=FTD_KERNEL_AUTO, wait_limit_us=0, proj_dim=0):
        import torch
        self.cfg = FtdConfig(max_batch, n_q_heads, n_kv_heads, head_dim, max_len, DTYPES[qkv_dtype],
                             DTYPES[cache_dtype], float(softmax_scale), DTYPES[out_dtype], int(window),
                             int(page_size), int(num_pages), int(q_len), int(kernel), int(proj_dim),
                             int(wait_limit_us))
        s = torch.cuda.current_stream().cuda_stream if stream is None else stream
        st, ctx = ftd_init(self.cfg, s)
        check(st)
        self.ctx = ctx

    def cache_ptrs(self):
        st, k, v, s = ftd_cache_ptrs(self.ctx)
        check(st)
        return k, v, s

    def __call__(self, q, k_new, v_new, seq_lens, out, bias=None, k_cache=None, v_cache=None, scales=None,
                 stream: Optional[int] = None):
        import torch
        s = torch.cuda.current_stream().cuda_stream if stream is None else stream
        if self.cfg.page_size:
            raise ValueError("a paged context takes paged(..., block_table, ...)")
        check(ftd_decode_mha(self.ctx, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(bias), _ptr(k_cache),
                             _ptr(v_cache), _ptr(seq_lens), _ptr(scales), _ptr(out), s))

    def proj(self, q, k_new, v_new, seq_lens, out, w_o, y, bias=None, k_cache=None, v_cache=None, scales=None,
             stream: Optional[int] = None):
        """The step followed by the output projection y = out . w_o^T (a context with proj_dim)."""
        import torch
        s = torch.cuda.current_stream().cuda_stream if stream is None else stream
        check(ftd_decode_mha_proj(self.ctx, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(bias), _ptr(k_cache),
                                  _ptr(v_cache), _ptr(seq_lens), _ptr(scales), _ptr(out), _ptr(w_o), _ptr(y), s))

    def paged(self, q, k_new, v_new, block_table, seq_lens, out, bias=None, k_pages=None, v_pages=None,
              scales=None, stream: Optional[int] = None):
        import torch
        s = torch.cuda.current_stream().cuda_stream if stream is None else stream
        check(ftd_decode_mha_paged(self.ctx, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(bias), _ptr(k_pages),
                                   _ptr(v_pages), _ptr(block_table), _ptr(seq_lens), _ptr(scales), _ptr(out),
                                   s))

    def get_error(self) -> int:
        return ftd_get_error(self.ctx)

    def close(self):
        if getattr(self, "ctx", None):
            ftd_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
