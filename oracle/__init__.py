"""Float64 CPU oracle of the masked multi-head attention decode step.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline / reference arm load it; the product library never does.
The arithmetic lives in ``oracle.c`` (plain C, float64); this module compiles
it with gcc and marshals numpy arrays through ctypes.  ``brute.py`` holds an
independent pure-Python restatement used to pin it.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(storage rounding against the IEEE definition and numpy, quantiser bounds and
round trip, attention against closed forms, invariants and the brute force).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LOCK = threading.Lock()
_LIBS: dict = {}

CODES = {"f32": 0, "f16": 1, "bf16": 2, "i8": 3}


class _Cfg(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int),
                ("D", ctypes.c_int), ("Lmax", ctypes.c_int), ("qkv_dtype", ctypes.c_int),
                ("cache_dtype", ctypes.c_int), ("softmax_scale", ctypes.c_double), ("window", ctypes.c_int),
                ("q_len", ctypes.c_int)]


def build(src: str = _SRC, out_dir: Optional[str] = None, defines=()) -> str:
    """Compile ``src`` into a shared library and return its path."""
    out_dir = out_dir or os.path.join(_HERE, "_build")
    os.makedirs(out_dir, exist_ok=True)
    tag = "_".join(d.replace("=", "-") for d in defines) or "base"
    out = os.path.join(out_dir, f"liboracle_{tag}.so")
    if os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           "-ffp-contract=off", src, "-o", out + ".tmp", "-lm"]
    cmd[1:1] = [f"-D{d}" for d in defines]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        self.lib = lib
        lib.oracle_bf16_to_f32.restype = ctypes.c_float
        lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
        lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.oracle_f16_to_f32.restype = ctypes.c_float
        lib.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
        lib.oracle_f32_to_f16.restype = ctypes.c_uint16
        lib.oracle_f32_to_f16.argtypes = [ctypes.c_float]
        P = ctypes.c_void_p
        lib.oracle_quant_i8.restype = None
        lib.oracle_quant_i8.argtypes = [P, ctypes.c_int, P, P]
        lib.oracle_attend.restype = None
        lib.oracle_attend.argtypes = [P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_double, P, P]
        lib.oracle_out_proj.restype = None
        lib.oracle_out_proj.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P]
        lib.oracle_decode_step.restype = ctypes.c_int
        lib.oracle_decode_step.argtypes = [ctypes.POINTER(_Cfg), P, P, P, P, P, P, P, P, P,
                                           ctypes.c_int]

    # -- storage formats -------------------------------------------------
    def f32_to_bf16(self, x) -> np.ndarray:
        x = np.asarray(x, np.float32).ravel()
        return np.array([self.lib.oracle_f32_to_bf16(float(v)) for v in x], np.uint16)

    def bf16_to_f32(self, h) -> np.ndarray:
        h = np.asarray(h, np.uint16).ravel()
        return np.array([self.lib.oracle_bf16_to_f32(int(v)) for v in h], np.float32)

    def f32_to_f16(self, x) -> np.ndarray:
        x = np.asarray(x, np.float32).ravel()
        return np.array([self.lib.oracle_f32_to_f16(float(v)) for v in x], np.uint16)

    def f16_to_f32(self, h) -> np.ndarray:
        h = np.asarray(h, np.uint16).ravel()
        return np.array([self.lib.oracle_f16_to_f32(int(v)) for v in h], np.float32)

    def quant_i8(self, x):
        x = np.ascontiguousarray(x, np.float32)
        code = np.zeros(x.shape[-1], np.int8)
        s = np.zeros(1, np.float32)
        self.lib.oracle_quant_i8(x.ctypes.data, x.shape[-1], code.ctypes.data, s.ctypes.data)
        return code, float(s[0])

    # -- attention ---------------------------------------------------------
    def attend(self, q, K, V, scale: float):
        q = np.ascontiguousarray(q, np.float64)
        K = np.ascontiguousarray(K, np.float64)
        V = np.ascontiguousarray(V, np.float64)
        n, D = K.shape
        o = np.zeros(D, np.float64)
        p = np.zeros(n, np.float64)
        self.lib.oracle_attend(q.ctypes.data, K.ctypes.data, V.ctypes.data, n, D, float(scale),
                               o.ctypes.data, p.ctypes.data)
        return o, p

    def decode_step(self, w, inputs: dict, nthreads: int = 1, softmax_scale: float = 0.0, window: int = 0,
                    q_len: Optional[int] = None):
        """Run one decode step on copies of the caches.

        ``w`` needs attributes B, Hq, Hkv, D, Lmax, qkv_dtype, cache_dtype
        (a ``synthetic.Workload``).  ``window`` > 0 attends only the last
        ``window`` positions.  ``q_len`` > 1 appends that many tokens per slot
        (q [B,T,Hq,D], k_new / v_new [B,T,Hkv,D]).  Returns a dict with
        ``out`` (float64 [B,Hq,D], or [B,T,Hq,D] when q_len > 1), the updated
        ``k_cache`` / ``v_cache`` / ``scales`` and the ``overflow`` flag.
        """
        if w.D > 1024:
            raise ValueError("oracle supports head_dim <= 1024")
        T = max(1, int(q_len or getattr(w, "q_len", 1)))
        cfg = _Cfg(w.B, w.Hq, w.Hkv, w.D, w.Lmax, CODES[w.qkv_dtype], CODES[w.cache_dtype],
                   float(softmax_scale), int(window), T)
        q = np.ascontiguousarray(inputs["q"])
        kn = np.ascontiguousarray(inputs["k_new"])
        vn = np.ascontiguousarray(inputs["v_new"])
        bias = inputs.get("bias")
        bias = None if bias is None else np.ascontiguousarray(bias)
        kc = np.array(inputs["k_cache"], copy=True, order="C")
        vc = np.array(inputs["v_cache"], copy=True, order="C")
        sc = inputs.get("scales")
        sc = None if sc is None else np.array(sc, np.float32, copy=True, order="C")
        lens = np.ascontiguousarray(inputs["seq_lens"], np.int32)
        if q.size != w.B * T * w.Hq * w.D or kn.size != w.B * T * w.Hkv * w.D:
            raise ValueError("q / k_new sizes do not match B, q_len and the heads")
        out = np.zeros((w.B, T, w.Hq, w.D) if T > 1 else (w.B, w.Hq, w.D), np.float64)
        ov = self.lib.oracle_decode_step(
            ctypes.byref(cfg), q.ctypes.data, kn.ctypes.data, vn.ctypes.data,
            None if bias is None else bias.ctypes.data, kc.ctypes.data, vc.ctypes.data,
            lens.ctypes.data, None if sc is None else sc.ctypes.data, out.ctypes.data,
            int(nthreads))
        return dict(out=out, k_cache=kc, v_cache=vc, scales=sc, overflow=bool(ov))


    def out_proj(self, x, W):
        """y [tokens][F] = x . W^T in float64: x is the step's output ([B,Hq,D] or [B,T,Hq,D], as
        float values), flattened to one row of Hq * D per token; W is [F][Hq * D] (float values)."""
        W = np.ascontiguousarray(W, np.float64)
        F, K = W.shape
        x = np.ascontiguousarray(np.asarray(x, np.float64).reshape(-1, K))
        y = np.zeros((x.shape[0], F), np.float64)
        self.lib.oracle_out_proj(x.ctypes.data, W.ctypes.data, x.shape[0], K, F, y.ctypes.data)
        return y


def load(path: Optional[str] = None) -> Oracle:
    """Build (if needed) and load the oracle library."""
    with _LOCK:
        path = path or build()
        if path not in _LIBS:
            _LIBS[path] = Oracle(path)
        return _LIBS[path]
