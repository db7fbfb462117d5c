"""Workload shapes and seeded input generators.

The five workloads mirror the decode-step shapes the FasterTransformer pages
reason about: a tiny fp32 case, Llama-2-7B / 13B-shaped multi-head caches, a
70B-shaped grouped-query cache and an INT8 cache with per-(token, head)
scales.  The pages measure whole models; no weights or datasets exist here, so
every tensor is drawn from the distributions below.

Storage formats (what the caller hands to the library and what the oracle
reads):

=======  ==========================  ========================
dtype    numpy array                 meaning
=======  ==========================  ========================
``f32``  ``float32``                 IEEE binary32
``f16``  ``float16``                 IEEE binary16
``bf16`` ``uint16`` (bit patterns)   bfloat16, top half of binary32
``i8``   ``int8``                    symmetric int8 code, fp32 scale
=======  ==========================  ========================

Random streams are keyed by ``(seed, purpose, slot)`` so one batch slot of a
multi-gigabyte cache can be regenerated on its own for a sampled check.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np

# Numeric codes shared with the C ABI's dtype enum.
DTYPE_CODES = {"f32": 0, "f16": 1, "bf16": 2, "i8": 3}

_STREAM_Q, _STREAM_KNEW, _STREAM_VNEW, _STREAM_BIAS = 11, 12, 13, 14
_STREAM_LENS, _STREAM_KCACHE, _STREAM_VCACHE = 15, 16, 17
_STREAM_KSCALE, _STREAM_VSCALE = 18, 19


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    Lmax: int
    qkv_dtype: str
    cache_dtype: str
    # ("fixed", L) -> every slot has L cached tokens (context L + 1)
    # ("ctx_uniform", lo, hi) -> context uniform over integers [lo, hi]
    lens: tuple = ("fixed", 0)
    bias_std: Optional[float] = None
    scale_range: tuple = (0.01, 0.05)
    seed: int = 0
    description: str = ""
    q_len: int = 1   # new tokens per slot per step (> 1: a speculative verification step)
    extra: dict = field(default_factory=dict)

    @property
    def group(self) -> int:
        return self.Hq // self.Hkv

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "tiny": Workload(
        "tiny", B=1, Hq=4, Hkv=4, D=64, Lmax=16, qkv_dtype="f32", cache_dtype="f32",
        lens=("fixed", 15), bias_std=0.1, seed=0,
        description="tiny decode step: B1 H4 D64, 15 cached + 1 new, fp32, bias N(0,0.1)"),
    "7b": Workload(
        "7b", B=8, Hq=32, Hkv=32, D=128, Lmax=4096, qkv_dtype="f16", cache_dtype="f16",
        lens=("fixed", 2047), seed=1,
        description="Llama-2-7B-shaped decode: B8 H32 D128, context 2048, fp16 cache Lmax 4096"),
    "13b": Workload(
        "13b", B=32, Hq=40, Hkv=40, D=128, Lmax=4096, qkv_dtype="bf16", cache_dtype="bf16",
        lens=("ctx_uniform", 128, 4096), seed=2,
        description="13B-shaped continuous batch: B32 H40 D128, context U{128..4096}, bf16"),
    "70b": Workload(
        "70b", B=16, Hq=64, Hkv=8, D=128, Lmax=8192, qkv_dtype="bf16", cache_dtype="bf16",
        lens=("fixed", 8191), seed=3,
        description="70B-shaped GQA decode: B16 Hq64 Hkv8 D128, context 8192, bf16"),
    "70b_i8": Workload(
        "70b_i8", B=16, Hq=64, Hkv=8, D=128, Lmax=8192, qkv_dtype="f16", cache_dtype="i8",
        lens=("fixed", 8191), scale_range=(0.01, 0.05), seed=6,
        description="70B-shaped GQA decode with an INT8 cache: B16 Hq64 Hkv8 D128, context 8192, fp16 q"),
    "mqa": Workload(
        "mqa", B=64, Hq=64, Hkv=1, D=128, Lmax=4096, qkv_dtype="bf16", cache_dtype="bf16",
        lens=("fixed", 4095), seed=5,
        description="MQA-shaped decode: B64, 64 query heads on one kv head, D128, context 4096, bf16"),
    "int8": Workload(
        "int8", B=64, Hq=32, Hkv=32, D=128, Lmax=2048, qkv_dtype="f16", cache_dtype="i8",
        lens=("ctx_uniform", 512, 2048), scale_range=(0.01, 0.05), seed=4,
        description="INT8 KV cache: B64 H32 D128, context U{512..2048}, fp16 q, fp32 scale per (token, head)"),
}


def storage_dtype(dt: str):
    return {"f32": np.float32, "f16": np.float16, "bf16": np.uint16, "i8": np.int8}[dt]


def to_storage(x: np.ndarray, dt: str) -> np.ndarray:
    """Store float32 samples in the format ``dt`` (round to nearest even)."""
    x = np.asarray(x, dtype=np.float32)
    if dt == "f32":
        return x.copy()
    if dt == "f16":
        return x.astype(np.float16)
    if dt == "bf16":
        u = x.view(np.uint32).astype(np.uint64)
        u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
        return u.astype(np.uint16)
    raise ValueError(f"to_storage: {dt}")


def _nan_bits(dt: str):
    return {"f32": np.float32(np.nan), "f16": np.float16(np.nan),
            "bf16": np.uint16(0x7FC0)}[dt]


def _rng(seed: int, stream: int, slot: int = 0) -> np.random.Generator:
    return np.random.default_rng([seed, stream, slot])


def gen_seq_lens(w: Workload, seed: Optional[int] = None) -> np.ndarray:
    """Cached tokens per slot before this step (the new token lands at that index)."""
    seed = w.seed if seed is None else seed
    kind = w.lens[0]
    if kind == "fixed":
        return np.full(w.B, w.lens[1], dtype=np.int32)
    if kind == "ctx_uniform":
        lo, hi = w.lens[1], w.lens[2]
        ctx = _rng(seed, _STREAM_LENS).integers(lo, hi + 1, size=w.B)
        return (ctx - 1).astype(np.int32)
    raise ValueError(f"lens kind {kind}")


def gen_qkv(w: Workload, seed: Optional[int] = None):
    """q [B,Hq,D], k_new / v_new [B,Hkv,D] ~ N(0,1); bias [(Hq+2Hkv)*D] or None.
    With q_len T > 1 the token axis follows the slot axis: q [B,T,Hq,D], k_new [B,T,Hkv,D]."""
    seed = w.seed if seed is None else seed
    tok = (w.q_len,) if w.q_len > 1 else ()
    q = _rng(seed, _STREAM_Q).standard_normal((w.B,) + tok + (w.Hq, w.D), dtype=np.float32)
    k = _rng(seed, _STREAM_KNEW).standard_normal((w.B,) + tok + (w.Hkv, w.D), dtype=np.float32)
    v = _rng(seed, _STREAM_VNEW).standard_normal((w.B,) + tok + (w.Hkv, w.D), dtype=np.float32)
    bias = None
    if w.bias_std is not None:
        n = (w.Hq + 2 * w.Hkv) * w.D
        bias = (_rng(seed, _STREAM_BIAS).standard_normal(n, dtype=np.float32)
                * np.float32(w.bias_std))
        bias = to_storage(bias, w.qkv_dtype)
    return (to_storage(q, w.qkv_dtype), to_storage(k, w.qkv_dtype),
            to_storage(v, w.qkv_dtype), bias)


def gen_cache_slot(w: Workload, seed: Optional[int], which: str, b: int,
                   seq_len: int, fill_beyond: str = "nan") -> np.ndarray:
    """Pre-filled cache rows for slot ``b``: array [Hkv, Lmax, D] in storage format.

    Rows ``0 .. seq_len-1`` hold the history.  Rows from ``seq_len`` on (the
    row the new token will take, and everything after it) hold ``fill_beyond``:
    ``"nan"`` (int8: code 127, whose scale is NaN) so any read past the mask
    poisons the result, or ``"zero"``.
    """
    seed = w.seed if seed is None else seed
    stream = _STREAM_KCACHE if which == "k" else _STREAM_VCACHE
    n_hist = max(0, min(int(seq_len), w.Lmax))
    rng = _rng(seed, stream, b)
    if w.cache_dtype == "i8":
        out = np.full((w.Hkv, w.Lmax, w.D), 127 if fill_beyond == "nan" else 0, np.int8)
        if n_hist:
            sscale = _scales_for(w, seed, which, b)[:, :n_hist]
            x = rng.standard_normal((w.Hkv, n_hist, w.D), dtype=np.float32)
            codes = np.clip(np.rint(x / sscale[:, :, None]), -128, 127)
            out[:, :n_hist] = codes.astype(np.int8)
        return out
    sd = storage_dtype(w.cache_dtype)
    fill = _nan_bits(w.cache_dtype) if fill_beyond == "nan" else sd(0)
    out = np.full((w.Hkv, w.Lmax, w.D), fill, dtype=sd)
    if n_hist:
        x = rng.standard_normal((w.Hkv, n_hist, w.D), dtype=np.float32)
        out[:, :n_hist] = to_storage(x, w.cache_dtype)
    return out


def _scales_for(w: Workload, seed: int, which: str, b: int) -> np.ndarray:
    stream = _STREAM_KSCALE if which == "k" else _STREAM_VSCALE
    lo, hi = w.scale_range
    return _rng(seed, stream, b).uniform(lo, hi, size=(w.Hkv, w.Lmax)).astype(np.float32)


def gen_scales_slot(w: Workload, seed: Optional[int], which: str, b: int,
                    seq_len: int, fill_beyond: str = "nan") -> np.ndarray:
    """Per-(token, head) fp32 scales [Hkv, Lmax] of an INT8 cache slot."""
    seed = w.seed if seed is None else seed
    s = _scales_for(w, seed, which, b)
    n_hist = max(0, min(int(seq_len), w.Lmax))
    s[:, n_hist:] = np.nan if fill_beyond == "nan" else 0.0
    return s


def gen_all(w: Workload, seed: Optional[int] = None, seq_lens: Optional[np.ndarray] = None,
            fill_beyond: str = "nan") -> dict:
    """Every input of one decode step, in storage formats (host arrays)."""
    seed = w.seed if seed is None else seed
    lens = gen_seq_lens(w, seed) if seq_lens is None else np.asarray(seq_lens, np.int32)
    q, k_new, v_new, bias = gen_qkv(w, seed)
    k_cache = np.stack([gen_cache_slot(w, seed, "k", b, lens[b], fill_beyond) for b in range(w.B)])
    v_cache = np.stack([gen_cache_slot(w, seed, "v", b, lens[b], fill_beyond) for b in range(w.B)])
    scales = None
    if w.cache_dtype == "i8":
        scales = np.stack([
            np.stack([gen_scales_slot(w, seed, "k", b, lens[b], fill_beyond) for b in range(w.B)]),
            np.stack([gen_scales_slot(w, seed, "v", b, lens[b], fill_beyond) for b in range(w.B)]),
        ])
    return dict(q=q, k_new=k_new, v_new=v_new, bias=bias, k_cache=k_cache, v_cache=v_cache,
                seq_lens=lens, scales=scales)
