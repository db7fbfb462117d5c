"""Pure-Python brute force of the decode step, for tiny inputs only.

TEST INFRASTRUCTURE ONLY.  An independent restatement of the decode step used
to pin ``oracle.c``: storage values are decoded with numpy (not with the C
oracle's helpers), the append rounding uses numpy's float16 cast and a
from-scratch bfloat16 rounding by comparing the two neighbouring
representable values, and attention is a triple loop over Python floats with
``math.exp``.  Slow by design; keep B*Hq*ctx*D below ~1e6.
"""
from __future__ import annotations

import math

import numpy as np


def _decode(x, dt):
    x = np.asarray(x)
    if dt == "f32":
        return x.astype(np.float64)
    if dt == "f16":
        return x.astype(np.float64)
    if dt == "bf16":
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


def _bf16_nearest(f: np.float32) -> int:
    """bfloat16 bits nearest to binary32 ``f`` (ties to even), by comparing neighbours."""
    u = int(np.float32(f).view(np.uint32))
    lo = u >> 16                       # truncation toward zero in magnitude
    hi = lo + 1                        # next bf16 away from zero
    flo = float(np.uint32(lo << 16).view(np.float32))
    fhi = float(np.uint32((hi & 0xFFFF) << 16).view(np.float32))
    fv = float(f)
    dlo, dhi = abs(fv - flo), abs(fhi - fv)
    if dlo < dhi:
        return lo
    if dhi < dlo:
        return hi & 0xFFFF
    return lo if lo % 2 == 0 else hi & 0xFFFF


def _store(x32: np.float32, dt):
    if dt == "f32":
        return np.float32(x32)
    if dt == "f16":
        return np.float16(x32)
    return np.uint16(_bf16_nearest(x32))


def _quant(row):
    """Symmetric absmax int8 code of a binary32 row (same reading as the oracle)."""
    amax = np.float32(max(abs(float(v)) for v in row))
    if amax == 0:
        return [0] * len(row), np.float32(1.0)
    s = np.float32(amax / np.float32(127.0))
    codes = []
    for v in row:
        r = np.float32(np.float32(v) / s)
        c = int(np.rint(r))
        codes.append(max(-127, min(127, c)))
    return codes, s


def decode_step(w, inp, softmax_scale: float = 0.0, window: int = 0, q_len=None):
    """Same contract as ``Oracle.decode_step`` (returns out, caches, scales, overflow).

    With q_len = T > 1, q is [B,T,Hq,D] and k_new / v_new [B,T,Hkv,D]: token j
    goes to position L + j and its query sees positions up to L + j."""
    B, Hq, Hkv, D, Lmax = w.B, w.Hq, w.Hkv, w.D, w.Lmax
    T = max(1, int(q_len or getattr(w, "q_len", 1)))
    g = Hq // Hkv
    scale = softmax_scale if softmax_scale > 0 else 1.0 / math.sqrt(D)
    kc = np.array(inp["k_cache"], copy=True)
    vc = np.array(inp["v_cache"], copy=True)
    sc = None if inp.get("scales") is None else np.array(inp["scales"], np.float32, copy=True)
    q = _decode(inp["q"], w.qkv_dtype).astype(np.float32).reshape(B, T, Hq, D)
    kn = _decode(inp["k_new"], w.qkv_dtype).astype(np.float32).reshape(B, T, Hkv, D)
    vn = _decode(inp["v_new"], w.qkv_dtype).astype(np.float32).reshape(B, T, Hkv, D)
    bias = inp.get("bias")
    bias = (np.zeros((Hq + 2 * Hkv) * D, np.float32) if bias is None
            else _decode(bias, w.qkv_dtype).astype(np.float32))
    bq = bias[: Hq * D].reshape(Hq, D)
    bk = bias[Hq * D:(Hq + Hkv) * D].reshape(Hkv, D)
    bv = bias[(Hq + Hkv) * D:].reshape(Hkv, D)
    overflow = False
    for b in range(B):
        L0 = int(inp["seq_lens"][b])
        if L0 < 0:
            continue
        if L0 + T > Lmax:
            overflow = True
            continue
        for j, h in ((j, h) for j in range(T) for h in range(Hkv)):
            L = L0 + j
            krow = [np.float32(kn[b, j, h, d] + bk[h, d]) for d in range(D)]
            vrow = [np.float32(vn[b, j, h, d] + bv[h, d]) for d in range(D)]
            if w.cache_dtype == "i8":
                kq, ks = _quant(krow)
                vq, vs = _quant(vrow)
                kc[b, h, L, :] = kq
                vc[b, h, L, :] = vq
                sc[0, b, h, L] = ks
                sc[1, b, h, L] = vs
            else:
                for d in range(D):
                    kc[b, h, L, d] = _store(krow[d], w.cache_dtype)
                    vc[b, h, L, d] = _store(vrow[d], w.cache_dtype)
    K = _decode(kc, w.cache_dtype)
    V = _decode(vc, w.cache_dtype)
    if w.cache_dtype == "i8":
        K = K * sc[0].astype(np.float64)[..., None]
        V = V * sc[1].astype(np.float64)[..., None]
    out = np.zeros((B, T, Hq, D))
    for b in range(B):
        L0 = int(inp["seq_lens"][b])
        if L0 < 0 or L0 + T > Lmax:
            continue
        for j, h in ((j, h) for j in range(T) for h in range(Hq)):
            L = L0 + j  # the last position token j sees
            kvh = h // g
            qv = [float(np.float32(q[b, j, h, d] + bq[h, d])) for d in range(D)]
            lo = max(0, L + 1 - window) if window > 0 else 0
            scores = []
            for t in range(lo, L + 1):
                acc = 0.0
                for d in range(D):
                    acc += qv[d] * float(K[b, kvh, t, d])
                scores.append(acc * scale)
            m = max(scores)
            ws = [math.exp(s - m) for s in scores]
            tot = sum(ws)
            for d in range(D):
                out[b, j, h, d] = sum(ws[i] * float(V[b, kvh, lo + i, d]) for i in range(L + 1 - lo)) / tot
    if T == 1:
        out = out[:, 0]
    return dict(out=out, k_cache=kc, v_cache=vc, scales=sc, overflow=overflow)


def out_proj(x, W):
    """The output projection as plain Python loops: y[t][f] = sum_k W[f][k] x[t][k]."""
    F, K = len(W), len(W[0])
    rows = [list(map(float, r)) for r in np.asarray(x, np.float64).reshape(-1, K)]
    return [[math.fsum(float(W[f][k]) * r[k] for k in range(K)) for f in range(F)] for r in rows]
