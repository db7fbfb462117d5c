"""Helpers for the GPU parity tests: move seeded inputs to the device, run one
step through the C ABI, compare with the oracle."""
from __future__ import annotations

import numpy as np

import decode_step_masked_gb300 as ftd
from synthetic import gen_cache_slot, gen_scales_slot, to_storage

# Parity bars: fp32/fp16/bf16 caches with fp32 accumulation, and INT8 caches
# against the oracle run on the dequantised values.
TOL_MAXABS = 2e-3
TOL_RELL2 = 1e-3
TOL_MAXABS_I8 = 1e-2


def dev(a):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def host(t, like):
    a = t.cpu().numpy()
    return a.view(like.dtype) if a.dtype != like.dtype else a


def make_step(w, softmax_scale=0.0, force_cuda_core=False, **opts):
    """A library context; force_cuda_core selects the CUDA-core kernel for grouped caches
    (the config's kernel field).  opts: out_dtype, window, page_size, num_pages, q_len,
    wait_limit_us (the config's option fields)."""
    kernel = ftd.FTD_KERNEL_CUDA_CORE if force_cuda_core else ftd.FTD_KERNEL_AUTO
    return ftd.DecodeStep(w.B, w.Hq, w.Hkv, w.D, w.Lmax, w.qkv_dtype, w.cache_dtype, softmax_scale,
                          kernel=kernel, **opts)


TORCH_OUT = {"f32": "float32", "f16": "float16", "bf16": "bfloat16"}


def run_step(w, inp, step=None, softmax_scale=0.0, use_bias=True, force_cuda_core=False, out_dtype="f32",
             window=0):
    """One decode step on the GPU with caller-owned device buffers.  The output
    comes back as float64 (exact for every out_dtype), [B,Hq,D] or, with
    w.q_len > 1, [B,T,Hq,D]."""
    import torch
    own = step is None
    T = getattr(w, "q_len", 1)
    if own:
        step = make_step(w, softmax_scale, force_cuda_core, out_dtype=out_dtype, window=window, q_len=T)
    q, kn, vn = dev(inp["q"]), dev(inp["k_new"]), dev(inp["v_new"])
    bias = dev(inp["bias"]) if (use_bias and inp.get("bias") is not None) else None
    kc, vc, sl = dev(inp["k_cache"]), dev(inp["v_cache"]), dev(inp["seq_lens"])
    sc = dev(inp["scales"]) if inp.get("scales") is not None else None
    shape = (w.B, T, w.Hq, w.D) if T > 1 else (w.B, w.Hq, w.D)
    out = torch.full(shape, float("nan"), dtype=getattr(torch, TORCH_OUT[out_dtype]), device="cuda")
    step(q, kn, vn, sl, out, bias=bias, k_cache=kc, v_cache=vc, scales=sc)
    torch.cuda.synchronize()
    status = step.get_error()
    res = dict(out=out.double().cpu().numpy(), out_raw=out.cpu(), k_cache=host(kc, inp["k_cache"]),
               v_cache=host(vc, inp["v_cache"]), scales=None if sc is None else sc.cpu().numpy(),
               status=status)
    if own:
        step.close()
    return res


def assert_close(got, ref, i8=False, what=""):
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = float(np.max(np.abs(got - ref))) if got.size else 0.0
    if i8:
        assert err <= TOL_MAXABS_I8, f"{what}: max-abs {err:.3e} > {TOL_MAXABS_I8}"
        return err, None
    nref = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(got - ref) / nref) if nref > 0 else float(np.linalg.norm(got))
    assert err <= TOL_MAXABS, f"{what}: max-abs {err:.3e} > {TOL_MAXABS}"
    assert rel <= TOL_RELL2, f"{what}: rel-L2 {rel:.3e} > {TOL_RELL2}"
    return err, rel


def assert_same_bytes(a, b, what):
    a = np.ascontiguousarray(a)
    b = np.ascontiguousarray(b)
    assert a.shape == b.shape and a.dtype.itemsize == b.dtype.itemsize, what
    diff = np.nonzero(a.reshape(-1).view(np.uint8) != b.reshape(-1).view(np.uint8))[0]
    if diff.size:
        first = np.unravel_index(diff[0] // a.dtype.itemsize, a.shape)
        raise AssertionError(f"{what}: {diff.size} bytes differ, first at element {tuple(int(i) for i in first)}")


class _CudaArray:
    """Wraps a raw device address so torch can view it (CUDA array interface)."""

    def __init__(self, ptr, shape, typestr):
        self.__cuda_array_interface__ = {"shape": tuple(int(x) for x in shape), "typestr": typestr,
                                         "data": (int(ptr), False), "version": 3, "strides": None}


def device_view(ptr, shape, np_dtype):
    """torch tensor aliasing library-owned device memory at ``ptr``."""
    import torch
    return torch.as_tensor(_CudaArray(ptr, shape, np.dtype(np_dtype).str), device="cuda")


def fill_device_cache(w, seed, lens, which, fill_beyond="nan"):
    """Device cache [B,Hkv,Lmax,D] filled slot by slot from the seeded generator."""
    import torch
    dt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.int16, "i8": torch.int8}[w.cache_dtype]
    t = torch.empty((w.B, w.Hkv, w.Lmax, w.D), dtype=dt, device="cuda")
    for b in range(w.B):
        t[b].copy_(dev(gen_cache_slot(w, seed, which, b, int(lens[b]), fill_beyond)))
    return t


def fill_device_scales(w, seed, lens, fill_beyond="nan"):
    import torch
    t = torch.empty((2, w.B, w.Hkv, w.Lmax), dtype=torch.float32, device="cuda")
    for b in range(w.B):
        t[0, b].copy_(dev(gen_scales_slot(w, seed, "k", b, int(lens[b]), fill_beyond)))
        t[1, b].copy_(dev(gen_scales_slot(w, seed, "v", b, int(lens[b]), fill_beyond)))
    return t


# ------------------------------------------------------------ paged caches
def page_layout(w, lens, page_size, spare, seed, q_len=1):
    """A shuffled page pool: every slot gets the pages covering positions 0 .. L_b;
    unused table entries hold an out-of-range sentinel the kernel must not read."""
    rng = np.random.default_rng(seed)
    pps = -(-w.Lmax // page_size)
    need = [(-(-(int(L) + q_len) // page_size) if 0 <= L <= w.Lmax - q_len else 0) for L in lens]
    num_pages = sum(need) + spare
    perm = rng.permutation(num_pages)
    table = np.full((w.B, pps), 1 << 30, np.int32)
    k = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[k:k + n]
        k += n
    return table, num_pages, perm[k:]


def to_pages(w, arr, table, num_pages, page_size, fill):
    """Scatter a contiguous [B][Hkv][Lmax](...) array into pages [num_pages][Hkv][page_size](...)."""
    tail = arr.shape[3:]
    pages = np.full((num_pages, w.Hkv, page_size) + tail, fill, dtype=arr.dtype)
    for b in range(w.B):
        for i, pg in enumerate(table[b]):
            if 0 <= pg < num_pages:
                lo = i * page_size
                n = min(page_size, w.Lmax - lo)
                pages[pg, :, :n] = arr[b, :, lo:lo + n]
    return pages


def from_pages(w, pages, table, page_size, lens, q_len=1):
    """Gather positions 0 .. L_b + q_len - 1 of each active slot back to a contiguous array (rest zero)."""
    out = np.zeros((w.B, w.Hkv, w.Lmax) + pages.shape[3:], dtype=pages.dtype)
    for b, L in enumerate(lens):
        if not 0 <= L <= w.Lmax - q_len:
            continue
        for t0 in range(0, int(L) + q_len, page_size):
            n = min(page_size, int(L) + q_len - t0)
            out[b, :, t0:t0 + n] = pages[table[b, t0 // page_size], :, :n]
    return out


def valid_rows(w, arr, lens, q_len=1):
    out = np.zeros_like(arr)
    for b, L in enumerate(lens):
        if 0 <= L <= w.Lmax - q_len:
            out[b, :, :L + q_len] = arr[b, :, :L + q_len]
    return out


def _from_storage(a, dt):
    a = np.asarray(a)
    if dt == "bf16":
        return (a.astype(np.uint32) << 16).view(np.float32)
    return a.astype(np.float32)


def rising_scores(w, inp, rise_log2=40.0, seed=5):
    """Inputs whose scores climb by about ``rise_log2`` (base-2 units) from the first
    cached position to the last: each kv head gets a unit direction u, its queries
    point along u and its cached keys carry a component growing linearly along u.
    The running maximum of every query row then moves again and again inside a
    context.  fp16 / bf16 caches only; positions past the lengths keep their fill."""
    rng = np.random.default_rng(seed)
    D, g = w.D, w.Hq // w.Hkv
    u = rng.standard_normal((w.Hkv, D))
    u /= np.linalg.norm(u, axis=1, keepdims=True)
    A = 12.0  # key component at the end of the cache
    sq = rise_log2 * np.sqrt(D) / (A * np.log2(np.e))
    q = _from_storage(inp["q"], w.qkv_dtype).astype(np.float64)
    lead = q.shape[:-2]  # [B] or [B, T]
    heads = np.repeat(u, g, axis=0)  # [Hq, D]
    q = sq * np.broadcast_to(heads, lead + heads.shape) + 0.1 * q
    k = _from_storage(inp["k_cache"], w.cache_dtype).astype(np.float64)  # [B, Hkv, Lmax, D]
    ramp = A * np.arange(w.Lmax, dtype=np.float64) / w.Lmax
    k = 0.3 * k + ramp[None, None, :, None] * u[None, :, None, :]
    return dict(inp, q=to_storage(q.astype(np.float32), w.qkv_dtype),
                k_cache=to_storage(k.astype(np.float32), w.cache_dtype))


def rising_scores_i8(w, inp, rise_log2=40.0, seed=5):
    """rising_scores for an INT8 cache: the keys' history rows (positions before each slot's
    length) become 0.3 x the dequantised key plus the same ramp along u, and are quantised
    again per (slot, kv head, position) row with the scale max|k| / 127.  Rows from the
    length on keep their fill (code 127 with a NaN scale)."""
    rng = np.random.default_rng(seed)
    D, g = w.D, w.Hq // w.Hkv
    u = rng.standard_normal((w.Hkv, D))
    u /= np.linalg.norm(u, axis=1, keepdims=True)
    A = 12.0
    sq = rise_log2 * np.sqrt(D) / (A * np.log2(np.e))
    q = _from_storage(inp["q"], w.qkv_dtype).astype(np.float64)
    lead = q.shape[:-2]
    heads = np.repeat(u, g, axis=0)
    q = sq * np.broadcast_to(heads, lead + heads.shape) + 0.1 * q
    codes = inp["k_cache"].copy()
    scales = inp["scales"].copy()
    ramp = A * np.arange(w.Lmax, dtype=np.float64) / w.Lmax
    for b, L in enumerate(np.asarray(inp["seq_lens"])):
        n = int(min(max(L, 0), w.Lmax))
        if n == 0:
            continue
        k = codes[b, :, :n].astype(np.float64) * scales[0, b, :, :n, None].astype(np.float64)
        k = 0.3 * k + ramp[None, :n, None] * u[:, None, :]
        s = (np.max(np.abs(k), axis=-1) / 127.0).astype(np.float32)
        codes[b, :, :n] = np.clip(np.rint(k / s[..., None].astype(np.float64)), -127, 127).astype(np.int8)
        scales[0, b, :, :n] = s
    return dict(inp, q=to_storage(q.astype(np.float32), w.qkv_dtype), k_cache=codes, scales=scales)


def scale_q(w, inp, factor):
    """The same inputs with the query multiplied by ``factor`` (stored again in the qkv dtype)."""
    q = _from_storage(inp["q"], w.qkv_dtype) * np.float32(factor)
    return dict(inp, q=to_storage(q, w.qkv_dtype))
