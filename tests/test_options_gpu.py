"""GPU parity of the step's options against the float64 oracle:

- half-precision output (out_dtype f16 / bf16): each element is the value of
  the fp32 path rounded once to nearest even, and within the fp32 bar plus half
  an output ulp of the oracle;
- sliding window (attend the last W positions): against the oracle's window,
  with the history before the window start poisoned with NaN so a read of it
  shows;
- paged cache (block table over a shuffled page pool): against the oracle on
  the contiguous cache the pages hold, appended rows checked in their pages,
  unused pages and table entries never touched, and an out-of-range table entry
  reported as FTD_ERR_BAD_PAGE.

Both kernels are covered: multi-head caches run the CUDA-core split-K kernel,
grouped fp16/bf16 caches with head_dim 128 and 8 query heads per kv head the
tensor-core kernel (forced onto the CUDA-core kernel in the `cuda_core` cases).
"""
import numpy as np
import pytest

import decode_step_masked_gb300 as ftd
import oracle
from synthetic import Workload, gen_all, to_storage
from tests.gpu_util import (TOL_MAXABS, TOL_MAXABS_I8, assert_close, assert_same_bytes, dev, from_pages,
                            make_step, page_layout, run_step, to_pages, valid_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    ftd.build_library()
    ftd.load_library()


def case(cache, qkv, B, Hq, Hkv, D, Lmax, lens, bias=0.1, seed=21):
    w = Workload("opt", B=B, Hq=Hq, Hkv=Hkv, D=D, Lmax=Lmax, qkv_dtype=qkv, cache_dtype=cache,
                 bias_std=bias, seed=seed)
    return w, gen_all(w, seed=seed, seq_lens=np.array(lens, np.int32), fill_beyond="nan")


# (cache, qkv, B, Hq, Hkv, D, Lmax, lens, force_cuda_core)
SHAPES = {
    "mha_bf16": ("bf16", "bf16", 5, 8, 8, 128, 768, [0, 127, 128, 500, 767], False),
    "mha_f16_d64": ("f16", "f16", 4, 4, 4, 64, 512, [1, 63, 300, 511], False),
    "mha_f32": ("f32", "f32", 3, 4, 4, 64, 384, [5, 200, 383], False),
    "mha_i8": ("i8", "f16", 4, 8, 8, 128, 512, [0, 100, 256, 511], False),
    "gqa_tc_bf16": ("bf16", "bf16", 4, 32, 4, 128, 1024, [0, 127, 700, 1023], False),
    "gqa_tc_f16": ("f16", "f16", 3, 16, 2, 128, 1024, [129, 512, 1000], False),
    "gqa_cc_bf16": ("bf16", "bf16", 4, 32, 4, 128, 1024, [0, 127, 700, 1023], True),
    "gqa_tc_i8": ("i8", "f16", 4, 32, 4, 128, 1024, [0, 127, 700, 1023], False),
    "gqa_cc_i8": ("i8", "f16", 4, 32, 4, 128, 1024, [0, 127, 700, 1023], True),
}


def _tol(cache):
    return TOL_MAXABS_I8 if cache == "i8" else TOL_MAXABS


# ------------------------------------------------------------ half output
def _ulp(x, dt):
    """Spacing of the format `dt` at magnitude x (normal range, subnormal floor)."""
    mant, emin = {"f16": (10, -14), "bf16": (7, -126)}[dt]
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** emin)))
    return 2.0 ** (e - mant)


@pytest.mark.parametrize("out_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("shape", list(SHAPES))
def test_half_output(shape, out_dtype):
    import torch
    cache, qkv, B, Hq, Hkv, D, Lmax, lens, cc = SHAPES[shape]
    w, inp = case(cache, qkv, B, Hq, Hkv, D, Lmax, lens)
    ref = oracle.load().decode_step(w, inp, nthreads=8)
    f32 = run_step(w, inp, force_cuda_core=cc)
    half = run_step(w, inp, force_cuda_core=cc, out_dtype=out_dtype)
    assert f32["status"] == ftd.FTD_OK and half["status"] == ftd.FTD_OK
    # the fp32 path meets the bar, and the half output is its single RNE rounding
    assert_close(f32["out"], ref["out"], i8=cache == "i8", what=f"{shape} fp32 out")
    rounded = f32["out_raw"].to(getattr(torch, {"f16": "float16", "bf16": "bfloat16"}[out_dtype]))
    assert torch.equal(half["out_raw"].view(torch.int16), rounded.view(torch.int16)), \
        f"{shape}: {out_dtype} output is not the rounded fp32 result"
    # against the oracle: fp32 bar plus half an ulp of the output format
    tol = _tol(cache)
    bound = tol + 0.5 * _ulp(np.abs(ref["out"]) + tol, out_dtype)
    err = np.abs(half["out"] - ref["out"])
    assert np.all(err <= bound), f"{shape}: worst {float(np.max(err - bound)):.3e} over the bound"
    # appends are unaffected by the output format
    assert_same_bytes(half["k_cache"], ref["k_cache"], f"{shape} K after append")
    assert_same_bytes(half["v_cache"], ref["v_cache"], f"{shape} V after append")


def test_half_output_inactive_slots_are_zero():
    w, inp = case("bf16", "bf16", 3, 8, 8, 128, 256, [-1, 40, 300])  # inactive, active, overflow
    got = run_step(w, inp, out_dtype="bf16")
    assert np.all(got["out"][0] == 0) and np.all(got["out"][2] == 0)
    assert got["status"] == ftd.FTD_ERR_SEQ_OVERFLOW


# ---------------------------------------------------------- sliding window
def _poison_before_window(w, inp, window):
    """NaN (int8: code 127 with a NaN scale) in every cached row before each slot's window start."""
    inp = dict(inp, k_cache=inp["k_cache"].copy(), v_cache=inp["v_cache"].copy())
    if inp.get("scales") is not None:
        inp["scales"] = inp["scales"].copy()
    nan = {"f32": np.float32(np.nan), "f16": np.float16(np.nan), "bf16": np.uint16(0x7FC0),
           "i8": np.int8(127)}[w.cache_dtype]
    for b, L in enumerate(inp["seq_lens"]):
        if L < 0 or L >= w.Lmax:
            continue
        start = max(0, int(L) + 1 - window)
        inp["k_cache"][b, :, :start] = nan
        inp["v_cache"][b, :, :start] = nan
        if inp.get("scales") is not None:
            inp["scales"][:, b, :, :start] = np.nan
    return inp


@pytest.mark.parametrize("window", [1, 2, 16, 100, 128, 129, 300, 5000])
@pytest.mark.parametrize("shape", list(SHAPES))
def test_sliding_window(shape, window):
    cache, qkv, B, Hq, Hkv, D, Lmax, lens, cc = SHAPES[shape]
    w, inp = case(cache, qkv, B, Hq, Hkv, D, Lmax, lens)
    inp = _poison_before_window(w, inp, window)
    ref = oracle.load().decode_step(w, inp, nthreads=8, window=window)
    got = run_step(w, inp, force_cuda_core=cc, window=window)
    assert got["status"] == ftd.FTD_OK
    assert_same_bytes(got["k_cache"], ref["k_cache"], f"{shape} W={window} K after append")
    assert_same_bytes(got["v_cache"], ref["v_cache"], f"{shape} W={window} V after append")
    if cache == "i8":
        assert_same_bytes(got["scales"], ref["scales"], f"{shape} W={window} scales")
    assert_close(got["out"], ref["out"], i8=cache == "i8", what=f"{shape} W={window}")


def test_window_one_returns_the_new_value():
    """W = 1: only the new token is visible, so the output is v' = v_new + b_v in the cache's precision."""
    w, inp = case("f32", "f32", 2, 4, 4, 64, 128, [0, 77])
    got = run_step(w, inp, window=1)
    vb = inp["v_new"].astype(np.float64) + inp["bias"][(w.Hq + w.Hkv) * w.D:].reshape(w.Hkv, w.D)
    np.testing.assert_allclose(got["out"], vb, rtol=0, atol=1e-6)


def test_window_with_half_output_and_consecutive_steps():
    """Window and bf16 output together over three steps of one context."""
    import torch
    w, inp = case("bf16", "bf16", 3, 32, 4, 128, 512, [126, 127, 300])
    o = oracle.load()
    W = 128
    step = make_step(w, out_dtype="bf16", window=W)
    q, kn, vn, bias = dev(inp["q"]), dev(inp["k_new"]), dev(inp["v_new"]), dev(inp["bias"])
    kc, vc = dev(inp["k_cache"]), dev(inp["v_cache"])
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    lens = inp["seq_lens"].copy()
    ref_inp = dict(inp)
    for it in range(3):
        step(q, kn, vn, dev(lens), out, bias=bias, k_cache=kc, v_cache=vc)
        ref = o.decode_step(w, dict(ref_inp, seq_lens=lens), window=W)
        torch.cuda.synchronize()
        got = out.double().cpu().numpy()
        bound = TOL_MAXABS + 0.5 * _ulp(np.abs(ref["out"]) + TOL_MAXABS, "bf16")
        assert np.all(np.abs(got - ref["out"]) <= bound), f"step {it}"
        ref_inp = dict(ref_inp, k_cache=ref["k_cache"], v_cache=ref["v_cache"])
        lens = lens + 1
    assert step.get_error() == ftd.FTD_OK
    step.close()


# --------------------------------------------------------------- paged
PAGED = {
    "mha_bf16_p128": ("bf16", "bf16", 5, 8, 8, 128, 768, [0, 127, 128, 500, 767], 128, False),
    "mha_f16_p256": ("f16", "f16", 4, 8, 8, 128, 1024, [255, 256, 700, 1023], 256, False),
    "mha_i8_p128": ("i8", "f16", 4, 8, 8, 128, 512, [0, 100, 256, 511], 128, False),
    "mha_f32_d64_p128": ("f32", "f32", 3, 4, 4, 64, 384, [5, -1, 383], 128, False),
    "gqa_tc_bf16_p256": ("bf16", "bf16", 4, 32, 4, 128, 1024, [0, 255, 700, 1023], 256, False),
    "gqa_tc_f16_p128": ("f16", "f16", 3, 16, 2, 128, 1024, [129, 512, 1000], 128, False),
    "gqa_cc_bf16_p256": ("bf16", "bf16", 4, 32, 4, 128, 1024, [0, 255, 700, 1023], 256, True),
    "gqa_tc_i8_p128": ("i8", "f16", 3, 16, 2, 128, 1024, [129, 512, 1000], 128, False),
}


def _run_paged(w, inp, table, num_pages, page_size, cc, window=0, out_dtype="f32", expect=ftd.FTD_OK):
    import torch
    nanv = {"f32": np.float32(np.nan), "f16": np.float16(np.nan), "bf16": np.uint16(0x7FC0),
            "i8": np.int8(127)}[w.cache_dtype]
    kp = to_pages(w, inp["k_cache"], table, num_pages, page_size, nanv)
    vp = to_pages(w, inp["v_cache"], table, num_pages, page_size, nanv)
    sp = None
    if inp.get("scales") is not None:
        sp = np.stack([to_pages(w, inp["scales"][i][..., None], table, num_pages, page_size, np.nan)[..., 0]
                       for i in range(2)])
    step = make_step(w, force_cuda_core=cc, out_dtype=out_dtype, window=window, page_size=page_size,
                     num_pages=num_pages)
    kd, vd = dev(kp), dev(vp)
    sd = dev(sp) if sp is not None else None
    out = torch.full((w.B, w.Hq, w.D), float("nan"), dtype=getattr(torch, {"f32": "float32", "f16": "float16",
                     "bf16": "bfloat16"}[out_dtype]), device="cuda")
    step.paged(dev(inp["q"]), dev(inp["k_new"]), dev(inp["v_new"]), dev(table), dev(inp["seq_lens"]), out,
               bias=dev(inp["bias"]), k_pages=kd, v_pages=vd, scales=sd)
    torch.cuda.synchronize()
    st = step.get_error()
    assert st == expect, ftd.ftd_status_str(st)
    step.close()
    like = inp["k_cache"]
    return dict(out=out.double().cpu().numpy(), k_pages=kd.cpu().numpy().view(like.dtype),
                v_pages=vd.cpu().numpy().view(like.dtype), scales=None if sd is None else sd.cpu().numpy(),
                k_in=kp, v_in=vp, s_in=sp)


@pytest.mark.parametrize("shape", list(PAGED))
def test_paged_cache(shape):
    cache, qkv, B, Hq, Hkv, D, Lmax, lens, ps, cc = PAGED[shape]
    w, inp = case(cache, qkv, B, Hq, Hkv, D, Lmax, lens)
    table, num_pages, spare = page_layout(w, inp["seq_lens"], ps, spare=3, seed=5)
    ref = oracle.load().decode_step(w, inp, nthreads=8)
    got = _run_paged(w, inp, table, num_pages, ps, cc)
    assert_close(got["out"], ref["out"], i8=cache == "i8", what=shape)
    L = inp["seq_lens"]
    # the appended rows landed in their pages, and every other held row is unchanged
    for name, key in (("K", "k"), ("V", "v")):
        assert_same_bytes(from_pages(w, got[f"{key}_pages"], table, ps, L),
                          valid_rows(w, ref[f"{key}_cache"], L), f"{shape} {name} pages after append")
        assert_same_bytes(got[f"{key}_pages"][spare], got[f"{key}_in"][spare], f"{shape} spare {name} pages")
    if cache == "i8":
        for i in range(2):
            g = from_pages(w, got["scales"][i][..., None], table, ps, L)[..., 0]
            assert_same_bytes(g, valid_rows(w, ref["scales"][i], L), f"{shape} scale plane {i}")


@pytest.mark.parametrize("window", [100, 256, 300])
@pytest.mark.parametrize("shape", ["mha_bf16_p128", "gqa_tc_bf16_p256", "mha_i8_p128", "gqa_tc_i8_p128"])
def test_paged_with_window_reads_only_window_pages(shape, window):
    """Entries of pages wholly before the window start are never read: they hold the sentinel."""
    cache, qkv, B, Hq, Hkv, D, Lmax, lens, ps, cc = PAGED[shape]
    w, inp = case(cache, qkv, B, Hq, Hkv, D, Lmax, lens)
    table, num_pages, _ = page_layout(w, inp["seq_lens"], ps, spare=1, seed=6)
    for b, L in enumerate(inp["seq_lens"]):
        if 0 <= L < w.Lmax:
            start = max(0, int(L) + 1 - window)
            table[b, :start // ps] = 1 << 30
    inp = _poison_before_window(w, inp, window)
    ref = oracle.load().decode_step(w, inp, nthreads=8, window=window)
    got = _run_paged(w, inp, table, num_pages, ps, cc, window=window, out_dtype="bf16")
    bound = _tol(cache) + 0.5 * _ulp(np.abs(ref["out"]) + _tol(cache), "bf16")
    assert np.all(np.abs(got["out"] - ref["out"]) <= bound), shape


@pytest.mark.parametrize("shape", ["mha_bf16_p128", "gqa_tc_bf16_p256"])
def test_bad_page_is_reported(shape):
    cache, qkv, B, Hq, Hkv, D, Lmax, lens, ps, cc = PAGED[shape]
    w, inp = case(cache, qkv, B, Hq, Hkv, D, Lmax, lens)
    table, num_pages, _ = page_layout(w, inp["seq_lens"], ps, spare=0, seed=7)
    table[2, 1] = num_pages  # slot 2 holds more than one page; one past the pool
    got = _run_paged(w, inp, table, num_pages, ps, cc, expect=ftd.FTD_ERR_BAD_PAGE)
    ref = oracle.load().decode_step(w, inp, nthreads=8)
    others = [b for b in range(w.B) if b != 2]
    assert_close(got["out"][others], ref["out"][others], what=f"{shape} slots with valid tables")


def test_paged_context_refuses_contiguous_call_and_vice_versa():
    import torch
    w, inp = case("bf16", "bf16", 2, 8, 8, 128, 256, [3, 4])
    step = make_step(w, page_size=128, num_pages=4)
    x = torch.zeros(16, dtype=torch.int32, device="cuda")
    p = x.data_ptr()
    assert ftd.ftd_decode_mha(step.ctx, p, p, p, 0, p, p, p, 0, p, 0) == ftd.FTD_ERR_INVALID_ARG
    assert ftd.ftd_decode_mha_paged(step.ctx, p, p, p, 0, p, p, 0, p, 0, p, 0) == ftd.FTD_ERR_INVALID_ARG
    step.close()
    flat = make_step(w)
    assert ftd.ftd_decode_mha_paged(flat.ctx, p, p, p, 0, p, p, p, p, 0, p, 0) == ftd.FTD_ERR_INVALID_ARG
    flat.close()
