"""GPU parity of steps with several new tokens per slot (speculative verification)
against the float64 oracle.

Token j of slot b is appended at position L_b + j and attends to positions
0 .. L_b + j.  The cases put the new rows across tile boundaries (16-row
CUDA-core tiles, 128-row tensor-core tiles) and page boundaries, at the
overflow edge L_b + T = Lmax, with windows and half-precision output, and on
both kernels: multi-head caches run the CUDA-core kernel while a kv head
carries fewer than 8 query rows (group x tokens), the tensor-core kernel from
8 rows on (fp16/bf16, head_dim 128), and `cuda_core` forces the CUDA-core one.
"""
import numpy as np
import pytest

import decode_step_masked_gb300 as ftd
import oracle
from synthetic import Workload, gen_all
from tests.gpu_util import (TOL_MAXABS, assert_close, assert_same_bytes, dev, from_pages, make_step, rising_scores,
                            page_layout, run_step, to_pages, valid_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    ftd.build_library()
    ftd.load_library()


def case(cache, qkv, B, Hq, Hkv, D, Lmax, lens, T, bias=0.1, seed=31):
    w = Workload("mq", B=B, Hq=Hq, Hkv=Hkv, D=D, Lmax=Lmax, qkv_dtype=qkv, cache_dtype=cache,
                 bias_std=bias, seed=seed, q_len=T)
    return w, gen_all(w, seed=seed, seq_lens=np.array(lens, np.int32), fill_beyond="nan")


# (cache, qkv, B, Hq, Hkv, D, Lmax, lens, T, force_cuda_core); the kernel each takes is in the name
CASES = {
    "mha_bf16_T2_cc": ("bf16", "bf16", 4, 8, 8, 128, 512, [0, 14, 15, 300], 2, False),
    "mha_f16_T4_cc": ("f16", "f16", 4, 4, 4, 128, 512, [13, 126, 200, 508], 4, False),
    "mha_f32_d64_T3_cc": ("f32", "f32", 3, 4, 4, 64, 256, [0, 30, 253], 3, False),
    "mha_f32_T32_cc": ("f32", "f32", 2, 2, 2, 128, 256, [5, 224], 32, False),  # 8-row tiles, 5 tiles of new rows
    "mha_i8_T4_cc": ("i8", "f16", 4, 8, 8, 128, 512, [0, 29, 60, 508], 4, False),
    "mha_bf16_T8_tc": ("bf16", "bf16", 3, 4, 4, 128, 1024, [0, 124, 1016], 8, False),
    "mha_f16_T16_tc": ("f16", "f16", 2, 4, 4, 128, 1024, [120, 1008], 16, False),
    "gqa_bf16_T2_tc": ("bf16", "bf16", 4, 32, 4, 128, 1024, [0, 127, 126, 1022], 2, False),
    "gqa_bf16_T3_tc": ("bf16", "bf16", 3, 16, 2, 128, 1024, [125, 500, 1021], 3, False),
    "gqa_bf16_T3_cc": ("bf16", "bf16", 3, 16, 2, 128, 1024, [125, 500, 1021], 3, True),
    "mqa_f16_T5_tc": ("f16", "f16", 2, 8, 1, 128, 512, [124, 300], 5, False),
    "mqa_f16_T5_cc": ("f16", "f16", 2, 8, 1, 128, 512, [124, 300], 5, True),
    "gqa_i8_T2_tc": ("i8", "f16", 4, 16, 4, 128, 1024, [0, 127, 126, 1022], 2, False),  # 8 rows per kv head
    "mqa_i8_T3_tc": ("i8", "bf16", 3, 8, 1, 128, 512, [125, 0, 509], 3, False),         # 24 rows: 3 blocks
}


def check(w, inp, cc, window=0, out_dtype="f32", what=""):
    ref = oracle.load().decode_step(w, inp, nthreads=8, window=window)
    got = run_step(w, inp, force_cuda_core=cc, window=window, out_dtype=out_dtype)
    want = ftd.FTD_ERR_SEQ_OVERFLOW if ref["overflow"] else ftd.FTD_OK
    assert got["status"] == want, (ftd.ftd_status_str(got["status"]), what)
    assert got["out"].shape == ref["out"].shape
    assert_same_bytes(got["k_cache"], ref["k_cache"], f"{what} K after append")
    assert_same_bytes(got["v_cache"], ref["v_cache"], f"{what} V after append")
    if w.cache_dtype == "i8":
        assert_same_bytes(got["scales"], ref["scales"], f"{what} INT8 scales after append")
    return got, ref


@pytest.mark.parametrize("name", ["gqa_bf16_T2_tc", "gqa_bf16_T3_tc", "mqa_f16_T5_tc", "mqa_f16_T5_cc"])
def test_multi_token_rising_scores(name):
    """Scores climbing along the context: the per-column running maxima move inside a
    piece while each new token's column still has its own causal limit."""
    *args, cc = CASES[name]
    w, inp = case(*args)
    got, ref = check(w, rising_scores(w, inp), cc, what=f"{name} rising")
    assert_close(got["out"], ref["out"], what=f"{name} rising")


@pytest.mark.parametrize("name", list(CASES))
def test_multi_token_step(name):
    cache, qkv, B, Hq, Hkv, D, Lmax, lens, T, cc = CASES[name]
    w, inp = case(cache, qkv, B, Hq, Hkv, D, Lmax, lens, T)
    got, ref = check(w, inp, cc, what=name)
    assert_close(got["out"], ref["out"], i8=cache == "i8", what=name)


@pytest.mark.parametrize("window", [1, 3, 100, 129])
@pytest.mark.parametrize("name", ["mha_bf16_T2_cc", "mha_i8_T4_cc", "gqa_bf16_T3_tc", "mqa_f16_T5_cc",
                                  "mha_f32_T32_cc"])
def test_multi_token_window(name, window):
    cache, qkv, B, Hq, Hkv, D, Lmax, lens, T, cc = CASES[name]
    w, inp = case(cache, qkv, B, Hq, Hkv, D, Lmax, lens, T)
    got, ref = check(w, inp, cc, window=window, what=f"{name} W={window}")
    assert_close(got["out"], ref["out"], i8=cache == "i8", what=f"{name} W={window}")


def test_multi_token_overflow_edge():
    """L + T = Lmax fits; L + T = Lmax + 1 overflows (zero output, cache untouched, status)."""
    for cc in (False, True):
        w, inp = case("bf16", "bf16", 3, 16, 2, 128, 256, [252, 253, 100], 4)
        got, ref = check(w, inp, cc, what=f"overflow edge cc={cc}")
        assert ref["overflow"] and not got["out"][1].any()
        assert_close(got["out"][[0, 2]], ref["out"][[0, 2]], what="slots that fit")


def test_multi_token_half_output_matches_rounded_fp32():
    import torch
    w, inp = case("bf16", "bf16", 3, 32, 4, 128, 512, [0, 250, 400], 3)
    f32 = run_step(w, inp)
    half = run_step(w, inp, out_dtype="bf16")
    assert torch.equal(half["out_raw"].view(torch.int16), f32["out_raw"].to(torch.bfloat16).view(torch.int16))


def test_multi_token_equals_single_steps_on_the_gpu():
    """One T-token step and T single-token steps in a row give the same caches; outputs within the bar."""
    import torch
    w, inp = case("f16", "f16", 2, 16, 2, 128, 512, [126, 40], 3)
    multi = run_step(w, inp)
    w1 = w.with_(q_len=1)
    step = make_step(w1)
    kc, vc = dev(inp["k_cache"]), dev(inp["v_cache"])
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.float32, device="cuda")
    for j in range(3):
        step(dev(inp["q"][:, j]), dev(inp["k_new"][:, j]), dev(inp["v_new"][:, j]),
             dev(inp["seq_lens"] + j), out, bias=dev(inp["bias"]), k_cache=kc, v_cache=vc)
        torch.cuda.synchronize()
        assert_close(out.double().cpu().numpy(), multi["out"][:, j], what=f"token {j}")
    assert step.get_error() == ftd.FTD_OK
    step.close()
    assert_same_bytes(kc.cpu().numpy().view(np.float16), multi["k_cache"], "K caches")
    assert_same_bytes(vc.cpu().numpy().view(np.float16), multi["v_cache"], "V caches")


@pytest.mark.parametrize("cc", [False, True])
def test_multi_token_paged_across_pages(cc):
    """New tokens that straddle a page boundary land in both pages."""
    import torch
    T, ps = 4, 128
    w, inp = case("bf16", "bf16", 3, 16, 2, 128, 512, [126, 0, 380], T)
    table, num_pages, spare = page_layout(w, inp["seq_lens"], ps, spare=2, seed=9, q_len=T)
    ref = oracle.load().decode_step(w, inp, nthreads=8)
    nan = np.uint16(0x7FC0)
    kp = to_pages(w, inp["k_cache"], table, num_pages, ps, nan)
    vp = to_pages(w, inp["v_cache"], table, num_pages, ps, nan)
    step = make_step(w, force_cuda_core=cc, page_size=ps, num_pages=num_pages, q_len=T)
    kd, vd = dev(kp), dev(vp)
    out = torch.empty((w.B, T, w.Hq, w.D), dtype=torch.float32, device="cuda")
    step.paged(dev(inp["q"]), dev(inp["k_new"]), dev(inp["v_new"]), dev(table), dev(inp["seq_lens"]), out,
               bias=dev(inp["bias"]), k_pages=kd, v_pages=vd)
    torch.cuda.synchronize()
    assert step.get_error() == ftd.FTD_OK
    step.close()
    assert_close(out.double().cpu().numpy(), ref["out"], what="paged multi-token")
    L = inp["seq_lens"]
    got_k = from_pages(w, kd.cpu().numpy().view(np.uint16), table, ps, L, q_len=T)
    assert_same_bytes(got_k, valid_rows(w, ref["k_cache"], L, q_len=T), "K pages after append")
    got_v = from_pages(w, vd.cpu().numpy().view(np.uint16), table, ps, L, q_len=T)
    assert_same_bytes(got_v, valid_rows(w, ref["v_cache"], L, q_len=T), "V pages after append")
    assert_same_bytes(kd.cpu().numpy().view(np.uint16)[spare], kp[spare], "spare pages untouched")


# every option at once: paged cache, sliding window, several tokens per step, half output
COMBINED = {
    "i8_cc": ("i8", "f16", 3, 8, 8, 128, 512, [126, 0, 380], 3, False),
    "i8_tc": ("i8", "f16", 3, 16, 4, 128, 1024, [126, 700, 1000], 2, False),  # 8 rows: INT8 tensor cores
    "bf16_tc": ("bf16", "bf16", 3, 32, 4, 128, 1024, [126, 700, 1000], 2, False),
    "bf16_cc": ("bf16", "bf16", 3, 32, 4, 128, 1024, [126, 700, 1000], 2, True),
    "f16_mha_tc": ("f16", "f16", 2, 4, 4, 128, 512, [250, 100], 4, False),
}


@pytest.mark.parametrize("window", [0, 200])
@pytest.mark.parametrize("name", list(COMBINED))
def test_all_options_together(name, window):
    import torch
    cache, qkv, B, Hq, Hkv, D, Lmax, lens, T, cc = COMBINED[name]
    ps = 128
    w, inp = case(cache, qkv, B, Hq, Hkv, D, Lmax, lens, T)
    table, num_pages, spare = page_layout(w, inp["seq_lens"], ps, spare=2, seed=11, q_len=T)
    ref = oracle.load().decode_step(w, inp, nthreads=8, window=window)
    nan = {"i8": np.int8(127), "bf16": np.uint16(0x7FC0), "f16": np.float16(np.nan)}[cache]
    kp = to_pages(w, inp["k_cache"], table, num_pages, ps, nan)
    vp = to_pages(w, inp["v_cache"], table, num_pages, ps, nan)
    sp = None
    if cache == "i8":
        sp = np.stack([to_pages(w, inp["scales"][i][..., None], table, num_pages, ps, np.nan)[..., 0]
                       for i in range(2)])
    step = make_step(w, force_cuda_core=cc, out_dtype="bf16", window=window, page_size=ps, num_pages=num_pages,
                     q_len=T)
    kd, vd = dev(kp), dev(vp)
    sd = dev(sp) if sp is not None else None
    out = torch.full((w.B, T, w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    step.paged(dev(inp["q"]), dev(inp["k_new"]), dev(inp["v_new"]), dev(table), dev(inp["seq_lens"]), out,
               bias=dev(inp["bias"]), k_pages=kd, v_pages=vd, scales=sd)
    torch.cuda.synchronize()
    assert step.get_error() == ftd.FTD_OK
    step.close()
    got = out.double().cpu().numpy()
    tol = 1e-2 if cache == "i8" else TOL_MAXABS
    mant = 7  # bf16 output: fp32 bar plus half an output ulp
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref["out"]) + tol, 2.0 ** -126))) - mant)
    assert np.all(np.abs(got - ref["out"]) <= tol + 0.5 * ulp), name
    L = inp["seq_lens"]
    like = inp["k_cache"].dtype
    got_k = from_pages(w, kd.cpu().numpy().view(like), table, ps, L, q_len=T)
    assert_same_bytes(got_k, valid_rows(w, ref["k_cache"], L, q_len=T), f"{name} K pages after append")
    if cache == "i8":
        g = from_pages(w, sd.cpu().numpy()[0][..., None], table, ps, L, q_len=T)[..., 0]
        assert_same_bytes(g, valid_rows(w, ref["scales"][0], L, q_len=T), f"{name} K scales after append")
