"""GPU parity of the wide tensor-core kernel (kv heads carrying 32 or 64 query rows:
multi-query caches, wide groups, or groups x several new tokens) against the float64
oracle, on the same seeded inputs.

The cases cover blocks of 64 and 32 rows, kv heads with several blocks (passes),
ragged and tile-edge lengths, inactive and overflowing slots, sliding windows,
several tokens per step, paged caches, half outputs and scores that climb along the
context, which makes every row move its reference many times inside a piece (the
rescale of O in TMEM).  Appended rows are compared bit for bit.
"""
import numpy as np
import pytest

import decode_step_masked_gb300 as ftd
import oracle
from synthetic import Workload, gen_all
from tests.gpu_util import (TOL_MAXABS, assert_close, assert_same_bytes, dev, from_pages, make_step, page_layout,
                            rising_scores, run_step, to_pages, valid_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    ftd.build_library()
    ftd.load_library()


def case(cache, B, Hq, Hkv, Lmax, lens, T=1, seed=71, bias=0.1):
    w = Workload("wide", B=B, Hq=Hq, Hkv=Hkv, D=128, Lmax=Lmax, qkv_dtype=cache, cache_dtype=cache, bias_std=bias,
                 seed=seed, q_len=T)
    return w, gen_all(w, seed=seed, seq_lens=np.array(lens, np.int32), fill_beyond="nan")


def check(w, inp, window=0, out_dtype="f32", what=""):
    ref = oracle.load().decode_step(w, inp, nthreads=8, window=window)
    got = run_step(w, inp, window=window, out_dtype=out_dtype)
    want = ftd.FTD_ERR_SEQ_OVERFLOW if ref["overflow"] else ftd.FTD_OK
    assert got["status"] == want, (ftd.ftd_status_str(got["status"]), what)
    assert_same_bytes(got["k_cache"], ref["k_cache"], f"{what} K after append")
    assert_same_bytes(got["v_cache"], ref["v_cache"], f"{what} V after append")
    if out_dtype == "f32":
        assert_close(got["out"], ref["out"], what=what)
    else:
        mant = 7 if out_dtype == "bf16" else 10
        ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref["out"]) + TOL_MAXABS, 2.0 ** -126))) - mant)
        assert np.all(np.abs(got["out"] - ref["out"]) <= TOL_MAXABS + 0.5 * ulp), what
    return got, ref


LENS = [0, 127, 128, 129, 1000, 2047, -1, 2048]  # one position, tile edges, long, inactive, overflow


@pytest.mark.parametrize("cache", ["bf16", "f16"])
@pytest.mark.parametrize("Hq,Hkv", [(64, 1), (32, 1), (64, 2), (128, 1), (96, 1), (128, 4)])
def test_wide_single_token(cache, Hq, Hkv):
    """Blocks of 64 rows (64/1, 128/1 in two passes, 128/4 = 32 rows -> 32), 32 rows (32/1, 64/2,
    96/1 in three passes)."""
    w, inp = case(cache, B=len(LENS), Hq=Hq, Hkv=Hkv, Lmax=2048, lens=LENS)
    got, _ = check(w, inp, what=f"wide {Hq}/{Hkv} {cache}")
    assert not got["out"][[6, 7]].any(), "inactive and overflowing slots are zero"


def test_wide_no_bias_and_many_tiles_per_cta():
    """The MQA shape at a long context: each CTA streams several tiles and starts new pieces
    mid-range; no bias."""
    w, inp = case("bf16", B=16, Hq=64, Hkv=1, Lmax=8192, lens=[8191] * 8 + [4000, 129, 7000, 8000, 1, 6143, 5000, 7777],
                  bias=None)
    check(w, inp, what="wide MQA long")


@pytest.mark.parametrize("Hq,Hkv,T", [(8, 1, 4), (16, 2, 4), (16, 1, 4), (8, 1, 8), (4, 1, 16), (32, 8, 8)])
def test_wide_multi_token(Hq, Hkv, T):
    """Several new tokens per step with group x tokens = 32 or 64 rows per kv head."""
    w, inp = case("bf16", B=4, Hq=Hq, Hkv=Hkv, Lmax=1024, lens=[0, 125, 1024 - T, 500], T=T)
    check(w, inp, what=f"wide multi-token {Hq}/{Hkv} T{T}")


@pytest.mark.parametrize("window", [0, 300])
@pytest.mark.parametrize("Hq,T", [(32, 1), (64, 1), (8, 4)])
def test_wide_many_short_segments(Hq, T, window):
    """200 slots with contexts up to 1000 tokens, some inactive: about five tiles per block,
    so blocks cross several pieces, and most segments end in a merge of partials; with a
    window, most pieces start on a tile whose rows before the window start are zeroed."""
    rng = np.random.default_rng(91)
    lens = rng.integers(-1, 1000, size=200)
    w, inp = case("bf16", B=200, Hq=Hq, Hkv=1, Lmax=1024, lens=lens, T=T, seed=92)
    check(w, inp, window=window, what=f"wide short segments Hq{Hq} T{T} window {window}")


@pytest.mark.parametrize("rise", [20.0, 60.0])
@pytest.mark.parametrize("Hq,Hkv,T", [(64, 1, 1), (32, 1, 1), (8, 1, 4), (16, 1, 4)])
def test_wide_rising_scores(Hq, Hkv, T, rise):
    """Scores climbing along the context: the row references move again and again within a
    piece, and O is rescaled in TMEM each time."""
    w, inp = case("bf16", B=3, Hq=Hq, Hkv=Hkv, Lmax=4096, lens=[4095 - T + 1, 1500, 700], T=T, seed=72)
    check(w, rising_scores(w, inp, rise_log2=rise), what=f"wide rising {rise} {Hq}/{Hkv} T{T}")


@pytest.mark.parametrize("window", [1, 100, 128, 129, 1000])
@pytest.mark.parametrize("Hq,Hkv,T", [(64, 1, 1), (8, 1, 4)])
def test_wide_window(Hq, Hkv, T, window):
    w, inp = case("f16", B=4, Hq=Hq, Hkv=Hkv, Lmax=2048, lens=[2048 - T, 300, 0, 1280], T=T, seed=73)
    check(w, inp, window=window, what=f"wide window {window} {Hq}/{Hkv} T{T}")


@pytest.mark.parametrize("out_dtype", ["bf16", "f16"])
def test_wide_half_output(out_dtype):
    w, inp = case("bf16", B=3, Hq=64, Hkv=1, Lmax=1024, lens=[1000, 3, 512], seed=74)
    check(w, inp, out_dtype=out_dtype, what=f"wide out {out_dtype}")


@pytest.mark.parametrize("rows,T,window", [(64, 1, 0), (64, 4, 0), (64, 4, 200), (32, 1, 0), (32, 4, 200)])
def test_wide_paged(rows, T, window):
    """Pages of 128 tokens in shuffled order, new tokens across a page boundary, a window;
    blocks of 64 and of 32 query rows."""
    import torch
    ps = 128
    w, inp = case("bf16", B=3, Hq=rows // T, Hkv=1, Lmax=1024, lens=[126, 0, 900], T=T, seed=75)
    table, num_pages, spare = page_layout(w, inp["seq_lens"], ps, spare=2, seed=12, q_len=T)
    ref = oracle.load().decode_step(w, inp, nthreads=8, window=window)
    nan = np.uint16(0x7FC0)
    kp = to_pages(w, inp["k_cache"], table, num_pages, ps, nan)
    vp = to_pages(w, inp["v_cache"], table, num_pages, ps, nan)
    step = make_step(w, page_size=ps, num_pages=num_pages, q_len=T, window=window)
    kd, vd = dev(kp), dev(vp)
    shape = (w.B, T, w.Hq, w.D) if T > 1 else (w.B, w.Hq, w.D)
    out = torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
    step.paged(dev(inp["q"]), dev(inp["k_new"]), dev(inp["v_new"]), dev(table), dev(inp["seq_lens"]), out,
               bias=dev(inp["bias"]), k_pages=kd, v_pages=vd)
    torch.cuda.synchronize()
    assert step.get_error() == ftd.FTD_OK
    step.close()
    assert_close(out.double().cpu().numpy(), ref["out"], what=f"wide paged T{T} window {window}")
    L = inp["seq_lens"]
    got_k = from_pages(w, kd.cpu().numpy().view(np.uint16), table, ps, L, q_len=T)
    assert_same_bytes(got_k, valid_rows(w, ref["k_cache"], L, q_len=T), "K pages after append")
    got_v = from_pages(w, vd.cpu().numpy().view(np.uint16), table, ps, L, q_len=T)
    assert_same_bytes(got_v, valid_rows(w, ref["v_cache"], L, q_len=T), "V pages after append")
