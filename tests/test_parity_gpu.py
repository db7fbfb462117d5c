"""GPU parity: the CUDA decode step against the float64 oracle on the same seeded inputs.

Append is compared bit for bit (caches and INT8 scales); attention outputs
within max-abs 2e-3 and relative L2 1e-3 (fp32/fp16/bf16 caches) or max-abs
1e-2 (INT8 cache, oracle on the dequantised values).
"""
import numpy as np
import pytest

import decode_step_masked_gb300 as ftd
import oracle
from synthetic import WORKLOADS, Workload, gen_all, gen_qkv, gen_seq_lens
from tests.gpu_util import (assert_close, assert_same_bytes, dev, device_view, fill_device_cache,
                            fill_device_scales, rising_scores, run_step)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    ftd.build_library()
    ftd.load_library()


def small(cache, qkv, B, Hq, Hkv, D, Lmax, lens, bias=0.1, seed=11):
    w = Workload("case", B=B, Hq=Hq, Hkv=Hkv, D=D, Lmax=Lmax, qkv_dtype=qkv, cache_dtype=cache,
                 bias_std=bias, seed=seed)
    return w, gen_all(w, seed=seed, seq_lens=np.array(lens, np.int32), fill_beyond="nan")


def check_step(w, inp, softmax_scale=0.0, use_bias=True, what="", force_cuda_core=False):
    o = oracle.load()
    ref_inp = dict(inp)
    if not use_bias:
        ref_inp["bias"] = None
    ref = o.decode_step(w, ref_inp, softmax_scale=softmax_scale, nthreads=8)
    got = run_step(w, inp, softmax_scale=softmax_scale, use_bias=use_bias, force_cuda_core=force_cuda_core)
    assert_same_bytes(got["k_cache"], ref["k_cache"], f"{what} K cache after append")
    assert_same_bytes(got["v_cache"], ref["v_cache"], f"{what} V cache after append")
    if w.cache_dtype == "i8":
        assert_same_bytes(got["scales"], ref["scales"], f"{what} INT8 scales after append")
    assert_close(got["out"], ref["out"], i8=w.cache_dtype == "i8", what=what)
    want = ftd.FTD_ERR_SEQ_OVERFLOW if ref["overflow"] else ftd.FTD_OK
    assert got["status"] == want, (ftd.ftd_status_str(got["status"]), what)
    return got, ref


def test_tiny_workload():
    w = WORKLOADS["tiny"]
    check_step(w, gen_all(w), what="tiny")


LENS = [0, 1, 15, 16, 17, 100, 255, 300]  # ctx 1, tile edges, ragged tails


@pytest.mark.parametrize("cache", ["f32", "f16", "bf16", "i8"])
@pytest.mark.parametrize("qkv", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
def test_dtype_grid(cache, qkv, D):
    w, inp = small(cache, qkv, B=len(LENS), Hq=4, Hkv=4, D=D, Lmax=304, lens=LENS)
    check_step(w, inp, what=f"{cache}/{qkv}/D{D}")


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (8, 4), (8, 2), (8, 1), (16, 2), (16, 1), (32, 1), (64, 8), (24, 8),
                                     (12, 2)])
@pytest.mark.parametrize("cache", ["bf16", "f16", "i8"])
@pytest.mark.parametrize("path", ["auto", "cuda_core"])
def test_gqa_mqa(Hq, Hkv, cache, path):
    """Groups of 8 or 16 query heads on fp16/bf16 caches take the tensor-core kernel under "auto"."""
    qkv = "f16" if cache == "i8" else cache
    w, inp = small(cache, qkv, B=3, Hq=Hq, Hkv=Hkv, D=128, Lmax=512, lens=[511, 37, 200])
    check_step(w, inp, what=f"gqa {Hq}/{Hkv} {cache} {path}", force_cuda_core=path == "cuda_core")


@pytest.mark.parametrize("lens", [[16000], [127], [128], [0], [129, 255, 256, 383, 1000, 3]])
@pytest.mark.parametrize("cache", ["bf16", "f16"])
def test_tensor_core_gqa_tile_edges(lens, cache):
    """Tensor-core path: 128-row tile edges, one token, and a long sequence merged across many CTAs."""
    Lmax = 16384 if max(lens) >= 4096 else 1024
    w, inp = small(cache, cache, B=len(lens), Hq=16, Hkv=2, D=128, Lmax=Lmax, lens=lens)
    check_step(w, inp, what=f"tc edges {lens} {cache}")


@pytest.mark.parametrize("cache", ["bf16", "f16"])
@pytest.mark.parametrize("B,Hq,Hkv,Lmax,lens", [
    (16, 8, 1, 8192, [8191] * 16),                                    # ~6.7 tiles per CTA, G = 8
    (8, 32, 2, 8192, [8191, 4000, 7000, 129, 8000, 6143, 5000, 7777]),  # G = 16, ragged
])
def test_tensor_core_many_tiles_per_cta(cache, B, Hq, Hkv, Lmax, lens):
    """Each CTA streams several 128-row tiles through its stage ring and starts new
    segments mid-range: the case that exposed a waiter skipping barrier phases."""
    w, inp = small(cache, cache, B=B, Hq=Hq, Hkv=Hkv, D=128, Lmax=Lmax, lens=lens, bias=0.1)
    check_step(w, inp, what=f"tc many tiles {B}x{Hq}/{Hkv} {cache}")


@pytest.mark.parametrize("B,Hq,Hkv,Lmax,lens", [
    (16, 64, 8, 8192, [8191] * 16),                                      # 70B-shaped, ~54 tiles per CTA
    (8, 16, 1, 8192, [8191, 4000, 7000, 129, 8000, 6143, 5000, 7777]),  # 16 rows: 2 blocks of 8, ragged
    (6, 16, 2, 1024, [16000 % 1024, 127, 128, 0, 129, 1023]),           # tile edges, one token
])
def test_tensor_core_int8(B, Hq, Hkv, Lmax, lens):
    """INT8 caches with blocks of 8 query rows: codes converted to fp16 on chip, scales on the
    scores and in the weights; appended codes and scales bit for bit."""
    w, inp = small("i8", "f16", B=B, Hq=Hq, Hkv=Hkv, D=128, Lmax=Lmax, lens=lens, bias=0.1)
    check_step(w, inp, what=f"tc int8 {B}x{Hq}/{Hkv}")


def test_inactive_and_overflow_slots():
    w, inp = small("bf16", "bf16", B=6, Hq=4, Hkv=2, D=128, Lmax=128, lens=[-1, 127, 128, 5, 1000, -7])
    got, ref = check_step(w, inp, what="inactive/overflow")
    assert not got["out"][[0, 2, 4, 5]].any(), "inactive and overflowing slots must be zero"
    assert got["status"] == ftd.FTD_ERR_SEQ_OVERFLOW


def test_error_is_sticky_then_cleared():
    import torch
    w, inp = small("bf16", "bf16", B=2, Hq=2, Hkv=2, D=64, Lmax=32, lens=[32, 3])
    step = ftd.DecodeStep(w.B, w.Hq, w.Hkv, w.D, w.Lmax, w.qkv_dtype, w.cache_dtype)
    run_step(w, inp, step=step)  # reads and clears the overflow
    assert step.get_error() == ftd.FTD_OK
    inp2 = dict(inp, seq_lens=np.array([3, 4], np.int32))
    assert run_step(w, inp2, step=step)["status"] == ftd.FTD_OK
    step.close()
    torch.cuda.synchronize()


def test_all_inactive():
    w, inp = small("f16", "f16", B=4, Hq=4, Hkv=4, D=128, Lmax=64, lens=[-1, -1, -1, -1])
    got, _ = check_step(w, inp, what="all inactive")
    assert not got["out"].any()


def test_no_bias_and_custom_scale():
    w, inp = small("bf16", "f32", B=3, Hq=8, Hkv=2, D=128, Lmax=256, lens=[200, 9, 255])
    check_step(w, inp, use_bias=False, what="no bias")
    check_step(w, inp, softmax_scale=0.37, what="scale 0.37")


def test_one_long_sequence_split_across_many_workers():
    # one segment spread over hundreds of warps: exercises the log-sum-exp merge
    w, inp = small("bf16", "bf16", B=1, Hq=1, Hkv=1, D=128, Lmax=16384, lens=[16000], bias=None)
    check_step(w, inp, what="one long sequence")


def test_many_short_segments_per_worker():
    rng = np.random.default_rng(5)
    lens = rng.integers(0, 40, 64)
    w, inp = small("f16", "f16", B=64, Hq=32, Hkv=32, D=128, Lmax=48, lens=lens)
    check_step(w, inp, what="many short segments")


def test_large_scores_stay_finite():
    w, inp = small("f32", "f32", B=2, Hq=4, Hkv=4, D=64, Lmax=512, lens=[400, 77], bias=None)
    inp = dict(inp, q=(inp["q"] * np.float32(40.0)).astype(np.float32))
    check_step(w, inp, what="large scores")


@pytest.mark.parametrize("cache,Hq,Hkv,cc", [
    ("bf16", 16, 2, False),  # tensor cores, 8 query columns
    ("f16", 32, 2, False),   # tensor cores, 16 query columns
    ("bf16", 16, 2, True),   # CUDA cores, grouped
    ("f16", 4, 4, False),    # CUDA cores, one query row per kv head
])
def test_scores_rising_along_the_context(cache, Hq, Hkv, cc):
    """Scores that climb by ~40 (base 2) along each context move every row's running
    maximum many times, tiles after the first included, so the softmax's rescaling
    of earlier weights and partial outputs is exercised, not just its first tile."""
    w, inp = small(cache, cache, B=4, Hq=Hq, Hkv=Hkv, D=128, Lmax=2048, lens=[1500, 700, 130, 2047])
    check_step(w, rising_scores(w, inp), what=f"rising scores {cache} {Hq}/{Hkv}", force_cuda_core=cc)


def test_consecutive_steps_continue_the_sequence():
    """Two decode steps in a row on one context: the second sees the first's append."""
    import torch
    w, inp = small("bf16", "bf16", B=4, Hq=8, Hkv=4, D=128, Lmax=256, lens=[10, 100, 250, 0])
    o = oracle.load()
    step = ftd.DecodeStep(w.B, w.Hq, w.Hkv, w.D, w.Lmax, w.qkv_dtype, w.cache_dtype)
    q, kn, vn, bias = dev(inp["q"]), dev(inp["k_new"]), dev(inp["v_new"]), dev(inp["bias"])
    kc, vc = dev(inp["k_cache"]), dev(inp["v_cache"])
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.float32, device="cuda")
    ref_inp = dict(inp)
    lens = inp["seq_lens"].copy()
    for it in range(3):
        step(q, kn, vn, dev(lens), out, bias=bias, k_cache=kc, v_cache=vc)
        ref = o.decode_step(w, dict(ref_inp, seq_lens=lens))
        torch.cuda.synchronize()
        assert_close(out.cpu().numpy().astype(np.float64), ref["out"], what=f"step {it}")
        assert_same_bytes(kc.cpu().numpy().view(np.uint16), ref["k_cache"], f"K after step {it}")
        ref_inp = dict(ref_inp, k_cache=ref["k_cache"], v_cache=ref["v_cache"])
        lens = lens + 1
    assert step.get_error() == ftd.FTD_OK
    step.close()


def test_pool_pointers_and_host_entry_point():
    """NULL caches select the context's own pool; the host-buffer entry point gives the same result."""
    import torch
    w, inp = small("i8", "f16", B=3, Hq=4, Hkv=2, D=128, Lmax=96, lens=[95, 20, 63])
    ref = oracle.load().decode_step(w, inp)
    step = ftd.DecodeStep(w.B, w.Hq, w.Hkv, w.D, w.Lmax, w.qkv_dtype, w.cache_dtype)
    kp, vp, sp = step.cache_ptrs()
    assert kp and vp and sp
    kview = device_view(kp, inp["k_cache"].shape, np.int8)
    vview = device_view(vp, inp["v_cache"].shape, np.int8)
    sview = device_view(sp, inp["scales"].shape, np.float32)
    kview.copy_(dev(inp["k_cache"]))
    vview.copy_(dev(inp["v_cache"]))
    sview.copy_(dev(inp["scales"]))
    torch.cuda.synchronize()
    host = {k: np.ascontiguousarray(inp[k]) for k in ("q", "k_new", "v_new", "bias", "seq_lens")}
    out = np.zeros((w.B, w.Hq, w.D), np.float32)
    s = torch.cuda.current_stream().cuda_stream
    st = ftd.ftd_decode_mha_host(step.ctx, host["q"].ctypes.data, host["k_new"].ctypes.data,
                                 host["v_new"].ctypes.data, host["bias"].ctypes.data, 0, 0,
                                 host["seq_lens"].ctypes.data, 0, out.ctypes.data, s)
    ftd.check(st)
    assert_close(out.astype(np.float64), ref["out"], i8=True, what="host entry point / pool")
    assert_same_bytes(kview.cpu().numpy(), ref["k_cache"], "pool K after append")
    assert_same_bytes(sview.cpu().numpy(), ref["scales"], "pool scales after append")
    assert step.get_error() == ftd.FTD_OK
    step.close()


@pytest.mark.parametrize("cache,Hq,Hkv", [("bf16", 2, 2), ("i8", 2, 2), ("f16", 8, 1)])
def test_maximum_batch(cache, Hq, Hkv):
    """1024 slots (the largest batch), ragged short contexts with inactive and overflowing slots:
    the prefix over slots and the weighted split search over the whole batch."""
    rng = np.random.default_rng(5)
    lens = rng.integers(-3, 64, size=1024).astype(np.int32)  # negative: inactive; 63: at Lmax - 1
    lens[17] = 64  # overflow
    w, inp = small(cache, "f16" if cache != "bf16" else "bf16", B=1024, Hq=Hq, Hkv=Hkv, D=64, Lmax=64,
                   lens=lens)
    check_step(w, inp, what=f"1024 slots {cache} Hq{Hq} Hkv{Hkv}")


def test_current_context_entry_point():
    """ftd_decode_mha_current (the specified ten-argument call) runs on the most recently
    initialised context and gives the same bytes as ftd_decode_mha on it; after that context
    is destroyed it refuses."""
    import torch
    w, inp = small("bf16", "bf16", B=3, Hq=16, Hkv=2, D=128, Lmax=256, lens=[0, 130, 255])
    step = ftd.DecodeStep(w.B, w.Hq, w.Hkv, w.D, w.Lmax, w.qkv_dtype, w.cache_dtype)
    q, kn, vn, bias, sl = (dev(inp[k]) for k in ("q", "k_new", "v_new", "bias", "seq_lens"))
    outs, caches = [], []
    for current in (False, True):
        kc, vc = dev(inp["k_cache"]), dev(inp["v_cache"])
        out = torch.full((w.B, w.Hq, w.D), float("nan"), dtype=torch.float32, device="cuda")
        s = torch.cuda.current_stream().cuda_stream
        args = (q.data_ptr(), kn.data_ptr(), vn.data_ptr(), bias.data_ptr(), kc.data_ptr(), vc.data_ptr(),
                sl.data_ptr(), 0, out.data_ptr(), s)
        st = ftd.ftd_decode_mha_current(*args) if current else ftd.ftd_decode_mha(step.ctx, *args)
        ftd.check(st)
        torch.cuda.synchronize()
        outs.append(out.cpu().numpy())
        caches.append(kc.cpu().numpy())
    assert step.get_error() == ftd.FTD_OK
    assert_same_bytes(outs[1], outs[0], "ftd_decode_mha_current output")
    assert_same_bytes(caches[1], caches[0], "ftd_decode_mha_current append")
    step.close()
    assert ftd.ftd_decode_mha_current(0, 0, 0, 0, 0, 0, 0, 0, 0, 0) == ftd.FTD_ERR_INVALID_ARG


def test_host_entry_point_with_pinned_buffers():
    """Pinned host buffers take the direct path (one launch that reads the inputs in place and
    writes the output to the host); the result matches the oracle and the caches get the
    appended rows."""
    import torch
    w, inp = small("bf16", "bf16", B=3, Hq=16, Hkv=2, D=128, Lmax=256, lens=[0, 130, 255])
    ref = oracle.load().decode_step(w, inp)
    step = ftd.DecodeStep(w.B, w.Hq, w.Hkv, w.D, w.Lmax, w.qkv_dtype, w.cache_dtype)
    kc, vc = dev(inp["k_cache"]), dev(inp["v_cache"])

    def pinned(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        return torch.from_numpy(a).pin_memory()

    hq, hk, hv, hb, hl = (pinned(inp[k]) for k in ("q", "k_new", "v_new", "bias", "seq_lens"))
    out = torch.full((w.B, w.Hq, w.D), float("nan"), dtype=torch.float32).pin_memory()
    s = torch.cuda.current_stream().cuda_stream
    for rep in range(2):  # the second call reuses the looked-up device addresses
        kcur, vcur = kc.clone(), vc.clone()
        n0 = ftd.ftd_kernel_launches()
        ftd.check(ftd.ftd_decode_mha_host(step.ctx, hq.data_ptr(), hk.data_ptr(), hv.data_ptr(), hb.data_ptr(),
                                          kcur.data_ptr(), vcur.data_ptr(), hl.data_ptr(), 0, out.data_ptr(), s))
        assert ftd.ftd_kernel_launches() - n0 == 1, "pinned buffers should take the one-launch direct path"
        assert_close(out.numpy().astype(np.float64), ref["out"], what=f"pinned host entry point, call {rep}")
        assert_same_bytes(kcur.cpu().numpy().view(np.uint16), ref["k_cache"], "K after append")
    assert step.get_error() == ftd.FTD_OK
    step.close()


def test_host_entry_point_lengths_change_between_calls():
    """The direct host path reads the lengths in place: calls that rewrite the pinned
    lengths between them each see their own lengths."""
    import torch
    w, inp = small("bf16", "bf16", B=3, Hq=16, Hkv=2, D=128, Lmax=256, lens=[255, 255, 255])
    step = ftd.DecodeStep(w.B, w.Hq, w.Hkv, w.D, w.Lmax, w.qkv_dtype, w.cache_dtype)
    kc, vc = dev(inp["k_cache"]), dev(inp["v_cache"])

    def pinned(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        return torch.from_numpy(a).pin_memory()

    hq, hk, hv, hb, hl = (pinned(inp[k]) for k in ("q", "k_new", "v_new", "bias", "seq_lens"))
    out = torch.full((w.B, w.Hq, w.D), float("nan"), dtype=torch.float32).pin_memory()
    s = torch.cuda.current_stream().cuda_stream
    for lens in ([0, 130, 255], [200, 7, 129], [128, 255, 1], [0, 130, 255]):
        hl.copy_(torch.tensor(lens, dtype=torch.int32))
        ref = oracle.load().decode_step(w, dict(inp, seq_lens=np.array(lens, np.int32)))
        kcur, vcur = kc.clone(), vc.clone()
        ftd.check(ftd.ftd_decode_mha_host(step.ctx, hq.data_ptr(), hk.data_ptr(), hv.data_ptr(), hb.data_ptr(),
                                          kcur.data_ptr(), vcur.data_ptr(), hl.data_ptr(), 0, out.data_ptr(), s))
        assert_close(out.numpy().astype(np.float64), ref["out"], what=f"host entry point, lengths {lens}")
        assert_same_bytes(kcur.cpu().numpy().view(np.uint16), ref["k_cache"], f"K after append, lengths {lens}")
    assert step.get_error() == ftd.FTD_OK
    step.close()


# ------------------------------------------------------------- full size
SAMPLED = {"7b": [(0, 0), (3, 17), (7, 31)], "13b": [(0, 5), (11, 39), (31, 0), (17, 22)],
           "70b": [(0, 0), (5, 37), (15, 63)], "int8": [(0, 1), (33, 30), (63, 31)],
           "mqa": [(0, 0), (21, 17), (63, 63)], "70b_i8": [(0, 0), (7, 40), (15, 63)]}


@pytest.mark.parametrize("name", ["7b", "13b", "70b", "int8", "mqa", "70b_i8"])
def test_full_size_workload_sampled(name):
    """Full-size workloads in the launch configuration the bench times; the oracle checks
    sampled (slot, head) outputs one slot at a time, and every appended row bit for bit."""
    import torch
    w = WORKLOADS[name]
    lens = gen_seq_lens(w)
    q, kn, vn, bias = gen_qkv(w)
    kc = fill_device_cache(w, w.seed, lens, "k")
    vc = fill_device_cache(w, w.seed, lens, "v")
    sc = fill_device_scales(w, w.seed, lens) if w.cache_dtype == "i8" else None
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.float32, device="cuda")
    step = ftd.DecodeStep(w.B, w.Hq, w.Hkv, w.D, w.Lmax, w.qkv_dtype, w.cache_dtype)
    step(dev(q), dev(kn), dev(vn), dev(lens), out, bias=None if bias is None else dev(bias),
         k_cache=kc, v_cache=vc, scales=sc)
    torch.cuda.synchronize()
    assert step.get_error() == ftd.FTD_OK
    got = out.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    o = oracle.load()
    idx = torch.arange(w.B, device="cuda")
    pos = torch.from_numpy(lens.astype(np.int64)).cuda()
    k_rows = kc[idx, :, pos, :].cpu().numpy()      # [B, Hkv, D]
    v_rows = vc[idx, :, pos, :].cpu().numpy()
    slots = sorted({b for b, _ in SAMPLED[name]})
    w1 = w.with_(B=1)
    for b in slots:
        from synthetic import gen_cache_slot, gen_scales_slot
        sub = dict(q=q[b:b + 1], k_new=kn[b:b + 1], v_new=vn[b:b + 1], bias=bias,
                   k_cache=gen_cache_slot(w, w.seed, "k", b, lens[b])[None],
                   v_cache=gen_cache_slot(w, w.seed, "v", b, lens[b])[None],
                   seq_lens=lens[b:b + 1], scales=None)
        if w.cache_dtype == "i8":
            sub["scales"] = np.stack([gen_scales_slot(w, w.seed, "k", b, lens[b])[None],
                                      gen_scales_slot(w, w.seed, "v", b, lens[b])[None]])
        ref = o.decode_step(w1, sub, nthreads=8)
        L = int(lens[b])
        assert_same_bytes(k_rows[b], ref["k_cache"][0, :, L, :].view(k_rows.dtype), f"{name} K row slot {b}")
        assert_same_bytes(v_rows[b], ref["v_cache"][0, :, L, :].view(v_rows.dtype), f"{name} V row slot {b}")
        heads = [h for bb, h in SAMPLED[name] if bb == b]
        assert_close(got[b, heads], ref["out"][0, heads], i8=w.cache_dtype == "i8", what=f"{name} slot {b}")
    step.close()
