"""ftd_decode_mha_noalloc against ftd_decode_mha on the same inputs, two calls in a row.

The no-allocation entry point serves callers that may not call cudaMalloc (a
plugin whose host runtime owns all device memory, or a loop that forbids
allocation after start-up); its scratch is a static device array shared by
every call.  This file is named to run last so that a run stopping at the
first failure has already run every other test; it also passes on its own.
"""
import numpy as np
import pytest

import decode_step_masked_gb300 as ftd
from synthetic import Workload, gen_all
from tests.gpu_util import TOL_MAXABS, TOL_RELL2, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    ftd.build_library()
    ftd.load_library()


def _case(lens, seed):
    w = Workload("noalloc", B=len(lens), Hq=16, Hkv=4, D=128, Lmax=1024, qkv_dtype="bf16", cache_dtype="bf16",
                 bias_std=0.1, seed=seed)
    return w, gen_all(w, seed=seed, seq_lens=np.array(lens, np.int32), fill_beyond="nan")


def test_noalloc_matches_context_entry_point_twice():
    import torch
    cases = [_case([1000, 3, 517, 64, -1, 255], seed=21), _case([15, 800, 1023, 2, 300, 999], seed=22)]
    w0 = cases[0][0]
    step = ftd.DecodeStep(w0.B, w0.Hq, w0.Hkv, w0.D, w0.Lmax, w0.qkv_dtype, w0.cache_dtype)
    cfg = ftd.FtdConfig(w0.B, w0.Hq, w0.Hkv, w0.D, w0.Lmax, ftd.FTD_BF16, ftd.FTD_BF16, 0.0)
    s = torch.cuda.current_stream().cuda_stream
    for call, (w, inp) in enumerate(cases):
        q, kn, vn, bias, sl = (dev(inp[k]) for k in ("q", "k_new", "v_new", "bias", "seq_lens"))
        kc_a, vc_a = dev(inp["k_cache"]), dev(inp["v_cache"])
        kc_b, vc_b = dev(inp["k_cache"]), dev(inp["v_cache"])
        out_a = torch.full((w.B, w.Hq, w.D), float("nan"), device="cuda")
        out_b = torch.full((w.B, w.Hq, w.D), float("nan"), device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        step(q, kn, vn, sl, out_a, bias=bias, k_cache=kc_a, v_cache=vc_a)
        st = ftd.ftd_decode_mha_noalloc(cfg, q.data_ptr(), kn.data_ptr(), vn.data_ptr(), bias.data_ptr(),
                                        kc_b.data_ptr(), vc_b.data_ptr(), sl.data_ptr(), 0, out_b.data_ptr(),
                                        err.data_ptr(), s)
        assert st == ftd.FTD_OK, ftd.ftd_last_error()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        a = out_a.cpu().numpy().astype(np.float64)
        b = out_b.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(b)), f"call {call}: non-finite output"
        assert np.max(np.abs(a - b)) <= TOL_MAXABS, f"call {call}"
        assert np.linalg.norm(a - b) / np.linalg.norm(a) <= TOL_RELL2, f"call {call}"
        assert torch.equal(kc_a, kc_b) and torch.equal(vc_a, vc_b), f"call {call}: appended rows differ"
    assert step.get_error() == ftd.FTD_OK
    step.close()


def test_noalloc_reports_overflow_and_rejects_oversized_configs():
    import torch
    w, inp = _case([1024, 5], seed=23)  # slot 0 overflows (seq_len == max_len)
    cfg = ftd.FtdConfig(w.B, w.Hq, w.Hkv, w.D, w.Lmax, ftd.FTD_BF16, ftd.FTD_BF16, 0.0)
    q, kn, vn, sl = (dev(inp[k]) for k in ("q", "k_new", "v_new", "seq_lens"))
    kc, vc = dev(inp["k_cache"]), dev(inp["v_cache"])
    out = torch.full((w.B, w.Hq, w.D), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    st = ftd.ftd_decode_mha_noalloc(cfg, q.data_ptr(), kn.data_ptr(), vn.data_ptr(), 0, kc.data_ptr(),
                                    vc.data_ptr(), sl.data_ptr(), 0, out.data_ptr(), err.data_ptr(), s)
    assert st == ftd.FTD_OK, ftd.ftd_last_error()
    torch.cuda.synchronize()
    assert int(err.item()) & 1, "overflow bit"
    assert not out[0].any().item() and torch.isfinite(out[1]).all().item()
    # 1024 slots x 128 kv heads of partials do not fit in the static array
    big = ftd.FtdConfig(1024, 128, 128, 128, 4096, ftd.FTD_BF16, ftd.FTD_BF16, 0.0)
    st = ftd.ftd_decode_mha_noalloc(big, q.data_ptr(), kn.data_ptr(), vn.data_ptr(), 0, kc.data_ptr(),
                                    vc.data_ptr(), sl.data_ptr(), 0, out.data_ptr(), 0, s)
    assert st == ftd.FTD_ERR_INVALID_ARG
    assert "static array" in ftd.ftd_last_error()


def test_noalloc_with_window_half_output_and_several_tokens():
    """The options the no-allocation entry point accepts (all but pages) give the context path's bytes."""
    import torch
    T = 3
    w = Workload("noalloc", B=3, Hq=8, Hkv=8, D=128, Lmax=512, qkv_dtype="f16", cache_dtype="i8", bias_std=0.1,
                 seed=24, q_len=T)
    inp = gen_all(w, seed=24, seq_lens=np.array([200, 0, 509], np.int32), fill_beyond="nan")
    opts = dict(out_dtype="bf16", window=64, q_len=T)
    step = ftd.DecodeStep(w.B, w.Hq, w.Hkv, w.D, w.Lmax, w.qkv_dtype, w.cache_dtype, **opts)
    cfg = ftd.FtdConfig(w.B, w.Hq, w.Hkv, w.D, w.Lmax, ftd.FTD_F16, ftd.FTD_I8, 0.0, ftd.FTD_BF16, 64, 0, 0, T)
    s = torch.cuda.current_stream().cuda_stream
    q, kn, vn, bias, sl = (dev(inp[k]) for k in ("q", "k_new", "v_new", "bias", "seq_lens"))
    outs, caches = [], []
    for use_noalloc in (False, True):
        kc, vc, sc = dev(inp["k_cache"]), dev(inp["v_cache"]), dev(inp["scales"])
        out = torch.full((w.B, T, w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
        if use_noalloc:
            err = torch.zeros(1, dtype=torch.int32, device="cuda")
            st = ftd.ftd_decode_mha_noalloc(cfg, q.data_ptr(), kn.data_ptr(), vn.data_ptr(), bias.data_ptr(),
                                            kc.data_ptr(), vc.data_ptr(), sl.data_ptr(), sc.data_ptr(),
                                            out.data_ptr(), err.data_ptr(), s)
            assert st == ftd.FTD_OK, ftd.ftd_last_error()
        else:
            step(q, kn, vn, sl, out, bias=bias, k_cache=kc, v_cache=vc, scales=sc)
        torch.cuda.synchronize()
        outs.append(out.float().cpu().numpy())
        caches.append((kc.cpu().numpy(), sc.cpu().numpy()))
    assert step.get_error() == ftd.FTD_OK
    step.close()
    assert np.all(np.isfinite(outs[1]))
    assert np.max(np.abs(outs[0] - outs[1])) <= 1e-2
    assert np.array_equal(caches[0][0], caches[1][0])
    assert np.array_equal(caches[0][1].view(np.uint32), caches[1][1].view(np.uint32))  # NaN fill past the lengths


def test_noalloc_int8_grouped_runs_the_tensor_core_kernel():
    """A grouped INT8 cache (8 query rows per kv head) runs the same tensor-core kernel as the
    context path: identical output, appended codes and scales."""
    import torch
    w = Workload("noalloc", B=4, Hq=16, Hkv=2, D=128, Lmax=1024, qkv_dtype="f16", cache_dtype="i8", bias_std=0.1,
                 seed=25)
    inp = gen_all(w, seed=25, seq_lens=np.array([1000, 0, 129, 511], np.int32), fill_beyond="nan")
    step = ftd.DecodeStep(w.B, w.Hq, w.Hkv, w.D, w.Lmax, w.qkv_dtype, w.cache_dtype)
    cfg = ftd.FtdConfig(w.B, w.Hq, w.Hkv, w.D, w.Lmax, ftd.FTD_F16, ftd.FTD_I8, 0.0)
    s = torch.cuda.current_stream().cuda_stream
    q, kn, vn, bias, sl = (dev(inp[k]) for k in ("q", "k_new", "v_new", "bias", "seq_lens"))
    outs, caches = [], []
    for use_noalloc in (False, True):
        kc, vc, sc = dev(inp["k_cache"]), dev(inp["v_cache"]), dev(inp["scales"])
        out = torch.full((w.B, w.Hq, w.D), float("nan"), device="cuda")
        if use_noalloc:
            err = torch.zeros(1, dtype=torch.int32, device="cuda")
            st = ftd.ftd_decode_mha_noalloc(cfg, q.data_ptr(), kn.data_ptr(), vn.data_ptr(), bias.data_ptr(),
                                            kc.data_ptr(), vc.data_ptr(), sl.data_ptr(), sc.data_ptr(),
                                            out.data_ptr(), err.data_ptr(), s)
            assert st == ftd.FTD_OK, ftd.ftd_last_error()
        else:
            step(q, kn, vn, sl, out, bias=bias, k_cache=kc, v_cache=vc, scales=sc)
        torch.cuda.synchronize()
        outs.append(out.cpu().numpy())
        caches.append((kc.cpu().numpy(), vc.cpu().numpy(), sc.cpu().numpy()))
    assert step.get_error() == ftd.FTD_OK
    step.close()
    assert np.all(np.isfinite(outs[1]))
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    assert np.array_equal(caches[0][0], caches[1][0]) and np.array_equal(caches[0][1], caches[1][1])
    assert np.array_equal(caches[0][2].view(np.uint32), caches[1][2].view(np.uint32))


@pytest.mark.parametrize("cache", ["bf16", "i8"])
def test_noalloc_matches_the_oracle_with_and_without_an_error_word(cache):
    """Against the float64 oracle (not only against ftd_decode_mha), two calls in a row: the first
    with an error word, the second with device_err NULL (its overflow bit is dropped, the
    overflowing slot still gets a zero output and an untouched cache)."""
    import oracle
    import torch
    from tests.gpu_util import TOL_MAXABS_I8, assert_same_bytes
    qkv = "f16" if cache == "i8" else "bf16"
    w = Workload("noalloc", B=5, Hq=16, Hkv=2, D=128, Lmax=1024, qkv_dtype=qkv, cache_dtype=cache,
                 bias_std=0.1, scale_range=(0.01, 0.05), seed=26)
    inp = gen_all(w, seed=26, seq_lens=np.array([1000, 1024, 3, 511, -1], np.int32), fill_beyond="nan")
    ref = oracle.load().decode_step(w, inp, nthreads=8)
    dt = ftd.DTYPES
    cfg = ftd.FtdConfig(w.B, w.Hq, w.Hkv, w.D, w.Lmax, dt[qkv], dt[cache], 0.0)
    s = torch.cuda.current_stream().cuda_stream
    q, kn, vn, bias, sl = (dev(inp[k]) for k in ("q", "k_new", "v_new", "bias", "seq_lens"))
    for call, with_err in enumerate((True, False)):
        kc, vc = dev(inp["k_cache"]), dev(inp["v_cache"])
        sc = dev(inp["scales"]) if cache == "i8" else None
        out = torch.full((w.B, w.Hq, w.D), float("nan"), device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        st = ftd.ftd_decode_mha_noalloc(cfg, q.data_ptr(), kn.data_ptr(), vn.data_ptr(), bias.data_ptr(),
                                        kc.data_ptr(), vc.data_ptr(), sl.data_ptr(),
                                        0 if sc is None else sc.data_ptr(), out.data_ptr(),
                                        err.data_ptr() if with_err else 0, s)
        assert st == ftd.FTD_OK, ftd.ftd_last_error()
        torch.cuda.synchronize()
        assert int(err.item()) == (1 if with_err else 0), f"call {call}: error word"
        got = out.double().cpu().numpy()
        assert np.all(np.isfinite(got)), f"call {call}"
        d = np.max(np.abs(got - ref["out"]))
        if cache == "i8":
            assert d <= TOL_MAXABS_I8, f"call {call}: max-abs {d:.3e}"
        else:
            assert d <= TOL_MAXABS, f"call {call}: max-abs {d:.3e}"
            assert np.linalg.norm(got - ref["out"]) / np.linalg.norm(ref["out"]) <= TOL_RELL2, f"call {call}"
        assert not got[1].any() and not got[4].any(), f"call {call}: overflowing / inactive slots"
        kh = kc.cpu().numpy()
        assert_same_bytes(kh.view(ref["k_cache"].dtype), ref["k_cache"], f"call {call}: K cache")
        if cache == "i8":
            assert_same_bytes(sc.cpu().numpy(), ref["scales"], f"call {call}: scales")
