"""Failure handling and ordering on the GPU, without faulting or hanging it.

- A kernel of the caller that writes seq_lens right before the step (the step is
  launched to start early, while its predecessor drains): the step must use the
  written lengths, since they are read again after the wait on the predecessor.
- The bounded-wait error path: ftd_debug_stall_next makes block 0 withhold one
  tile copy, so its waits run out after the context's short wait limit; the call
  then reports FTD_ERR_DEVICE_TIMEOUT, and the next call on the same context
  matches the oracle (ftd_get_error reset the split-K counters).  Every wait is
  bounded and the copies in flight are drained before a block exits.
"""
import numpy as np
import pytest

import decode_step_masked_gb300 as ftd
import oracle
from synthetic import Workload, gen_all
from tests.gpu_util import assert_close, assert_same_bytes, dev, make_step, run_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    ftd.build_library()
    ftd.load_library()


# name: (cache, qkv, Hq, Hkv, force the CUDA-core kernel)
CASES = {"tc_bf16": ("bf16", "bf16", 16, 2, False), "splitk_bf16": ("bf16", "bf16", 16, 2, True),
         "splitk_mha_f16": ("f16", "f16", 4, 4, False), "tc_i8": ("i8", "f16", 16, 2, False),
         "splitk_i8": ("i8", "f16", 4, 4, False), "tc_wide_mqa": ("bf16", "bf16", 64, 1, False),
         "tc_wide_32": ("f16", "f16", 32, 1, False)}


def case(name, lens, seed):
    cache, qkv, Hq, Hkv, cc = CASES[name]
    w = Workload("fail", B=len(lens), Hq=Hq, Hkv=Hkv, D=128, Lmax=2048, qkv_dtype=qkv, cache_dtype=cache,
                 bias_std=0.1, seed=seed)
    return w, gen_all(w, seed=seed, seq_lens=np.array(lens, np.int32), fill_beyond="nan"), cc


@pytest.mark.parametrize("name", sorted(CASES))
def test_lengths_written_right_before_the_step(name):
    """seq_lens - 1 is on the device; a torch kernel adds 1 on the step's stream just before
    the step.  Result, appended rows and error status follow the new lengths."""
    import torch
    lens = np.array([1500, 0, 2047, 333, 128, -1], np.int32)
    w, inp, cc = case(name, lens, seed=51)
    ref = oracle.load().decode_step(w, inp, nthreads=8)
    step = make_step(w, force_cuda_core=cc)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        q, kn, vn, bias = (dev(inp[k]) for k in ("q", "k_new", "v_new", "bias"))
        kc, vc = dev(inp["k_cache"]), dev(inp["v_cache"])
        sc = dev(inp["scales"]) if inp["scales"] is not None else None
        delta = (lens >= 0).astype(np.int32)
        stale = dev((lens - delta).astype(np.int32))  # one token short (slot 1 then looks inactive)
        d = dev(delta)
        sl = stale.clone()
        out = torch.full((w.B, w.Hq, w.D), float("nan"), device="cuda")
        torch.cuda.synchronize()
        for _ in range(3):  # the step follows the add kernel directly, three times in a row
            sl.copy_(stale)
            sl.add_(d)
            step(q, kn, vn, sl, out, bias=bias, k_cache=kc, v_cache=vc, scales=sc, stream=stream.cuda_stream)
    torch.cuda.synchronize()
    assert step.get_error() == ftd.FTD_OK
    step.close()
    assert_close(out.double().cpu().numpy(), ref["out"], i8=w.cache_dtype == "i8", what=name)
    kh = kc.cpu().numpy()
    assert_same_bytes(kh.view(ref["k_cache"].dtype), ref["k_cache"], f"{name}: K cache")


@pytest.mark.parametrize("name", sorted(CASES))
def test_lengths_written_after_the_step_read_them(name):
    """The preceding kernel (ftd_debug_late_lengths) lets the step start at once and writes
    seq_lens only ~50 us later: the step plans from the stale lengths, finds after its wait
    that they changed, and re-plans.  Result, appended rows and status follow the new lengths."""
    import torch
    lens = np.array([1500, 0, 2047, 333, 128, -1], np.int32)
    w, inp, cc = case(name, lens, seed=53)
    ref = oracle.load().decode_step(w, inp, nthreads=8)
    step = make_step(w, force_cuda_core=cc)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        q, kn, vn, bias = (dev(inp[k]) for k in ("q", "k_new", "v_new", "bias"))
        kc, vc = dev(inp["k_cache"]), dev(inp["v_cache"])
        sc = dev(inp["scales"]) if inp["scales"] is not None else None
        stale = dev(np.array([700, -1, 5, 333, 2047, 9], np.int32))  # every slot but one differs
        new = dev(lens)
        sl = stale.clone()
        out = torch.full((w.B, w.Hq, w.D), float("nan"), device="cuda")
        torch.cuda.synchronize()
        for _ in range(3):
            sl.copy_(stale)
            assert ftd.ftd_debug_late_lengths(new.data_ptr(), sl.data_ptr(), w.B, 50, stream.cuda_stream) == 0
            step(q, kn, vn, sl, out, bias=bias, k_cache=kc, v_cache=vc, scales=sc, stream=stream.cuda_stream)
    torch.cuda.synchronize()
    assert step.get_error() == ftd.FTD_OK
    step.close()
    assert_close(out.double().cpu().numpy(), ref["out"], i8=w.cache_dtype == "i8", what=name)
    assert_same_bytes(kc.cpu().numpy().view(ref["k_cache"].dtype), ref["k_cache"], f"{name}: K cache")
    assert_same_bytes(vc.cpu().numpy().view(ref["v_cache"].dtype), ref["v_cache"], f"{name}: V cache")


@pytest.mark.parametrize("name", sorted(CASES))
def test_timeout_path_reports_and_recovers(name):
    lens = [1800, 40, 1000, 2047]
    w, inp, cc = case(name, lens, seed=52)
    step = make_step(w, force_cuda_core=cc, wait_limit_us=2000)
    assert ftd.ftd_debug_stall_next(step.ctx, 1) == ftd.FTD_OK
    got = run_step(w, inp, step=step)
    assert got["status"] == ftd.FTD_ERR_DEVICE_TIMEOUT, ftd.ftd_status_str(got["status"])
    # the same context, the next call: correct again
    ref = oracle.load().decode_step(w, inp, nthreads=8)
    for _ in range(2):
        got = run_step(w, inp, step=step)
        assert got["status"] == ftd.FTD_OK, ftd.ftd_status_str(got["status"])
        assert_close(got["out"], ref["out"], i8=w.cache_dtype == "i8", what=f"{name} after a timeout")
        assert_same_bytes(got["k_cache"], ref["k_cache"], f"{name}: K cache after a timeout")
    step.close()
