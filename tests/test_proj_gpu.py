"""The output projection (ftd_decode_mha_proj) against the float64 oracle.

One call runs the decode step and then y = out . W_o^T on the tensor cores.  The
checks, on the same seeded inputs:
  * out and the appended cache rows as in ftd_decode_mha (the decode parity bars);
  * y against the oracle's projection of the oracle's own output (the whole chain),
    within the decode bars (max-abs 2e-3, rel-L2 1e-3; INT8 caches max-abs 1e-2);
  * y against the oracle's projection of the GPU's out as stored: the projection
    alone, whose hi / lo operand split keeps about 16 mantissa bits
    (rel-L2 3e-5 for an fp32 y; half an output ulp more for a half-precision y);
  * rows of inactive and overflowing slots are zero.
"""
import numpy as np
import pytest

import decode_step_masked_gb300 as ftd
import oracle
from synthetic import Workload, gen_all, to_storage
from tests.gpu_util import TOL_MAXABS, TOL_MAXABS_I8, TOL_RELL2, TORCH_OUT, assert_close, assert_same_bytes, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    ftd.build_library()
    ftd.load_library()


def weight(F, K, dt, seed):
    """W_o ~ N(0, 1/K) stored in dt, and its float64 values."""
    w = np.random.default_rng([seed, 99]).standard_normal((F, K)).astype(np.float32) / np.float32(np.sqrt(K))
    st = to_storage(w, dt)
    vals = (st.astype(np.uint32) << 16).view(np.float32) if dt == "bf16" else st.astype(np.float32)
    return st, vals.astype(np.float64)


def run_proj(w, inp, F, out_dtype="f32", force_cuda_core=False, seed=0, calls=1):
    import torch
    T = getattr(w, "q_len", 1)
    Wst, Wf = weight(F, w.Hq * w.D, w.qkv_dtype, seed)
    kernel = ftd.FTD_KERNEL_CUDA_CORE if force_cuda_core else ftd.FTD_KERNEL_AUTO
    step = ftd.DecodeStep(w.B, w.Hq, w.Hkv, w.D, w.Lmax, w.qkv_dtype, w.cache_dtype, out_dtype=out_dtype,
                          q_len=T, kernel=kernel, proj_dim=F)
    tdt = getattr(torch, TORCH_OUT[out_dtype])
    lead = (w.B, T) if T > 1 else (w.B,)
    q, kn, vn = dev(inp["q"]), dev(inp["k_new"]), dev(inp["v_new"])
    bias = dev(inp["bias"]) if inp.get("bias") is not None else None
    sl = dev(inp["seq_lens"])
    wd = dev(Wst)
    for _ in range(calls):  # the same step again: the counters and planes are reused
        kc, vc = dev(inp["k_cache"]), dev(inp["v_cache"])
        sc = dev(inp["scales"]) if inp.get("scales") is not None else None
        out = torch.full(lead + (w.Hq, w.D), float("nan"), dtype=tdt, device="cuda")
        y = torch.full(lead + (F,), float("nan"), dtype=tdt, device="cuda")
        step.proj(q, kn, vn, sl, out, wd, y, bias=bias, k_cache=kc, v_cache=vc, scales=sc)
        torch.cuda.synchronize()
    status = step.get_error()
    step.close()
    return dict(out=out.double().cpu().numpy(), y=y.double().cpu().numpy(), k_cache=kc.cpu().numpy(),
                status=status, W=Wf)


def check(w, inp, F, out_dtype="f32", force_cuda_core=False, what="", calls=1):
    o = oracle.load()
    ref = o.decode_step(w, inp, nthreads=8)
    got = run_proj(w, inp, F, out_dtype, force_cuda_core, seed=w.seed, calls=calls)
    want = ftd.FTD_ERR_SEQ_OVERFLOW if ref["overflow"] else ftd.FTD_OK
    assert got["status"] == want, (ftd.ftd_status_str(got["status"]), what)
    i8 = w.cache_dtype == "i8"
    assert_same_bytes(got["k_cache"].view(ref["k_cache"].dtype), ref["k_cache"], f"{what}: K cache")
    if out_dtype == "f32":
        assert_close(got["out"], ref["out"], i8=i8, what=f"{what}: out")
    T = getattr(w, "q_len", 1)
    F_ = got["W"].shape[0]
    y = got["y"].reshape(-1, F_)
    # the whole chain: the oracle's projection of the oracle's output
    y_ref = o.out_proj(ref["out"], got["W"])
    assert np.all(np.isfinite(y)), f"{what}: non-finite y"
    half = out_dtype != "f32"
    if i8:
        assert np.max(np.abs(y - y_ref)) <= TOL_MAXABS_I8, f"{what}: y vs oracle"
    else:
        err = np.max(np.abs(y - y_ref))
        rel = np.linalg.norm(y - y_ref) / max(np.linalg.norm(y_ref), 1e-30)
        ulp = np.max(np.abs(y_ref)) * (2.0 ** -8 if out_dtype == "bf16" else 2.0 ** -11) if half else 0.0
        assert err <= TOL_MAXABS + ulp, f"{what}: y max-abs {err:.3e}"
        assert rel <= TOL_RELL2 + (4e-3 if half else 0.0), f"{what}: y rel-L2 {rel:.3e}"
    # the projection alone: the oracle's projection of the output the GPU stored
    y_own = o.out_proj(got["out"], got["W"])
    rel = np.linalg.norm(y - y_own) / max(np.linalg.norm(y_own), 1e-30)
    if half:
        bound = np.abs(y_own) * (2.0 ** -8 if out_dtype == "bf16" else 2.0 ** -11) + 1e-4 * np.max(np.abs(y_own))
        assert np.all(np.abs(y - y_own) <= bound), f"{what}: y vs projection of the stored out"
    else:
        assert rel <= 3e-5, f"{what}: y vs projection of the stored out, rel-L2 {rel:.3e}"
    # inactive and overflowing slots give zero rows
    lens = np.asarray(inp["seq_lens"])
    dead = (lens < 0) | (lens > w.Lmax - T)
    yb = got["y"].reshape(w.B, -1)
    assert not yb[dead].any(), f"{what}: rows of inactive slots"
    return y, y_ref


def case(cache, qkv, B, Hq, Hkv, D, Lmax, lens, seed, q_len=1):
    w = Workload("proj", B=B, Hq=Hq, Hkv=Hkv, D=D, Lmax=Lmax, qkv_dtype=qkv, cache_dtype=cache, bias_std=0.1,
                 scale_range=(0.01, 0.05), seed=seed, q_len=q_len)
    return w, gen_all(w, seed=seed, seq_lens=np.array(lens, np.int32), fill_beyond="nan")


@pytest.mark.parametrize("cache,qkv,Hq,Hkv,D,F,cc", [
    ("bf16", "bf16", 16, 2, 128, 256, False),   # tensor-core decode, K = 2048
    ("bf16", "bf16", 16, 2, 128, 384, True),    # the same on the CUDA-core kernel, 3 feature tiles
    ("f16", "f16", 4, 4, 64, 128, False),       # multi-head, head_dim 64, K = 256, one tile
    ("i8", "f16", 16, 2, 128, 256, False),      # INT8 cache on the tensor cores
    ("i8", "f16", 8, 8, 128, 640, False),       # INT8 multi-head (dp4a), 5 tiles
])
def test_projection(cache, qkv, Hq, Hkv, D, F, cc):
    w, inp = case(cache, qkv, B=5, Hq=Hq, Hkv=Hkv, D=D, Lmax=1024, lens=[1000, 0, -1, 517, 1024], seed=61)
    check(w, inp, F, force_cuda_core=cc, what=f"{cache}/{Hq}/{Hkv}/D{D}/F{F}")


@pytest.mark.parametrize("out_dtype", ["bf16", "f16"])
def test_projection_half_output(out_dtype):
    qkv = "bf16" if out_dtype == "bf16" else "f16"
    w, inp = case(qkv, qkv, B=6, Hq=16, Hkv=2, D=128, Lmax=512, lens=[511, 3, 200, 0, 128, 300], seed=62)
    check(w, inp, 256, out_dtype=out_dtype, what=f"half out {out_dtype}")


def test_projection_several_tokens_per_step():
    w, inp = case("bf16", "bf16", B=3, Hq=8, Hkv=2, D=128, Lmax=512, lens=[100, 0, 508], seed=63, q_len=4)
    check(w, inp, 256, what="q_len 4")


def test_projection_many_tokens_two_blocks_and_repeat():
    """150 tokens: two token blocks of the projection kernel (128 + 22), and two calls in a row
    on one context (the arrival counters return to zero after every tile)."""
    lens = [(37 * i) % 60 for i in range(150)]
    lens[7] = -1
    w, inp = case("bf16", "bf16", B=150, Hq=2, Hkv=2, D=64, Lmax=64, lens=lens, seed=64)
    check(w, inp, 256, what="150 tokens", calls=2)


def test_projection_large_feature_count():
    """A 70B-like projection shape on a small batch: K = 64 x 128 = 8192 and F = 1024 (8 tiles x
    128 chunks of K over the 152 CTAs: every tile merges pieces of several CTAs)."""
    w, inp = case("bf16", "bf16", B=4, Hq=64, Hkv=8, D=128, Lmax=256, lens=[255, 100, 3, 200], seed=65)
    check(w, inp, 1024, what="K 8192")


def test_projection_refused_without_proj_dim():
    import torch
    w, inp = case("bf16", "bf16", B=2, Hq=4, Hkv=4, D=64, Lmax=64, lens=[3, 4], seed=66)
    step = ftd.DecodeStep(w.B, w.Hq, w.Hkv, w.D, w.Lmax, w.qkv_dtype, w.cache_dtype)
    x = torch.zeros(4096, device="cuda")
    st = ftd.ftd_decode_mha_proj(step.ctx, x.data_ptr(), x.data_ptr(), x.data_ptr(), 0, 0, 0, x.data_ptr(), 0,
                                 x.data_ptr(), x.data_ptr(), x.data_ptr(), 0)
    assert st == ftd.FTD_ERR_INVALID_ARG and "proj_dim" in ftd.ftd_last_error()
    step.close()
