"""INT8 caches with large-magnitude queries and large scores, on both INT8 paths.

The CUDA-core INT8 path splits the scaled query into two int8 levels for its dp4a
scores (about 1.5e-5 of max|q| per element), and its P.V weights into three; the
tensor-core INT8 path splits q and the weights into fp16 hi / lo halves.  Both
errors grow with the magnitude of q and of the scores, so these cases drive q to
8, 32 and 128 times N(0, 1) and let scores climb along the context, and hold every
output to the INT8 bar (max-abs 1e-2 against the oracle on the dequantised cache).
The measured error of each case is printed (pytest -s).
"""
import numpy as np
import pytest

import decode_step_masked_gb300 as ftd
import oracle
from synthetic import Workload, gen_all
from tests.gpu_util import TOL_MAXABS_I8, assert_same_bytes, rising_scores_i8, run_step, scale_q

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    ftd.build_library()
    ftd.load_library()


# (query heads, kv heads): 1 and 2 query rows per kv head run the dp4a CUDA-core path,
# 8 rows the tensor-core INT8 variant
PATHS = {"dp4a_g1": (4, 4), "dp4a_g2": (8, 4), "tc_g8": (16, 2)}


def case(path, seed):
    Hq, Hkv = PATHS[path]
    w = Workload("i8prec", B=4, Hq=Hq, Hkv=Hkv, D=128, Lmax=2048, qkv_dtype="f16", cache_dtype="i8",
                 bias_std=0.1, scale_range=(0.01, 0.05), seed=seed)
    return w, gen_all(w, seed=seed, seq_lens=np.array([2047, 700, 129, 1500], np.int32), fill_beyond="nan")


def check(w, inp, what):
    ref = oracle.load().decode_step(w, inp, nthreads=8)
    got = run_step(w, inp)
    assert got["status"] == ftd.FTD_OK, what
    assert_same_bytes(got["k_cache"], ref["k_cache"], f"{what}: K codes after append")
    assert_same_bytes(got["scales"], ref["scales"], f"{what}: scales after append")
    assert np.all(np.isfinite(got["out"])), f"{what}: non-finite output"
    err = float(np.max(np.abs(got["out"] - ref["out"])))
    print(f"{what}: max-abs {err:.3e} (bar {TOL_MAXABS_I8:.0e})")
    assert err <= TOL_MAXABS_I8, f"{what}: max-abs {err:.3e} > {TOL_MAXABS_I8}"
    return err


@pytest.mark.parametrize("factor", [1, 8, 32, 128])
@pytest.mark.parametrize("path", sorted(PATHS))
def test_large_queries(path, factor):
    w, inp = case(path, seed=41)
    check(w, scale_q(w, inp, factor), f"{path} q x{factor}")


@pytest.mark.parametrize("rise", [20.0, 60.0])
@pytest.mark.parametrize("path", sorted(PATHS))
def test_rising_scores(path, rise):
    """Scores climbing by `rise` base-2 units along the context move every query row's running
    maximum many times; the top scores are large and close together."""
    w, inp = case(path, seed=42)
    check(w, rising_scores_i8(w, inp, rise_log2=rise), f"{path} rising {rise:g}")
