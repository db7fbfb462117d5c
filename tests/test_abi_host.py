"""The C ABI on the host: the library loads, exports what include/ftd.h declares,
and rejects bad arguments synchronously without touching a GPU."""
import ctypes
import os
import re

import pytest

import decode_step_masked_gb300 as ftd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    ftd.build_library()
    return ftd.load_library()


def declared_functions():
    with open(os.path.join(ROOT, "include", "ftd.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ftd_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 9, names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ftd.h but not exported"
    assert set(names) == set(ftd.EXPORTS)


def test_status_strings(lib):
    for code, name in [(0, "FTD_OK"), (1, "FTD_ERR_INVALID_ARG"), (2, "FTD_ERR_UNSUPPORTED"),
                       (3, "FTD_ERR_OOM"), (4, "FTD_ERR_CUDA"), (5, "FTD_ERR_SEQ_OVERFLOW"),
                       (6, "FTD_ERR_DEVICE_TIMEOUT"), (7, "FTD_ERR_BAD_PAGE")]:
        assert ftd.ftd_status_str(code) == name
    assert ftd.ftd_status_str(99) == "FTD_ERR_UNKNOWN"


def cfg(**kw):
    base = dict(max_batch=4, n_q_heads=8, n_kv_heads=2, head_dim=128, max_len=256,
                qkv_dtype=ftd.FTD_BF16, cache_dtype=ftd.FTD_BF16, softmax_scale=0.0,
                out_dtype=ftd.FTD_F32, window=0, page_size=0, num_pages=0, q_len=0, kernel=0, proj_dim=0,
                wait_limit_us=0)
    base.update(kw)
    return ftd.FtdConfig(*[base[f] for f, _ in ftd.FtdConfig._fields_])


@pytest.mark.parametrize("kw,status", [
    (dict(max_batch=0), ftd.FTD_ERR_INVALID_ARG),
    (dict(max_batch=1025), ftd.FTD_ERR_INVALID_ARG),
    (dict(n_kv_heads=0), ftd.FTD_ERR_INVALID_ARG),
    (dict(n_q_heads=6, n_kv_heads=4), ftd.FTD_ERR_INVALID_ARG),
    (dict(n_q_heads=2, n_kv_heads=4), ftd.FTD_ERR_INVALID_ARG),
    (dict(max_len=0), ftd.FTD_ERR_INVALID_ARG),
    (dict(max_len=100), ftd.FTD_ERR_INVALID_ARG),
    (dict(head_dim=0), ftd.FTD_ERR_INVALID_ARG),
    (dict(head_dim=96), ftd.FTD_ERR_UNSUPPORTED),
    (dict(qkv_dtype=ftd.FTD_I8), ftd.FTD_ERR_UNSUPPORTED),
    (dict(cache_dtype=7), ftd.FTD_ERR_UNSUPPORTED),
    (dict(softmax_scale=-1.0), ftd.FTD_ERR_INVALID_ARG),
    (dict(softmax_scale=float("nan")), ftd.FTD_ERR_INVALID_ARG),
    (dict(softmax_scale=float("inf")), ftd.FTD_ERR_INVALID_ARG),
    (dict(out_dtype=ftd.FTD_I8), ftd.FTD_ERR_UNSUPPORTED),
    (dict(out_dtype=9), ftd.FTD_ERR_UNSUPPORTED),
    (dict(window=-1), ftd.FTD_ERR_INVALID_ARG),
    (dict(page_size=64, num_pages=8), ftd.FTD_ERR_INVALID_ARG),
    (dict(page_size=-128, num_pages=8), ftd.FTD_ERR_INVALID_ARG),
    (dict(page_size=128, num_pages=0), ftd.FTD_ERR_INVALID_ARG),
    (dict(page_size=384, num_pages=8), ftd.FTD_ERR_INVALID_ARG),
    (dict(q_len=-1), ftd.FTD_ERR_INVALID_ARG),
    (dict(q_len=65), ftd.FTD_ERR_INVALID_ARG),
    (dict(kernel=2), ftd.FTD_ERR_INVALID_ARG),
    (dict(kernel=-1), ftd.FTD_ERR_INVALID_ARG),
    (dict(wait_limit_us=-5), ftd.FTD_ERR_INVALID_ARG),
    (dict(proj_dim=-128), ftd.FTD_ERR_INVALID_ARG),
    (dict(proj_dim=100), ftd.FTD_ERR_INVALID_ARG),
    (dict(proj_dim=128, qkv_dtype=ftd.FTD_F32), ftd.FTD_ERR_UNSUPPORTED),
    # rows fit 32 bits (1024 x 1 x 2^20) but the tile space of 4096 query rows per kv head does not
    (dict(max_batch=1024, n_q_heads=64, n_kv_heads=1, max_len=1 << 20, q_len=64), ftd.FTD_ERR_UNSUPPORTED),
])
def test_init_rejects_bad_config(lib, kw, status):
    st, ctx = ftd.ftd_init(cfg(**kw))
    assert st == status, (ftd.ftd_status_str(st), ftd.ftd_last_error())
    assert ctx is None
    assert ftd.ftd_last_error() != ""


def test_null_arguments(lib):
    assert lib.ftd_init(None, None, None) == ftd.FTD_ERR_INVALID_ARG
    out = ctypes.c_void_p(1234)
    assert lib.ftd_init(None, None, ctypes.byref(out)) == ftd.FTD_ERR_INVALID_ARG
    assert out.value is None, "ftd_init must clear *out on failure"
    assert ftd.ftd_decode_mha(0, 16, 16, 16, 0, 16, 16, 16, 0, 16, 0) == ftd.FTD_ERR_INVALID_ARG
    assert ftd.ftd_decode_mha_host(0, 16, 16, 16, 0, 16, 16, 16, 0, 16, 0) == ftd.FTD_ERR_INVALID_ARG
    assert ftd.ftd_decode_mha_paged(0, 16, 16, 16, 0, 16, 16, 16, 16, 0, 16, 0) == ftd.FTD_ERR_INVALID_ARG
    assert ftd.ftd_decode_mha_proj(0, 16, 16, 16, 0, 16, 16, 16, 0, 16, 16, 16, 0) == ftd.FTD_ERR_INVALID_ARG
    assert ftd.ftd_get_error(0) == ftd.FTD_ERR_INVALID_ARG
    assert ftd.ftd_cache_ptrs(0)[0] == ftd.FTD_ERR_INVALID_ARG
    assert ftd.ftd_debug_stall_next(0, 1) == ftd.FTD_ERR_INVALID_ARG
    ftd.ftd_destroy(0)  # no-op
    # without a live context the handle-free entry point refuses (no context exists on a CPU host)
    assert ftd.ftd_decode_mha_current(16, 16, 16, 0, 16, 16, 16, 0, 16, 0) == ftd.FTD_ERR_INVALID_ARG
    assert "no context" in ftd.ftd_last_error()


def test_no_launches_from_host_failures(lib):
    n = ftd.ftd_kernel_launches()
    ftd.ftd_init(cfg(max_batch=0))
    ftd.ftd_decode_mha(0, 16, 16, 16, 0, 16, 16, 16, 0, 16, 0)
    assert ftd.ftd_kernel_launches() == n


def test_config_struct_matches_header():
    """The ctypes mirror lists ftd_config's fields in the header's order."""
    with open(os.path.join(ROOT, "include", "ftd.h")) as f:
        text = f.read()
    body = re.search(r"typedef struct \{(.*?)\} ftd_config;", text, re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    names = re.findall(r"\b([a-z_]+)\s*;", body)
    assert names == [f for f, _ in ftd.FtdConfig._fields_]


def test_noalloc_rejects_paged_and_bad_options(lib):
    for kw in (dict(page_size=128, num_pages=4), dict(window=-3), dict(out_dtype=ftd.FTD_I8), dict(q_len=99)):
        st = ftd.ftd_decode_mha_noalloc(cfg(**kw), 16, 16, 16, 0, 16, 16, 16, 0, 16, 0, 0)
        assert st in (ftd.FTD_ERR_INVALID_ARG, ftd.FTD_ERR_UNSUPPORTED), kw
        assert ftd.ftd_last_error() != ""


def test_noalloc_applies_the_context_paths_checks(lib):
    """The no-allocation entry point makes ftd_init's and ftd_decode_mha's checks: the 32-bit
    tile-space bound and the natural alignment of every pointer, before any device work."""
    huge = cfg(max_batch=1024, n_q_heads=64, n_kv_heads=1, max_len=1 << 20, q_len=64)
    assert ftd.ftd_decode_mha_noalloc(huge, 16, 16, 16, 0, 16, 16, 16, 0, 16, 0, 0) == ftd.FTD_ERR_UNSUPPORTED
    assert "tile indices" in ftd.ftd_last_error()
    ok = dict(q=16, k_new=16, v_new=16, bias=0, k_cache=256, v_cache=512, seq_lens=16, scales=0, out=1024)
    for name, bad in (("q", 17), ("k_new", 33), ("v_new", 49), ("bias", 3), ("seq_lens", 18), ("k_cache", 264),
                      ("v_cache", 520), ("out", 1032)):
        a = dict(ok, **{name: bad})
        st = ftd.ftd_decode_mha_noalloc(cfg(), a["q"], a["k_new"], a["v_new"], a["bias"], a["k_cache"],
                                        a["v_cache"], a["seq_lens"], a["scales"], a["out"], 0, 0)
        assert st == ftd.FTD_ERR_INVALID_ARG, name
        assert "aligned" in ftd.ftd_last_error(), name
    i8 = cfg(cache_dtype=ftd.FTD_I8, qkv_dtype=ftd.FTD_F16)
    st = ftd.ftd_decode_mha_noalloc(i8, 16, 16, 16, 0, 256, 512, 16, 0, 1024, 0, 0)
    assert st == ftd.FTD_ERR_INVALID_ARG and "scales" in ftd.ftd_last_error()
    st = ftd.ftd_decode_mha_noalloc(i8, 16, 16, 16, 0, 256, 512, 16, 8, 1024, 0, 0)
    assert st == ftd.FTD_ERR_INVALID_ARG and "aligned" in ftd.ftd_last_error()


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(FileNotFoundError, match="no fallback"):
        ftd.load_library(str(tmp_path / "libftd.so"))
