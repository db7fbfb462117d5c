"""Host-side logic of bench.py: algorithmic byte counts, and the multi-rank
reduction (max of the timed region, sum of the units) on 2 gloo ranks."""
import os
import socket

import numpy as np
import pytest

import bench
from synthetic import WORKLOADS, gen_seq_lens


def test_step_bytes_7b_matches_hand_count():
    w = WORKLOADS["7b"]
    by = bench.step_bytes(w, gen_seq_lens(w))
    # 2 (K and V) x 8 slots x 32 heads x 2048 rows x 128 x 2 bytes: 2047 cached rows read, 1 appended
    assert by["kv"] == 2 * 8 * 32 * 2048 * 128 * 2 == 268435456
    assert by["ctx"] == 8 * 2048
    small = (8 * 32 * 128 + 2 * 8 * 32 * 128) * 2 + 4 * 8 + 4 * 8 * 32 * 128
    assert by["total"] == by["kv"] + small


def test_step_bytes_int8_counts_scales_and_skips_inactive():
    w = WORKLOADS["int8"].with_(B=3)
    lens = np.array([10, -1, w.Lmax], np.int32)  # one active, one inactive, one overflowing
    by = bench.step_bytes(w, lens)
    assert by["ctx"] == 11
    assert by["kv"] == 2 * w.Hkv * w.D * 1 * 11 + 8 * w.Hkv * 11


def test_gqa_counts_kv_once_per_kv_head():
    w = WORKLOADS["70b"]
    by = bench.step_bytes(w, gen_seq_lens(w))
    assert by["kv"] == 2 * 16 * 8 * 8192 * 128 * 2  # 537 MB: K/V read once per kv head, not per q head


def test_step_bytes_window_counts_visible_rows_only():
    w = WORKLOADS["7b"].with_(B=3)
    lens = np.array([10, 2047, -1], np.int32)  # short slot, long slot, inactive
    by = bench.step_bytes(w, lens, window=100)
    assert by["ctx"] == 11 + 100
    assert by["kv"] == 2 * w.Hkv * w.D * 2 * (11 + 100)  # reads of visible history + the appended rows
    assert bench.step_bytes(w, lens, window=0)["ctx"] == 11 + 2048


def test_step_bytes_half_output():
    w = WORKLOADS["70b"]
    lens = gen_seq_lens(w)
    assert (bench.step_bytes(w, lens)["total"] - bench.step_bytes(w, lens, out_dtype="bf16")["total"]
            == 2 * w.B * w.Hq * w.D)


def test_step_bytes_several_new_tokens():
    w = WORKLOADS["7b"].with_(B=2)
    lens = np.array([100, 4093], np.int32)  # 4093 + 4 > Lmax 4096: overflow, no work
    by = bench.step_bytes(w, lens, q_len=4)
    assert by["ctx"] == 104
    assert by["kv"] == 2 * w.Hkv * w.D * 2 * 104  # 100 history rows read + 4 rows appended
    by_w = bench.step_bytes(w, lens, window=10, q_len=4)
    assert by_w["ctx"] == 13  # rows some token sees: positions 91 .. 103
    assert bench.kernel_name(w, 8) == "decode_gqa_tc_kernel" and bench.kernel_name(w, 4) == "decode_gqa_tc_kernel"
    assert bench.kernel_name(w, 2) == "decode_splitk_kernel"
    i8 = WORKLOADS["int8"]  # INT8: the tensor-core variant takes blocks of 8 query rows
    assert bench.kernel_name(i8) == "decode_splitk_kernel" and bench.kernel_name(i8, 4) == "decode_splitk_kernel"
    assert bench.kernel_name(i8, 8) == "decode_gqa_tc_kernel"
    assert bench.kernel_name(i8.with_(Hq=64, Hkv=8)) == "decode_gqa_tc_kernel"


def test_page_table_is_a_permutation():
    w = WORKLOADS["13b"]
    table, n = bench.page_table(w, 256, 3)
    assert table.shape == (w.B, w.Lmax // 256) and n == w.B * w.Lmax // 256
    assert sorted(table.reshape(-1).tolist()) == list(range(n))


def test_pool_rotation_exceeds_l2():
    for name in ("7b", "13b", "70b", "int8"):
        w = WORKLOADS[name]
        kv = bench.step_bytes(w, gen_seq_lens(w))["kv"]
        n = bench.n_pools_for(w, kv)
        assert (n - 1) * kv > 2 * 129e6, name  # traffic between two reads of one pool


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [12.5, 20.0][rank]
        local_units = [1e9, 3e9][rank]
        q.put((rank, bench.reduce_over_ranks(local_ms, local_units, world)))
    finally:
        dist.destroy_process_group()


def test_reduce_over_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        t, u = res[r]
        assert t == pytest.approx(20.0) and u == pytest.approx(4e9)  # slowest rank, all units


def test_reduce_single_rank_is_identity():
    assert bench.reduce_over_ranks(3.0, 7.0, 1) == (3.0, 7.0)


def test_cpu_baseline_helpers():
    """The CPU baseline records the host CPU's model and times the brute force on the tiny step."""
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()
    assert bench.brute_tiny_ms() > 0.0
