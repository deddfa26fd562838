"""Host logic of bench.py (CPU only): the byte model against the numbers the
pages print, the L2-defeating layer counts, and the multi-rank aggregation
run as two gloo ranks."""
import json
import os
import pathlib
import socket

import pytest
import torch.multiprocessing as mp

import bench

GOLD = json.loads((pathlib.Path(__file__).parent / "golden" / "s2pro_byte_model.json").read_text())


def test_expanded_full_capacity_bytes_match_the_page():
    g = GOLD
    per_layer = bench.expanded_full_capacity_bytes(g["n_head"], g["max_seq_len"], g["head_dim"],
                                                   g["bytes_per_element_fp16"])
    assert per_layer == g["expanded_kv_bytes_per_layer"] == 512 * 2**20
    assert per_layer * g["layers"] == g["expanded_kv_bytes_36_layers"] == 18 * 2**30


def test_active_prefix_bytes_read_kv_heads_once():
    g = GOLD
    # the slice reads only kv_len rows of the 8 KV heads (no expansion): 1/4 of
    # the expanded heads, kv_len/capacity of the rows
    kv_len = 634
    active = bench.attend_bytes(1, g["n_head"], g["n_local_heads"], g["head_dim"], [kv_len], elem=2)
    kv_part = active - 2 * 2 * g["n_head"] * g["head_dim"]
    expanded = bench.expanded_full_capacity_bytes(g["n_head"], g["max_seq_len"], g["head_dim"], 2)
    assert kv_part * (g["n_head"] // g["n_local_heads"]) * g["max_seq_len"] == expanded * kv_len


def test_layers_defeat_l2():
    l2 = 126 * 2**20
    for kv in bench.SWEEP:
        n = bench.layers_for(kv, l2)
        assert n * 2 * bench.N_KV_HEAD * kv * bench.HEAD_DIM * bench.ELEM >= 3 * l2


def test_aggregate_value_is_whole_job():
    # 2 ranks x 1 GB per step x 10 steps in 10 ms (slowest rank) = 2000 GB/s
    assert bench.aggregate_value(10**9, 10, 2, 10.0) == pytest.approx(2000.0)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, results):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [12.0, 15.0][rank]
    m = bench.max_over_ranks(local_ms, world)
    bench.barrier(world)
    results[rank] = (m, bench.aggregate_value(10**9, 10, world, m))
    dist.destroy_process_group()


def test_two_rank_max_and_aggregate():
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        results = mgr.dict()
        mp.start_processes(_rank_main, args=(2, port, results), nprocs=2, join=True, start_method="spawn")
        r = dict(results)
    assert r[0][0] == r[1][0] == 15.0
    assert r[0][1] == pytest.approx(2 * 10**9 * 10 / 0.015 / 1e9)


def test_kernel_hash_ignores_comments_only():
    """The ncu figures under profiles/ stay tied to the kernel code: a comment
    edit keeps the hash, a code edit changes it."""
    src = "int f(int x) {\n  // doubles x\n  return 2 * x; /* cheap */\n}\n"
    assert bench.strip_comments(src) == bench.strip_comments(src.replace("doubles x", "twice x"))
    assert bench.strip_comments(src) != bench.strip_comments(src.replace("2 * x", "3 * x"))
    assert "//" not in bench.strip_comments(src) and "/*" not in bench.strip_comments(src)


def test_profile_traffic_matches_current_kernel_code():
    """When profiles/ holds ncu traffic for the current kernel code, it is the
    algorithmic bytes plus at most 2% (no re-reads)."""
    traffic = bench.traffic_from_profiles(bench.kernel_source_hash())
    if traffic is None:
        pytest.skip("profiles/ holds no ncu traffic for the current kernel code (bench reports null)")
    for kv in bench.SWEEP:
        algorithmic = bench.attend_bytes(1, bench.N_HEAD, bench.N_KV_HEAD, bench.HEAD_DIM, [kv])
        assert 1.0 <= traffic[kv] / algorithmic < 1.02
