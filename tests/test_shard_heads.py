"""KV-head partition of one decode step over several ranks
(decode_attn_shard_heads): the host arithmetic of the partition, and two gloo
ranks on CPU that each run the oracle on their own block of KV heads (with
their query heads) and gather the outputs: laid side by side on the head
axis they are, bit for bit, the single-rank oracle's output, and each rank's
cache block after the append is the matching block of the single-rank cache.
Every (sequence, KV head) group is independent, so no data is exchanged
before the gather; one GPU per rank is not needed to check that."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import decode_attention_static_gb300 as da
from decode_attention_static_gb300 import build as da_build


@pytest.fixture(scope="module", autouse=True)
def _library():
    da_build.build_library()
    da.load_library()


@pytest.mark.parametrize("n_head,n_kv_head", [(32, 8), (16, 16), (4, 1), (64, 8), (24, 6), (40, 5)])
@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
def test_partition_covers_every_head_once_in_rank_order(n_head, n_kv_head, world):
    G = n_head // n_kv_head
    parts = [da.shard_heads(n_head, n_kv_head, world, r) for r in range(world)]
    kv_next = h_next = 0
    for kv0, nkv, h0, nh in parts:
        assert kv0 == kv_next and h0 == h_next          # contiguous, in rank order
        assert nh == G * nkv and h0 == G * kv0          # every KV head with its own query heads
        kv_next, h_next = kv0 + nkv, h0 + nh
    assert kv_next == n_kv_head and h_next == n_head    # everything, once
    sizes = [p[1] for p in parts]
    assert max(sizes) - min(sizes) <= 1 and sizes == sorted(sizes, reverse=True)


def test_partition_rejects_bad_arguments():
    for args in [(30, 8, 2, 0), (32, 8, 0, 0), (32, 8, 2, 2), (32, 8, 2, -1), (0, 8, 2, 0)]:
        with pytest.raises(da.DecodeAttnError) as e:
            da.shard_heads(*args)
        assert e.value.status == -2
    assert da.shard_heads(4, 2, 4, 3) == (2, 0, 4, 0)  # more ranks than KV heads: the last hold none


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _step():
    import workloads as W

    # batched streaming shape, ragged positions (one at 0), NaN tails
    return W.decode_step(3, 16, 8, 64, 700, "bf16", [699, 0, 345], seed=81)


def _rank_main(rank, world, port, results):
    import torch
    import torch.distributed as dist

    import oracle
    import workloads as W

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ora = oracle.default()
    step = _step()
    kv0, nkv, h0, nh = da.shard_heads(step.n_head, step.n_kv_head, world, rank)
    # this rank's own contiguous block of every tensor (what it would hold on its GPU)
    q = W.raw_bits(step.q[:, h0:h0 + nh]).copy()
    kc = W.raw_bits(step.k_cache[:, kv0:kv0 + nkv]).copy()
    vc = W.raw_bits(step.v_cache[:, kv0:kv0 + nkv]).copy()
    kn = W.raw_bits(step.k_new[:, kv0:kv0 + nkv]).copy()
    vn = W.raw_bits(step.v_new[:, kv0:kv0 + nkv]).copy()
    ora.kvcache_append(kc, vc, kn, vn, step.position_ids.numpy())
    out = ora.decode_attn(q, kc, vc, step.kv_len.numpy(), nh, nkv, step.dtype)
    gathered = [None] * world
    dist.all_gather_object(gathered, (out, kc, vc))
    if rank == 0:
        results["out"] = np.concatenate([g[0] for g in gathered], axis=1)
        results["k"] = np.concatenate([g[1] for g in gathered], axis=1)
        results["v"] = np.concatenate([g[2] for g in gathered], axis=1)
    dist.destroy_process_group()


def test_two_ranks_gather_the_single_rank_result(ora):
    import workloads as W

    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        results = mgr.dict()
        mp.start_processes(_rank_main, args=(2, port, results), nprocs=2, join=True, start_method="spawn")
        r = dict(results)
    step = _step()
    kb, vb = W.raw_bits(step.k_cache).copy(), W.raw_bits(step.v_cache).copy()
    ora.kvcache_append(kb, vb, W.raw_bits(step.k_new), W.raw_bits(step.v_new), step.position_ids.numpy())
    ref = ora.decode_attn(W.raw_bits(step.q), kb, vb, step.kv_len.numpy(), step.n_head, step.n_kv_head, step.dtype)
    assert np.array_equal(r["k"], kb) and np.array_equal(r["v"], vb)
    assert np.array_equal(r["out"], ref)
