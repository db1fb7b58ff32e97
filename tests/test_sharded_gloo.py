"""KV-sequence sharding across ranks, host logic on 2 and 3 gloo ranks (CPU).

Each rank takes its part of every request's keys (kv_shard_range: prefix
slices and page-aligned suffix slices), computes the state of its part, and
the ranks exchange the states with gather_states.  Here the per-rank states
come from the oracle (the CUDA kernels need a GPU; they are covered by the
GPU test of the same path), and the gathered states are merged with the
oracle's n-ary merge: the result must be the oracle's attention over the
whole key set ("Attention States and Recursive Attention", Applications)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from paged_kv_cascade_gb300.sharded import gather_states, kv_shard_range


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _problem():
    import workloads
    return workloads.make_problem(batch=6, hq=8, hkv=2, d=128, dtype="bf16", prefix_lens=[100, 37],
                                  prefix_groups=[3, 2], suffix=("list", [0, 5, 70, 16, 33, 129]),
                                  page_size=16, seed=71, poison=True, extra_pages=2)


def _worker(rank, world, port, out):
    import oracle
    import workloads
    from pkc_testing import oracle_args
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        p = _problem()
        part = workloads.shard_problem(p, rank, world, kv_shard_range)
        o, lse = oracle.attention_rows(part["q"], **oracle_args(part))
        B, Hq, D = p["q"].shape
        o_all, lse_all = gather_states(torch.from_numpy(o.reshape(B, Hq, D)),
                                       torch.from_numpy(lse.reshape(B, Hq)))
        v, s = oracle.merge_n(o_all.numpy().reshape(world, B * Hq, D), lse_all.numpy().reshape(world, B * Hq))
        out[rank] = (v, s, int(part["cache_seqlens"].sum()), int(part["prefix_kv_indptr"][-1]))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_sharded_states_merge_to_the_whole_key_set(world):
    import oracle
    from pkc_testing import oracle_args
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
    p = _problem()
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p))
    # every rank merged the same states in the same order: identical results
    for r in range(1, world):
        assert np.array_equal(out[r][0], out[0][0]) and np.array_equal(out[r][1], out[0][1])
    v, s = out[0][0], out[0][1]
    fin = ~np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(s), ~fin)
    assert np.max(np.abs(v - ref_o)) < 1e-12 and np.max(np.abs(s[fin] - ref_lse[fin])) < 1e-12
    # the shards hold every key once
    assert sum(out[r][2] for r in range(world)) == int(p["cache_seqlens"].sum())
    assert sum(out[r][3] for r in range(world)) == int(p["prefix_kv_indptr"][-1])


def test_shard_ranges_cover_every_token_once_page_aligned():
    for n in (0, 1, 15, 16, 17, 100, 4097):
        for world in (1, 2, 3, 8):
            for align in (1, 16):
                spans = [kv_shard_range(n, r, world, align) for r in range(world)]
                assert spans[0][0] == 0 and spans[-1][1] == n
                for (a, b), (c, d) in zip(spans, spans[1:]):
                    assert b == c
                for a, b in spans:
                    assert a % align == 0 and a <= b
                    assert b == n or b % align == 0
    with pytest.raises(ValueError):
        kv_shard_range(10, 2, 2)
