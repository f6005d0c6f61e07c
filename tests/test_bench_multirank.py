"""The multi-rank path of the benchmark (replicas, max over ranks), run as
two gloo ranks on the CPU."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    w, r, local = bench.dist_setup("gloo")
    assert (w, r, local) == (world, rank, rank)
    step_ms = [1.0 + rank, 2.0 + rank, 3.0 + rank]  # rank 1 is the slow one: 9 ms in all
    bench.barrier(w)
    agg = bench.aggregate(step_ms, 1000, w, torch.device("cpu"))
    results[rank] = (agg["total_ms"], agg["ms_per_step"], agg["value"])
    dist.destroy_process_group()


def test_two_rank_aggregate_takes_the_slowest_rank():
    world, port = 2, _free_port()
    results = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, port, results), nprocs=world, join=True)
    for rank in range(world):
        total_ms, ms_per_step, value = results[rank]
        assert total_ms == pytest.approx(9.0)
        assert ms_per_step == pytest.approx(3.0)
        # 2 ranks x 1000 tokens x 3 steps in 9 ms
        assert value == pytest.approx(2 * 1000 * 3 / 9e-3)


def test_single_rank_aggregate():
    agg = bench.aggregate([2.0, 2.0], 500, 1, torch.device("cpu"))
    assert agg["value"] == pytest.approx(500 * 2 / 4e-3)
    assert agg["ms_per_step"] == pytest.approx(2.0)


def test_layer_accounting_counts_keys():
    from csa_inputs import packs
    spec = packs.pack_spec("tiny")
    acc = bench.layer_accounting(spec, spec.layers[0])
    # window: min(16, pos+1) per token; compressed: min(8, floor((pos+1)/4))
    keys = 0
    for L in spec.lengths:
        for pos in range(L):
            keys += min(16, pos + 1) + min(8, (pos + 1) // 4)
    assert acc["keys"] == keys
    assert acc["kv_bytes"] == keys * 1024
    assert acc["mla_flops"] == 4 * 512 * 4 * keys


def test_layer_accounting_counts_listed_rows():
    """cmp_keys (the KL gradient's listed rows) = per token the oracle's
    visible-block count, capped at top-k."""
    import numpy as np

    import oracle
    from csa_inputs import packs
    lengths = (1, 3, 37, 120, 9)
    layer = packs.LayerSpec(cmp_ratio=4, indexer=True, topk=8, index_heads=4, index_dim=64)
    spec = packs.PackSpec("custom", lengths, heads=4, dim=512, win_left=15, layers=(layer,),
                          seed=1)
    acc = bench.layer_accounting(spec, layer)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    cuc = oracle.compress_cu_seqlens(cu, 4)
    T, tc = int(cu[-1]), int(cuc[-1])
    rng = np.random.default_rng(0)
    _, _, _, _, nvis = oracle.indexer_topk(rng.standard_normal((T, 4, 64)),
                                           rng.standard_normal((tc, 64)),
                                           rng.standard_normal((T, 4)), T, cu, cuc, 4, 8)
    assert acc["cmp_keys"] == int(np.minimum(nvis, 8).sum())
