"""Host side of the vocab-parallel exchange (invariant_lm_head_gb300.vocab_parallel)
on CPU with gloo, world size 2: the shard layout check, the rank-ordered
all-gather of chunk planes with unequal chunk counts, the stacked gather of
grad_hidden partials, and the exact label-logit sum. No GPU is involved; the
kernels these feed are covered by tests/test_gpu_vocab_parallel.py."""

import os
import socket

import pytest
import torch.multiprocessing as mp

from invariant_lm_head_gb300 import vocab_parallel as vp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    import torch
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        res = {}
        V_total = 5000  # 5 chunks: rank 0 holds 3 (rows 0..3071), rank 1 holds 2 (3072..4999)
        b0, b1 = vp.shard_bounds(V_total, world, rank)
        res["bounds"] = (b0, b1)
        counts = vp.exchange_layout(b0, b1 - b0, V_total)
        res["counts"] = counts
        T = 6
        n = -(-(b1 - b0) // vp.CHUNK)
        # plane p, local chunk c, row t -> a value naming (rank, p, c, t)
        planes = torch.tensor([[[1000 * rank + 100 * p + 10 * c + t for t in range(T)]
                                for c in range(n)] for p in range(3)], dtype=torch.float32)
        res["whole"] = vp.gather_chunks(planes, counts).tolist()
        part = torch.full((T, 4), float(rank + 1))
        res["ranks"] = vp.gather_ranks(part).tolist()
        # label logits: rank r holds rows whose label is in its shard, 0 elsewhere
        zl = torch.zeros(T)
        zl[rank::2] = torch.tensor([-0.1234567, 3.5, 7.25], dtype=torch.float32)[: len(range(rank, T, 2))]
        res["zl"] = vp.sum_label_logits(zl).tolist()
        # a layout that does not tile the vocabulary is refused on every rank
        try:
            vp.exchange_layout(b0 + (512 if rank == 1 else 0), b1 - b0, V_total)
            res["bad"] = "accepted"
        except ValueError as e:
            res["bad"] = str(e)
        out[rank] = res
    finally:
        dist.destroy_process_group()


def _three_rank_worker(rank, world, port, out):
    import torch
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        V_total, T = 5000, 4  # 5 chunks over 3 ranks: 2, 2, 1
        b0, b1 = vp.shard_bounds(V_total, world, rank)
        counts = vp.exchange_layout(b0, b1 - b0, V_total)
        n = -(-(b1 - b0) // vp.CHUNK)
        planes = torch.full((3, n, T), float(rank))
        whole = vp.gather_chunks(planes, counts)
        out[rank] = (counts, whole[0, :, 0].tolist(), vp.gather_ranks(torch.tensor([rank])).tolist())
    finally:
        dist.destroy_process_group()


def test_exchange_on_three_gloo_ranks():
    world = 3
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_three_rank_worker, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn")
    for r in range(world):
        counts, chunk_owner, ranks = out[r]
        assert counts == [2, 2, 1]
        assert chunk_owner == [0.0, 0.0, 1.0, 1.0, 2.0]  # rank order along the vocabulary
        assert ranks == [[0], [1], [2]]


def test_exchange_on_two_gloo_ranks():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    r0, r1 = out[0], out[1]
    assert r0["bounds"] == (0, 3072) and r1["bounds"] == (3072, 5000)
    assert r0["counts"] == r1["counts"] == [3, 2]
    # chunk planes: rank 0's three chunks, then rank 1's two, on both ranks
    assert r0["whole"] == r1["whole"]
    whole = r0["whole"]
    assert len(whole) == 3 and all(len(p) == 5 for p in whole)
    for p in range(3):
        for c in range(5):
            rank, lc = (0, c) if c < 3 else (1, c - 3)
            assert whole[p][c] == [1000 * rank + 100 * p + 10 * lc + t for t in range(6)]
    assert r0["ranks"] == r1["ranks"] == [[[1.0] * 4] * 6, [[2.0] * 4] * 6]
    # the sum picks each row's single nonzero term exactly
    import numpy as np

    want = np.array([-0.1234567, -0.1234567, 3.5, 3.5, 7.25, 7.25], dtype=np.float32)
    assert np.array_equal(np.array(r0["zl"], dtype=np.float32), want)
    assert r0["zl"] == r1["zl"]
    assert "tile the vocabulary" in r0["bad"] and "tile the vocabulary" in r1["bad"]


@pytest.mark.parametrize("V,world", [(152064, 2), (152064, 4), (1025, 2), (4096, 3), (100, 1)])
def test_shard_bounds_tile_the_vocabulary(V, world):
    bounds = [vp.shard_bounds(V, world, r) for r in range(world)]
    assert bounds[0][0] == 0 and bounds[-1][1] == V
    for (a0, a1), (b0, b1) in zip(bounds, bounds[1:]):
        assert a1 == b0 and a0 % vp.CHUNK == 0 and b0 % vp.CHUNK == 0
    chunks = [-(-(b - a) // vp.CHUNK) for a, b in bounds]
    assert min(chunks) >= 1 and max(chunks) - min(chunks) <= 1


def test_shard_bounds_refuses_more_ranks_than_chunks():
    with pytest.raises(ValueError):
        vp.shard_bounds(1024, 2, 0)
