"""Host logic of bench.py for N > 1 ranks, on CPU with gloo (world size 2):
max-over-ranks timing and the whole-job throughput aggregate."""

import os
import socket

import json

import pytest
import torch.multiprocessing as mp

import bench


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
        ms = 100.0 + 50.0 * rank  # rank 1 is the slow one
        bench.barrier(world)
        worst = bench.reduce_max(ms, world, torch.device("cpu"))
        out[rank] = (worst, bench.aggregate_tokens_per_s(16384, world, 10, worst))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_aggregate():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    assert out[0][0] == out[1][0] == 150.0
    assert out[0][1] == pytest.approx(16384 * 2 * 10 / 0.150)


def test_single_rank_aggregate_and_defaults():
    assert bench.aggregate_tokens_per_s(100, 1, 4, 200.0) == pytest.approx(2000.0)
    assert bench.reduce_max(3.0, 1, None) == 3.0
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_traffic_lookup_ignores_stale_counters(tmp_path, monkeypatch):
    assert bench.traffic_for("no_such_kernel") is None
    # a fake repository: the entry counts only while its sources are unchanged
    (tmp_path / "profiles").mkdir()
    (tmp_path / "a.cu").write_text("one")
    (tmp_path / "b.cu").write_text("two")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench.sources_sha(["a.cu", "b.cu"])
    entry = {"source_files": ["a.cu", "b.cu"], "source_sha": sha,
             "dram_bytes_per_full_launch": 1234}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"kernels": {"k": entry}}))
    assert bench.traffic_for("k") == 1234
    (tmp_path / "b.cu").write_text("changed")
    assert bench.traffic_for("k") is None
    assert bench.sources_sha(["a.cu", "missing.cu"]) is None


def test_backward_rooflines():
    # the joint bound of a backward whose kernels may overlap: the three
    # GEMMs' 6THV flops at the tensor peak or their algorithmic bytes at HBM
    # speed, whichever is longer; never above the serial sum of per-kernel
    # bounds, and equal to the flop term once the batch is compute-bound
    peaks = {"bf16_tflops": 2000.0, "hbm_gbs": 8000.0}
    H, V = 3584, 152064
    for T in (1, 128, 512, 2048, 16384):
        joint = bench.bwd_joint_roofline_ms(T, H, V, peaks)
        serial = sum(bench.bwd_roofline_ms(T, H, V, peaks).values())
        flop_ms = 6.0 * T * H * V / 2000e12 * 1e3
        byte_ms = (2.0 * V * H * 2 + 4.0 * V * H + 6.0 * T * H + 6.0 * T * V) / 8000e9 * 1e3
        assert joint == pytest.approx(max(flop_ms, byte_ms), rel=1e-12)
        assert joint <= serial * (1 + 1e-12)
    # one row: all bytes (W read twice, grad_weight written in fp32)
    assert bench.bwd_joint_roofline_ms(1, H, V, peaks) == pytest.approx(
        (8.0 * V * H + 6.0 * H + 6.0 * V) / 8000e9 * 1e3, rel=1e-12)
    # a long batch: all flops
    assert bench.bwd_joint_roofline_ms(16384, H, V, peaks) == pytest.approx(
        6.0 * 16384 * H * V / 2000e12 * 1e3, rel=1e-12)


def test_invariance_cases_count_only_real_mismatches():
    # a row-wise map has no mismatch in any case; one that depends on the
    # batch size (a per-batch offset) is caught in every case but the whole
    # batch, and so is one whose rows see their position in the batch
    import torch

    x = torch.randn(300, 5, generator=torch.Generator().manual_seed(3))
    cpu = torch.device("cpu")
    subs = ((1, (0, 299)), (7, (0, 100)), (64, (5,)))
    row_wise = bench.invariance_cases(lambda r: (x[r] * 2.0, (x[r] + 1).to(torch.bfloat16)), 300,
                                      subs, window=128, dev=cpu)
    assert row_wise["mismatched_values"] == 0
    assert len(row_wise["cases"]) == 5 + 3 + 3 + 1
    assert row_wise["rows_compared"] == 2 + 14 + 64 + 3 * 128 + 3 * 300 + 300
    by_size = bench.invariance_cases(lambda r: (x[r] + float(r.numel()),), 300, subs,
                                     window=128, dev=cpu)
    assert all(c["mismatched"] > 0 for c in by_size["cases"]
               if c.get("batch") not in (300, None) or "embedded_rows" in c)
    assert all(c["mismatched"] == 0 for c in by_size["cases"] if "shuffled" in c)
    by_pos = bench.invariance_cases(lambda r: (x[r] + torch.arange(r.numel()).float()[:, None],),
                                    300, subs, window=128, dev=cpu)
    # (the embedded case keeps every row's position, so it cannot show this one)
    assert all(c["mismatched"] > 0 for c in by_pos["cases"]
               if c.get("start", 1) != 0 and "embedded_rows" not in c)


def test_packed_invariance_over_sequences():
    import torch

    lengths = (5, 9, 3, 12, 7, 4, 8, 6)
    T = sum(lengths)
    x = torch.randn(T, 3, generator=torch.Generator().manual_seed(4))
    cpu = torch.device("cpu")
    ok = bench.packed_invariance(lambda r: (x[r].exp(),), lengths, seeds=(1, 2), alone=(0, 3, 7),
                                 dev=cpu)
    assert ok["mismatched_values"] == 0 and ok["rows_compared"] == 2 * T + 5 + 12 + 6
    # a result that depends on the packing (each row plus the batch mean) is caught
    bad = bench.packed_invariance(lambda r: (x[r] + x[r].mean(),), lengths, seeds=(1,),
                                  alone=(3,), dev=cpu)
    assert bad["cases"][-1]["mismatched"] > 0


def test_cpu_model_names_the_host():
    name = bench.cpu_model()
    assert isinstance(name, str) and name and name != "unknown"
