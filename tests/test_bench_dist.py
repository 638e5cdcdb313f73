"""The multi-rank bench logic on CPU: two gloo ranks agree on the slowest rank's
time and the whole-job throughput; the reference arm runs on rank 0 only."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms_local = 10.0 + 5.0 * rank          # rank 1 is the slow one
    ms = bench.max_over_ranks(ms_local, world)
    val = bench.whole_job_tokens_per_s(64, world, 20, ms)
    bench.barrier(world)
    out[rank] = (ms, val)
    dist.destroy_process_group()


def test_two_ranks_agree_on_max_time_and_value():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0] == out[1]
    ms, val = out[0]
    assert ms == 15.0
    assert val == pytest.approx(64 * 2 * 20 / 0.015)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    import argparse
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    args = argparse.Namespace(config=1, steps=1, warmup=0, cpu_seconds=0.1)
    assert bench.run_reference(args) is None


def test_reference_arm_line_on_cpu(monkeypatch):
    """Rank 0 of the reference arm times the oracle on a bounded sample (tiny
    workload here) and prints the contract's keys."""
    import argparse
    import bench
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.delenv("RANK", raising=False)
    args = argparse.Namespace(config=1, steps=2, warmup=1, cpu_seconds=0.5)
    line = bench.run_reference(args)
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


def test_algorithmic_bytes_of_the_quantised_variants():
    """Per-step byte accounting: MXFP8 keys move d code bytes plus d/G scale bytes
    per visible position; an FP8 latent row moves 576 code bytes plus five fp32
    tile scales; the bf16 forms 2 bytes per element."""
    import bench
    from indexed_sparse_attention_indexer_gb300 import workloads as W
    lens = [100, 37]
    base = W.make_decode(2, 0, 4, 64, 16, 16, seed=1, lengths=lens)
    mx = W.make_decode(2, 0, 4, 64, 16, 16, seed=1, lengths=lens, k_mx_group=32)
    l8 = W.make_decode(2, 0, 4, 64, 16, 16, seed=1, lengths=lens, latent_fp8=True)
    n = sum(lens)
    sel = sum(min(16, x) for x in lens)
    assert bench.algorithmic_bytes(base)["index_keys"] == n * 64 * 2
    assert bench.algorithmic_bytes(mx)["index_keys"] == n * (64 + 2)
    assert bench.algorithmic_bytes(base)["gather"] == sel * 576 * 2
    assert bench.algorithmic_bytes(l8)["gather"] == sel * (576 + 5 * 4)
