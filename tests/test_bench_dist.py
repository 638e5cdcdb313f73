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
    args = argparse.Namespace(config=1, steps=1, warmup=0, cpu_seconds=0.1, tokens_per_seq=1)
    assert bench.run_reference(args) is None


def test_reference_arm_line_on_cpu(monkeypatch):
    """Rank 0 of the reference arm times the oracle on a bounded sample (tiny
    workload here) and prints the contract's keys."""
    import argparse
    import bench
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.delenv("RANK", raising=False)
    args = argparse.Namespace(config=1, steps=2, warmup=1, cpu_seconds=0.5, tokens_per_seq=1)
    line = bench.run_reference(args)
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == bench.host_cores() and cb["nproc"] >= 1
    assert cb["single_core_value"] > 0
    # the GPU arm's config keys, so both arms describe the same workload
    assert set(line["config"]) == {"workload", "batch", "history", "indexer", "topk", "mla_heads",
                                   "parallelism", "l2"}
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


def test_algorithmic_flops_count_the_scored_prefill_rows():
    """Indexer flops: every visible position of a decode row; for a prefill,
    only the rows with more than K positions of history (a row seeing at most
    K takes them all, whatever the scores).  Attention flops: min(K, visible)
    rows per query, either way."""
    import bench
    from indexed_sparse_attention_indexer_gb300 import workloads as W
    K = 16
    pf = W.make_prefill(40, 50, 4, 64, K, 16, seed=2, q_offset=10)
    vis = [10 + t + 1 for t in range(40)]                 # 11 .. 50
    scored = sum(v for v in vis if v > K)
    fl = bench.algorithmic_flops(pf)
    assert fl["indexer"] == 2 * scored * 4 * 64
    assert fl["mla"] == 2 * sum(min(K, v) for v in vis) * 16 * (576 + 512)
    dec = W.make_decode(2, 0, 4, 64, K, 16, seed=1, lengths=[100, 9])
    assert bench.algorithmic_flops(dec)["indexer"] == 2 * (100 + 9) * 4 * 64


def test_zigzag_partition_covers_and_balances():
    from indexed_sparse_attention_indexer_gb300 import partition as P
    for T, world in ((8192, 2), (8192, 8), (4096, 4), (130, 3), (7, 4), (1, 2)):
        segs = P.zigzag_segments(T, world)
        rows = sorted(t for r in range(world) for t in P.rank_rows(T, world, r))
        assert rows == list(range(T)), (T, world)
        if T >= 64 * world:
            work = [P.causal_pairs(s, q_offset=0) for s in segs]
            assert max(work) / min(work) < 1.01, (T, world, work)
            cont = [P.causal_pairs(s) for s in P.contiguous_segments(T, world)]
            assert max(cont) / min(cont) > 2.0          # what the zigzag avoids
    # the pair count is the sum of the visible lengths
    assert P.causal_pairs([(0, 3)], q_offset=5) == 6 + 7 + 8


def _zigzag_rank(rank, world, port, out):
    """Each rank runs its zigzag rows of a tiny prefill through the oracle (the
    CPU stand-in for its GPU) and the rows are reassembled on rank 0."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from indexed_sparse_attention_indexer_gb300 import partition as P
    from indexed_sparse_attention_indexer_gb300 import workloads as W
    ws = W.make_prefill(40, 70, 4, 64, 8, 16, seed=9, q_offset=30)   # same seeded cache on every rank
    mine = {t: oracle.prefill_row(ws, t) for t in P.rank_rows(ws.T, world, rank)}
    got = [None] * world
    dist.all_gather_object(got, {t: (r["idx"], r["out"]) for t, r in mine.items()})
    if rank == 0:
        merged = {}
        for part in got:
            assert not (set(part) & set(merged))
            merged.update(part)
        out["rows"] = sorted(merged)
        ref = oracle.layer(ws)
        out["same"] = all(
            (merged[t][0] == ref[t]["idx"]).all() and (merged[t][1] == ref[t]["out"]).all()
            for t in range(ws.T))
    dist.destroy_process_group()


def test_zigzag_rows_reassemble_to_the_one_rank_result():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_zigzag_rank, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out["rows"] == list(range(40))
    assert out["same"]
