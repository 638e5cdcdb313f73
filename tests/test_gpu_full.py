"""The five measured workloads at full size, in the launch configuration the
bench times (one dsi_indexed_attention call per batch), checked row by row
against the oracle on sampled rows (indices bit-exact, outputs within the
relative tolerance), plus properties that hold for every row."""
import numpy as np
import pytest
import torch

import oracle
from indexed_sparse_attention_indexer_gb300 import binding
from indexed_sparse_attention_indexer_gb300 import workloads as W
from tests.parity import assert_lse_close, assert_out_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def decode_subset(g, rows):
    """CPU copy of the sampled sequences of a device decode workload, laid out
    for the oracle (a paged pool keeps only the pages of those sequences, in
    the block table's order)."""
    sub = g.to(DEV)
    sub.q_idx, sub.w, sub.q = g.q_idx[rows], g.w[rows], g.q[rows]
    sub.seq_lens = g.seq_lens[rows]
    if g.block_table is None:
        sub.k_idx, sub.latent = g.k_idx[rows], g.latent[rows]
        sub.k_scale = None if g.k_scale is None else g.k_scale[rows]
    else:
        bt = g.block_table[rows].long()
        used = bt.clamp(min=0)
        P = used.numel()
        flat = used.view(-1)
        sub.k_idx = g.k_idx.view(torch.uint8)[flat].view(g.k_idx.dtype)
        sub.latent = g.latent[flat]
        sub.k_scale = None if g.k_scale is None else g.k_scale[used.view(-1)]
        nb = torch.arange(P, device=DEV, dtype=torch.int32).view(bt.shape)
        sub.block_table = torch.where(bt >= 0, nb, torch.full_like(nb, -1))
    return sub.to("cpu")


def check_decode(g, out, lse, idx, count, rows):
    ws = decode_subset(g, rows)
    for i, b in enumerate(rows):
        ref = oracle.decode_row(ws, i)
        assert np.array_equal(idx[b].cpu().numpy(), ref["idx"]), f"row {b}"
        assert int(count[b]) == ref["count"]
        assert_out_close(out[b].float().cpu().numpy(), ref["out"], f"row {b}")
        assert_lse_close(lse[b].cpu().numpy(), ref["lse"], f"row {b}")


def check_all_rows_properties(idx, count, lens_of_row):
    """Every row: ascending valid indices below its visible length, -1 tail."""
    idx = idx.cpu()
    count = count.cpu()
    K = idx.shape[1]
    n = torch.as_tensor(lens_of_row).to(torch.int64)
    assert torch.equal(count.to(torch.int64), torch.clamp(n, max=K))
    ar = torch.arange(K).view(1, K)
    valid = ar < count.view(-1, 1)
    assert torch.all((idx >= 0) == valid)
    x = torch.where(valid, idx.to(torch.int64), torch.full_like(idx, 1 << 40, dtype=torch.int64))
    assert torch.all((x[:, 1:] > x[:, :-1]) | ~valid[:, 1:])
    assert torch.all(torch.where(valid, idx.to(torch.int64) < n.view(-1, 1), torch.ones_like(valid)))


def _run(g):
    out, lse, idx, count = binding.layer(g)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    return out, lse, idx, count


def test_config1_decode_s2048():
    g = W.make_config(1, device=DEV)
    out, lse, idx, count = _run(g)
    check_decode(g, out, lse, idx, count, [0])


def test_config2_decode_b64_s32768():
    g = W.make_config(2, device=DEV)
    out, lse, idx, count = _run(g)
    check_all_rows_properties(idx, count, g.seq_lens.cpu())
    check_decode(g, out, lse, idx, count, [0, 17, 42, 63])


def test_config5_paged_fp8_decode():
    g = W.make_config(5, device=DEV)
    out, lse, idx, count = _run(g)
    check_all_rows_properties(idx, count, g.seq_lens.cpu())
    lens = g.seq_lens.cpu()
    rows = [int(lens.argmax()), int(lens.argmin()), 3, 77]
    check_decode(g, out, lse, idx, count, rows)


def _prefill_rows(T, seed=0):
    rng = np.random.default_rng(seed)
    return sorted(set(list(range(8)) + list(range(T - 8, T)) + rng.integers(0, T, 16).tolist()))


def check_prefill(g, out, lse, idx, count, rows):
    cpu = g.to("cpu")
    for t in rows:
        ref = oracle.prefill_row(cpu, t)
        assert np.array_equal(idx[t].cpu().numpy(), ref["idx"]), f"row {t}"
        assert_out_close(out[t].float().cpu().numpy(), ref["out"], f"row {t}")
        assert_lse_close(lse[t].cpu().numpy(), ref["lse"], f"row {t}")


def test_config3_prefill_t8192():
    g = W.make_config(3, device=DEV)
    out, lse, idx, count = _run(g)
    check_all_rows_properties(idx, count, torch.arange(1, g.T + 1))
    check_prefill(g, out, lse, idx, count, _prefill_rows(g.T))


@pytest.mark.parametrize("chunk", [0, 15, 31])
def test_config4_chunked_prefill(chunk):
    c = W.CONFIGS[4]
    k_idx, latent = W.make_long_cache(c["S"], c["d"], c["seed"], DEV)
    g = W.make_chunk(k_idx, latent, chunk, c["T"], c["H_i"], c["K"], c["H"], c["seed"])
    out, lse, idx, count = _run(g)
    check_all_rows_properties(idx, count, torch.arange(1, g.T + 1) + g.q_offset)
    check_prefill(g, out, lse, idx, count, _prefill_rows(g.T, seed=chunk))
