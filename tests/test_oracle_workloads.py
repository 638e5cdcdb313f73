"""The oracle's per-row drivers on seeded workloads, and the workload recipes (CPU)."""
import numpy as np
import torch

import oracle
from indexed_sparse_attention_indexer_gb300 import workloads as W


def test_recipe_values():
    ws = W.make_decode(3, 100, 4, 16, 8, 2, seed=1, k_fp8=True, page_size=16,
                       lengths=[100, 1, 37])
    qi = ws.q_idx.float()
    assert qi.min() >= -3 and qi.max() <= 3 and torch.equal(qi, qi.round())
    ki = ws.k_idx.float()
    assert ki.min() >= -3 and ki.max() <= 3 and torch.equal(ki, ki.round())
    assert torch.equal(ws.w * 128, torch.floor(ws.w * 128)) and ws.w.min() >= 0 and ws.w.max() < 1
    e = torch.log2(ws.k_scale)
    assert torch.equal(e, e.round()) and e.min() >= -4 and e.max() <= 0
    # block table: every used page id distinct, unused entries -1
    used = [int(x) for b in range(3) for x in ws.block_table[b] if x >= 0]
    assert len(used) == len(set(used)) == (100 + 15) // 16 + 1 + (37 + 15) // 16
    L = W.loguniform_lengths(4096, 1024, 131072, torch.Generator().manual_seed(7), "cpu")
    assert L.min() >= 1024 and L.max() <= 131072
    # log-uniform: the median sits near the geometric mean (~11585)
    assert 9000 < float(L.float().median()) < 14500


def _as_paged(ws, page):
    """Re-lay a contiguous decode workload into a shuffled page pool (test helper)."""
    B, S = ws.k_idx.shape[:2]
    npg = (S + page - 1) // page
    P = B * npg
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(5))
    kp = torch.zeros((P, page) + ws.k_idx.shape[2:], dtype=ws.k_idx.dtype)
    lp = torch.zeros((P, page) + ws.latent.shape[2:], dtype=ws.latent.dtype)
    bt = torch.full((B, npg), -1, dtype=torch.int32)
    for b in range(B):
        for j in range(npg):
            p = int(perm[b * npg + j])
            n = min(page, S - j * page)
            kp[p, :n] = ws.k_idx[b, j * page:j * page + n]
            lp[p, :n] = ws.latent[b, j * page:j * page + n]
            bt[b, j] = p
    out = ws.to("cpu")
    out.k_idx, out.latent, out.block_table, out.page_size = kp, lp, bt, page
    return out


def test_paged_equals_contiguous():
    ws = W.make_decode(3, 150, 4, 16, 20, 4, seed=3, lengths=[150, 61, 64])
    pg = _as_paged(ws, 16)
    for b in range(3):
        a = oracle.decode_row(ws, b)
        c = oracle.decode_row(pg, b)
        assert np.array_equal(a["idx"], c["idx"]) and a["count"] == c["count"]
        assert np.array_equal(a["out"], c["out"])


def test_prefill_causality_and_chunk_invariance():
    T, S = 24, 40
    ws = W.make_prefill(T, S, 4, 16, 6, 2, seed=4, q_offset=16)
    res = oracle.layer(ws)
    for t, r in res.items():
        sel = r["idx"][:r["count"]]
        assert sel.max() <= ws.q_offset + t
        assert r["count"] == min(ws.K, ws.q_offset + t + 1)
    full = W.make_prefill(4, 8, 4, 16, 6, 2, seed=4, q_offset=0)
    r0 = oracle.prefill_row(full, 0)
    assert r0["count"] == 1 and r0["idx"][0] == 0
    # a row's result depends only on its own query and the visible prefix
    sub = ws.to("cpu")
    sub.q_idx, sub.w, sub.q = ws.q_idx[5:9], ws.w[5:9], ws.q[5:9]
    sub.q_offset = ws.q_offset + 5
    for t in range(4):
        a = oracle.prefill_row(sub, t)
        b = res[5 + t]
        assert np.array_equal(a["idx"], b["idx"]) and np.array_equal(a["out"], b["out"])


def test_decode_row_short_history_takes_all():
    ws = W.make_decode(2, 0, 4, 16, 32, 2, seed=6, lengths=[5, 40])
    r = oracle.decode_row(ws, 0)
    assert r["count"] == 5 and list(r["idx"][:6]) == [0, 1, 2, 3, 4, -1]
    r = oracle.decode_row(ws, 1)
    assert r["count"] == 32


def test_multi_token_rows_reduce_to_decode_rows():
    """A multi-token step: T = 1 is a decode row; the last candidate sees the whole
    history (a decode row of the full length); candidate t of a sequence of length L
    equals a one-token decode of the same query over a history of L - (T-1-t) rows."""
    T = 3
    ws = W.make_decode(2, 0, 4, 16, 8, 2, seed=12, lengths=[20, 9], tokens_per_seq=T)
    assert ws.T == 2 * T and ws.tokens_per_seq == T
    one = W.make_decode(2, 0, 4, 16, 8, 2, seed=12, lengths=[20, 9])
    assert np.array_equal(oracle.multi_token_row(one, 1, 1)["out"], oracle.decode_row(one, 1)["out"])
    for r in range(ws.T):
        b, t = divmod(r, T)
        got = oracle.multi_token_row(ws, r, T)
        # the same query on a workload whose sequence b is cut to L - (T-1-t) rows
        cut = ws.to("cpu")
        cut.q_idx, cut.w, cut.q = ws.q_idx[r:r + 1].repeat(2, 1, 1), ws.w[r:r + 1].repeat(2, 1), \
            ws.q[r:r + 1].repeat(2, 1, 1)
        lens = ws.seq_lens.clone()
        lens[b] = int(ws.seq_lens[b]) - (T - 1 - t)
        cut.seq_lens = lens
        ref = oracle.decode_row(cut, b)
        assert np.array_equal(got["idx"], ref["idx"]) and got["count"] == ref["count"]
        assert np.array_equal(got["out"], ref["out"])
        # causality: no candidate sees a later candidate's key
        sel = got["idx"][:got["count"]]
        assert sel.size == 0 or sel.max() <= int(ws.seq_lens[b]) - (T - t)


def test_mxfp8_and_fp8_latent_recipes():
    """MXFP8 keys: integer codes, E8M0 bytes in {125, 126, 127}, one per group;
    FP8 latent: exponent fields 4..10 (no NaN codes), tile scales in [0.02, 0.2)."""
    ws = W.make_decode(2, 0, 8, 64, 8, 16, seed=4, lengths=[40, 9], k_mx_group=32,
                       latent_fp8=True)
    k = ws.k_idx.float()
    assert torch.equal(k, k.round()) and k.abs().max() <= 3
    assert ws.k_scale.dtype == torch.uint8 and ws.k_scale.shape[-1] == 2
    assert int(ws.k_scale.min()) >= 125 and int(ws.k_scale.max()) <= 127
    raw = ws.latent.view(torch.uint8)
    ex = (raw >> 3) & 15
    assert int(ex.min()) >= 4 and int(ex.max()) <= 10
    assert ws.latent_scale.shape == ws.latent.shape[:-1] + (5,)
    assert float(ws.latent_scale.min()) >= 0.02 and float(ws.latent_scale.max()) < 0.2
    # the MXFP8 key scores of a row equal the unquantised scores of its dequantised keys
    b = 0
    kb = ws.k_idx[b, :40].float().numpy() * np.repeat(
        2.0 ** (ws.k_scale[b, :40].numpy().astype(np.int64) - 127), 32, axis=1)
    qd = oracle.mxfp8_dequantize(*oracle.mxfp8_quantize(ws.q_idx[b].float(), 32), 32)
    assert np.array_equal(oracle.row_scores(ws, b), oracle.index_scores(qd, ws.w[b], kb))
