"""CUDA path (through the C ABI) against the CPU oracle on seeded inputs at
sizes the oracle finishes in seconds: several tiles, ragged tails, paged and
FP8 caches, prefill with offsets, and the degenerate cases."""
import math
import zlib

import numpy as np
import pytest
import torch

import oracle
from indexed_sparse_attention_indexer_gb300 import binding
from indexed_sparse_attention_indexer_gb300 import workloads as W
from tests.parity import assert_lse_close, assert_out_close

pytestmark = pytest.mark.gpu

DEV = "cuda"

DECODE_CASES = {
    # name: (B, lengths, H_i, d, K, H, page, fp8, extra)
    "small_heads_d64": (3, [300, 77, 1], 4, 64, 32, 16, 0, False, {}),
    "small_heads_d128": (2, [513, 1000], 2, 128, 100, 16, 0, False, {}),
    "hi64_d128_h128": (4, [700, 129, 64, 1000], 64, 128, 64, 128, 0, False, {}),
    "hi64_ragged_tiles": (3, [4097, 127, 2049], 64, 128, 256, 128, 0, False, {}),
    "paged_bf16": (3, [650, 64, 1], 64, 128, 128, 128, 64, False, {}),
    "paged_fp8": (4, [1100, 300, 65, 2], 64, 128, 128, 128, 64, True, {}),
    "paged_fp8_small_heads": (2, [333, 90], 4, 64, 40, 16, 16, True, {}),
    "k_ge_history": (2, [200, 31], 4, 64, 512, 16, 0, False, {}),
    # a single row splits its selection eight ways, merged inside one cluster
    "single_seq_h16_cluster_merge8": (1, [900], 4, 64, 256, 16, 0, False, {}),
    # four-way clusters per head group; the short row's later splits hold no index
    "h48_cluster_merge4": (2, [400, 60], 4, 64, 128, 48, 0, False, {}),
    "heads_8": (2, [100, 257], 4, 64, 16, 8, 0, False, {}),
    "heads_48_hi16": (2, [300, 90], 16, 64, 50, 48, 0, False, {}),
    "softmax_stress": (2, [400, 150], 4, 64, 64, 16, 0, False, {"q_std": 1.0, "scale": 1.0}),
    "hi64_fp8_contiguous": (3, [900, 129, 2], 64, 128, 100, 128, 0, True, {}),
    # s_max not a multiple of 4: the key scales are copied lane by lane
    "hi64_fp8_contiguous_odd_s_max": (2, [901, 37], 64, 128, 64, 128, 0, True, {}),
    "hi64_paged_page128": (3, [1000, 128, 300], 64, 128, 200, 128, 128, False, {}),
    "hi64_paged_page16_generic": (2, [333, 40], 64, 128, 64, 128, 16, False, {}),
    "zero_length_sequence": (3, [100, 0, 5], 64, 128, 16, 128, 0, False, {}),
    "zero_length_paged_fp8": (3, [0, 70, 200], 64, 128, 16, 128, 64, True, {}),
    "softmax_stress_h128": (2, [3000, 700], 4, 64, 2048, 128, 0, False,
                            {"q_std": 1.0, "scale": 1.0}),
    "k100_h128": (3, [900, 50, 101], 4, 64, 100, 128, 0, False, {}),
    "single_seq_h128_splitk": (1, [5000], 64, 128, 2048, 128, 0, False, {}),
    # runs of sequences of one key tile (groups of a single tile): the query
    # slots turn over as fast as the tiles arrive
    "hi64_many_one_tile_seqs": (24, [1, 128, 77, 64, 3, 128, 90, 129, 100, 5, 128, 60,
                                     33, 128, 2, 127, 128, 700, 41, 128, 9, 64, 128, 16],
                                64, 128, 16, 128, 0, False, {}),
    # more rows than the attention core's cluster slots (a second wave of
    # clusters), with zero-length and one-tile sequences
    "hi64_many_rows_paged": (96, [90, 1179, 952, 64, 1193, 0, 1297, 502, 1452, 478, 537, 585,
                                  490, 1202, 281, 137, 1366, 0, 316, 1187, 1094, 1138, 1108, 906,
                                  1456, 196, 1158, 540, 1012, 1306, 64, 1467, 307, 1061, 214,
                                  242, 62, 1317, 276, 243, 0, 0, 389, 530, 498, 582, 957, 174,
                                  823, 279, 825, 1132, 511, 114, 1446, 589, 687, 5, 1495, 692,
                                  64, 131, 558, 52, 1035, 1218, 504, 310, 80, 1216, 1406, 403,
                                  652, 1200, 622, 663, 1245, 1006, 1079, 1461, 1215, 311, 962,
                                  947, 161, 125, 1114, 698, 0, 242, 991, 1149, 26, 161, 468, 667],
                             64, 128, 192, 128, 64, False, {}),
    "hi64_many_one_tile_seqs_paged_fp8": (20, [64, 128, 7, 100, 128, 1, 65, 128, 30, 128,
                                               300, 12, 128, 128, 99, 2, 128, 64, 50, 128],
                                          64, 128, 16, 128, 64, True, {}),
}


def _decode(name):
    B, lens, Hi, d, K, H, page, fp8, extra = DECODE_CASES[name]
    return W.make_decode(B, max(lens), Hi, d, K, H, seed=zlib.crc32(name.encode()) % 1000, lengths=lens,
                         page_size=page, k_fp8=fp8, **extra)


def _check_scores(ws, g, cache):
    decode = ws.mode == "decode"
    scores = binding.index_score(g.q_idx, g.w, cache, decode, ws.q_offset)
    torch.cuda.synchronize()
    sc = scores.cpu().numpy()
    for r in range(ws.T):
        ref = oracle.row_scores(ws, r).astype(np.float32)
        n = ref.shape[0]
        assert np.array_equal(sc[r, :n], ref), f"scores differ in row {r}"
    return scores


@pytest.mark.parametrize("name", sorted(DECODE_CASES))
def test_decode_entry_points(name):
    ws = _decode(name)
    g = ws.to(DEV)
    cache = binding.Cache.of(g)
    scores = _check_scores(ws, g, cache)
    idx, count = binding.topk(scores, ws.K, row_len=g.seq_lens)
    ref = oracle.layer(ws)
    idx_h, cnt_h = idx.cpu().numpy(), count.cpu().numpy()
    for b in range(ws.B):
        assert np.array_equal(idx_h[b], ref[b]["idx"]), f"indices differ, row {b}"
        assert cnt_h[b] == ref[b]["count"]
    # attention core on the oracle's own indices
    ref_idx = torch.tensor(np.stack([ref[b]["idx"] for b in range(ws.B)]), dtype=torch.int32,
                           device=DEV)
    out, lse = binding.sparse_mla_decode(g.q, cache, ref_idx, ws.scale)
    torch.cuda.synchronize()
    assert_out_close(out.float().cpu().numpy(), np.stack([ref[b]["out"] for b in range(ws.B)]), name)
    assert_lse_close(lse.cpu().numpy(), np.stack([ref[b]["lse"] for b in range(ws.B)]), name)
    assert binding.device_status() == 0


@pytest.mark.parametrize("name", sorted(DECODE_CASES))
def test_decode_fused(name):
    ws = _decode(name)
    g = ws.to(DEV)
    out, lse, idx, count = binding.layer(g)
    torch.cuda.synchronize()
    ref = oracle.layer(ws)
    for b in range(ws.B):
        assert np.array_equal(idx[b].cpu().numpy(), ref[b]["idx"]), f"row {b}"
        assert int(count[b]) == ref[b]["count"]
    assert_out_close(out.float().cpu().numpy(), np.stack([ref[b]["out"] for b in range(ws.B)]), name)
    assert_lse_close(lse.cpu().numpy(), np.stack([ref[b]["lse"] for b in range(ws.B)]), name)
    assert binding.device_status() == 0


PREFILL_CASES = {
    # name: (T, S, q_offset, H_i, d, K, H)
    "from_start_small_heads": (130, 130, 0, 4, 64, 32, 16),
    "offset_hi64": (200, 400, 150, 64, 128, 64, 128),
    "from_start_hi64": (300, 300, 0, 64, 128, 128, 128),
    "k_ge_history": (70, 100, 20, 4, 64, 128, 16),
    "ragged_groups_hi64": (130, 333, 203, 64, 128, 100, 128),   # T not a multiple of 4
    "single_token_hi64": (1, 50, 49, 64, 128, 8, 128),
}


@pytest.mark.parametrize("name", sorted(PREFILL_CASES))
def test_prefill(name):
    T, S, off, Hi, d, K, H = PREFILL_CASES[name]
    ws = W.make_prefill(T, S, Hi, d, K, H, seed=5, q_offset=off)
    g = ws.to(DEV)
    cache = binding.Cache.of(g)
    scores = _check_scores(ws, g, cache)
    idx, count = binding.topk(scores, K, q_offset=off)
    ref = oracle.layer(ws)
    idx_h = idx.cpu().numpy()
    for t in range(T):
        assert np.array_equal(idx_h[t], ref[t]["idx"]), f"row {t}"
        sel = idx_h[t][idx_h[t] >= 0]
        assert sel.max() <= off + t          # causality
    ref_idx = torch.tensor(np.stack([ref[t]["idx"] for t in range(T)]), dtype=torch.int32,
                           device=DEV)
    out, lse = binding.sparse_mla_prefill(g.q, cache, ref_idx, off, ws.scale)
    ref_out = np.stack([ref[t]["out"] for t in range(T)])
    assert_out_close(out.float().cpu().numpy(), ref_out, name)
    out2, lse2, idx2, _ = binding.layer(g)
    torch.cuda.synchronize()
    assert np.array_equal(idx2.cpu().numpy(), idx_h)
    assert_out_close(out2.float().cpu().numpy(), ref_out, name + " fused")
    assert_lse_close(lse2.cpu().numpy(), np.stack([ref[t]["lse"] for t in range(T)]), name)
    assert binding.device_status() == 0


def test_prefill_attention_on_given_indices():
    """The attention core over index sets it is handed, with several rows per
    cluster slot (each cluster takes rows in turn): rows with no valid entry,
    a first tile of skipped entries, a single entry in the last tile, and
    entries past the row's history (skipped), against the oracle's attention
    over the valid rows."""
    T, S, off, K, H = 400, 820, 400, 192, 128
    ws = W.make_prefill(T, S, 4, 64, K, H, seed=31, q_offset=off)
    rng = np.random.default_rng(31)
    idx = np.full((T, K), -1, dtype=np.int32)
    for t in range(T):
        n_vis = off + t + 1
        kind = t % 5
        if kind == 1:
            idx[t] = rng.choice(n_vis, K, replace=False)
        elif kind == 2:
            idx[t, 64:] = rng.choice(n_vis, K - 64, replace=False)
        elif kind == 3:
            idx[t, K - 1] = rng.integers(0, n_vis)
        elif kind == 4:
            idx[t] = rng.choice(n_vis, K, replace=False)
            bad = rng.choice(K, 20, replace=False)
            idx[t, bad] = rng.integers(n_vis, S + 50, 20)   # past the history
    g = ws.to(DEV)
    cache = binding.Cache.of(g)
    out, lse = binding.sparse_mla_prefill(g.q, cache, torch.tensor(idx, device=DEV), off,
                                          ws.scale)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    lat = ws.latent[0].float().numpy()
    q = ws.q.float().numpy()
    ref_o = np.zeros((T, H, W.D_LATENT))
    ref_l = np.zeros((T, H))
    for t in range(T):
        v = idx[t][(idx[t] >= 0) & (idx[t] < off + t + 1)]
        ref_o[t], ref_l[t] = oracle.sparse_mla(q[t], lat[v], ws.scale)
    assert_out_close(out.float().cpu().numpy(), ref_o, "given indices")
    assert_lse_close(lse.cpu().numpy(), ref_l, "given indices")


FUSED_PREFILL_CASES = [
    # T, S, q_offset, K: rows longer than the 4096-entry candidate buffer force
    # compactions; odd T leaves a half-empty last group
    (300, 6000, 5700, 2048),
    (257, 5000, 0, 100),
    (64, 9000, 8936, 1),
    (33, 4200, 4000, 2048),
    # rows with at most K positions of history take all of them unscored:
    # every row, from the start and after an offset, and the first 98 of 200
    (40, 40, 0, 64),
    (64, 1000, 900, 2048),
    (200, 2150, 1950, 2048),
]


@pytest.mark.parametrize("case", FUSED_PREFILL_CASES, ids=[str(c) for c in FUSED_PREFILL_CASES])
def test_fused_prefill_topk_matches_unfused(case):
    """The fused prefill indexer (scores never leave the chip) selects exactly what
    scoring + select in two kernels selects, and what the oracle selects."""
    T, S, off, K = case
    ws = W.make_prefill(T, S, 64, 128, K, 16, seed=11, q_offset=off)
    g = ws.to(DEV)
    out, lse, idx, count = binding.layer(g)
    scores = binding.index_score(g.q_idx, g.w, binding.Cache.of(g), False, off)
    idx2, cnt2 = binding.topk(scores, K, q_offset=off)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    assert torch.equal(idx, idx2)
    assert torch.equal(count, cnt2)
    # the fused indexer through its own entry point
    idx3, cnt3 = binding.index_topk_prefill(g.q_idx, g.w, binding.Cache.of(g), K, off)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    assert torch.equal(idx3, idx2)
    assert torch.equal(cnt3, cnt2)
    for t in (0, T // 2, T - 1):
        ref = oracle.prefill_row(ws, t)
        assert np.array_equal(idx[t].cpu().numpy(), ref["idx"]), f"row {t}"


def test_prefill_chunk_invariance():
    """A prefill split into query chunks gives the same indices (and outputs) as one call."""
    T, S, Hi, d, K, H = 256, 256, 64, 128, 64, 128
    ws = W.make_prefill(T, S, Hi, d, K, H, seed=9)
    g = ws.to(DEV)
    out, _, idx, _ = binding.layer(g)
    for c0 in (0, 96, 200):
        c1 = min(T, c0 + 96)
        sub = g.to(DEV)
        sub.q_idx, sub.w, sub.q, sub.q_offset = g.q_idx[c0:c1], g.w[c0:c1], g.q[c0:c1], c0
        o2, _, i2, _ = binding.layer(sub)
        torch.cuda.synchronize()
        assert torch.equal(i2, idx[c0:c1])
        d = (o2.float() - out[c0:c1].float()).abs().max().item()
        assert d <= 1e-2 * out.float().abs().max().item()


TOPK_CASES = [
    # rows, ld, K, value levels (ties), with -inf, staged in shared memory?
    (5, 1000, 7, 4, False),
    (3, 5000, 2048, 16, True),
    (2, 50000, 2048, 1000, True),     # longer than the shared-memory stage
    (4, 33000, 1, 3, False),
    (3, 600, 600, 5, False),          # K == n
    (2, 70000, 4096, 1 << 20, False),
    (3, 32768, 2048, 1 << 20, True),  # the register-resident kernel at its largest rows
    (2, 32767, 2048, 7, False),       # odd row stride (unaligned rows, scalar loads)
    (2, 32769, 100, 50, False),       # one past the register-resident rows: two chunks
    (2, 131072, 2048, 1 << 16, True), # four chunks, the longest rows the chunked kernel takes
    (1, 140000, 512, 100, False),     # beyond: the 8-bit radix kernel, re-reading from L2
    (160, 4000, 256, 9, True),        # enough rows for one CTA each (no cluster)
    (320, 40000, 512, 1 << 12, False),  # enough long rows for one CTA each: chunked reloads
    (9, 2048, 128, 3, True),          # short rows, heavy ties
    (7, 1999, 1, 1 << 20, False),     # short rows, K = 1, odd row stride
    (6, 2048, 2000, 50, True),        # short rows, K near n
    (3, 16384, 2048, 50, True),       # the largest row one CTA of a two-CTA cluster takes alone
    (3, 16385, 2048, 50, False),      # one past it: both CTAs share the row (9 keys a thread)
]


@pytest.mark.parametrize("case", TOPK_CASES, ids=[str(c) for c in TOPK_CASES])
def test_topk_ties_and_lengths(case):
    rows, ld, K, levels, with_inf = case
    gen = torch.Generator().manual_seed(rows * 1000 + K)
    sc = torch.randint(0, levels, (rows, ld), generator=gen).float() / 8 - levels / 16
    if with_inf:
        sc[:, ::7] = -math.inf
    lens = torch.randint(1, ld + 1, (rows,), generator=gen).to(torch.int32)
    lens[0] = ld
    g = sc.to(DEV)
    idx, count = binding.topk(g, K, row_len=lens.to(DEV))
    torch.cuda.synchronize()
    for r in range(rows):
        n = int(lens[r])
        exp, cnt = oracle.topk_select(sc[r, :n].numpy(), K)
        assert np.array_equal(idx[r].cpu().numpy(), exp), f"row {r}"
        assert int(count[r]) == cnt


MULTI_CASES = {
    # name: (lengths, T, H_i, d, K, H, page_size, fp8)
    "contig_hi64_t2": ([300, 64, 130], 2, 64, 128, 64, 128, 0, False),
    "paged_fp8_t4": ([1000, 200], 4, 64, 128, 128, 128, 64, True),
    "small_heads_t3": ([50, 7, 90], 3, 4, 64, 16, 16, 0, False),
    "shorter_than_t": ([1, 40], 2, 64, 128, 8, 128, 0, False),   # candidate 0 of seq 0 sees nothing
    # sequences of one key tile among longer ones: the query slots turn over
    # at every tile for the groups of four candidates
    "one_tile_seqs_t4_paged_fp8": ([128, 64, 700, 2, 128, 129, 30, 128], 4, 64, 128, 32, 128, 64,
                                   True),
    # 90 candidate rows: more than the attention core's cluster slots
    "many_rows_t2": ([242, 63, 330, 424, 223, 798, 890, 692, 144, 426, 705, 829, 207, 440, 4,
                       232, 172, 127, 451, 735, 542, 135, 707, 583, 801, 776, 874, 233, 460, 676,
                       562, 105, 619, 33, 832, 608, 333, 388, 897, 856, 480, 842, 42, 681, 736],
                     2, 64, 128, 128, 128, 0, False),
}


@pytest.mark.parametrize("name", sorted(MULTI_CASES))
def test_multi_token_decode(name):
    """Speculative verification: T candidate rows per sequence, each causal over the
    history and the earlier candidates, through dsi_indexed_attention_multi."""
    lengths, T, Hi, d, K, H, page, fp8 = MULTI_CASES[name]
    ws = W.make_decode(len(lengths), 0, Hi, d, K, H, seed=23, lengths=lengths, page_size=page,
                       k_fp8=fp8, tokens_per_seq=T)
    g = ws.to(DEV)
    out, lse, idx, count = binding.indexed_attention_multi(g.q_idx, g.w, g.q, binding.Cache.of(g),
                                                           T, K, ws.scale)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    for r in range(ws.T):
        ref = oracle.multi_token_row(ws, r, T)
        assert np.array_equal(idx[r].cpu().numpy(), ref["idx"]), f"row {r}"
        assert int(count[r]) == ref["count"]
        if ref["count"] == 0:
            assert torch.all(out[r] == 0) and torch.all(torch.isinf(lse[r]))
            continue
        assert_out_close(out[r].float().cpu().numpy(), ref["out"], f"{name} row {r}")
        assert_lse_close(lse[r].cpu().numpy(), ref["lse"], f"{name} row {r}")


def test_topk_wide_key_range_and_constant_rows():
    """Scores spread over many binades (and signs), plus rows that are constant or
    hold one distinct value above a constant floor."""
    rows, ld, K = 4, 32768, 2048
    gen = torch.Generator().manual_seed(11)
    mag = torch.exp2(torch.rand((rows, ld), generator=gen) * 120 - 60)
    sign = torch.where(torch.rand((rows, ld), generator=gen) < 0.3, -1.0, 1.0)
    sc = mag * sign
    sc[2] = 1.5
    sc[3] = -2.0
    sc[3, 12345] = 7.0
    g = sc.to(DEV)
    idx, count = binding.topk(g, K, row_len=torch.full((rows,), ld, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    for r in range(rows):
        exp, cnt = oracle.topk_select(sc[r].numpy(), K)
        assert np.array_equal(idx[r].cpu().numpy(), exp), f"row {r}"
        assert int(count[r]) == cnt


def test_topk_negative_zero_ties_positive_zero():
    sc = torch.zeros((1, 64))
    sc[0, ::2] = -0.0
    g = sc.to(DEV)
    idx, _ = binding.topk(g, 5, row_len=torch.tensor([64], dtype=torch.int32, device=DEV))
    assert idx[0].tolist() == [0, 1, 2, 3, 4]


@pytest.mark.parametrize("heads,d", [(64, 128), (4, 64)])
def test_fp8_keys_round_queries_to_e4m3(heads, d):
    """Non-integer index queries with FP8 keys: both sides score with E4M3 queries."""
    ws = W.make_decode(2, 0, heads, d, 32, 16, seed=31, lengths=[500, 77], page_size=64,
                       k_fp8=True)
    gen = torch.Generator().manual_seed(3)
    ws.q_idx = (torch.randn(ws.q_idx.shape, generator=gen) * 2).to(torch.bfloat16)
    g = ws.to(DEV)
    scores = binding.index_score(g.q_idx, g.w, binding.Cache.of(g), True)
    torch.cuda.synchronize()
    for b in range(ws.B):
        n = int(ws.seq_lens[b])
        ref = oracle.row_scores(ws, b)
        got = scores[b, :n].cpu().numpy().astype(np.float64)
        # products are no longer small integers: compare within fp32 summation noise
        assert np.allclose(got, ref, rtol=1e-5, atol=1e-4 * np.abs(ref).max())


def test_zeroed_head_weight_matches_removed_head():
    ws = _decode("hi64_d128_h128")
    g = ws.to(DEV)
    w0 = g.w.clone()
    w0[:, 5] = 0
    s0 = binding.index_score(g.q_idx, w0, binding.Cache.of(g), True)
    keep = [h for h in range(64) if h != 5]
    s1 = binding.index_score(g.q_idx[:, keep].contiguous(), g.w[:, keep].contiguous(),
                             binding.Cache.of(g), True)
    torch.cuda.synchronize()
    for b in range(ws.B):
        n = int(ws.seq_lens[b])
        assert torch.equal(s0[b, :n], s1[b, :n])


def test_checked_build_flags_out_of_range_index():
    """With the bounds-checked library an index >= seq_len is skipped and reported."""
    ws = _decode("small_heads_d64")
    g = ws.to(DEV)
    idx = torch.zeros((ws.B, 4), dtype=torch.int32, device=DEV)
    idx[1, 2] = int(ws.seq_lens[1]) + 5     # beyond the history, inside the allocation
    binding.sparse_mla_decode(g.q, binding.Cache.of(g), idx, ws.scale, checked=True)
    assert binding.device_status(checked=True) == binding.DSI_ERR_BOUNDS
    assert binding.device_status(checked=True) == 0   # read clears it


@pytest.mark.parametrize("H,paged", [(16, 0), (128, 0), (128, 64)])
def test_indices_past_the_history_are_skipped_in_every_build(H, paged):
    """Entries beyond a row's visible history (here up to 2^30, far outside the
    cache) take no part in the attention in the release build either: the
    result equals the same call with those entries set to -1, and no row
    outside the cache is read."""
    Hi, d = (4, 64) if H == 16 else (64, 128)
    ws = W.make_decode(3, 0, Hi, d, 64, H, seed=37, lengths=[300, 90, 200], page_size=paged)
    g = ws.to(DEV)
    cache = binding.Cache.of(g)
    gen = torch.Generator().manual_seed(3)
    good = torch.stack([torch.randperm(int(L), generator=gen)[:64].sort().values
                        for L in ws.seq_lens]).to(torch.int32)
    bad = good.clone()
    bad[0, 5], bad[1, 0], bad[2, 63] = 300, 1 << 30, 5000     # past each row's history
    clean = good.clone()
    clean[0, 5], clean[1, 0], clean[2, 63] = -1, -1, -1
    ref, ref_lse = binding.sparse_mla_decode(g.q, cache, clean.to(DEV), ws.scale)
    out, lse = binding.sparse_mla_decode(g.q, cache, bad.to(DEV), ws.scale)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    assert torch.equal(out, ref) and torch.equal(lse, ref_lse)


@pytest.mark.parametrize("Hi,d,H", [(64, 128, 128), (4, 64, 16)])
def test_decode_length_above_s_max_is_clamped(Hi, d, H):
    """A seq_lens entry above a contiguous cache's s_max (here 100, not a
    multiple of 64) counts as s_max in every kernel: scoring, Top-K (whose
    score rows are 128 wide) and attention see the same clamped history, and
    the result equals the oracle on that history."""
    ws = W.make_decode(3, 100, Hi, d, 32, H, seed=31, lengths=[100, 77, 100])
    g = ws.to(DEV)
    g.seq_lens = torch.tensor([130, 77, 5000], dtype=torch.int32, device=DEV)
    cache = binding.Cache.of(g)
    for _ in range(2):     # the second call runs over the first call's workspace
        out, lse, idx, count = binding.indexed_attention(g.q_idx, g.w, g.q, cache, ws.K, ws.scale,
                                                         True)
        torch.cuda.synchronize()
        ref = oracle.layer(ws)     # ws keeps the clamped lengths [100, 77, 100]
        for b in range(ws.B):
            assert np.array_equal(idx[b].cpu().numpy(), ref[b]["idx"]), f"row {b}"
            assert int(count[b]) == ref[b]["count"]
            assert int(idx[b].max()) < 100
        assert_out_close(out.float().cpu().numpy(), np.stack([ref[b]["out"] for b in range(ws.B)]),
                         "clamped")
    assert binding.device_status() == 0
