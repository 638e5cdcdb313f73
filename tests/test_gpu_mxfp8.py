"""MXFP8 index path on the GPU (through the C ABI) against the CPU oracle: the
quantiser bit for bit, and scoring / the fused layer with MXFP8 key caches
(E4M3 codes, one E8M0 scale per group of 32, 64 or 128 elements)."""
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


def _codes_f64(codes: torch.Tensor) -> np.ndarray:
    return codes.cpu().view(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


QUANT_CASES = [
    # (rows, d, group, row pitch)
    (1000, 128, 32, 128),
    (37, 128, 64, 136),
    (9, 256, 128, 256),
    (8, 32, 32, 40),
    (3000, 64, 32, 64),
]


@pytest.mark.parametrize("case", QUANT_CASES, ids=[str(c) for c in QUANT_CASES])
def test_quantize_bit_exact(case):
    """Codes and scale bytes equal the oracle's, element for element, on normal
    rows with outliers and on the special rows (zeros, subnormals, huge values,
    powers of two, groups that saturate at 448)."""
    n, d, group, ld = case
    x_full = W.make_mx_input(n, ld, seed=n + d + group)
    x = x_full[:, :d]
    codes, scales = binding.mxfp8_quantize(x_full.to(DEV)[:, :d], group)
    torch.cuda.synchronize()
    ref_c, ref_X = oracle.mxfp8_quantize(x.float(), group)
    got_c = _codes_f64(codes)
    assert np.array_equal(got_c, ref_c), f"codes differ at {np.argwhere(got_c != ref_c)[:5]}"
    assert np.array_equal(scales.cpu().numpy().astype(np.int64), ref_X + 127)


def test_quantize_appends_into_cache_rows():
    """dst_rows scatters each row into its cache row; -1 skips; other rows untouched."""
    n, d, P = 40, 128, 100
    x = W.make_mx_input(n, d, seed=5)
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(1))[:n].to(torch.int64)
    perm[7] = -1
    codes = torch.full((P, d), 0x7E, dtype=torch.uint8, device=DEV).view(torch.float8_e4m3fn)
    scales = torch.full((P, d // 32), 0xAB, dtype=torch.uint8, device=DEV)
    binding.mxfp8_quantize(x.to(DEV), 32, dst_rows=perm.to(DEV), codes=codes, scales=scales)
    torch.cuda.synchronize()
    ref_c, ref_X = oracle.mxfp8_quantize(x.float(), 32)
    got_c, got_s = _codes_f64(codes), scales.cpu().numpy()
    written = set()
    for i in range(n):
        r = int(perm[i])
        if r < 0:
            continue
        written.add(r)
        assert np.array_equal(got_c[r], ref_c[i]) and np.array_equal(got_s[r], ref_X[i] + 127)
    for r in range(P):
        if r not in written:
            assert np.all(codes[r].cpu().view(torch.uint8).numpy() == 0x7E) and np.all(got_s[r] == 0xAB)


MX_CASES = {
    # name: (lengths, tokens per sequence, K, H, page size, group)
    "contig_g32": ([700, 132, 64, 1000], 1, 64, 128, 0, 32),
    "contig_ragged_tiles_g64": ([4104, 128, 2052], 1, 256, 128, 0, 64),
    "paged_g32": ([1100, 300, 65, 2], 1, 128, 128, 64, 32),
    "paged_g128_page128": ([1000, 128, 301], 1, 200, 128, 128, 128),
    "zero_length_g32": ([100, 0, 8], 1, 16, 128, 0, 32),
    "multi_t2_g32": ([300, 64, 132], 2, 64, 128, 0, 32),
    "multi_t4_paged_g64": ([1000, 200], 4, 128, 128, 64, 64),
    # sequences of one key tile: query slots turn over every tile
    "one_tile_seqs_g32": ([128, 1, 64, 127, 128, 30, 128, 128, 9, 100, 128, 64, 2, 128, 128, 77],
                          1, 16, 128, 0, 32),
    "one_tile_seqs_paged_g64": ([64, 128, 1, 128, 128, 30, 100, 128, 128, 5, 128, 64], 1, 16,
                                128, 64, 64),
    # candidate pairs (two issuers on alternate tiles, two accumulators) over
    # paged keys, with sequences of one tile among longer ones
    "multi_t2_paged_g32_one_tile_seqs": ([700, 128, 64, 129, 3, 128, 1000, 66], 2, 64, 128, 64, 32),
}


def _mx_decode(name):
    lengths, T, K, H, page, group = MX_CASES[name]
    return W.make_decode(len(lengths), 0, 64, 128, K, H, seed=zlib.crc32(name.encode()) % 1000,
                         lengths=lengths, page_size=page, tokens_per_seq=T, k_mx_group=group)


@pytest.mark.parametrize("name", sorted(MX_CASES))
def test_mx_decode_layer(name):
    """Integer-valued index queries and codes with scales 2^-2..2^0: the MXFP8
    scores are exact in fp32, so scores and selections match the oracle exactly;
    the attention core then runs on the oracle's selections' rows."""
    ws = _mx_decode(name)
    T = ws.tokens_per_seq
    g = ws.to(DEV)
    cache = binding.Cache.of(g)
    assert cache.struct.k_dtype == binding.DSI_MXFP8_E4M3
    if T == 1:
        scores = binding.index_score(g.q_idx, g.w, cache, True)
        torch.cuda.synchronize()
        sc = scores.cpu().numpy()
        for r in range(ws.T):
            ref = oracle.row_scores(ws, r).astype(np.float32)
            assert np.array_equal(sc[r, :ref.shape[0]], ref), f"scores differ in row {r}"
        out, lse, idx, count = binding.layer(g)
    else:
        out, lse, idx, count = binding.indexed_attention_multi(g.q_idx, g.w, g.q, cache, T,
                                                               ws.K, ws.scale)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    for r in range(ws.T):
        ref = oracle.multi_token_row(ws, r, T) if T > 1 else oracle.decode_row(ws, r)
        assert np.array_equal(idx[r].cpu().numpy(), ref["idx"]), f"row {r}"
        assert int(count[r]) == ref["count"]
        if ref["count"] == 0:
            continue
        assert_out_close(out[r].float().cpu().numpy(), ref["out"], f"{name} row {r}")
        assert_lse_close(lse[r].cpu().numpy(), ref["lse"], f"{name} row {r}")


@pytest.mark.parametrize("group", [32, 128])
def test_mx_prefill_scores_and_layer(group):
    """Causal prefill with MXFP8 keys (groups of 4 query tokens per tile pass),
    with an offset so that rows start mid-cache."""
    ws = W.make_prefill(70, 608, 64, 128, 64, 16, seed=group, q_offset=500, k_mx_group=group)
    g = ws.to(DEV)
    cache = binding.Cache.of(g)
    scores = binding.index_score(g.q_idx, g.w, cache, False, ws.q_offset)
    torch.cuda.synchronize()
    sc = scores.cpu().numpy()
    for t in range(ws.T):
        ref = oracle.row_scores(ws, t).astype(np.float32)
        assert np.array_equal(sc[t, :ref.shape[0]], ref), f"scores differ in row {t}"
    out, lse, idx, count = binding.layer(g)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    for t in (0, 1, 33, 69):
        ref = oracle.prefill_row(ws, t)
        assert np.array_equal(idx[t].cpu().numpy(), ref["idx"]), f"row {t}"
        assert_out_close(out[t].float().cpu().numpy(), ref["out"], f"prefill row {t}")


def test_mx_nonint_queries_subnormal_codes_and_large_scales():
    """Non-integer index queries (quantised in the kernel, rounding decisions
    identical to the oracle's), E4M3 subnormal key codes and scales above 2^7
    (the second rescaling multiply): scores within fp32 summation noise."""
    ws = W.make_decode(2, 0, 64, 128, 32, 16, seed=41, lengths=[500, 76], page_size=64,
                       k_mx_group=32)
    gen = torch.Generator().manual_seed(9)
    ws.q_idx = (torch.randn(ws.q_idx.shape, generator=gen) * 3).to(torch.bfloat16)
    raw = ws.k_idx.view(torch.uint8)
    sub = torch.randint(1, 8, raw.shape, generator=gen, dtype=torch.uint8)      # 1..7: subnormal codes
    pick = torch.rand(raw.shape, generator=gen) < 0.25
    raw[pick] = sub[pick] | (torch.rand(raw.shape, generator=gen)[pick] < 0.5).to(torch.uint8) * 0x80
    big = torch.rand(ws.k_scale.shape, generator=gen) < 0.3
    ws.k_scale[big] = torch.randint(130, 140, ws.k_scale.shape, generator=gen,
                                    dtype=torch.int64)[big].to(torch.uint8)
    g = ws.to(DEV)
    scores = binding.index_score(g.q_idx, g.w, binding.Cache.of(g), True)
    torch.cuda.synchronize()
    for b in range(ws.B):
        n = int(ws.seq_lens[b])
        ref = oracle.row_scores(ws, b)
        got = scores[b, :n].cpu().numpy().astype(np.float64)
        assert np.allclose(got, ref, rtol=1e-5, atol=1e-5 * np.abs(ref).max()), b


def test_mx_append_then_score_matches_oracle_quantisation():
    """bf16 keys appended into a paged MXFP8 cache by the quantiser, then scored;
    the oracle quantises the same bf16 keys itself and scores them."""
    B, L, page = 2, 300, 64
    npg = (L + page - 1) // page
    keys = W.make_mx_input(B * L, 128, seed=77)[:, :]
    keys[:8] = keys[8:16]                        # ordinary rows only (no special rows)
    ws = W.make_decode(B, L, 64, 128, 32, 16, seed=78, page_size=page, k_mx_group=32)
    gen = torch.Generator().manual_seed(2)
    ws.q_idx = torch.randn(ws.q_idx.shape, generator=gen).to(torch.bfloat16)
    # slot mapping: position p of sequence b -> its physical cache row
    bt = ws.block_table
    dst = torch.tensor([int(bt[b, p // page]) * page + p % page for b in range(B) for p in range(L)],
                       dtype=torch.int64)
    g = ws.to(DEV)
    binding.mxfp8_quantize(keys.to(DEV), 32, dst_rows=dst.to(DEV), codes=g.k_idx, scales=g.k_scale)
    scores = binding.index_score(g.q_idx, g.w, binding.Cache.of(g), True)
    torch.cuda.synchronize()
    assert npg * B <= ws.k_idx.shape[0]
    for b in range(B):
        kb = keys[b * L:(b + 1) * L].float()
        codes, X = oracle.mxfp8_quantize(kb, 32)
        ref = oracle.index_scores(ws.q_idx[b], ws.w[b], codes, (X + 127).astype(np.uint8))
        got = scores[b, :L].cpu().numpy().astype(np.float64)
        assert np.allclose(got, ref, rtol=1e-5, atol=1e-5 * np.abs(ref).max()), b


def test_mx_contiguous_needs_aligned_s_max():
    """A contiguous MXFP8 cache whose rows per sequence do not start a 16-byte
    row of scales (s_max a multiple of 4 for groups of 32) is refused on the
    host (nothing launched)."""
    ws = W.make_decode(2, 0, 64, 128, 16, 16, seed=3, lengths=[10, 9], k_mx_group=32)
    g = ws.to(DEV)
    with pytest.raises(binding.DsiError) as e:
        binding.index_score(g.q_idx, g.w, binding.Cache.of(g), True)
    assert e.value.status == binding.DSI_ERR_UNSUPPORTED
