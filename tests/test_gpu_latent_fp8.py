"""FP8 latent cache on the GPU (through the C ABI) against the CPU oracle: the
append kernel bit for bit, and the attention core over E4M3 latent rows with
one fp32 scale per tile of 128 dims (the rope dims a fifth tile)."""
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


def _latent_rows(n: int, ld: int, seed: int) -> torch.Tensor:
    """bf16 latent rows: normal values with per-row and per-tile magnitudes, one
    all-zero tile, one tile with a single large value."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((n, ld), generator=g)
    x *= torch.exp(torch.empty((n, 1)).uniform_(-4, 4, generator=g))
    x[:, :576] *= torch.exp(torch.empty((1, 576)).uniform_(-1, 1, generator=g))
    if n > 2:
        x[1, 128:256] = 0.0
        x[2, 300] = 3.0e4
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("n,ld", [(1000, 576), (37, 584), (3, 640)])
def test_append_bit_exact(n, ld):
    x = _latent_rows(n, ld, seed=n)
    codes, scales = binding.latent_fp8_append(x.to(DEV)[:, :576] if ld == 576 else x.to(DEV)[:, :576])
    torch.cuda.synchronize()
    ref_c, ref_s = oracle.latent_fp8_quantize(x[:, :576].float())
    got_c = _codes_f64(codes)
    assert np.array_equal(got_c, ref_c), f"codes differ at {np.argwhere(got_c != ref_c)[:5]}"
    assert np.array_equal(scales.cpu().numpy().astype(np.float64), ref_s)


def test_append_into_cache_rows():
    """dst_rows scatters each row into its cache row; -1 skips; other rows untouched."""
    n, P = 20, 64
    x = _latent_rows(n, 576, seed=5)
    perm = torch.randperm(P, generator=torch.Generator().manual_seed(2))[:n].to(torch.int64)
    perm[3] = -1
    codes = torch.full((P, 576), 0x11, dtype=torch.uint8, device=DEV).view(torch.float8_e4m3fn)
    scales = torch.full((P, 5), -1.0, dtype=torch.float32, device=DEV)
    binding.latent_fp8_append(x.to(DEV), dst_rows=perm.to(DEV), codes=codes, scales=scales)
    torch.cuda.synchronize()
    ref_c, ref_s = oracle.latent_fp8_quantize(x.float())
    got_c, got_s = _codes_f64(codes), scales.cpu().numpy()
    written = set()
    for i in range(n):
        r = int(perm[i])
        if r < 0:
            continue
        written.add(r)
        assert np.array_equal(got_c[r], ref_c[i]) and np.array_equal(got_s[r].astype(np.float64), ref_s[i])
    for r in range(P):
        if r not in written:
            assert np.all(codes[r].cpu().view(torch.uint8).numpy() == 0x11) and np.all(got_s[r] == -1.0)


CASES = {
    # name: (lengths, H_i, d, K, H, page size)
    "contig_h16": ([300, 77, 1], 4, 64, 32, 16, 0),
    "paged_h128": ([650, 64, 129], 64, 128, 128, 128, 64),
    "zero_length_h16": ([100, 0, 5], 4, 64, 16, 16, 0),
    "k_ge_history_h48": ([200, 31], 16, 64, 512, 48, 0),
    "single_seq_h16_cluster_merge8": ([900], 4, 64, 256, 16, 0),
    "single_seq_splitk_h128": ([5000], 64, 128, 2048, 128, 0),
    # 128 heads run on the tensor-core kernel (rows converted to bf16 as they land)
    "contig_h128_ragged": ([3000, 129, 64, 1, 700], 64, 128, 256, 128, 0),
    "zero_length_h128": ([0, 300, 2], 64, 128, 64, 128, 0),
    "paged128_h128": ([1000, 128, 300], 64, 128, 200, 128, 128),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_decode_layer_fp8_latent(name):
    lens, Hi, d, K, H, page = CASES[name]
    ws = W.make_decode(len(lens), 0, Hi, d, K, H, seed=zlib.crc32(name.encode()) % 1000,
                       lengths=lens, page_size=page, latent_fp8=True)
    g = ws.to(DEV)
    out, lse, idx, count = binding.layer(g)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    for b in range(ws.B):
        ref = oracle.decode_row(ws, b)
        assert np.array_equal(idx[b].cpu().numpy(), ref["idx"]), f"row {b}"
        if ref["count"] == 0:
            assert torch.all(out[b] == 0) and torch.all(torch.isinf(lse[b]))
            continue
        assert_out_close(out[b].float().cpu().numpy(), ref["out"], f"{name} row {b}")
        assert_lse_close(lse[b].cpu().numpy(), ref["lse"], f"{name} row {b}")


def test_prefill_fp8_latent():
    ws = W.make_prefill(40, 120, 4, 64, 16, 16, seed=3, q_offset=70, latent_fp8=True)
    g = ws.to(DEV)
    out, lse, idx, count = binding.layer(g)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    for t in (0, 1, 20, 39):
        ref = oracle.prefill_row(ws, t)
        assert np.array_equal(idx[t].cpu().numpy(), ref["idx"]), f"row {t}"
        assert_out_close(out[t].float().cpu().numpy(), ref["out"], f"prefill row {t}")
        assert_lse_close(lse[t].cpu().numpy(), ref["lse"], f"prefill row {t}")


def test_prefill_fp8_latent_h128():
    """Causal prefill with 128 heads over an FP8 latent cache: the fused
    prefill indexer, then the tensor-core attention kernel on FP8 rows."""
    ws = W.make_prefill(130, 333, 64, 128, 100, 128, seed=13, q_offset=203, latent_fp8=True)
    g = ws.to(DEV)
    out, lse, idx, count = binding.layer(g)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    for t in (0, 1, 64, 100, 129):
        ref = oracle.prefill_row(ws, t)
        assert np.array_equal(idx[t].cpu().numpy(), ref["idx"]), f"row {t}"
        assert_out_close(out[t].float().cpu().numpy(), ref["out"], f"prefill row {t}")
        assert_lse_close(lse[t].cpu().numpy(), ref["lse"], f"prefill row {t}")


@pytest.mark.parametrize("H,page", [(16, 64), (128, 64), (128, 0)])
def test_append_then_attend_matches_oracle_quantisation_heads(H, page):
    """bf16 rows quantised by the append kernel, attended by the CUDA-core (16
    heads) or tensor-core (128 heads) kernel; the oracle quantises the same
    rows itself."""
    Hi, d = (4, 64) if H == 16 else (64, 128)
    ws = W.make_decode(3, 0, Hi, d, 64, H, seed=19, lengths=[900, 70, 130], page_size=page)
    pool = ws.latent.reshape(-1, 576)
    g = ws.to(DEV)
    codes, scales = binding.latent_fp8_append(pool.to(DEV))
    g.latent = codes.view(ws.latent.shape)
    g.latent_scale = scales.view(ws.latent.shape[:-1] + (5,))
    out, lse, idx, count = binding.layer(g)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    rc, rs = oracle.latent_fp8_quantize(pool.float())
    wq = ws.to("cpu")
    wq.latent = torch.tensor(rc).to(torch.float8_e4m3fn).view(ws.latent.shape)
    wq.latent_scale = torch.tensor(rs, dtype=torch.float32).view(ws.latent.shape[:-1] + (5,))
    for b in range(ws.B):
        ref = oracle.decode_row(wq, b)
        assert np.array_equal(idx[b].cpu().numpy(), ref["idx"])
        assert_out_close(out[b].float().cpu().numpy(), ref["out"], f"row {b}")
        assert_lse_close(lse[b].cpu().numpy(), ref["lse"], f"row {b}")


def test_append_then_attend_matches_oracle_quantisation():
    """bf16 latent rows quantised into the cache by the append kernel, then the
    decode layer; the oracle quantises the same rows itself and attends."""
    ws = W.make_decode(2, 0, 4, 64, 32, 16, seed=9, lengths=[200, 70], page_size=64)
    pool = ws.latent.reshape(-1, 576)                       # bf16 rows of the page pool
    g = ws.to(DEV)
    codes, scales = binding.latent_fp8_append(pool.to(DEV))
    g.latent = codes.view(ws.latent.shape)
    g.latent_scale = scales.view(ws.latent.shape[:-1] + (5,))
    out, lse, idx, count = binding.layer(g)
    torch.cuda.synchronize()
    rc, rs = oracle.latent_fp8_quantize(pool.float())
    wq = ws.to("cpu")
    wq.latent = torch.tensor(rc).to(torch.float8_e4m3fn).view(ws.latent.shape)
    wq.latent_scale = torch.tensor(rs, dtype=torch.float32).view(ws.latent.shape[:-1] + (5,))
    for b in range(ws.B):
        ref = oracle.decode_row(wq, b)
        assert np.array_equal(idx[b].cpu().numpy(), ref["idx"])
        assert_out_close(out[b].float().cpu().numpy(), ref["out"], f"row {b}")
        assert_lse_close(lse[b].cpu().numpy(), ref["lse"], f"row {b}")
