"""Oracle for the indexed sparse attention layer — TEST INFRASTRUCTURE ONLY.

A plain, slow CPU restatement in fp64 of what the layer computes.  Only the
tests, the package's ``smoke()`` check and the bench's CPU-baseline leg may
import it; the library never does, and it shares no code, tables or helpers
with the CUDA path (inputs come from the seeded generators in the package's
``workloads`` module, which hold none of the arithmetic).

Sources (page titles, sections):
* "Day 0 Inference Support for New LLM Architectures: Optimization Practices"
  — "Index-Based Sparse Attention": an indexer scores history positions,
  applies head-weight weighting and keeps the Top-K; the attention core reads
  the KV entries at those indices.  "Internal Fusion of the Indexer": the three
  steps are scoring, weighted sum over heads, top-k, read from a paged K cache.
* "Day 0 Inference Acceleration for New LLM Architectures..." §2–§3: relevance
  scoring, head weight summation, Top-K selection; only the index sequence is
  passed to the attention kernel, which reads the key-values at those indices.
* "Day 0 Inference Adaptation and Performance Optimization for New Models" §1:
  index selection sits on top of Multi-head Latent Attention (MLA).

Readings where the pages are silent (each also listed in the design notes):
* gate = ReLU; one index key per position shared by all indexer heads; the
  head weights are per query token.
* Top-K: the K largest scores, equal scores go to the lower position; rows
  with at most K candidates keep all of them; the selected positions are
  reported in ascending order, padded with -1.
* FP8 index keys carry one scale per token; the oracle dequantises each
  element (key * scale) before the dot product, and the index query takes
  part rounded to E4M3 (the index path quantises both index Q and K, "Day 0
  Inference Support...", "A Layered Strategy").
* MXFP8 index keys carry one E8M0 scale per group of 32 (or G) elements; the
  group exponent is floor(log2(amax)) - 8 (the microscaling rule for E4M3),
  and the index query is quantised the same way before the dot product.
* Attention core = absorbed MLA: the key of a position is its whole 576-wide
  latent row (512 latent + 64 rope), the value is the first 512 dims; logits
  are ``scale * q . c``, softmax over the selected positions, ``lse`` is the
  natural-log log-sum-exp of the scaled logits.
* Decode row b sees positions 0..seq_lens[b]-1 (the new token's key is already
  in the cache); prefill token t at position q_offset+t sees 0..q_offset+t.
* FP8 latent cache: E4M3 codes with one fp32 scale per token and tile of 128
  dims (the 64 rope dims form a fifth tile); scale = tile max / 448 in fp32,
  code = nearest E4M3 of x / scale in fp32; the oracle attends over code * scale.

Every function is pinned by the CPU tests to closed forms, brute force and
textbook routines (exact rational arithmetic, a rank-count definition of the
selection, torch's scaled_dot_product_attention in fp64).  The pages print no
worked example, so nothing is pinned to values printed on the pages.
"""
from __future__ import annotations

import math

import numpy as np

D_V = 512


def _f64(x) -> np.ndarray:
    """Any array-like (numpy or a CPU torch tensor of any float type) -> fp64."""
    if hasattr(x, "detach"):
        x = x.detach().cpu()
        if x.dtype.is_floating_point and x.dtype != __import__("torch").float64:
            x = x.float()
        x = x.numpy()
    return np.asarray(x, dtype=np.float64)


# ----------------------------------------------------------------------------
# step 1-2: indexer score (dot product per indexer head, ReLU gate, weighted
# sum over heads)
# ----------------------------------------------------------------------------

def e4m3_round(x) -> np.ndarray:
    """Round to the nearest FP8 E4M3 value (ties to even), saturating at +-448."""
    import torch
    t = torch.as_tensor(np.clip(_f64(x), -448.0, 448.0))
    return t.to(torch.float8_e4m3fn).to(torch.float64).numpy()


# MXFP8 ("Day 0 Inference Support for New LLM Architectures: Optimization
# Practices", "A Layered Strategy"; "Day 0 Inference Acceleration ...: Hybrid
# Attention Adaptation and Optimization Practices" §4, quantisation of the index
# Q/K): every group of G consecutive elements (G = 32 on the pages) shares one
# power-of-two scale, chosen dynamically from the group's largest magnitude.
# The reading taken here is the usual microscaling rule: the shared exponent is
# X = floor(log2(amax)) - emax, emax = 8 being the exponent of E4M3's largest
# normal (448 = 1.75 * 2**8); X is stored as an E8M0 byte X + 127 and held in
# [-127, 127]; an all-zero group takes X = -127.  Elements are x / 2**X rounded
# to the nearest E4M3 value (ties to even), saturating at +-448.

E4M3_EMAX = 8
E8M0_BIAS = 127


def mx_exponent(amax) -> int:
    """Shared exponent X of one group from its largest magnitude."""
    a = abs(float(amax))
    if a == 0.0:
        return -E8M0_BIAS
    m, e = math.frexp(a)              # a = m * 2**e with 0.5 <= m < 1: floor(log2 a) = e - 1
    return int(min(E8M0_BIAS, max(-E8M0_BIAS, e - 1 - E4M3_EMAX)))


def mxfp8_quantize(x, group: int = 32):
    """x [..., d] -> (codes [..., d] as E4M3 values in fp64, X [..., d/group] int64)."""
    a = _f64(x)
    d = a.shape[-1]
    assert d % group == 0
    blocks = a.reshape(a.shape[:-1] + (d // group, group))
    amax = np.abs(blocks).max(axis=-1)
    X = np.vectorize(mx_exponent, otypes=[np.int64])(amax) if amax.size else \
        np.zeros(amax.shape, dtype=np.int64)
    codes = e4m3_round(blocks / np.ldexp(1.0, X)[..., None])
    return codes.reshape(a.shape), X


def mxfp8_dequantize(codes, X, group: int = 32) -> np.ndarray:
    """codes [..., d] (E4M3 values) and X [..., d/group] -> values codes * 2**X."""
    c = _f64(codes)
    d = c.shape[-1]
    blocks = c.reshape(c.shape[:-1] + (d // group, group))
    return (blocks * np.ldexp(1.0, np.asarray(X, dtype=np.int64))[..., None]).reshape(c.shape)


def index_scores(q_idx, w, k_rows, k_scale=None) -> np.ndarray:
    """Indexer score of each given history row for one query token.

    q_idx [H_i, d], w [H_i], k_rows [n, d] -> I [n] fp64:
        I[s] = sum_h w[h] * max(0, sum_j q[h, j] * k[s, j]),
    where the keys are dequantised first when they are quantised:
    * k_scale [n] (FP8, one scale per token): k = k_rows * k_scale[s] and the
      index query takes part rounded to E4M3 (the index path quantises both
      index Q and K);
    * k_scale [n, d/G] of E8M0 bytes (MXFP8, one scale per group of G = d /
      k_scale.shape[1] elements): k = k_rows * 2**(byte - 127) group by group,
      and the index query is MXFP8-quantised with the same G and dequantised.
    """
    q = _f64(q_idx)
    k = _f64(k_rows)
    if k_scale is not None and np.ndim(_f64(k_scale)) == 2:
        byt = _f64(k_scale)
        group = k.shape[-1] // byt.shape[-1]
        qc, qX = mxfp8_quantize(q, group)
        q = mxfp8_dequantize(qc, qX, group)
        k = mxfp8_dequantize(k, byt.astype(np.int64) - E8M0_BIAS, group)
    elif k_scale is not None:
        q = e4m3_round(q)
        k = k * _f64(k_scale)[:, None]
    u = k @ q.T                       # relevance of row s for indexer head h: [n, H_i]
    gated = np.maximum(u, 0.0)        # ReLU gate
    return gated @ _f64(w)            # head-weight weighted sum over heads


# ----------------------------------------------------------------------------
# step 3: Top-K selection
# ----------------------------------------------------------------------------

def topk_select(scores, K: int):
    """Top-K positions of one score row.

    Returns (idx [K] int64 ascending, -1 padded; count).  Ordering: larger score
    first, equal scores by lower position; the first min(K, n) of that order
    are kept.
    """
    I = _f64(scores)
    n = I.shape[0]
    pos = np.arange(n)
    order = np.lexsort((pos, -I))     # primary: score descending, secondary: position
    keep = np.sort(order[:min(K, n)])
    out = np.full(K, -1, dtype=np.int64)
    out[:keep.shape[0]] = keep
    return out, int(keep.shape[0])


# ----------------------------------------------------------------------------
# steps 4-5: gather + attention over the selected latent rows
# ----------------------------------------------------------------------------

def sparse_mla(q, rows, scale: float, d_v: int = D_V):
    """Multi-head attention of one query token over the given latent rows.

    q [H, D], rows [n, D] -> (o [H, d_v], lse [H]):
        l[h, s] = scale * q[h] . rows[s]      (keys: the whole row)
        p = softmax_s(l),  o[h] = sum_s p[h, s] * rows[s, :d_v]  (values)
        lse[h] = log sum_s exp(l[h, s]).
    An empty row set gives o = 0 and lse = -inf.
    """
    qq = _f64(q)
    c = _f64(rows)
    H = qq.shape[0]
    if c.shape[0] == 0:
        return np.zeros((H, d_v)), np.full(H, -np.inf)
    logits = scale * (qq @ c.T)                   # [H, n]
    m = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - m)
    z = e.sum(axis=1, keepdims=True)
    o = (e @ c[:, :d_v]) / z
    lse = m[:, 0] + np.log(z[:, 0])
    return o, lse


def dense_mla(q, rows, scale: float, d_v: int = D_V):
    """Attention over every given row (the K >= history special case)."""
    return sparse_mla(q, rows, scale, d_v)


# ----------------------------------------------------------------------------
# FP8 latent cache ("Day 0 Inference Support for New LLM Architectures:
# Optimization Practices", "A Layered Strategy": the KV cache in FP8 with one
# scale per token and head tile of 128 elements).  The latent row (one MLA
# "head") splits into tiles of 128: dims 0-127, 128-255, 256-383, 384-511, and
# the 64 rope dims 512-575 as a fifth tile.  Reading: the scale of a tile is
# its largest magnitude over 448 (E4M3's largest normal), computed in fp32;
# each element is x / scale computed in fp32, rounded to the nearest E4M3
# value (ties to even); an all-zero tile has scale 0 and zero codes.
# ----------------------------------------------------------------------------

LATENT_TILES = ((0, 128), (128, 256), (256, 384), (384, 512), (512, 576))


def latent_fp8_quantize(rows):
    """rows [n, 576] -> (codes [n, 576] as E4M3 values in fp64, scales [n, 5]
    holding fp32 values)."""
    x = _f64(rows).astype(np.float32)
    codes = np.zeros(x.shape, dtype=np.float64)
    scales = np.zeros(x.shape[:-1] + (len(LATENT_TILES),), dtype=np.float32)
    for t, (a, b) in enumerate(LATENT_TILES):
        seg = x[..., a:b]
        amax = np.abs(seg).max(axis=-1)
        sc = (amax / np.float32(448.0)).astype(np.float32)
        safe = np.where(sc > 0, sc, np.float32(1.0)).astype(np.float32)
        y = np.where((sc > 0)[..., None], seg / safe[..., None], np.float32(0.0))
        codes[..., a:b] = e4m3_round(y.astype(np.float64))
        scales[..., t] = sc
    return codes, scales.astype(np.float64)


def latent_fp8_dequantize(codes, scales) -> np.ndarray:
    """codes [n, 576] (E4M3 values) and scales [n, 5] -> code * scale, tile by tile."""
    c = _f64(codes).copy()
    sc = _f64(scales)
    for t, (a, b) in enumerate(LATENT_TILES):
        c[..., a:b] *= sc[..., t:t + 1]
    return c


# ----------------------------------------------------------------------------
# cache addressing (contiguous or paged through a block table)
# ----------------------------------------------------------------------------

def history_rows(cache, b: int, positions, block_table=None, page_size: int = 0):
    """Rows of sequence b at the given logical positions.

    Contiguous cache: cache[b, pos].  Paged cache (a pool [P, page, ...]):
    cache[block_table[b, pos // page], pos % page].
    """
    pos = np.asarray(positions, dtype=np.int64)
    fp8 = getattr(cache, "dtype", None) is not None and "float8" in str(cache.dtype)
    if fp8:   # index the raw bytes (not every torch build indexes float8 tensors)
        return history_rows(cache.view(__import__("torch").uint8), b, pos, block_table,
                            page_size).view(cache.dtype)
    if block_table is None:
        return cache[b][pos] if len(pos) else cache[b][:0]
    bt = block_table[b]
    if hasattr(bt, "numpy"):
        bt = bt.cpu().numpy()
    pages = np.asarray(bt, dtype=np.int64)[pos // page_size]
    slots = pos % page_size
    return cache[pages, slots]


# ----------------------------------------------------------------------------
# one row of the whole layer
# ----------------------------------------------------------------------------

def _latent_reader(ws, b: int, bt):
    """latent_of(positions) for sequence b: bf16 rows, or FP8 codes dequantised
    with their tile scales."""
    lat = ws.latent.cpu()
    lsc = getattr(ws, "latent_scale", None)
    lsc = None if lsc is None else lsc.cpu()

    def latent_of(p):
        rows = history_rows(lat, b, p, bt, ws.page_size)
        if lsc is None:
            return rows
        return latent_fp8_dequantize(rows, history_rows(lsc, b, p, bt, ws.page_size))
    return latent_of


def layer_row(q_idx_t, w_t, q_t, k_hist, k_scale_hist, latent_of, n_hist: int, K: int,
              scale: float):
    """Indexer -> Top-K -> sparse MLA for one query token with n_hist visible rows.

    ``k_hist`` [n_hist, d] (and ``k_scale_hist``) are the visible index keys;
    ``latent_of(positions)`` returns the latent rows at those positions.
    Returns a dict with scores (fp64 and fp32-rounded), idx, count, out, lse.
    """
    I = index_scores(q_idx_t, w_t, k_hist, k_scale_hist)
    idx, count = topk_select(I, K)
    rows = latent_of(idx[:count])
    o, lse = sparse_mla(q_t, rows, scale)
    return {"scores": I, "scores_fp32": I.astype(np.float32), "idx": idx, "count": count,
            "out": o, "lse": lse}


def decode_row(ws, b: int):
    """Row b of a decode batch (attributes as laid out by the seeded generators)."""
    L = int(ws.seq_lens[b])
    pos = np.arange(L)
    bt = ws.block_table.cpu() if ws.block_table is not None else None
    k_hist = history_rows(ws.k_idx.cpu(), b, pos, bt, ws.page_size)
    ks = None
    if ws.k_scale is not None:
        ks = history_rows(ws.k_scale.cpu(), b, pos, bt, ws.page_size)
    return layer_row(ws.q_idx[b].cpu(), ws.w[b].cpu(), ws.q[b].cpu(), k_hist, ks,
                     _latent_reader(ws, b, bt), L, ws.K, ws.scale)


def multi_token_row(ws, r: int, tokens_per_seq: int):
    """Row r of a multi-token decode step (speculative verification, "Day 0
    Inference Acceleration for New LLM Architectures: Hybrid Attention Adaptation
    and Optimization Practices" §6): candidate t = r % T of sequence b = r // T.
    The T candidates' keys are the last T positions of the sequence's history;
    candidate t sees its own position and everything before it, i.e. the first
    seq_lens[b] - (T - 1 - t) positions, and runs the same index selection and
    attention as a single decode token."""
    T = int(tokens_per_seq)
    b, t = divmod(int(r), T)
    L = max(0, int(ws.seq_lens[b]) - (T - 1 - t))
    pos = np.arange(L)
    bt = ws.block_table.cpu() if ws.block_table is not None else None
    k_hist = history_rows(ws.k_idx.cpu(), b, pos, bt, ws.page_size)
    ks = None
    if ws.k_scale is not None:
        ks = history_rows(ws.k_scale.cpu(), b, pos, bt, ws.page_size)
    return layer_row(ws.q_idx[r].cpu(), ws.w[r].cpu(), ws.q[r].cpu(), k_hist, ks,
                     _latent_reader(ws, b, bt), L, ws.K, ws.scale)


def _rows_prefix(k_idx, n: int):
    """The first n key rows of the single prefill sequence (FP8 keys are
    sliced as raw bytes: not every torch build slices float8 tensors)."""
    k = k_idx.cpu()
    if "float8" in str(k.dtype):
        return k.view(__import__("torch").uint8)[0, :n].view(k.dtype)
    return k[0, :n]


def prefill_row(ws, t: int):
    """Query token t (position q_offset+t) of a causal prefill of one sequence."""
    n = ws.q_offset + t + 1
    k_hist = _rows_prefix(ws.k_idx, n)
    ks = None if ws.k_scale is None else ws.k_scale[0, :n].cpu()
    return layer_row(ws.q_idx[t].cpu(), ws.w[t].cpu(), ws.q[t].cpu(), k_hist, ks,
                     _latent_reader(ws, 0, None), n, ws.K, ws.scale)


def row_scores(ws, r: int) -> np.ndarray:
    """Indexer scores only, for row r (decode sequence or prefill token)."""
    if ws.mode == "decode":
        L = int(ws.seq_lens[r])
        pos = np.arange(L)
        bt = ws.block_table.cpu() if ws.block_table is not None else None
        k_hist = history_rows(ws.k_idx.cpu(), r, pos, bt, ws.page_size)
        ks = None if ws.k_scale is None else history_rows(ws.k_scale.cpu(), r, pos, bt,
                                                           ws.page_size)
        return index_scores(ws.q_idx[r].cpu(), ws.w[r].cpu(), k_hist, ks)
    n = ws.q_offset + r + 1
    ks = None if ws.k_scale is None else ws.k_scale[0, :n].cpu()
    return index_scores(ws.q_idx[r].cpu(), ws.w[r].cpu(), _rows_prefix(ws.k_idx, n), ks)


def layer(ws, rows=None):
    """The whole layer for the given rows (all rows by default)."""
    R = ws.q_idx.shape[0]
    rows = range(R) if rows is None else rows
    f = decode_row if ws.mode == "decode" else prefill_row
    return {r: f(ws, r) for r in rows}
