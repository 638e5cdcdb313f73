/*
 * dsi.h — C ABI of libdsi: the index-based sparse attention layer on one GPU.
 *
 * The layer has two stages ("Day 0 Inference Support for New LLM
 * Architectures: Optimization Practices", section "Index-Based Sparse
 * Attention"): a lightweight indexer scores the history positions of every
 * query token, weights the per-head scores with per-token head weights and
 * keeps the Top-K positions; a sparse attention core then reads only the
 * latent (MLA) cache rows at those positions and attends over them.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Memory: every pointer argument is caller-owned DEVICE memory unless its
 *   comment says otherwise.  The library allocates nothing per call; scratch
 *   space is a caller-provided workspace sized by dsi_workspace_size().
 * - Execution: calls enqueue kernels on `stream` (a cudaStream_t passed as
 *   void*, NULL = legacy default stream) and return after launch, without a
 *   host synchronisation.  Errors detectable on the host (null pointers,
 *   shapes, alignment, unsupported sizes) return before anything is launched
 *   and leave every output untouched.  Errors found by kernels (an index out
 *   of range when the library is built with DSI_CHECKED, a bounded wait that
 *   ran out) set a device status word that dsi_get_device_status() reads.
 * - No CPU fallback: a shape without a kernel returns DSI_ERR_UNSUPPORTED.
 * - Numbers: bf16 = IEEE bfloat16 (2 bytes), fp8 = E4M3 ("e4m3fn", 1 byte),
 *   scores fp32, indices int32.  Arrays are row-major, densely packed except
 *   where a leading dimension is passed.
 *
 * Cache layout (struct dsi_cache)
 * -------------------------------
 * One index key of width d per history position, shared by all indexer heads
 * (the pages read "the paged K cache"; "Internal Fusion of the Indexer"), and
 * one latent row of DSI_D_QK = 576 bf16 per position (512 latent + 64 rope;
 * "Day 0 Inference Adaptation and Performance Optimization for New Models" §1:
 * index selection on top of Multi-head Latent Attention).
 * - Contiguous (block_table == NULL): k_idx [batch, s_max, d],
 *   k_scale [batch, s_max], latent [batch, s_max, 576].
 * - Paged (block_table != NULL): pools k_idx [num_pages, page_size, d],
 *   k_scale [num_pages, page_size], latent [num_pages, page_size, 576];
 *   logical position p of sequence b lives in page block_table[b, p/page_size]
 *   at slot p % page_size.
 * - FP8 latent cache (latent_dtype == DSI_FP8_E4M3; "Day 0 Inference Support
 *   for New LLM Architectures: Optimization Practices", "A Layered Strategy":
 *   the KV cache in FP8 with one scale per token and head tile of 128
 *   elements): latent holds E4M3 codes [positions, 576] and latent_scale fp32
 *   [positions, 5], one scale per tile of dims 0-127, 128-255, 256-383,
 *   384-511 and 512-575 (the rope dims); the row's value is code * scale of
 *   its tile (see dsi_latent_fp8_append).
 * Row semantics:
 * - decode != 0: one query token per sequence; row b sees positions
 *   0 .. seq_lens[b]-1 (the new token's own key is already in the cache).
 *   A length above s_max counts as s_max (a negative one as 0) in every
 *   kernel: scoring, Top-K and attention agree on the clamped history.
 * - decode == 0 (prefill): one sequence (batch == 1); query token t sits at
 *   position q_offset + t and sees positions 0 .. q_offset + t.
 */
#ifndef DSI_H
#define DSI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSI_D_LATENT 512
#define DSI_D_ROPE 64
#define DSI_D_QK 576
#define DSI_MAX_K 4096          /* largest supported top-k */
#define DSI_VERSION 2          /* 2: MXFP8 keys and FP8 latent caches in dsi_cache */

typedef enum {
  DSI_OK = 0,
  DSI_ERR_INVALID_ARG = 1,   /* null pointer, negative size, inconsistent shape */
  DSI_ERR_UNSUPPORTED = 2,   /* valid, but no kernel for this shape / dtype */
  DSI_ERR_CUDA = 3,          /* a CUDA runtime call failed (launch, attribute) */
  DSI_ERR_TIMEOUT = 4,       /* a bounded device wait ran out (device status) */
  DSI_ERR_BOUNDS = 5,        /* an index or page id out of range (device status) */
  DSI_ERR_WORKSPACE = 6      /* workspace NULL or smaller than dsi_workspace_size() */
} dsi_status;

/* Index key formats.  DSI_MXFP8_E4M3: microscaled FP8 ("Day 0 Inference
 * Support for New LLM Architectures: Optimization Practices", "A Layered
 * Strategy": index Q/K in MXFP8, one scale per 32 elements, quantised
 * dynamically) -- E4M3 codes plus one E8M0 byte (scale 2^(byte-127)) per
 * group of k_group consecutive elements of a key. */
typedef enum { DSI_BF16 = 0, DSI_FP8_E4M3 = 1, DSI_MXFP8_E4M3 = 2 } dsi_dtype;

typedef struct dsi_cache {
  const void*    k_idx;        /* index keys, k_dtype elements */
  int32_t        k_dtype;      /* dsi_dtype of k_idx */
  int32_t        d;            /* index key width (64 or 128; any multiple of 8 on the generic kernel) */
  const void*    k_scale;      /* FP8: fp32 [positions], one scale per position;
                                  MXFP8: uint8 E8M0 [positions, d / k_group];
                                  NULL for bf16 (laid out like k_idx, minus d) */
  const void*    latent;       /* latent rows, 576 per position (bf16, or E4M3 codes) */
  const int32_t* block_table;  /* [batch, max_pages] page ids, or NULL for contiguous */
  int32_t        page_size;    /* positions per page (paged only; multiple of 8) */
  int32_t        max_pages;    /* columns of block_table (paged only) */
  const int32_t* seq_lens;     /* [batch] history length per sequence (decode); may be NULL for prefill */
  int32_t        batch;        /* number of sequences */
  int64_t        s_max;        /* contiguous: rows per sequence; paged: max_pages * page_size */
  int64_t        num_pages;    /* paged: pages in the pools (bounds checks); contiguous: 0 */
  int32_t        k_group;      /* MXFP8: elements per scale, 32, 64 or 128 (0 = 32); else unused */
  int32_t        latent_dtype; /* dsi_dtype of latent: DSI_BF16 (0) or DSI_FP8_E4M3 */
  const float*   latent_scale; /* FP8 latent: fp32 [positions, 5] tile scales; else NULL */
} dsi_cache;

/*
 * dsi_index_score — indexer scores of every visible position.
 * ("Day 0 Inference Support for New LLM Architectures: Optimization
 * Practices", "Internal Fusion of the Indexer": relevance scoring, then the
 * weighted sum over heads; "Day 0 Inference Adaptation and Performance
 * Optimization for New Models" §3, indexing stage.)
 *
 *   scores[r, s] = k_scale_s * sum_h w[r, h] * max(0, q_idx[r, h, :] . k[s, :])
 *
 * with k_scale_s = 1 for bf16 keys.  The ReLU gate is this library's stated
 * choice (the pages leave the activation open).  With FP8 keys the index
 * query takes part rounded to E4M3.  With MXFP8 keys k[s, :] is the
 * dequantised key (code * 2^(byte-127) group by group, k_scale_s = 1) and
 * the index query is MXFP8-quantised on the fly with the same group size (see
 * dsi_mxfp8_quantize) and dequantised; MXFP8 keys need n_heads_idx == 64,
 * d == 128, a 16-byte aligned k_scale, and either a paged page_size that is a
 * multiple of 64 or a contiguous s_max (and batch * s_max) that is a multiple
 * of 4, 8 or 16 for k_group 32, 64 or 128 (else DSI_ERR_UNSUPPORTED /
 * DSI_ERR_INVALID_ARG).
 *   q_idx   bf16 [rows, n_heads_idx, d]
 *   w       fp32 [rows, n_heads_idx] head weights per query token
 *   cache   see above; decode: rows == batch
 *   scores  fp32 [rows, ld_scores]; entries s < visible length of row r are
 *           written, the rest are left untouched.  ld_scores >= s_max
 *           (decode) or >= q_offset + rows (prefill).
 * Errors: DSI_ERR_INVALID_ARG (null, rows < 0, ld too small, prefill with
 * batch != 1 or q_offset + rows > s_max), DSI_ERR_UNSUPPORTED (d not a
 * multiple of 8, n_heads_idx outside 1..128, page_size not a multiple of 8).
 */
dsi_status dsi_index_score(const void* q_idx, const float* w, const dsi_cache* cache,
                           int32_t rows, int32_t n_heads_idx, int32_t decode, int64_t q_offset,
                           float* scores, int64_t ld_scores, void* stream);

/*
 * dsi_topk — per-row Top-K selection.
 * ("Day 0 Inference Support for New LLM Architectures: Optimization
 * Practices", "Internal Fusion of the Indexer": top-k over the weighted
 * scores, indices fed to the attention core.)
 *
 * For each row r with n_r candidates scores[r, 0 .. n_r-1]: keeps the
 * min(K, n_r) largest scores; equal scores are ranked by lower position.  The
 * kept positions are written to idx[r, 0 .. count-1] in ascending order, the
 * rest of the row is -1.  (Ascending order and -1 padding are this library's
 * reading; the pages only say an index sequence is output.)
 *   scores   fp32 [rows, ld_scores]; NaN is not allowed (undefined rank)
 *   row_len  int32 [rows] candidate count per row, or NULL for the causal
 *            prefill rule n_r = q_offset + r + 1
 *   idx      int32 [rows, K]
 *   count    int32 [rows] or NULL
 * Errors: DSI_ERR_INVALID_ARG (null, K < 1, rows < 0), DSI_ERR_UNSUPPORTED
 * (K > DSI_MAX_K).  A row length outside 0..ld_scores is clamped to that range.
 */
dsi_status dsi_topk(const float* scores, int64_t ld_scores, int32_t rows,
                    const int32_t* row_len, int64_t q_offset, int32_t K,
                    int32_t* idx, int32_t* count, void* stream);

/*
 * dsi_indexed_attention_multi — the fused layer for a multi-token decode step
 * (speculative verification: T candidate tokens per sequence checked at once).
 * ("Day 0 Inference Acceleration for New LLM Architectures: Hybrid Attention
 * Adaptation and Optimization Practices" §6: the speculative path reuses the
 * same index selection with a different candidate length.)
 *
 * Rows come tokens_per_seq (T) to a sequence: row r is candidate t = r % T of
 * sequence b = r / T.  The T candidates' keys are the last T cached positions
 * of sequence b (seq_lens[b] counts them), and candidate t sees positions
 * 0 .. seq_lens[b] - T + t (itself and everything before it).  Each row then
 * goes through the same indexer, Top-K and sparse attention as one decode
 * token (dsi_indexed_attention with decode = 1 is the T = 1 case).
 *   q_idx  bf16 [batch*T, n_heads_idx, d];  w  fp32 [batch*T, n_heads_idx]
 *   q      bf16 [batch*T, n_heads, 576];    out bf16 [batch*T, n_heads, 512]
 *   idx_out / count_out / lse / workspace as for dsi_indexed_attention with
 *   rows = batch*T (dsi_workspace_size(batch*T, n_heads_idx, n_heads, K, s_max, 1)).
 * Errors: as dsi_indexed_attention; DSI_ERR_INVALID_ARG for T < 1.
 */
dsi_status dsi_indexed_attention_multi(const void* q_idx, const float* w, const void* q,
                                       const dsi_cache* cache, int32_t tokens_per_seq,
                                       int32_t n_heads_idx, int32_t n_heads, int32_t K,
                                       float scale, int32_t* idx_out, int32_t* count_out,
                                       void* out, float* lse, void* workspace,
                                       size_t workspace_bytes, void* stream);

/*
 * dsi_index_topk_prefill — the prefill indexer in one kernel: scores, ReLU
 * gate, head weights and the running per-row Top-K, writing only indices.
 * ("Day 0 Inference Support for New LLM Architectures: Optimization
 * Practices", "Internal Fusion of the Indexer": scoring, weighting and
 * Top-K fused so the score matrix never leaves the chip; "Load Imbalance in
 * Causal Indexing and the Zigzag Layout": early and late query tokens paired.)
 *
 * Same result as dsi_index_score followed by dsi_topk with the causal rule
 * (row r sees positions 0 .. q_offset + r): identical indices, order, -1
 * padding and counts.
 *   q_idx   bf16 [T, n_heads_idx, d]
 *   w       fp32 [T, n_heads_idx]
 *   cache   bf16 index keys, contiguous (batch 1) or paged
 *   idx     int32 [T, K];  count  int32 [T] or NULL
 * Errors: DSI_ERR_INVALID_ARG (null, T < 0, K < 1, batch != 1, q_offset + T >
 * s_max), DSI_ERR_UNSUPPORTED when the fused kernel does not cover the shape
 * (n_heads_idx != 64, d != 128, FP8 keys, page_size not a multiple of 64,
 * K > 2048, q_offset + T > 131072): use dsi_index_score + dsi_topk there.
 */
dsi_status dsi_index_topk_prefill(const void* q_idx, const float* w, const dsi_cache* cache,
                                  int32_t T, int32_t n_heads_idx, int64_t q_offset, int32_t K,
                                  int32_t* idx, int32_t* count, void* stream);

/*
 * dsi_sparse_mla_decode — attention of one query token per sequence over the
 * latent rows at the selected positions.
 * ("Day 0 Inference Support for New LLM Architectures: Optimization
 * Practices", "Index-Based Sparse Attention": the attention core reads the KV
 * entries at the selected indices; "Day 0 Inference Adaptation and
 * Performance Optimization for New Models" §3, sparse attention stage.)
 *
 * Absorbed-MLA reading (the pages give no formula): for head h,
 *   l_s = scale * q[b, h, :] . c_s  (c_s = latent row of position s, 576 wide)
 *   out[b, h, :] = sum_s softmax(l)_s * c_s[0:512];  lse[b, h] = ln sum_s exp(l_s)
 * over the positions s = idx[b, j] >= 0.  With an FP8 latent cache c_s is the
 * dequantised row (code * tile scale); the 128-head tensor-core kernel reads
 * bf16 rows only, so FP8 latent caches take the CUDA-core kernel.
 *   q       bf16 [batch, n_heads, 576]
 *   idx     int32 [batch, K] logical positions (< seq_lens[b]); entries < 0 skipped
 *   out     bf16 [batch, n_heads, 512]
 *   lse     fp32 [batch, n_heads] or NULL; a row with no valid index gives
 *           out = 0 and lse = -inf
 *   workspace / workspace_bytes: optional (NULL, 0 allowed); with room for
 *           dsi_workspace_size(batch, 0, n_heads, K, 0, 1) bytes the kernel
 *           splits each row's K positions over several blocks.
 * Errors: DSI_ERR_INVALID_ARG, DSI_ERR_UNSUPPORTED (n_heads outside 1..128 or
 * not a multiple of 16 when > 16), DSI_ERR_BOUNDS (device status, DSI_CHECKED
 * builds) for an index >= seq_lens[b].
 */
dsi_status dsi_sparse_mla_decode(const void* q, const dsi_cache* cache, const int32_t* idx,
                                 int32_t batch, int32_t n_heads, int32_t K, float scale,
                                 void* out, float* lse, void* workspace, size_t workspace_bytes,
                                 void* stream);

/*
 * dsi_sparse_mla_prefill — the same attention for T query tokens of one
 * sequence (batch == 1); token t sits at position q_offset + t and its
 * indices must be <= q_offset + t.
 *   q    bf16 [T, n_heads, 576];  idx int32 [T, K];  out bf16 [T, n_heads, 512]
 *   lse  fp32 [T, n_heads] or NULL.  workspace as for decode (may be NULL).
 */
dsi_status dsi_sparse_mla_prefill(const void* q, const dsi_cache* cache, const int32_t* idx,
                                  int32_t T, int32_t n_heads, int32_t K, int64_t q_offset,
                                  float scale, void* out, float* lse, void* workspace,
                                  size_t workspace_bytes, void* stream);

/*
 * dsi_indexed_attention — the whole layer: indexer scores -> Top-K -> sparse
 * MLA, enqueued back to back on one stream (the only dependency is "Top-K
 * ready"; "Day 0 Inference Adaptation and Performance Optimization for New
 * Models" §3).  Arguments as in the entry points above.
 *   idx_out   int32 [rows, K] or NULL (then the indices live in the workspace)
 *   count_out int32 [rows] or NULL
 *   workspace at least dsi_workspace_size(rows, n_heads_idx, n_heads, K,
 *             s_max or q_offset + rows, decode) bytes, 256-byte aligned.
 * Errors: as for the parts; DSI_ERR_WORKSPACE when the workspace is too small.
 */
dsi_status dsi_indexed_attention(const void* q_idx, const float* w, const void* q,
                                 const dsi_cache* cache, int32_t rows, int32_t n_heads_idx,
                                 int32_t n_heads, int32_t K, int64_t q_offset, float scale,
                                 int32_t decode, int32_t* idx_out, int32_t* count_out,
                                 void* out, float* lse, void* workspace, size_t workspace_bytes,
                                 void* stream);

/*
 * dsi_indexed_attention_static — dsi_indexed_attention for callers that
 * cannot allocate device memory.  The pages have no counterpart: this entry
 * exists for callers such as a plugin inside a runtime that owns every device
 * allocation and offers its kernels no scratch, or a latency-critical path
 * that cannot afford cudaMalloc's implicit device synchronisation.
 *
 * Same arguments and results as dsi_indexed_attention, minus the workspace:
 * the scratch (score rows, indices, split-K partials) lives in one device
 * array of DSI_STATIC_SCRATCH_BYTES inside the library, which every GPU that
 * loads the library keeps until the process exits.  The caller still owns
 * inputs and outputs.  Returns DSI_ERR_WORKSPACE, before launching anything,
 * when dsi_layer_workspace_size() for the call exceeds
 * DSI_STATIC_SCRATCH_BYTES (a prefill on the fused indexer needs no score
 * rows, so e.g. 8192 tokens with K = 2048 fit where their score matrix
 * would not).  The first call on a device (with that device current) looks
 * up the array's device address and caches it; make that first call before
 * any stream capture.  The cached address belongs to the device's primary
 * context: after cudaDeviceReset() on that device the library must not be
 * called again in the process.  All calls share the array: calls whose
 * kernels overlap on the GPU race.  Nothing in the array needs to start at
 * zero.  Allocates nothing.
 */
#define DSI_STATIC_SCRATCH_BYTES (16u << 20)
dsi_status dsi_indexed_attention_static(const void* q_idx, const float* w, const void* q,
                                        const dsi_cache* cache, int32_t rows, int32_t n_heads_idx,
                                        int32_t n_heads, int32_t K, int64_t q_offset, float scale,
                                        int32_t decode, int32_t* idx_out, int32_t* count_out,
                                        void* out, float* lse, void* stream);

/* Bytes of workspace dsi_indexed_attention needs for any cache of these
 * sizes (and the larger, split-K sizing of the dsi_sparse_mla_* calls when
 * n_heads_idx == 0 and s_max == 0).  It counts the fp32 score rows of the
 * unfused scoring + Top-K pair, rows x round_up(s_max, 64) x 4 bytes, which a
 * prefill that takes the fused indexer does not use: dsi_layer_workspace_size
 * gives the exact figure for one call. */
size_t dsi_workspace_size(int32_t rows, int32_t n_heads_idx, int32_t n_heads, int32_t K,
                          int64_t s_max, int32_t decode);

/* Exact bytes of workspace one dsi_indexed_attention call with these
 * arguments needs (a multi-token step: rows = batch * tokens_per_seq,
 * decode = 1): the score rows only when the call runs the unfused scoring +
 * Top-K pair (every decode call; a prefill whose shape the fused indexer
 * does not cover), the indices, and the split-K partials.  Never more than
 * dsi_workspace_size(rows, n_heads_idx, n_heads, K, s_max or q_offset + rows,
 * decode).  Host only; returns 256 for non-positive sizes or a NULL cache. */
size_t dsi_layer_workspace_size(const dsi_cache* cache, int32_t rows, int32_t n_heads_idx,
                                int32_t n_heads, int32_t K, int64_t q_offset, int32_t decode);

/*
 * dsi_mxfp8_quantize — dynamic MXFP8 quantisation of bf16 rows: index keys on
 * their way into the cache (an append: dst_rows are the cache rows of the new
 * positions) or any index vectors.
 * ("Day 0 Inference Support for New LLM Architectures: Optimization
 * Practices", "A Layered Strategy": MXFP8 index Q/K, dynamic per-group
 * quantisation, 32 elements per scale; "Day 0 Inference Acceleration for New
 * LLM Architectures: Hybrid Attention Adaptation and Optimization Practices"
 * §4, per-group dynamic quantisation of the index Q/K; "Day 0 Inference
 * Adaptation and Performance Optimization for New Models" §4 and §7: the group
 * size as a configurable parameter to scan.)
 *
 * For row i and group g (elements g*group .. g*group+group-1):
 *   X = floor(log2(max |x|)) - 8 over the group, held in [-127, 127]
 *       (8 = exponent of E4M3's largest normal, 448); an all-zero group has X = -127
 *   codes[dst(i), j]  = E4M3 of x[i, j] / 2^X, nearest (ties to even),
 *                       saturating at +-448
 *   scales[dst(i), g] = X + 127 (E8M0)
 * with dst(i) = dst_rows[i], or i when dst_rows is NULL; a negative dst_rows
 * entry skips the row.  This library's reading of the scale rule is the usual
 * microscaling one; the pages fix only the group size and the dynamic choice.
 *   x         bf16 [n_rows, ld_x] (16-byte aligned, ld_x a multiple of 8, >= d);
 *             the first d elements of each row are quantised
 *   group     32, 64 or 128; d a multiple of group
 *   dst_rows  int64 [n_rows] device array, or NULL
 *   codes     uint8 E4M3 [*, d] (16-byte aligned), rows addressed by dst(i)
 *   scales    uint8 E8M0 [*, d / group], rows addressed by dst(i)
 * The caller guarantees every dst(i) lies inside codes and scales.
 * Errors: DSI_ERR_INVALID_ARG (null pointer, n_rows < 0, ld_x < d, ld_x not a
 * multiple of 8, misaligned x or codes), DSI_ERR_UNSUPPORTED (group not 32,
 * 64 or 128; d < 1 or not a multiple of group).
 */
dsi_status dsi_mxfp8_quantize(const void* x, int64_t n_rows, int32_t d, int64_t ld_x,
                              int32_t group, const int64_t* dst_rows, void* codes, void* scales,
                              void* stream);

/*
 * dsi_latent_fp8_append — quantise bf16 latent rows into an FP8 latent cache
 * (the on-the-fly cache write of new positions; "Day 0 Inference Adaptation
 * and Sparse Attention Optimization for New Large Model Architectures": cache
 * writes compressed to FP8 as they happen).
 *
 * For row i and tile t (dims 0-127, 128-255, 256-383, 384-511, 512-575):
 *   scale = (largest |x| of the tile) / 448 in fp32 (0 for an all-zero tile)
 *   codes[dst(i), j] = E4M3 of x[i, j] / scale computed in fp32, nearest
 *                      (ties to even), saturating at +-448 (0 when scale is 0)
 *   scales[dst(i), t] = scale
 * with dst(i) = dst_rows[i], or i when dst_rows is NULL; a negative entry
 * skips the row.  The scale rule is this library's reading; the pages fix the
 * tile of 128 per token and the FP8 format only.
 *   x         bf16 [n_rows, ld_x] (16-byte aligned, ld_x a multiple of 8, >= 576)
 *   dst_rows  int64 [n_rows] device array, or NULL
 *   codes     uint8 E4M3 [*, 576] (16-byte aligned)
 *   scales    fp32 [*, 5]
 * The caller guarantees every dst(i) lies inside codes and scales.
 * Errors: DSI_ERR_INVALID_ARG (null pointer, n_rows < 0, ld_x < 576, ld_x not
 * a multiple of 8, misaligned x, codes or scales).
 */
dsi_status dsi_latent_fp8_append(const void* x, int64_t n_rows, int64_t ld_x,
                                 const int64_t* dst_rows, void* codes, float* scales,
                                 void* stream);

/*
 * dsi_selftest_wait_timeout — exercises the failure-detection path.  The
 * pages have no counterpart: every wait inside the library's kernels is
 * bounded, and a wait that runs out sets the device status word to
 * DSI_ERR_TIMEOUT, drains its CTA and returns instead of hanging.  This call
 * launches one warp that waits, with the given limit, on a barrier nothing
 * ever completes, so that path can be tested: afterwards
 * dsi_get_device_status() returns DSI_ERR_TIMEOUT once, and the device stays
 * usable.  No memory is touched but the status word.
 *   limit_ns  1000 .. 1e9 (1 us .. 1 s); the kernel ends after about that long
 * Errors: DSI_ERR_INVALID_ARG for a limit outside the range.
 */
dsi_status dsi_selftest_wait_timeout(uint64_t limit_ns, void* stream);

/* Synchronises `stream`, returns and clears the device status word of the
 * current device (DSI_OK, DSI_ERR_BOUNDS or DSI_ERR_TIMEOUT), or DSI_ERR_CUDA
 * when the stream reports an asynchronous CUDA error. */
dsi_status dsi_get_device_status(void* stream);

/* Static description of a status code (never NULL). */
const char* dsi_status_string(dsi_status status);

/* DSI_VERSION of the built library. */
int32_t dsi_version(void);

/* Number of kernels this library has launched in this process (all devices,
 * all streams; counted on the host at launch).  For accounting in benchmarks. */
uint64_t dsi_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* DSI_H */
