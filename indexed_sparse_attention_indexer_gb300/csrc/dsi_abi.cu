// libdsi C ABI: argument validation on the host, then kernel launches on the
// caller's stream.  Nothing here computes; see include/dsi.h for the contract.
#include <stdio.h>
#include <string.h>

#include <atomic>

#include "kernels.h"
#include "latent_fp8.h"

using namespace dsi;

namespace {

std::atomic<unsigned long long> g_launches{0};

__device__ int g_status_word;  // device status (DSI_ERR_BOUNDS / DSI_ERR_TIMEOUT), 0 = ok

constexpr int kMaxDevices = 64;
// per-device address of g_status_word; atomics, so host threads that look it
// up at once store the same value without a data race
std::atomic<int*> g_status_ptr[kMaxDevices];

// Device address of the status word on the current device (looked up once;
// valid while the device's primary context lives).
int* status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  int* p = g_status_ptr[dev].load(std::memory_order_acquire);
  if (!p) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_status_word) != cudaSuccess) return nullptr;
    p = static_cast<int*>(a);
    g_status_ptr[dev].store(p, std::memory_order_release);
  }
  return p;
}

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

dsi_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return DSI_OK;
  if (e == cudaErrorInvalidValue) return DSI_ERR_UNSUPPORTED;
  return DSI_ERR_CUDA;
}

// Validate a cache description for rows of a decode batch or of a prefill.
dsi_status check_cache(const dsi_cache* c, int rows, int decode, int64_t q_offset, bool need_keys,
                       bool need_latent, int tokens_per_seq = 1) {
  if (!c) return DSI_ERR_INVALID_ARG;
  if (c->batch < 0) return DSI_ERR_INVALID_ARG;
  if (need_keys) {
    if (!c->k_idx) return DSI_ERR_INVALID_ARG;
    if (c->k_dtype != DSI_BF16 && c->k_dtype != DSI_FP8_E4M3 && c->k_dtype != DSI_MXFP8_E4M3)
      return DSI_ERR_UNSUPPORTED;
    if (c->d <= 0) return DSI_ERR_INVALID_ARG;
    const int chunk = c->k_dtype == DSI_BF16 ? 8 : 16;  // elements per 16-byte load
    if (c->d % chunk != 0 || c->d > 256) return DSI_ERR_UNSUPPORTED;
    if (!aligned(c->k_idx, 16)) return DSI_ERR_INVALID_ARG;
    if (c->k_dtype != DSI_BF16 && !c->k_scale) return DSI_ERR_INVALID_ARG;
    if (c->k_dtype == DSI_MXFP8_E4M3) {
      const int g = c->k_group ? c->k_group : 32;
      if (g != 32 && g != 64 && g != 128) return DSI_ERR_UNSUPPORTED;
      if (c->d % g != 0) return DSI_ERR_UNSUPPORTED;
      if (!aligned(c->k_scale, 16)) return DSI_ERR_INVALID_ARG;
    }
  }
  if (need_latent) {
    if (!c->latent || !aligned(c->latent, 16)) return DSI_ERR_INVALID_ARG;
    if (c->latent_dtype != DSI_BF16 && c->latent_dtype != DSI_FP8_E4M3) return DSI_ERR_UNSUPPORTED;
    if (c->latent_dtype == DSI_FP8_E4M3 && (!c->latent_scale || !aligned(c->latent_scale, 4)))
      return DSI_ERR_INVALID_ARG;
  }
  if (c->block_table) {
    if (c->page_size <= 0 || c->max_pages <= 0 || c->num_pages <= 0) return DSI_ERR_INVALID_ARG;
    if (c->page_size % 8 != 0) return DSI_ERR_UNSUPPORTED;
    if (c->s_max != (int64_t)c->max_pages * c->page_size) return DSI_ERR_INVALID_ARG;
  } else if (c->s_max <= 0) {
    return DSI_ERR_INVALID_ARG;
  }
  if (decode) {
    if ((int64_t)rows != (int64_t)c->batch * tokens_per_seq || !c->seq_lens)
      return DSI_ERR_INVALID_ARG;
  } else {
    if (c->batch != 1 || q_offset < 0 || q_offset + rows > c->s_max) return DSI_ERR_INVALID_ARG;
  }
  return DSI_OK;
}

CacheView view_of(const dsi_cache* c) {
  CacheView v;
  v.k_idx = c->k_idx;
  v.k_scale = c->k_dtype == DSI_FP8_E4M3 ? static_cast<const float*>(c->k_scale) : nullptr;
  v.k_mx_scale =
      c->k_dtype == DSI_MXFP8_E4M3 ? static_cast<const uint8_t*>(c->k_scale) : nullptr;
  v.k_group = c->k_group ? c->k_group : 32;
  v.latent = reinterpret_cast<const bf16*>(c->latent);
  v.block_table = c->block_table;
  v.seq_lens = c->seq_lens;
  v.s_max = c->s_max;
  v.num_pages = c->num_pages;
  v.page_size = c->page_size;
  v.max_pages = c->max_pages;
  v.d = c->d;
  v.k_dtype = c->k_dtype;
  v.batch = c->batch;
  v.tokens_per_seq = 1;
  return v;
}

// The attention core over the cache's latent rows: bf16 rows, or FP8 codes
// with their tile scales.
cudaError_t attend(const bf16* q, const CacheView& v, const dsi_cache* c, const int32_t* idx,
                   int rows, int H, int K, int decode, int64_t q_offset, float scale, bf16* out,
                   float* lse, void* ws, size_t ws_bytes, int* err, cudaStream_t st) {
  if (c->latent_dtype == DSI_FP8_E4M3)
    return launch_sparse_mla_fp8(q, v, c->latent_scale, idx, rows, H, K, decode, q_offset, scale,
                                 out, lse, ws, ws_bytes, err, st);
  return launch_sparse_mla(q, v, idx, rows, H, K, decode, q_offset, scale, out, lse, ws, ws_bytes,
                           err, st);
}

dsi_status check_mla_heads(int H) {
  if (H <= 0 || H > 128) return DSI_ERR_UNSUPPORTED;
  if (H > 16 && H % 16 != 0) return DSI_ERR_UNSUPPORTED;
  return DSI_OK;
}

// Workspace carving (every piece 256-byte aligned).
struct WsPlan {
  size_t scores_off, idx_off, mla_off, total;
  int64_t ld;
  int splits;
};

WsPlan plan_workspace(int rows, int Hi, int H, int K, int64_t s_max, size_t mla_budget_hint,
                      bool with_scores, bool with_idx) {
  WsPlan p;
  p.ld = (int64_t)round_up((size_t)(s_max > 0 ? s_max : 1), 64);
  size_t off = 0;
  p.scores_off = off;
  if (with_scores) off += round_up((size_t)rows * p.ld * sizeof(float), 256);
  p.idx_off = off;
  if (with_idx) off += round_up((size_t)rows * K * sizeof(int32_t), 256);
  p.mla_off = off;
  p.splits = mla_pick_splits(rows, H, K, mla_budget_hint);
  off += round_up(mla_partials_bytes(rows, H, p.splits), 256);
  p.total = off;
  (void)Hi;
  return p;
}

// Whether a call of the fused layer takes the fused prefill indexer (scores
// stay on chip) rather than the scoring kernel + Top-K pair.
bool uses_fused_prefill(const CacheView& v, int n_heads_idx, int rows, int64_t q_offset, int K,
                        int decode) {
  return !decode && fused_prefill_topk_supported(v, n_heads_idx, rows, q_offset, K);
}

// Workspace of one fused-layer call: score rows only for the unfused pair.
WsPlan layer_plan(const dsi_cache* c, int rows, int Hi, int H, int K, int64_t q_offset, int decode,
                  bool fused_prefill) {
  const int64_t span = decode ? c->s_max : q_offset + rows;
  return plan_workspace(rows, Hi, H, K, span, (size_t)-1, !fused_prefill, true);
}

}  // namespace

void dsi::note_launch(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

extern "C" {

uint64_t dsi_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }


const char* dsi_status_string(dsi_status s) {
  switch (s) {
    case DSI_OK: return "ok";
    case DSI_ERR_INVALID_ARG: return "invalid argument";
    case DSI_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case DSI_ERR_CUDA: return "CUDA error";
    case DSI_ERR_TIMEOUT: return "device wait timed out";
    case DSI_ERR_BOUNDS: return "index or page out of range";
    case DSI_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

int32_t dsi_version(void) { return DSI_VERSION; }

dsi_status dsi_index_score(const void* q_idx, const float* w, const dsi_cache* cache, int32_t rows,
                           int32_t n_heads_idx, int32_t decode, int64_t q_offset, float* scores,
                           int64_t ld_scores, void* stream) {
  if (!q_idx || !w || !scores || rows < 0) return DSI_ERR_INVALID_ARG;
  if (n_heads_idx < 1 || n_heads_idx > 128) return DSI_ERR_UNSUPPORTED;
  dsi_status s = check_cache(cache, rows, decode, q_offset, true, false);
  if (s != DSI_OK) return s;
  if (!aligned(q_idx, 16)) return DSI_ERR_INVALID_ARG;
  if (ld_scores < (decode ? cache->s_max : q_offset + rows)) return DSI_ERR_INVALID_ARG;
  if (rows == 0) return DSI_OK;
  CacheView v = view_of(cache);
  if (!index_score_supported(v, n_heads_idx, rows, decode)) return DSI_ERR_UNSUPPORTED;
  return from_cuda(launch_index_score(reinterpret_cast<const bf16*>(q_idx), w, v, rows,
                                      n_heads_idx, decode, q_offset, scores, ld_scores,
                                      status_ptr(), reinterpret_cast<cudaStream_t>(stream)));
}

dsi_status dsi_topk(const float* scores, int64_t ld_scores, int32_t rows, const int32_t* row_len,
                    int64_t q_offset, int32_t K, int32_t* idx, int32_t* count, void* stream) {
  if (!scores || !idx || rows < 0 || K < 1 || ld_scores < 1 || q_offset < 0)
    return DSI_ERR_INVALID_ARG;
  if (K > DSI_MAX_K) return DSI_ERR_UNSUPPORTED;
  if (rows == 0) return DSI_OK;
  return from_cuda(launch_topk(scores, ld_scores, rows, row_len, q_offset, K, idx, count,
                               reinterpret_cast<cudaStream_t>(stream)));
}

dsi_status dsi_index_topk_prefill(const void* q_idx, const float* w, const dsi_cache* cache,
                                  int32_t T, int32_t n_heads_idx, int64_t q_offset, int32_t K,
                                  int32_t* idx, int32_t* count, void* stream) {
  if (!q_idx || !w || !idx || T < 0 || K < 1) return DSI_ERR_INVALID_ARG;
  if (n_heads_idx < 1 || n_heads_idx > 128 || K > DSI_MAX_K) return DSI_ERR_UNSUPPORTED;
  dsi_status s = check_cache(cache, T, 0, q_offset, true, false);
  if (s != DSI_OK) return s;
  if (!aligned(q_idx, 16)) return DSI_ERR_INVALID_ARG;
  if (T == 0) return DSI_OK;
  CacheView v = view_of(cache);
  if (!fused_prefill_topk_supported(v, n_heads_idx, T, q_offset, K)) return DSI_ERR_UNSUPPORTED;
  return from_cuda(launch_index_topk_prefill(reinterpret_cast<const bf16*>(q_idx), w, v, T,
                                             q_offset, K, idx, count, status_ptr(),
                                             reinterpret_cast<cudaStream_t>(stream)));
}

static dsi_status mla_common(const void* q, const dsi_cache* cache, const int32_t* idx, int rows,
                             int H, int K, int decode, int64_t q_offset, float scale, void* out,
                             float* lse, void* ws, size_t ws_bytes, void* stream) {
  if (!q || !idx || !out || rows < 0 || K < 1) return DSI_ERR_INVALID_ARG;
  dsi_status s = check_mla_heads(H);
  if (s != DSI_OK) return s;
  s = check_cache(cache, rows, decode, q_offset, false, true);
  if (s != DSI_OK) return s;
  if (!aligned(q, 16) || !aligned(out, 16)) return DSI_ERR_INVALID_ARG;
  if (ws && !aligned(ws, 256)) return DSI_ERR_INVALID_ARG;
  if (!(scale == scale)) return DSI_ERR_INVALID_ARG;
  if (rows == 0) return DSI_OK;
  CacheView v = view_of(cache);
  return from_cuda(attend(reinterpret_cast<const bf16*>(q), v, cache, idx, rows, H, K, decode,
                          q_offset, scale, reinterpret_cast<bf16*>(out), lse, ws,
                          ws ? ws_bytes : 0, status_ptr(), reinterpret_cast<cudaStream_t>(stream)));
}

dsi_status dsi_sparse_mla_decode(const void* q, const dsi_cache* cache, const int32_t* idx,
                                 int32_t batch, int32_t n_heads, int32_t K, float scale, void* out,
                                 float* lse, void* workspace, size_t workspace_bytes,
                                 void* stream) {
  return mla_common(q, cache, idx, batch, n_heads, K, 1, 0, scale, out, lse, workspace,
                    workspace_bytes, stream);
}

dsi_status dsi_sparse_mla_prefill(const void* q, const dsi_cache* cache, const int32_t* idx,
                                  int32_t T, int32_t n_heads, int32_t K, int64_t q_offset,
                                  float scale, void* out, float* lse, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  return mla_common(q, cache, idx, T, n_heads, K, 0, q_offset, scale, out, lse, workspace,
                    workspace_bytes, stream);
}

size_t dsi_workspace_size(int32_t rows, int32_t n_heads_idx, int32_t n_heads, int32_t K,
                          int64_t s_max, int32_t decode) {
  (void)decode;
  if (rows <= 0 || K <= 0 || n_heads <= 0) return 256;
  const bool layer = n_heads_idx > 0 || s_max > 0;
  WsPlan p = plan_workspace(rows, n_heads_idx, n_heads, K, s_max, (size_t)-1, layer, layer);
  return p.total > 0 ? p.total : 256;
}

size_t dsi_layer_workspace_size(const dsi_cache* cache, int32_t rows, int32_t n_heads_idx,
                                int32_t n_heads, int32_t K, int64_t q_offset, int32_t decode) {
  if (!cache || rows <= 0 || K <= 0 || n_heads <= 0) return 256;
  if (!decode && q_offset < 0) return 256;
  const CacheView v = view_of(cache);
  const bool fused = uses_fused_prefill(v, n_heads_idx, rows, q_offset, K, decode);
  const WsPlan p = layer_plan(cache, rows, n_heads_idx, n_heads, K, q_offset, decode, fused);
  return p.total > 0 ? p.total : 256;
}

// The fused layer for rows of a decode batch (tokens_per_seq query tokens per
// sequence) or of a prefill.
static dsi_status layer_common(const void* q_idx, const float* w, const void* q,
                               const dsi_cache* cache, int32_t rows, int32_t n_heads_idx,
                               int32_t n_heads, int32_t K, int64_t q_offset, float scale,
                               int32_t decode, int32_t tokens_per_seq, int32_t* idx_out,
                               int32_t* count_out, void* out, float* lse, void* workspace,
                               size_t workspace_bytes, void* stream) {
  if (!q_idx || !w || !q || !out || rows < 0 || K < 1) return DSI_ERR_INVALID_ARG;
  if (n_heads_idx < 1 || n_heads_idx > 128 || K > DSI_MAX_K) return DSI_ERR_UNSUPPORTED;
  dsi_status s = check_mla_heads(n_heads);
  if (s != DSI_OK) return s;
  s = check_cache(cache, rows, decode, q_offset, true, true, tokens_per_seq);
  if (s != DSI_OK) return s;
  if (!aligned(q_idx, 16) || !aligned(q, 16) || !aligned(out, 16)) return DSI_ERR_INVALID_ARG;
  if (!(scale == scale)) return DSI_ERR_INVALID_ARG;
  if (rows == 0) return DSI_OK;
  CacheView v = view_of(cache);
  v.tokens_per_seq = tokens_per_seq;
  const bool fused_prefill = uses_fused_prefill(v, n_heads_idx, rows, q_offset, K, decode);
  if (!fused_prefill && !index_score_supported(v, n_heads_idx, rows, decode))
    return DSI_ERR_UNSUPPORTED;
  // the score rows only exist when the unfused scoring/select pair runs
  const WsPlan p = layer_plan(cache, rows, n_heads_idx, n_heads, K, q_offset, decode, fused_prefill);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < p.total) return DSI_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  float* scores = reinterpret_cast<float*>(ws + p.scores_off);
  int32_t* idx = idx_out ? idx_out : reinterpret_cast<int32_t*>(ws + p.idx_off);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int* err = status_ptr();
  cudaError_t e;
  if (fused_prefill) {
    // prefill: scores stay on chip, only the selected indices are written
    e = launch_index_topk_prefill(reinterpret_cast<const bf16*>(q_idx), w, v, rows, q_offset, K,
                                  idx, count_out, err, st);
    if (e != cudaSuccess) return from_cuda(e);
  } else {
    e = launch_index_score(reinterpret_cast<const bf16*>(q_idx), w, v, rows, n_heads_idx, decode,
                           q_offset, scores, p.ld, err, st);
    if (e != cudaSuccess) return from_cuda(e);
    // rows are clamped to what the scorer wrote: a decode length above s_max
    // counts as s_max, as in visible_len()
    e = launch_topk(scores, p.ld, rows, decode ? cache->seq_lens : nullptr, q_offset, K, idx,
                    count_out, st, tokens_per_seq, decode ? cache->s_max : q_offset + rows);
    if (e != cudaSuccess) return from_cuda(e);
  }
  e = attend(reinterpret_cast<const bf16*>(q), v, cache, idx, rows, n_heads, K, decode, q_offset,
             scale, reinterpret_cast<bf16*>(out), lse, ws + p.mla_off, p.total - p.mla_off, err,
             st);
  return from_cuda(e);
}

dsi_status dsi_indexed_attention(const void* q_idx, const float* w, const void* q,
                                 const dsi_cache* cache, int32_t rows, int32_t n_heads_idx,
                                 int32_t n_heads, int32_t K, int64_t q_offset, float scale,
                                 int32_t decode, int32_t* idx_out, int32_t* count_out, void* out,
                                 float* lse, void* workspace, size_t workspace_bytes,
                                 void* stream) {
  return layer_common(q_idx, w, q, cache, rows, n_heads_idx, n_heads, K, q_offset, scale, decode,
                      1, idx_out, count_out, out, lse, workspace, workspace_bytes, stream);
}

dsi_status dsi_indexed_attention_multi(const void* q_idx, const float* w, const void* q,
                                       const dsi_cache* cache, int32_t tokens_per_seq,
                                       int32_t n_heads_idx, int32_t n_heads, int32_t K,
                                       float scale, int32_t* idx_out, int32_t* count_out,
                                       void* out, float* lse, void* workspace,
                                       size_t workspace_bytes, void* stream) {
  if (!cache || tokens_per_seq < 1 || cache->batch < 0) return DSI_ERR_INVALID_ARG;
  const int64_t rows = (int64_t)cache->batch * tokens_per_seq;
  if (rows > 0x7fffffff) return DSI_ERR_INVALID_ARG;
  return layer_common(q_idx, w, q, cache, (int32_t)rows, n_heads_idx, n_heads, K, 0, scale, 1,
                      tokens_per_seq, idx_out, count_out, out, lse, workspace, workspace_bytes,
                      stream);
}

dsi_status dsi_mxfp8_quantize(const void* x, int64_t n_rows, int32_t d, int64_t ld_x,
                              int32_t group, const int64_t* dst_rows, void* codes, void* scales,
                              void* stream) {
  if (!x || !codes || !scales || n_rows < 0) return DSI_ERR_INVALID_ARG;
  if (group != 32 && group != 64 && group != 128) return DSI_ERR_UNSUPPORTED;
  if (d < 1 || d % group != 0) return DSI_ERR_UNSUPPORTED;
  if (ld_x < d || ld_x % 8 != 0 || !aligned(x, 16) || !aligned(codes, 16))
    return DSI_ERR_INVALID_ARG;
  if (n_rows == 0) return DSI_OK;
  return from_cuda(launch_mxfp8_quantize(reinterpret_cast<const bf16*>(x), n_rows, d, ld_x, group,
                                         dst_rows, static_cast<uint8_t*>(codes),
                                         static_cast<uint8_t*>(scales),
                                         reinterpret_cast<cudaStream_t>(stream)));
}

dsi_status dsi_latent_fp8_append(const void* x, int64_t n_rows, int64_t ld_x,
                                 const int64_t* dst_rows, void* codes, float* scales,
                                 void* stream) {
  if (!x || !codes || !scales || n_rows < 0) return DSI_ERR_INVALID_ARG;
  if (ld_x < DSI_D_QK || ld_x % 8 != 0 || !aligned(x, 16) || !aligned(codes, 16) ||
      !aligned(scales, 4))
    return DSI_ERR_INVALID_ARG;
  if (n_rows == 0) return DSI_OK;
  return from_cuda(launch_latent_fp8_append(reinterpret_cast<const bf16*>(x), n_rows, ld_x,
                                            dst_rows, static_cast<uint8_t*>(codes), scales,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

dsi_status dsi_selftest_wait_timeout(uint64_t limit_ns, void* stream) {
  if (limit_ns < 1000 || limit_ns > 1000000000ull) return DSI_ERR_INVALID_ARG;
  int* err = status_ptr();
  if (!err) return DSI_ERR_CUDA;
  return from_cuda(launch_selftest_wait_timeout(limit_ns, err,
                                                reinterpret_cast<cudaStream_t>(stream)));
}

dsi_status dsi_get_device_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return DSI_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof(int)) != cudaSuccess) return DSI_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int)) != cudaSuccess) return DSI_ERR_CUDA;
  }
  if (v == DSI_ERR_BOUNDS) return DSI_ERR_BOUNDS;
  if (v == DSI_ERR_TIMEOUT) return DSI_ERR_TIMEOUT;
  return v == 0 ? DSI_OK : DSI_ERR_CUDA;
}

}  // extern "C"
