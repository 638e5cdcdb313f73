// Device-side helpers shared by the libdsi kernels: cache addressing, the
// device status word, bf16/fp8 unpacking and block-wide scans.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "dsi.h"

namespace dsi {

typedef __nv_bfloat16 bf16;

// Kernel-side copy of dsi_cache (passed by value).
struct CacheView {
  const void* k_idx;
  const float* k_scale;
  const bf16* latent;
  const int32_t* block_table;
  const int32_t* seq_lens;
  int64_t s_max;
  int64_t num_pages;
  int32_t page_size;
  int32_t max_pages;
  int32_t d;
  int32_t k_dtype;
  int32_t batch;
  int32_t tokens_per_seq;   // decode: query rows per sequence (1; T for a multi-token step)
};

// Device status word codes (mirrors dsi_status).
enum : int { kErrNone = 0, kErrTimeout = DSI_ERR_TIMEOUT, kErrBounds = DSI_ERR_BOUNDS };

__device__ __forceinline__ void report(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// Sequence of query row r: decode rows come tokens_per_seq to a sequence
// (row r is token r % T of sequence r / T); prefill rows all belong to one.
__device__ __forceinline__ int seq_of_row(const CacheView& c, int r, int decode) {
  if (!decode) return 0;
  return c.tokens_per_seq == 1 ? r : r / c.tokens_per_seq;   // no division in the common case
}

// Number of history positions visible to row r.  Decode: the T new tokens of
// a sequence are its last T cached positions, token t sees everything before
// the later ones (a length beyond the cache's rows per sequence is clamped).
__device__ __forceinline__ int64_t visible_len(const CacheView& c, int r, int decode,
                                               int64_t q_offset) {
  if (!decode) return q_offset + r + 1;
  const int T = c.tokens_per_seq;
  int64_t n = T == 1 ? (int64_t)__ldg(c.seq_lens + r)
                     : (int64_t)__ldg(c.seq_lens + r / T) - (T - 1 - r % T);
  n = n < 0 ? 0 : n;
  return n > c.s_max ? c.s_max : n;
}

// Physical row (in the contiguous array or the page pool) of logical position
// p of sequence b.  With DSI_CHECKED the page id is range-checked and -1 is
// returned (after flagging the status word) when it is out of range.
__device__ __forceinline__ int64_t phys_row(const CacheView& c, int b, int64_t p, int* err) {
  if (c.block_table == nullptr) return (int64_t)b * c.s_max + p;
  // positions come from int32 indices: divide in 32 bits when they fit
  const int64_t pg = (p >= 0 && p <= 0x7fffffff) ? (int64_t)((int)p / c.page_size) : p / c.page_size;
#ifdef DSI_CHECKED
  if (pg < 0 || pg >= c.max_pages) { report(err, kErrBounds); return -1; }
#endif
  const int page = __ldg(c.block_table + (int64_t)b * c.max_pages + pg);
#ifdef DSI_CHECKED
  if (page < 0 || page >= c.num_pages) { report(err, kErrBounds); return -1; }
#endif
  (void)err;
  return (int64_t)page * c.page_size + (p - pg * c.page_size);
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float* f) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

__device__ __forceinline__ void fp8x16_to_f32(const uint4& v, float* f) {
  const __nv_fp8x2_e4m3* h = reinterpret_cast<const __nv_fp8x2_e4m3*>(&v);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float2 t = static_cast<float2>(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

// Exclusive block-wide prefix sum of one int per thread.  `ws` holds >= 33
// ints of shared memory.  Returns the exclusive prefix; `total` gets the sum.
// Every thread of the block must call it.
__device__ __forceinline__ int block_exclusive_scan(int v, int* ws, int& total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) ws[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int s = lane < nw ? ws[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    ws[lane] = s;
  }
  __syncthreads();
  const int before = wid > 0 ? ws[wid - 1] : 0;
  total = ws[nw - 1];
  __syncthreads();
  return before + x - v;
}

// Order-preserving map of an fp32 score to an unsigned key: a larger score
// gives a larger key, -0 and +0 map to the same key (they compare equal), NaN
// is not expected.
__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

}  // namespace dsi
