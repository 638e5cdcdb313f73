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
  const float* k_scale;      // FP8 keys: one scale per position (null otherwise)
  const uint8_t* k_mx_scale; // MXFP8 keys: E8M0 bytes [positions, d / k_group] (null otherwise)
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
  int32_t k_group;          // MXFP8 keys: elements per scale (32, 64 or 128)
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

// ---- MXFP8 (E4M3 codes with one power-of-two scale per group) -------------
// Shared exponent of a group from its largest magnitude (a non-negative
// float): floor(log2(amax)) - 8, held in [-127, 127].  floor(log2) is the
// biased exponent field minus 127 for normal numbers; zero and subnormal
// maxima lie below the E8M0 range and clamp to -127.
__device__ __forceinline__ int mx_exponent(float amax) {
  const int e = (int)(__float_as_uint(amax) >> 23);   // sign bit is clear
  if (e == 0) return -127;
  const int x = e - 127 - 8;
  return x < -127 ? -127 : x;                          // e <= 254 keeps x <= 119
}

// 16 floats scaled by 2^-X (exact: a power of two) and rounded to E4M3,
// nearest-even, saturating at +-448; byte i of the result is element i.
__device__ __forceinline__ uint4 mx_encode16(const float* f, int X) {
  const float inv = __uint_as_float((uint32_t)(127 - X) << 23);   // 2^-X, -X in [-119, 127]
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
        make_float2(f[4 * k] * inv, f[4 * k + 1] * inv), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
        make_float2(f[4 * k + 2] * inv, f[4 * k + 3] * inv), __NV_SATFINITE, __NV_E4M3);
    w[k] = (uint32_t)lo | ((uint32_t)hi << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// 16 E4M3 codes -> the 16 bf16 values code * 2^X (exact down to bf16's
// subnormal range).  Each code's sign, exponent and mantissa bits are moved
// into a bf16 bit pattern whose exponent field is the E4M3 field itself (so
// a subnormal code lands on a bf16 subnormal with the same mantissa); that
// pattern is the code's value times 2^-120, and one bf16 multiply by
// 2^(120 + X) rebiases and scales it (X > 7 takes a second multiply, since
// 2^(120 + X) would leave bf16's range).  lo = elements 0..7, hi = 8..15.
__device__ __forceinline__ void mx_decode16(const uint4& v, int X, uint4& lo, uint4& hi) {
  const uint32_t e1 = (uint32_t)(X <= 7 ? X + 247 : 247);
  const uint32_t m1 = (e1 << 7) | (e1 << 23);
  const uint32_t in[4] = {v.x, v.y, v.z, v.w};
  uint32_t out[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    // codes 0,1 (then 2,3) of the word into the high bytes of two halves
    const uint32_t a = __byte_perm(in[k], 0u, 0x1404);
    const uint32_t b = __byte_perm(in[k], 0u, 0x3424);
    out[2 * k] = bf16x2_mul((a & 0x80008000u) | ((a >> 4) & 0x07F007F0u), m1);
    out[2 * k + 1] = bf16x2_mul((b & 0x80008000u) | ((b >> 4) & 0x07F007F0u), m1);
  }
  if (X > 7) {
    const uint32_t e2 = (uint32_t)(X + 127);
    const uint32_t m2 = (e2 << 7) | (e2 << 23);
#pragma unroll
    for (int i = 0; i < 8; ++i) out[i] = bf16x2_mul(out[i], m2);
  }
  lo = make_uint4(out[0], out[1], out[2], out[3]);
  hi = make_uint4(out[4], out[5], out[6], out[7]);
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
