// Sparse MLA attention core on CUDA cores (any head count that is a multiple
// of 16, or fewer than 16 heads).
//
// ("Day 0 Inference Support for New LLM Architectures: Optimization
// Practices", "Index-Based Sparse Attention": read the KV entries at the
// selected indices and run the attention over them; "Day 0 Inference
// Adaptation and Performance Optimization for New Models" §7: fuse the index
// reading with the computation.)  Absorbed-MLA reading: the key of a
// position is its whole 576-wide latent row, the value its first 512 dims.
//
// One block = (query row, group of 16 heads, split of the K indices).  The
// selected latent rows are gathered in tiles of 32 with cp.async into a
// double-buffered shared-memory tile (row stride padded to 1168 bytes so that
// 16-byte reads of different rows fall in different banks), logits are dot
// products against the block's fp32 query rows, the softmax is online (running
// max and sum per head) and P.V accumulates in registers.  With several
// splits, each block writes an unnormalised partial (o, m, l) and a combine
// kernel merges them with their log-sum-exp weights.
//
// FP8 latent cache ("Day 0 Inference Support...", "A Layered Strategy": the
// KV cache in FP8 with one scale per token and tile of 128 elements): the same
// kernel gathers the E4M3 codes (576 bytes per row) and the row's five tile
// scales; a logit sums code * q tile by tile and multiplies each tile's sum by
// its scale, and P.V scales each row's probability by the scale of the tile
// that holds the thread's output dims.
#include <math.h>

#include "kernels.h"
#include "latent_fp8.h"

namespace dsi {

constexpr int kHB = 16;        // heads per block
constexpr int kNT = 32;        // gathered rows per tile
constexpr int kRS = 584;       // shared row stride (bf16), 1168 bytes
constexpr int kRS8 = 656;      // FP8 rows: shared row stride in bytes (164 words: 16-byte reads of
                               // 8 consecutive rows fall in different banks)
constexpr int kMlaThreads = 256;
static_assert(sizeof(uint8_t[2][kNT][kRS8]) + sizeof(float[2][kNT][8]) <=
                  sizeof(bf16[2][kNT][kRS]), "FP8 tile fits the bf16 tile's space");
constexpr float kLog2e = 1.4426950408889634f;

struct MlaSmem {
  float q[kHB][DSI_D_QK];          // 36864 B
  union {
    bf16 c[2][kNT][kRS];           // 74752 B
    struct {
      uint8_t c8[2][kNT][kRS8];    // FP8 latent codes: 41984 B
      float sc[2][kNT][8];         // and the rows' tile scales (5 used)
    };
  };
  float p[kHB][kNT];               // 2048 B
  float m[kHB], l[kHB], alpha[kHB];
  int valid[2][kNT];
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }

// 8 E4M3 codes (byte i = element i) -> floats
__device__ __forceinline__ void fp8x8_to_f32(const uint2& v, float* f) {
  const __nv_fp8x2_e4m3* h = reinterpret_cast<const __nv_fp8x2_e4m3*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = static_cast<float2>(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n"); }

template <bool F8>
__global__ void __launch_bounds__(kMlaThreads)
mla_simt(const bf16* __restrict__ q, CacheView c, const float* __restrict__ lscale,
         const int32_t* __restrict__ idx, int H, int K, int decode, int64_t q_offset, float scale,
         bf16* __restrict__ out, float* __restrict__ lse, float* __restrict__ part_o,
         float2* __restrict__ part_ml, int splits, int* err) {
  extern __shared__ float4 mla_smem_raw[];
  MlaSmem& S = *reinterpret_cast<MlaSmem*>(mla_smem_raw);
  const int g = blockIdx.x, r = blockIdx.y, sp = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = seq_of_row(c, r, decode);
  const int64_t n_vis = visible_len(c, r, decode, q_offset);
  const int hcount = H - g * kHB < kHB ? H - g * kHB : kHB;  // heads of this block
  const int per = (K + splits - 1) / splits;
  const int j_begin = sp * per;
  const int j_end = min(K, j_begin + per);
  const int32_t* irow = idx + (int64_t)r * K;
  const float sl2 = scale * kLog2e;  // logits in log2 units

  // the block's query rows in fp32 (pre-scaled): every 16-byte load is issued
  // before any is converted, so their latencies overlap
  {
    constexpr int kQv = kHB * DSI_D_QK / 8;                     // 8-element pieces
    constexpr int kQPer = (kQv + kMlaThreads - 1) / kMlaThreads;
    uint4 qr[kQPer];
#pragma unroll
    for (int k = 0; k < kQPer; ++k) {
      const int i = tid + k * kMlaThreads;
      const int h = i / (DSI_D_QK / 8), pc = i - h * (DSI_D_QK / 8);
      qr[k] = (i < kQv && h < hcount)
                  ? __ldg(reinterpret_cast<const uint4*>(
                        q + ((int64_t)r * H + g * kHB + h) * DSI_D_QK + pc * 8))
                  : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int k = 0; k < kQPer; ++k) {
      const int i = tid + k * kMlaThreads;
      if (i < kQv) {
        const int h = i / (DSI_D_QK / 8), pc = i - h * (DSI_D_QK / 8);
        float f[8];
        bf16x8_to_f32(qr[k], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) S.q[h][pc * 8 + e] = f[e] * sl2;
      }
    }
  }
  // the indices come from the kernel launched before this one (the query rows
  // do not); the kernel after this one may start its set-up
  grid_dep_wait();
  grid_dep_launch();
  if (tid < kHB) { S.m[tid] = -INFINITY; S.l[tid] = 0.f; }

  auto gather = [&](int buf, int j0) {
    // bf16: 32 rows x 72 chunks of 16 bytes; FP8: 36 chunks of codes + 5 scales
    constexpr int kPer = F8 ? 41 : 72;
    for (int i = tid; i < kNT * kPer; i += kMlaThreads) {
      const int rr = i / kPer, ch = i - rr * kPer;
      const int j = j0 + rr;
      int pos = (j < j_end) ? __ldg(irow + j) : -1;
      // an index past the visible history is skipped in every build (the
      // checked build also reports it), so indices left unwritten by a
      // failed earlier kernel can never address rows outside the cache
      if (pos >= n_vis) {
#ifdef DSI_CHECKED
        report(err, kErrBounds);
#endif
        pos = -1;
      }
      int64_t row = pos >= 0 ? phys_row(c, b, pos, err) : -1;
      if (ch == 0) S.valid[buf][rr] = row >= 0;
      if (row < 0) continue;
      if (F8) {
        const uint8_t* codes = reinterpret_cast<const uint8_t*>(c.latent);
        if (ch < 36) cp_async16(&S.c8[buf][rr][ch * 16], codes + row * DSI_D_QK + ch * 16);
        else cp_async4(&S.sc[buf][rr][ch - 36], lscale + row * kLatentTiles + (ch - 36));
      } else {
        cp_async16(&S.c[buf][rr][ch * 8], c.latent + row * DSI_D_QK + ch * 8);
      }
    }
    cp_async_commit();
  };

  const int ntiles = (j_end - j_begin + kNT - 1) / kNT;
  // PV ownership: 8 dims (dc) x 4 heads (hq) per thread
  const int dc = tid & 63, hq = (tid >> 6) * 4;
  float acc[4][8];
#pragma unroll
  for (int h = 0; h < 4; ++h)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[h][e] = 0.f;

  if (ntiles > 0) gather(0, j_begin);
  for (int t = 0; t < ntiles; ++t) {
    const int buf = t & 1;
    cp_async_wait_all();
    __syncthreads();
    if (t + 1 < ntiles) gather(buf ^ 1, j_begin + (t + 1) * kNT);
    // ---- logits: lane = row of the tile, 2 heads per thread ----------------
    {
      const int pr = lane, h0 = warp * 2;
      float a0 = 0.f, a1 = 0.f;
      if (F8 && S.valid[buf][pr]) {
        // tile by tile: sum code * q over the tile, then times the tile's scale
        const uint8_t* crow = &S.c8[buf][pr][0];
#pragma unroll 1
        for (int t = 0; t < kLatentTiles; ++t) {
          const int ch0 = t * 8, ch1 = t < 4 ? ch0 + 8 : 36;   // 16-code chunks of the tile
          float b0 = 0.f, b1 = 0.f;
#pragma unroll 2
          for (int ch = ch0; ch < ch1; ++ch) {
            float cf[16];
            fp8x16_to_f32(*reinterpret_cast<const uint4*>(crow + ch * 16), cf);
            const float4* q0 = reinterpret_cast<const float4*>(&S.q[h0][ch * 16]);
            const float4* q1 = reinterpret_cast<const float4*>(&S.q[h0 + 1][ch * 16]);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float4 x = q0[k], y = q1[k];
              b0 = fmaf(x.x, cf[4 * k], b0); b0 = fmaf(x.y, cf[4 * k + 1], b0);
              b0 = fmaf(x.z, cf[4 * k + 2], b0); b0 = fmaf(x.w, cf[4 * k + 3], b0);
              b1 = fmaf(y.x, cf[4 * k], b1); b1 = fmaf(y.y, cf[4 * k + 1], b1);
              b1 = fmaf(y.z, cf[4 * k + 2], b1); b1 = fmaf(y.w, cf[4 * k + 3], b1);
            }
          }
          const float st = S.sc[buf][pr][t];
          a0 = fmaf(st, b0, a0);
          a1 = fmaf(st, b1, a1);
        }
      } else if (!F8 && S.valid[buf][pr]) {
        // four partial sums per head (dims 8ch + {0,4}, {1,5}, ...), so the
        // multiply-adds form four short chains instead of one long one
        const bf16* crow = &S.c[buf][pr][0];
        float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
        for (int ch = 0; ch < 72; ++ch) {
          float cf[8];
          bf16x8_to_f32(*reinterpret_cast<const uint4*>(crow + ch * 8), cf);
          const float4* q0 = reinterpret_cast<const float4*>(&S.q[h0][ch * 8]);
          const float4* q1 = reinterpret_cast<const float4*>(&S.q[h0 + 1][ch * 8]);
          float4 x0 = q0[0], x1 = q0[1], y0 = q1[0], y1 = q1[1];
          s0[0] = fmaf(x0.x, cf[0], s0[0]); s0[1] = fmaf(x0.y, cf[1], s0[1]);
          s0[2] = fmaf(x0.z, cf[2], s0[2]); s0[3] = fmaf(x0.w, cf[3], s0[3]);
          s0[0] = fmaf(x1.x, cf[4], s0[0]); s0[1] = fmaf(x1.y, cf[5], s0[1]);
          s0[2] = fmaf(x1.z, cf[6], s0[2]); s0[3] = fmaf(x1.w, cf[7], s0[3]);
          s1[0] = fmaf(y0.x, cf[0], s1[0]); s1[1] = fmaf(y0.y, cf[1], s1[1]);
          s1[2] = fmaf(y0.z, cf[2], s1[2]); s1[3] = fmaf(y0.w, cf[3], s1[3]);
          s1[0] = fmaf(y1.x, cf[4], s1[0]); s1[1] = fmaf(y1.y, cf[5], s1[1]);
          s1[2] = fmaf(y1.z, cf[6], s1[2]); s1[3] = fmaf(y1.w, cf[7], s1[3]);
        }
        a0 = (s0[0] + s0[1]) + (s0[2] + s0[3]);
        a1 = (s1[0] + s1[1]) + (s1[2] + s1[3]);
      } else {
        a0 = -INFINITY; a1 = -INFINITY;
      }
      // ---- online softmax for heads h0, h0+1 (whole warp owns them) --------
#pragma unroll
      for (int k2 = 0; k2 < 2; ++k2) {
        const int h = h0 + k2;
        const float v = k2 ? a1 : a0;
        float mx = v;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float m_old = S.m[h];
        const float m_new = fmaxf(m_old, mx);
        const float pv = (m_new == -INFINITY) ? 0.f : exp2f(v - m_new);
        float sum = pv;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        const float al = (m_old == -INFINITY) ? 0.f : exp2f(m_old - m_new);
        S.p[h][pr] = pv;
        __syncwarp();
        if (lane == 0) {
          S.alpha[h] = al;
          S.l[h] = S.l[h] * al + sum;
          S.m[h] = m_new;
        }
      }
    }
    __syncthreads();
    // ---- P.V: o[h, dims] = o * alpha + sum_j p[h, j] * c[j, dims] -----------
    {
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const float al = S.alpha[hq + h];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[h][e] *= al;
      }
      for (int j = 0; j < kNT; ++j) {
        if (!S.valid[buf][j]) continue;
        float cf[8];
        float sj = 1.f;   // FP8: the scale of the tile holding dims dc*8 .. dc*8+7
        if (F8) {
          fp8x8_to_f32(*reinterpret_cast<const uint2*>(&S.c8[buf][j][dc * 8]), cf);
          sj = S.sc[buf][j][dc >> 4];
        } else {
          bf16x8_to_f32(*reinterpret_cast<const uint4*>(&S.c[buf][j][dc * 8]), cf);
        }
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float pj = F8 ? S.p[hq + h][j] * sj : S.p[hq + h][j];
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[h][e] = fmaf(pj, cf[e], acc[h][e]);
        }
      }
    }
  }
  __syncthreads();
  // ---- epilogue ---------------------------------------------------------------
  if (splits == 1) {
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const int hh = hq + h;
      if (hh >= hcount) continue;
      const float l = S.l[hh];
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __align__(16) bf16 o8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) o8[e] = __float2bfloat16(acc[h][e] * inv);
      *reinterpret_cast<uint4*>(out + ((int64_t)r * H + g * kHB + hh) * DSI_D_LATENT + dc * 8) =
          *reinterpret_cast<const uint4*>(o8);
      if (lse && dc == 0)
        lse[(int64_t)r * H + g * kHB + hh] = l > 0.f ? (S.m[hh] + log2f(l)) / kLog2e : -INFINITY;
    }
  } else {
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const int hh = hq + h;
      if (hh >= hcount) continue;
      const int64_t pr = (((int64_t)r * splits + sp) * H + g * kHB + hh);
      float4* po = reinterpret_cast<float4*>(part_o + pr * DSI_D_LATENT + dc * 8);
      po[0] = make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
      po[1] = make_float4(acc[h][4], acc[h][5], acc[h][6], acc[h][7]);
      if (dc == 0) part_ml[pr] = make_float2(S.m[hh], S.l[hh]);
    }
  }
}

// Merge split-K partials: o = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s.
__global__ void __launch_bounds__(128)
mla_combine(const float* __restrict__ part_o, const float2* __restrict__ part_ml, int H,
            int splits, bf16* __restrict__ out, float* __restrict__ lse) {
  const int r = blockIdx.y, h = blockIdx.x, tid = threadIdx.x;
  grid_dep_wait();   // the partials come from the attention kernel launched just before
  float M = -INFINITY;
  for (int s = 0; s < splits; ++s) M = fmaxf(M, part_ml[((int64_t)r * splits + s) * H + h].x);
  float L = 0.f;
  float o[4] = {0.f, 0.f, 0.f, 0.f};
  for (int s = 0; s < splits; ++s) {
    const int64_t pr = ((int64_t)r * splits + s) * H + h;
    const float2 ml = part_ml[pr];
    if (ml.x == -INFINITY) continue;
    const float f = exp2f(ml.x - M);
    L += f * ml.y;
    const float4 v = reinterpret_cast<const float4*>(part_o + pr * DSI_D_LATENT)[tid];
    o[0] += f * v.x; o[1] += f * v.y; o[2] += f * v.z; o[3] += f * v.w;
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  __align__(8) bf16 o4[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) o4[e] = __float2bfloat16(o[e] * inv);
  *reinterpret_cast<uint2*>(out + ((int64_t)r * H + h) * DSI_D_LATENT + tid * 4) =
      *reinterpret_cast<const uint2*>(o4);
  if (lse && tid == 0) lse[(int64_t)r * H + h] = L > 0.f ? (M + log2f(L)) / kLog2e : -INFINITY;
}

cudaError_t launch_mla_combine(const float* part_o, const float2* part_ml, int rows, int H,
                               int splits, bf16* out, float* lse, cudaStream_t st) {
  const cudaError_t e = launch_overlapped(mla_combine, dim3(H, rows), dim3(128), 0, st, part_o,
                                          part_ml, H, splits, out, lse);
  note_launch();
  return e;
}

size_t mla_partials_bytes(int rows, int n_heads, int splits) {
  if (splits <= 1) return 0;
  const size_t n = (size_t)rows * splits * n_heads;
  return n * DSI_D_LATENT * sizeof(float) + n * sizeof(float2) + 256;
}

int mla_pick_splits(int rows, int n_heads, int K, size_t ws_bytes) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int groups = (n_heads + kHB - 1) / kHB;
  const long blocks = (long)rows * groups;
  int splits = 1;
  // aim for >= 2 blocks per SM, each split keeping >= 4 tiles of work; a
  // batch that fills under a quarter of the SMs (a single decode row) is
  // latency-bound and splits down to one tile per block
  const int min_tiles = blocks < sms / 4 ? 1 : 4;
  while (blocks * splits < 2L * sms && (K / (splits * 2)) >= min_tiles * kNT && splits < 16)
    splits *= 2;
  while (splits > 1 && mla_partials_bytes(rows, n_heads, splits) > ws_bytes) splits /= 2;
  return splits;
}

cudaError_t launch_sparse_mla_tc(const bf16* q, const CacheView& c, const float* latent_scale,
                                 const int32_t* idx, int rows, int n_heads, int K, int decode,
                                 int64_t q_offset, float scale, bf16* out, float* lse, void* ws,
                                 size_t ws_bytes, int* err, cudaStream_t st);
bool tc_mla_supported(int n_heads);
bool tc_mla_cache_ok(const CacheView& c);
bool tc_mla_fp8_ok(const CacheView& c, const float* latent_scale);

template <bool F8>
static cudaError_t launch_simt(const bf16* q, const CacheView& c, const float* lscale,
                               const int32_t* idx, int rows, int H, int K, int decode,
                               int64_t q_offset, float scale, bf16* out, float* lse, void* ws,
                               size_t ws_bytes, int* err, cudaStream_t st) {
  const int splits = mla_pick_splits(rows, H, K, ws ? ws_bytes : 0);
  const size_t smem = sizeof(MlaSmem);
  cudaError_t e = cudaFuncSetAttribute(mla_simt<F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  float* part_o = nullptr;
  float2* part_ml = nullptr;
  if (splits > 1) {
    const size_t n = (size_t)rows * splits * H;
    part_o = reinterpret_cast<float*>(ws);
    part_ml = reinterpret_cast<float2*>(reinterpret_cast<char*>(ws) + n * DSI_D_LATENT * sizeof(float));
  }
  dim3 grid((H + kHB - 1) / kHB, rows, splits);
  e = launch_overlapped(mla_simt<F8>, grid, dim3(kMlaThreads), smem, st, q, c, lscale, idx, H, K,
                        decode, q_offset, scale, out, lse, part_o, part_ml, splits, err);
  note_launch();
  if (e != cudaSuccess || splits == 1) return e;
  return launch_mla_combine(part_o, part_ml, rows, H, splits, out, lse, st);
}

cudaError_t launch_sparse_mla(const bf16* q, const CacheView& c, const int32_t* idx, int rows,
                              int H, int K, int decode, int64_t q_offset, float scale, bf16* out,
                              float* lse, void* ws, size_t ws_bytes, int* err, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  if (tc_mla_supported(H) && tc_mla_cache_ok(c))
    return launch_sparse_mla_tc(q, c, nullptr, idx, rows, H, K, decode, q_offset, scale, out, lse,
                                ws, ws_bytes, err, st);
  return launch_simt<false>(q, c, nullptr, idx, rows, H, K, decode, q_offset, scale, out, lse, ws,
                            ws_bytes, err, st);
}

cudaError_t launch_sparse_mla_fp8(const bf16* q, const CacheView& c, const float* latent_scale,
                                  const int32_t* idx, int rows, int H, int K, int decode,
                                  int64_t q_offset, float scale, bf16* out, float* lse, void* ws,
                                  size_t ws_bytes, int* err, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  // 128 heads: the tensor-core kernel, rows converted to bf16 as they land
  if (tc_mla_supported(H) && tc_mla_cache_ok(c) && tc_mla_fp8_ok(c, latent_scale))
    return launch_sparse_mla_tc(q, c, latent_scale, idx, rows, H, K, decode, q_offset, scale, out,
                                lse, ws, ws_bytes, err, st);
  return launch_simt<true>(q, c, latent_scale, idx, rows, H, K, decode, q_offset, scale, out,
                           lse, ws, ws_bytes, err, st);
}

}  // namespace dsi
