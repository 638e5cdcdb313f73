// Indexer scoring on CUDA cores.
//
//   scores[r, s] = scale_s * sum_h w[r, h] * relu(q_idx[r, h, :] . k[s, :])
//
// ("Day 0 Inference Support for New LLM Architectures: Optimization
// Practices", "Internal Fusion of the Indexer": relevance scoring followed by
// the weighted sum over heads.)  Two kernels live here:
//  * score_stream: few indexer heads.  A bandwidth kernel: every lane loads one
//    16-byte slice of a key row, computes the partial dot products of its slice
//    against all heads and the slices of one row are combined with warp
//    shuffles; the key stream is read once with 128-bit loads.
//  * score_simt: any head count; one thread per position keeps the per-head
//    dot products in registers, the query rows sit in shared memory.
// The tensor-core kernel for 64 heads x 128 dims is in index_score_tc.cu.
#include "kernels.h"

namespace dsi {

template <typename KT> struct KeyTraits;
// kPerChunk: key elements per 16-byte load.  query(): the value an index
// query element takes part in the dot product with (with FP8 keys the index
// query is quantised to E4M3 as well).
template <> struct KeyTraits<bf16> {
  static constexpr int kPerChunk = 8;
  __device__ static void unpack(const uint4& v, float* f) { bf16x8_to_f32(v, f); }
  __device__ static float query(float x) { return x; }
};
template <> struct KeyTraits<__nv_fp8_e4m3> {
  static constexpr int kPerChunk = 16;
  __device__ static void unpack(const uint4& v, float* f) { fp8x16_to_f32(v, f); }
  __device__ static float query(float x) { return static_cast<float>(__nv_fp8_e4m3(x)); }
};

constexpr int kStreamWarps = 8;

template <int D, int HI, typename KT>
__global__ void __launch_bounds__(kStreamWarps * 32)
score_stream(const bf16* __restrict__ q_idx, const float* __restrict__ w, CacheView c,
             int decode, int64_t q_offset, float* __restrict__ scores, int64_t ld, int* err) {
  constexpr int EPC = KeyTraits<KT>::kPerChunk;
  constexpr int LPP = D / EPC;   // lanes per key row
  constexpr int PPW = 32 / LPP;  // key rows per warp step
  static_assert(D % EPC == 0 && LPP <= 32 && (LPP & (LPP - 1)) == 0, "shape");
  const int r = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = lane % LPP, grp = lane / LPP;
  const int b = seq_of_row(c, r, decode);
  const int64_t n = visible_len(c, r, decode, q_offset);

  float qr[HI][EPC];
  float wr[HI];
#pragma unroll
  for (int h = 0; h < HI; ++h) {
    const bf16* qp = q_idx + ((int64_t)r * HI + h) * D + sub * EPC;
#pragma unroll
    for (int e = 0; e < EPC; e += 8) {
      uint4 v = *reinterpret_cast<const uint4*>(qp + e);
      bf16x8_to_f32(v, &qr[h][e]);
    }
#pragma unroll
    for (int e = 0; e < EPC; ++e) qr[h][e] = KeyTraits<KT>::query(qr[h][e]);
    wr[h] = w[(int64_t)r * HI + h];
  }
  const KT* kbase = reinterpret_cast<const KT*>(c.k_idx);
  const int64_t step = (int64_t)gridDim.x * kStreamWarps * PPW;
  for (int64_t base = ((int64_t)blockIdx.x * kStreamWarps + warp) * PPW; base < n; base += step) {
    const int64_t p = base + grp;
    const bool valid = p < n;
    float kf[EPC];
    int64_t row = 0;
    if (valid) {
      row = phys_row(c, b, p, err);
      if (row < 0) row = 0;
      uint4 v = __ldg(reinterpret_cast<const uint4*>(kbase + row * D + sub * EPC));
      KeyTraits<KT>::unpack(v, kf);
    } else {
#pragma unroll
      for (int e = 0; e < EPC; ++e) kf[e] = 0.f;
    }
    float part[HI];
#pragma unroll
    for (int h = 0; h < HI; ++h) {
      float a = 0.f;
#pragma unroll
      for (int e = 0; e < EPC; ++e) a = fmaf(qr[h][e], kf[e], a);
      part[h] = a;
    }
#pragma unroll
    for (int o = LPP / 2; o > 0; o >>= 1) {
#pragma unroll
      for (int h = 0; h < HI; ++h) part[h] += __shfl_xor_sync(0xffffffffu, part[h], o);
    }
    if (valid && sub == 0) {
      float s = 0.f;
#pragma unroll
      for (int h = 0; h < HI; ++h) s = fmaf(wr[h], part[h] > 0.f ? part[h] : 0.f, s);
      if (c.k_scale) s *= __ldg(c.k_scale + row);
      scores[(int64_t)r * ld + p] = s;
    }
  }
}

// Generic: one thread per key row, q rows staged in shared memory as fp32.
template <int HMAX, typename KT>
__global__ void __launch_bounds__(128)
score_simt(const bf16* __restrict__ q_idx, const float* __restrict__ w, CacheView c, int H,
           int decode, int64_t q_offset, float* __restrict__ scores, int64_t ld, int* err) {
  extern __shared__ float4 smem_f4[];
  float* qs = reinterpret_cast<float*>(smem_f4);  // [H][D]
  float* ws = qs + H * c.d;                       // [H]
  const int D = c.d;
  const int r = blockIdx.y;
  const int b = seq_of_row(c, r, decode);
  const int64_t n = visible_len(c, r, decode, q_offset);
  for (int i = threadIdx.x; i < H * D; i += blockDim.x)
    qs[i] = KeyTraits<KT>::query(__bfloat162float(q_idx[(int64_t)r * H * D + i]));
  for (int i = threadIdx.x; i < H; i += blockDim.x) ws[i] = w[(int64_t)r * H + i];
  __syncthreads();
  constexpr int EPC = KeyTraits<KT>::kPerChunk;
  const KT* kbase = reinterpret_cast<const KT*>(c.k_idx);
  for (int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < n;
       p += (int64_t)gridDim.x * blockDim.x) {
    int64_t row = phys_row(c, b, p, err);
    if (row < 0) continue;
    float acc[HMAX];
#pragma unroll
    for (int h = 0; h < HMAX; ++h) acc[h] = 0.f;
    const KT* kr = kbase + row * D;
    for (int j = 0; j < D; j += EPC) {
      float kf[EPC];
      KeyTraits<KT>::unpack(__ldg(reinterpret_cast<const uint4*>(kr + j)), kf);
#pragma unroll
      for (int h = 0; h < HMAX; ++h) {
        if (h < H) {
          const float* qh = qs + h * D + j;
          float a = acc[h];
#pragma unroll
          for (int e = 0; e < EPC; e += 4) {
            float4 qv = *reinterpret_cast<const float4*>(qh + e);
            a = fmaf(qv.x, kf[e], a);
            a = fmaf(qv.y, kf[e + 1], a);
            a = fmaf(qv.z, kf[e + 2], a);
            a = fmaf(qv.w, kf[e + 3], a);
          }
          acc[h] = a;
        }
      }
    }
    float s = 0.f;
#pragma unroll
    for (int h = 0; h < HMAX; ++h)
      if (h < H) s = fmaf(ws[h], acc[h] > 0.f ? acc[h] : 0.f, s);
    if (c.k_scale) s *= __ldg(c.k_scale + row);
    scores[(int64_t)r * ld + p] = s;
  }
}

cudaError_t launch_index_score_tc(const bf16* q_idx, const float* w, const CacheView& c,
                                  int rows, int decode, int64_t q_offset, float* scores,
                                  int64_t ld, int* err, cudaStream_t st);
bool tc_score_supported(const CacheView& c, int n_heads_idx);
bool tc_score_shape_ok(const CacheView& c, int rows, int decode);

ScoreKernel pick_score_kernel(const CacheView& c, int H) {
  if (tc_score_supported(c, H)) return kScoreTc;
  const bool fp8 = c.k_dtype == DSI_FP8_E4M3;
  if ((c.d == 64 || c.d == 128) && ((!fp8 && H <= 8 && (H == 1 || H == 2 || H == 4 || H == 8)) ||
                                    (fp8 && (H == 1 || H == 2 || H == 4))))
    return kScoreStream;
  return kScoreSimt;
}

template <int D, int HI, typename KT>
static cudaError_t go_stream(const bf16* q, const float* w, const CacheView& c, int rows,
                             int decode, int64_t q_offset, float* scores, int64_t ld, int* err,
                             cudaStream_t st) {
  constexpr int EPC = KeyTraits<KT>::kPerChunk;
  constexpr int PPB = kStreamWarps * (32 / (D / EPC));
  const int64_t span = decode ? c.s_max : q_offset + rows;
  int64_t gx = (span + PPB - 1) / PPB;
  if (gx > 1024) gx = 1024;
  if (gx < 1) gx = 1;
  dim3 grid((unsigned)gx, (unsigned)rows);
  score_stream<D, HI, KT><<<grid, kStreamWarps * 32, 0, st>>>(q, w, c, decode, q_offset, scores,
                                                               ld, err);
  note_launch();
  return cudaGetLastError();
}

template <typename KT>
static cudaError_t dispatch_stream(const bf16* q, const float* w, const CacheView& c, int rows,
                                   int H, int decode, int64_t q_offset, float* scores,
                                   int64_t ld, int* err, cudaStream_t st) {
#define DSI_GO(DD, HH)                                                                    \
  if (c.d == DD && H == HH)                                                               \
    return go_stream<DD, HH, KT>(q, w, c, rows, decode, q_offset, scores, ld, err, st);
  DSI_GO(64, 1) DSI_GO(64, 2) DSI_GO(64, 4) DSI_GO(128, 1) DSI_GO(128, 2) DSI_GO(128, 4)
  if (KeyTraits<KT>::kPerChunk == 8) { DSI_GO(64, 8) DSI_GO(128, 8) }
#undef DSI_GO
  return cudaErrorInvalidValue;
}

template <typename KT>
static cudaError_t dispatch_simt(const bf16* q, const float* w, const CacheView& c, int rows,
                                 int H, int decode, int64_t q_offset, float* scores, int64_t ld,
                                 int* err, cudaStream_t st) {
  const int64_t span = decode ? c.s_max : q_offset + rows;
  int64_t gx = (span + 127) / 128;
  if (gx > 512) gx = 512;
  if (gx < 1) gx = 1;
  dim3 grid((unsigned)gx, (unsigned)rows);
  const size_t smem = (size_t)(H * c.d + H) * sizeof(float);
#define DSI_GO(HM)                                                                         \
  if (H <= HM) {                                                                           \
    if (smem > 48 * 1024)                                                                  \
      cudaFuncSetAttribute(score_simt<HM, KT>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                           (int)smem);                                                     \
    score_simt<HM, KT><<<grid, 128, smem, st>>>(q, w, c, H, decode, q_offset, scores, ld,  \
                                                err);                                      \
    note_launch();                                                                         \
    return cudaGetLastError();                                                             \
  }
  DSI_GO(8) DSI_GO(16) DSI_GO(32) DSI_GO(64) DSI_GO(128)
#undef DSI_GO
  return cudaErrorInvalidValue;
}

bool index_score_supported(const CacheView& c, int H, int rows, int decode) {
  if (c.k_dtype != DSI_MXFP8_E4M3) return true;
  return tc_score_supported(c, H) && tc_score_shape_ok(c, rows, decode);
}

cudaError_t launch_index_score(const bf16* q_idx, const float* w, const CacheView& c, int rows,
                               int H, int decode, int64_t q_offset, float* scores, int64_t ld,
                               int* err, cudaStream_t st) {
  const bool fp8 = c.k_dtype == DSI_FP8_E4M3;
  if (!index_score_supported(c, H, rows, decode)) return cudaErrorInvalidValue;
  ScoreKernel k = pick_score_kernel(c, H);
  if (k == kScoreTc && !tc_score_shape_ok(c, rows, decode)) k = kScoreSimt;
  switch (k) {
    case kScoreTc:
      return launch_index_score_tc(q_idx, w, c, rows, decode, q_offset, scores, ld, err, st);
    case kScoreStream:
      return fp8 ? dispatch_stream<__nv_fp8_e4m3>(q_idx, w, c, rows, H, decode, q_offset, scores,
                                                  ld, err, st)
                 : dispatch_stream<bf16>(q_idx, w, c, rows, H, decode, q_offset, scores, ld, err,
                                         st);
    default:
      return fp8 ? dispatch_simt<__nv_fp8_e4m3>(q_idx, w, c, rows, H, decode, q_offset, scores,
                                                ld, err, st)
                 : dispatch_simt<bf16>(q_idx, w, c, rows, H, decode, q_offset, scores, ld, err,
                                       st);
  }
}

}  // namespace dsi
