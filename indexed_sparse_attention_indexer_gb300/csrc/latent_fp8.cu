// FP8 latent cache append: bf16 latent rows -> E4M3 codes with one fp32 scale
// per tile of 128 dims (the 64 rope dims form a fifth tile).
//
// ("Day 0 Inference Support for New LLM Architectures: Optimization
// Practices", "A Layered Strategy": the KV cache in FP8, one scale per token
// and head tile of 128 elements; "Day 0 Inference Adaptation and Sparse
// Attention Optimization for New Large Model Architectures": cache writes
// compressed to FP8 on the fly.)  Per tile: scale = max|x| / 448 in fp32, code
// = E4M3 of x / scale in fp32 (nearest even, saturating), both divisions IEEE
// round-to-nearest; an all-zero tile has scale 0 and zero codes.
//
// One warp per row: lane l holds dims 16l .. 16l+15 of the 512 latent dims
// (tile l / 8, whose maximum is a butterfly over 8 lanes), lanes 0-3 also the
// 64 rope dims.  HBM-bound: 1152 bytes read, 596 written per row.
#include "kernels.h"
#include "latent_fp8.h"

namespace dsi {
namespace {

__device__ __forceinline__ uint4 encode16_scaled(const float* f, float s) {
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float y[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) y[e] = s > 0.f ? __fdiv_rn(f[4 * k + e], s) : 0.f;
    const __nv_fp8x2_storage_t lo =
        __nv_cvt_float2_to_fp8x2(make_float2(y[0], y[1]), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi =
        __nv_cvt_float2_to_fp8x2(make_float2(y[2], y[3]), __NV_SATFINITE, __NV_E4M3);
    w[k] = (uint32_t)lo | ((uint32_t)hi << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__global__ void __launch_bounds__(256)
latent_fp8_append_kernel(const bf16* __restrict__ x, int64_t n_rows, int64_t ld_x,
                         const int64_t* __restrict__ dst_rows, uint8_t* __restrict__ codes,
                         float* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t row = warp0; row < n_rows; row += nwarps) {   // the whole warp takes one row
    const bf16* src = x + row * ld_x;
    float f[16], r[16];
    bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(src + lane * 16)), f);
    bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(src + lane * 16 + 8)), f + 8);
    float amax = 0.f, rmax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
    if (lane < 4) {
      bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(src + 512 + lane * 16)), r);
      bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(src + 512 + lane * 16 + 8)), r + 8);
#pragma unroll
      for (int i = 0; i < 16; ++i) rmax = fmaxf(rmax, fabsf(r[i]));
    }
#pragma unroll
    for (int m = 1; m < 8; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
#pragma unroll
    for (int m = 1; m < 4; m <<= 1) rmax = fmaxf(rmax, __shfl_xor_sync(0xffffffffu, rmax, m));
    const int64_t dst = dst_rows ? __ldg(dst_rows + row) : row;
    if (dst < 0) continue;
    const float s = __fdiv_rn(amax, 448.f);
    *reinterpret_cast<uint4*>(codes + dst * DSI_D_QK + lane * 16) = encode16_scaled(f, s);
    if ((lane & 7) == 0) scales[dst * kLatentTiles + (lane >> 3)] = s;
    if (lane < 4) {
      const float sr = __fdiv_rn(rmax, 448.f);
      *reinterpret_cast<uint4*>(codes + dst * DSI_D_QK + 512 + lane * 16) = encode16_scaled(r, sr);
      if (lane == 0) scales[dst * kLatentTiles + 4] = sr;
    }
  }
}

}  // namespace

cudaError_t launch_latent_fp8_append(const bf16* x, int64_t n_rows, int64_t ld_x,
                                     const int64_t* dst_rows, uint8_t* codes, float* scales,
                                     cudaStream_t st) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (n_rows + 7) / 8;                 // 8 rows (warps) per block
  const int64_t cap = (int64_t)sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  latent_fp8_append_kernel<<<(unsigned)blocks, 256, 0, st>>>(x, n_rows, ld_x, dst_rows, codes,
                                                              scales);
  note_launch();
  return cudaGetLastError();
}

}  // namespace dsi
