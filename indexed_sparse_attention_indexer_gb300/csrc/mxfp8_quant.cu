// Dynamic MXFP8 quantisation of bf16 rows (index keys on their way into the
// cache, or index queries).
//
// ("Day 0 Inference Support for New LLM Architectures: Optimization
// Practices", "A Layered Strategy": the index Q/K are MXFP8, every 32
// elements share one scale chosen on the fly.)  Per group of G elements:
// X = floor(log2(amax)) - 8 held in [-127, 127] (8 = exponent of E4M3's
// largest normal), codes = E4M3(x / 2^X) rounded to nearest even and
// saturated at +-448, scale byte = X + 127.
//
// An HBM-bound elementwise kernel: one thread per 16 elements (two 16-byte
// loads, one 16-byte store), the G/16 threads of a group sit in adjacent lanes
// and find the group maximum with butterfly shuffles.
#include "kernels.h"

namespace dsi {
namespace {

__global__ void __launch_bounds__(256)
mxfp8_quantize_kernel(const bf16* __restrict__ x, int64_t n_rows, int d, int64_t ld_x,
                      int group, const int64_t* __restrict__ dst_rows,
                      uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  const int upr = d >> 4;                      // 16-element units per row
  const int upg = group >> 4;                  // units per group (2, 4 or 8)
  const int64_t total = n_rows * upr;
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  // whole warps step together (the shuffles need every lane); groups never
  // straddle a warp because 32 and the row's unit count are multiples of upg
  for (int64_t base = warp0 * 32; base < total; base += nwarps * 32) {
    const int64_t unit = base + lane;
    const bool valid = unit < total;
    int64_t row = 0;
    int u = 0;
    float f[16];
    float amax = 0.f;
    if (valid) {
      row = unit / upr;
      u = (int)(unit - row * upr);
      const bf16* src = x + row * ld_x + u * 16;
      bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(src)), f);
      bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(src + 8)), f + 8);
#pragma unroll
      for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
    }
    for (int m = 1; m < upg; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
    if (!valid) continue;
    const int64_t dst = dst_rows ? __ldg(dst_rows + row) : row;
    if (dst < 0) continue;
    const int X = mx_exponent(amax);
    *reinterpret_cast<uint4*>(codes + dst * d + u * 16) = mx_encode16(f, X);
    if (u % upg == 0) scales[dst * (d / group) + u / upg] = (uint8_t)(X + 127);
  }
}

}  // namespace

cudaError_t launch_mxfp8_quantize(const bf16* x, int64_t n_rows, int d, int64_t ld_x, int group,
                                  const int64_t* dst_rows, uint8_t* codes, uint8_t* scales,
                                  cudaStream_t st) {
  const int64_t units = n_rows * (d / 16);
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (units + 255) / 256;
  const int64_t cap = (int64_t)sms * 8;        // 8 resident CTAs of 256 threads per SM
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  mxfp8_quantize_kernel<<<(unsigned)blocks, 256, 0, st>>>(x, n_rows, d, ld_x, group, dst_rows,
                                                           codes, scales);
  note_launch();
  return cudaGetLastError();
}

}  // namespace dsi
