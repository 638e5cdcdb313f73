// Internal launchers of the FP8 latent cache: the append (quantising) kernel
// and the attention core over FP8 latent rows.  Argument validation happens
// in dsi_abi.cu.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace dsi {

// Tiles of one latent row: dims 0-127, 128-255, 256-383, 384-511 and the 64
// rope dims 512-575, one fp32 scale each.
constexpr int kLatentTiles = 5;

// codes[dst(i), :576] / scales[dst(i), :5] of bf16 latent rows x[i, :576] (pitch ld_x).
cudaError_t launch_latent_fp8_append(const bf16* x, int64_t n_rows, int64_t ld_x,
                                     const int64_t* dst_rows, uint8_t* codes, float* scales,
                                     cudaStream_t st);

// Sparse MLA over FP8 latent rows (c.latent holds E4M3 codes, latent_scale
// fp32 [positions, 5]); CUDA-core kernel, any head count the bf16 CUDA-core
// kernel takes.
cudaError_t launch_sparse_mla_fp8(const bf16* q, const CacheView& c, const float* latent_scale,
                                  const int32_t* idx, int rows, int H, int K, int decode,
                                  int64_t q_offset, float scale, bf16* out, float* lse, void* ws,
                                  size_t ws_bytes, int* err, cudaStream_t st);

}  // namespace dsi
