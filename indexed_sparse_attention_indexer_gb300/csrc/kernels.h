// Internal launchers of the libdsi kernels (host side).  Each returns the
// cudaError_t of its launch; argument validation happens in dsi_abi.cu.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace dsi {

// Counts kernel launches made by the library (dsi_launch_count()).
void note_launch(int n = 1);

// Launch with programmatic stream serialisation: the kernel may start while
// the previous kernel on the stream finishes (once that kernel has signalled
// griddepcontrol.launch_dependents, or at its end); the kernel itself executes
// griddepcontrol.wait before it reads anything the previous kernel writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Device side of the same: wait for the previous kernel's results / let the
// next kernel start its set-up.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

// ---- indexer scoring -------------------------------------------------------
// scores[r, s] for s < visible_len(r); kernels: warp-shuffle streaming (few
// heads), tcgen05 tensor-core tiles (64 heads x 128 dims), generic SIMT.
cudaError_t launch_index_score(const bf16* q_idx, const float* w, const CacheView& c, int rows,
                               int n_heads_idx, int decode, int64_t q_offset, float* scores,
                               int64_t ld, int* err, cudaStream_t st);

// Whether a scoring kernel exists for the shape (MXFP8 keys: the tensor-core
// kernel only).
bool index_score_supported(const CacheView& c, int n_heads_idx, int rows, int decode);

// Which scoring kernel a shape takes (for tests and the bench's accounting).
enum ScoreKernel { kScoreStream = 0, kScoreSimt = 1, kScoreTc = 2 };
ScoreKernel pick_score_kernel(const CacheView& c, int n_heads_idx);

// Fused prefill indexer: scoring + running per-row Top-K in the epilogue;
// writes only idx [rows, K] (ascending, -1 padded) and count [rows] (may be null).
bool fused_prefill_topk_supported(const CacheView& c, int n_heads_idx, int rows, int64_t q_offset,
                                  int K);
cudaError_t launch_index_topk_prefill(const bf16* q_idx, const float* w, const CacheView& c,
                                      int rows, int64_t q_offset, int K, int32_t* idx,
                                      int32_t* count, int* err, cudaStream_t st);

// ---- Top-K -------------------------------------------------------------------
// row_len: candidates per row, or per sequence when tokens_per_seq > 1 (row r
// is token r % T of sequence r / T and has row_len[r / T] - (T - 1 - r % T));
// null: the causal prefill rule q_offset + r + 1.  Row lengths are clamped
// to n_cap (negative: ld), the longest row the scorer wrote (s_max for a
// decode batch: its visible lengths never exceed the cache's rows).
cudaError_t launch_topk(const float* scores, int64_t ld, int rows, const int32_t* row_len,
                        int64_t q_offset, int K, int32_t* idx, int32_t* count,
                        cudaStream_t st, int tokens_per_seq = 1, int64_t n_cap = -1);

// ---- sparse MLA ----------------------------------------------------------------
// part_o / part_ml: split-K partials (may be null when splits == 1).
size_t mla_partials_bytes(int rows, int n_heads, int splits);
// Merges split-K partials (unnormalised o, running max m in log2 units, sum l).
cudaError_t launch_mla_combine(const float* part_o, const float2* part_ml, int rows, int H,
                               int splits, bf16* out, float* lse, cudaStream_t st);
int mla_pick_splits(int rows, int n_heads, int K, size_t ws_bytes);
cudaError_t launch_sparse_mla(const bf16* q, const CacheView& c, const int32_t* idx, int rows,
                              int n_heads, int K, int decode, int64_t q_offset, float scale,
                              bf16* out, float* lse, void* ws, size_t ws_bytes, int* err,
                              cudaStream_t st);

// ---- MXFP8 quantisation ------------------------------------------------------
// codes[dst(i), :d] / scales[dst(i), :d/group] of bf16 rows x[i, :d] (row pitch ld_x).
cudaError_t launch_mxfp8_quantize(const bf16* x, int64_t n_rows, int d, int64_t ld_x, int group,
                                  const int64_t* dst_rows, uint8_t* codes, uint8_t* scales,
                                  cudaStream_t st);

// ---- failure detection self-test (selftest.cu) ------------------------------
// One warp waits, with the given limit, on an mbarrier nothing arrives at:
// the timeout path of every bounded wait, run on purpose.
cudaError_t launch_selftest_wait_timeout(uint64_t limit_ns, int* err, cudaStream_t st);

}  // namespace dsi
