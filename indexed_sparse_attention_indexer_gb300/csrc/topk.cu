// Per-row Top-K selection: radix select in shared memory with the
// lower-position tie rule, then an order-preserving compaction.
//
// ("Day 0 Inference Support for New LLM Architectures: Optimization
// Practices", "Internal Fusion of the Indexer": Top-K completed on chip, only
// the selected indices leave the kernel.)
//
// One block per row.  Scores become order-preserving 32-bit keys.  Four
// 8-bit MSB-first histogram passes find the exact K-th largest key T and how
// many keys equal to T must be kept (the lowest positions among them).  A
// final pass walks the row in position order with block-wide prefix sums and
// writes the kept positions ascending.  Rows that fit are staged in shared
// memory once; longer rows are re-read from global memory (L2) each pass.
#include "kernels.h"

namespace dsi {

constexpr int kTopkThreads = 1024;
constexpr int kTopkItems = 4;                       // positions per thread per compaction step
constexpr int kTopkSmemKeys = 40 * 1024;            // keys staged in shared memory (160 KB)

__device__ __forceinline__ uint32_t load_key(const uint32_t* skeys, const float* grow, int64_t i) {
  return skeys ? skeys[i] : score_key(__ldg(grow + i));
}

__global__ void __launch_bounds__(kTopkThreads)
topk_rows(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ row_len,
          int64_t q_offset, int K, int32_t* __restrict__ idx, int32_t* __restrict__ count,
          int stage) {
  extern __shared__ uint32_t topk_smem[];
  __shared__ int hist[256];
  __shared__ int scan_ws[40];
  __shared__ uint32_t s_digit;
  __shared__ int s_krem;
  const int r = blockIdx.x;
  const int tid = threadIdx.x;
  int64_t n = row_len ? (int64_t)row_len[r] : q_offset + r + 1;
  if (n < 0) n = 0;
  if (n > ld) n = ld;
  int32_t* out = idx + (int64_t)r * K;
  const float* grow = scores + (int64_t)r * ld;

  if (n <= K) {  // every candidate is kept
    for (int64_t j = tid; j < K; j += blockDim.x) out[j] = j < n ? (int32_t)j : -1;
    if (count && tid == 0) count[r] = (int32_t)n;
    return;
  }
  uint32_t* skeys = nullptr;
  if (stage && n <= kTopkSmemKeys) {
    skeys = topk_smem;
    for (int64_t j = tid; j < n; j += blockDim.x) skeys[j] = score_key(__ldg(grow + j));
  }
  // ---- radix select of the K-th largest key --------------------------------
  uint32_t prefix = 0, mask = 0;
  int krem = K;  // how many keys still to take within the current prefix
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int64_t j = tid; j < n; j += blockDim.x) {
      const uint32_t k = load_key(skeys, grow, j);
      if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1);
    }
    __syncthreads();
    if (tid < 32) {
      // warp 0: find the digit where the count of larger-or-equal digits reaches krem
      int c[8];
      int tot = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) { c[e] = hist[255 - (tid * 8 + e)]; tot += c[e]; }
      int incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (tid >= o) incl += y;
      }
      int excl = incl - tot;  // keys in digits above this lane's 8 digits
      if (excl < krem && incl >= krem) {
        int run = excl;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (run < krem && run + c[e] >= krem) {
            s_digit = 255u - (uint32_t)(tid * 8 + e);
            s_krem = krem - run;
          }
          run += c[e];
        }
      }
    }
    __syncthreads();
    prefix |= s_digit << shift;
    mask |= 255u << shift;
    krem = s_krem;
    __syncthreads();
  }
  // prefix = T (the K-th largest key); krem = number of keys == T to keep.
  const uint32_t T = prefix;
  // ---- ordered compaction ---------------------------------------------------
  int eq_seen = 0, written = 0;
  const int64_t chunk = (int64_t)blockDim.x * kTopkItems;
#pragma unroll 1
  for (int64_t base = 0; base < n && written < K; base += chunk) {
    const int64_t j0 = base + (int64_t)tid * kTopkItems;
    uint32_t kk[kTopkItems];
    int gt = 0, eq = 0;
#pragma unroll
    for (int e = 0; e < kTopkItems; ++e) {
      const int64_t j = j0 + e;
      kk[e] = j < n ? load_key(skeys, grow, j) : 0u;
      if (j < n) { gt += kk[e] > T; eq += kk[e] == T; }
    }
    int eq_tot;
    const int eq_before = eq_seen + block_exclusive_scan(eq, scan_ws, eq_tot);
    // keys equal to T are kept while their rank among equals is < krem
    int take_eq = krem - eq_before;
    take_eq = take_eq < 0 ? 0 : (take_eq > eq ? eq : take_eq);
    int sel_tot;
    int pos = written + block_exclusive_scan(gt + take_eq, scan_ws, sel_tot);
    int eq_rank = eq_before;
#pragma unroll
    for (int e = 0; e < kTopkItems; ++e) {
      const int64_t j = j0 + e;
      if (j < n) {
        bool keep = kk[e] > T;
        if (kk[e] == T) { keep = eq_rank < krem; ++eq_rank; }
        if (keep) out[pos++] = (int32_t)j;
      }
    }
    eq_seen += eq_tot;
    written += sel_tot;
  }
  if (count && tid == 0) count[r] = K;
}

cudaError_t launch_topk(const float* scores, int64_t ld, int rows, const int32_t* row_len,
                        int64_t q_offset, int K, int32_t* idx, int32_t* count, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  // stage rows in shared memory when the longest possible row fits
  const int64_t longest = row_len ? ld : (q_offset + rows < ld ? q_offset + rows : ld);
  const int stage = longest <= kTopkSmemKeys;
  const size_t smem = stage ? (size_t)longest * sizeof(uint32_t) : 0;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(topk_rows, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  topk_rows<<<rows, kTopkThreads, smem, st>>>(scores, ld, row_len, q_offset, K, idx, count, stage);
  note_launch();
  return cudaGetLastError();
}

}  // namespace dsi
