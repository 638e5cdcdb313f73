// Per-row Top-K selection: radix select in shared memory with the
// lower-position tie rule, then an order-preserving compaction.
//
// ("Day 0 Inference Support for New LLM Architectures: Optimization
// Practices", "Internal Fusion of the Indexer": Top-K completed on chip, only
// the selected indices leave the kernel.)
//
// One block per row.  Scores become order-preserving 32-bit keys; the search
// finds the exact K-th largest key T and how many keys equal to T must be kept
// (the lowest positions among them), then the kept positions are written
// ascending with block-wide prefix sums.
//
// Rows of up to 131072 positions (topk_rows_reg): 32768-position chunks, each
// warp holding 1024 consecutive positions of a chunk in registers; a row of
// one chunk stays in registers, longer rows reload their chunks from L2 for
// each pass.  The search narrows an interval [lo, hi]
// that holds T, starting from the row's min and max key: each pass splits the
// interval into 2048 equal bins (11 bits of the key range per pass, so at most
// three passes) and keeps the bin where the count from the top reaches K.
// Bins follow the keys' actual range, so the histogram atomics stay spread
// out even when most scores share their top bits.  The compaction ranks the
// warps once (per-warp counts) and then each warp walks its positions in
// order with ballots, so every store of a round is one contiguous run.
//
// Still longer rows (topk_rows): four 8-bit MSB-first histogram passes and a
// compaction walking the row in chunks; rows that fit are staged in shared
// memory once, longer ones re-read from global memory (L2) each pass.
#include "kernels.h"
#include "tc_common.cuh"

namespace dsi {

constexpr int kTopkThreads = 1024;
constexpr int kTopkItems = 4;                       // positions per thread per compaction step
constexpr int kTopkSmemKeys = 40 * 1024;            // keys staged in shared memory (160 KB)

__device__ __forceinline__ uint32_t load_key(const uint32_t* skeys, const float* grow, int64_t i) {
  return skeys ? skeys[i] : score_key(__ldg(grow + i));
}

__global__ void __launch_bounds__(kTopkThreads)
topk_rows(const float* __restrict__ scores, int64_t ld, int64_t n_cap,
          const int32_t* __restrict__ row_len, int64_t q_offset, int K, int32_t* __restrict__ idx,
          int32_t* __restrict__ count, int stage, int tps) {
  extern __shared__ uint32_t topk_smem[];
  __shared__ int hist[256];
  __shared__ int scan_ws[40];
  __shared__ uint32_t s_digit;
  __shared__ int s_krem;
  const int r = blockIdx.x;
  const int tid = threadIdx.x;
  int64_t n = !row_len ? q_offset + r + 1
              : tps == 1 ? (int64_t)row_len[r]
                         : (int64_t)row_len[r / tps] - (tps - 1 - r % tps);
  if (n < 0) n = 0;
  if (n > n_cap) n = n_cap;   // the scorer's visible length never exceeds it
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

constexpr int kRegPer = 32;                               // keys per thread
constexpr int kRegKeysMax = kTopkThreads * kRegPer;        // 32768 per chunk
constexpr int kRegChunks = 4;                              // rows up to 131072 positions
constexpr int kBins = 2048;                                // 11-bit digits of the key range
constexpr int kWarps = kTopkThreads / 32;
static_assert(kBins == 64 * kWarps, "each warp owns 64 bins in the bin search");

// Loads chunk c (32768 positions) of the row into the thread's registers.
__device__ __forceinline__ void load_chunk(uint32_t* key, const float* grow, int64_t n, int c,
                                           int wpos, int lane) {
#pragma unroll
  for (int i = 0; i < kRegPer; ++i) {
    const int64_t p = (int64_t)c * kRegKeysMax + wpos + 32 * i + lane;
    key[i] = p < n ? max(score_key(__ldg(grow + p)), 1u) : 0u;
  }
}

// The chosen bin [lo, hi] holds at most kRankMax of the CTA's keys: they are
// collected and ranked against each other (each lane counts the keys above
// and equal to its own), which gives T and the number of keys equal to T to
// take, without the passes that would narrow the bin to one value.  On return
// lo == hi == T and krem counts the keys equal to T to keep.
constexpr int kRankMax = 32;
constexpr int kPackRows = kTopkThreads;   // rows a packed cluster launch can order
template <int N>
__device__ __forceinline__ void rank_bin(const uint32_t (&key)[N], uint32_t& lo, uint32_t& hi,
                                         int& krem, uint32_t* cand, int* nc, uint32_t* sel,
                                         int tid, int lane, int wid) {
  const uint32_t span = hi - lo;
#pragma unroll
  for (int i = 0; i < N; ++i)
    if (key[i] - lo <= span) cand[atomicAdd(nc, 1)] = key[i];
  __syncthreads();
  if (wid == 0) {
    const int m = *nc;
    const uint32_t kv = lane < m ? cand[lane] : 0u;
    int g = 0, e = 0;
    for (int j = 0; j < m; ++j) {
      const uint32_t c = cand[j];
      g += c > kv;
      e += c == kv;
    }
    if (lane < m && g < krem && krem <= g + e) { sel[0] = kv; sel[1] = (uint32_t)g; }
  }
  __syncthreads();
  lo = hi = sel[0];
  krem -= (int)sel[1];
}

template <bool kChunked>
__global__ void __launch_bounds__(kTopkThreads, 1)
topk_rows_reg(const float* __restrict__ scores, int64_t ld, int64_t n_cap,
              const int32_t* __restrict__ row_len, int64_t q_offset, int K,
              int32_t* __restrict__ idx, int32_t* __restrict__ count, int tps) {
  __shared__ int hist[2][kBins];          // alternate passes; each is cleared as it is read
  __shared__ int wsum[2][kWarps];
  __shared__ int wbase[2][kWarps];
  __shared__ uint32_t s_sel[3];
  __shared__ uint32_t s_cand[kRankMax];
  __shared__ int s_nc;
  // the scores come from the previous kernel; the attention kernel after this
  // one may start its set-up now
  grid_dep_wait();
  grid_dep_launch();
  const int r = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const unsigned kAll = 0xffffffffu;
  const unsigned lt_mask = (1u << lane) - 1u;
  int64_t n = !row_len ? q_offset + r + 1
              : tps == 1 ? (int64_t)row_len[r]
                         : (int64_t)row_len[r / tps] - (tps - 1 - r % tps);
  if (n < 0) n = 0;
  if (n > n_cap) n = n_cap;   // the scorer's visible length never exceeds it
  int32_t* out = idx + (int64_t)r * K;
  const float* grow = scores + (int64_t)r * ld;
  if (n <= K) {  // every candidate is kept
    for (int64_t j = tid; j < K; j += blockDim.x) out[j] = j < n ? (int32_t)j : -1;
    if (count && tid == 0) count[r] = (int32_t)n;
    return;
  }
  // ---- keys: the row in chunks of 32768 positions; within a chunk warp w
  // holds positions 1024w .. 1024w+1023, in round i lane l position
  // 1024w + 32i + l (every load is one coalesced line per warp).  A row of one
  // chunk stays in registers throughout; longer rows reload each chunk per
  // pass (from L2).  Valid keys are at least 1 (every non-NaN score maps far
  // above it); slots past the row end hold 0, so they fall below every
  // interval searched and below T, and need no separate validity test.
  const int nchunks = kChunked ? (int)((n + kRegKeysMax - 1) / kRegKeysMax) : 1;
  const bool resident = !kChunked;
  const int wpos = wid * (kRegPer * 32);
  uint32_t key[kRegPer];
  if (resident) load_chunk(key, grow, n, 0, wpos, lane);
  for (int i = tid; i < 2 * kBins; i += blockDim.x) (&hist[0][0])[i] = 0;
  if (tid == 0) s_nc = 0;
  // ---- the row's key range ------------------------------------------------
  {
    uint32_t kmax = 0u, kmin = 0xffffffffu;
    for (int c = 0; c < nchunks; ++c) {
      if (!resident) load_chunk(key, grow, n, c, wpos, lane);
#pragma unroll
      for (int i = 0; i < kRegPer; ++i) {
        kmax = max(kmax, key[i]);
        kmin = min(kmin, key[i] == 0u ? 0xffffffffu : key[i]);
      }
    }
    kmax = __reduce_max_sync(kAll, kmax);
    kmin = __reduce_min_sync(kAll, kmin);
    if (lane == 0) { wsum[0][wid] = (int)kmax; wsum[1][wid] = (int)kmin; }
    __syncthreads();
    if (wid == 0) {
      kmax = __reduce_max_sync(kAll, (uint32_t)wsum[0][lane]);
      kmin = __reduce_min_sync(kAll, (uint32_t)wsum[1][lane]);
      if (lane == 0) { s_sel[0] = kmin; s_sel[1] = kmax; }
    }
    __syncthreads();
  }
  uint32_t lo = s_sel[0], hi = s_sel[1];
  int krem = K;   // keys to take from [lo, hi], counted from the top; T is in [lo, hi]
  // ---- narrow [lo, hi] to T, 11 bits of the range per pass -------------------
  int pass = 0;
#pragma unroll 1
  while (lo != hi) {
    const uint32_t span = hi - lo;
    const int bits = 32 - __clz(span);
    const int sh = bits > 11 ? bits - 11 : 0;          // bins of 2^sh keys cover [lo, hi]
    int* h = hist[pass & 1];
    for (int c = 0; c < nchunks; ++c) {
      if (!resident) load_chunk(key, grow, n, c, wpos, lane);
#pragma unroll
      for (int i = 0; i < kRegPer; ++i) {
        const uint32_t off = key[i] - lo;                 // wraps for keys below lo
        if (off <= span) atomicAdd(&h[off >> sh], 1);
      }
    }
    __syncthreads();
    // warp w owns bins 2047-64w down to 1984-64w, lane l the pair starting at
    // 2047-64w-2l; both are cleared for the pass after next
    const int b0 = kBins - 1 - 64 * wid - 2 * lane;
    const int c0 = h[b0], c1 = h[b0 - 1];
    h[b0] = 0;
    h[b0 - 1] = 0;
    int incl = c0 + c1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kAll, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[pass & 1][wid] = incl;
    __syncthreads();
    // keys in the bins of the warps above this one
    const int wt = wsum[pass & 1][lane];
    int wincl = wt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kAll, wincl, o);
      if (lane >= o) wincl += y;
    }
    const int above_w = __shfl_sync(kAll, wincl - wt, wid);
    const int above = above_w + incl - (c0 + c1);       // keys in the bins above this pair
    if (above < krem && above + c0 + c1 >= krem) {
      if (above + c0 >= krem) {
        s_sel[0] = (uint32_t)b0; s_sel[1] = (uint32_t)above; s_sel[2] = (uint32_t)c0;
      } else {
        s_sel[0] = (uint32_t)(b0 - 1); s_sel[1] = (uint32_t)(above + c0); s_sel[2] = (uint32_t)c1;
      }
    }
    __syncthreads();
    const uint32_t b = s_sel[0];
    krem -= (int)s_sel[1];
    const uint64_t top = (uint64_t)lo + ((uint64_t)(b + 1) << sh) - 1;
    lo += b << sh;
    hi = top < (uint64_t)hi ? (uint32_t)top : hi;
    ++pass;
    if (sh == 0) break;
    if (resident && s_sel[2] <= (uint32_t)kRankMax) {
      rank_bin(key, lo, hi, krem, s_cand, &s_nc, s_sel, tid, lane, wid);
      break;
    }
  }
  const uint32_t T = lo;
  // ---- ordered compaction, chunk by chunk -------------------------------------
  // per-warp counts of keys above T and equal to T; warp 0 turns them into
  // each warp's rank among equals and output offset, carrying both across
  // chunks (a chunk's positions all follow the previous chunk's)
  int eq_run = 0, sel_run = 0;           // warp 0: equals and kept keys in earlier chunks
  __syncthreads();                       // s_sel / wsum readers of the last pass are done
  for (int c = 0; c < nchunks; ++c) {
    if (!resident) load_chunk(key, grow, n, c, wpos, lane);
    int gt = 0, eq = 0;
#pragma unroll
    for (int i = 0; i < kRegPer; ++i) { gt += key[i] > T; eq += key[i] == T; }
    gt = __reduce_add_sync(kAll, gt);
    eq = __reduce_add_sync(kAll, eq);
    if (lane == 0) { wsum[0][wid] = gt; wsum[1][wid] = eq; }
    __syncthreads();
    if (wid == 0) {
      const int g = wsum[0][lane], e = wsum[1][lane];
      int ei = e;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kAll, ei, o);
        if (lane >= o) ei += y;
      }
      const int ebase = eq_run + ei - e;
      int take = krem - ebase;
      take = take < 0 ? 0 : (take > e ? e : take);
      const int sel = g + take;
      int si = sel;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kAll, si, o);
        if (lane >= o) si += y;
      }
      wbase[0][lane] = ebase;
      wbase[1][lane] = sel_run + si - sel;
      eq_run += __shfl_sync(kAll, ei, 31);
      sel_run += __shfl_sync(kAll, si, 31);
    }
    __syncthreads();
    int eq_rank = wbase[0][wid], pos = wbase[1][wid];
    const int cpos = c * kRegKeysMax + wpos;
    if (eq == 0) {                       // warp-uniform: no ties at T in this warp
#pragma unroll
      for (int i = 0; i < kRegPer; ++i) {
        const bool keep = key[i] > T;
        const unsigned km = __ballot_sync(kAll, keep);
        if (keep) out[pos + __popc(km & lt_mask)] = cpos + 32 * i + lane;
        pos += __popc(km);
      }
    } else {
#pragma unroll
      for (int i = 0; i < kRegPer; ++i) {
        const bool is_eq = key[i] == T;
        const unsigned em = __ballot_sync(kAll, is_eq);
        const bool keep = key[i] > T || (is_eq && eq_rank + __popc(em & lt_mask) < krem);
        const unsigned km = __ballot_sync(kAll, keep);
        if (keep) out[pos + __popc(km & lt_mask)] = cpos + 32 * i + lane;
        pos += __popc(km);
        eq_rank += __popc(em);
      }
    }
    __syncthreads();                     // wsum / wbase are rewritten for the next chunk
  }
  if (count && tid == 0) count[r] = K;
}

// ---------------------------------------------------------------------------
// Cluster form: the CL CTAs of a cluster share one row.  The row is cut into
// CL equal runs of kpt * 1024 positions (kpt <= KPT keys a thread, chosen per
// row from its length), CTA q holding run q in registers with the same
// warp-major layout as above.  Each pass every CTA histograms its own keys,
// and after a cluster barrier every CTA sums the CL histograms through
// distributed shared memory, so all of them take the same bin and the same
// number of passes.  The compaction offsets of run q are the kept counts of
// runs 0 .. q-1, read the same way.  A row that fits one CTA's registers
// (KPT keys a thread) is taken by CTA 0 alone, the others leave at once, so
// short rows cost one CTA.  Used when the rows are too few (or too long) to
// fill the GPU with one CTA each.
__device__ __forceinline__ int ld_peer_s32(const void* local, uint32_t rank) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];\n"
               : "=r"(v)
               : "r"(tc::map_to_rank(tc::smem_u32(local), rank))
               : "memory");
  return v;
}
// Two adjacent counters (8-byte aligned) of the same CTA of the cluster.
__device__ __forceinline__ int2 ld_peer_v2(const void* local, uint32_t rank) {
  int2 v;
  asm volatile("ld.shared::cluster.v2.s32 {%0, %1}, [%2];\n"
               : "=r"(v.x), "=r"(v.y)
               : "r"(tc::map_to_rank(tc::smem_u32(local), rank))
               : "memory");
  return v;
}

// rank_bin over the runs of all `parts` CTAs of the cluster: each collects its
// own keys of the bin, and warp 0 of every CTA gathers all of them (at most
// kRankMax) through distributed shared memory, so all take the same T.
template <int N>
__device__ __forceinline__ void rank_bin_cluster(const uint32_t (&key)[N], uint32_t& lo,
                                                 uint32_t& hi, int& krem, uint32_t* cand, int* nc,
                                                 uint32_t* sel, int parts, int lane, int wid) {
  const uint32_t span = hi - lo;
#pragma unroll
  for (int i = 0; i < N; ++i)
    if (key[i] - lo <= span) cand[atomicAdd(nc, 1)] = key[i];
  tc::cluster_sync();                    // every run's candidates in place
  if (wid == 0) {
    // lane l takes candidate l of the concatenated lists
    uint32_t kv = 0u;
    int m = 0;
    for (int rk = 0; rk < parts; ++rk) {
      const int mr = ld_peer_s32(nc, rk);
      if (lane >= m && lane < m + mr) kv = (uint32_t)ld_peer_s32(cand + (lane - m), rk);
      m += mr;
    }
    int g = 0, e = 0;
    for (int j = 0; j < m; ++j) {
      const uint32_t c = __shfl_sync(0xffffffffu, kv, j);
      g += c > kv;
      e += c == kv;
    }
    if (lane < m && g < krem && krem <= g + e) { sel[0] = kv; sel[1] = (uint32_t)g; }
  }
  __syncthreads();
  lo = hi = sel[0];
  krem -= (int)sel[1];
}

template <int CL, int KPT, bool PACK>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(kTopkThreads, 1)
topk_rows_cl(const float* __restrict__ scores, int64_t ld, int64_t n_cap,
             const int32_t* __restrict__ row_len, int64_t q_offset, int K,
             int32_t* __restrict__ idx, int32_t* __restrict__ count, int tps, int rows) {
  __shared__ __align__(16) int hist[2][kBins];   // alternate passes (the peers read both)
  __shared__ int wsum[2][kWarps];
  __shared__ int wbase[2][kWarps];
  __shared__ uint32_t s_sel[3];
  __shared__ uint32_t s_range[2];         // this CTA's smallest and largest key (peers read them)
  __shared__ uint32_t s_cand[kRankMax];
  __shared__ int s_nc;
  __shared__ int s_cnt[2];                // this CTA's keys above T and equal to T (peers read them)
  __shared__ int s_rows[PACK ? kPackRows : 1];   // PACK: the long rows in row order, then the others
  __shared__ int s_wl[kWarps];
  grid_dep_wait();
  grid_dep_launch();
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const unsigned kAll = 0xffffffffu;
  const unsigned lt_mask = (1u << lane) - 1u;
  const int qc = (int)tc::cluster_ctarank();
  auto row_n = [&](int rr) {
    int64_t v = !row_len ? q_offset + rr + 1
                : tps == 1 ? (int64_t)row_len[rr]
                           : (int64_t)row_len[rr / tps] - (tps - 1 - rr % tps);
    if (v < 0) v = 0;
    return v > n_cap ? n_cap : v;   // the scorer's visible length never exceeds it
  };
  // row of this cluster.  PACK: rows longer than one CTA's registers take a
  // cluster each (first, in row order), the others one CTA each, CL to a
  // cluster, so short rows do not hold the SMs of a whole cluster (every CTA
  // derives the same order from the row lengths)
  int r = blockIdx.x / CL;
  bool solo = false;                      // this CTA takes a row of its own
  if constexpr (PACK) {
    const bool lng = tid < rows && row_n(tid) > (int64_t)KPT * kTopkThreads;
    const unsigned bl = __ballot_sync(kAll, lng);
    if (lane == 0) s_wl[wid] = __popc(bl);
    __syncthreads();
    int lb = 0, nlong = 0;
    for (int w2 = 0; w2 < kWarps; ++w2) {
      lb += w2 < wid ? s_wl[w2] : 0;
      nlong += s_wl[w2];
    }
    if (tid < rows) {
      const int lp = lb + __popc(bl & lt_mask);
      s_rows[lng ? lp : nlong + tid - lp] = tid;
    }
    __syncthreads();
    const int cl = blockIdx.x / CL;
    if (cl >= nlong) {
      const int si = nlong + (cl - nlong) * CL + qc;
      if (si >= rows) return;
      r = s_rows[si];
      solo = true;
    } else {
      r = s_rows[cl];
    }
  }
  const int q = solo ? 0 : qc;            // this CTA's run of the row
  const int64_t n = row_n(r);
  int32_t* out = idx + (int64_t)r * K;
  const float* grow = scores + (int64_t)r * ld;
  if (n <= K) {  // every candidate is kept (the same decision in every CTA of the cluster)
    const int ncta = solo ? 1 : CL;
    for (int64_t j = q * kTopkThreads + tid; j < K; j += ncta * kTopkThreads)
      out[j] = j < n ? (int32_t)j : -1;
    if (count && q == 0 && tid == 0) count[r] = (int32_t)n;
    return;
  }
  // ---- this CTA's run of the row: kpt keys a thread --------------------------
  // coop: the CL CTAs share the row; otherwise one CTA takes it alone (a
  // decision every CTA of the cluster makes the same way)
  const bool coop = !solo && n > (int64_t)KPT * kTopkThreads;
  if (!coop && !solo && q != 0) return;
  const int parts = coop ? CL : 1;
  const int kpt = (int)((n + parts * kTopkThreads - 1) / (parts * kTopkThreads));   // <= KPT
  const int64_t run0 = (int64_t)q * kpt * kTopkThreads;
  const int64_t wpos = run0 + (int64_t)wid * kpt * 32;
  uint32_t key[KPT];
#pragma unroll
  for (int i = 0; i < KPT; ++i) {
    const int64_t p = wpos + 32 * i + lane;
    key[i] = (i < kpt && p < n) ? max(score_key(__ldg(grow + p)), 1u) : 0u;
  }
  for (int i = tid; i < 2 * kBins; i += blockDim.x) (&hist[0][0])[i] = 0;
  if (tid == 0) s_nc = 0;
  {
    uint32_t kmax = 0u, kmin = 0xffffffffu;
#pragma unroll
    for (int i = 0; i < KPT; ++i) {
      kmax = max(kmax, key[i]);
      kmin = min(kmin, key[i] == 0u ? 0xffffffffu : key[i]);
    }
    kmax = __reduce_max_sync(kAll, kmax);
    kmin = __reduce_min_sync(kAll, kmin);
    if (lane == 0) { wsum[0][wid] = (int)kmax; wsum[1][wid] = (int)kmin; }
    __syncthreads();
    if (wid == 0) {
      kmax = __reduce_max_sync(kAll, (uint32_t)wsum[0][lane]);
      kmin = __reduce_min_sync(kAll, (uint32_t)wsum[1][lane]);
      if (lane == 0) { s_range[0] = kmin; s_range[1] = kmax; }
    }
  }
  // every CTA's range (and cleared histograms) in place
  if (coop) tc::cluster_sync(); else __syncthreads();
  if (wid == 0) {
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    if (lane < parts) {
      // the cluster's runs, or (a CTA alone on its row) this CTA's own range:
      // a CTA alone never reads another CTA's shared memory, which may belong
      // to another row or be gone
      const uint32_t rk = coop ? (uint32_t)lane : (uint32_t)qc;
      kmin = (uint32_t)ld_peer_s32(&s_range[0], rk);
      kmax = (uint32_t)ld_peer_s32(&s_range[1], rk);
    }
    kmin = __reduce_min_sync(kAll, kmin);
    kmax = __reduce_max_sync(kAll, kmax);
    if (lane == 0) { s_sel[0] = kmin; s_sel[1] = kmax; }
  }
  __syncthreads();
  uint32_t lo = s_sel[0], hi = s_sel[1];
  int krem = K;
  // ---- narrow [lo, hi] to T over the cluster's summed histograms --------------
  int pass = 0;
#pragma unroll 1
  while (lo != hi) {
    const uint32_t span = hi - lo;
    const int bits = 32 - __clz(span);
    const int sh = bits > 11 ? bits - 11 : 0;
    int* h = hist[pass & 1];
#pragma unroll
    for (int i = 0; i < KPT; ++i) {
      const uint32_t off = key[i] - lo;
      if (off <= span) atomicAdd(&h[off >> sh], 1);
    }
    // every CTA's histogram of this pass is complete, and every CTA is done
    // reading the previous pass's buffer, which is cleared for the next pass
    if (coop) tc::cluster_sync(); else __syncthreads();
    {
      int* hp = hist[(pass + 1) & 1];
      hp[tid] = 0;
      hp[tid + kTopkThreads] = 0;
    }
    const int b0 = kBins - 1 - 64 * wid - 2 * lane;
    int c0 = 0, c1 = 0;
    if (coop) {
#pragma unroll
      for (int rk = 0; rk < CL; ++rk) {
        const int2 v = ld_peer_v2(&h[b0 - 1], rk);
        c0 += v.y;
        c1 += v.x;
      }
    } else {
      c0 = h[b0];
      c1 = h[b0 - 1];
    }
    int incl = c0 + c1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kAll, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[pass & 1][wid] = incl;
    __syncthreads();
    const int wt = wsum[pass & 1][lane];
    int wincl = wt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kAll, wincl, o);
      if (lane >= o) wincl += y;
    }
    const int above_w = __shfl_sync(kAll, wincl - wt, wid);
    const int above = above_w + incl - (c0 + c1);
    if (above < krem && above + c0 + c1 >= krem) {
      if (above + c0 >= krem) {
        s_sel[0] = (uint32_t)b0; s_sel[1] = (uint32_t)above; s_sel[2] = (uint32_t)c0;
      } else {
        s_sel[0] = (uint32_t)(b0 - 1); s_sel[1] = (uint32_t)(above + c0); s_sel[2] = (uint32_t)c1;
      }
    }
    __syncthreads();
    const uint32_t b = s_sel[0];
    krem -= (int)s_sel[1];
    const uint64_t top = (uint64_t)lo + ((uint64_t)(b + 1) << sh) - 1;
    lo += b << sh;
    hi = top < (uint64_t)hi ? (uint32_t)top : hi;
    ++pass;
    if (sh == 0) break;
    // a chosen bin of few keys: rank them directly (the counts are the
    // cluster's sums, so every CTA of it decides the same way; on four-CTA
    // clusters gathering the candidates measured slower than narrowing on)
    if (s_sel[2] <= (uint32_t)kRankMax && (!coop || CL == 2)) {
      if (coop) rank_bin_cluster(key, lo, hi, krem, s_cand, &s_nc, s_sel, parts, lane, wid);
      else rank_bin(key, lo, hi, krem, s_cand, &s_nc, s_sel, tid, lane, wid);
      break;
    }
  }
  const uint32_t T = lo;
  // ---- ordered compaction: this run's offsets follow runs 0 .. q-1 -----------
  int gt = 0, eq = 0;
#pragma unroll
  for (int i = 0; i < KPT; ++i) { gt += key[i] > T; eq += key[i] == T; }
  gt = __reduce_add_sync(kAll, gt);
  eq = __reduce_add_sync(kAll, eq);
  __syncthreads();                       // s_sel / wsum readers of the last pass are done
  if (lane == 0) { wsum[0][wid] = gt; wsum[1][wid] = eq; }
  __syncthreads();
  if (wid == 0) {
    const int gs = __reduce_add_sync(kAll, wsum[0][lane]);
    const int es = __reduce_add_sync(kAll, wsum[1][lane]);
    if (lane == 0) { s_cnt[0] = gs; s_cnt[1] = es; }
  }
  if (coop) tc::cluster_sync();          // every run's counts in place
  else __syncthreads();
  if (wid == 0) {
    int eq_run = 0, sel_run = 0;         // equals and kept keys of the runs before this one
    for (int rk = 0; rk < q; ++rk) {
      const int g = ld_peer_s32(&s_cnt[0], rk), e = ld_peer_s32(&s_cnt[1], rk);
      int take = krem - eq_run;
      take = take < 0 ? 0 : (take > e ? e : take);
      sel_run += g + take;
      eq_run += e;
    }
    const int g = wsum[0][lane], e = wsum[1][lane];
    int ei = e;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kAll, ei, o);
      if (lane >= o) ei += y;
    }
    const int ebase = eq_run + ei - e;
    int take = krem - ebase;
    take = take < 0 ? 0 : (take > e ? e : take);
    const int sel = g + take;
    int si = sel;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kAll, si, o);
      if (lane >= o) si += y;
    }
    wbase[0][lane] = ebase;
    wbase[1][lane] = sel_run + si - sel;
  }
  if (coop) tc::cluster_sync();          // no peer reads this CTA's shared memory past here
  else __syncthreads();
  int eq_rank = wbase[0][wid], pos = wbase[1][wid];
  if (eq == 0) {                         // warp-uniform: no ties at T in this warp
#pragma unroll
    for (int i = 0; i < KPT; ++i) {
      const bool keep = key[i] > T;
      const unsigned km = __ballot_sync(kAll, keep);
      if (keep) out[pos + __popc(km & lt_mask)] = (int32_t)(wpos + 32 * i + lane);
      pos += __popc(km);
    }
  } else {
#pragma unroll
    for (int i = 0; i < KPT; ++i) {
      const bool is_eq = key[i] == T;
      const unsigned em = __ballot_sync(kAll, is_eq);
      const bool keep = key[i] > T || (is_eq && eq_rank + __popc(em & lt_mask) < krem);
      const unsigned km = __ballot_sync(kAll, keep);
      if (keep) out[pos + __popc(km & lt_mask)] = (int32_t)(wpos + 32 * i + lane);
      pos += __popc(km);
      eq_rank += __popc(em);
    }
  }
  if (count && q == 0 && tid == 0) count[r] = K;
}

cudaError_t launch_topk(const float* scores, int64_t ld, int rows, const int32_t* row_len,
                        int64_t q_offset, int K, int32_t* idx, int32_t* count, cudaStream_t st,
                        int tps, int64_t n_cap) {
  if (rows <= 0) return cudaSuccess;
  n_cap = (n_cap < 0 || n_cap > ld) ? ld : n_cap;
  const int64_t longest = row_len ? n_cap : (q_offset + rows < n_cap ? q_offset + rows : n_cap);
  if (longest <= kRegChunks * kRegKeysMax) {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaError_t e;
    if (longest <= kRegKeysMax) {
      // rows of one chunk: two CTAs a row while that still fits in one wave
      e = 2L * rows <= sms
              ? launch_overlapped(topk_rows_cl<2, kRegPer / 2, false>, dim3(2 * rows),
                                  dim3(kTopkThreads), 0, st, scores, ld, n_cap, row_len, q_offset,
                                  K, idx, count, tps, rows)
              : launch_overlapped(topk_rows_reg<false>, dim3(rows), dim3(kTopkThreads), 0, st,
                                  scores, ld, n_cap, row_len, q_offset, K, idx, count, tps);
    } else {
      // longer rows: four CTAs a row hold up to 131072 keys in registers
      e = (long)rows <= 2L * sms && rows <= kPackRows
              ? launch_overlapped(topk_rows_cl<4, kRegPer, true>, dim3(4 * rows),
                                  dim3(kTopkThreads), 0, st, scores, ld, n_cap, row_len, q_offset,
                                  K, idx, count, tps, rows)
              : launch_overlapped(topk_rows_reg<true>, dim3(rows), dim3(kTopkThreads), 0, st,
                                  scores, ld, n_cap, row_len, q_offset, K, idx, count, tps);
    }
    note_launch();
    return e;
  }
  // stage rows in shared memory when the longest possible row fits
  const int stage = longest <= kTopkSmemKeys;
  const size_t smem = stage ? (size_t)longest * sizeof(uint32_t) : 0;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(topk_rows, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  topk_rows<<<rows, kTopkThreads, smem, st>>>(scores, ld, n_cap, row_len, q_offset, K, idx, count,
                                                stage, tps);
  note_launch();
  return cudaGetLastError();
}

}  // namespace dsi
