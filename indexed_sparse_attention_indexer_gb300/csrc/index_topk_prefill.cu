// Fused prefill indexer: tcgen05 scoring with ReLU, head weights and a running
// per-row Top-K in the epilogue; only the selected indices leave the kernel.
//
// ("Day 0 Inference Support for New LLM Architectures: Optimization
// Practices", "Internal Fusion of the Indexer": scoring, head-weight
// weighting and Top-K in one kernel that writes only the selected indices;
// "Load Imbalance in Causal Indexing and the Zigzag Layout": later positions
// have more history, so early and late segments are paired.)
//
// Work unit = a group of 2 query tokens (N = 2 x 64 heads).  Each CTA owns
// whole groups, taken in zigzag pairs (group i with group G-1-i), so every row
// is selected by one CTA and the causal triangle balances across CTAs.  For a
// group, the 128-position key tiles stream through TMA stages into
// tcgen05.mma (as in the scoring kernel); the epilogue computes the fp32
// scores, and each token keeps a candidate buffer in shared memory of unique
// 64-bit keys (order-preserving score key << 32 | ~position): larger key =
// larger score, then lower position, so ties need no special handling.  A
// candidate is kept when its key beats the current threshold (the K-th best
// key of the last compaction); when a buffer nears capacity the token's 128
// threads radix-select the K-th key and compact the buffer to the best K.
// At the end of the group a final select picks the K best, and their
// positions are written in ascending order through a bitmap prefix scan.
// A row whose history holds at most K positions selects all of them whatever
// the scores, so the leading rows of a prefill (up to K - q_offset of them)
// are not scored: a small kernel launched just before writes their positions
// in order, and the groups cover the remaining rows only.
#include <algorithm>

#include "kernels.h"
#include "tc_common.cuh"
#include "tma_host.h"

namespace dsi {
using namespace tc;

namespace {

constexpr int kD = 128;
constexpr int kHeads = 64;
constexpr int kTileM = 128;
constexpr int kSub = 64;
constexpr int NT = 2;                        // tokens per group
constexpr int N = NT * kHeads;               // 128
constexpr int kStages = 3;                   // key tiles in flight (L2 latency per tile)
constexpr int kQSlots = 1;                   // the next group's queries load while the epilogue selects
constexpr int A_BYTES = kTileM * kD * 2;     // 32 KB
constexpr int B_BYTES = N * kD * 2;          // 32 KB
constexpr int kCap = 4096;                   // candidates per token
constexpr int kMaxK = kCap / 2;              // 2048
constexpr int kMaxRow = kCap * 64 / 2;       // bitmap of a row fits the 32 KB buffer: 131072 positions
constexpr int EPI_WARPS = 16;                // 8 per token: two sets of 4 taking alternate tiles
constexpr int TOKT = 256;                    // threads per token (both sets)
constexpr int EPI_THREADS = EPI_WARPS * 32;
// MMA issuers: warp 1 and the last warp take alternate tiles (a thread
// issuing tcgen05.mma back to back waits ~120 cycles per instruction; two
// issuing at once halve the eight-MMA tile's issue time)
constexpr int kMmaWarps = 2;

constexpr int kMmaWarp1 = 2 + EPI_WARPS;     // the second issuer
constexpr int THREADS = 64 + EPI_THREADS + 32 * (kMmaWarps - 1);   // 608
constexpr int kAccBufs = 4;                  // score accumulators in TMEM
constexpr int TMEM_COLS = kAccBufs * N;      // 512
// an issuer reuses only accumulators it used last (parity waits)
static_assert(kAccBufs % kMmaWarps == 0, "issuer phases");
constexpr uint32_t IDESC = idesc_f32(1, kTileM, N);

constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + kStages * A_BYTES;
constexpr int OFF_BUF = OFF_B + kQSlots * B_BYTES;              // NT x kCap x 8 bytes
constexpr int OFF_W = OFF_BUF + NT * kCap * 8;                  // NT x 64 fp32
constexpr int kSelBits = 11;
constexpr int kSelBins = 1 << kSelBits;                         // select histogram bins
constexpr int kRankMax = 128;                                   // bin size ranked directly
constexpr int kHistInts = kSelBins + 32;                        // + reduction scratch
constexpr int OFF_HIST = OFF_W + NT * kHeads * 4;               // NT x kHistInts int
constexpr int OFF_TOK = OFF_HIST + NT * kHistInts * 4;          // per-token state
constexpr int OFF_BAR = (OFF_TOK + NT * 64 + 7) & ~7;
constexpr int NBARS = 2 * kStages + 2 * kAccBufs + 2 * kQSlots + 1;
constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
constexpr int SMEM = OFF_MISC + 64 + 1024;
static_assert(SMEM <= 227 * 1024, "shared memory");

struct TokState {
  unsigned long long theta;   // keys <= theta are rejected
  unsigned long long lo, hi;  // select scratch
  int cnt;                    // candidates in the buffer
  int digit;                  // select scratch
  int krem;
  int total;
  int stop;                   // set (never cleared) when a wait failed: the token's threads leave
  int cnt2;                   // select scratch: keys collected from the final bin
};
static_assert(sizeof(TokState) <= 64, "token state");

struct Args {
  const bf16* q_idx;
  const float* w;
  int32_t* idx;
  int32_t* count;
  int64_t q_offset;
  int rows;
  int K;
  int groups;
  int pairs_per_cta;   // zigzag pairs handled by each CTA (ceil)
};

// Two independent fp32 FMAs in one instruction (each rounded as fmaf would).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  uint64_t ra, rb, rc, rd;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rc) : "f"(c.x), "f"(c.y));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
  float2 d;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
  return d;
}

__device__ __forceinline__ void bar_tok(int tk) {    // the TOKT threads of one token
  asm volatile("bar.sync %0, %1;\n" ::"r"(2 + tk), "n"(TOKT) : "memory");
}

// k-th group (0-based) processed by CTA `cta`: zigzag pairs (i, G-1-i), pairs
// dealt round-robin over the CTAs.  Returns -1 past the end.
__device__ __forceinline__ int zigzag_group(int k, int cta, int ncta, int G) {
  const int pair = cta + (k >> 1) * ncta;
  const int npairs = (G + 1) / 2;
  if (pair >= npairs) return -1;
  const int g = (k & 1) ? G - 1 - pair : pair;
  if ((k & 1) && g == pair) return -1;             // middle group of an odd count
  return g;
}

__device__ __forceinline__ int group_tiles(const Args& a, int g) {
  const int last = min(a.rows, (g + 1) * NT) - 1;
  return (int)((a.q_offset + last + 1 + kTileM - 1) / kTileM);
}

// Select over the token's candidate buffer: the k-th largest key (keys are
// unique).  128 threads of the token (tt = 0..127) take part.  An interval
// [lo, hi] holding the answer starts at the candidates' min and max; each pass
// splits it into kSelBins equal bins and keeps the bin where the count from
// the top reaches k.  Bins follow the keys' actual spread, so the histogram
// atomics do not pile onto a few addresses the way fixed top digits of
// similar scores would.  Once the chosen bin holds at most kRankMax keys, they
// are collected and ranked against each other directly (each thread counts
// the keys above its own), which ends the search without further passes.
__device__ unsigned long long select_kth(const unsigned long long* buf, int n, int k, int* hist,
                                         TokState* ts, int tt, int tk) {
  const int lane = tt & 31, wq = tt >> 5;
  const unsigned kAll = 0xffffffffu;
  unsigned long long mn = ~0ull, mx = 0ull;
#pragma unroll 4
  for (int i = tt; i < n; i += TOKT) {
    const unsigned long long c = buf[i];
    mn = c < mn ? c : mn;
    mx = c > mx ? c : mx;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const unsigned long long a = __shfl_xor_sync(kAll, mn, o), b = __shfl_xor_sync(kAll, mx, o);
    mn = a < mn ? a : mn;
    mx = b > mx ? b : mx;
  }
  constexpr int kW = TOKT / 32;                  // warps of the token
  unsigned long long* red = reinterpret_cast<unsigned long long*>(hist + kSelBins);   // 2 kW words
  if (lane == 0) { red[wq] = mn; red[kW + wq] = mx; }
  bar_tok(tk);
  if (tt == 0) {
    unsigned long long l = red[0], h = red[kW];
    for (int x = 1; x < kW; ++x) { l = red[x] < l ? red[x] : l; h = red[kW + x] > h ? red[kW + x] : h; }
    ts->lo = l;
    ts->hi = h;
  }
  bar_tok(tk);
  unsigned long long lo = ts->lo, hi = ts->hi;
  int krem = k;
  bar_tok(tk);
  while (lo != hi) {
    const unsigned long long span = hi - lo;
    const int bits = 64 - __clzll((long long)span);
    const int sh = bits > kSelBits ? bits - kSelBits : 0;
    for (int i = tt; i < kSelBins; i += TOKT) hist[i] = 0;
    bar_tok(tk);
#pragma unroll 4
    for (int i = tt; i < n; i += TOKT) {
      const unsigned long long off = buf[i] - lo;         // wraps for keys below lo
      if (off <= span) atomicAdd(&hist[(int)(off >> sh)], 1);
    }
    bar_tok(tk);
    // thread tt owns bins kSelBins-1-kPerT*tt down to kSelBins-kPerT-kPerT*tt
    constexpr int kPerT = kSelBins / TOKT;
    int cs[kPerT], tot = 0;
#pragma unroll
    for (int e = 0; e < kPerT; ++e) { cs[e] = hist[kSelBins - 1 - kPerT * tt - e]; tot += cs[e]; }
    int incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kAll, incl, o);
      if (lane >= o) incl += y;
    }
    int* wsum = hist + kSelBins + 16;
    if (lane == 31) wsum[wq] = incl;
    bar_tok(tk);
    int above = incl - tot;
    for (int x = 0; x < wq; ++x) above += wsum[x];
    if (above < krem && above + tot >= krem) {
      int run = above;
#pragma unroll
      for (int e = 0; e < kPerT; ++e) {
        if (run < krem && run + cs[e] >= krem) {
          ts->digit = kSelBins - 1 - kPerT * tt - e;
          ts->krem = krem - run;
          ts->total = cs[e];
        }
        run += cs[e];
      }
    }
    bar_tok(tk);
    const unsigned long long b = (unsigned long long)ts->digit;
    const int in_bin = ts->total;
    krem = ts->krem;
    const unsigned long long t1 = (b << sh) + ((1ull << sh) - 1ull);
    hi = t1 > span ? hi : lo + t1;
    lo += b << sh;
    bar_tok(tk);
    if (sh == 0) break;
    if (in_bin <= kRankMax) {
      // collect the bin's keys (unique) and rank them: the key with exactly
      // krem-1 larger keys in the bin is the k-th of the buffer
      unsigned long long* small = reinterpret_cast<unsigned long long*>(hist);
      if (tt == 0) ts->cnt2 = 0;
      bar_tok(tk);
      for (int i = tt; i < n; i += TOKT) {
        const unsigned long long c = buf[i];
        if (c >= lo && c <= hi) small[atomicAdd(&ts->cnt2, 1)] = c;
      }
      bar_tok(tk);
      const int m = ts->cnt2;
      if (tt < m) {
        const unsigned long long mine = small[tt];
        int above = 0;
        for (int x = 0; x < m; ++x) above += small[x] > mine ? 1 : 0;
        if (above == krem - 1) ts->lo = mine;
      }
      bar_tok(tk);
      lo = ts->lo;
      bar_tok(tk);
      break;
    }
  }
  return lo;
}

// Keep the entries >= t (exactly k of them) at the front of the buffer.
__device__ void compact_ge(unsigned long long* buf, int n, unsigned long long t, TokState* ts,
                           int tt, int tk) {
  constexpr int PER = kCap / TOKT;
  unsigned long long keep[PER];
  int nk = 0;
  for (int i = tt, e = 0; e < PER; i += TOKT, ++e) {
    const unsigned long long c = i < n ? buf[i] : 0ull;
    keep[e] = c;
    nk += (i < n && c >= t) ? 1 : 0;
  }
  if (tt == 0) ts->total = 0;
  bar_tok(tk);
  int base = nk ? atomicAdd(&ts->total, nk) : 0;
  bar_tok(tk);
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const int i = tt + e * TOKT;
    if (i < n && keep[e] >= t) buf[base++] = keep[e];
  }
  bar_tok(tk);
}

__global__ void __launch_bounds__(THREADS, 1)
index_topk_prefill(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                   CacheView c, Args a, int* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  grid_dep_wait();   // inputs may come from the kernel launched just before
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* acc_full = bars + 2 * kStages;
  uint64_t* acc_empty = acc_full + kAccBufs;
  uint64_t* q_full = acc_empty + kAccBufs;
  uint64_t* q_empty = q_full + kQSlots;
  uint64_t* done_bar = q_empty + kQSlots;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int i = 0; i < kAccBufs; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], NT * 128);   // one warp set (4 warps) of each token reads a tile
    }
    for (int i = 0; i < kQSlots; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], kMmaWarps);
    }
    mbar_init(done_bar, kMmaWarps);
    *abort_flag = 0;
    for (int i = 0; i < NT; ++i) reinterpret_cast<TokState*>(smem + OFF_TOK)[i].stop = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int nmax = 2 * a.pairs_per_cta;   // groups this CTA may own

  if (warp == 0) {
    // ======================= TMA producer =====================================
    if (lane == 0) {
      prefetch_tmap(&kmap);
      prefetch_tmap(&qmap);
      int stage = 0, qcount = 0, n_issued = 0;
      uint32_t ph = 0;
      bool ok = true;
      // contiguous keys: a tile is one 128-row box per 64-dim block (rows past
      // the group's history are read and masked by the epilogue); paged:
      // 64-row boxes through the block table.  The rows are worked out before
      // the stage wait: one thread issues every tile, so its instruction
      // latency bounds the tile rate.
      const bool whole = c.block_table == nullptr;
      for (int k = 0; ok && k < nmax; ++k) {
        const int g = zigzag_group(k, blockIdx.x, gridDim.x, a.groups);
        if (g < 0) continue;
        const int slot = qcount % kQSlots;
        if (!(ok = mbar_wait(&q_empty[slot], ((qcount / kQSlots) & 1) ^ 1, abort_flag, err))) break;
        uint8_t* qs = smem + OFF_B + slot * B_BYTES;
        mbar_arrive_expect_tx(&q_full[slot], B_BYTES);
        for (int t = 0; t < NT; ++t)
          for (int cc = 0; cc < 2; ++cc)
            tma_load_2d(qs + cc * (N * 128) + t * kHeads * 128, &qmap, cc * 64, (g * NT + t) * kHeads,
                        &q_full[slot]);
        ++qcount;
        const int ntile = group_tiles(a, g);
        const int64_t nvis = a.q_offset + min(a.rows, (g + 1) * NT);
        for (int j = 0; j < ntile; ++j) {
          int nsub = 2;
          int64_t prow[2];
          prow[0] = (int64_t)j * kTileM;
          prow[1] = prow[0] + kSub;
          if (!whole) {
            nsub = 0;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const int64_t p = (int64_t)j * kTileM + i * kSub;
              prow[i] = -1;
              if (p < nvis) { prow[i] = phys_row(c, 0, p, err); if (prow[i] >= 0) ++nsub; }
            }
          }
          if (!(ok = mbar_wait(&empty[stage], ph ^ 1, abort_flag, err))) break;
          uint8_t* as = smem + OFF_A + stage * A_BYTES;
          mbar_arrive_expect_tx(&full[stage], (uint32_t)(nsub * (A_BYTES / 2)));
          if (whole) {
            tma_load_2d(as, &kmap, 0, (int)prow[0], &full[stage]);
            tma_load_2d(as + 16384, &kmap, 64, (int)prow[0], &full[stage]);
          } else {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              if (prow[i] < 0) continue;
              tma_load_2d(as + i * (kSub * 128), &kmap, 0, (int)prow[i], &full[stage]);
              tma_load_2d(as + 16384 + i * (kSub * 128), &kmap, 64, (int)prow[i], &full[stage]);
            }
          }
          ++n_issued;
          if (++stage == kStages) { stage = 0; ph ^= 1; }
        }
      }
      // after an abort, wait (bounded by time) for the last tiles' copies
      if (*abort_flag) {
        volatile int no_abort = 0;
        for (int t = max(0, n_issued - kStages); t < n_issued; ++t)
          mbar_wait(&full[t % kStages], (uint32_t)((t / kStages) & 1), &no_abort, err, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 1 || warp == kMmaWarp1) {
    // ======================= MMA issuer ========================================
    // Issuer mw takes the CTA's tiles kt = mw, mw + 2, ...; both wait for a
    // group's queries and both release them (a commit after its own MMAs on
    // them, else a plain arrival).
    const int mw = warp == 1 ? 0 : 1;
    if (lane == 0) {
      int stage = 0, abuf = 0, qcount = 0, kt = 0;
      uint32_t ph = 0, aph = 0;
      bool ok = true, any = false;
      for (int k = 0; ok && k < nmax; ++k) {
        const int g = zigzag_group(k, blockIdx.x, gridDim.x, a.groups);
        if (g < 0) continue;
        const int slot = qcount % kQSlots;
        if (!(ok = mbar_wait(&q_full[slot], (qcount / kQSlots) & 1, abort_flag, err))) break;
        ++qcount;
        const int ntile = group_tiles(a, g);
        bool used = false;
        for (int j = 0; j < ntile; ++j, ++kt) {
          if (kt % kMmaWarps != mw) {
            // the other issuer's tile: wait for its keys all the same.  With
            // an odd stage count the stages alternate between the issuers, and
            // a parity wait on a stage cannot tell its next phase from the one
            // after; having seen every phase in order, an issuer is never two
            // phases ahead of a stage.
            if (!(ok = mbar_wait(&full[stage], ph, abort_flag, err))) break;
            if (++stage == kStages) { stage = 0; ph ^= 1; }
            if (++abuf == kAccBufs) { abuf = 0; aph ^= 1; }
            continue;
          }
          if (!(ok = mbar_wait(&full[stage], ph, abort_flag, err))) break;
          if (!(ok = mbar_wait(&acc_empty[abuf], aph ^ 1, abort_flag, err))) break;
          tc_fence_after();
          const uint64_t ad = desc_sw128(smem_u32(smem + OFF_A + stage * A_BYTES));
          const uint64_t bd = desc_sw128(smem_u32(smem + OFF_B + slot * B_BYTES));
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16(tmem + abuf * N, ad + (uint64_t)(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4),
                     bd + (uint64_t)(((kk >> 2) * (N * 128) + (kk & 3) * 32) >> 4), IDESC, kk > 0);
          mma_commit(&empty[stage]);
          mma_commit(&acc_full[abuf]);
          used = any = true;
          if (++stage == kStages) { stage = 0; ph ^= 1; }
          if (++abuf == kAccBufs) { abuf = 0; aph ^= 1; }
        }
        if (!ok) break;
        if (used) mma_commit(&q_empty[slot]); else mbar_arrive(&q_empty[slot]);
      }
      if (any) mma_commit(done_bar); else mbar_arrive(done_bar);
      mbar_wait(done_bar, 0, abort_flag, err, 100000000ull);
    }
    __syncwarp();
  } else {
    // ======================= epilogue + running Top-K ===========================
    const int ew = warp - 2;                  // 0..15
    const int tk = ew >> 3;                   // token of the group this warp serves
    const int set = (ew >> 2) & 1;            // tiles of this parity (each set covers 4 lane quarters)
    const int quarter = warp & 3;             // TMEM lane quarter
    const int tt = (ew & 7) * 32 + lane;      // thread index within the token's TOKT
    const int row = quarter * 32 + lane;      // position within the tile (TMEM lane)
    unsigned long long* buf = reinterpret_cast<unsigned long long*>(smem + OFF_BUF) + tk * kCap;
    float* wts = reinterpret_cast<float*>(smem + OFF_W) + tk * kHeads;
    int* hist = reinterpret_cast<int*>(smem + OFF_HIST) + tk * kHistInts;
    TokState* ts = reinterpret_cast<TokState*>(smem + OFF_TOK) + tk;
    int gbase = 0;                            // the CTA's tile count before this group
    bool ok = true;
    for (int k = 0; ok && k < nmax; ++k) {
      const int g = zigzag_group(k, blockIdx.x, gridDim.x, a.groups);
      if (g < 0) continue;
      const int r = g * NT + tk;                        // query row this token slot holds
      const bool live = r < a.rows;
      const int64_t nvis = live ? a.q_offset + r + 1 : 0;
      if (tt < kHeads) wts[tt] = live ? __ldg(a.w + (int64_t)r * kHeads + tt) : 0.f;
      if (tt == 0) { ts->theta = 0ull; ts->cnt = 0; }
      bar_tok(tk);
      const int ntile = group_tiles(a, g);
      // the two sets take tiles j0 and j0 + 1 at once; the token's barrier
      // then publishes both tiles' appends
      for (int j0 = 0; j0 < ntile; j0 += 2) {
        const int j = j0 + set;
        // the stop decision is published before the token's barrier and read
        // after it, so its warps leave together (none is left waiting); a
        // warp whose wait failed appends nothing
        bool got = true;
        unsigned long long key = 0ull;
        bool take = false;
        if (j < ntile) {
          const int gi = gbase + j;                       // the CTA's tile index
          const int abuf = gi & (kAccBufs - 1);
          const uint32_t aph = (uint32_t)(gi / kAccBufs) & 1u;
          got = warp_wait(&acc_full[abuf], aph, abort_flag, err);
          if (got) {
            tc_fence_after();
            // the token's 64 head scores in two halves of 32 (fewer live
            // registers); weights four at a time, products two per instruction
            const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + abuf * N + tk * kHeads;
            const int64_t p = (int64_t)j * kTileM + row;
            float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
            const float4* w4 = reinterpret_cast<const float4*>(wts);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              float v[32];
              tmem_ld32(taddr + hh * 32, v);
              tmem_ld_wait();
#pragma unroll
              for (int h4 = 0; h4 < 8; ++h4) {
                const float4 ww = w4[hh * 8 + h4];
                a0 = ffma2(make_float2(ww.x, ww.y),
                           make_float2(fmaxf(v[4 * h4], 0.f), fmaxf(v[4 * h4 + 1], 0.f)), a0);
                a1 = ffma2(make_float2(ww.z, ww.w),
                           make_float2(fmaxf(v[4 * h4 + 2], 0.f), fmaxf(v[4 * h4 + 3], 0.f)), a1);
              }
            }
            tc_fence_before();
            mbar_arrive(&acc_empty[abuf]);
            if (live && p < nvis) {
              key = ((unsigned long long)score_key((a0.x + a1.x) + (a0.y + a1.y)) << 32) |
                    (unsigned long long)(0xFFFFFFFFu - (uint32_t)p);
              take = key > ts->theta;
            }
          }
        }
        // append with one atomic per warp
        const unsigned tm = __ballot_sync(0xffffffffu, take);
        if (tm) {
          int slot0 = 0;
          if (lane == __ffs(tm) - 1) slot0 = atomicAdd(&ts->cnt, __popc(tm));
          slot0 = __shfl_sync(0xffffffffu, slot0, __ffs(tm) - 1);
          if (take) buf[slot0 + __popc(tm & ((1u << lane) - 1u))] = key;
        }
        if (lane == 0 && (!got || *abort_flag)) ts->stop = 1;
        bar_tok(tk);
        if (ts->stop) { ok = false; break; }
        // keep room for two more tiles: compact a buffer that could overflow
        if (ts->cnt > kCap - 2 * kTileM) {
          const int n = ts->cnt;
          const unsigned long long t = select_kth(buf, n, a.K, hist, ts, tt, tk);
          compact_ge(buf, n, t, ts, tt, tk);
          if (tt == 0) { ts->cnt = a.K; ts->theta = t - 1ull; }
        }
        bar_tok(tk);
      }
      gbase += ntile;
      if (!ok) break;
      // ---- final selection of the group's rows -------------------------------
      if (live) {
        int n = ts->cnt;
        if (n > a.K) {
          const unsigned long long t = select_kth(buf, n, a.K, hist, ts, tt, tk);
          compact_ge(buf, n, t, ts, tt, tk);
          n = a.K;
        }
        // winners' positions -> registers, then the buffer becomes a bitmap
        constexpr int PER = kMaxK / TOKT;
        int mypos[PER];
#pragma unroll
        for (int e = 0; e < PER; ++e) {
          const int i = tt + e * TOKT;
          mypos[e] = i < n ? (int)(0xFFFFFFFFu - (uint32_t)(buf[i] & 0xFFFFFFFFull)) : -1;
        }
        bar_tok(tk);
        uint32_t* bits = reinterpret_cast<uint32_t*>(buf);
        const int nwords = (int)((nvis + 31) / 32);
        for (int i = tt; i < nwords; i += TOKT) bits[i] = 0u;
        bar_tok(tk);
#pragma unroll
        for (int e = 0; e < PER; ++e)
          if (mypos[e] >= 0) atomicOr(&bits[mypos[e] >> 5], 1u << (mypos[e] & 31));
        bar_tok(tk);
        // ascending output: each thread owns a contiguous run of words
        const int per = (nwords + TOKT - 1) / TOKT;
        const int w0 = min(nwords, tt * per), w1 = min(nwords, w0 + per);
        int mine = 0;
        for (int i = w0; i < w1; ++i) mine += __popc(bits[i]);
        // exclusive scan of `mine` over the token's TOKT threads
        int incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        int* wsum = hist;   // the token's warp totals
        if (lane == 31) wsum[tt >> 5] = incl;
        bar_tok(tk);
        int before = incl - mine;
        for (int x = 0; x < (tt >> 5); ++x) before += wsum[x];
        int32_t* out = a.idx + (int64_t)r * a.K;
        for (int i = w0; i < w1; ++i) {
          uint32_t m = bits[i];
          while (m) {
            const int bpos = __ffs(m) - 1;
            m &= m - 1;
            out[before++] = i * 32 + bpos;
          }
        }
        for (int i = n + tt; i < a.K; i += TOKT) out[i] = -1;
        if (a.count && tt == 0) a.count[r] = n;
      }
      bar_tok(tk);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

// Leading rows whose history holds at most K positions: 0, 1, .., n - 1, then
// -1 (the selection of every position, whatever the scores).
__global__ void __launch_bounds__(256)
prefill_take_all(int32_t* __restrict__ idx, int32_t* __restrict__ count, int rows, int K,
                 int64_t q_offset) {
  grid_dep_wait();     // the kernel launched before may still read these outputs
  grid_dep_launch();   // the fused indexer may start its set-up
  for (int t = blockIdx.x; t < rows; t += gridDim.x) {
    const int64_t n = q_offset + t + 1;
    int32_t* o = idx + (int64_t)t * K;
    for (int j = threadIdx.x; j < K; j += blockDim.x) o[j] = j < n ? j : -1;
    if (count && threadIdx.x == 0) count[t] = (int)n;
  }
}

}  // namespace

bool fused_prefill_topk_supported(const CacheView& c, int n_heads_idx, int rows, int64_t q_offset,
                                  int K) {
  if (n_heads_idx != kHeads || c.d != kD || c.k_dtype != DSI_BF16) return false;
  if (c.block_table && c.page_size % kSub != 0) return false;
  if (K < 1 || K > kMaxK) return false;
  if (q_offset + rows > kMaxRow) return false;
  const uint64_t krows = c.block_table ? (uint64_t)c.num_pages * c.page_size
                                       : (uint64_t)c.batch * c.s_max;
  if (krows >= (1ull << 31) || (int64_t)rows * kHeads >= (1ll << 31)) return false;
  return tma_encode_fn() != nullptr;
}

cudaError_t launch_index_topk_prefill(const bf16* q_idx, const float* w, const CacheView& c,
                                      int rows, int64_t q_offset, int K, int32_t* idx,
                                      int32_t* count, int* err, cudaStream_t st) {
  const uint64_t krows = c.block_table ? (uint64_t)c.num_pages * c.page_size
                                       : (uint64_t)c.batch * c.s_max;
  // rows r < K - q_offset see at most K positions and take them all
  const int r0 = (int)std::max<int64_t>(0, std::min<int64_t>(rows, (int64_t)K - q_offset));
  const int fr = rows - r0;                        // rows scored and selected
  const bf16* fq = q_idx + (int64_t)r0 * kHeads * kD;
  CUtensorMap kmap, qmap;
  // contiguous keys: one 128-row box per 64-dim block of a tile; paged: 64-row boxes
  if (!tma_map_2d(&kmap, c.k_idx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, krows, kD, 64,
                  c.block_table ? kSub : kTileM))
    return cudaErrorInvalidValue;
  // (with no row to score the map is never used)
  if (!tma_map_2d(&qmap, fr > 0 ? fq : q_idx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  (uint64_t)(fr > 0 ? fr : rows) * kHeads, kD, 64, kHeads))
    return cudaErrorInvalidValue;
  Args a;
  a.q_idx = fq;
  a.w = w + (int64_t)r0 * kHeads;
  a.idx = idx + (int64_t)r0 * K;
  a.count = count ? count + r0 : nullptr;
  a.q_offset = q_offset + r0;
  a.rows = fr;
  a.K = K;
  a.groups = (fr + NT - 1) / NT;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (r0 > 0) {
    const cudaError_t te = launch_overlapped(prefill_take_all, dim3(std::min(r0, sms)), dim3(256),
                                             0, st, idx, count, r0, K, q_offset);
    note_launch();
    if (te != cudaSuccess || fr == 0) return te;
  }
  const int npairs = (a.groups + 1) / 2;
  const int grid = npairs < sms ? npairs : sms;
  a.pairs_per_cta = (npairs + grid - 1) / grid;
  cudaError_t e = cudaFuncSetAttribute(index_topk_prefill,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (e != cudaSuccess) return e;
  cudaError_t le = launch_overlapped(index_topk_prefill, dim3(grid), dim3(THREADS), SMEM,
                                     st, kmap, qmap, c, a, err);
  note_launch();
  return le;
}

}  // namespace dsi
