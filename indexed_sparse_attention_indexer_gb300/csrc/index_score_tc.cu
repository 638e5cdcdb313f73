// Indexer scoring on the tcgen05 tensor cores (64 indexer heads x 128 dims).
//
// ("Day 0 Inference Support for New LLM Architectures: Optimization
// Practices", "Internal Fusion of the Indexer": relevance scoring then the
// weighted sum over heads, reading the paged K cache directly.)
//
// One tile is a GEMM D[128 positions x N] = K_tile[128 x 128] . Q^T with
// N = 64 heads x NT query tokens, accumulated in fp32 in TMEM:
//  * A (index keys) streams through a ring of shared-memory stages filled by
//    TMA (128-byte swizzle); paged caches are read page by page through the
//    block table (64-position sub-tiles, so any page size that is a multiple
//    of 64 works).
//  * B (the index queries of the current group of NT tokens) stays resident
//    in one of two shared-memory slots while its tiles stream by.
//  * the epilogue warps read one TMEM lane (= one position) per thread,
//    apply the ReLU gate and the per-token head weights, sum over heads and
//    (FP8 keys) multiply by the token's key scale.  Every head sum is
//    thread-local: no shuffles.
// Roles: warp 0 = TMA producer, warp 1 = TMEM owner + MMA issuer, the rest =
// epilogue.  Two TMEM accumulators let the epilogue of tile i overlap the MMA
// of tile i+1.  Work = (group, tile) items in causal order, split into equal
// contiguous ranges over one CTA per SM, so causal prefill rows balance
// without a special order.  FP8 keys use kind::f8f6f4 with the queries
// rounded to E4M3 (exact for the integer-valued index queries).
//
// MXFP8 keys (E4M3 codes, one E8M0 scale per group of 32, 64 or 128
// elements; "Day 0 Inference Support...", "A Layered Strategy"): the codes
// land by TMA as FP8 keys do and the tile's group scales by one bulk copy; the
// index queries are MXFP8-quantised group by group on the fly (codes in the
// B slot, scale bytes beside it).  Four scale warps, one per TMEM lane
// quarter, copy each tile's key scales and each query group's scales into
// TMEM, and the block-scaled MMA (kind::mxf8f6f4, one scale per 32 elements
// of K on both operands) applies them inside the tensor core: the
// dequantisation is fused into the contraction and nothing else in the
// kernel touches a code.  HBM carries one byte per key element plus a byte
// per group.
#include "kernels.h"
#include "tc_common.cuh"
#include "tma_host.h"

namespace dsi {
using namespace tc;

namespace {

constexpr int kD = 128;          // index key width
constexpr int kHeads = 64;       // indexer heads
constexpr int kTileM = 128;      // positions per tile
constexpr int kSub = 64;         // positions per TMA sub-tile
constexpr int kMaxGroups = 2048;

enum : int { kKeyBf16 = 0, kKeyFp8 = 1, kKeyMx = 2 };

template <int NT, int KK>
struct Cfg {
  static constexpr bool FP8 = KK == kKeyFp8;
  static constexpr bool MX = KK == kKeyMx;
  static constexpr bool K8 = FP8 || MX;                   // one byte per key element in HBM
  static constexpr int N = NT * kHeads;
  static constexpr int EB = K8 ? 1 : 2;                   // MMA operand element bytes
  static constexpr int ST_BYTES = kTileM * kD * EB;       // one stage = one MMA A tile: 16 or 32 KB
  static constexpr int B_BYTES = N * kD * EB;
  static constexpr int STAGES = K8 ? 8 : (NT == 1 ? 4 : 2);
  // MXFP8: one stage's key scales (128 keys x up to 4 bytes) and one query
  // slot's scale words (a 32-bit word per query row: the E8M0 bytes of its
  // four 32-element blocks of K)
  static constexpr int SC_BYTES = MX ? kTileM * 4 : 0;
  static constexpr int SQ_BYTES = MX ? N * 4 : 0;
  static constexpr int SF_WARPS = MX ? 4 : 0;             // scale warps, one per TMEM lane quarter
  static constexpr int EPI_WARPS = NT == 1 ? 4 : 8;
  static constexpr int EPI_THREADS = EPI_WARPS * 32;
  // producer warps: tile k is issued by producer k % PRODUCERS (one warp's
  // serial per-tile path cannot keep up with single-token decode over
  // one-byte keys, whose 16 KB tiles arrive twice as often as bf16 tiles)
  static constexpr int PRODUCERS = NT == 1 && K8 ? 2 : 1;
  static constexpr int PROD_WARP1 = 2 + EPI_WARPS + SF_WARPS;   // the extra producer warp
  // MMA issuers: tile k is issued by issuer k % MMA_WARPS.  A thread issuing
  // tcgen05.mma back to back waits ~120 cycles per instruction whatever N
  // (64 or 128) and kind (bf16 or E4M3), while two threads issuing at once
  // reach ~60 cycles per M = 128, N = 64 instruction (measured); a
  // single-token tile (N = 64) would otherwise be bound by its issuer's chain
  // of waits, four or eight MMAs and commits.
  static constexpr int MMA_WARPS = NT == 1 || (MX && NT == 2) ? 2 : 1;
  static constexpr int MMA_WARP1 = PROD_WARP1 + PRODUCERS - 1;   // the extra MMA warps
  static constexpr int THREADS =
      64 + EPI_THREADS + 32 * SF_WARPS + 32 * (PRODUCERS - 1) + 32 * (MMA_WARPS - 1);
  // MXFP8 scale columns in TMEM: per stage four (key row m's word in column
  // m / 32 of lane m), per query slot N / 32 (at least four)
  static constexpr int SFB_STRIDE = N / 32 < 4 ? 4 : N / 32;
  static constexpr int SF_COLS = MX ? STAGES * 4 + 2 * SFB_STRIDE : 0;
  // TMEM accumulators: four where they fit (the epilogue of tile i then
  // releases its accumulator four tiles ahead of the MMA that reuses it)
  static constexpr int ACCS_FIT = 4 * N + SF_COLS <= 512   ? 4
                                 : 3 * N + SF_COLS <= 512 ? 3
                                 : 2 * N + SF_COLS <= 512 ? 2
                                                          : 1;
  // Each issuer must be the one that used a stage or an accumulator last
  // before it waits on its barrier again (a parity wait cannot tell a phase
  // from the one two later), so both counts are multiples of the issuers.
  static constexpr int ACCS = MMA_WARPS == 2 ? ACCS_FIT & ~1 : ACCS_FIT;
  static_assert(ACCS >= 1 && ACCS % MMA_WARPS == 0 && STAGES % MMA_WARPS == 0, "issuer phases");
  static constexpr int SFA_COL = ACCS * N;
  static constexpr int SFB_COL = SFA_COL + STAGES * 4;
  static constexpr int TMEM_USED = ACCS * N + SF_COLS;
  static constexpr int TMEM_COLS = TMEM_USED <= 128 ? 128 : (TMEM_USED <= 256 ? 256 : 512);
  static_assert(TMEM_USED <= 512, "TMEM columns");
  static constexpr int KSTEPS = K8 ? 4 : 8;               // 32 bytes of K per MMA
  static constexpr uint32_t IDESC =
      MX ? idesc_mxf8(kTileM, N, 0, 0) : idesc_f32(FP8 ? 0u : 1u, kTileM, N);
  static constexpr int TOK_PER_THREAD = NT == 1 ? 1 : NT / 2;   // epilogue column split
  static constexpr bool SEQ_TOK = MX && TOK_PER_THREAD > 1;      // epilogue loads a token at a time
  // shared memory carve (offsets from a 1024-aligned base)
  static constexpr int OFF_A = 0;                                   // TMA stages
  static constexpr int OFF_B = OFF_A + STAGES * ST_BYTES;
  static constexpr int OFF_SC = OFF_B + 2 * B_BYTES;                // MXFP8: key scales
  static constexpr int OFF_SQ = OFF_SC + STAGES * SC_BYTES;         // MXFP8: query scale words
  static constexpr int OFF_KS = OFF_SQ + 2 * SQ_BYTES;              // FP8: per-stage key scales
  static constexpr int OFF_W = OFF_KS + (FP8 ? STAGES * kTileM * 4 : 0); // per epilogue warp: weights
  static constexpr int OFF_PREFIX = OFF_W + EPI_WARPS * TOK_PER_THREAD * kHeads * 4;
  static constexpr int OFF_BAR = (OFF_PREFIX + (kMaxGroups + 1) * 4 + 7) & ~7;
  static constexpr int NBARS = 2 * STAGES + 2 * ACCS + 2 + 2 + 1 + (MX ? STAGES : 0);
  static constexpr int OFF_MISC = OFF_BAR + NBARS * 8 + 8;
  static constexpr int SMEM = OFF_MISC + 64 + 1024;                 // + alignment slack
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

struct ScoreArgs {
  const bf16* q_idx;
  const float* w;
  float* scores;
  int64_t ld;
  int64_t q_offset;
  int rows;      // query rows (decode: sequences)
  int groups;
  int decode;
  int lg_group;  // MXFP8: log2 of the elements per scale (5, 6 or 7)
  int sc_bulk;   // FP8: key scales by one bulk copy per box (aligned) instead of per lane
};

// Group g holds query rows g*NT .. g*NT+NT-1: NT tokens of the prefill, or
// (decode) the NT candidate rows of one sequence, which share its key tiles.
// The group's last row sees the most history.
template <int NT>
__device__ __forceinline__ int64_t group_visible(const CacheView& c, const ScoreArgs& a, int g) {
  const int last = min(a.rows, (g + 1) * NT) - 1;
  return a.decode ? visible_len(c, last, 1, 0) : a.q_offset + last + 1;
}

template <int NT>
__device__ __forceinline__ int group_tiles(const CacheView& c, const ScoreArgs& a, int g) {
  return (int)((group_visible<NT>(c, a, g) + kTileM - 1) / kTileM);
}

// Walks the CTA's contiguous range of (group, tile) items.  The current
// group's tile count is kept in a register, so a step within a group reads
// no shared memory.
struct ItemIter {
  int g, j, left, gtiles;
  const int* prefix;
  int groups;
  __device__ void init(const int* pre, int G, int64_t begin, int64_t end) {
    prefix = pre;
    groups = G;
    left = (int)(end - begin);
    // largest g with prefix[g] <= begin
    int lo = 0, hi = G;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] <= begin) lo = mid; else hi = mid;
    }
    g = lo;
    j = (int)(begin - prefix[g]);
    skip_empty();
  }
  __device__ void skip_empty() {
    gtiles = g < groups ? prefix[g + 1] - prefix[g] : 0;
    while (g < groups && j >= gtiles) {
      ++g;
      j = 0;
      gtiles = g < groups ? prefix[g + 1] - prefix[g] : 0;
    }
  }
  __device__ bool valid() const { return left > 0; }
  __device__ void next() {
    --left;
    if (++j >= gtiles) skip_empty();
  }
  // group of the item after the current one (or -1 when none)
  __device__ int next_group() const {
    if (left <= 1) return -1;
    if (j + 1 < gtiles) return g;
    int gg = g + 1;
    while (gg < groups && prefix[gg + 1] == prefix[gg]) ++gg;
    return gg;
  }
};

template <int NT, int KK>
__global__ void __launch_bounds__(Cfg<NT, KK>::THREADS, 1)
score_tc(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
         CacheView c, ScoreArgs a, int* err) {
  using C = Cfg<NT, KK>;
  constexpr bool FP8 = C::FP8;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  grid_dep_wait();   // inputs may come from the kernel launched just before
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  float* wbuf = reinterpret_cast<float*>(smem + C::OFF_W);
  int* prefix = reinterpret_cast<int*>(smem + C::OFF_PREFIX);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::STAGES;
  uint64_t* acc_full = bars + 2 * C::STAGES;
  uint64_t* acc_empty = acc_full + C::ACCS;
  uint64_t* q_full = acc_empty + C::ACCS;
  uint64_t* q_empty = q_full + 2;
  uint64_t* done_bar = q_empty + 2;
  uint64_t* sf_full = done_bar + 1;         // MXFP8: the stage's scales are in TMEM
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  __shared__ int scan_tmp[40];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- per-CTA set-up: tile prefix over groups, barriers, TMEM --------------
  {
    const int G = a.groups;
    const int per = (G + C::THREADS - 1) / C::THREADS;
    const int g0 = min(G, tid * per), g1 = min(G, g0 + per);
    int mine = 0;
    for (int g = g0; g < g1; ++g) mine += group_tiles<NT>(c, a, g);
    int total;
    int run = block_exclusive_scan(mine, scan_tmp, total);
    for (int g = g0; g < g1; ++g) {
      prefix[g] = run;
      run += group_tiles<NT>(c, a, g);
    }
    if (tid == 0) prefix[G] = total;
  }
  if (tid == 0) {
    // FP8: the producer warp's 32 lanes also arrive on full when they copy the
    // key scales themselves, and a stage is empty once the MMAs and every
    // epilogue warp (which reads its scales) are done with it.  MXFP8: the
    // scale warps read the stage's scales before the MMAs are issued, so
    // the MMAs' commit empties it.
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], FP8 && !a.sc_bulk ? 33 : 1);
      mbar_init(&empty[s], FP8 ? 1 + C::EPI_WARPS : 1);
      if (C::MX) mbar_init(&sf_full[s], C::SF_WARPS);
    }
    for (int i = 0; i < C::ACCS; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], C::EPI_THREADS);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], C::MMA_WARPS);
    }
    mbar_init(done_bar, C::MMA_WARPS);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int64_t total_items = prefix[a.groups];
  const int64_t it_begin = total_items * blockIdx.x / gridDim.x;
  const int64_t it_end = total_items * (blockIdx.x + 1) / gridDim.x;

  const bool producer = warp == 0 || (C::PRODUCERS > 1 && warp == C::PROD_WARP1);
  const bool issuer = warp == 1 || (warp >= C::MMA_WARP1 && warp < C::MMA_WARP1 + C::MMA_WARPS - 1);
  if (producer) {
    // ======================= TMA producers ===================================
    // Producer pw issues the tiles k = pw, pw + PRODUCERS, ... of the CTA's
    // range; producer 0 also loads each group's queries.
    const int pw = warp == 0 ? 0 : 1;
    ItemIter it;
    it.init(prefix, a.groups, it_begin, it_end);
    int gprev = -1, qcount = 0, stage = 0;
    int gvis = -1, gb = 0, win = -1;     // group whose visible length / block-table window is held
    int64_t gnvis = 0, win0 = -1, rbase = 0;
    // log2 of a power-of-two page size (the common case: shifts instead of
    // 64-bit divisions per sub-tile), else -1
    const int pshift = (c.block_table && (c.page_size & (c.page_size - 1)) == 0)
                           ? __ffs(c.page_size) - 1 : -1;
    uint32_t phase = 0;
    int k = 0, last_k = -1;              // item index; last tile this warp issued (stage k % STAGES)
    // contiguous keys: one 128-row box per tile (the map's box is 128 rows);
    // paged caches: two 64-row boxes
    const bool whole = c.block_table == nullptr;
    const int spr = kD >> a.lg_group;    // MXFP8: scale bytes per key
    if (lane == 0) {
      prefetch_tmap(&kmap);
      if (!C::K8) prefetch_tmap(&qmap);
    }
    // The per-tile path is short: a warp's own instruction latency bounds its
    // tile rate.  Page ids and rows are worked out before the stage wait;
    // lane 0's wait result (false on abort or timeout) is the one value the
    // warp shares per tile.
    for (; it.valid(); ++k, it.next()) {
      if (k != 0 && ++stage == C::STAGES) { stage = 0; phase ^= 1; }
      const int g = it.g, j = it.j;
      if (pw == 0 && g != gprev) {
        const int slot = qcount & 1;
        const uint32_t qph = (qcount >> 1) & 1;
        bool ok = true;
        if (lane == 0) ok = mbar_wait(&q_empty[slot], qph ^ 1, abort_flag, err);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        uint8_t* qs = smem + C::OFF_B + slot * C::B_BYTES;
        if (C::MX) {
          // MXFP8-quantise the index queries group by group: E4M3 codes into
          // the swizzled B slot, the group's E8M0 byte into the row's scale
          // word (once per 32-element block it covers); the lanes of one
          // group are adjacent, so the group maximum is a butterfly
          const int upg = 1 << (a.lg_group - 4);     // 16-element units per group
          uint8_t* sq = smem + C::OFF_SQ + slot * C::SQ_BYTES;
          constexpr int kIters = C::N * 8 / 32, kBatch = 4;
          static_assert(kIters % kBatch == 0, "whole batches");
          for (int i0 = 0; i0 < kIters; i0 += kBatch) {
            // the loads of a batch of units first, then their quantisation
            uint4 v[kBatch][2];
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
              const int i = lane + (i0 + k) * 32;
              const int n = i >> 3, u = i & 7;
              const int r = g * NT + n / kHeads;
              v[k][0] = v[k][1] = make_uint4(0, 0, 0, 0);
              if (r < a.rows) {
                const bf16* src = a.q_idx + ((int64_t)r * kHeads + n % kHeads) * kD + u * 16;
                v[k][0] = __ldg(reinterpret_cast<const uint4*>(src));
                v[k][1] = __ldg(reinterpret_cast<const uint4*>(src + 8));
              }
            }
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
              const int i = lane + (i0 + k) * 32;
              const int n = i >> 3, u = i & 7;
              float f[16];
              bf16x8_to_f32(v[k][0], f);
              bf16x8_to_f32(v[k][1], f + 8);
              float amax = 0.f;
#pragma unroll
              for (int e = 0; e < 16; ++e) amax = fmaxf(amax, fabsf(f[e]));
              for (int m = 1; m < upg; m <<= 1)
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
              const int X = mx_exponent(amax);
              *reinterpret_cast<uint4*>(qs + sw128_offset(n, u)) = mx_encode16(f, X);
              if ((u & (upg - 1)) == 0) {
                const int kb0 = u >> 1, nkb = upg >> 1;
                for (int t = 0; t < nkb; ++t) sq[n * 4 + kb0 + t] = (uint8_t)(X + 127);
              }
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&q_full[slot]);
        } else if (FP8) {
          // round the bf16 index queries to E4M3 into the swizzled B slot; the
          // loads of eight units are issued before any of them is converted
          constexpr int kIters = C::N * 8 / 32, kBatch = 8;
          static_assert(kIters % kBatch == 0, "whole batches");
          for (int i0 = 0; i0 < kIters; i0 += kBatch) {
            uint4 v[kBatch][2];
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
              const int i = lane + (i0 + k) * 32;
              const int n = i >> 3, u = i & 7;
              const int r = g * NT + n / kHeads;
              v[k][0] = v[k][1] = make_uint4(0, 0, 0, 0);
              if (r < a.rows) {
                const bf16* src = a.q_idx + ((int64_t)r * kHeads + n % kHeads) * kD + u * 16;
                v[k][0] = __ldg(reinterpret_cast<const uint4*>(src));
                v[k][1] = __ldg(reinterpret_cast<const uint4*>(src + 8));
              }
            }
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
              const int i = lane + (i0 + k) * 32;
              const int n = i >> 3, u = i & 7;
              float f[16];
              bf16x8_to_f32(v[k][0], f);
              bf16x8_to_f32(v[k][1], f + 8);
              uint32_t wds[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const __nv_fp8x2_storage_t lo =
                    __nv_cvt_float2_to_fp8x2(make_float2(f[4 * e], f[4 * e + 1]), __NV_SATFINITE,
                                             __NV_E4M3);
                const __nv_fp8x2_storage_t hi =
                    __nv_cvt_float2_to_fp8x2(make_float2(f[4 * e + 2], f[4 * e + 3]),
                                             __NV_SATFINITE, __NV_E4M3);
                wds[e] = (uint32_t)lo | ((uint32_t)hi << 16);
              }
              *reinterpret_cast<uint4*>(qs + sw128_offset(n, u)) =
                  make_uint4(wds[0], wds[1], wds[2], wds[3]);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&q_full[slot]);
        } else if (lane == 0) {
          mbar_arrive_expect_tx(&q_full[slot], C::B_BYTES);
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            const int r = g * NT + t;   // rows past the end read as zeros
#pragma unroll
            for (int cc = 0; cc < 2; ++cc)
              tma_load_2d(qs + cc * (C::N * 128) + t * kHeads * 128, &qmap, cc * 64, r * kHeads,
                          &q_full[slot]);
          }
        }
        __syncwarp();
        ++qcount;
        gprev = g;
      }
      if (k % C::PRODUCERS != pw) continue;
      // ---- one key tile -----------------------------------------------------
      if (g != gvis) {               // the group's sequence and visible length, once
        gb = seq_of_row(c, g * NT, a.decode);
        gnvis = group_visible<NT>(c, a, g);
        rbase = (int64_t)gb * c.s_max;
        gvis = g;
        win0 = -1;
      }
      const int64_t p0 = (int64_t)j * kTileM;
      // physical row of each 64-position sub-tile (-1: past the visible
      // history).  Paged caches: the page ids come from a window of 32
      // block-table entries that the warp loads at once (one load per lane),
      // so no lane waits on a dependent page-table read per tile.
      int64_t prow[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int64_t pp = p0 + i * kSub;
        prow[i] = -1;
        if (pp >= gnvis) continue;
        if (c.block_table == nullptr) {
          prow[i] = rbase + pp;
          continue;
        }
        const int64_t pg = pshift >= 0 ? (pp >> pshift) : pp / c.page_size;
        if (win0 < 0 || pg < win0 || pg >= win0 + 32) {
          win0 = pg;
          const int64_t e = win0 + lane;
          win = e < c.max_pages ? __ldg(c.block_table + (int64_t)gb * c.max_pages + e) : -1;
        }
        const int page = __shfl_sync(0xffffffffu, win, (int)(pg - win0));
#ifdef DSI_CHECKED
        if (page < 0 || page >= c.num_pages) {
          if (lane == 0) report(err, kErrBounds);
          continue;
        }
#endif
        prow[i] = (int64_t)page * c.page_size + (pp - pg * c.page_size);
      }
      int nsub = 0;
#pragma unroll
      for (int i = 0; i < 2; ++i) nsub += prow[i] >= 0;
      bool ok = true;
      if (lane == 0) {
        ok = mbar_wait(&empty[stage], phase ^ 1, abort_flag, err);
        if (ok) {
          uint8_t* as = smem + C::OFF_A + stage * C::ST_BYTES;
          float* ks = reinterpret_cast<float*>(smem + C::OFF_KS) + stage * kTileM;
          uint8_t* ms = smem + C::OFF_SC + stage * C::SC_BYTES;
          if (whole) {
            // contiguous keys: the tile is one 128-row box (rows past the
            // history are read and ignored; past the array, zero-filled); the
            // key scales of the sequence's rows in the tile follow by one bulk
            // copy (16-byte aligned: sequences start at multiples of s_max)
            const uint32_t kr = (uint32_t)(c.s_max - p0 < kTileM ? c.s_max - p0 : kTileM);
            const uint32_t sc_bytes = FP8 && a.sc_bulk ? kr * 4u : C::MX ? kr * (uint32_t)spr : 0u;
            mbar_arrive_expect_tx(&full[stage], (uint32_t)C::ST_BYTES + sc_bytes);
            tma_load_2d(as, &kmap, 0, (int)prow[0], &full[stage]);
            if (!C::K8) tma_load_2d(as + 16384, &kmap, 64, (int)prow[0], &full[stage]);
            if (FP8 && sc_bytes) bulk_load(ks, c.k_scale + prow[0], sc_bytes, &full[stage]);
            if (C::MX) bulk_load(ms, c.k_mx_scale + prow[0] * spr, sc_bytes, &full[stage]);
          } else {
            // 64-row boxes (paged: one page's run each), each with its 64
            // keys' scales by one bulk copy
            mbar_arrive_expect_tx(
                &full[stage],
                (uint32_t)(nsub * (C::ST_BYTES / 2 + (C::MX ? kSub * spr : 0) +
                                   (FP8 && a.sc_bulk ? kSub * 4 : 0))));
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              if (prow[i] < 0) continue;
              if (C::K8) {
                tma_load_2d(as + i * (kSub * 128), &kmap, 0, (int)prow[i], &full[stage]);
              } else {
                tma_load_2d(as + i * (kSub * 128), &kmap, 0, (int)prow[i], &full[stage]);
                tma_load_2d(as + 16384 + i * (kSub * 128), &kmap, 64, (int)prow[i], &full[stage]);
              }
              if (C::MX)
                bulk_load(ms + i * kSub * spr, c.k_mx_scale + prow[i] * spr, kSub * spr,
                          &full[stage]);
              if (FP8 && a.sc_bulk)
                bulk_load(ks + i * kSub, c.k_scale + prow[i], kSub * 4, &full[stage]);
            }
          }
        }
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      if (FP8 && !a.sc_bulk) {
        // the tile's per-position key scales into the stage's scale slot, four
        // positions a lane (only visible positions are copied or read); the
        // lanes' barrier arrivals land with their copies
        float* ks = reinterpret_cast<float*>(smem + C::OFF_KS) + stage * kTileM;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int q = lane * 4 + k;
          const int64_t pr = prow[q / kSub];
          if (pr >= 0 && p0 + q < gnvis)
            cp_async_4(smem_u32(ks + q), c.k_scale + pr + (q % kSub));
        }
        cp_async_mbar_arrive_noinc(&full[stage]);
      }
      last_k = k;
    }
    // never leave the CTA with a copy still landing in shared memory: after
    // an abort, wait (bounded by time) for the stages of this warp's last
    // tiles (any tile still in flight is one of the last STAGES issued)
    if (FP8) cp_async_wait<0>();
    if (lane == 0 && *abort_flag) {
      volatile int no_abort = 0;
      for (int t = last_k; t >= 0 && t > last_k - C::STAGES; t -= C::PRODUCERS)
        mbar_wait(&full[t % C::STAGES], (uint32_t)((t / C::STAGES) & 1), &no_abort, err,
                  100000000ull);
    }
  } else if (issuer) {
    // ======================= MMA issuers ======================================
    // Issuer mw takes the tiles k = mw, mw + MMA_WARPS, ... (disjoint stages
    // and accumulators); a group's query slot is released once every issuer
    // has passed the group's last tile (a commit after its own MMAs on it,
    // else a plain arrival).
    const int mw = warp == 1 ? 0 : warp - C::MMA_WARP1 + 1;
    if (lane == 0) {
      ItemIter it;
      it.init(prefix, a.groups, it_begin, it_end);
      int gprev = -1, qcount = 0, stage = 0, abuf = 0, slot = 0;
      uint32_t phase = 0, aph = 0, qph = 0;
      bool qwait = false, used = false, any = false;
      for (int kt = 0; it.valid(); ++kt) {
        const int g = it.g;
        if (g != gprev) {
          slot = qcount & 1;
          qph = (qcount >> 1) & 1;
          ++qcount;
          gprev = g;
          qwait = true;
          used = false;
        }
        const bool last_of_group = it.next_group() != g;
        if (kt % C::MMA_WARPS != mw) {
          if (last_of_group) {
            // an issuer with no tile of the group still waits for its queries
            // before it arrives, so it cannot run a whole slot cycle ahead
            // and complete the slot's next phase for the group after
            if (qwait && !mbar_wait(&q_full[slot], qph, abort_flag, err)) break;
            qwait = false;
            if (used) mma_commit(&q_empty[slot]); else mbar_arrive(&q_empty[slot]);
          }
          if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
          if (++abuf == C::ACCS) { abuf = 0; aph ^= 1; }
          it.next();
          continue;
        }
        if (qwait) {
          if (!mbar_wait(&q_full[slot], qph, abort_flag, err)) break;
          qwait = false;
        }
        if (!mbar_wait(&full[stage], phase, abort_flag, err)) break;
        // MXFP8: the tile's key scales (and the group's query scales) in TMEM
        if (C::MX && !mbar_wait(&sf_full[stage], phase, abort_flag, err)) break;
        if (!mbar_wait(&acc_empty[abuf], aph ^ 1, abort_flag, err)) break;
        tc_fence_after();
        const uint32_t a_base = smem_u32(smem + C::OFF_A + stage * C::ST_BYTES);
        const uint32_t b_base = smem_u32(smem + C::OFF_B + slot * C::B_BYTES);
        const uint32_t d_tmem = tmem + abuf * C::N;
#pragma unroll
        for (int k = 0; k < C::KSTEPS; ++k) {
          uint32_t ao, bo;
          if (C::K8) { ao = k * 32; bo = k * 32; }
          else { ao = (k >> 2) * 16384 + (k & 3) * 32; bo = (k >> 2) * (C::N * 128) + (k & 3) * 32; }
          const uint64_t ad = desc_sw128(a_base + ao);
          const uint64_t bd = desc_sw128(b_base + bo);
          if (C::MX)   // K step k = 32-element block k: byte k of every scale word
            mma_mxf8(d_tmem, ad, bd, C::IDESC | ((uint32_t)k << 4) | ((uint32_t)k << 29),
                     tmem + C::SFA_COL + stage * 4, tmem + C::SFB_COL + slot * C::SFB_STRIDE,
                     k > 0);
          else if (FP8) mma_fp8(d_tmem, ad, bd, C::IDESC, k > 0);
          else mma_bf16(d_tmem, ad, bd, C::IDESC, k > 0);
        }
        mma_commit(&empty[stage]);
        mma_commit(&acc_full[abuf]);
        used = any = true;
        if (last_of_group) mma_commit(&q_empty[slot]);
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1;
        }
        if (++abuf == C::ACCS) { abuf = 0; aph ^= 1; }
        it.next();
      }
      // all MMAs of this CTA complete before TMEM is released
      if (any) mma_commit(done_bar); else mbar_arrive(done_bar);
      mbar_wait(done_bar, 0, abort_flag, err, 100000000ull);
    }
    __syncwarp();
  } else if (C::MX && warp >= 2 + C::EPI_WARPS) {   // (the warps before PROD_WARP1)
    // ======================= scale warps (MXFP8 keys) =========================
    // Warp q of the four (q = its TMEM lane quarter) copies into its lanes,
    // per query group, the scale words of query rows lane + 32c into column c
    // of the slot's (every lane quarter holds them all) and, per tile, the
    // scale word of key row 32q + lane into column q of the stage's four.
    const int quarter = warp & 3;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const int spr = kD >> a.lg_group;
    constexpr int NBC = C::N / 32;
    ItemIter it;
    it.init(prefix, a.groups, it_begin, it_end);
    int gprev = -1, qcount = 0, stage = 0;
    uint32_t phase = 0;
    while (it.valid()) {
      const int g = it.g;
      if (g != gprev) {
        const int slot = qcount & 1;
        if (!warp_wait(&q_full[slot], (qcount >> 1) & 1, abort_flag, err)) break;
        const uint32_t* sq = reinterpret_cast<const uint32_t*>(smem + C::OFF_SQ + slot * C::SQ_BYTES);
        uint32_t r[NBC];
#pragma unroll
        for (int cc = 0; cc < NBC; ++cc) r[cc] = sq[lane + 32 * cc];
        tmem_st_words<NBC>(tmem + lane_base + C::SFB_COL + slot * C::SFB_STRIDE, r);
        ++qcount;
        gprev = g;
      }
      if (!warp_wait(&full[stage], phase, abort_flag, err)) break;
      // the key's spr scale bytes, each repeated over the 32-element blocks
      // of its group
      const uint8_t* ks = smem + C::OFF_SC + stage * C::SC_BYTES + (quarter * 32 + lane) * spr;
      uint32_t wd;
      if (spr == 4) wd = *reinterpret_cast<const uint32_t*>(ks);
      else if (spr == 2) wd = __byte_perm(*reinterpret_cast<const uint16_t*>(ks), 0u, 0x1100);
      else wd = *ks * 0x01010101u;
      tmem_st_words<1>(tmem + lane_base + C::SFA_COL + stage * 4 + quarter, &wd);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sf_full[stage]);
      if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
      it.next();
    }
  } else {
    // ======================= epilogue =========================================
    const int ew = warp - 2;                 // 0 .. EPI_WARPS-1
    const int quarter = warp & 3;            // TMEM lane quarter this warp may read
    const int half = ew / 4;                 // column half (8-warp epilogue)
    const int row = quarter * 32 + lane;     // position within the tile
    ItemIter it;
    it.init(prefix, a.groups, it_begin, it_end);
    int gprev = -1, abuf = 0, kst = 0;
    uint32_t aph = 0, kph = 0;
    constexpr int TPT = C::TOK_PER_THREAD;
    // this warp's private copy of the head weights of its tokens (no
    // cross-warp barrier: a warp that leaves early can never block the others)
    float* wg = wbuf + ew * TPT * kHeads;
    int64_t nv[TPT];                         // visible length of each of the thread's tokens
    while (it.valid()) {
      const int g = it.g, j = it.j;
      if (g != gprev) {
        __syncwarp();
        for (int i = lane; i < TPT * kHeads; i += 32) {
          const int t = half * TPT + i / kHeads, h = i % kHeads;
          const int r = g * NT + t;
          wg[i] = r < a.rows ? __ldg(a.w + (int64_t)r * kHeads + h) : 0.f;
        }
#pragma unroll
        for (int tt = 0; tt < TPT; ++tt) {
          const int r = g * NT + half * TPT + tt;
          nv[tt] = r >= a.rows ? 0 : a.decode ? visible_len(c, r, 1, 0) : a.q_offset + r + 1;
        }
        __syncwarp();
        gprev = g;
      }
      if (!warp_wait(&acc_full[abuf], aph, abort_flag, err)) break;
      tc_fence_after();
      const int64_t p = (int64_t)j * kTileM + row;
      // the weighted ReLU head sum of token tt of this thread's tokens
      auto store = [&](int tt, const float* vt, float ksc) {
        const int t = half * TPT + tt;
        const int r = g * NT + t;
        if (r >= a.rows || p >= nv[tt]) return;
        const float* wt = wg + tt * kHeads;
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int h = 0; h < kHeads; h += 2) {
          s0 = fmaf(wt[h], fmaxf(vt[h], 0.f), s0);
          s1 = fmaf(wt[h + 1], fmaxf(vt[h + 1], 0.f), s1);
        }
        float sc = s0 + s1;
        if (FP8) sc *= ksc;
        a.scores[(int64_t)r * a.ld + p] = sc;
      };
      if constexpr (C::SEQ_TOK) {
        // one token's 64 columns at a time (the scale warps leave 128
        // registers a thread); the accumulator is released after the last
        // token's loads
#pragma unroll
        for (int tt = 0; tt < TPT; ++tt) {
          float v[kHeads];
          const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + abuf * C::N +
                                 (half * TPT + tt) * kHeads;
          tmem_ld32(taddr, v);
          tmem_ld32(taddr + 32, v + 32);
          tmem_ld_wait();
          if (tt == TPT - 1) {
            tc_fence_before();
            mbar_arrive(&acc_empty[abuf]);
          }
          store(tt, v, 1.f);
        }
        if (++abuf == C::ACCS) { abuf = 0; aph ^= 1; }
        it.next();
        continue;
      }
      float v[TPT][kHeads];
#pragma unroll
      for (int tt = 0; tt < TPT; ++tt) {
        const int t = half * TPT + tt;
        const uint32_t col = abuf * C::N + t * kHeads;
        const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + col;
        tmem_ld32(taddr, v[tt]);
        tmem_ld32(taddr + 32, v[tt] + 32);
      }
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&acc_empty[abuf]);
      // FP8 keys: this position's scale from the stage the producer filled
      // (acquire its copies through the stage's barrier), then release the
      // stage's scale slot
      float ksc = 1.f;
      if (FP8) {
        if (!warp_wait(&full[kst], kph, abort_flag, err)) break;
        ksc = reinterpret_cast<const float*>(smem + C::OFF_KS)[kst * kTileM + row];
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[kst]);
        if (++kst == C::STAGES) { kst = 0; kph ^= 1; }
      }
#pragma unroll
      for (int tt = 0; tt < TPT; ++tt) store(tt, v[tt], ksc);
      if (++abuf == C::ACCS) { abuf = 0; aph ^= 1; }
      it.next();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

// ---------------------------------------------------------------- host side
template <int NT, int KK>
cudaError_t go(const bf16* q_idx, const float* w, const CacheView& c, int rows, int decode,
               int64_t q_offset, float* scores, int64_t ld, int* err, cudaStream_t st) {
  using C = Cfg<NT, KK>;
  const uint64_t krows = c.block_table ? (uint64_t)c.num_pages * c.page_size
                                       : (uint64_t)c.batch * c.s_max;
  CUtensorMap kmap, qmap;
  memset(&qmap, 0, sizeof(qmap));
  // contiguous keys are copied a whole 128-position tile per box
  const uint32_t box_rows = c.block_table ? kSub : kTileM;
  if (C::K8) {
    if (!tma_map_2d(&kmap, c.k_idx, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, krows, kD, 128, box_rows))
      return cudaErrorInvalidValue;
  } else {
    if (!tma_map_2d(&kmap, c.k_idx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, krows, kD, 64, box_rows))
      return cudaErrorInvalidValue;
    if (!tma_map_2d(&qmap, q_idx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)rows * kHeads, kD,
                  64, kHeads))
      return cudaErrorInvalidValue;
  }
  ScoreArgs a;
  a.q_idx = q_idx;
  a.w = w;
  a.scores = scores;
  a.ld = ld;
  a.q_offset = q_offset;
  a.rows = rows;
  a.decode = decode;
  a.groups = (rows + NT - 1) / NT;
  a.lg_group = c.k_group == 128 ? 7 : c.k_group == 64 ? 6 : 5;
  // FP8 key scales by bulk copy: 16-byte aligned runs (a page's rows start at
  // multiples of 64 positions; a sequence's at multiples of s_max)
  a.sc_bulk = C::FP8 && (reinterpret_cast<uintptr_t>(c.k_scale) & 15) == 0 &&
              (c.block_table != nullptr || c.s_max % 4 == 0);
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaError_t e = cudaFuncSetAttribute(score_tc<NT, KK>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  cudaError_t le = launch_overlapped(score_tc<NT, KK>, dim3(sms), dim3(C::THREADS), C::SMEM,
                                     st, kmap, qmap, c, a, err);
  note_launch();
  return le;
}

template <int NT>
cudaError_t go_kind(const bf16* q_idx, const float* w, const CacheView& c, int rows, int decode,
                    int64_t q_offset, float* scores, int64_t ld, int* err, cudaStream_t st) {
  switch (c.k_dtype) {
    case DSI_FP8_E4M3:
      return go<NT, kKeyFp8>(q_idx, w, c, rows, decode, q_offset, scores, ld, err, st);
    case DSI_MXFP8_E4M3:
      return go<NT, kKeyMx>(q_idx, w, c, rows, decode, q_offset, scores, ld, err, st);
    default:
      return go<NT, kKeyBf16>(q_idx, w, c, rows, decode, q_offset, scores, ld, err, st);
  }
}

}  // namespace

bool tc_score_supported(const CacheView& c, int H) {
  if (H != kHeads || c.d != kD) return false;
  if (c.block_table && c.page_size % kSub != 0) return false;
  const uint64_t krows = c.block_table ? (uint64_t)c.num_pages * c.page_size
                                       : (uint64_t)c.batch * c.s_max;
  if (krows >= (1ull << 31)) return false;
  if ((reinterpret_cast<uintptr_t>(c.k_idx) & 15) != 0) return false;
  if (c.k_dtype == DSI_MXFP8_E4M3) {
    // the scales are copied as rows of 16 bytes, 64 keys at a time: a
    // sequence's (contiguous) or page's first key must start such a row
    if (!c.k_mx_scale || (reinterpret_cast<uintptr_t>(c.k_mx_scale) & 15) != 0) return false;
    if (c.k_group != 32 && c.k_group != 64 && c.k_group != 128) return false;
    const int per16 = 16 / (kD / c.k_group);             // keys per 16 bytes of scales
    if (!c.block_table && c.s_max % per16 != 0) return false;
    if (krows % per16 != 0) return false;
  }
  return tma_encode_fn() != nullptr;
}

// Query rows per group: prefill 4 tokens; decode one row, or the 2 or 4
// candidate rows of a sequence in a multi-token step (they share its keys,
// which are then read once for all of them).
static int tokens_per_group(const CacheView& c, int decode) {
  if (!decode) return 4;
  return (c.tokens_per_seq == 2 || c.tokens_per_seq == 4) ? c.tokens_per_seq : 1;
}

bool tc_score_shape_ok(const CacheView& c, int rows, int decode) {
  const int nt = tokens_per_group(c, decode);
  const int groups = (rows + nt - 1) / nt;
  return groups <= kMaxGroups && (int64_t)rows * kHeads < (1ll << 31);
}

cudaError_t launch_index_score_tc(const bf16* q_idx, const float* w, const CacheView& c, int rows,
                                  int decode, int64_t q_offset, float* scores, int64_t ld,
                                  int* err, cudaStream_t st) {
  if (decode) {
    switch (tokens_per_group(c, decode)) {
      case 4: return go_kind<4>(q_idx, w, c, rows, 1, 0, scores, ld, err, st);
      case 2: return go_kind<2>(q_idx, w, c, rows, 1, 0, scores, ld, err, st);
      default: return go_kind<1>(q_idx, w, c, rows, 1, 0, scores, ld, err, st);
    }
  }
  return go_kind<4>(q_idx, w, c, rows, 0, q_offset, scores, ld, err, st);
}

}  // namespace dsi
