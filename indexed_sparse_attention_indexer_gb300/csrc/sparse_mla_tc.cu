// Sparse MLA attention core on the tcgen05 tensor cores (128 heads).
//
// ("Day 0 Inference Support for New LLM Architectures: Optimization
// Practices", "Index-Based Sparse Attention": read the KV entries at the
// selected indices and attend over them; "Day 0 Inference Adaptation and
// Performance Optimization for New Models" §7: fuse index reading with the
// computation.)  Absorbed-MLA reading: key = the whole 576-wide latent row,
// value = its first 512 dims.
//
// One (query row, K split) is a cluster of two CTAs.  With all 128 heads as
// the MMA M dimension, the fp32 output of one row (128 x 512) alone fills a
// CTA's tensor memory, so the work is split by dimension:
//   CTA 0: logits over key dims   0..255 and 512..543, output dims   0..255
//   CTA 1: logits over key dims 256..511 and 544..575, output dims 256..511
// Each CTA gathers only the 288 dims of every selected row that it uses
// (no dim is gathered twice), keeps its half of the output accumulator in
// TMEM (256 columns), one logit tile (64 columns) and its query slice (four
// 64-dim blocks, 128 columns, and its half of the rope dims in 16 more): 18
// logit MMAs a tile on each CTA.  Stage block 4 holds the rope half in the
// first 64 bytes of each 128-byte row.
// The two partial logit tiles (128 heads x 64 positions, fp32) are swapped
// through distributed shared memory, so both CTAs hold the same logits and
// take the same softmax decisions.  Per 64-position tile, 12 warps:
//   producers (warps 0-2): the tile's rows into a 128-byte-swizzled stage
//     (ring of 4), by TMA gather4 (four rows per instruction) and cp.async at
//     once, so both copy engines work; the cp.async threads arrive on the
//     stage's barrier when their copies land, without waiting for them;
//   MMA (warp 3, one thread): S = Qslice . C^T into the logit tile once both
//     readers of the previous tile have loaded it, O += P . V (A = P K-major,
//     B = V MN-major, same stage);
//   exchange (warps 4-7): this CTA's partial logits out of TMEM and into the
//     peer's buffer (st.async, bytes counted on the peer's barrier);
//   softmax (warps 8-11, one head per thread): own partial from TMEM plus the
//     peer's from the buffer (one buffer credit per warp returns to the
//     peer), online softmax in log2 units with a lazily moved reference max
//     (the accumulator is rescaled only when the max grows by more than 2^8),
//     P in bf16 to the shared-memory P tile once P.V of the previous tile is
//     done, and the epilogue.
// Every wait is bounded; the cluster syncs once after set-up and once before
// exit so no CTA leaves while its peer may still write into it.
#include <atomic>

#include "kernels.h"
#include "tc_common.cuh"
#include "tma_host.h"

namespace dsi {
using namespace tc;

namespace {

constexpr int kH = 128;                        // heads (MMA M)
constexpr int kNp = 64;                        // positions per tile (MMA N of the logits)
constexpr int kChunks = 5;                     // stage blocks per row: four 64-dim blocks and the rope half
// Four stages: the logit tile and the P tile are single (their next use waits
// only for the readers of the previous one), and the query's rope half sits
// in the TMEM columns the second logit tile would take, which leaves the
// shared memory for a fourth 40 KB stage of gathered rows.
constexpr int kStages = 4;
constexpr int kXBufs = 1;                      // exchange buffers for the peer's partial logits
constexpr int kQkTmem = 4;                     // query blocks of the main logit MMAs (the rope half apart)
constexpr int kRopeHalf = 32;                  // rope dims each CTA takes (512.. or 544..)
constexpr int kChunkBytes = kNp * 128;         // one 64-dim block of a tile: 8 KB
constexpr int kStageBytes = kChunks * kChunkBytes;
// 12 warps (three per SM sub-partition): at most 168 registers a thread
constexpr int kProducerWarps = 3;
constexpr int kMmaWarp = kProducerWarps;       // warp 3: lane 0 issues the MMAs
constexpr int kExWarp0 = kMmaWarp + 1;         // warps 4-7: logit exchange with the peer
constexpr int kSmWarp0 = kExWarp0 + 4;         // warps 8-11: softmax and epilogue
constexpr int kThreads = (kSmWarp0 + 4) * 32;  // 384
// Each tile is gathered by two engines at once: TMA gather4 (warp 0) for the
// first kTmaChunks 64-dim blocks of the first kTmaRows rows, cp.async (warps
// 1-2) for the rest.
constexpr int kTmaChunks = 3;
// rows of those blocks by TMA (cp.async takes the rest): rows from HBM (one
// cluster a row, the decode batches) gather faster with more of them on
// cp.async, rows from L2 (the persistent prefill form) with more on TMA
constexpr int kTmaRows = 40;
constexpr int kTmaRowsP = 48;
static_assert(kTmaRows % 4 == 0 && kTmaRows <= kNp && kTmaRowsP % 4 == 0 && kTmaRowsP <= kNp,
              "whole gather4 groups");
constexpr int kLdgWarps = kProducerWarps - 1;
constexpr int kLdgThreads = kLdgWarps * 32;

constexpr int kMaxEntries = DSI_MAX_K;         // index entries one split can hold

constexpr int OFF_C = 0;
constexpr int OFF_P = OFF_C + kStages * kStageBytes;      // the P tile [128 x 64] bf16, 16 KB
constexpr int OFF_X = OFF_P + kH * kNp * 2;               // kXBufs x peer logits [128 x 64] fp32
constexpr int OFF_ROWS = OFF_X + kXBufs * kH * kNp * 4;   // physical row of each entry (or -1)
constexpr int OFF_BAR = OFF_ROWS + kMaxEntries * 4;
constexpr int NBARS = 2 * kStages + 12 + 2 * kXBufs;
constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
constexpr int SMEM = OFF_MISC + 64 + 1024;
static_assert(SMEM <= 227 * 1024, "shared memory");

constexpr uint32_t TM_S = 0;      // logits, 64 columns
constexpr uint32_t TM_Q4 = 64;    // the query's rope half (16 of 32 columns used)
constexpr uint32_t TM_Q = 128;    // query slice: four 64-dim blocks, 128 columns
constexpr uint32_t TM_O = 256;    // output half, 256 columns
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t IDESC_S = idesc_f32(1, kH, kNp);
constexpr uint32_t IDESC_O = idesc_f32_bmn(1, kH, 256);
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.f;  // move the reference max only when it grows by > 2^8

struct MlaArgs {
  const bf16* q;
  const int32_t* idx;
  bf16* out;
  float* lse;
  float* part_o;
  float2* part_ml;
  int64_t q_offset;
  float scale;
  int rows, K, decode, splits;
};

// An entry takes part when it names a visible position.  Checked in every
// build (the checked build also reports entries past the history), so indices
// left unwritten by a failed earlier kernel never address rows outside the cache.
__device__ __forceinline__ bool pos_ok(int pos, int64_t n_vis) {
  return pos >= 0 && pos < n_vis;
}

// A tile's cp.async part, thread lt of kLdgThreads: the fourth 64-dim block
// of every row (8 pieces a row), the rope half (4 pieces, into the first half
// of block 4) and the first kTmaChunks blocks of the rows past kTmaRows, each
// 16-byte piece to its swizzled place (consecutive threads take consecutive
// pieces of a row).  `rows` holds the tile's physical rows (-1: row 0).
template <int TR>
__device__ __forceinline__ void ldg_tile(uint32_t st_addr, const bf16* latent, const int32_t* rows,
                                         int lt, uint32_t rho, int g0) {
  static_assert((kNp - TR) * kTmaChunks * 8 % kLdgThreads == 0, "whole rounds of pieces");
#pragma unroll
  for (int k = 0; k < kNp * 8 / kLdgThreads; ++k) {
    const int q = lt + k * kLdgThreads, rr = q >> 3, u = q & 7;
    const int pr = max(rows[rr], 0);
    cp_async_16(st_addr + 3 * kChunkBytes + sw128_offset(rr, u),
                latent + (int64_t)pr * DSI_D_QK + (g0 + 3) * 64 + u * 8);
  }
#pragma unroll
  for (int k = 0; k < kNp * 4 / kLdgThreads; ++k) {
    const int q = lt + k * kLdgThreads, rr = q >> 2, u = q & 3;
    const int pr = max(rows[rr], 0);
    cp_async_16(st_addr + kQkTmem * kChunkBytes + sw128_offset(rr, u),
                latent + (int64_t)pr * DSI_D_QK + DSI_D_LATENT + (int)rho * kRopeHalf + u * 8);
  }
  constexpr int kTail = (kNp - TR) * kTmaChunks * 8;
#pragma unroll
  for (int k = 0; k < kTail / kLdgThreads; ++k) {
    const int q = lt + k * kLdgThreads;
    const int rr = TR + q / (kTmaChunks * 8), w = q % (kTmaChunks * 8);
    const int pr = max(rows[rr], 0);
    cp_async_16(st_addr + (w >> 3) * kChunkBytes + sw128_offset(rr, w & 7),
                latent + (int64_t)pr * DSI_D_QK + (g0 + (w >> 3)) * 64 + (w & 7) * 8);
  }
}
static_assert(kNp * 8 % kLdgThreads == 0 && kNp * 4 % kLdgThreads == 0, "whole rounds of pieces");

__device__ __forceinline__ void tmem_st32f(uint32_t taddr, const float* v) {
  uint32_t r[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(v[i]);
  tmem_st32(taddr, r);
}

// FP8 latent rows: 16 codes a piece, 18 pieces of this CTA's 288 dims per
// row, 1152 pieces a tile over the three producer warps.
constexpr int kF8RowPieces = (kQkTmem * 64 + kRopeHalf) / 16;   // 18 pieces of 16 codes a row
constexpr int kF8Pieces = kNp * kF8RowPieces;
constexpr int kF8PerThread = (kF8Pieces + kProducerWarps * 32 - 1) / (kProducerWarps * 32);
// first latent dim of piece u of a row: the four 64-dim blocks, then the rope half
__device__ __forceinline__ int f8_piece_dim(int u, uint32_t rho, int g0) {
  return u < kQkTmem * 4 ? g0 * 64 + u * 16
                         : DSI_D_LATENT + (int)rho * kRopeHalf + (u - kQkTmem * 4) * 16;
}

// 16 E4M3 codes times their tile scale, rounded to bf16 (lo = codes 0..7).
__device__ __forceinline__ void fp8x16_scaled_bf16(const uint4& v, float sc, uint4& lo, uint4& hi) {
  const uint32_t in[4] = {v.x, v.y, v.z, v.w};
  uint32_t out[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const __nv_fp8x2_storage_t pr = (__nv_fp8x2_storage_t)((in[k] >> (16 * hh)) & 0xFFFFu);
      const __half2 h2 = __half2(__nv_cvt_fp8x2_to_halfraw2(pr, __NV_E4M3));
      const float2 f = __half22float2(h2);
      const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * sc, f.y * sc);
      out[2 * k + hh] = *reinterpret_cast<const uint32_t*>(&b);
    }
  }
  lo = make_uint4(out[0], out[1], out[2], out[3]);
  hi = make_uint4(out[4], out[5], out[6], out[7]);
}

template <bool F8L>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
mla_tc(const __grid_constant__ CUtensorMap lmap, CacheView c, const float* lscale, MlaArgs a,
       int* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* full = bars;                       // [kStages] gather landed (TMA bytes + cp.async threads)
  uint64_t* empty = bars + kStages;            // [kStages] stage free (MMA commit)
  uint64_t* s_full = bars + 2 * kStages;       // [2] logits in TMEM (MMA commit)
  uint64_t* s_empty = s_full + 2;              // [2] logits read out (softmax threads)
  uint64_t* p_full = s_full + 4;               // [2] P written (softmax threads)
  uint64_t* p_empty = s_full + 6;              // [2] P.V done (MMA commit)
  uint64_t* q_ready = s_full + 8;              // query slice in place (softmax threads)
  uint64_t* o_done = s_full + 9;               // last P.V done (MMA commit)
  uint64_t* x_full = s_full + 10;              // [kXBufs] peer's partial logits landed (byte count)
  uint64_t* x_empty = x_full + kXBufs;         // [kXBufs] peer has read what we sent (one credit per peer softmax warp)
  int32_t* rows_s = reinterpret_cast<int32_t*>(smem + OFF_ROWS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  int* last_valid = reinterpret_cast<int*>(smem + OFF_MISC + 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rho = cluster_ctarank();          // which half of the dims this CTA owns
  const uint32_t peer = rho ^ 1u;
  const int pair = blockIdx.x >> 1;
  const int r = pair / a.splits, sp = pair % a.splits;
  const int b = seq_of_row(c, r, a.decode);
  const int64_t n_vis = visible_len(c, r, a.decode, a.q_offset);
  const int tiles_all = (a.K + kNp - 1) / kNp;
  const int tiles_per = (tiles_all + a.splits - 1) / a.splits;
  const int j_begin = sp * tiles_per * kNp;
  const int j_end = min(a.K, j_begin + tiles_per * kNp);
  const int span = tiles_per * kNp;                // entries this split owns (<= kMaxEntries)
  const int32_t* irow = a.idx + (int64_t)r * a.K;
  const int g0 = rho ? 4 : 0;                      // first gathered 64-dim block
  // this CTA's slice of the head's query row is loaded first, so it lands
  // while the entries are being staged (and, launched behind the select
  // kernel, while that kernel finishes): the exchange warps take the first two
  // of its four main blocks, the softmax warps the other two and the rope half
  // (eight 16-byte pieces a block, four for the rope half)
  uint4 qv[24];
  if (warp >= kExWarp0) {
    const int b0 = g0 + (warp < kSmWarp0 ? 0 : 2);
    const int nq = warp < kSmWarp0 ? 16 : 16 + kRopeHalf / 8;
    const uint4* qrow = reinterpret_cast<const uint4*>(
        a.q + ((int64_t)r * kH + (warp & 3) * 32 + lane) * DSI_D_QK);
#pragma unroll
    for (int i = 0; i < 24; ++i)
      qv[i] = i < nq ? __ldg(qrow + (i < 16 ? b0 * 8 + i
                                            : (DSI_D_LATENT + (int)rho * kRopeHalf) / 8 + (i - 16)))
                     : make_uint4(0, 0, 0, 0);
  }

  if (tid == 0) {
    // bf16 rows: the TMA lane's byte count plus the cp.async threads; FP8
    // rows: every producer thread once its converted pieces are stored
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], F8L ? kProducerWarps * 32 : 1 + kLdgThreads);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 256);
      mbar_init(&p_full[i], 128);
      mbar_init(&p_empty[i], 1);
    }
    mbar_init(q_ready, 256);
    mbar_init(o_done, 1);
    for (int i = 0; i < kXBufs; ++i) {
      mbar_init(&x_full[i], 1);
      mbar_init(&x_empty[i], 4);
    }
    *abort_flag = 0;
    *last_valid = -1;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, TMEM_COLS);
  // the selected indices come from the previous kernel
  grid_dep_wait();
  constexpr int kPer = (kMaxEntries + kThreads - 1) / kThreads;
  int pos[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int jj = tid + u * kThreads;
    pos[u] = (jj < span && j_begin + jj < j_end) ? __ldg(irow + j_begin + jj) : -1;
  }
  __syncthreads();
  // the split's entries, translated once to physical cache rows (-1 = skipped)
  {
    int lv = -1;
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int jj = tid + u * kThreads;
      if (jj >= span) break;
      int pr = -1;
#ifdef DSI_CHECKED
      if (pos[u] >= n_vis) report(err, kErrBounds);
#endif
      if (pos_ok(pos[u], n_vis)) {
        const int64_t x = phys_row(c, b, pos[u], err);
        if (x >= 0) { pr = (int)x; lv = jj; }
      }
      rows_s[jj] = pr;
    }
    if (lv >= 0) atomicMax(last_valid, lv);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int n_tiles = *last_valid < 0 ? 0 : *last_valid / kNp + 1;
  constexpr uint32_t kXBytes = kH * kNp * 4;       // one partial logit tile
  if (tid == 0) {                                  // expect the peer's first two tiles
    for (int i = 0; i < kXBufs && i < n_tiles; ++i) mbar_arrive_expect_tx(&x_full[i], kXBytes);
  }
  cluster_sync();   // the peer's barriers exist (and are armed) before anyone uses them
  grid_dep_launch();   // the next kernel on the stream may start its set-up
  const uint32_t tmem = *tmem_slot;

  if (F8L && warp < kProducerWarps) {
    // ======================= gather: FP8 rows ===================================
    // Each thread owns kF8PerThread pieces of every tile (16 codes of one row)
    // and keeps one tile of them in registers: piece k of tile t is converted
    // (code * tile scale, rounded to bf16) into the swizzled stage, and its
    // registers at once take piece k of tile t+1, so a tile's loads are in
    // flight while the previous tile is converted and processed.  The stage
    // is occupied from conversion to its P.V only.
    const uint8_t* codes = reinterpret_cast<const uint8_t*>(c.latent);
    uint4 cv[kF8PerThread];
    float sc[kF8PerThread];
    auto load_tile = [&](int t) {
#pragma unroll
      for (int k = 0; k < kF8PerThread; ++k) {
        const int q = tid + k * kProducerWarps * 32;
        if (q < kF8Pieces) {
          const int rr = q / kF8RowPieces, u = q % kF8RowPieces;
          const int64_t pr = max(rows_s[t * kNp + rr], 0);
          const int d0 = f8_piece_dim(u, rho, g0);     // first dim of the piece
          cv[k] = __ldg(reinterpret_cast<const uint4*>(codes + pr * DSI_D_QK + d0));
          sc[k] = __ldg(lscale + pr * 5 + (d0 >> 7));
        }
      }
    };
    if (n_tiles > 0) load_tile(0);
    int stage = 0;
    uint32_t ph = 0;
    for (int t = 0; t < n_tiles; ++t) {
      if (!mbar_wait(&empty[stage], ph ^ 1, abort_flag, err)) break;
      uint8_t* st_base = smem + OFF_C + stage * kStageBytes;
#pragma unroll
      for (int k = 0; k < kF8PerThread; ++k) {
        const int q = tid + k * kProducerWarps * 32;
        if (q < kF8Pieces) {
          const int rr = q / kF8RowPieces, u = q % kF8RowPieces;
          uint4 lo, hi;
          fp8x16_scaled_bf16(cv[k], sc[k], lo, hi);
          uint8_t* blk = st_base + (u >> 2) * kChunkBytes;
          *reinterpret_cast<uint4*>(blk + sw128_offset(rr, (u & 3) * 2)) = lo;
          *reinterpret_cast<uint4*>(blk + sw128_offset(rr, (u & 3) * 2 + 1)) = hi;
          if (t + 1 < n_tiles) {
            const int64_t pr = max(rows_s[(t + 1) * kNp + rr], 0);
            const int d0 = f8_piece_dim(u, rho, g0);
            cv[k] = __ldg(reinterpret_cast<const uint4*>(codes + pr * DSI_D_QK + d0));
            sc[k] = __ldg(lscale + pr * 5 + (d0 >> 7));
          }
        }
      }
      fence_proxy_async_smem();   // the tensor core reads the stage through the async proxy
      mbar_arrive(&full[stage]);
      if (++stage == kStages) { stage = 0; ph ^= 1; }
    }
  } else if (warp == 0) {
    // ======================= gather: TMA part =================================
    // kTmaRows/4 lanes: lane g gathers rows 4g..4g+3 of the tile for the
    // first kTmaChunks 64-dim blocks, each a TMA gather of four 128-byte rows
    // into the swizzled stage.  Lane 0 first arms the stage's barrier.
    // Skipped entries fetch row 0 (their probability is zero).
    if (lane < kTmaRows / 4) {
      if (lane == 0) prefetch_tmap(&lmap);
      int stage = 0;
      uint32_t ph = 0;
      bool issued[kStages] = {};
      uint32_t issued_ph[kStages] = {};
      const unsigned gmask = (1u << (kTmaRows / 4)) - 1u;
      for (int t = 0; t < n_tiles; ++t) {
        bool ok = true;
        if (lane == 0) {
          ok = mbar_wait(&empty[stage], ph ^ 1, abort_flag, err);
          if (ok) mbar_arrive_expect_tx(&full[stage], kTmaChunks * kTmaRows * 128);
        }
        ok = __shfl_sync(gmask, ok, 0);
        if (!ok) break;
        issued[stage] = true;
        issued_ph[stage] = ph;
        uint8_t* st_base = smem + OFF_C + stage * kStageBytes;
        const int r4 = lane * 4;
        const int32_t* rw = rows_s + t * kNp + r4;
        const int y0 = max(rw[0], 0), y1 = max(rw[1], 0), y2 = max(rw[2], 0), y3 = max(rw[3], 0);
#pragma unroll
        for (int ch = 0; ch < kTmaChunks; ++ch)
          tma_gather4(st_base + ch * kChunkBytes + r4 * 128, &lmap, (g0 + ch) * 64, y0, y1, y2, y3,
                      &full[stage]);
        if (++stage == kStages) { stage = 0; ph ^= 1; }
      }
      // never leave the CTA with a gather still landing in shared memory
      if (lane == 0 && *abort_flag) {
        volatile int no_abort = 0;   // the drain is bounded by time only
        for (int s2 = 0; s2 < kStages; ++s2)
          if (issued[s2]) mbar_wait(&full[s2], issued_ph[s2], &no_abort, err, 100000000ull);
      }
    }
  } else if (!F8L && warp < kProducerWarps) {
    // ======================= gather: cp.async part ============================
    // the fourth 64-dim block and the rope half of every row, and the first
    // blocks of the rows past kTmaRows, each 16-byte piece to its swizzled
    // place (consecutive lanes take consecutive pieces of a row); each tile is
    // signalled (after a proxy fence) once its copies have landed.  The split
    // balances the two engines.
    int stage = 0;
    uint32_t ph = 0;
    for (int t = 0; t < n_tiles; ++t) {
      if (!mbar_wait(&empty[stage], ph ^ 1, abort_flag, err)) break;
      const uint32_t st_addr = smem_u32(smem + OFF_C + stage * kStageBytes);
      ldg_tile<kTmaRows>(st_addr, c.latent, rows_s + t * kNp, (warp - 1) * 32 + lane, rho, g0);
      // the stage's barrier counts this thread once its copies have landed;
      // the thread goes on to the next stage without waiting for them
      cp_async_mbar_arrive_noinc(&full[stage]);
      if (++stage == kStages) { stage = 0; ph ^= 1; }
    }
    cp_async_wait<0>();
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      // ===================== MMA issuer =======================================
      // Event-driven with non-blocking probes (nothing in this warp ever
      // suspends): a P.V tile is issued when its P is ready, a logit tile (QK)
      // when its gather has landed and the TMEM logit tile is free.
      bool ok = mbar_wait(q_ready, 0, abort_flag, err);
      tc_fence_after();
      int qk_next = 0, pv_next = 0;
      const uint32_t pbase = smem_u32(smem + OFF_P);
      uint64_t t_last = global_ns();
      uint32_t idle = 0;
      while (ok && pv_next < n_tiles) {
        bool progress = false;
        if (pv_next < qk_next && mbar_test_wait(&p_full[0], pv_next & 1)) {
          tc_fence_after();
          const int st = pv_next % kStages;
          const uint64_t pd = desc_sw128(pbase);
          const uint64_t vd = desc_sw128_mn(smem_u32(smem + OFF_C + st * kStageBytes), kChunkBytes);
#pragma unroll
          for (int kk = 0; kk < kNp / 16; ++kk)
            mma_bf16(tmem + TM_O, pd + (uint64_t)((kk * 32) >> 4), vd + (uint64_t)((kk * 2048) >> 4),
                     IDESC_O, (pv_next > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&p_empty[0]);
          mma_commit(&empty[st]);
          ++pv_next;
          progress = true;
        }
        if (qk_next < n_tiles) {
          const int st = qk_next % kStages;
          if (mbar_test_wait(&full[st], (qk_next / kStages) & 1) &&
              mbar_test_wait(&s_empty[0], (qk_next & 1) ^ 1)) {
            tc_fence_after();
            // the stage's cp.async part was written through the generic proxy
            fence_proxy_async_smem();
            const uint32_t t_s = tmem + TM_S;
            const uint32_t st_base = smem_u32(smem + OFF_C + st * kStageBytes);
            const uint64_t d0 = desc_sw128(st_base);
            for (int k = 0; k < kQkTmem * 4; ++k)
              mma_bf16_tmem_a(t_s, tmem + TM_Q + k * 8,
                              d0 + (uint64_t)(((k >> 2) * kChunkBytes + (k & 3) * 32) >> 4),
                              IDESC_S, k > 0 ? 1u : 0u);
            {   // this CTA's half of the rope dims, in the first half of stage block 4
              const uint64_t cd = desc_sw128(st_base + kQkTmem * kChunkBytes);
#pragma unroll
              for (int kk = 0; kk < kRopeHalf / 16; ++kk)
                mma_bf16_tmem_a(t_s, tmem + TM_Q4 + kk * 8, cd + (uint64_t)((kk * 32) >> 4),
                                IDESC_S, 1u);
            }
            mma_commit(&s_full[0]);
            ++qk_next;
            progress = true;
          }
        }
        // bounded: give up after kWaitLimitNs without progress (the clock is
        // read once per 256 idle probes)
        if (progress) {
          idle = 0;
          t_last = global_ns();
        } else if (*abort_flag) {
          ok = false;
        } else if ((++idle & 255u) == 0 && global_ns() - t_last > kWaitLimitNs) {
          *abort_flag = 1;
          report(err, kErrTimeout);
          ok = false;
        }
      }
      mma_commit(o_done);
    }
    __syncwarp();
  } else if (warp < kSmWarp0) {
    // ======================= logit exchange ===================================
    // Per tile: read this CTA's partial logits from TMEM and store them into
    // the peer's exchange buffer (st.async, bytes counted on the peer's
    // barrier) once the peer has read the previous tile out of it.  The
    // softmax warps read the same TMEM tile and add the peer's partial.
    const int quarter = warp & 3;
    const int h = quarter * 32 + lane;               // head = TMEM lane
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
      uint32_t w32[32];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 v = qv[8 * ch + i];
        w32[4 * i] = v.x; w32[4 * i + 1] = v.y; w32[4 * i + 2] = v.z; w32[4 * i + 3] = v.w;
      }
      tmem_st32(tmem + lane_base + TM_Q + ch * 32, w32);
    }
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(q_ready);
    // exchange buffer layout [buffer][4-position group][head] x float4: a
    // warp's stores (and loads) of one group are 512 contiguous bytes
    const uint32_t x_remote = map_to_rank(smem_u32(smem + OFF_X), peer) + h * 16;
    const uint32_t xfull_remote = map_to_rank(smem_u32(x_full), peer);
    bool ok = true;
    for (int t = 0; ok && t < n_tiles; ++t) {
      const int bsel = t % kXBufs;
      float v[kNp];
      if (!(ok = warp_wait(&s_full[0], t & 1, abort_flag, err))) break;
      tc_fence_after();
      tmem_ld32(tmem + lane_base + TM_S, v);
      tmem_ld32(tmem + lane_base + TM_S + 32, v + 32);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&s_empty[0]);
      // this CTA's partial to the peer, once the peer has read the buffer
      if (!(ok = warp_wait_cluster(&x_empty[bsel], ((t / kXBufs) & 1) ^ 1, abort_flag, err))) break;
      const uint32_t dst = x_remote + bsel * kXBytes;
#pragma unroll
      for (int q4 = 0; q4 < kNp / 4; ++q4)
        st_async_v4(dst + q4 * (kH * 16),
                    make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]),
                    xfull_remote + bsel * 8);
    }
  } else {
    // ======================= softmax + epilogue ================================
    const int quarter = warp & 3;
    const int h = quarter * 32 + lane;               // head = TMEM lane
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    // query blocks 2-3 and the rope half into TMEM
    {
#pragma unroll
      for (int ch = 2; ch < kQkTmem; ++ch) {
        uint32_t w32[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 v = qv[8 * (ch - 2) + i];
          w32[4 * i] = v.x; w32[4 * i + 1] = v.y; w32[4 * i + 2] = v.z; w32[4 * i + 3] = v.w;
        }
        tmem_st32(tmem + lane_base + TM_Q + ch * 32, w32);
      }
      {
        uint32_t w32[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 v = qv[8 * (kQkTmem - 2) + i];
          w32[4 * i] = v.x; w32[4 * i + 1] = v.y; w32[4 * i + 2] = v.z; w32[4 * i + 3] = v.w;
        }
        tmem_st32(tmem + lane_base + TM_Q4, w32);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(q_ready);
    }
    uint8_t* const pbuf = smem + OFF_P;
    const uint8_t* xrow = smem + OFF_X + h * 16;
    const uint32_t xempty_remote = map_to_rank(smem_u32(x_empty), peer);
    const float sl2 = a.scale * kLog2e;
    float m_ref = -INFINITY, l_sum = 0.f;
    bool ok = true;
    for (int t = 0; ok && t < n_tiles; ++t) {
      // summed logits of tile t (frees the TMEM tile for the logits of t+1)
      float vc[kNp];
      const int bsel = t % kXBufs;
      if (!(ok = warp_wait(&s_full[0], t & 1, abort_flag, err))) break;
      tc_fence_after();
      tmem_ld32(tmem + lane_base + TM_S, vc);
      tmem_ld32(tmem + lane_base + TM_S + 32, vc + 32);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&s_empty[0]);
      // the peer's partial logits of the same tile, summed here
      if (!(ok = warp_wait_cluster(&x_full[bsel], (t / kXBufs) & 1, abort_flag, err))) break;
#pragma unroll
      for (int q4 = 0; q4 < kNp / 4; ++q4) {
        const float4 pv4 = *reinterpret_cast<const float4*>(xrow + bsel * kXBytes +
                                                            q4 * (kH * 16));
        vc[4 * q4] += pv4.x; vc[4 * q4 + 1] += pv4.y; vc[4 * q4 + 2] += pv4.z; vc[4 * q4 + 3] += pv4.w;
      }
      // buffer credit, one per warp; warp 0 re-arms the byte count first
      __syncwarp();
      if (lane == 0 && t + kXBufs < n_tiles) {
        if (quarter == 0) mbar_arrive_expect_tx_relaxed(&x_full[bsel], kXBytes);
        mbar_arrive_remote_relaxed(xempty_remote + bsel * 8);
      }
      // validity of the tile's 64 entries
      const uint32_t m_lo = __ballot_sync(0xffffffffu, rows_s[t * kNp + lane] >= 0);
      const uint32_t m_hi = __ballot_sync(0xffffffffu, rows_s[t * kNp + 32 + lane] >= 0);
      if ((m_lo & m_hi) != 0xffffffffu) {   // warp-uniform: the tile has skipped entries
#pragma unroll
        for (int j = 0; j < kNp; ++j)
          if ((((j < 32 ? m_lo >> j : m_hi >> (j - 32)) & 1u)) == 0) vc[j] = -INFINITY;
      }
      // online softmax in log2 units.  The tile max is taken on the raw sums
      // (scaling by sl2 > 0 keeps the order, and rounding is monotone) in
      // eight independent chains.
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = vc[i];
#pragma unroll
      for (int j = 8; j < kNp; ++j) mx[j & 7] = fmaxf(mx[j & 7], vc[j]);
#pragma unroll
      for (int w2 = 4; w2 >= 1; w2 >>= 1)
#pragma unroll
        for (int i = 0; i < w2; ++i) mx[i] = fmaxf(mx[i], mx[i + w2]);
      const float tmax = mx[0] * sl2;
      float alpha = 1.f;
      bool rescale = false;
      if (m_ref == -INFINITY) {
        m_ref = tmax;                      // accumulator is still zero: nothing to rescale
      } else if (tmax > m_ref + kRescaleLog2) {
        alpha = exp2f(m_ref - tmax);
        m_ref = tmax;
        rescale = true;
      }
      // the P tile is free, and PV(t-1) has landed in the accumulator, once
      // PV(t-1) is done
      if (!(ok = warp_wait(&p_empty[0], (t & 1) ^ 1, abort_flag, err))) break;
      tc_fence_after();
      uint8_t* prow = pbuf;
      // P = 2^(logit * sl2 - reference) in bf16, straight into the swizzled P
      // tile; the row sum adds the rounded values (what P.V multiplies), in
      // eight independent chains
      float ps[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) ps[i] = 0.f;
      // 2^(-inf) is 0 for skipped entries; a reference of -inf means every
      // entry so far was skipped (all probabilities 0)
      const float nmr = (m_ref == -INFINITY) ? 0.f : -m_ref;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        uint32_t w4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = 8 * u + 2 * e;
          const float e0 = ex2_approx(fmaf(vc[j], sl2, nmr));
          const float e1 = ex2_approx(fmaf(vc[j + 1], sl2, nmr));
          const __nv_bfloat162 p2 = __floats2bfloat162_rn(e0, e1);
          const float2 pr = __bfloat1622float2(p2);
          ps[2 * e] += pr.x;
          ps[2 * e + 1] += pr.y;
          w4[e] = *reinterpret_cast<const uint32_t*>(&p2);
        }
        *reinterpret_cast<uint4*>(prow + sw128_offset(h, u)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
      const float psum = ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
      l_sum = l_sum * alpha + psum;     // alpha == 1 for heads that did not move their reference
      // the accumulator rescaled once P is written (the logits are no longer
      // live); TMEM loads/stores are warp-collective: rescale when any head of
      // the warp needs it (the others multiply by 1)
      if (__any_sync(0xffffffffu, rescale)) {
        for (int c0 = 0; c0 < 256; c0 += 32) {
          float o[32];
          tmem_ld32(tmem + lane_base + TM_O + c0, o);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32f(tmem + lane_base + TM_O + c0, o);
        }
        tmem_st_wait();
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full[0]);
    }
    // ---- epilogue: normalise and store this CTA's 256 output dims ------------
    if (ok && warp_wait(o_done, 0, abort_flag, err)) {
      tc_fence_after();
      const int col0 = (int)rho * 256;
      const bool have = n_tiles > 0 && l_sum > 0.f;
      const float inv = have ? 1.f / l_sum : 0.f;
      for (int c0 = 0; c0 < 256; c0 += 32) {
        float o[32];
        if (n_tiles > 0) {
          tmem_ld32(tmem + lane_base + TM_O + c0, o);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0.f;
        }
        if (a.splits == 1) {
          bf16* dst = a.out + ((int64_t)r * kH + h) * DSI_D_LATENT + col0 + c0;
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            __align__(16) bf16 o8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) o8[e] = __float2bfloat16(o[i + e] * inv);
            *reinterpret_cast<uint4*>(dst + i) = *reinterpret_cast<const uint4*>(o8);
          }
        } else {
          float* dst = a.part_o + (((int64_t)r * a.splits + sp) * kH + h) * DSI_D_LATENT + col0 + c0;
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(dst + i) = make_float4(o[i], o[i + 1], o[i + 2], o[i + 3]);
        }
      }
      if (rho == 0) {
        if (a.splits == 1) {
          if (a.lse) a.lse[(int64_t)r * kH + h] = have ? (m_ref + log2f(l_sum)) / kLog2e : -INFINITY;
        } else {
          a.part_ml[((int64_t)r * a.splits + sp) * kH + h] =
              make_float2(have ? m_ref : -INFINITY, have ? l_sum : 0.f);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, TMEM_COLS);
  cluster_sync();   // the peer may still arrive on / write into this CTA until here
}

// ---------------------------------------------------------------------------
// Persistent form for prefills of at least two rows per cluster slot (bf16
// rows, no split, K <= 2048): each cluster takes rows pair, pair + nclu, ... in turn,
// so a row's set-up, first gathers and first logits overlap the end of the
// previous row instead of a new cluster's launch and pipeline fill.
//   - The exchange warps prepare the next row while the current one runs
//     (its entries translated into the other half of the entries' space, and
//     its tile count), after sending the current row's third partial tile;
//     `rows_ready[b]` publishes a row's entries, `rows_free[b]` returns them
//     (producers, softmax warps and the MMA thread).  At a row's start the
//     same warps write its query slice into TMEM (the previous row's logit
//     MMAs are complete by then: they have seen every one of its logit tiles)
//     and arrive on `q_ready`.
//   - Stages, logit/P tiles and exchange buffers run on the cluster's tile
//     count across rows, as if the rows were one long row; the accumulator
//     starts afresh at each row's first P.V, which follows the previous row's
//     epilogue (the softmax warps write the row's first P only after it).
//   - `q_ready` and `o_done` complete one phase per row with tiles, and rows
//     without tiles skip them, so no phase can complete twice before it is
//     waited for.
constexpr int kPerEntries = kMaxEntries / 2;   // each of the two row buffers
constexpr int NBARS_R = NBARS + 5;             // + rows_ready[2], rows_free[2], setup_bar
constexpr int OFF_MISC_R = OFF_BAR + NBARS_R * 8;
constexpr int SMEM_R = OFF_MISC_R + 64 + 1024;
static_assert(SMEM_R <= 227 * 1024, "shared memory (persistent form)");
constexpr int kSetupThreads = 128;             // the exchange warps
constexpr int kFreeArrivals = kProducerWarps + 4 + 1;   // producer warps, softmax warps, MMA thread

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
mla_tc_rows(const __grid_constant__ CUtensorMap lmap, CacheView c, MlaArgs a, int* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* s_full = bars + 2 * kStages;
  uint64_t* s_empty = s_full + 2;
  uint64_t* p_full = s_full + 4;
  uint64_t* p_empty = s_full + 6;
  uint64_t* q_ready = s_full + 8;
  uint64_t* o_done = s_full + 9;
  uint64_t* x_full = s_full + 10;
  uint64_t* x_empty = x_full + kXBufs;
  uint64_t* rows_ready = bars + NBARS;           // [2] a row's entries and tile count in place
  uint64_t* rows_free = rows_ready + 2;          // [2] every reader is done with them
  uint64_t* setup_bar = rows_ready + 4;          // the preparing warps' entries written
  int32_t* rows_s = reinterpret_cast<int32_t*>(smem + OFF_ROWS);   // [2][kPerEntries]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC_R);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC_R + 4);
  int* ntiles_s = reinterpret_cast<int*>(smem + OFF_MISC_R + 8);   // [2]
  int* lastv_s = reinterpret_cast<int*>(smem + OFF_MISC_R + 16);   // [2]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rho = cluster_ctarank();
  const uint32_t peer = rho ^ 1u;
  const int pair = blockIdx.x >> 1, nclu = gridDim.x >> 1;
  const int items = pair < a.rows ? (a.rows - pair + nclu - 1) / nclu : 0;   // rows of this cluster
  const int tiles_all = (a.K + kNp - 1) / kNp;
  const int span = tiles_all * kNp;                // entries of a row (<= kPerEntries)
  const int g0 = rho ? 4 : 0;
  constexpr uint32_t kXBytes = kH * kNp * 4;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1 + kLdgThreads);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 256);
      mbar_init(&p_full[i], 128);
      mbar_init(&p_empty[i], 1);
      mbar_init(&rows_ready[i], kSetupThreads);
      mbar_init(&rows_free[i], kFreeArrivals);
      lastv_s[i] = -1;
    }
    mbar_init(q_ready, kSetupThreads);
    mbar_init(o_done, 1);
    mbar_init(setup_bar, kSetupThreads);
    for (int i = 0; i < kXBufs; ++i) {
      mbar_init(&x_full[i], 1);
      mbar_init(&x_empty[i], 4);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, TMEM_COLS);
  grid_dep_wait();   // the indices (and queries) come from the kernels launched before
  __syncthreads();
  // the peer's first partial tile (every later one is expected as the
  // previous is consumed)
  if (tid == 0) mbar_arrive_expect_tx(&x_full[0], kXBytes);
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  grid_dep_launch();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ======================= gather: TMA part =================================
    if (lane < kTmaRowsP / 4) {
      if (lane == 0) prefetch_tmap(&lmap);
      int stage = 0;
      uint32_t ph = 0;
      bool issued[kStages] = {};
      uint32_t issued_ph[kStages] = {};
      const unsigned gmask = (1u << (kTmaRowsP / 4)) - 1u;
      bool ok = true;
      for (int i = 0; ok && i < items; ++i) {
        const int bsel = i & 1;
        ok = mbar_wait(&rows_ready[bsel], (uint32_t)(i >> 1) & 1u, abort_flag, err);
        ok = __all_sync(gmask, ok);
        if (!ok) break;
        const int n = ntiles_s[bsel];
        const int32_t* rs = rows_s + bsel * kPerEntries;
        for (int t = 0; t < n; ++t) {
          if (lane == 0) {
            ok = mbar_wait(&empty[stage], ph ^ 1, abort_flag, err);
            if (ok) mbar_arrive_expect_tx(&full[stage], kTmaChunks * kTmaRowsP * 128);
          }
          ok = __shfl_sync(gmask, ok, 0);
          if (!ok) break;
          issued[stage] = true;
          issued_ph[stage] = ph;
          uint8_t* st_base = smem + OFF_C + stage * kStageBytes;
          const int r4 = lane * 4;
          const int32_t* rw = rs + t * kNp + r4;
          const int y0 = max(rw[0], 0), y1 = max(rw[1], 0), y2 = max(rw[2], 0), y3 = max(rw[3], 0);
#pragma unroll
          for (int ch = 0; ch < kTmaChunks; ++ch)
            tma_gather4(st_base + ch * kChunkBytes + r4 * 128, &lmap, (g0 + ch) * 64, y0, y1, y2, y3,
                        &full[stage]);
          if (++stage == kStages) { stage = 0; ph ^= 1; }
        }
        __syncwarp(gmask);
        if (ok && lane == 0) mbar_arrive(&rows_free[bsel]);
      }
      if (lane == 0 && *abort_flag) {
        volatile int no_abort = 0;
        for (int s2 = 0; s2 < kStages; ++s2)
          if (issued[s2]) mbar_wait(&full[s2], issued_ph[s2], &no_abort, err, 100000000ull);
      }
    }
  } else if (warp < kProducerWarps) {
    // ======================= gather: cp.async part ============================
    int stage = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int i = 0; ok && i < items; ++i) {
      const int bsel = i & 1;
      if (!(ok = warp_wait(&rows_ready[bsel], (uint32_t)(i >> 1) & 1u, abort_flag, err))) break;
      const int n = ntiles_s[bsel];
      const int32_t* rs = rows_s + bsel * kPerEntries;
      for (int t = 0; t < n; ++t) {
        if (!(ok = mbar_wait(&empty[stage], ph ^ 1, abort_flag, err))) break;
        const uint32_t st_addr = smem_u32(smem + OFF_C + stage * kStageBytes);
        ldg_tile<kTmaRowsP>(st_addr, c.latent, rs + t * kNp, (warp - 1) * 32 + lane, rho, g0);
        cp_async_mbar_arrive_noinc(&full[stage]);
        if (++stage == kStages) { stage = 0; ph ^= 1; }
      }
      ok = __all_sync(0xffffffffu, ok);
      if (ok && lane == 0) mbar_arrive(&rows_free[bsel]);
    }
    cp_async_wait<0>();
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      // ===================== MMA issuer =======================================
      // Two cursors over the cluster's tiles: the logits (QK) and P.V, each
      // with its row and tile within the row; the QK cursor learns each row's
      // tile count (returning its entries' buffer at once) and stays at most
      // three rows ahead of P.V.
      int n0 = 0, n1 = 0, n2 = 0;                // tile counts of rows pi, pi + 1, pi + 2
      int qi = 0, qt = 0, qg = 0, nq = 0;        // QK: row, tile, tile count so far, rows with tiles
      bool qin = false;                          // the QK cursor has entered row qi
      bool qq = false;                           // ... and its queries are in TMEM
      int pi = 0, pt = 0, pg = 0;                // P.V: row, tile, tile count so far
      const uint32_t pbase = smem_u32(smem + OFF_P);
      uint64_t t_last = global_ns();
      uint32_t idle = 0;
      bool ok = true;
      while (ok && pi < items) {
        bool progress = false;
        // ---- P.V ----
        if (pi < qi || (pi == qi && qin)) {
          const int pn = n0;
          if (pt >= pn) {            // a row without tiles, or one just finished
            ++pi;
            pt = 0;
            n0 = n1;
            n1 = n2;
            progress = true;
          } else if (pg < qg && mbar_test_wait(&p_full[0], pg & 1)) {
            tc_fence_after();
            const int st = pg % kStages;
            const uint64_t pd = desc_sw128(pbase);
            const uint64_t vd = desc_sw128_mn(smem_u32(smem + OFF_C + st * kStageBytes), kChunkBytes);
#pragma unroll
            for (int kk = 0; kk < kNp / 16; ++kk)
              mma_bf16(tmem + TM_O, pd + (uint64_t)((kk * 32) >> 4), vd + (uint64_t)((kk * 2048) >> 4),
                       IDESC_O, (pt > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&p_empty[0]);
            mma_commit(&empty[st]);
            ++pg;
            if (++pt == pn) mma_commit(o_done);   // the row's output is complete
            progress = true;
          }
        }
        // ---- QK ----
        if (qi < items) {
          if (!qin) {
            if (qi - pi < 3 && mbar_test_wait(&rows_ready[qi & 1], (uint32_t)(qi >> 1) & 1u)) {
              const int nn = ntiles_s[qi & 1];
              if (qi == pi) n0 = nn; else if (qi == pi + 1) n1 = nn; else n2 = nn;
              mbar_arrive(&rows_free[qi & 1]);
              qin = true;
              qq = false;
              qt = 0;
              progress = true;
            }
          } else if (qt >= (qi == pi ? n0 : qi == pi + 1 ? n1 : n2)) {
            ++qi;
            qin = false;
            progress = true;
          } else if (!qq) {
            if (mbar_test_wait(q_ready, (uint32_t)nq & 1u)) {
              tc_fence_after();
              ++nq;
              qq = true;
              progress = true;
            }
          } else {
            const int st = qg % kStages;
            if (mbar_test_wait(&full[st], (qg / kStages) & 1) &&
                mbar_test_wait(&s_empty[0], (qg & 1) ^ 1)) {
              tc_fence_after();
              fence_proxy_async_smem();
              const uint32_t t_s = tmem + TM_S;
              const uint32_t st_base = smem_u32(smem + OFF_C + st * kStageBytes);
              const uint64_t d0 = desc_sw128(st_base);
              for (int k = 0; k < kQkTmem * 4; ++k)
                mma_bf16_tmem_a(t_s, tmem + TM_Q + k * 8,
                                d0 + (uint64_t)(((k >> 2) * kChunkBytes + (k & 3) * 32) >> 4),
                                IDESC_S, k > 0 ? 1u : 0u);
              {
                const uint64_t cd = desc_sw128(st_base + kQkTmem * kChunkBytes);
#pragma unroll
                for (int kk = 0; kk < kRopeHalf / 16; ++kk)
                  mma_bf16_tmem_a(t_s, tmem + TM_Q4 + kk * 8, cd + (uint64_t)((kk * 32) >> 4),
                                  IDESC_S, 1u);
              }
              mma_commit(&s_full[0]);
              ++qg;
              ++qt;
              progress = true;
            }
          }
        }
        if (progress) {
          idle = 0;
          t_last = global_ns();
        } else if (*abort_flag) {
          ok = false;
        } else if ((++idle & 255u) == 0 && global_ns() - t_last > kWaitLimitNs) {
          *abort_flag = 1;
          report(err, kErrTimeout);
          ok = false;
        }
      }
    }
    __syncwarp();
  } else if (warp < kSmWarp0) {
    // ======================= row preparation + logit exchange =================
    const int quarter = warp & 3;
    const int h = quarter * 32 + lane;
    const int et = tid - kExWarp0 * 32;              // 0..127
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    int setups = 0;
    // entries of row item i, translated into buffer i & 1, and its tile count
    auto prepare = [&](int i) -> bool {
      const int bsel = i & 1, use = i >> 1;
      if (use > 0 && !warp_wait(&rows_free[bsel], (uint32_t)(use - 1) & 1u, abort_flag, err))
        return false;
      const int r = pair + i * nclu;
      const int64_t n_vis = visible_len(c, r, a.decode, a.q_offset);
      const int b = seq_of_row(c, r, a.decode);
      const int32_t* irow = a.idx + (int64_t)r * a.K;
      int32_t* rs = rows_s + bsel * kPerEntries;
      // every index load is issued before any is used
      constexpr int kPP = kPerEntries / kSetupThreads;
      int pos[kPP];
#pragma unroll
      for (int u = 0; u < kPP; ++u) {
        const int jj = et + u * kSetupThreads;
        pos[u] = (jj < span && jj < a.K) ? __ldg(irow + jj) : -1;
      }
      int lv = -1;
#pragma unroll
      for (int u = 0; u < kPP; ++u) {
        const int jj = et + u * kSetupThreads;
        if (jj >= span) break;
        int pr = -1;
#ifdef DSI_CHECKED
        if (pos[u] >= n_vis) report(err, kErrBounds);
#endif
        if (pos_ok(pos[u], n_vis)) {
          const int64_t x = phys_row(c, b, pos[u], err);
          if (x >= 0) { pr = (int)x; lv = jj; }
        }
        rs[jj] = pr;
      }
      lv = __reduce_max_sync(0xffffffffu, lv);
      if (lane == 0 && lv >= 0) atomicMax(&lastv_s[bsel], lv);
      // the next row's query slice toward L2 (it is read at the row's start)
      if (i + 1 < items) {
        const bf16* qn = a.q + ((int64_t)(r + nclu) * kH + h) * DSI_D_QK;
#pragma unroll
        for (int k = 0; k < kQkTmem; ++k)
          asm volatile("prefetch.global.L2 [%0];" ::"l"(qn + (g0 + k) * 64));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(qn + DSI_D_LATENT + (int)rho * kRopeHalf));
      }
      mbar_arrive(setup_bar);
      if (et == 0) {
        if (!mbar_wait(setup_bar, (uint32_t)setups & 1u, abort_flag, err)) return false;
        const int l = lastv_s[bsel];
        ntiles_s[bsel] = l < 0 ? 0 : l / kNp + 1;
        lastv_s[bsel] = -1;
      }
      ++setups;
      mbar_arrive(&rows_ready[bsel]);
      return true;
    };
    // this row's query slice (four 64-dim blocks and the rope half) into
    // TMEM, eight 16-byte pieces a block
    auto load_q = [&](int r) {
      const uint4* qrow = reinterpret_cast<const uint4*>(a.q + ((int64_t)r * kH + h) * DSI_D_QK);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint4 qv[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) qv[k] = __ldg(qrow + (g0 + half * 2) * 8 + k);
#pragma unroll
        for (int cb = 0; cb < 2; ++cb) {
          uint32_t w32[32];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint4 v = qv[cb * 8 + k];
            w32[4 * k] = v.x; w32[4 * k + 1] = v.y; w32[4 * k + 2] = v.z; w32[4 * k + 3] = v.w;
          }
          tmem_st32(tmem + lane_base + TM_Q + (half * 2 + cb) * 32, w32);
        }
      }
      {
        uint32_t w32[32];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint4 v = k < kRopeHalf / 8
                              ? __ldg(qrow + (DSI_D_LATENT + (int)rho * kRopeHalf) / 8 + k)
                              : make_uint4(0, 0, 0, 0);
          w32[4 * k] = v.x; w32[4 * k + 1] = v.y; w32[4 * k + 2] = v.z; w32[4 * k + 3] = v.w;
        }
        tmem_st32(tmem + lane_base + TM_Q4, w32);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(q_ready);
    };
    const uint32_t x_remote = map_to_rank(smem_u32(smem + OFF_X), peer) + h * 16;
    const uint32_t xfull_remote = map_to_rank(smem_u32(x_full), peer);
    bool ok = items > 0 ? prepare(0) : true;
    int tg = 0;
    for (int i = 0; ok && i < items; ++i) {
      const int bsel = i & 1;
      if (!(ok = warp_wait(&rows_ready[bsel], (uint32_t)(i >> 1) & 1u, abort_flag, err))) break;
      const int n = ntiles_s[bsel];
      const bool more = i + 1 < items;
      if (n == 0) {
        if (more) ok = prepare(i + 1);
        continue;
      }
      // every logit tile of the previous rows has been seen complete, so no
      // MMA reads the query slice any more
      load_q(pair + i * nclu);
      const int prep_at = n > 2 ? 2 : n - 1;
      for (int t = 0; ok && t < n; ++t, ++tg) {
        float v[kNp];
        if (!(ok = warp_wait(&s_full[0], tg & 1, abort_flag, err))) break;
        tc_fence_after();
        tmem_ld32(tmem + lane_base + TM_S, v);
        tmem_ld32(tmem + lane_base + TM_S + 32, v + 32);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&s_empty[0]);
        if (!(ok = warp_wait_cluster(&x_empty[0], (tg & 1) ^ 1, abort_flag, err))) break;
#pragma unroll
        for (int q4 = 0; q4 < kNp / 4; ++q4)
          st_async_v4(x_remote + q4 * (kH * 16),
                      make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]),
                      xfull_remote);
        if (t == prep_at && more) ok = prepare(i + 1);
      }
    }
  } else {
    // ======================= softmax + epilogue ================================
    const int quarter = warp & 3;
    const int h = quarter * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    uint8_t* const pbuf = smem + OFF_P;
    const uint8_t* xrow = smem + OFF_X + h * 16;
    const uint32_t xempty_remote = map_to_rank(smem_u32(x_empty), peer);
    const float sl2 = a.scale * kLog2e;
    bool ok = true;
    int tg = 0, nrows = 0;                          // tiles so far; rows with tiles so far
    for (int i = 0; ok && i < items; ++i) {
      const int bsel = i & 1;
      const int r = pair + i * nclu;
      if (!(ok = warp_wait(&rows_ready[bsel], (uint32_t)(i >> 1) & 1u, abort_flag, err))) break;
      const int n = ntiles_s[bsel];
      const int32_t* rs = rows_s + bsel * kPerEntries;
      float m_ref = -INFINITY, l_sum = 0.f;
      for (int t = 0; ok && t < n; ++t, ++tg) {
        float vc[kNp];
        if (!(ok = warp_wait(&s_full[0], tg & 1, abort_flag, err))) break;
        tc_fence_after();
        tmem_ld32(tmem + lane_base + TM_S, vc);
        tmem_ld32(tmem + lane_base + TM_S + 32, vc + 32);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&s_empty[0]);
        if (!(ok = warp_wait_cluster(&x_full[0], tg & 1, abort_flag, err))) break;
#pragma unroll
        for (int q4 = 0; q4 < kNp / 4; ++q4) {
          const float4 pv4 = *reinterpret_cast<const float4*>(xrow + q4 * (kH * 16));
          vc[4 * q4] += pv4.x; vc[4 * q4 + 1] += pv4.y; vc[4 * q4 + 2] += pv4.z; vc[4 * q4 + 3] += pv4.w;
        }
        // buffer credit (the next tile may be in a later row; none after the
        // cluster's last row)
        __syncwarp();
        if (lane == 0 && !(i + 1 == items && t + 1 == n)) {
          if (quarter == 0) mbar_arrive_expect_tx_relaxed(&x_full[0], kXBytes);
          mbar_arrive_remote_relaxed(xempty_remote);
        }
        const uint32_t m_lo = __ballot_sync(0xffffffffu, rs[t * kNp + lane] >= 0);
        const uint32_t m_hi = __ballot_sync(0xffffffffu, rs[t * kNp + 32 + lane] >= 0);
        if ((m_lo & m_hi) != 0xffffffffu) {
#pragma unroll
          for (int j = 0; j < kNp; ++j)
            if ((((j < 32 ? m_lo >> j : m_hi >> (j - 32)) & 1u)) == 0) vc[j] = -INFINITY;
        }
        float mx[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mx[k] = vc[k];
#pragma unroll
        for (int j = 8; j < kNp; ++j) mx[j & 7] = fmaxf(mx[j & 7], vc[j]);
#pragma unroll
        for (int w2 = 4; w2 >= 1; w2 >>= 1)
#pragma unroll
          for (int k = 0; k < w2; ++k) mx[k] = fmaxf(mx[k], mx[k + w2]);
        const float tmax = mx[0] * sl2;
        float alpha = 1.f;
        bool rescale = false;
        if (m_ref == -INFINITY) {
          m_ref = tmax;
        } else if (tmax > m_ref + kRescaleLog2) {
          alpha = exp2f(m_ref - tmax);
          m_ref = tmax;
          rescale = true;
        }
        if (!(ok = warp_wait(&p_empty[0], (tg & 1) ^ 1, abort_flag, err))) break;
        tc_fence_after();
        float ps[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) ps[k] = 0.f;
        const float nmr = (m_ref == -INFINITY) ? 0.f : -m_ref;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          uint32_t w4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = 8 * u + 2 * e;
            const float e0 = ex2_approx(fmaf(vc[j], sl2, nmr));
            const float e1 = ex2_approx(fmaf(vc[j + 1], sl2, nmr));
            const __nv_bfloat162 p2 = __floats2bfloat162_rn(e0, e1);
            const float2 pr = __bfloat1622float2(p2);
            ps[2 * e] += pr.x;
            ps[2 * e + 1] += pr.y;
            w4[e] = *reinterpret_cast<const uint32_t*>(&p2);
          }
          *reinterpret_cast<uint4*>(pbuf + sw128_offset(h, u)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
        const float psum = ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
        l_sum = l_sum * alpha + psum;
        // the accumulator rescaled once this tile's P is written (the logits
        // are no longer live): P.V of the previous tile has landed in it, and
        // this tile's P.V waits for the arrival below
        if (__any_sync(0xffffffffu, rescale)) {
          for (int c0 = 0; c0 < 256; c0 += 32) {
            float o[32];
            tmem_ld32(tmem + lane_base + TM_O + c0, o);
            tmem_ld_wait();
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] *= alpha;
            tmem_st32f(tmem + lane_base + TM_O + c0, o);
          }
          tmem_st_wait();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&p_full[0]);
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&rows_free[bsel]);
      // ---- this row's output: normalise and store this CTA's 256 dims ---------
      const bool have = n > 0 && l_sum > 0.f;
      if (n > 0) {
        if (!(ok = warp_wait(o_done, (uint32_t)nrows & 1u, abort_flag, err))) break;
        tc_fence_after();
        ++nrows;
      }
      const int col0 = (int)rho * 256;
      const float inv = have ? 1.f / l_sum : 0.f;
      bf16* dst0 = a.out + ((int64_t)r * kH + h) * DSI_D_LATENT + col0;
      for (int c0 = 0; c0 < 256; c0 += 32) {
        float o[32];
        if (n > 0) {
          tmem_ld32(tmem + lane_base + TM_O + c0, o);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = 0.f;
        }
#pragma unroll
        for (int k = 0; k < 32; k += 8) {
          __align__(16) bf16 o8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) o8[e] = __float2bfloat16(o[k + e] * inv);
          *reinterpret_cast<uint4*>(dst0 + c0 + k) = *reinterpret_cast<const uint4*>(o8);
        }
      }
      if (rho == 0 && a.lse)
        a.lse[(int64_t)r * kH + h] = have ? (m_ref + log2f(l_sum)) / kLog2e : -INFINITY;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, TMEM_COLS);
  cluster_sync();
}

}  // namespace

bool tc_mla_supported(int n_heads) { return n_heads == kH; }

// FP8 latent rows are read as 16-byte pieces at row offsets of 576 bytes.
bool tc_mla_fp8_ok(const CacheView& c, const float* latent_scale) {
  return latent_scale != nullptr && (reinterpret_cast<uintptr_t>(c.latent) & 15) == 0;
}

// Physical rows must fit the kernel's 32-bit row ids.
bool tc_mla_cache_ok(const CacheView& c) {
  const uint64_t rows = c.block_table ? (uint64_t)c.num_pages * c.page_size
                                      : (uint64_t)c.batch * c.s_max;
  return rows < (1ull << 31);
}

int tc_mla_splits(int rows, int K, size_t ws_bytes) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int tiles = (K + kNp - 1) / kNp;
  int splits = 1;
  while (2L * rows * splits * 2 <= sms && tiles / (splits * 2) >= 4) splits *= 2;
  while (splits > 1 && mla_partials_bytes(rows, kH, splits) > ws_bytes) splits /= 2;
  return splits;
}

// Two-CTA clusters of the persistent form that fit on the device at once
// (queried once per device; 0 when the query fails).
static int rows_slots() {
  static std::atomic<int> cached[16];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 16) return 0;
  const int v = cached[dev].load(std::memory_order_relaxed);
  if (v != 0) return v > 0 ? v : 0;
  int slots = 0;
  cudaLaunchConfig_t qc = {};
  qc.gridDim = dim3(2);
  qc.blockDim = dim3(kThreads);
  qc.dynamicSmemBytes = SMEM_R;
  cudaLaunchAttribute ca;
  ca.id = cudaLaunchAttributeClusterDimension;
  ca.val.clusterDim.x = 2;
  ca.val.clusterDim.y = 1;
  ca.val.clusterDim.z = 1;
  qc.attrs = &ca;
  qc.numAttrs = 1;
  if (cudaOccupancyMaxActiveClusters(&slots, mla_tc_rows, &qc) != cudaSuccess) {
    cudaGetLastError();
    slots = 0;
  }
  cached[dev].store(slots > 0 ? slots : -1, std::memory_order_relaxed);
  return slots;
}

cudaError_t launch_sparse_mla_tc(const bf16* q, const CacheView& c, const float* latent_scale,
                                 const int32_t* idx, int rows, int H, int K, int decode,
                                 int64_t q_offset, float scale, bf16* out, float* lse, void* ws,
                                 size_t ws_bytes, int* err, cudaStream_t st) {
  MlaArgs a;
  a.q = q;
  a.idx = idx;
  a.out = out;
  a.lse = lse;
  a.q_offset = q_offset;
  a.scale = scale;
  a.rows = rows;
  a.K = K;
  a.decode = decode;
  a.splits = tc_mla_splits(rows, K, ws ? ws_bytes : 0);
  a.part_o = nullptr;
  a.part_ml = nullptr;
  if (a.splits > 1) {
    const size_t n = (size_t)rows * a.splits * H;
    a.part_o = reinterpret_cast<float*>(ws);
    a.part_ml = reinterpret_cast<float2*>(reinterpret_cast<char*>(ws) + n * DSI_D_LATENT * sizeof(float));
  }
  // bf16 latent rows as a 2D tensor [rows, 576], one-row boxes of 64 dims
  // (gather4); FP8 rows are read with plain loads (no tensor map)
  const bool f8 = latent_scale != nullptr;
  const uint64_t lrows = c.block_table ? (uint64_t)c.num_pages * c.page_size
                                       : (uint64_t)c.batch * c.s_max;
  CUtensorMap lmap;
  memset(&lmap, 0, sizeof(lmap));
  if (!f8 &&
      !tma_map_2d(&lmap, c.latent, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, lrows, DSI_D_QK, 64, 1))
    return cudaErrorInvalidValue;
  // a prefill of at least two rows per cluster slot (bf16 rows, no split,
  // K <= 2048): the persistent form, one cluster per slot taking rows in turn
  // (rows of a prefill are dealt round-robin, so every slot gets a like mix;
  // decode batches, whose rows differ in length at random, keep one cluster a
  // row, which the hardware places as slots free up)
  if (!decode && !f8 && a.splits == 1 && (K + kNp - 1) / kNp * kNp <= kPerEntries) {
    cudaError_t e = cudaFuncSetAttribute(mla_tc_rows, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SMEM_R);
    if (e != cudaSuccess) return e;
    const int slots = rows_slots();
    if (slots > 0 && rows >= 2 * slots) {
      e = launch_overlapped(mla_tc_rows, dim3(2u * (unsigned)slots), dim3(kThreads), SMEM_R, st,
                            lmap, c, a, err);
      note_launch();
      return e;
    }
  }
  auto kern = f8 ? mla_tc<true> : mla_tc<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (e != cudaSuccess) return e;
  const long blocks = 2L * rows * a.splits;
  if (blocks > 0x7fffffffL) return cudaErrorInvalidValue;
  e = launch_overlapped(kern, dim3((unsigned)blocks), dim3(kThreads), SMEM, st, lmap, c,
                        latent_scale, a, err);
  note_launch();
  if (e != cudaSuccess || a.splits == 1) return e;
  return launch_mla_combine(a.part_o, a.part_ml, rows, H, a.splits, out, lse, st);
}

}  // namespace dsi
