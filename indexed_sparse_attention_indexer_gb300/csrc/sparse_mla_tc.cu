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
//   CTA 0: logits over key dims   0..319, output dims   0..255
//   CTA 1: logits over key dims 320..575, output dims 256..511
// Each CTA gathers only the 320 dims of every selected row that it needs (no
// row is fetched twice), keeps its slice of the queries in TMEM as the A
// operand of the logit MMA, and keeps its half of the output accumulator in
// TMEM.  The two partial logit tiles (128 heads x 64 positions, fp32) are
// swapped through distributed shared memory, so both CTAs hold the same
// logits and take the same softmax decisions.  Per 64-position tile:
//   producers (4 warps): cp.async gather of the tile's rows into a
//     128-byte-swizzled stage (ring of 4), zero rows for skipped entries;
//   MMA (1 thread):  S = Qslice . C^T  (A from TMEM, B K-major from the stage)
//                    O += P . V        (A = P K-major, B = V MN-major, same stage)
//   softmax (4 warps, one head per thread): read S from TMEM, exchange with
//     the peer, online softmax in log2 units with a lazily moved reference max
//     (the accumulator is rescaled only when the max grows by more than 2^8),
//     P in bf16 to shared memory.
// Every wait is bounded; the cluster syncs once after set-up and once before
// exit so no CTA leaves while its peer may still write into it.
#include "kernels.h"
#include "tc_common.cuh"

namespace dsi {
using namespace tc;

namespace {

constexpr int kH = 128;                        // heads (MMA M)
constexpr int kNp = 64;                        // positions per tile (MMA N of the logits)
constexpr int kChunks = 5;                     // 64-dim blocks each CTA gathers per row
constexpr int kStages = 4;
constexpr int kChunkBytes = kNp * 128;         // one 64-dim block of a tile: 8 KB
constexpr int kStageBytes = kChunks * kChunkBytes;
constexpr int kProducerWarps = 4;
constexpr int kMmaWarp = kProducerWarps;       // warp 4
constexpr int kThreads = (kProducerWarps + 1 + 4) * 32;   // 288
constexpr int kProducers = kProducerWarps * 32;

constexpr int OFF_C = 0;
constexpr int OFF_P = OFF_C + kStages * kStageBytes;      // P [128 x 64] bf16, 16 KB
constexpr int OFF_X = OFF_P + kH * kNp * 2;               // peer logits [128 x 64] fp32, 32 KB
constexpr int OFF_BAR = OFF_X + kH * kNp * 4;
constexpr int NBARS = 2 * kStages + 8;
constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
constexpr int SMEM = OFF_MISC + 64 + 1024;

constexpr uint32_t TM_S = 0;      // logits, 64 columns
constexpr uint32_t TM_Q = 64;     // query slice, 160 (CTA 0) or 128 (CTA 1) columns
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

__device__ __forceinline__ bool pos_ok(int pos, int64_t n_vis) {
#ifdef DSI_CHECKED
  return pos >= 0 && pos < n_vis;
#else
  (void)n_vis;
  return pos >= 0;
#endif
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
mla_tc(CacheView c, MlaArgs a, int* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* s_full = bars + 2 * kStages;
  uint64_t* s_empty = s_full + 1;
  uint64_t* p_full = s_full + 2;
  uint64_t* p_empty = s_full + 3;
  uint64_t* q_ready = s_full + 4;
  uint64_t* x_full = s_full + 5;
  uint64_t* x_empty = s_full + 6;
  uint64_t* o_done = s_full + 7;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  int* last_valid = reinterpret_cast<int*>(smem + OFF_MISC + 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rho = cluster_ctarank();          // which half of the dims this CTA owns
  const int pair = blockIdx.x >> 1;
  const int r = pair / a.splits, sp = pair % a.splits;
  const int b = a.decode ? r : 0;
  const int64_t n_vis = visible_len(c, r, a.decode, a.q_offset);
  const int tiles_all = (a.K + kNp - 1) / kNp;
  const int tiles_per = (tiles_all + a.splits - 1) / a.splits;
  const int j_begin = sp * tiles_per * kNp;
  const int j_end = min(a.K, j_begin + tiles_per * kNp);
  const int32_t* irow = a.idx + (int64_t)r * a.K;
  const int g0 = rho ? 4 : 0;                      // first gathered 64-dim block
  const int qk_first = rho ? 1 : 0;                // first stage block used by the logits

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) { mbar_init(&full[s], kProducers); mbar_init(&empty[s], 1); }
    mbar_init(s_full, 1);
    mbar_init(s_empty, 128);
    mbar_init(p_full, 128);
    mbar_init(p_empty, 1);
    mbar_init(q_ready, 128);
    mbar_init(x_full, 128);
    mbar_init(x_empty, 128);
    mbar_init(o_done, 1);
    *abort_flag = 0;
    *last_valid = -1;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) tmem_alloc(tmem_slot, TMEM_COLS);
  __syncthreads();
  // last valid entry of this split (tiles past it are skipped)
  for (int j = j_begin + tid; j < j_end; j += kThreads)
    if (pos_ok(__ldg(irow + j), n_vis)) atomicMax(last_valid, j);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();   // the peer's barriers exist before anyone arrives on them
  const uint32_t tmem = *tmem_slot;
  const int n_tiles = *last_valid < 0 ? 0 : (*last_valid - j_begin) / kNp + 1;

  if (warp < kProducerWarps) {
    // ======================= gather producers =================================
    const int pt = tid;                 // 0..127
    const int rr = pt >> 1;             // row of the tile
    const int half = pt & 1;            // which 20 of the row's 40 16-byte pieces
    int stage = 0, prev = -1;
    uint32_t ph = 0;
    for (int t = 0; t < n_tiles; ++t) {
      if (!mbar_wait(&empty[stage], ph ^ 1, abort_flag, err)) break;
      const int j = j_begin + t * kNp + rr;
      int pos = j < j_end ? __ldg(irow + j) : -1;
#ifdef DSI_CHECKED
      if (pos >= n_vis) { report(err, kErrBounds); pos = -1; }
#endif
      const int64_t prow = pos >= 0 ? phys_row(c, b, pos, err) : -1;
      uint8_t* st_base = smem + OFF_C + stage * kStageBytes;
      const uint32_t st_addr = smem_u32(st_base);
#pragma unroll 4
      for (int i = 0; i < 20; ++i) {
        const int pi = half * 20 + i;
        const int ch = pi >> 3, u = pi & 7;
        const uint32_t off = ch * kChunkBytes + sw128_offset(rr, u);
        if (prow >= 0)
          cp_async_16(st_addr + off, c.latent + prow * DSI_D_QK + (g0 + ch) * 64 + u * 8);
        else
          *reinterpret_cast<uint4*>(st_base + off) = make_uint4(0, 0, 0, 0);
      }
      cp_async_commit();
      if (prev >= 0) {
        cp_async_wait<1>();
        fence_proxy_async_smem();
        mbar_arrive(&full[prev]);
      }
      prev = stage;
      if (++stage == kStages) { stage = 0; ph ^= 1; }
    }
    cp_async_wait<0>();
    fence_proxy_async_smem();
    if (prev >= 0) mbar_arrive(&full[prev]);
  } else if (warp == kMmaWarp) {
    // ======================= MMA issuer =======================================
    if (lane == 0) {
      bool ok = mbar_wait(q_ready, 0, abort_flag, err);
      tc_fence_after();
      int stage = 0, prev = -1;
      uint32_t ph = 0;
      auto pv = [&](int tt, int st) -> bool {
        if (!mbar_wait(p_full, tt & 1, abort_flag, err)) return false;
        tc_fence_after();
        const uint32_t pbase = smem_u32(smem + OFF_P);
        const uint32_t vbase = smem_u32(smem + OFF_C + st * kStageBytes);
#pragma unroll
        for (int kk = 0; kk < kNp / 16; ++kk)
          mma_bf16(tmem + TM_O, desc_sw128(pbase + kk * 32), desc_sw128_mn(vbase + kk * 2048, kChunkBytes),
                   IDESC_O, (tt > 0 || kk > 0) ? 1u : 0u);
        mma_commit(p_empty);
        mma_commit(&empty[st]);
        return true;
      };
      for (int t = 0; ok && t < n_tiles; ++t) {
        if (!mbar_wait(&full[stage], ph, abort_flag, err)) break;
        if (!mbar_wait(s_empty, (t & 1) ^ 1, abort_flag, err)) break;
        tc_fence_after();
        const uint32_t cbase = smem_u32(smem + OFF_C + stage * kStageBytes);
        int k = 0;
        for (int kc = qk_first; kc < kChunks; ++kc) {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks, ++k)
            mma_bf16_tmem_a(tmem + TM_S, tmem + TM_Q + k * 8,
                            desc_sw128(cbase + kc * kChunkBytes + ks * 32), IDESC_S, k > 0 ? 1u : 0u);
        }
        mma_commit(s_full);
        if (prev >= 0 && !pv(t - 1, prev)) break;
        prev = stage;
        if (++stage == kStages) { stage = 0; ph ^= 1; }
      }
      if (!*abort_flag && prev >= 0) pv(n_tiles - 1, prev);
      mma_commit(o_done);
    }
    __syncwarp();
  } else {
    // ======================= softmax + epilogue ================================
    const int quarter = warp & 3;
    const int h = quarter * 32 + lane;               // head = TMEM lane
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    // this CTA's slice of the query row into TMEM (columns pack bf16 pairs)
    {
      const int qcols = (kChunks - qk_first) * 32;
      const uint32_t* qsrc = reinterpret_cast<const uint32_t*>(
          a.q + ((int64_t)r * kH + h) * DSI_D_QK + (g0 + qk_first) * 64);
      for (int c0 = 0; c0 < qcols; c0 += 32) {
        uint32_t w32[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(qsrc + c0) + i);
          w32[4 * i] = v.x; w32[4 * i + 1] = v.y; w32[4 * i + 2] = v.z; w32[4 * i + 3] = v.w;
        }
        tmem_st32(tmem + lane_base + TM_Q + c0, w32);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(q_ready);
    }
    const uint32_t peer = rho ^ 1u;
    const uint32_t x_remote = map_to_rank(smem_u32(smem + OFF_X), peer);
    const uint32_t xfull_remote = map_to_rank(smem_u32(x_full), peer);
    const uint32_t xempty_remote = map_to_rank(smem_u32(x_empty), peer);
    const float* xrow = reinterpret_cast<const float*>(smem + OFF_X) + h * kNp;
    uint8_t* prow = smem + OFF_P;
    const float sl2 = a.scale * kLog2e;
    float m_ref = -INFINITY, l_sum = 0.f;
    bool ok = true;
    for (int t = 0; t < n_tiles; ++t) {
      if (!(ok = warp_wait(s_full, t & 1, abort_flag, err))) break;
      tc_fence_after();
      float v[kNp];
      tmem_ld32(tmem + lane_base + TM_S, v);
      tmem_ld32(tmem + lane_base + TM_S + 32, v + 32);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(s_empty);
      // validity of the tile's 64 positions (two ballots per warp)
      const int jt = j_begin + t * kNp;
      const int pa = jt + lane < j_end ? __ldg(irow + jt + lane) : -1;
      const int pb = jt + 32 + lane < j_end ? __ldg(irow + jt + 32 + lane) : -1;
      const uint32_t m_lo = __ballot_sync(0xffffffffu, pos_ok(pa, n_vis));
      const uint32_t m_hi = __ballot_sync(0xffffffffu, pos_ok(pb, n_vis));
      // swap partial logits with the peer CTA
      if (!(ok = warp_wait_cluster(x_empty, (t & 1) ^ 1, abort_flag, err))) break;
#pragma unroll
      for (int q4 = 0; q4 < kNp / 4; ++q4)
        st_cluster_v4(x_remote + h * kNp * 4 + ((q4 ^ (h & 15)) << 4),
                      make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]));
      mbar_arrive_remote(xfull_remote);
      if (!(ok = warp_wait_cluster(x_full, t & 1, abort_flag, err))) break;
#pragma unroll
      for (int q4 = 0; q4 < kNp / 4; ++q4) {
        const float4 pv4 = *reinterpret_cast<const float4*>(
            reinterpret_cast<const uint8_t*>(xrow) + ((q4 ^ (h & 15)) << 4));
        v[4 * q4] += pv4.x; v[4 * q4 + 1] += pv4.y; v[4 * q4 + 2] += pv4.z; v[4 * q4 + 3] += pv4.w;
      }
      mbar_arrive_remote(xempty_remote);
      // online softmax in log2 units
      float tmax = -INFINITY;
#pragma unroll
      for (int j = 0; j < kNp; ++j) {
        const bool on = ((j < 32 ? m_lo >> j : m_hi >> (j - 32)) & 1u) != 0;
        v[j] = on ? v[j] * sl2 : -INFINITY;
        tmax = fmaxf(tmax, v[j]);
      }
      float alpha = 1.f;
      bool rescale = false;
      if (m_ref == -INFINITY) {
        m_ref = tmax;                      // accumulator is still zero: nothing to rescale
      } else if (tmax > m_ref + kRescaleLog2) {
        alpha = exp2f(m_ref - tmax);
        m_ref = tmax;
        rescale = true;
      }
      uint32_t pk[kNp / 2];
      float psum = 0.f;
#pragma unroll
      for (int j = 0; j < kNp; j += 2) {
        const float e0 = (v[j] == -INFINITY) ? 0.f : exp2f(v[j] - m_ref);
        const float e1 = (v[j + 1] == -INFINITY) ? 0.f : exp2f(v[j + 1] - m_ref);
        const __nv_bfloat162 p2 = __floats2bfloat162_rn(e0, e1);
        const float2 pr = __bfloat1622float2(p2);
        psum += pr.x + pr.y;
        pk[j / 2] = *reinterpret_cast<const uint32_t*>(&p2);
      }
      // PV(t-1) must be complete before P and the accumulator are touched
      if (!(ok = warp_wait(p_empty, (t & 1) ^ 1, abort_flag, err))) break;
      tc_fence_after();
      // TMEM loads/stores are warp-collective: rescale when any head of the
      // warp needs it (the others multiply by 1)
      if (__any_sync(0xffffffffu, rescale)) {
        for (int c0 = 0; c0 < 256; c0 += 32) {
          float o[32];
          tmem_ld32(tmem + lane_base + TM_O + c0, o);
          tmem_ld_wait();
          uint32_t ob[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) ob[i] = __float_as_uint(o[i] * alpha);
          tmem_st32(tmem + lane_base + TM_O + c0, ob);
        }
        tmem_st_wait();
        l_sum *= alpha;   // alpha == 1 for heads that did not move their reference
      }
      l_sum += psum;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        *reinterpret_cast<uint4*>(prow + sw128_offset(h, u)) =
            make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
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

}  // namespace

bool tc_mla_supported(int n_heads) { return n_heads == kH; }

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

cudaError_t launch_sparse_mla_tc(const bf16* q, const CacheView& c, const int32_t* idx, int rows,
                                 int H, int K, int decode, int64_t q_offset, float scale, bf16* out,
                                 float* lse, void* ws, size_t ws_bytes, int* err, cudaStream_t st) {
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
  cudaError_t e = cudaFuncSetAttribute(mla_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (e != cudaSuccess) return e;
  const long blocks = 2L * rows * a.splits;
  if (blocks > 0x7fffffffL) return cudaErrorInvalidValue;
  mla_tc<<<(unsigned)blocks, kThreads, SMEM, st>>>(c, a, err);
  note_launch();
  e = cudaGetLastError();
  if (e != cudaSuccess || a.splits == 1) return e;
  return launch_mla_combine(a.part_o, a.part_ml, rows, H, a.splits, out, lse, st);
}

}  // namespace dsi
