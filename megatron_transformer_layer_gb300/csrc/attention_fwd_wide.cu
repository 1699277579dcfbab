// Causal flash attention forward with 256-key blocks (sm_103a, tcgen05),
// over the whole score matrix or over one rectangle of it (the
// context-parallel path: each rectangle merges its O and log-sum-exp into
// the rows' running fp32 result).
//
// S_j = Q K_j^T runs as 128 x 256 x 16 MMAs, which keep the tensor pipe
// busier per instruction than 128 x 128 ones (the shared-memory operand
// reads per flop drop by a quarter), and P gets tensor-memory columns of its
// own, so S_{j+1} can be formed while the softmax of block j still runs and
// the tensor core alternates S_{j+1} and O += P_j V_j without waiting.
//
// One CTA per (128-query tile, head, batch), heaviest tiles first; 320
// threads:
//   warp 0      TMA: Q once; K_j (256 keys) into a 2-deep ring; V_j as two
//               128-key halves into a ring of kVSlots half-tiles (2 at
//               D = 128, where shared memory ends), each half released as
//               soon as its 8 PV steps are done
//   warp 1      allocates the 512 TMEM columns and issues tcgen05.mma from
//               one thread
//   warps 2..9  softmax, two warps per TMEM lane quarter: warp (quarter,
//               half) takes keys [128 half, 128 half + 128) of its 32 rows;
//               the halves of a row exchange their maxima and sums through
//               shared memory behind an mbarrier (bounded wait)
// TMEM: S [0, 256), O [256, 256 + D), P [384, 512) (bf16 pairs, 256 keys).
// Products in issue order: S_0, S_1, then for each block j: O += P_j V_j
// (once the softmax has written P_j), S_{j+2} (once the softmax holds S_{j+1}
// in registers).  Before it overwrites P the softmax of block j waits for
// PV_{j-1}; before it rescales O, for the same product.
// Softmax as in the 128-key kernel: exp2 with log2(e)/sqrt(d) folded in, O
// rescaled in TMEM only when a row's max grows by more than 8 (log2 units),
// the final division by the sum taken against the same max.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>

#include "mc_layer_internal.h"
#include "ptx.cuh"

namespace mc {
namespace {

constexpr int kWideThreads = 320;
constexpr int kKeys = 256;  // keys per block
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;

template <int D>
struct WideCfg {
  static constexpr int kChunks = D / 64;             // 128-byte boxes per row
  static constexpr int kQTile = 128 * D * 2;         // Q [128][D] bf16
  static constexpr int kKVTile = kKeys * D * 2;      // K or V [256][D] bf16
  static constexpr int kChunkBytes = kKeys * 128;    // one 64-wide d chunk of 256 rows
  static constexpr int kVHalf = 128 * D * 2;         // V half-tile [128][D] bf16
  static constexpr int kVSlots = D == 64 ? 4 : 2;
  static constexpr int kXch = 2 * 2 * 128 * 4;       // [parity][half][row] floats
  static constexpr int kBars = 24 * 8;
  // The dynamic shared memory starts 1024-byte aligned (checked at run time),
  // so no alignment slack is reserved: at D = 128 it would not fit.
  static constexpr int kUsed = kQTile + 2 * kKVTile + kVSlots * kVHalf + kXch + kBars;
  static constexpr int kSmem = kUsed > 116 * 1024 ? kUsed : 116 * 1024;
  static_assert(kUsed <= 227 * 1024, "wide forward shared memory");
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0, kColO = 256, kColP = 384;
};

// A rectangle of the causal score matrix: query rows [base, base + len)
// (whole 128-row tiles) against keys [key_lo, key_hi) (key_lo a multiple of
// 128).  The whole matrix is {0, s, 0, INT_MAX} and writes bf16 O and the
// fp32 log-sum-exp.  A partial rectangle (the context-parallel path) merges
// its O and log-sum-exp into the rows' running ones by the log-sum-exp rule:
// `out` [b, s, a] holds O normalised over the keys seen so far, `lse2`
// [b, H, s] their log2-sum-exp (indexed by the absolute row).  Without
// kCpAccMerge in `mode` there is nothing to merge with; with kCpAccFinal
// the merged result goes to the kernel's bf16 O and natural-log lse.
struct WideRect {
  int base, len;
  int key_lo, key_hi;
  int mode;
};

// The rectangles of one launch (disjoint query rows): CTAs
// [cta_end[i - 1], cta_end[i]) take the 128-row query tiles of rectangle i,
// heaviest first.
struct WideRects {
  int n;
  int cta_end[kCpMaxRects];
  WideRect r[kCpMaxRects];
  float* out;
  float* lse2;
  int head_major;  // the whole matrix: the grid order (attention_cta)
};

template <int D, bool PART>
__global__ void __launch_bounds__(kWideThreads, 1)
    attn_fwd_wide_kernel(const __grid_constant__ CUtensorMap tm, uint16_t* __restrict__ out,
                         float* __restrict__ lse, int s, int H, int* status,
                         const __grid_constant__ WideRects rects) {
  using C = WideCfg<D>;
  constexpr int VS = C::kVSlots;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {  // the 128-byte swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) record_error(status, MC_ERR_DEVICE_BOUNDS, kSiteAttention);
    return;
  }
  uint8_t* sQ = smem;
  uint8_t* sK[2] = {smem + C::kQTile, smem + C::kQTile + C::kKVTile};
  uint8_t* sV0 = smem + C::kQTile + 2 * C::kKVTile;
  float* xch = reinterpret_cast<float*>(sV0 + VS * C::kVHalf);
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(xch) + C::kXch);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;    // [2]
  uint64_t* k_empty = bars + 3;   // [2]  after S_j
  uint64_t* v_full = bars + 5;    // [4] per half-tile slot (VS used)
  uint64_t* v_empty = bars + 9;   // [4]  after the half's PV steps
  uint64_t* s_full = bars + 13;   // S_j in TMEM
  uint64_t* s_free = bars + 14;   // the softmax holds S_j in registers (256 threads)
  uint64_t* p_full = bars + 15;   // P_j in TMEM (256 threads)
  uint64_t* pv_done = bars + 16;  // PV_j complete
  uint64_t* o_final = bars + 17;  // single use: the last PV is complete
  uint64_t* drain = bars + 18;
  uint64_t* xbar = bars + 19;     // [4] per lane quarter: the two halves' exchange (64 threads)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 23);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int a = H * D;
  // this CTA's rectangle (the whole matrix: one) and query tile, heaviest first
  int ri = 0;
  if constexpr (PART)
    while (ri + 1 < rects.n && static_cast<int>(blockIdx.x) >= rects.cta_end[ri]) ++ri;
  const WideRect rect = rects.r[ri];
  const int cta0 = ri > 0 ? rects.cta_end[ri - 1] : 0;
  int t_heavy, hh, bi;
  attention_cta(!PART && rects.head_major, H, t_heavy, hh, bi);
  const int q_blk =
      PART ? rect.base / 128 + (rect.len / 128 - 1 - (static_cast<int>(blockIdx.x) - cta0))
           : (s + 127) / 128 - 1 - t_heavy;
  const int q0 = q_blk * 128;
  // (the whole matrix: keys from 0, masked past s)
  const int k_lo = PART ? rect.key_lo : 0;
  const int k_end = PART ? min(s, rect.key_hi) : s;  // keys past it are masked
  const int k_last = min(q0 + 128, k_end);           // no block starts at or after it
  const int n_kb = (k_last - k_lo + kKeys - 1) / kKeys;   // 256-key blocks
  if (n_kb < 1) {  // an empty rectangle: the caller's schedule never makes one
    if (threadIdx.x == 0) record_error(status, MC_ERR_DEVICE_BOUNDS, kSiteAttention);
    return;
  }

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < VS; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, 256);
    mbar_init(p_full, 256);
    mbar_init(pv_done, 1);
    mbar_init(o_final, 1);
    mbar_init(drain, 1);
    for (int i = 0; i < 4; ++i) mbar_init(&xbar[i], 64);
    fence_mbar_init();
    tma_prefetch_desc(&tm);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the previous kernel on the stream has completed
  const uint32_t tS = tmem + C::kColS, tO = tmem + C::kColO, tP = tmem + C::kColP;

  if (warp == 0) {
    if (lane == 0) {
      // -------------------------------------------------------- producer
      mbar_arrive_expect_tx(q_full, C::kQTile);
      for (int c = 0; c < C::kChunks; ++c)
        tma_load_3d(sQ + c * 16384, &tm, q_full, hh * D + c * 64, q0, bi);
      // Order K_0, then per block j >= 1: K_j, V_{j-1} (both halves); V_{n-1}
      // last.  K_j waits for S_{j-2}, a V half for the PV steps that read
      // its slot last.
      int k_issued = 0, v_issued = 0;  // V counted in half-tiles
      bool ok = true;
      auto load_v = [&](int jv) {
        for (int h = 0; ok && h < 2; ++h) {
          const int u = 2 * jv + h, slot = u % VS;
          if (!mbar_wait(&v_empty[slot], ((u / VS) & 1) ^ 1u, status, kSiteAttention)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&v_full[slot], C::kVHalf);
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d(sV0 + slot * C::kVHalf + c * 16384, &tm, &v_full[slot],
                        2 * a + hh * D + c * 64, k_lo + jv * kKeys + h * 128, bi);
          ++v_issued;
        }
      };
      for (int j = 0; ok && j <= n_kb; ++j) {
        if (j < n_kb) {
          const int ks = j & 1;
          if (!mbar_wait(&k_empty[ks], ((j >> 1) & 1) ^ 1u, status, kSiteAttention)) break;
          mbar_arrive_expect_tx(&k_full[ks], C::kKVTile);
          for (int c = 0; c < C::kChunks; ++c)
            for (int h = 0; h < 2; ++h)
              tma_load_3d(sK[ks] + c * C::kChunkBytes + h * 16384, &tm, &k_full[ks],
                          a + hh * D + c * 64, k_lo + j * kKeys + h * 128, bi);
          ++k_issued;
        }
        if (j >= 1) load_v(j - 1);
      }
      pdl_launch();  // every load of this CTA is issued
      // Copies still in flight must land before the CTA exits.
      mbar_wait(q_full, 0, status, kSiteAttention, 200000000ull, false);
      for (int j = k_issued - 1; j >= 0 && j >= k_issued - 2; --j)
        mbar_wait(&k_full[j & 1], (j >> 1) & 1, status, kSiteAttention, 200000000ull, false);
      for (int u = v_issued - 1; u >= 0 && u >= v_issued - VS; --u)
        mbar_wait(&v_full[u % VS], (u / VS) & 1, status, kSiteAttention, 200000000ull, false);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // -------------------------------------------------------- MMA issuer
      constexpr uint32_t kIdescQK = idesc_bf16_f32(128, kKeys, false, false);
      constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, false, true);
      const uint32_t qb = smem_u32(sQ);
      auto issue_s = [&](int j) -> bool {
        const int ks = j & 1;
        if (!mbar_wait(&k_full[ks], (j >> 1) & 1, status, kSiteAttention)) return false;
        // S still holds S_{j-1} until the softmax has it in registers.
        if (j > 0 && !mbar_wait(s_free, (j - 1) & 1, status, kSiteAttention)) return false;
        tc_fence_after();
        const uint32_t kbase = smem_u32(sK[ks]);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          // K-major: Q chunk of 128 rows, K chunk of 256 rows (1024 B per 8 rows)
          const uint32_t qoff = (kk >> 2) * 16384 + (kk & 3) * 32;
          const uint32_t koff = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
          umma_bf16(tS, smem_desc_sw128(qb + qoff, 16, 1024),
                    smem_desc_sw128(kbase + koff, 16, 1024), kIdescQK, kk > 0 ? 1u : 0u);
        }
        umma_commit(s_full);
        umma_commit(&k_empty[ks]);
        return true;
      };
      bool ok = mbar_wait(q_full, 0, status, kSiteAttention) && issue_s(0);
      if (ok && n_kb > 1) ok = issue_s(1);
      for (int j = 0; ok && j < n_kb; ++j) {
        if (!mbar_wait(p_full, j & 1, status, kSiteAttention)) break;
        bool vok = true;
        for (int h = 0; h < 2; ++h) {
          const int u = 2 * j + h, slot = u % VS;
          if (!mbar_wait(&v_full[slot], (u / VS) & 1, status, kSiteAttention)) {
            vok = false;
            break;
          }
          tc_fence_after();
          const uint32_t vb = smem_u32(sV0 + slot * C::kVHalf);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            // P: 16 keys = 8 packed columns; V (MN-major): 16 key rows of
            // 128 B, 64-wide d chunks 16 KB apart.
            umma_bf16_ts(tO, tP + (8 * h + kk) * 8, smem_desc_sw128(vb + kk * 2048, 16384, 1024),
                         kIdescPV, (j > 0 || h > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&v_empty[slot]);
        }
        if (!vok) break;
        umma_commit(pv_done);
        if (j == n_kb - 1) umma_commit(o_final);
        if (j + 2 < n_kb && !issue_s(j + 2)) break;
      }
      umma_commit(drain);
      mbar_wait(drain, 0, status, kSiteAttention, 200000000ull, false);
    }
  } else {
    // ---------------------------------------------------------- softmax
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    const int q = q0 + row;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float scale = rsqrtf(static_cast<float>(D)) * kLog2e;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    // Exchange with the other half of the row (bounded wait on the quarter's
    // barrier); slots alternate by phase so a fast peer never overwrites a
    // value the other has not read.
    int xphase = 0;
    auto exchange = [&](float v) -> float {
      float* slot = xch + (xphase & 1) * 256;
      slot[half * 128 + row] = v;
      mbar_arrive(&xbar[quarter]);
      if (!mbar_wait(&xbar[quarter], xphase & 1, status, kSiteAttention)) ok = false;
      const float peer = slot[(half ^ 1) * 128 + row];
      ++xphase;
      return peer;
    };
    for (int j = 0; ok && j < n_kb; ++j) {
      if (PART && (rect.mode & kCpAccMerge) && j == max(n_kb - 3, 0) && q < s)
        // the running O that this thread merges into at the end: into L2 now
        bulk_prefetch_l2(rects.out + (static_cast<int64_t>(bi) * s + q) * a + hh * D + half * (D / 2),
                         D * 2);
      if (!mbar_wait_warp(s_full, j & 1, status, kSiteAttention)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float x[128];
#pragma unroll
      for (int c = 0; c < 4; ++c)
        tmem_ld_32x32b_x32_nowait(tS + lane_off + half * 128 + 32 * c, x + 32 * c);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(s_free);
      const int key0 = k_lo + j * kKeys + half * 128;
      if (key0 + 127 > q0 || key0 + 128 > k_end) {  // diagonal, ragged or past the keys: mask
        const int lim = min(q + 1, k_end) - key0;   // keys [0, lim) of this half are visible
#pragma unroll
        for (int i = 0; i < 128; ++i) x[i] = i < lim ? x[i] : -INFINITY;
      }
      // Row maximum: four chains of three-input maxima, then a tree.
      float mc[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
      for (int p = 0; p < 62; ++p) mc[p & 3] = fmax3f(mc[p & 3], x[4 + 2 * p], x[5 + 2 * p]);
      float mx = fmaxf(fmax3f(mc[0], mc[1], mc[2]), mc[3]);
      mx = fmaxf(mx, exchange(mx));
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      mx *= scale;  // raw scores; scale > 0 commutes with max
      const float m_new = fmaxf(m, mx);
      const bool need = j > 0 && m_new > m + kRescaleThreshold;
      float alpha = 1.f;
      if (j == 0) m = m_new;  // key 0 is visible to every row: m is finite
      if (need) {
        alpha = fast_exp2(m - m_new);
        l *= alpha;
        m = m_new;
      }
      // exp2, row sum and the bf16 P in registers while PV_{j-1} may still
      // run; pairs of elements in packed f32x2 arithmetic.
      uint32_t pk[64];
      float2 sm2[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
      const float2 scale2 = make_float2(scale, scale), negm2 = make_float2(-m, -m);
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        const float2 y = __ffma2_rn(make_float2(x[2 * i], x[2 * i + 1]), scale2, negm2);
        const float2 pv = make_float2(fast_exp2(y.x), fast_exp2(y.y));
        sm2[i & 3] = __fadd2_rn(sm2[i & 3], pv);
        pk[i] = pack_bf16x2(pv.x, pv.y);
      }
      const float2 s01 = __fadd2_rn(__fadd2_rn(sm2[0], sm2[1]), __fadd2_rn(sm2[2], sm2[3]));
      l += s01.x + s01.y;
      // PV_{j-1} has to be complete before O is rescaled or P overwritten.
      if (j > 0 && !mbar_wait_warp(pv_done, (j - 1) & 1, status, kSiteAttention)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
        for (int c = half * (D / 32); c < (half + 1) * (D / 32); ++c) {
          float v[16];
          tmem_ld_32x32b_x16(tO + lane_off + c * 16, v);
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) w[i] = __float_as_uint(v[i] * alpha);
          tmem_st_32x32b_x16(tO + lane_off + c * 16, w);
        }
      }
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = pk[c * 32 + i];
        tmem_st_32x32b_x32(tP + lane_off + half * 64 + c * 32, w);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    if (__all_sync(0xffffffffu, ok) && mbar_wait_warp(o_final, 0, status, kSiteAttention)) {
      tc_fence_after();
      float run_l2 = 0.f;  // the rows' running log2-sum-exp
      const bool merge = PART && (rect.mode & kCpAccMerge);
      const int64_t lrow = (static_cast<int64_t>(bi) * H + hh) * s + q;
      // Both halves read it before either passes the exchange below, after
      // which half 0 may overwrite it.
      if (merge && q < s) run_l2 = rects.lse2[lrow];
      l += exchange(l);  // both halves' sums, taken against the same max
      const float inv = 1.f / l;
      if constexpr (PART) {
        // this rectangle's log2-sum-exp m + log2(l), merged with the running one
        float l2 = m + log2f(l), c_new = inv, c_old = 0.f;
        if (merge) {
          const float mx = fmaxf(run_l2, l2);
          l2 = mx + log2f(fast_exp2(run_l2 - mx) + fast_exp2(l2 - mx));
          c_old = fast_exp2(run_l2 - l2);
          c_new = fast_exp2(m - l2);  // = exp2(this rectangle's l2 - merged l2) / l
        }
        const bool final = rect.mode & kCpAccFinal;
        const int64_t row_off = (static_cast<int64_t>(bi) * s + q) * a + hh * D;
#pragma unroll 1
        for (int c = half * (D / 64); c < (half + 1) * (D / 64); ++c) {
          float v[32];
          tmem_ld_32x32b_x32(tO + lane_off + c * 32, v);
          if (q < s && MC_DCHECK(q - rect.base >= 0 && q - rect.base < rect.len &&
                                     hh * D + c * 32 + 32 <= a,
                                 status, kSiteAttention))
            accumulate_row32(v, c_new, c_old, rects.out + row_off + c * 32,
                             out + row_off + c * 32, merge, final);
        }
        if (q < s && half == 0) {
          if (final)
            lse[lrow] = l2 * kLn2;
          else
            rects.lse2[lrow] = l2;
        }
      } else {
        uint16_t* orow = out + (static_cast<int64_t>(bi) * s + q) * a + hh * D;
#pragma unroll 1
        for (int c = half * (D / 64); c < (half + 1) * (D / 64); ++c) {
          float v[32];
          tmem_ld_32x32b_x32(tO + lane_off + c * 32, v);
          if (q < s && MC_DCHECK(q >= 0 && hh * D + c * 32 + 32 <= a, status, kSiteAttention)) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint4 wv;
              wv.x = pack_bf16x2(v[8 * i + 0] * inv, v[8 * i + 1] * inv);
              wv.y = pack_bf16x2(v[8 * i + 2] * inv, v[8 * i + 3] * inv);
              wv.z = pack_bf16x2(v[8 * i + 4] * inv, v[8 * i + 5] * inv);
              wv.w = pack_bf16x2(v[8 * i + 6] * inv, v[8 * i + 7] * inv);
              dst[i] = wv;
            }
          }
        }
        if (q < s && half == 0) lse[(static_cast<int64_t>(bi) * H + hh) * s + q] = (m + log2f(l)) * kLn2;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, bool PART>
int launch_wide(const uint16_t* qkv, uint16_t* o, float* lse, int b, int s, int H, int* status,
                cudaStream_t st, const WideRects& rects) {
  using C = WideCfg<D>;
  const uint64_t a3 = 3ull * H * D;
  CUtensorMap tm;
  const uint64_t dims[3] = {a3, static_cast<uint64_t>(s), static_cast<uint64_t>(b)};
  const uint64_t strides[2] = {a3 * 2, a3 * 2 * static_cast<uint64_t>(s)};
  const uint32_t box[3] = {64, 128, 1};
  if (!make_tmap_bf16(&tm, qkv, 3, dims, strides, box)) return MC_ERR_CUDA;
  auto kern = attn_fwd_wide_kernel<D, PART>;
  static PerDeviceInit init;
  const cudaError_t attr = once_per_device(init, [&](long long*) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  });
  if (attr != cudaSuccess) return MC_ERR_CUDA;
  const dim3 grid = PART ? dim3(rects.cta_end[rects.n - 1], H, b)
                         : attention_grid(rects.head_major, (s + 127) / 128, H, b);
  launch_kernel(kern, grid, dim3(kWideThreads), C::kSmem, st, 1, tm, o, lse, s, H, status, rects);
  return cudaGetLastError() == cudaSuccess ? MC_OK : MC_ERR_CUDA;
}

}  // namespace

int launch_attention_forward_wide(const uint16_t* qkv, uint16_t* o, float* lse, int b, int s,
                                  int H, int d, int* status, cudaStream_t st) {
  WideRects whole = {};
  whole.n = 1;
  whole.cta_end[0] = (s + 127) / 128;
  whole.r[0] = {0, s, 0, INT_MAX, 0};
  whole.head_major = attention_head_major((s + 127) / 128, H, b) ? 1 : 0;
  return d == 64 ? launch_wide<64, false>(qkv, o, lse, b, s, H, status, st, whole)
                 : launch_wide<128, false>(qkv, o, lse, b, s, H, status, st, whole);
}

int launch_attention_forward_parts(const uint16_t* qkv, uint16_t* o, float* lse, int b, int s,
                                   int H, int d, const CpRect* rects, int n, float* acc_o,
                                   float* acc_lse2, int* status, cudaStream_t st) {
  if (check_cp_rects(rects, n, s) != MC_OK) return MC_ERR_ARGUMENT;
  // Rectangles off the diagonal (every tile the same length) first, then the
  // diagonal ones, whose tiles the kernel takes heaviest first.
  WideRects w = {};
  w.out = acc_o;
  w.lse2 = acc_lse2;
  for (int pass = 0; pass < 2; ++pass)
    for (int i = 0; i < n; ++i) {
      const CpRect& r = rects[i];
      if ((r.q_base == r.k_base) != (pass == 1)) continue;
      w.r[w.n] = {r.q_base, r.q_len, r.k_base, r.k_base + r.k_len, r.mode_q};
      w.cta_end[w.n] = (w.n > 0 ? w.cta_end[w.n - 1] : 0) + r.q_len / 128;
      ++w.n;
    }
  return d == 64 ? launch_wide<64, true>(qkv, o, lse, b, s, H, status, st, w)
                 : launch_wide<128, true>(qkv, o, lse, b, s, H, status, st, w);
}

}  // namespace mc
