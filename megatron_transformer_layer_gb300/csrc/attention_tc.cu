// Causal flash attention backward on the sm_103a tensor cores (tcgen05):
// the dK/dV and dQ kernels, over the whole score matrix or over the
// rectangles that the context-parallel path combines.  The forward (whole
// matrix and rectangles) is attention_fwd_wide.cu; the delta pre-pass and
// the argument checks are attention.cu.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "mc_layer_internal.h"
#include "ptx.cuh"

namespace mc {
namespace {

constexpr int kBwdThreads = 320;  // producer, MMA, 8 compute warps
constexpr float kLog2e = 1.4426950408889634f;
constexpr int64_t kDsTileBytes = 128 * 128 * 2;  // one bf16 dS^T tile (128 keys x 128 queries)

// A rectangle of the causal score matrix, for the context-parallel path:
// dK/dV take key rows [base, base + len) against query blocks
// [blk_lo, blk_hi).  Results are added to running fp32 sums dK | dV
// [b, s, 2a] indexed by the absolute row.  Without kCpAccMerge in `mode`
// there is no earlier sum to add; with kCpAccFinal the sum goes to dqkv as
// bf16 instead.  The rectangle's dS^T tiles start at tile `tile0` of the
// workspace.  The fused kernel uses the whole matrix (base 0, blocks
// [0, INT_MAX)) and no sums.
struct AttnPart {
  int base, len;
  int blk_lo, blk_hi;
  int mode;
  int64_t tile0;
};

// The rectangles of one launch (disjoint key rows): CTAs
// [cta_end[i - 1], cta_end[i]) take the 128-key blocks of rectangle i.
struct AttnParts {
  int n;
  int cta_end[kCpMaxRects];
  AttnPart r[kCpMaxRects];
  float* acc;
  int head_major;  // the whole matrix: the grid order (attention_cta)
};

// ---------------------------------------------------------------- backward
// Two kernels after the delta pre-pass:
//   dkdv: rows = keys (K, V resident; Q_i, dO_i streamed), accumulates dV,
//         dK and, given a dS workspace, writes each block pair's dS^T tile.
//   dq:   rows = queries.  With the tiles, dQ = dS K streams them and K_j
//         (attn_bwd_dq_gemm_kernel; also the context-parallel rectangles);
//         without, Q and dO stay resident, K_j and V_j stream in, and S and
//         dP are formed again (attn_bwd_dq_tc_kernel).
template <int D>
struct BwdCfg {
  static constexpr int kChunks = D / 64;
  static constexpr int kTile = 128 * D * 2;
  // K, V, two (Q_i, dO_i) stages, the dS^T tile staged for its bulk store,
  // lse/delta staging [2][2][128], barriers.  The dynamic shared memory
  // starts 1024-byte aligned (checked at run time): no slack is reserved.
  static constexpr int kUsed = 6 * kTile + static_cast<int>(kDsTileBytes) + 4 * 128 * 4 + 24 * 8;
  static constexpr int kSmem = kUsed > 116 * 1024 ? kUsed : 116 * 1024;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kUsed <= 227 * 1024, "dkdv kernel shared memory");
};

// dK, dV for one 128-key block.  TMEM: S^T [0, 128), dP^T [128, 256),
// dV [256, 256 + D), dK [384, 384 + D).  Per query block i:
//   MMA      S^T_i = K Q_i^T (as soon as the compute warps hold S^T_{i-1} in
//            registers), then dV += P^T_{i-1} dO_{i-1}, dK += dS^T_{i-1} Q_{i-1},
//            then (those done) dP^T_i = V dO_i^T.
//   compute  load S^T_i, release it; P^T = exp2(S^T c - lse2) while the MMAs
//            above run; then load dP^T_i and form dS^T = P^T (dP^T - delta);
//            with a dS workspace, also into the shared-memory tile image
//            that one thread then sends out with a bulk store.
// Each compute thread owns one key row and 64 query columns of dP^T, and
// writes its P^T and dS^T (bf16 pairs) back over exactly those columns: the
// 16 queries of group g (dP^T columns [16g, 16g + 16)) leave P at columns
// [16g, 16g + 8) and dS at [16g + 8, 16g + 16).  No thread overwrites
// columns another thread still has to read.
template <int D, bool PART>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv,
                            const __grid_constant__ CUtensorMap tm_do, const float* __restrict__ lse,
                            const float* __restrict__ delta, uint16_t* __restrict__ dqkv, int s,
                            int H, int* status, const __grid_constant__ AttnParts parts,
                            uint8_t* __restrict__ ds_tiles) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {  // the 128-byte swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) record_error(status, MC_ERR_DEVICE_BOUNDS, kSiteAttention);
    return;
  }
  uint8_t* sK = smem;
  uint8_t* sV = smem + C::kTile;
  uint8_t* sQ[2] = {smem + 2 * C::kTile, smem + 3 * C::kTile};
  uint8_t* sdO[2] = {smem + 4 * C::kTile, smem + 5 * C::kTile};
  uint8_t* sDs = smem + 6 * C::kTile;  // dS^T tile image (swizzled), 32 KB
  float* sL = reinterpret_cast<float*>(sDs + kDsTileBytes);  // [2][128] lse * log2(e)
  float* sD = sL + 256;                                       // [2][128] delta
  uint64_t* bars = reinterpret_cast<uint64_t*>(sD + 256);
  uint64_t* r_full = bars + 0;
  uint64_t* st_full = bars + 1;    // [2]
  uint64_t* st_empty = bars + 3;   // [2]
  uint64_t* s_full = bars + 5;     // S^T_i in TMEM
  uint64_t* s_free = bars + 6;     // compute warps hold S^T_i in registers
  uint64_t* dp_full = bars + 7;    // dP^T_i in TMEM
  uint64_t* p_full = bars + 8;     // P^T_i, dS^T_i in TMEM
  uint64_t* acc_done = bars + 9;   // dV, dK products of block i complete
  uint64_t* drain = bars + 10;
  uint64_t* lse_ready = bars + 11;  // [2]
  uint64_t* ds_full = bars + 13;    // the dS^T tile of block i is in sDs (256 threads)
  uint64_t* ds_free = bars + 14;    // its bulk store has read sDs
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 15);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int a = H * D;
  const int nblk = (s + 127) / 128;
  // this CTA's rectangle (the whole matrix: one) and key block (heaviest:
  // the first of a head's)
  int t_heavy, hh, bi;
  attention_cta(!PART && parts.head_major, H, t_heavy, hh, bi);
  int ri = 0;
  if constexpr (PART)
    while (ri + 1 < parts.n && static_cast<int>(blockIdx.x) >= parts.cta_end[ri]) ++ri;
  const AttnPart part = parts.r[ri];
  const int cta0 = ri > 0 ? parts.cta_end[ri - 1] : 0;
  const int kb = PART ? part.base / 128 + static_cast<int>(blockIdx.x) - cta0 : t_heavy;
  const int r0 = kb * 128;
  // query blocks qb0 .. qb0 + count - 1 (fused: kb .. nblk - 1)
  const int qb0 = max(kb, part.blk_lo);
  const int count = min(nblk, part.blk_hi) - qb0;

  if (threadIdx.x == 0) {
    mbar_init(r_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&st_full[i], 1);
      mbar_init(&st_empty[i], 1);
      mbar_init(&lse_ready[i], 256);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, 256);
    mbar_init(dp_full, 1);
    mbar_init(p_full, 256);
    mbar_init(acc_done, 1);
    mbar_init(drain, 1);
    mbar_init(ds_full, 256);
    mbar_init(ds_free, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tm_qkv);
    tma_prefetch_desc(&tm_do);
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
  const uint32_t tS = tmem, tdP = tmem + 128, tdV = tmem + 256, tdK = tmem + 384;

  if (warp == 0) {
    if (lane == 0) {
      // -------------------------------------------------------- producer
      const int cq = hh * D, ck = a + hh * D, cv = 2 * a + hh * D;
      mbar_arrive_expect_tx(r_full, 2 * C::kTile);
      for (int c = 0; c < C::kChunks; ++c) {
        tma_load_3d(sK + c * 16384, &tm_qkv, r_full, ck + c * 64, r0, bi);
        tma_load_3d(sV + c * 16384, &tm_qkv, r_full, cv + c * 64, r0, bi);
      }
      int issued = 0;
      for (int i = 0; i < count; ++i) {
        const int st = i & 1;
        const int row = (qb0 + i) * 128;
        if (!mbar_wait(&st_empty[st], ((i >> 1) & 1) ^ 1u, status, kSiteAttention)) break;
        mbar_arrive_expect_tx(&st_full[st], 2 * C::kTile);
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_3d(sQ[st] + c * 16384, &tm_qkv, &st_full[st], cq + c * 64, row, bi);
          tma_load_3d(sdO[st] + c * 16384, &tm_do, &st_full[st], hh * D + c * 64, row, bi);
        }
        ++issued;
      }
      pdl_launch();  // every load of this CTA is issued
      mbar_wait(r_full, 0, status, kSiteAttention, 200000000ull, false);
      for (int i = issued - 1; i >= 0 && i >= issued - 2; --i)
        mbar_wait(&st_full[i & 1], (i >> 1) & 1, status, kSiteAttention, 200000000ull, false);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // -------------------------------------------------------- MMA issuer
      constexpr uint32_t kIdescSq = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t kIdescAcc = idesc_bf16_f32(128, D, false, true);
      bool ok = mbar_wait(r_full, 0, status, kSiteAttention);
      const uint32_t kbase = smem_u32(sK), vbase = smem_u32(sV);
      for (int i = 0; ok && i <= count; ++i) {
        const int st = i & 1;
        if (i < count) {
          if (!mbar_wait(&st_full[st], (i >> 1) & 1, status, kSiteAttention)) break;
          // tS was read into registers for block i - 1.
          if (i > 0 && !mbar_wait(s_free, (i - 1) & 1, status, kSiteAttention)) break;
          tc_fence_after();
          const uint32_t qb = smem_u32(sQ[st]);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            umma_bf16(tS, smem_desc_sw128(kbase + off, 16, 1024), smem_desc_sw128(qb + off, 16, 1024),
                      kIdescSq, kk > 0 ? 1u : 0u);
          }
          umma_commit(s_full);
        }
        if (i > 0) {
          const int pi = i - 1, pst = pi & 1;
          if (!mbar_wait(p_full, pi & 1, status, kSiteAttention)) break;
          tc_fence_after();
          const uint32_t qb = smem_u32(sQ[pst]), dob = smem_u32(sdO[pst]);
#pragma unroll
          for (int kk = 0; kk < 128 / 16; ++kk) {
            // 16 queries = group kk: P at 16 kk, dS at 16 kk + 8; B tiles viewed MN-major
            const uint32_t pcol = static_cast<uint32_t>(kk * 16);
            const uint32_t acc = (pi > 0 || kk > 0) ? 1u : 0u;
            umma_bf16_ts(tdV, tdP + pcol, smem_desc_sw128(dob + kk * 2048, 16384, 1024), kIdescAcc,
                         acc);
            umma_bf16_ts(tdK, tdP + pcol + 8, smem_desc_sw128(qb + kk * 2048, 16384, 1024),
                         kIdescAcc, acc);
          }
          umma_commit(&st_empty[pst]);
          umma_commit(acc_done);
        }
        if (i < count) {
          // dP^T_i overwrites the P^T / dS^T that the products above read.
          if (i > 0 && !mbar_wait(acc_done, (i - 1) & 1, status, kSiteAttention)) break;
          tc_fence_after();
          const uint32_t dob = smem_u32(sdO[st]);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            umma_bf16(tdP, smem_desc_sw128(vbase + off, 16, 1024),
                      smem_desc_sw128(dob + off, 16, 1024), kIdescSq, kk > 0 ? 1u : 0u);
          }
          umma_commit(dp_full);
        }
      }
      umma_commit(drain);
      mbar_wait(drain, 0, status, kSiteAttention, 200000000ull, false);
    }
  } else {
    // ---------------------------------------------------------- compute
    // Two warps per TMEM lane quarter; `half` picks 64 of the 128 query
    // columns (the per-element work needs no reduction along the row).
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int t = quarter * 32 + lane;  // key row within the block
    const int r = r0 + t;               // this thread's key
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t my_cols = lane_off + static_cast<uint32_t>(half * 64);
    const float scale2 = rsqrtf(static_cast<float>(D)) * kLog2e;
    const float* L = lse + (static_cast<int64_t>(bi) * H + hh) * s;
    const float* Dl = delta + (static_cast<int64_t>(bi) * H + hh) * s;
    // lse / delta of query t of the next block, loaded one block ahead (half 0)
    float nl2 = 0.f, nd = 0.f;
    if (half == 0 && qb0 * 128 + t < s) {
      nl2 = L[qb0 * 128 + t] * kLog2e;
      nd = Dl[qb0 * 128 + t];
    }
    bool ok = true;
    for (int i = 0; i < count; ++i) {
      const int c0 = (qb0 + i) * 128;  // first query of this block
      const float* l2 = sL + (i & 1) * 128 + half * 64;
      const float* dl = sD + (i & 1) * 128 + half * 64;
      if (half == 0) {
        sL[(i & 1) * 128 + t] = nl2;
        sD[(i & 1) * 128 + t] = nd;
        const int qn = c0 + 128 + t;
        nl2 = qn < s ? L[qn] * kLog2e : 0.f;
        nd = qn < s ? Dl[qn] : 0.f;
      }
      mbar_arrive(&lse_ready[i & 1]);
      if (!mbar_wait_warp(&lse_ready[i & 1], (i >> 1) & 1, status, kSiteAttention) ||
          !mbar_wait_warp(s_full, i & 1, status, kSiteAttention)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float p[64];
      tmem_ld_32x32b_x32_nowait(tS + my_cols, p);
      tmem_ld_32x32b_x32_nowait(tS + my_cols + 32, p + 32);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(s_free);
      // Visible: query >= key, both within the sequence.
      const int q0 = c0 + half * 64;
      const bool edge = q0 < r0 + 127 || q0 + 64 > s;
      const float2 sc2 = make_float2(scale2, scale2);
#pragma unroll
      for (int e = 0; e < 64; e += 4) {
        const float4 lv = *reinterpret_cast<const float4*>(l2 + e);
        const float2 y0 = __ffma2_rn(make_float2(p[e], p[e + 1]), sc2, make_float2(-lv.x, -lv.y));
        const float2 y1 =
            __ffma2_rn(make_float2(p[e + 2], p[e + 3]), sc2, make_float2(-lv.z, -lv.w));
        p[e] = fast_exp2(y0.x);
        p[e + 1] = fast_exp2(y0.y);
        p[e + 2] = fast_exp2(y1.x);
        p[e + 3] = fast_exp2(y1.y);
      }
      if (edge) {
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          const int q = q0 + e;
          p[e] = (q >= r && q < s) ? p[e] : 0.f;
        }
      }
      if (!mbar_wait_warp(dp_full, i & 1, status, kSiteAttention)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // dS^T of this (query block, key block) pair also goes to `ds_tiles`
      // for the dQ product, as the 128-byte-swizzled shared-memory image of
      // an MN-major A operand: query chunk `half` at 16 KB, key row t at
      // 128 B, the 16-byte unit of queries [8u, 8u + 8) at unit u ^ (t & 7).
      // It is assembled in sDs (conflict-free 16-byte writes) and leaves as
      // one bulk store; the previous block's store must have read sDs first.
      const bool store_ds = ds_tiles != nullptr;
      uint8_t* ds_row = sDs + half * 16384 + t * 128;
      if (store_ds && i > 0) {
        if (threadIdx.x == 64) {
          bulk_wait_read();
          mbar_arrive(ds_free);
        }
        if (!mbar_wait_warp(ds_free, (i - 1) & 1, status, kSiteAttention)) {
          ok = false;
          break;
        }
      }
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        float dv[16];
        tmem_ld_32x32b_x16(tdP + my_cols + g * 16, dv);
        uint32_t w[16];  // [P of the 16 queries | dS of the 16 queries]
#pragma unroll
        for (int e = 0; e < 16; e += 4) {
          const float4 dlv = *reinterpret_cast<const float4*>(dl + g * 16 + e);
          const float* pp = p + g * 16 + e;
          const float2 d0 = __fmul2_rn(make_float2(pp[0], pp[1]),
                                       __fadd2_rn(make_float2(dv[e], dv[e + 1]),
                                                  make_float2(-dlv.x, -dlv.y)));
          const float2 d1 = __fmul2_rn(make_float2(pp[2], pp[3]),
                                       __fadd2_rn(make_float2(dv[e + 2], dv[e + 3]),
                                                  make_float2(-dlv.z, -dlv.w)));
          w[e / 2] = pack_bf16x2(pp[0], pp[1]);
          w[e / 2 + 1] = pack_bf16x2(pp[2], pp[3]);
          w[8 + e / 2] = pack_bf16x2(d0.x, d0.y);
          w[8 + e / 2 + 1] = pack_bf16x2(d1.x, d1.y);
        }
        if (store_ds) {
          *reinterpret_cast<uint4*>(ds_row + (((2 * g) ^ (t & 7)) << 4)) =
              make_uint4(w[8], w[9], w[10], w[11]);
          *reinterpret_cast<uint4*>(ds_row + (((2 * g + 1) ^ (t & 7)) << 4)) =
              make_uint4(w[12], w[13], w[14], w[15]);
        }
        // over this thread's own dP^T columns, already in registers
        tmem_st_32x32b_x16(tdP + my_cols + g * 16, w);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(p_full);
      if (store_ds) {
        fence_proxy_async_smem();  // sDs writes visible to the bulk copy
        mbar_arrive(ds_full);
        if (warp == 2) {
          // one thread stores the assembled tile
          if (!mbar_wait_warp(ds_full, i & 1, status, kSiteAttention)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            // the whole matrix: the lower triangle of (query block, key block)
            // pairs per head; a rectangle: its nq x nk pairs per head
            const int qb = qb0 + i;
            const int nq = part.blk_hi - part.blk_lo, nk = part.len / 128;
            const int kr = kb - part.base / 128;
            const int64_t tile =
                PART ? part.tile0 + ((static_cast<int64_t>(bi) * H + hh) * nq + (qb - part.blk_lo)) * nk + kr
                     : (static_cast<int64_t>(bi) * H + hh) *
                               (static_cast<int64_t>(nblk) * (nblk + 1) / 2) +
                           static_cast<int64_t>(qb) * (qb + 1) / 2 + kb;
            const bool in_rect =
                PART ? qb >= part.blk_lo && qb < part.blk_hi && kr >= 0 && kr < nk : true;
            if (MC_DCHECK(kb <= qb && qb < nblk && in_rect, status, kSiteAttention)) {
              bulk_store(ds_tiles + tile * kDsTileBytes, sDs, static_cast<uint32_t>(kDsTileBytes));
              bulk_commit();
            }
          }
        }
      }
    }
    // the tile stores must be complete (and done with sDs) before exit
    if (ds_tiles && threadIdx.x == 64) bulk_wait_all();
    if (ok && mbar_wait_warp(acc_done, (count - 1) & 1, status, kSiteAttention)) {
      tc_fence_after();
      const float scale = rsqrtf(static_cast<float>(D));
      const int64_t base = (static_cast<int64_t>(bi) * s + r) * 3 * static_cast<int64_t>(a);
#pragma unroll 1
      for (int w = 0; w < 2; ++w) {
        // w = 0: dV (V's columns of dqkv), w = 1: dK scaled by 1/sqrt(d)
        const uint32_t tacc = w == 0 ? tdV : tdK;
        const float mul = w == 0 ? 1.f : scale;
        const int col = (w == 0 ? 2 * a : a) + hh * D;
#pragma unroll 1
        for (int c = half * (D / 64); c < (half + 1) * (D / 64); ++c) {
          float v[32];
          tmem_ld_32x32b_x32(tacc + lane_off + c * 32, v);
          const bool in_range = MC_DCHECK(
              r >= 0 && col + c * 32 + 32 <= 3 * a && (!PART || r - part.base < part.len), status,
              kSiteAttention);
          if (PART && r < s && in_range) {
            // the running sums: dK at [0, a), dV at [a, 2a) of the key's row
            float* run = parts.acc + (static_cast<int64_t>(bi) * s + r) * 2 * a +
                         (w == 0 ? a : 0) + hh * D + c * 32;
            accumulate_row32(v, mul, 1.f, run, dqkv + base + col + c * 32,
                             part.mode & kCpAccMerge, part.mode & kCpAccFinal);
          } else if (!PART && r < s && in_range) {
            uint4* dst = reinterpret_cast<uint4*>(dqkv + base + col + c * 32);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              uint4 wv;
              wv.x = pack_bf16x2(v[8 * k + 0] * mul, v[8 * k + 1] * mul);
              wv.y = pack_bf16x2(v[8 * k + 2] * mul, v[8 * k + 3] * mul);
              wv.z = pack_bf16x2(v[8 * k + 4] * mul, v[8 * k + 5] * mul);
              wv.w = pack_bf16x2(v[8 * k + 6] * mul, v[8 * k + 7] * mul);
              dst[k] = wv;
            }
          }
        }
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

template <int D>
struct DqCfg {
  static constexpr int kChunks = D / 64;
  static constexpr int kTile = 128 * D * 2;
  // Q, dO, three K stages, two V stages, barriers, alignment slack
  static constexpr int kUsed = 7 * kTile + 24 * 8 + 1024;
  static constexpr int kSmem = kUsed > 116 * 1024 ? kUsed : 116 * 1024;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kUsed <= 227 * 1024, "dq kernel shared memory");
};

// dQ, with the next block's products overlapping this block's dS.
//   TMEM: S [0, 128), dP [128, 256), dQ [256, 256 + D), dS (bf16) [384, 448).
// The compute warps read S_j and dP_j into registers and release them at once
// (s_free), so S_{j+1} = Q K_{j+1}^T and dP_{j+1} = dO V_{j+1}^T run while
// dS_j is formed; dQ += dS_j K_j follows when dS_j is in TMEM (ds_full), and
// its completion (ds_free) lets dS_{j+1} be written.
template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv,
                          const __grid_constant__ CUtensorMap tm_do, const float* __restrict__ lse,
                          const float* __restrict__ delta, uint16_t* __restrict__ dqkv, int s,
                          int H, int* status, int head_major) {
  using C = DqCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  // K_j is needed until dQ_j, V_j only until dP_j: separate rings (K 3 deep,
  // V 2 deep) keep the next blocks' loads ahead of the overlapped products.
  uint8_t* sQ = smem;
  uint8_t* sdO = smem + C::kTile;
  uint8_t* sK[3] = {smem + 2 * C::kTile, smem + 3 * C::kTile, smem + 4 * C::kTile};
  uint8_t* sV[2] = {smem + 5 * C::kTile, smem + 6 * C::kTile};
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 7 * C::kTile);
  uint64_t* r_full = bars + 0;
  uint64_t* k_full = bars + 1;    // [3]
  uint64_t* k_empty = bars + 4;   // [3]
  uint64_t* v_full = bars + 7;    // [2]
  uint64_t* v_empty = bars + 9;   // [2]
  uint64_t* s_full = bars + 11;
  uint64_t* s_free = bars + 12;
  uint64_t* ds_full = bars + 13;
  uint64_t* ds_free = bars + 14;
  uint64_t* drain = bars + 15;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int a = H * D;
  // heaviest first: query blocks 0 .. nblk - 1 against key blocks 0 .. qb
  int t_heavy, hh, bi;
  attention_cta(head_major != 0, H, t_heavy, hh, bi);
  const int qb = (s + 127) / 128 - 1 - t_heavy;
  const int q0 = qb * 128;
  const int count = qb + 1;  // key blocks 0 .. qb

  if (threadIdx.x == 0) {
    mbar_init(r_full, 1);
    for (int i = 0; i < 3; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, 256);
    mbar_init(ds_full, 256);
    mbar_init(ds_free, 1);
    mbar_init(drain, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tm_qkv);
    tma_prefetch_desc(&tm_do);
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
  const uint32_t tS = tmem, tdP = tmem + 128, tdQ = tmem + 256, tdS = tmem + 384;

  if (warp == 0) {
    if (lane == 0) {
      // -------------------------------------------------------- producer
      mbar_arrive_expect_tx(r_full, 2 * C::kTile);
      for (int c = 0; c < C::kChunks; ++c) {
        tma_load_3d(sQ + c * 16384, &tm_qkv, r_full, hh * D + c * 64, q0, bi);
        tma_load_3d(sdO + c * 16384, &tm_do, r_full, hh * D + c * 64, q0, bi);
      }
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < count; ++j) {
        const int ks = j % 3, kph = (j / 3) & 1, vs = j & 1, vph = (j >> 1) & 1;
        if (!mbar_wait(&k_empty[ks], kph ^ 1u, status, kSiteAttention)) break;
        mbar_arrive_expect_tx(&k_full[ks], C::kTile);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(sK[ks] + c * 16384, &tm_qkv, &k_full[ks], a + hh * D + c * 64,
                      j * 128, bi);
        ++k_issued;
        if (!mbar_wait(&v_empty[vs], vph ^ 1u, status, kSiteAttention)) break;
        mbar_arrive_expect_tx(&v_full[vs], C::kTile);
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(sV[vs] + c * 16384, &tm_qkv, &v_full[vs], 2 * a + hh * D + c * 64,
                      j * 128,
                      bi);
        ++v_issued;
      }
      pdl_launch();  // every load of this CTA is issued
      // Copies still in flight must land before the CTA exits: the last
      // K loads (up to 3) and V loads (up to 2).
      mbar_wait(r_full, 0, status, kSiteAttention, 200000000ull, false);
      for (int j = k_issued - 1; j >= 0 && j >= k_issued - 3; --j)
        mbar_wait(&k_full[j % 3], (j / 3) & 1, status, kSiteAttention, 200000000ull, false);
      for (int j = v_issued - 1; j >= 0 && j >= v_issued - 2; --j)
        mbar_wait(&v_full[j & 1], (j >> 1) & 1, status, kSiteAttention, 200000000ull, false);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // -------------------------------------------------------- MMA issuer
      constexpr uint32_t kIdescSq = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t kIdescAcc = idesc_bf16_f32(128, D, false, true);
      bool ok = mbar_wait(r_full, 0, status, kSiteAttention);
      const uint32_t qb0 = smem_u32(sQ), dob = smem_u32(sdO);
      for (int j = 0; ok && j <= count; ++j) {
        if (j < count) {
          const int ks = j % 3, vs = j & 1;
          if (!mbar_wait(&k_full[ks], (j / 3) & 1, status, kSiteAttention)) break;
          if (!mbar_wait(&v_full[vs], (j >> 1) & 1, status, kSiteAttention)) break;
          // S / dP of block j - 1 are in the compute warps' registers.
          if (j > 0 && !mbar_wait(s_free, (j - 1) & 1, status, kSiteAttention)) break;
          tc_fence_after();
          const uint32_t kb = smem_u32(sK[ks]), vb = smem_u32(sV[vs]);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            umma_bf16(tS, smem_desc_sw128(qb0 + off, 16, 1024), smem_desc_sw128(kb + off, 16, 1024),
                      kIdescSq, kk > 0 ? 1u : 0u);
            umma_bf16(tdP, smem_desc_sw128(dob + off, 16, 1024),
                      smem_desc_sw128(vb + off, 16, 1024), kIdescSq, kk > 0 ? 1u : 0u);
          }
          umma_commit(s_full);
          umma_commit(&v_empty[vs]);  // V_j is done once dP_j is
        }
        if (j > 0) {
          const int pj = j - 1, pks = pj % 3;
          if (!mbar_wait(ds_full, pj & 1, status, kSiteAttention)) break;
          tc_fence_after();
          const uint32_t kb = smem_u32(sK[pks]);
#pragma unroll
          for (int kk = 0; kk < 128 / 16; ++kk)
            umma_bf16_ts(tdQ, tdS + kk * 8, smem_desc_sw128(kb + kk * 2048, 16384, 1024), kIdescAcc,
                         (pj > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&k_empty[pks]);
          umma_commit(ds_free);
        }
      }
      umma_commit(drain);
      mbar_wait(drain, 0, status, kSiteAttention, 200000000ull, false);
    }
  } else {
    // ---------------------------------------------------------- compute
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;   // 64 of the block's 128 key columns
    const int r = q0 + quarter * 32 + lane;  // this thread's query row
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float scale2 = rsqrtf(static_cast<float>(D)) * kLog2e;
    const float* L = lse + (static_cast<int64_t>(bi) * H + hh) * s;
    const float* Dl = delta + (static_cast<int64_t>(bi) * H + hh) * s;
    const float my_l2 = r < s ? L[r] * kLog2e : 0.f;
    const float my_d = r < s ? Dl[r] : 0.f;
    bool ok = true;
    for (int j = 0; j < count; ++j) {
      if (!mbar_wait_warp(s_full, j & 1, status, kSiteAttention)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sv[64], dv[64];
      tmem_ld_32x32b_x32_nowait(tS + lane_off + half * 64, sv);
      tmem_ld_32x32b_x32_nowait(tS + lane_off + half * 64 + 32, sv + 32);
      tmem_ld_32x32b_x32_nowait(tdP + lane_off + half * 64, dv);
      tmem_ld_32x32b_x32_nowait(tdP + lane_off + half * 64 + 32, dv + 32);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(s_free);
      const int c0 = j * 128 + half * 64;
      const bool edge = c0 + 63 > q0 || c0 + 64 > s;
      uint32_t dw[32];
      const float2 sc2 = make_float2(scale2, scale2), nl2 = make_float2(-my_l2, -my_l2);
      const float2 nd2 = make_float2(-my_d, -my_d);
#pragma unroll
      for (int e = 0; e < 64; e += 2) {
        const float2 y = __ffma2_rn(make_float2(sv[e], sv[e + 1]), sc2, nl2);
        float2 pv = make_float2(fast_exp2(y.x), fast_exp2(y.y));
        if (edge) {
          const int col = c0 + e;
          pv.x = (col <= r && col < s) ? pv.x : 0.f;
          pv.y = (col + 1 <= r && col + 1 < s) ? pv.y : 0.f;
        }
        const float2 ds = __fmul2_rn(pv, __fadd2_rn(make_float2(dv[e], dv[e + 1]), nd2));
        dw[e / 2] = pack_bf16x2(ds.x, ds.y);
      }
      // dS_{j-1} must have been consumed by its dQ product.
      if (j > 0 && !mbar_wait_warp(ds_free, (j - 1) & 1, status, kSiteAttention)) {
        ok = false;
        break;
      }
      tc_fence_after();
      tmem_st_32x32b_x32(tdS + lane_off + half * 32, dw);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(ds_full);
    }
    if (ok && mbar_wait_warp(ds_free, (count - 1) & 1, status, kSiteAttention)) {
      tc_fence_after();
      const float scale = rsqrtf(static_cast<float>(D));
      const int64_t base = (static_cast<int64_t>(bi) * s + r) * 3 * static_cast<int64_t>(a);
#pragma unroll 1
      for (int c = half * (D / 64); c < (half + 1) * (D / 64); ++c) {
        float v[32];
        tmem_ld_32x32b_x32(tdQ + lane_off + c * 32, v);
        const bool in_range =
            MC_DCHECK(r >= 0 && hh * D + c * 32 + 32 <= a, status, kSiteAttention);
        if (r < s && in_range) {
          uint4* dst = reinterpret_cast<uint4*>(dqkv + base + hh * D + c * 32);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 wv;
            wv.x = pack_bf16x2(v[8 * k + 0] * scale, v[8 * k + 1] * scale);
            wv.y = pack_bf16x2(v[8 * k + 2] * scale, v[8 * k + 3] * scale);
            wv.z = pack_bf16x2(v[8 * k + 4] * scale, v[8 * k + 5] * scale);
            wv.w = pack_bf16x2(v[8 * k + 6] * scale, v[8 * k + 7] * scale);
            dst[k] = wv;
          }
        }
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

template <int D>
int launch_bwd_dq_tc(const CUtensorMap& tq, const CUtensorMap& td, const float* lse,
                     const float* delta, uint16_t* dqkv, int b, int s, int H, int* status,
                     cudaStream_t st) {
  using C = DqCfg<D>;
  auto kern = attn_bwd_dq_tc_kernel<D>;
  static PerDeviceInit init;
  const cudaError_t attr = once_per_device(init, [&](long long*) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  });
  if (attr != cudaSuccess) return MC_ERR_CUDA;
  const int nb = (s + 127) / 128;
  const bool hm = attention_head_major(nb, H, b);
  launch_kernel(kern, attention_grid(hm, nb, H, b), dim3(kBwdThreads), C::kSmem, st, 1, tq, td, lse,
                delta, dqkv, s, H, status, hm ? 1 : 0);
  return cudaGetLastError() == cudaSuccess ? MC_OK : MC_ERR_CUDA;
}

template <int D, bool PART>
int launch_bwd_dkdv_tc(const CUtensorMap& tq, const CUtensorMap& td, const float* lse,
                       const float* delta, uint16_t* dqkv, int b, int s, int H, int* status,
                       cudaStream_t st, const AttnParts& parts, uint8_t* ds_tiles = nullptr) {
  using C = BwdCfg<D>;
  auto kern = attn_bwd_dkdv_tc_kernel<D, PART>;
  static PerDeviceInit init;
  const cudaError_t attr = once_per_device(init, [&](long long*) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  });
  if (attr != cudaSuccess) return MC_ERR_CUDA;
  const dim3 grid = PART ? dim3(parts.cta_end[parts.n - 1], H, b)
                         : attention_grid(parts.head_major, (s + 127) / 128, H, b);
  launch_kernel(kern, grid, dim3(kBwdThreads), C::kSmem, st, 1, tq, td, lse, delta, dqkv, s, H,
                status, parts, ds_tiles);
  return cudaGetLastError() == cudaSuccess ? MC_OK : MC_ERR_CUDA;
}

// dQ from the dS^T tiles that the dK/dV kernel wrote: dQ_i = sum_{j <= i}
// dS_ij K_j, without forming S and dP again.  Persistent: one CTA per SM
// walks a share of the (128-query block, head, batch) items -- each head's
// blocks heaviest first, handed out in a snake over the CTAs -- with its
// ring and accumulators carried across items.  192 threads:
//   warp 0      producer: per key block j the 32 KB dS^T tile (one bulk copy
//               of its swizzled image) and K_j (TMA) into a 3-deep ring,
//               running on into the next item's tiles without a gap
//   warp 1      TMEM (two accumulators of 128 columns) and the MMA thread:
//               dQ += dS_ij K_j with A = dS (queries contiguous: MN-major)
//               and B = K_j (MN-major), the items alternating accumulators
//   warps 2..5  epilogue: dQ / sqrt(d) as bf16 into the dQ columns of dqkv,
//               while the next item accumulates into the other accumulator
// The tiles are read once from HBM; the kernel is bound by that stream, not
// by the 128 x 128 products.  The whole matrix reads each head's lower
// triangle of tiles; a context-parallel rectangle (PART) the nq x nk tiles
// that the dK/dV kernel wrote for it, adding dQ to the running fp32 sums.
template <int D>
struct DqGemmCfg {
  static constexpr int kChunks = D / 64;
  static constexpr int kKTile = 128 * D * 2;
  static constexpr int kStage = static_cast<int>(kDsTileBytes) + kKTile;
  static constexpr int kStages = 3;
  static constexpr int kUsed = kStages * kStage + 16 * 8;
  static constexpr int kSmem = kUsed + 1024;  // + alignment slack
  static_assert(kSmem <= 227 * 1024, "dq gemm shared memory");
  static constexpr uint32_t kTmemCols = 256;  // two accumulators of 128 columns
};

// Query blocks [q_lo, q_lo + nq) against key blocks [k_lo, k_lo + nk)
// (key blocks past a query block are not visible); its dS^T tiles start at
// tile `tile0`; `mode` as in AttnPart.  The whole matrix is {0, nb, 0, nb}.
struct DqRect {
  int q_lo, nq, k_lo, nk;
  int mode;
  int64_t tile0;
};

// The rectangles of one launch (disjoint query rows): items
// [item_end[i - 1], item_end[i]) are rectangle i's (query block, head,
// batch) triples; `acc` holds the running dQ sums [b, s, a].
struct DqRects {
  int n;
  int item_end[kCpMaxRects];
  DqRect r[kCpMaxRects];
  float* acc;
  int head_major;  // the whole matrix: every head's heaviest query block first
};

// Item r of CTA blockIdx.x (snake over the dispatch order): rectangle,
// query block within it, head and batch; false once the CTA's share is done.
__device__ __forceinline__ bool dq_item(int r, const DqRects& rects, int H, int& ri, int& qr,
                                        int& hh, int& bi) {
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  const int64_t k = static_cast<int64_t>(r) * G + ((r & 1) ? G - 1 - c : c);
  if (k >= rects.item_end[rects.n - 1]) return false;
  ri = 0;
  while (ri + 1 < rects.n && k >= rects.item_end[ri]) ++ri;
  const int kr = static_cast<int>(k - (ri > 0 ? rects.item_end[ri - 1] : 0));
  const int nq = rects.r[ri].nq;
  int hb;
  if (rects.head_major) {  // (the whole matrix: one rectangle)
    const int n_hb = rects.item_end[0] / nq;
    hb = kr % n_hb;
    qr = nq - 1 - kr / n_hb;
  } else {
    qr = nq - 1 - kr % nq;  // heaviest first within a head
    hb = kr / nq;
  }
  hh = hb % H;
  bi = hb / H;
  return true;
}

template <int D, bool PART>
__global__ void __launch_bounds__(192, 1)
    attn_bwd_dq_gemm_kernel(const __grid_constant__ CUtensorMap tm_qkv,
                            const uint8_t* __restrict__ ds_tiles, uint16_t* __restrict__ dqkv,
                            int s, int H, int* status, const __grid_constant__ DqRects rects) {
  using C = DqGemmCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStage);
  uint64_t* full = bars + 0;       // [3]
  uint64_t* empty = bars + 3;      // [3]
  uint64_t* acc_full = bars + 6;   // [2]  an item's dQ is complete in accumulator a
  uint64_t* acc_empty = bars + 8;  // [2]  the epilogue has read accumulator a (128 threads)
  uint64_t* drain = bars + 10;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 11);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int a = H * D;
  const int nb = (s + 127) / 128;
  const int64_t ntri = static_cast<int64_t>(nb) * (nb + 1) / 2;
  // key blocks R.k_lo .. + n_keys(R, qb) - 1 and the first tile of an item
  auto n_keys = [&](const DqRect& R, int qb) { return PART ? min(R.nk, qb + 1 - R.k_lo) : qb + 1; };
  auto first_tile = [&](const DqRect& R, int qr, int hh, int bi) {
    const int qb = R.q_lo + qr;
    return PART ? R.tile0 + ((static_cast<int64_t>(bi) * H + hh) * R.nq + qr) * R.nk
                : (static_cast<int64_t>(bi) * H + hh) * ntri + static_cast<int64_t>(qb) * (qb + 1) / 2;
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 128);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tm_qkv);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the dK/dV kernel (the dS^T tiles) has completed

  if (warp == 0) {
    if (lane == 0) {
      // -------------------------------------------------------- producer
      int gt = 0;  // tiles issued, across items
      bool ok = true;
      int ri, qr, hh, bi;
      for (int r = 0; ok && dq_item(r, rects, H, ri, qr, hh, bi); ++r) {
        const DqRect& R = rects.r[ri];
        const int64_t tile0 = first_tile(R, qr, hh, bi);
        const int nj = n_keys(R, R.q_lo + qr);
        for (int j = 0; j < nj; ++j, ++gt) {
          const int st = gt % C::kStages;
          if (!mbar_wait(&empty[st], ((gt / C::kStages) & 1) ^ 1u, status, kSiteAttention)) {
            ok = false;
            break;
          }
          uint8_t* dst = smem + st * C::kStage;
          mbar_arrive_expect_tx(&full[st], C::kStage);
          bulk_load(dst, ds_tiles + (tile0 + j) * kDsTileBytes,
                    static_cast<uint32_t>(kDsTileBytes), &full[st]);
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d(dst + kDsTileBytes + c * 16384, &tm_qkv, &full[st], a + hh * D + c * 64,
                        (R.k_lo + j) * 128, bi);
        }
      }
      pdl_launch();  // every load of this CTA is issued
      for (int g = gt - 1; g >= 0 && g >= gt - C::kStages; --g)
        mbar_wait(&full[g % C::kStages], (g / C::kStages) & 1, status, kSiteAttention,
                  200000000ull, false);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // -------------------------------------------------------- MMA issuer
      constexpr uint32_t kIdesc = idesc_bf16_f32(128, D, true, true);
      bool ok = true;
      int gt = 0, ri, qr, hh, bi;
      for (int r = 0; ok && dq_item(r, rects, H, ri, qr, hh, bi); ++r) {
        const int nj = n_keys(rects.r[ri], rects.r[ri].q_lo + qr);
        const int acc = r & 1;
        // the epilogue of item r - 2 has read this accumulator
        if (!mbar_wait(&acc_empty[acc], ((r >> 1) & 1) ^ 1u, status, kSiteAttention)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * 128);
        for (int j = 0; j < nj; ++j, ++gt) {
          const int st = gt % C::kStages;
          if (!mbar_wait(&full[st], (gt / C::kStages) & 1, status, kSiteAttention)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ab = smem_u32(smem + st * C::kStage);
          const uint32_t kbase = ab + static_cast<uint32_t>(kDsTileBytes);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            // 16 keys per step: 16 rows of 128 B in both MN-major operands;
            // 64-wide query (A) or d (B) chunks 16 KB apart
            umma_bf16(d_tmem, smem_desc_sw128(ab + kk * 2048, 16384, 1024),
                      smem_desc_sw128(kbase + kk * 2048, 16384, 1024), kIdesc,
                      (j > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&empty[st]);
        }
        if (ok) umma_commit(&acc_full[acc]);
      }
      umma_commit(drain);
      mbar_wait(drain, 0, status, kSiteAttention, 200000000ull, false);
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float scale = rsqrtf(static_cast<float>(D));
    int ri, qr, hh, bi;
    for (int r = 0; dq_item(r, rects, H, ri, qr, hh, bi); ++r) {
      const int acc = r & 1;
      const DqRect& R = rects.r[ri];
      const int row = (R.q_lo + qr) * 128 + quarter * 32 + lane;  // this thread's query row
      if (!mbar_wait_warp(&acc_full[acc], (r >> 1) & 1, status, kSiteAttention)) break;
      tc_fence_after();
      const int64_t base = (static_cast<int64_t>(bi) * s + row) * 3 * static_cast<int64_t>(a);
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        float v[32];
        tmem_ld_32x32b_x32(tmem + static_cast<uint32_t>(acc * 128) + lane_off + c * 32, v);
        if (row < s && MC_DCHECK(row >= 0 && hh * D + c * 32 + 32 <= a, status, kSiteAttention)) {
          if constexpr (PART) {
            float* run = rects.acc + (static_cast<int64_t>(bi) * s + row) * a + hh * D + c * 32;
            accumulate_row32(v, scale, 1.f, run, dqkv + base + hh * D + c * 32,
                             R.mode & kCpAccMerge, R.mode & kCpAccFinal);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(dqkv + base + hh * D + c * 32);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              uint4 wv;
              wv.x = pack_bf16x2(v[8 * k + 0] * scale, v[8 * k + 1] * scale);
              wv.y = pack_bf16x2(v[8 * k + 2] * scale, v[8 * k + 3] * scale);
              wv.z = pack_bf16x2(v[8 * k + 4] * scale, v[8 * k + 5] * scale);
              wv.w = pack_bf16x2(v[8 * k + 6] * scale, v[8 * k + 7] * scale);
              dst[k] = wv;
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[acc]);  // the accumulator may take the item after next
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
int launch_bwd_dq_gemm(const CUtensorMap& tq, const uint8_t* ds_tiles, uint16_t* dqkv, int b,
                       int s, int H, const DqRects& rects, int* status, cudaStream_t st) {
  using C = DqGemmCfg<D>;
  auto kern = attn_bwd_dq_gemm_kernel<D, PART>;
  static PerDeviceInit init;
  const cudaError_t attr = once_per_device(init, [&](long long*) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  });
  if (attr != cudaSuccess) return MC_ERR_CUDA;
  const int n_items = rects.item_end[rects.n - 1];
  const int grid = n_items < num_sms() ? n_items : num_sms();
  launch_kernel(kern, dim3(grid), dim3(192), C::kSmem, st, 1, tq, ds_tiles, dqkv, s, H, status,
                rects);
  return cudaGetLastError() == cudaSuccess ? MC_OK : MC_ERR_CUDA;
}

// Tensor maps over Q|K|V [b, s, 3a] and dO [b, s, a] with 64 x 128 boxes.
bool make_qkv_map(CUtensorMap* tq, const uint16_t* qkv, int b, int s, int a_) {
  const uint64_t a = static_cast<uint64_t>(a_);
  const uint32_t box[3] = {64, 128, 1};
  const uint64_t dq[3] = {3 * a, static_cast<uint64_t>(s), static_cast<uint64_t>(b)};
  const uint64_t sq[2] = {3 * a * 2, 3 * a * 2 * static_cast<uint64_t>(s)};
  return make_tmap_bf16(tq, qkv, 3, dq, sq, box);
}

bool make_bwd_maps(CUtensorMap* tq, CUtensorMap* td, const uint16_t* qkv, const uint16_t* dout,
                   int b, int s, int a_) {
  const uint64_t a = static_cast<uint64_t>(a_);
  const uint32_t box[3] = {64, 128, 1};
  const uint64_t dd[3] = {a, static_cast<uint64_t>(s), static_cast<uint64_t>(b)};
  const uint64_t sd[2] = {a * 2, a * 2 * static_cast<uint64_t>(s)};
  return make_qkv_map(tq, qkv, b, s, a_) && make_tmap_bf16(td, dout, 3, dd, sd, box);
}


// With `ds_tiles` (attention_ds_workspace_bytes of device memory) the dK/dV
// kernel also writes dS^T and dQ is its product with K; without, the dQ
// kernel forms S and dP again.
template <int D>
int launch_bwd_tc(const uint16_t* qkv, const float* lse, const uint16_t* dout, uint16_t* dqkv,
                  const float* delta, int b, int s, int H, int* status, cudaStream_t st,
                  uint8_t* ds_tiles) {
  CUtensorMap tq, td;
  if (!make_bwd_maps(&tq, &td, qkv, dout, b, s, H * D)) return MC_ERR_CUDA;
  const int nb = (s + 127) / 128;
  AttnParts whole = {};
  whole.n = 1;
  whole.cta_end[0] = nb;
  whole.r[0] = {0, s, 0, 0x7fffffff, 0, 0};
  whole.head_major = attention_head_major(nb, H, b) ? 1 : 0;
  int rc = launch_bwd_dkdv_tc<D, false>(tq, td, lse, delta, dqkv, b, s, H, status, st, whole,
                                        ds_tiles);
  if (rc != MC_OK) return rc;
  if (ds_tiles) {
    const int64_t n_items = static_cast<int64_t>(nb) * H * b;
    if (n_items > 0x7fffffff) return MC_ERR_UNSUPPORTED;
    DqRects dq = {};
    dq.n = 1;
    dq.item_end[0] = static_cast<int>(n_items);
    dq.r[0] = {0, nb, 0, nb, 0, 0};
    dq.head_major = attention_head_major(nb, H, b) ? 1 : 0;
    return launch_bwd_dq_gemm<D, false>(tq, ds_tiles, dqkv, b, s, H, dq, status, st);
  }
  return launch_bwd_dq_tc<D>(tq, td, lse, delta, dqkv, b, s, H, status, st);
}

}  // namespace

int64_t attention_ds_workspace_bytes(int64_t b, int64_t s, int64_t H) {
  const int64_t nb = (s + 127) / 128;
  return b * H * (nb * (nb + 1) / 2) * kDsTileBytes;
}

int launch_attention_backward_tc(const uint16_t* qkv, const float* lse, const uint16_t* dout,
                                 uint16_t* dqkv, const float* delta, int b, int s, int H, int d,
                                 int* status, cudaStream_t st, uint8_t* ds_tiles) {
  return d == 64 ? launch_bwd_tc<64>(qkv, lse, dout, dqkv, delta, b, s, H, status, st, ds_tiles)
                 : launch_bwd_tc<128>(qkv, lse, dout, dqkv, delta, b, s, H, status, st, ds_tiles);
}

int64_t attention_cp_tile_bytes(const CpRect* rects, int n, int64_t b, int64_t H) {
  int64_t tiles = 0;
  for (int i = 0; i < n; ++i)
    tiles += b * H * (rects[i].q_len / 128) * static_cast<int64_t>(rects[i].k_len / 128);
  return tiles * kDsTileBytes;
}

namespace {
// Rectangles off the diagonal (every CTA or item the same length) go first
// in a launch, the diagonal ones (heaviest first inside) after them; the
// dS^T tiles keep the order given.
template <typename F>
void for_each_rect_heavy_first(const CpRect* rects, int n, F&& f) {
  for (int pass = 0; pass < 2; ++pass)
    for (int i = 0; i < n; ++i)
      if ((rects[i].q_base == rects[i].k_base) == (pass == 1)) f(i);
}

void rect_tile_offsets(const CpRect* rects, int n, int64_t b, int64_t H, int64_t* tile0) {
  int64_t t0 = 0;
  for (int i = 0; i < n; ++i) {
    tile0[i] = t0;
    t0 += b * H * (rects[i].q_len / 128) * static_cast<int64_t>(rects[i].k_len / 128);
  }
}
}  // namespace

int launch_attention_dkdv_parts(const uint16_t* qkv, const float* lse, const uint16_t* dout,
                                const float* delta, uint16_t* dqkv, int b, int s, int H, int d,
                                const CpRect* rects, int n, float* acc_dkv, uint8_t* ds_tiles,
                                int* status, cudaStream_t st) {
  if (check_cp_rects(rects, n, s) != MC_OK || !ds_tiles) return MC_ERR_ARGUMENT;
  CUtensorMap tq, td;
  if (!make_bwd_maps(&tq, &td, qkv, dout, b, s, H * d)) return MC_ERR_CUDA;
  int64_t tile0[kCpMaxRects];
  rect_tile_offsets(rects, n, b, H, tile0);
  AttnParts p = {};
  p.acc = acc_dkv;
  for_each_rect_heavy_first(rects, n, [&](int i) {
    const CpRect& r = rects[i];
    p.r[p.n] = {r.k_base, r.k_len, r.q_base / 128, (r.q_base + r.q_len) / 128, r.mode_k, tile0[i]};
    p.cta_end[p.n] = (p.n > 0 ? p.cta_end[p.n - 1] : 0) + r.k_len / 128;
    ++p.n;
  });
  return d == 64 ? launch_bwd_dkdv_tc<64, true>(tq, td, lse, delta, dqkv, b, s, H, status, st, p,
                                                ds_tiles)
                 : launch_bwd_dkdv_tc<128, true>(tq, td, lse, delta, dqkv, b, s, H, status, st, p,
                                                 ds_tiles);
}

int launch_attention_dq_parts(const uint16_t* qkv, const uint8_t* ds_tiles, uint16_t* dqkv, int b,
                              int s, int H, int d, const CpRect* rects, int n, float* acc_dq,
                              int* status, cudaStream_t st) {
  if (check_cp_rects(rects, n, s) != MC_OK || !ds_tiles) return MC_ERR_ARGUMENT;
  CUtensorMap tq;
  if (!make_qkv_map(&tq, qkv, b, s, H * d)) return MC_ERR_CUDA;
  int64_t tile0[kCpMaxRects];
  rect_tile_offsets(rects, n, b, H, tile0);
  DqRects q = {};
  q.acc = acc_dq;
  int64_t items = 0;
  for_each_rect_heavy_first(rects, n, [&](int i) {
    const CpRect& r = rects[i];
    q.r[q.n] = {r.q_base / 128, r.q_len / 128, r.k_base / 128, r.k_len / 128, r.mode_q, tile0[i]};
    items += static_cast<int64_t>(r.q_len / 128) * H * b;
    q.item_end[q.n] = static_cast<int>(items < 0x7fffffff ? items : 0x7fffffff);
    ++q.n;
  });
  if (items > 0x7fffffff) return MC_ERR_UNSUPPORTED;
  return d == 64 ? launch_bwd_dq_gemm<64, true>(tq, ds_tiles, dqkv, b, s, H, q, status, st)
                 : launch_bwd_dq_gemm<128, true>(tq, ds_tiles, dqkv, b, s, H, q, status, st);
}

}  // namespace mc
