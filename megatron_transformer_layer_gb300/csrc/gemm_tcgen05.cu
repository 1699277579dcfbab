// Persistent, warp-specialised BF16 GEMM on the sm_103a tensor cores.
//
//   C[M, N] = sum_k A[m, k] * B[n, k]      (fp32 accumulation in TMEM)
//
// One CTA per SM walks a grouped sequence of 128 x BN output tiles.
//   warp 0      TMA producer: 128B-swizzled A/B boxes -> STAGES-deep smem ring
//   warp 1      allocates TMEM (2 accumulators of BN fp32 columns) and, from
//               one thread, issues tcgen05.mma (M = 128, N = BN, K = 16)
//   warps 2..9  epilogue: tcgen05.ld the accumulator, apply the fused
//               epilogue, store to global memory; two warps per TMEM lane
//               quarter, each taking half of the tile's columns; the second
//               accumulator lets the next tile's main loop run underneath.
//               Each warp's 32 x 32 blocks pass through shared memory so
//               that its global accesses cover whole rows (coalesced).
//
// Operands may be K-major ([rows, K] in memory) or MN-major ([K, rows] in
// memory); the latter is how the dgrad (W used as [K, N]) and wgrad
// (activations used transposed) products read their operands without any
// transpose pass.  For a row-parallel product the K range is the
// concatenation of the tp_parts partitions' K-slices, so each partition's
// partial product is added into the same fp32 accumulator in partition order:
// the cross-partition sum happens inside the accumulator and the epilogue
// applies bias and residual once, after the sum.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "mc_layer_internal.h"
#include "ptx.cuh"

namespace mc {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;  // one 128-byte swizzle atom of bf16 along K
constexpr int kEpilogueWarps = 8;  // two per TMEM lane quarter, splitting the columns
constexpr int kThreads = 64 + 32 * kEpilogueWarps;
constexpr int kEpilogueThreads = 32 * kEpilogueWarps;

struct GemmArgs {
  int M, N, K;
  int num_kb;
  int m_tiles, n_tiles, num_tiles;
  int m_pairs, num_units;  // paired variant: units = (pair of M-tiles, N-tile)
  void* out;
  int64_t ldc;
  const __nv_bfloat16* bias;
  const void* aux;
  int64_t ldaux;
  int accumulate;
  int* status;
  // 8-bit operands: the instruction descriptor (formats) and the device
  // scalars whose product dequantises the fp32 accumulator
  uint32_t idesc_f8;
  const float* a_scale_inv;
  const float* b_scale_inv;
};

// Execution modes of the GEMM kernel.
//   kSolo   one CTA per 128 x BN tile
//   kDuo    clusters of two CTAs run one 256 x BN tile (M-tiles 2p, 2p + 1 of
//           one N-tile) with tcgen05.mma.cta_group::2: each CTA holds only its
//           own 128 rows of A and its half of B, and the even CTA issues the
//           MMAs for both.  Per flop each SM receives 2/3 of the operand bytes
//           of a 128 x 256 tile, which is what keeps the tensor pipe fed from L2.
constexpr int kSolo = 0, kDuo = 1;

template <int BN, int MODE, int EPI>
struct GemmCfg {
  static constexpr int kABytes = BM * BK * 2;
  // B bytes held per CTA and stage
  static constexpr int kBBytes = (MODE == kDuo ? BN / 2 : BN) * BK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = kStageBytes > 32768 ? 4 : 6;
  // bytes that complete one stage's full barrier (kDuo: both CTAs' copies
  // land on the even CTA's barrier)
  static constexpr int kTxBytes = MODE == kDuo ? 2 * kStageBytes : kStageBytes;
  static constexpr int kTmemCols = 2 * BN;
  // ring + barriers (full, empty, acc_full x2, acc_empty x2, drain) + tmem slot
  static constexpr int kBarrierBytes = (2 * kStages + 5) * 8 + 8;
  // the epilogue's 32 x 33-float block per epilogue warp
  static constexpr int kEpiBytes = kEpilogueWarps * 32 * 33 * 4;
  static constexpr int kSmemBytes =
      kStages * kStageBytes + kBarrierBytes + kEpiBytes + 1024;  // +align
  static_assert(kSmemBytes <= 227 * 1024, "gemm shared memory");
};

__device__ __forceinline__ void tile_coords(int tile, int m_tiles, int n_tiles, int& mb, int& nb) {
  constexpr int G = 8;  // M tiles per group; a group sweeps all N tiles
  const int per_group = G * n_tiles;
  const int group = tile / per_group;
  const int first_m = group * G;
  const int gsize = min(G, m_tiles - first_m);
  const int r = tile - group * per_group;
  mb = first_m + r % gsize;
  nb = r / gsize;
}

__device__ __forceinline__ float gelu_tanh(float x) {
  const float c = 0.7978845608028654f;  // sqrt(2/pi)
  const float u = c * fmaf(0.044715f * x, x * x, x);
  return 0.5f * x * (1.0f + tanhf(u));
}

__device__ __forceinline__ float gelu_tanh_grad(float x) {
  const float c = 0.7978845608028654f;
  const float x2 = x * x;
  const float th = tanhf(c * fmaf(0.044715f * x, x2, x));
  return 0.5f * (1.0f + th) + 0.5f * x * (1.0f - th * th) * c * fmaf(3.0f * 0.044715f, x2, 1.0f);
}

// 8 bf16 values (16 bytes) <-> 8 floats.
__device__ __forceinline__ void unpack_bf16x8(const uint4 w, float (&v)[8]) {
  v[0] = bf16_lo(w.x);
  v[1] = bf16_hi(w.x);
  v[2] = bf16_lo(w.y);
  v[3] = bf16_hi(w.y);
  v[4] = bf16_lo(w.z);
  v[5] = bf16_hi(w.z);
  v[6] = bf16_lo(w.w);
  v[7] = bf16_hi(w.w);
}

__device__ __forceinline__ uint4 pack_bf16x8(const float (&v)[8]) {
  return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                    pack_bf16x2(v[6], v[7]));
}

// The fused epilogue of one warp's 32 x 32 block of the accumulator: rows
// r0 + [0, 32), columns col0 + [0, 32).  tcgen05.ld leaves one row per lane
// (v); the block goes through shared memory (`blk`, rows padded to 33
// floats, so that both phases are free of bank conflicts) and comes back
// with several lanes on one row, so that each 16-byte global access of the
// warp touches 4 (fp32) or 8 (bf16) rows instead of 32.  Every global read
// of the epilogue (residual, pre-activation, the output added to) is issued
// before the first store, which could alias it.
template <int EPI>
__device__ __forceinline__ void epilogue_block(const float (&v)[32], float* blk, int lane, int r0,
                                               int col0, const GemmArgs& g) {
  auto stage = [&] {
#pragma unroll
    for (int k = 0; k < 32; ++k) blk[lane * 33 + k] = v[k];
    __syncwarp();
  };
  const bool cols_ok =
      col0 < g.N && MC_DCHECK(col0 + 32 <= g.N && g.N <= g.ldc && r0 >= 0, g.status,
                              kSiteGemmEpilogue);
  if constexpr (EPI == MC_EPI_STORE_F32 || EPI == MC_EPI_BIAS_RESID_F32) {
    // fp32: 8 lanes per row, 4 columns each; rows 4 i + lane / 8
    stage();
    const int sub = lane & 7;
    constexpr bool kResid = EPI == MC_EPI_BIAS_RESID_F32;
    const bool reads = kResid || g.accumulate;
    float4 bias4 = make_float4(0.f, 0.f, 0.f, 0.f);
    if constexpr (kResid) {
      const uint2 bw = *reinterpret_cast<const uint2*>(g.bias + col0 + 4 * sub);
      bias4 = make_float4(bf16_lo(bw.x), bf16_hi(bw.x), bf16_lo(bw.y), bf16_hi(bw.y));
    }
    float4 x[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int grow = r0 + 4 * i + (lane >> 3);
      x[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (reads && cols_ok && grow < g.M) {
        const float* base = kResid ? static_cast<const float*>(g.aux) + (int64_t)grow * g.ldaux
                                   : static_cast<const float*>(g.out) + (int64_t)grow * g.ldc;
        x[i] = *reinterpret_cast<const float4*>(base + col0 + 4 * sub);
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int lr = 4 * i + (lane >> 3);
      const int grow = r0 + lr;
      const float* src = blk + lr * 33 + 4 * sub;
      float4 w = make_float4(src[0], src[1], src[2], src[3]);
      if (cols_ok && grow < g.M) {
        if constexpr (kResid)  // (acc + bias) + residual
          w = make_float4(w.x + bias4.x + x[i].x, w.y + bias4.y + x[i].y, w.z + bias4.z + x[i].z,
                          w.w + bias4.w + x[i].w);
        else if (g.accumulate)
          w = make_float4(w.x + x[i].x, w.y + x[i].y, w.z + x[i].z, w.w + x[i].w);
        *reinterpret_cast<float4*>(static_cast<float*>(g.out) + (int64_t)grow * g.ldc + col0 +
                                   4 * sub) = w;
      }
    }
    __syncwarp();  // the block is read before the next chunk overwrites it
  } else {
    // bf16: 4 lanes per row, 8 columns each; rows 8 i + lane / 4
    stage();
    const int sub = lane & 3;
    float b[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if constexpr (EPI == MC_EPI_BIAS_BF16 || EPI == MC_EPI_BIAS_GELU)
      unpack_bf16x8(*reinterpret_cast<const uint4*>(g.bias + col0 + 8 * sub), b);
    uint4 hp[4];  // GELU_BWD: the pre-activation
    if constexpr (EPI == MC_EPI_GELU_BWD) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int grow = r0 + 8 * i + (lane >> 2);
        hp[i] = make_uint4(0u, 0u, 0u, 0u);
        if (cols_ok && grow < g.M)
          hp[i] = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(g.aux) +
                                                  (int64_t)grow * g.ldaux + col0 + 8 * sub);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int lr = 8 * i + (lane >> 2);
      const int grow = r0 + lr;
      float x[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) x[k] = blk[lr * 33 + 8 * sub + k];
      if (!cols_ok || grow >= g.M) continue;
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(g.out) + (int64_t)grow * g.ldc + col0 + 8 * sub;
      if constexpr (EPI == MC_EPI_BIAS_BF16 || EPI == MC_EPI_BIAS_GELU) {
#pragma unroll
        for (int k = 0; k < 8; ++k) x[k] += b[k];
      }
      if constexpr (EPI == MC_EPI_BIAS_GELU) {
        // the pre-activation for the backward, then the activation
        *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(const_cast<void*>(g.aux)) +
                                  (int64_t)grow * g.ldaux + col0 + 8 * sub) = pack_bf16x8(x);
#pragma unroll
        for (int k = 0; k < 8; ++k) x[k] = gelu_tanh(x[k]);
      }
      if constexpr (EPI == MC_EPI_GELU_BWD) {
        float h[8];
        unpack_bf16x8(hp[i], h);
#pragma unroll
        for (int k = 0; k < 8; ++k) x[k] *= gelu_tanh_grad(h[k]);
      }
      *reinterpret_cast<uint4*>(out) = pack_bf16x8(x);
    }
    __syncwarp();  // the block is read before the next chunk overwrites it
  }
}

// kDuo: CTAs run in clusters of two along M.  Each CTA loads its A rows and
// its half of B into its own shared memory, both signalling the even CTA's
// full barrier; the even CTA issues 256 x BN x 16 MMAs that read both CTAs'
// operands and write each CTA's 128 accumulator rows into its own TMEM, and
// its commits arrive on the barriers of both CTAs (a stage is refilled, an
// accumulator read, only then); the odd CTA's epilogue releases the
// accumulator on the even CTA's barrier.
// F8: operands are 8-bit floats (E4M3 / E5M2, K-major only): a 128-byte
// swizzled row then holds 128 elements of K instead of 64, each MMA takes
// K = 32 (kind::f8f6f4) and the epilogue multiplies by the two operands'
// dequantisation scales before the fused epilogue.
template <bool A_MN, bool B_MN, int BN, int EPI, int MODE, bool F8>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, const GemmArgs g) {
  using Cfg = GemmCfg<BN, MODE, EPI>;
  constexpr int S = Cfg::kStages;
  constexpr bool kDuoMode = MODE == kDuo;
  static_assert(!F8 || (!A_MN && !B_MN), "8-bit operands are K-major");
  constexpr int kBKE = F8 ? 2 * BK : BK;  // K elements per 128-byte row
  constexpr uint32_t kIdesc = idesc_bf16_f32(kDuoMode ? 2 * BM : BM, BN, A_MN, B_MN);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + S * Cfg::kABytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * Cfg::kStageBytes);
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  float* epi_stage = reinterpret_cast<float*>(smem + S * Cfg::kStageBytes + Cfg::kBarrierBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t crank = kDuoMode ? cluster_ctarank() : 0u;
  const bool issuer_cta = crank == 0u;  // kDuo: the CTA that issues the pair's MMAs
  // Work units: output tiles, or (pairs) pairs of M-tiles sharing an N-tile.
  const int unit0 = kDuoMode ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int ustride = kDuoMode ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  const int n_units = kDuoMode ? g.num_units : g.num_tiles;
  auto unit_coords = [&](int u, int& mb, int& nb) {
    if constexpr (kDuoMode) {
      int mp;
      tile_coords(u, g.m_pairs, g.n_tiles, mp, nb);
      mb = 2 * mp + static_cast<int>(crank);
    } else {
      tile_coords(u, g.m_tiles, g.n_tiles, mb, nb);
    }
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      // kDuo: one arrival per epilogue warp of both CTAs
      mbar_init(&acc_empty[i], kDuoMode ? 2 * kEpilogueWarps : kEpilogueThreads);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    if constexpr (kDuoMode) {
      tmem_alloc_pair(tmem_slot, Cfg::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, Cfg::kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // The peer's copies, commits and arrivals target this CTA's
  // barriers: both CTAs must have initialised theirs first.
  if constexpr (kDuoMode) cluster_sync();
  pdl_wait();  // the previous kernel on the stream has completed

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      // kDuo: the even CTA's full barriers, which count both CTAs' bytes
      const uint32_t full0_pair = kDuoMode ? mapa_shared(full, 0) : 0u;
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      for (int u = unit0; ok && u < n_units; u += ustride) {
        int mb, nb;
        unit_coords(u, mb, nb);
        for (int kb = 0; kb < g.num_kb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, g.status, kSiteGemmProducer)) {
            ok = false;
            break;
          }
          const int k0 = kb * kBKE;
          uint8_t* a_dst = sA + stage * Cfg::kABytes;
          uint8_t* b_dst = sB + stage * Cfg::kBBytes;
          if constexpr (kDuoMode) {
            if (issuer_cta) mbar_arrive_expect_tx(&full[stage], Cfg::kTxBytes);
            const uint32_t fb = full0_pair + static_cast<uint32_t>(stage) * 8u;
            if constexpr (!A_MN) {
              tma_load_2d_pair(a_dst, &tmA, fb, k0, mb * BM);
            } else {
              tma_load_2d_pair(a_dst, &tmA, fb, mb * BM, k0);
              tma_load_2d_pair(a_dst + 64 * BK * 2, &tmA, fb, mb * BM + 64, k0);
            }
            // this CTA's half of the B tile: N rows [nb BN + crank BN/2, + BN/2)
            if constexpr (!B_MN) {
              tma_load_2d_pair(b_dst, &tmB, fb, k0, nb * BN + static_cast<int>(crank) * (BN / 2));
            } else {
#pragma unroll
              for (int j = 0; j < BN / 128; ++j) {
                const int jj = static_cast<int>(crank) * (BN / 128) + j;
                tma_load_2d_pair(b_dst + j * 64 * BK * 2, &tmB, fb, nb * BN + jj * 64, k0);
              }
            }
          } else {
            mbar_arrive_expect_tx(&full[stage], Cfg::kTxBytes);
            if constexpr (!A_MN) {
              tma_load_2d(a_dst, &tmA, &full[stage], k0, mb * BM);
            } else {
              tma_load_2d(a_dst, &tmA, &full[stage], mb * BM, k0);
              tma_load_2d(a_dst + 64 * BK * 2, &tmA, &full[stage], mb * BM + 64, k0);
            }
            if constexpr (!B_MN) {
              tma_load_2d(b_dst, &tmB, &full[stage], k0, nb * BN);
            } else {
#pragma unroll
              for (int j = 0; j < BN / 64; ++j)
                tma_load_2d(b_dst + j * 64 * BK * 2, &tmB, &full[stage], nb * BN + j * 64, k0);
            }
          }
          ++issued;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Every load of this CTA is issued: the next kernel on the stream may
      // start its prologue on SMs this grid releases.
      pdl_launch();
      // Wait for the copies still in flight (the last use of each stage)
      // before the CTA may exit.  kDuo: the even CTA's full barriers count
      // both CTAs' copies, and the closing cluster barrier holds the odd CTA
      // until the even one has seen them land.
      if (!kDuoMode || issuer_cta) {
        const int pending = issued < S ? issued : S;
        for (int i = 0; i < pending; ++i) {
          stage = stage == 0 ? S - 1 : stage - 1;
          if (stage == S - 1) phase ^= 1u;
          mbar_wait(&full[stage], phase, g.status, kSiteGemmDrain, 200000000ull, false);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && (!kDuoMode || issuer_cta)) {
      // ---------------------------------------------------------- MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int u = unit0; ok && u < n_units; u += ustride) {
        const bool got = kDuoMode ? mbar_wait<true>(&acc_empty[acc], acc_phase ^ 1u, g.status,
                                                    kSiteGemmMma)
                                  : mbar_wait(&acc_empty[acc], acc_phase ^ 1u, g.status,
                                              kSiteGemmMma);
        if (!got) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        // The K loop runs over the partitions' K-slices in order; all of them
        // accumulate into d_tmem.
        for (int kb = 0; kb < g.num_kb; ++kb) {
          if (!mbar_wait(&full[stage], phase, g.status, kSiteGemmMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * Cfg::kABytes);
          const uint32_t b0 = smem_u32(sB + stage * Cfg::kBBytes);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            // K-major: a K step of 16 bf16 (32 fp8) is 32 bytes inside the swizzled row.
            // MN-major: a K step is 16 rows of 128 bytes; LBO = 64-wide MN chunk.
            const uint64_t ad = A_MN ? smem_desc_sw128(a0 + k * 2048, 64 * BK * 2, 1024)
                                     : smem_desc_sw128(a0 + k * 32, 16, 1024);
            const uint64_t bd = B_MN ? smem_desc_sw128(b0 + k * 2048, 64 * BK * 2, 1024)
                                     : smem_desc_sw128(b0 + k * 32, 16, 1024);
            if constexpr (F8 && kDuoMode)
              umma_f8_pair(d_tmem, ad, bd, g.idesc_f8, (kb | k) != 0 ? 1u : 0u);
            else if constexpr (F8)
              umma_f8(d_tmem, ad, bd, g.idesc_f8, (kb | k) != 0 ? 1u : 0u);
            else if constexpr (kDuoMode)
              umma_bf16_pair(d_tmem, ad, bd, kIdesc, (kb | k) != 0 ? 1u : 0u);
            else
              umma_bf16(d_tmem, ad, bd, kIdesc, (kb | k) != 0 ? 1u : 0u);
          }
          if constexpr (kDuoMode)
            umma_commit_pair_mc(&empty[stage], 0x3);  // frees the stage in both CTAs
          else
            umma_commit(&empty[stage]);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (kDuoMode)
          umma_commit_pair_mc(&acc_full[acc], 0x3);
        else
          umma_commit(&acc_full[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // Every MMA issued by this thread must be complete before TMEM is freed.
      if constexpr (kDuoMode)
        umma_commit_pair_mc(drain, 0x3);
      else
        umma_commit(drain);
      mbar_wait(drain, 0, g.status, kSiteGemmDrain, 200000000ull, false);
    } else if (kDuoMode && lane == 0) {
      // The odd CTA's TMEM is written by the even CTA's MMAs.
      mbar_wait(drain, 0, g.status, kSiteGemmDrain, 200000000ull, false);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;      // TMEM lanes [32 q, 32 q + 32)
    const int half = (warp - 2) >> 2;  // which half of the tile's columns
    const uint32_t acc_empty_pair = kDuoMode ? mapa_shared(acc_empty, 0) : 0u;
    const float dq = F8 ? *g.a_scale_inv * *g.b_scale_inv : 1.f;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = unit0; u < n_units; u += ustride) {
      int mb, nb;
      unit_coords(u, mb, nb);
      if (!mbar_wait_warp(&acc_full[acc], acc_phase, g.status, kSiteGemmEpilogue)) break;
      tc_fence_after();
      const int r0 = mb * BM + quarter * 32;  // the warp's 32 rows
      float* blk = epi_stage + (warp - 2) * (32 * 33);
      const uint32_t t_row = tmem_base + static_cast<uint32_t>(acc * BN) +
                             (static_cast<uint32_t>(quarter * 32) << 16);
#pragma unroll 1
      for (int c = half * (BN / 64); c < (half + 1) * (BN / 64); ++c) {
        float v[32];
        tmem_ld_32x32b_x32(t_row + c * 32, v);
        const int col0 = nb * BN + c * 32;
        if constexpr (F8) {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= dq;
        }
        epilogue_block<EPI>(v, blk, lane, r0, col0, g);
      }
      tc_fence_before();
      if constexpr (kDuoMode) {
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(acc_empty_pair + static_cast<uint32_t>(acc) * 8u);
      } else {
        mbar_arrive(&acc_empty[acc]);
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  if constexpr (kDuoMode) {
    // Both CTAs are done with both CTAs' TMEM, barriers and shared memory
    // before the pair frees its tensor memory together and exits.
    cluster_sync();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
    }
  } else {
    __syncthreads();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tmem_base, Cfg::kTmemCols);
    }
  }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2D bf16 tensor map over a row-major matrix [outer, inner] with row stride
// `ld` elements, box [box_outer, box_inner], 128-byte swizzle, zero fill.
// u8: 8-bit elements (ld in elements = bytes) instead of bf16.
bool make_tmap(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t ld,
               uint32_t box_inner, uint32_t box_outer, bool u8 = false) {
  auto enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld * (u8 ? 1 : 2)};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, u8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <bool A_MN, bool B_MN, int BN, int EPI, int MODE, bool F8 = false>
int launch_variant(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& g,
                   cudaStream_t stream) {
  using Cfg = GemmCfg<BN, MODE, EPI>;
  constexpr bool PAIR = MODE == kDuo;
  auto kern = gemm_tcgen05_kernel<A_MN, B_MN, BN, EPI, MODE, F8>;
  static PerDeviceInit init;
  long long max_clusters = 0;
  const cudaError_t attr_err = once_per_device(init, [&](long long* value) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::kSmemBytes);
    if (e == cudaSuccess && PAIR) {
      // Clusters of two that fit on the device at once (pairs must share a
      // GPC, so this can be below half the SM count).
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = 2;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(2 * num_sms(), 1, 1);
      cfg.blockDim = dim3(kThreads, 1, 1);
      cfg.dynamicSmemBytes = Cfg::kSmemBytes;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      int n = 0;
      e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
      if (e == cudaSuccess && n < 1) e = cudaErrorInvalidConfiguration;
      *value = n;
    }
    return e;
  }, &max_clusters);
  if (attr_err != cudaSuccess) return MC_ERR_CUDA;
  if constexpr (PAIR) {
    const int clusters =
        g.num_units < max_clusters ? g.num_units : static_cast<int>(max_clusters);
    if (launch_kernel(kern, dim3(2 * clusters), dim3(kThreads), Cfg::kSmemBytes, stream, 2u, ta,
                      tb, g) != cudaSuccess)
      return MC_ERR_CUDA;
  } else {
    const int grid = g.num_tiles < num_sms() ? g.num_tiles : num_sms();
    if (launch_kernel(kern, dim3(grid), dim3(kThreads), Cfg::kSmemBytes, stream, 1u, ta, tb, g) !=
        cudaSuccess)
      return MC_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? MC_OK : MC_ERR_CUDA;
}

template <int BN, int EPI, int MODE>
int dispatch_layouts(int a_layout, int b_layout, const CUtensorMap& ta, const CUtensorMap& tb,
                     const GemmArgs& g, cudaStream_t stream) {
  if (!a_layout && !b_layout) return launch_variant<false, false, BN, EPI, MODE>(ta, tb, g, stream);
  if (!a_layout && b_layout) return launch_variant<false, true, BN, EPI, MODE>(ta, tb, g, stream);
  if (a_layout && b_layout) return launch_variant<true, true, BN, EPI, MODE>(ta, tb, g, stream);
  return launch_variant<true, false, BN, EPI, MODE>(ta, tb, g, stream);
}

template <int BN, int MODE>
int dispatch_epilogue(int epi, int a_layout, int b_layout, const CUtensorMap& ta,
                      const CUtensorMap& tb, const GemmArgs& g, cudaStream_t stream) {
  switch (epi) {
    case MC_EPI_STORE_F32:
      return dispatch_layouts<BN, MC_EPI_STORE_F32, MODE>(a_layout, b_layout, ta, tb, g, stream);
    case MC_EPI_STORE_BF16:
      return dispatch_layouts<BN, MC_EPI_STORE_BF16, MODE>(a_layout, b_layout, ta, tb, g, stream);
    case MC_EPI_BIAS_BF16:
      return dispatch_layouts<BN, MC_EPI_BIAS_BF16, MODE>(a_layout, b_layout, ta, tb, g, stream);
    case MC_EPI_BIAS_GELU:
      return dispatch_layouts<BN, MC_EPI_BIAS_GELU, MODE>(a_layout, b_layout, ta, tb, g, stream);
    case MC_EPI_BIAS_RESID_F32:
      return dispatch_layouts<BN, MC_EPI_BIAS_RESID_F32, MODE>(a_layout, b_layout, ta, tb, g,
                                                               stream);
    case MC_EPI_GELU_BWD:
      return dispatch_layouts<BN, MC_EPI_GELU_BWD, MODE>(a_layout, b_layout, ta, tb, g, stream);
    default:
      return MC_ERR_ARGUMENT;
  }
}

template <int BN, int MODE>
int dispatch_epilogue_f8(int epi, const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& g,
                         cudaStream_t stream) {
  switch (epi) {
    case MC_EPI_STORE_F32:
      return launch_variant<false, false, BN, MC_EPI_STORE_F32, MODE, true>(ta, tb, g, stream);
    case MC_EPI_STORE_BF16:
      return launch_variant<false, false, BN, MC_EPI_STORE_BF16, MODE, true>(ta, tb, g, stream);
    case MC_EPI_BIAS_BF16:
      return launch_variant<false, false, BN, MC_EPI_BIAS_BF16, MODE, true>(ta, tb, g, stream);
    case MC_EPI_BIAS_GELU:
      return launch_variant<false, false, BN, MC_EPI_BIAS_GELU, MODE, true>(ta, tb, g, stream);
    case MC_EPI_BIAS_RESID_F32:
      return launch_variant<false, false, BN, MC_EPI_BIAS_RESID_F32, MODE, true>(ta, tb, g,
                                                                                  stream);
    case MC_EPI_GELU_BWD:
      return launch_variant<false, false, BN, MC_EPI_GELU_BWD, MODE, true>(ta, tb, g, stream);
    default:
      return MC_ERR_ARGUMENT;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Tile shape of an M x N product: the one whose estimated time, waves x time
// per tile, is smallest.  Clocks per 16-deep K step (bf16; 32-deep fp8)
// measured on this GPU with one MMA stream per SM and operands resident:
// SM-pair 256 x 256 tile 128 (each SM reads 8 KB of operands per step), one
// CTA 128 x 256 161, one CTA 128 x 128 97 (shared-memory operand reads bound
// the single-CTA shapes).  Pairs need N % 256 == 0 and two M-tiles.
struct TileChoice {
  int bn;
  bool pair;
};
TileChoice choose_tiles(int64_t m_tiles, int64_t N) {
  const int64_t sms = num_sms();
  const int64_t clusters = sms / 2;
  auto waves = [](int64_t units, int64_t slots) { return (units + slots - 1) / slots; };
  TileChoice best = {128, false};
  int64_t best_cost = waves(m_tiles * ((N + 127) / 128), sms) * 97;
  if (N % 256 == 0) {
    const int64_t solo = waves(m_tiles * (N / 256), sms) * 161;
    if (solo < best_cost) best = {256, false}, best_cost = solo;
    if (m_tiles >= 2) {
      const int64_t duo = waves(((m_tiles + 1) / 2) * (N / 256), clusters) * 128;
      if (duo <= best_cost) best = {256, true}, best_cost = duo;
    }
  }
  return best;
}

}  // namespace

bool make_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box) {
  auto enc = get_encode_fn();
  if (!enc || rank < 1 || rank > 5) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) st[i] = strides_bytes[i];
  }
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), d, st, bx,
                   es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int launch_gemm(int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda, int a_layout,
                const uint16_t* B, int64_t ldb, int b_layout, void* out, int64_t ldc, int epi,
                const uint16_t* bias, const void* aux, int64_t ldaux, int accumulate, int k_parts,
                int* status, cudaStream_t stream) {
  if (M < 1 || N < 64 || K < 1 || N % 64 != 0) return MC_ERR_UNSUPPORTED;
  if (M > (1 << 30) || N > (1 << 30) || K > (1 << 30)) return MC_ERR_UNSUPPORTED;
  if (a_layout == 0 && (K % 64 != 0)) return MC_ERR_UNSUPPORTED;
  if (k_parts < 1 || K % k_parts != 0) return MC_ERR_ARGUMENT;
  if (a_layout < 0 || a_layout > 1 || b_layout < 0 || b_layout > 1) return MC_ERR_ARGUMENT;
  if (epi < MC_EPI_STORE_F32 || epi > MC_EPI_GELU_BWD) return MC_ERR_ARGUMENT;
  if (!A || !B || !out) return MC_ERR_NULLPTR;
  const bool needs_bias =
      epi == MC_EPI_BIAS_BF16 || epi == MC_EPI_BIAS_GELU || epi == MC_EPI_BIAS_RESID_F32;
  const bool needs_aux =
      epi == MC_EPI_BIAS_GELU || epi == MC_EPI_BIAS_RESID_F32 || epi == MC_EPI_GELU_BWD;
  if ((needs_bias && !bias) || (needs_aux && !aux)) return MC_ERR_NULLPTR;
  if (!aligned16(A) || !aligned16(B) || !aligned16(out) || (bias && !aligned16(bias)) ||
      (aux && !aligned16(aux)))
    return MC_ERR_ALIGN;
  if (lda % 8 || ldb % 8 || ldc % 8 || (needs_aux && ldaux % 8)) return MC_ERR_ALIGN;
  // Leading dimensions must cover the rows they describe.
  if ((a_layout == 0 ? lda < K : lda < M) || (b_layout == 0 ? ldb < K : ldb < N) || ldc < N ||
      (needs_aux && ldaux < N))
    return MC_ERR_ARGUMENT;

  const int64_t m_tiles = (M + BM - 1) / BM;
  const TileChoice tc = choose_tiles(m_tiles, N);
  const int bn = tc.bn;
  const bool pair = tc.pair;

  CUtensorMap ta, tb;
  bool ok = a_layout == 0 ? make_tmap(&ta, A, K, M, lda, BK, BM)
                          : make_tmap(&ta, A, M, K, lda, 64, BK);
  // K-major B: a paired CTA loads half of the tile's rows
  ok = ok && (b_layout == 0 ? make_tmap(&tb, B, K, N, ldb, BK, pair ? bn / 2 : bn)
                            : make_tmap(&tb, B, N, K, ldb, 64, BK));
  if (!ok) return MC_ERR_CUDA;

  GemmArgs g;
  g.M = static_cast<int>(M);
  g.N = static_cast<int>(N);
  g.K = static_cast<int>(K);
  g.num_kb = static_cast<int>((K + BK - 1) / BK);
  g.m_tiles = static_cast<int>(m_tiles);
  g.n_tiles = static_cast<int>((N + bn - 1) / bn);
  const int64_t tiles = m_tiles * g.n_tiles;
  if (tiles > (1 << 30)) return MC_ERR_UNSUPPORTED;
  g.num_tiles = static_cast<int>(tiles);
  g.m_pairs = static_cast<int>((m_tiles + 1) / 2);
  g.num_units = g.m_pairs * g.n_tiles;
  g.out = out;
  g.ldc = ldc;
  g.bias = reinterpret_cast<const __nv_bfloat16*>(bias);
  g.aux = aux;
  g.ldaux = ldaux;
  g.accumulate = accumulate;
  g.status = status;
  g.idesc_f8 = 0;
  g.a_scale_inv = g.b_scale_inv = nullptr;
  if (pair) return dispatch_epilogue<256, kDuo>(epi, a_layout, b_layout, ta, tb, g, stream);
  return bn == 256 ? dispatch_epilogue<256, kSolo>(epi, a_layout, b_layout, ta, tb, g, stream)
                   : dispatch_epilogue<128, kSolo>(epi, a_layout, b_layout, ta, tb, g, stream);
}

int launch_gemm_fp8(int64_t M, int64_t N, int64_t K, const uint8_t* A, int64_t lda, int a_format,
                    const uint8_t* B, int64_t ldb, int b_format, const float* a_scale_inv,
                    const float* b_scale_inv, void* out, int64_t ldc, int epi,
                    const uint16_t* bias, const void* aux, int64_t ldaux, int accumulate,
                    int k_parts, int* status, cudaStream_t stream) {
  if (M < 1 || N < 64 || K < 1 || N % 64 != 0 || K % 16 != 0) return MC_ERR_UNSUPPORTED;
  if (M > (1 << 30) || N > (1 << 30) || K > (1 << 30)) return MC_ERR_UNSUPPORTED;
  if (k_parts < 1 || K % k_parts != 0) return MC_ERR_ARGUMENT;
  if (a_format < 0 || a_format > 1 || b_format < 0 || b_format > 1) return MC_ERR_ARGUMENT;
  if (epi < MC_EPI_STORE_F32 || epi > MC_EPI_GELU_BWD) return MC_ERR_ARGUMENT;
  if (!A || !B || !out || !a_scale_inv || !b_scale_inv) return MC_ERR_NULLPTR;
  const bool needs_bias =
      epi == MC_EPI_BIAS_BF16 || epi == MC_EPI_BIAS_GELU || epi == MC_EPI_BIAS_RESID_F32;
  const bool needs_aux =
      epi == MC_EPI_BIAS_GELU || epi == MC_EPI_BIAS_RESID_F32 || epi == MC_EPI_GELU_BWD;
  if ((needs_bias && !bias) || (needs_aux && !aux)) return MC_ERR_NULLPTR;
  if (!aligned16(A) || !aligned16(B) || !aligned16(out) || (bias && !aligned16(bias)) ||
      (aux && !aligned16(aux)) || (reinterpret_cast<uintptr_t>(a_scale_inv) & 3u) ||
      (reinterpret_cast<uintptr_t>(b_scale_inv) & 3u))
    return MC_ERR_ALIGN;
  if (lda % 16 || ldb % 16 || ldc % 8 || (needs_aux && ldaux % 8)) return MC_ERR_ALIGN;
  if (lda < K || ldb < K || ldc < N || (needs_aux && ldaux < N)) return MC_ERR_ARGUMENT;

  const int64_t m_tiles = (M + BM - 1) / BM;
  const TileChoice tc = choose_tiles(m_tiles, N);
  const int bn = tc.bn;
  const bool pair = tc.pair;
  constexpr int kBKE = 2 * BK;  // 128 one-byte elements per swizzled row
  CUtensorMap ta, tb;
  if (!make_tmap(&ta, A, K, M, lda, kBKE, BM, true) ||
      !make_tmap(&tb, B, K, N, ldb, kBKE, pair ? bn / 2 : bn, true))
    return MC_ERR_CUDA;

  GemmArgs g;
  g.M = static_cast<int>(M);
  g.N = static_cast<int>(N);
  g.K = static_cast<int>(K);
  g.num_kb = static_cast<int>((K + kBKE - 1) / kBKE);
  g.m_tiles = static_cast<int>(m_tiles);
  g.n_tiles = static_cast<int>((N + bn - 1) / bn);
  const int64_t tiles = m_tiles * g.n_tiles;
  if (tiles > (1 << 30)) return MC_ERR_UNSUPPORTED;
  g.num_tiles = static_cast<int>(tiles);
  g.m_pairs = static_cast<int>((m_tiles + 1) / 2);
  g.num_units = g.m_pairs * g.n_tiles;
  g.out = out;
  g.ldc = ldc;
  g.bias = reinterpret_cast<const __nv_bfloat16*>(bias);
  g.aux = aux;
  g.ldaux = ldaux;
  g.accumulate = accumulate;
  g.status = status;
  g.idesc_f8 = idesc_f8_f32(pair ? 2 * BM : BM, bn, a_format, b_format);
  g.a_scale_inv = a_scale_inv;
  g.b_scale_inv = b_scale_inv;
  if (pair) return dispatch_epilogue_f8<256, kDuo>(epi, ta, tb, g, stream);
  return bn == 256 ? dispatch_epilogue_f8<256, kSolo>(epi, ta, tb, g, stream)
                   : dispatch_epilogue_f8<128, kSolo>(epi, ta, tb, g, stream);
}

}  // namespace mc
