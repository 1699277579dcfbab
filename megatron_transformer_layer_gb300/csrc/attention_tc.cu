// Causal flash attention forward on the sm_103a tensor cores (tcgen05).
//
// One CTA per (128-query tile, head, batch), heaviest tiles first:
//   warp 0      TMA: the Q tile once, then K/V tiles of 128 keys into a
//               2-deep ring (3-D tensor map over Q|K|V [b, s, 3a]: rows past
//               the sequence read zeros)
//   warp 1      allocates 512 TMEM columns and issues tcgen05.mma from one
//               thread: S_j = Q K_j^T (M = 128, N = 128, K = d) into one of
//               two S buffers, then O += P_{j-1} V_{j-1} (M = 128, N = d,
//               K = 128) with P read from tensor memory
//   warps 2..5  one thread per query row: load the S row from TMEM, mask,
//               online softmax (running max and sum, exp2 with log2(e)/sqrt(d)
//               folded in), write P back into the S buffer as bf16 pairs;
//               at the end normalise O and store O and the log-sum-exp.
// O is rescaled in TMEM only when a row's running max grows by more than 8
// (log2 units); otherwise P is formed against the stale max (values <= 2^8),
// which is exact because the final normalisation divides by the sum taken
// against the same max.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "mc_layer_internal.h"
#include "ptx.cuh"

namespace mc {
namespace {

constexpr int kThreads = 192;
constexpr int BQ = 128;   // query rows per CTA
constexpr int BKV = 128;  // keys per block
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;

template <int D>
struct FwdCfg {
  static constexpr int kChunks = D / 64;              // 128-byte boxes per row
  static constexpr int kTile = 128 * D * 2;           // [128 rows][D] bf16
  static constexpr int kBarBytes = 16 * 8;
  static constexpr int kUsed = 5 * kTile + kBarBytes + 1024;
  // At least 116 KB so that two CTAs never share an SM (each holds all 512
  // TMEM columns).
  static constexpr int kSmem = kUsed > 116 * 1024 ? kUsed : 116 * 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm, uint16_t* __restrict__ out,
                       float* __restrict__ lse, int s, int H, int* status) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sK[2] = {smem + C::kTile, smem + 2 * C::kTile};
  uint8_t* sV[2] = {smem + 3 * C::kTile, smem + 4 * C::kTile};
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 5 * C::kTile);
  uint64_t* q_full = bars + 0;
  uint64_t* kv_full = bars + 1;   // [2]
  uint64_t* kv_empty = bars + 3;  // [2]
  uint64_t* s_full = bars + 5;    // [2]
  uint64_t* p_full = bars + 7;    // [2]
  uint64_t* o_ready = bars + 9;
  uint64_t* drain = bars + 10;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 11);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int a = H * D;
  const int q_blk = gridDim.x - 1 - blockIdx.x;
  const int hh = blockIdx.y, bi = blockIdx.z;
  const int q0 = q_blk * BQ;
  const int n_kb = (min(q0 + BQ, s) + BKV - 1) / BKV;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
    }
    mbar_init(o_ready, 1);
    mbar_init(drain, 1);
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
  const uint32_t tS[2] = {tmem + C::kColS0, tmem + C::kColS1};
  const uint32_t tO = tmem + C::kColO;

  if (warp == 0) {
    if (lane == 0) {
      // -------------------------------------------------------- producer
      mbar_arrive_expect_tx(q_full, C::kTile);
      for (int c = 0; c < C::kChunks; ++c)
        tma_load_3d(sQ + c * 16384, &tm, q_full, hh * D + c * 64, q0, bi);
      int issued = 0;
      for (int j = 0; j < n_kb; ++j) {
        const int st = j & 1;
        if (!mbar_wait(&kv_empty[st], ((j >> 1) & 1) ^ 1u, status, kSiteAttention)) break;
        mbar_arrive_expect_tx(&kv_full[st], 2 * C::kTile);
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_3d(sK[st] + c * 16384, &tm, &kv_full[st], a + hh * D + c * 64, j * BKV, bi);
          tma_load_3d(sV[st] + c * 16384, &tm, &kv_full[st], 2 * a + hh * D + c * 64, j * BKV, bi);
        }
        ++issued;
      }
      // Copies still in flight must land before the CTA exits.
      mbar_wait(q_full, 0, status, kSiteAttention, 200000000ull, false);
      for (int j = issued - 1; j >= 0 && j >= issued - 2; --j)
        mbar_wait(&kv_full[j & 1], (j >> 1) & 1, status, kSiteAttention, 200000000ull, false);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // -------------------------------------------------------- MMA issuer
      constexpr uint32_t kIdescQK = idesc_bf16_f32(128, BKV, false, false);
      constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, false, true);
      bool ok = mbar_wait(q_full, 0, status, kSiteAttention);
      const uint32_t q_base = smem_u32(sQ);
      for (int j = 0; ok && j <= n_kb; ++j) {
        if (j < n_kb) {
          const int st = j & 1;
          if (!mbar_wait(&kv_full[st], (j >> 1) & 1, status, kSiteAttention)) break;
          // S buffer st was last read (as P) by PV_{j-2}.
          if (j >= 2 && !mbar_wait(o_ready, (j - 2) & 1, status, kSiteAttention)) break;
          tc_fence_after();
          const uint32_t k_base = smem_u32(sK[st]);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            umma_bf16(tS[st], smem_desc_sw128(q_base + off, 16, 1024),
                      smem_desc_sw128(k_base + off, 16, 1024), kIdescQK, kk > 0 ? 1u : 0u);
          }
          umma_commit(&s_full[st]);
        }
        if (j >= 1) {
          const int pj = j - 1, pst = pj & 1;
          if (!mbar_wait(&p_full[pst], (pj >> 1) & 1, status, kSiteAttention)) break;
          tc_fence_after();
          const uint32_t v_base = smem_u32(sV[pst]);
#pragma unroll
          for (int kk = 0; kk < BKV / 16; ++kk) {
            // P: 16 keys = 8 packed columns; V (MN-major): 16 key rows of 128 B,
            // 64-wide d chunks 16 KB apart.
            umma_bf16_ts(tO, tS[pst] + kk * 8,
                         smem_desc_sw128(v_base + kk * 2048, 16384, 1024), kIdescPV,
                         (pj > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&kv_empty[pst]);
          umma_commit(o_ready);
        }
      }
      umma_commit(drain);
      mbar_wait(drain, 0, status, kSiteAttention, 200000000ull, false);
    }
  } else {
    // ---------------------------------------------------------- softmax
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int q = q0 + row;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float scale = rsqrtf(static_cast<float>(D)) * kLog2e;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kb; ++j) {
      const int st = j & 1;
      if (!mbar_wait(&s_full[st], (j >> 1) & 1, status, kSiteAttention)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float x[BKV];
#pragma unroll
      for (int c = 0; c < BKV / 32; ++c) {
        float v[32];
        tmem_ld_32x32b_x32(tS[st] + lane_off + c * 32, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) x[c * 32 + i] = v[i];
      }
      const int key0 = j * BKV;
      const bool need_mask = key0 + BKV - 1 > q0 || key0 + BKV > s;
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < BKV; ++i) {
        float v = x[i] * scale;
        if (need_mask && (key0 + i > q || key0 + i >= s)) v = -INFINITY;
        x[i] = v;
        mx = fmaxf(mx, v);
      }
      const float m_new = fmaxf(m, mx);
      const bool need = j > 0 && m_new > m + kRescaleThreshold;
      if (j == 0) m = m_new;  // key 0 is visible to every row: m is finite
      if (__any_sync(0xffffffffu, need)) {
        const float alpha = need ? exp2f(m - m_new) : 1.f;
        if (!mbar_wait(o_ready, (j - 1) & 1, status, kSiteAttention)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float v[32];
          tmem_ld_32x32b_x32(tO + lane_off + c * 32, v);
          uint32_t w[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(v[i] * alpha);
          tmem_st_32x32b_x32(tO + lane_off + c * 32, w);
        }
        tmem_st_wait();
        if (need) {
          l *= alpha;
          m = m_new;
        }
      }
      uint32_t pk[BKV / 2];
      float sum = 0.f;
#pragma unroll
      for (int i = 0; i < BKV / 2; ++i) {
        const float p0 = exp2f(x[2 * i] - m);
        const float p1 = exp2f(x[2 * i + 1] - m);
        sum += p0 + p1;
        pk[i] = pack_bf16x2(p0, p1);
      }
      l += sum;
#pragma unroll
      for (int c = 0; c < BKV / 64; ++c) {
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = pk[c * 32 + i];
        tmem_st_32x32b_x32(tS[st] + lane_off + c * 32, w);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_full[st]);
    }
    if (ok && mbar_wait(o_ready, (n_kb - 1) & 1, status, kSiteAttention)) {
      tc_fence_after();
      const float inv = 1.f / l;
      uint16_t* orow = out + (static_cast<int64_t>(bi) * s + q) * a + hh * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        float v[32];
        tmem_ld_32x32b_x32(tO + lane_off + c * 32, v);
        if (q < s) {
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
      if (q < s) lse[(static_cast<int64_t>(bi) * H + hh) * s + q] = (m + log2f(l)) * kLn2;
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
int launch_fwd_tc(const uint16_t* qkv, uint16_t* o, float* lse, int b, int s, int H, int* status,
                  cudaStream_t st) {
  using C = FwdCfg<D>;
  const uint64_t a3 = 3ull * H * D;
  CUtensorMap tm;
  const uint64_t dims[3] = {a3, static_cast<uint64_t>(s), static_cast<uint64_t>(b)};
  const uint64_t strides[2] = {a3 * 2, a3 * 2 * static_cast<uint64_t>(s)};
  const uint32_t box[3] = {64, 128, 1};
  if (!make_tmap_bf16(&tm, qkv, 3, dims, strides, box)) return MC_ERR_CUDA;
  auto kern = attn_fwd_tc_kernel<D>;
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [&] {
    attr = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  });
  if (attr != cudaSuccess) return MC_ERR_CUDA;
  dim3 grid((s + BQ - 1) / BQ, H, b);
  kern<<<grid, kThreads, C::kSmem, st>>>(tm, o, lse, s, H, status);
  return cudaGetLastError() == cudaSuccess ? MC_OK : MC_ERR_CUDA;
}

}  // namespace

int launch_attention_forward_tc(const uint16_t* qkv, uint16_t* o, float* lse, int b, int s, int H,
                                int d, int* status, cudaStream_t st) {
  return d == 64 ? launch_fwd_tc<64>(qkv, o, lse, b, s, H, status, st)
                 : launch_fwd_tc<128>(qkv, o, lse, b, s, H, status, st);
}

}  // namespace mc
