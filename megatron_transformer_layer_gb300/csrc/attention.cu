// Causal flash attention backward for head_dim 64 and 128 (the forward is
// the tcgen05 kernel in attention_tc.cu; this file also holds the launcher
// entry points and the allocation-free variant).
//
// Layout: qkv [T, 3a] bf16 (token-major; Q | K | V blocks, head k at columns
// k*d of its block), o / dO [T, a] bf16, lse / delta [b, H, s] fp32.
// Key/query blocks of 64 are streamed through double-buffered, XOR-swizzled
// shared memory with cp.async; products run on mma.sync m16n8k16
// (bf16 -> fp32) with exp2 and the log2(e)/sqrt(d) scale folded in.
//
// Backward (recompute P from the saved log-sum-exp):
//   pre:   delta_i = sum_c dO_ic O_ic
//   dq:    per query block:  S = Q K^T, P, dP = dO V^T, dS = P (dP - delta),
//          dQ += dS K
//   dkdv:  per key block:    S^T = K Q^T, P^T, dV += P^T dO,
//          dP^T = V dO^T, dS^T = P^T (dP^T - delta), dK += dS^T Q
// Two passes keep every accumulator in registers and avoid atomics; the price
// is recomputing S and dP once more in the dq pass.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "mc_layer_internal.h"
#include "ptx.cuh"

namespace mc {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------- helpers
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;  // 0 => zero fill
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D (16x8 fp32) += A (16x16 bf16, row) * B (16x8 bf16, col)
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of element (row, col) in a [rows][D] bf16 tile whose 16-byte
// chunks are XOR-swizzled by (row & 7).
template <int D>
__device__ __forceinline__ uint32_t swz(int row, int col) {
  const int chunk = (col >> 3) ^ (row & 7);
  return static_cast<uint32_t>(row * D * 2 + chunk * 16 + (col & 7) * 2);
}

// Copies rows [r0, r0 + ROWS) of a head's D columns (global row stride ld
// elements, base already offset to the head's first column) into a swizzled
// smem tile; rows >= nrows are zero-filled.
template <int D, int ROWS, int THREADS>
__device__ __forceinline__ void load_tile(uint32_t s_base, const uint16_t* g_base, int64_t ld,
                                          int r0, int nrows) {
  constexpr int CH = D / 8;  // 16-byte chunks per row
  for (int i = threadIdx.x; i < ROWS * CH; i += THREADS) {
    const int r = i / CH, c = i % CH;
    const int gr = r0 + r;
    const bool valid = gr < nrows;
    const uint16_t* src = g_base + static_cast<int64_t>(valid ? gr : 0) * ld + c * 8;
    cp_async16(s_base + swz<D>(r, c * 8), src, valid);
  }
}

// A fragments (16 rows x D) of a swizzled tile, rows [row0, row0 + 16).
template <int D>
__device__ __forceinline__ void load_a_frags(uint32_t s_base, int row0, uint32_t (&f)[D / 16][4]) {
  const int l = threadIdx.x & 31;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk)
    ldsm_x4(s_base + swz<D>(row0 + (l & 15), kk * 16 + (l >> 4) * 8), f[kk][0], f[kk][1], f[kk][2],
            f[kk][3]);
}

// B fragments for two n8 blocks [n0, n0 + 16) at k-step kk, from a tile stored
// [n][k] (rows = n): b[0..1] for n-block n0, b[2..3] for n0 + 8.
template <int D>
__device__ __forceinline__ void load_b_nk(uint32_t s_base, int n0, int kk, uint32_t (&b)[4]) {
  const int l = threadIdx.x & 31;
  ldsm_x4(s_base + swz<D>(n0 + (l & 7) + ((l >> 4) << 3), kk * 16 + ((l >> 3) & 1) * 8), b[0],
          b[1], b[2], b[3]);
}

// B fragments for two n8 blocks [n0, n0 + 16) at k-step kk, from a tile stored
// [k][n] (rows = k), via ldmatrix.trans.
template <int D>
__device__ __forceinline__ void load_b_kn(uint32_t s_base, int k0, int n0, uint32_t (&b)[4]) {
  const int l = threadIdx.x & 31;
  ldsm_x4_t(s_base + swz<D>(k0 + (l & 7) + ((l >> 3) & 1) * 8, n0 + (l >> 4) * 8), b[0], b[1],
            b[2], b[3]);
}

// A fragment (16 x 16) from two adjacent 16x8 fp32 accumulator blocks.
__device__ __forceinline__ void c_to_a(const float (&c0)[4], const float (&c1)[4],
                                       uint32_t (&a)[4]) {
  a[0] = pack_bf16x2(c0[0], c0[1]);
  a[1] = pack_bf16x2(c0[2], c0[3]);
  a[2] = pack_bf16x2(c1[0], c1[1]);
  a[3] = pack_bf16x2(c1[2], c1[3]);
}

// ---------------------------------------------------------------- backward
constexpr int kBwdB = 64, kBwdThreads = 128;

// delta[b, h, i] = sum_c dO[i, h*D + c] * O[i, h*D + c]; one warp per (token, head).
template <int D>
__global__ void attn_bwd_pre_kernel(const uint16_t* __restrict__ o, const uint16_t* __restrict__ dout,
                                    float* __restrict__ delta, int64_t T, int s, int H) {
  const int64_t wid = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
  const int l = threadIdx.x & 31;
  if (wid >= T * H) return;
  const int64_t tok = wid / H;
  const int hh = static_cast<int>(wid % H);
  const int a = H * D;
  constexpr int PER = D / 32;  // 2 or 4 elements per lane
  const uint16_t* po = o + tok * a + hh * D + l * PER;
  const uint16_t* pd = dout + tok * a + hh * D + l * PER;
  float acc = 0.f;
  if constexpr (PER == 4) {
    const uint2 x = *reinterpret_cast<const uint2*>(po), y = *reinterpret_cast<const uint2*>(pd);
    acc = bf16_lo(x.x) * bf16_lo(y.x) + bf16_hi(x.x) * bf16_hi(y.x) + bf16_lo(x.y) * bf16_lo(y.y) +
          bf16_hi(x.y) * bf16_hi(y.y);
  } else {
    const uint32_t x = *reinterpret_cast<const uint32_t*>(po), y = *reinterpret_cast<const uint32_t*>(pd);
    acc = bf16_lo(x) * bf16_lo(y) + bf16_hi(x) * bf16_hi(y);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (l == 0) {
    const int64_t bi = tok / s, i = tok % s;
    delta[(bi * H + hh) * s + i] = acc;
  }
}

// dQ for one 64-row query block (4 warps x 16 rows).
template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_dq_kernel(const uint16_t* __restrict__ qkv, const uint16_t* __restrict__ dout,
                       const float* __restrict__ lse, const float* __restrict__ delta,
                       uint16_t* __restrict__ dqkv, int s, int H) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr uint32_t kTile = kBwdB * D * 2;
  const uint32_t sQ = smem_u32(smem), sdO = sQ + kTile, sK0 = sdO + kTile, sV0 = sK0 + 2 * kTile;

  const int a = H * D;
  const int64_t ld = 3 * static_cast<int64_t>(a);
  const int q_blk = gridDim.x - 1 - blockIdx.x;
  const int hh = blockIdx.y, bi = blockIdx.z;
  const int q0 = q_blk * kBwdB;
  const uint16_t* base = qkv + static_cast<int64_t>(bi) * s * ld;
  const uint16_t* gQ = base + hh * D;
  const uint16_t* gK = base + a + hh * D;
  const uint16_t* gV = base + 2 * a + hh * D;
  const uint16_t* gdO = dout + static_cast<int64_t>(bi) * s * a + hh * D;
  const int warp = threadIdx.x >> 5, l = threadIdx.x & 31;
  const int g = l >> 2, t = l & 3;
  const int row_a = q0 + warp * 16 + g, row_b = row_a + 8;

  const float* L = lse + (static_cast<int64_t>(bi) * H + hh) * s;
  const float* Dl = delta + (static_cast<int64_t>(bi) * H + hh) * s;
  const float lse2_a = row_a < s ? L[row_a] * kLog2e : 0.f;
  const float lse2_b = row_b < s ? L[row_b] * kLog2e : 0.f;
  const float del_a = row_a < s ? Dl[row_a] : 0.f;
  const float del_b = row_b < s ? Dl[row_b] : 0.f;

  const int kv_end = min(q0 + kBwdB, s);
  const int n_kb = (kv_end + kBwdB - 1) / kBwdB;

  load_tile<D, kBwdB, kBwdThreads>(sQ, gQ, ld, q0, s);
  load_tile<D, kBwdB, kBwdThreads>(sdO, gdO, a, q0, s);
  load_tile<D, kBwdB, kBwdThreads>(sK0, gK, ld, 0, s);
  load_tile<D, kBwdB, kBwdThreads>(sV0, gV, ld, 0, s);
  cp_async_commit();

  const float scale = rsqrtf(static_cast<float>(D));
  const float scale2 = scale * kLog2e;
  uint32_t qf[D / 16][4], df[D / 16][4];
  float dq[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) dq[i][0] = dq[i][1] = dq[i][2] = dq[i][3] = 0.f;

  for (int kb = 0; kb < n_kb; ++kb) {
    const int buf = kb & 1;
    if (kb + 1 < n_kb) {
      load_tile<D, kBwdB, kBwdThreads>(sK0 + (buf ^ 1) * kTile, gK, ld, (kb + 1) * kBwdB, s);
      load_tile<D, kBwdB, kBwdThreads>(sV0 + (buf ^ 1) * kTile, gV, ld, (kb + 1) * kBwdB, s);
    }
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    if (kb == 0) {
      load_a_frags<D>(sQ, warp * 16, qf);
      load_a_frags<D>(sdO, warp * 16, df);
    }
    const uint32_t sK = sK0 + buf * kTile, sV = sV0 + buf * kTile;
    float sc[kBwdB / 8][4], dp[kBwdB / 8][4];
#pragma unroll
    for (int i = 0; i < kBwdB / 8; ++i) {
      sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
      dp[i][0] = dp[i][1] = dp[i][2] = dp[i][3] = 0.f;
    }
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
      for (int nb = 0; nb < kBwdB / 16; ++nb) {
        uint32_t b[4];
        load_b_nk<D>(sK, nb * 16, kk, b);
        mma16816(sc[2 * nb], qf[kk], b[0], b[1]);
        mma16816(sc[2 * nb + 1], qf[kk], b[2], b[3]);
        load_b_nk<D>(sV, nb * 16, kk, b);
        mma16816(dp[2 * nb], df[kk], b[0], b[1]);
        mma16816(dp[2 * nb + 1], df[kk], b[2], b[3]);
      }
    }
    const int key0 = kb * kBwdB;
#pragma unroll
    for (int i = 0; i < kBwdB / 8; ++i) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int key = key0 + i * 8 + 2 * t + (j & 1);
        const int row = j < 2 ? row_a : row_b;
        const float p = (key > row || key >= s)
                            ? 0.f
                            : exp2f(sc[i][j] * scale2 - (j < 2 ? lse2_a : lse2_b));
        sc[i][j] = p * (dp[i][j] - (j < 2 ? del_a : del_b));  // dS
      }
    }
#pragma unroll
    for (int kk = 0; kk < kBwdB / 16; ++kk) {
      uint32_t da[4];
      c_to_a(sc[2 * kk], sc[2 * kk + 1], da);
#pragma unroll
      for (int nb = 0; nb < D / 16; ++nb) {
        uint32_t b[4];
        load_b_kn<D>(sK, kk * 16, nb * 16, b);
        mma16816(dq[2 * nb], da, b[0], b[1]);
        mma16816(dq[2 * nb + 1], da, b[2], b[3]);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();
  __syncthreads();

  // Stage dQ (scaled) through sQ and write the Q block of dqkv.
  uint8_t* sq = smem;
#pragma unroll
  for (int i = 0; i < D / 8; ++i) {
    const int col = i * 8 + 2 * t;
    *reinterpret_cast<uint32_t*>(sq + swz<D>(warp * 16 + g, col)) =
        pack_bf16x2(dq[i][0] * scale, dq[i][1] * scale);
    *reinterpret_cast<uint32_t*>(sq + swz<D>(warp * 16 + g + 8, col)) =
        pack_bf16x2(dq[i][2] * scale, dq[i][3] * scale);
  }
  __syncwarp();
  uint16_t* gdQ = dqkv + static_cast<int64_t>(bi) * s * ld + hh * D;
  constexpr int CH = D / 8;
  for (int i = l; i < 16 * CH; i += 32) {
    const int r = i / CH, c = i % CH;
    const int row = q0 + warp * 16 + r;
    if (row < s)
      *reinterpret_cast<uint4*>(gdQ + static_cast<int64_t>(row) * ld + c * 8) =
          *reinterpret_cast<const uint4*>(sq + swz<D>(warp * 16 + r, c * 8));
  }
}

// dK, dV for one 64-key block (4 warps x 16 keys).
template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_dkdv_kernel(const uint16_t* __restrict__ qkv, const uint16_t* __restrict__ dout,
                         const float* __restrict__ lse, const float* __restrict__ delta,
                         uint16_t* __restrict__ dqkv, int s, int H) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr uint32_t kTile = kBwdB * D * 2;
  const uint32_t sK = smem_u32(smem), sV = sK + kTile, sQ0 = sV + kTile, sdO0 = sQ0 + 2 * kTile;
  float* sL = reinterpret_cast<float*>(smem + 6 * kTile);  // [2][kBwdB] lse * log2e
  float* sD = sL + 2 * kBwdB;                               // [2][kBwdB] delta

  const int a = H * D;
  const int64_t ld = 3 * static_cast<int64_t>(a);
  const int k_blk = blockIdx.x;  // low key blocks see the most queries: first
  const int hh = blockIdx.y, bi = blockIdx.z;
  const int k0 = k_blk * kBwdB;
  const uint16_t* base = qkv + static_cast<int64_t>(bi) * s * ld;
  const uint16_t* gQ = base + hh * D;
  const uint16_t* gK = base + a + hh * D;
  const uint16_t* gV = base + 2 * a + hh * D;
  const uint16_t* gdO = dout + static_cast<int64_t>(bi) * s * a + hh * D;
  const float* L = lse + (static_cast<int64_t>(bi) * H + hh) * s;
  const float* Dl = delta + (static_cast<int64_t>(bi) * H + hh) * s;
  const int warp = threadIdx.x >> 5, l = threadIdx.x & 31;
  const int g = l >> 2, t = l & 3;
  const int key_a = k0 + warp * 16 + g, key_b = key_a + 8;

  const int qb_first = k0 / kBwdB;
  const int n_qb = (s + kBwdB - 1) / kBwdB;

  auto load_q_block = [&](int qb, int buf) {
    load_tile<D, kBwdB, kBwdThreads>(sQ0 + buf * kTile, gQ, ld, qb * kBwdB, s);
    load_tile<D, kBwdB, kBwdThreads>(sdO0 + buf * kTile, gdO, a, qb * kBwdB, s);
    for (int i = threadIdx.x; i < kBwdB; i += kBwdThreads) {
      const int q = qb * kBwdB + i;
      sL[buf * kBwdB + i] = q < s ? L[q] * kLog2e : 0.f;
      sD[buf * kBwdB + i] = q < s ? Dl[q] : 0.f;
    }
  };

  load_tile<D, kBwdB, kBwdThreads>(sK, gK, ld, k0, s);
  load_tile<D, kBwdB, kBwdThreads>(sV, gV, ld, k0, s);
  load_q_block(qb_first, 0);
  cp_async_commit();

  const float scale = rsqrtf(static_cast<float>(D));
  const float scale2 = scale * kLog2e;
  float dk[D / 8][4], dv[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) {
    dk[i][0] = dk[i][1] = dk[i][2] = dk[i][3] = 0.f;
    dv[i][0] = dv[i][1] = dv[i][2] = dv[i][3] = 0.f;
  }

  for (int qb = qb_first; qb < n_qb; ++qb) {
    const int buf = (qb - qb_first) & 1;
    if (qb + 1 < n_qb) load_q_block(qb + 1, buf ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const uint32_t sQ = sQ0 + buf * kTile, sdO = sdO0 + buf * kTile;
    const float* bl = sL + buf * kBwdB;
    const float* bd = sD + buf * kBwdB;

    float st[kBwdB / 8][4], dpt[kBwdB / 8][4];
#pragma unroll
    for (int i = 0; i < kBwdB / 8; ++i) {
      st[i][0] = st[i][1] = st[i][2] = st[i][3] = 0.f;
      dpt[i][0] = dpt[i][1] = dpt[i][2] = dpt[i][3] = 0.f;
    }
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t ka[4], va[4];
      {
        const int l2 = threadIdx.x & 31;
        ldsm_x4(sK + swz<D>(warp * 16 + (l2 & 15), kk * 16 + (l2 >> 4) * 8), ka[0], ka[1], ka[2], ka[3]);
        ldsm_x4(sV + swz<D>(warp * 16 + (l2 & 15), kk * 16 + (l2 >> 4) * 8), va[0], va[1], va[2], va[3]);
      }
#pragma unroll
      for (int nb = 0; nb < kBwdB / 16; ++nb) {
        uint32_t b[4];
        load_b_nk<D>(sQ, nb * 16, kk, b);
        mma16816(st[2 * nb], ka, b[0], b[1]);
        mma16816(st[2 * nb + 1], ka, b[2], b[3]);
        load_b_nk<D>(sdO, nb * 16, kk, b);
        mma16816(dpt[2 * nb], va, b[0], b[1]);
        mma16816(dpt[2 * nb + 1], va, b[2], b[3]);
      }
    }
    const int q_base = qb * kBwdB;
    // P^T and dS^T; columns are queries.
#pragma unroll
    for (int i = 0; i < kBwdB / 8; ++i) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int qc = i * 8 + 2 * t + (j & 1);
        const int q = q_base + qc;
        const int key = j < 2 ? key_a : key_b;
        const float p = (q < key || q >= s) ? 0.f : exp2f(st[i][j] * scale2 - bl[qc]);
        st[i][j] = p;
        dpt[i][j] = p * (dpt[i][j] - bd[qc]);
      }
    }
#pragma unroll
    for (int kk = 0; kk < kBwdB / 16; ++kk) {
      uint32_t pa[4], da[4];
      c_to_a(st[2 * kk], st[2 * kk + 1], pa);
      c_to_a(dpt[2 * kk], dpt[2 * kk + 1], da);
#pragma unroll
      for (int nb = 0; nb < D / 16; ++nb) {
        uint32_t b[4];
        load_b_kn<D>(sdO, kk * 16, nb * 16, b);
        mma16816(dv[2 * nb], pa, b[0], b[1]);
        mma16816(dv[2 * nb + 1], pa, b[2], b[3]);
        load_b_kn<D>(sQ, kk * 16, nb * 16, b);
        mma16816(dk[2 * nb], da, b[0], b[1]);
        mma16816(dk[2 * nb + 1], da, b[2], b[3]);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();
  __syncthreads();

  // Stage dK (scaled) in sK and dV in sV, then write the K and V blocks.
  uint8_t* sk = smem;
  uint8_t* sv = smem + kTile;
#pragma unroll
  for (int i = 0; i < D / 8; ++i) {
    const int col = i * 8 + 2 * t;
    *reinterpret_cast<uint32_t*>(sk + swz<D>(warp * 16 + g, col)) =
        pack_bf16x2(dk[i][0] * scale, dk[i][1] * scale);
    *reinterpret_cast<uint32_t*>(sk + swz<D>(warp * 16 + g + 8, col)) =
        pack_bf16x2(dk[i][2] * scale, dk[i][3] * scale);
    *reinterpret_cast<uint32_t*>(sv + swz<D>(warp * 16 + g, col)) = pack_bf16x2(dv[i][0], dv[i][1]);
    *reinterpret_cast<uint32_t*>(sv + swz<D>(warp * 16 + g + 8, col)) =
        pack_bf16x2(dv[i][2], dv[i][3]);
  }
  __syncwarp();
  uint16_t* gdK = dqkv + static_cast<int64_t>(bi) * s * ld + a + hh * D;
  uint16_t* gdV = gdK + a;
  constexpr int CH = D / 8;
  for (int i = l; i < 16 * CH; i += 32) {
    const int r = i / CH, c = i % CH;
    const int key = k0 + warp * 16 + r;
    if (key < s) {
      *reinterpret_cast<uint4*>(gdK + static_cast<int64_t>(key) * ld + c * 8) =
          *reinterpret_cast<const uint4*>(sk + swz<D>(warp * 16 + r, c * 8));
      *reinterpret_cast<uint4*>(gdV + static_cast<int64_t>(key) * ld + c * 8) =
          *reinterpret_cast<const uint4*>(sv + swz<D>(warp * 16 + r, c * 8));
    }
  }
}

template <typename K>
bool set_smem(K kern, int bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) ==
         cudaSuccess;
}

template <int D>
int bwd_launch(const uint16_t* qkv, const uint16_t* o, const float* lse, const uint16_t* dout,
               uint16_t* dqkv, float* delta, int b, int s, int H, cudaStream_t st) {
  const int64_t T = static_cast<int64_t>(b) * s;
  const int64_t warps = T * H;
  attn_bwd_pre_kernel<D><<<static_cast<unsigned>((warps * 32 + 255) / 256), 256, 0, st>>>(
      o, dout, delta, T, s, H);
  if (cudaGetLastError() != cudaSuccess) return MC_ERR_CUDA;
  const int tile = kBwdB * D * 2;
  const int smem_dq = 6 * tile;
  const int smem_kv = 6 * tile + 4 * kBwdB * 4;
  if (!set_smem(attn_bwd_dq_kernel<D>, smem_dq) || !set_smem(attn_bwd_dkdv_kernel<D>, smem_kv))
    return MC_ERR_CUDA;
  dim3 grid((s + kBwdB - 1) / kBwdB, H, b);
  attn_bwd_dkdv_kernel<D><<<grid, kBwdThreads, smem_kv, st>>>(qkv, dout, lse, delta, dqkv, s, H);
  if (cudaGetLastError() != cudaSuccess) return MC_ERR_CUDA;
  attn_bwd_dq_kernel<D><<<grid, kBwdThreads, smem_dq, st>>>(qkv, dout, lse, delta, dqkv, s, H);
  return cudaGetLastError() == cudaSuccess ? MC_OK : MC_ERR_CUDA;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

int launch_attention_forward(const uint16_t* qkv, uint16_t* o, float* lse, int b, int s, int H,
                             int d, int* status, cudaStream_t st) {
  (void)status;
  if (b < 1 || s < 1 || H < 1) return MC_ERR_SHAPE;
  if (d != 64 && d != 128) return MC_ERR_UNSUPPORTED;
  if (H > 65535 || b > 65535) return MC_ERR_UNSUPPORTED;
  if (!qkv || !o || !lse) return MC_ERR_NULLPTR;
  if (!al16(qkv) || !al16(o)) return MC_ERR_ALIGN;
  return launch_attention_forward_tc(qkv, o, lse, b, s, H, d, status, st);
}

int launch_attention_backward(const uint16_t* qkv, const uint16_t* o, const float* lse,
                              const uint16_t* dout, uint16_t* dqkv, float* delta, int b, int s,
                              int H, int d, int* status, cudaStream_t st) {
  (void)status;
  if (b < 1 || s < 1 || H < 1) return MC_ERR_SHAPE;
  if (d != 64 && d != 128) return MC_ERR_UNSUPPORTED;
  if (H > 65535 || b > 65535) return MC_ERR_UNSUPPORTED;
  if (!qkv || !o || !lse || !dout || !dqkv || !delta) return MC_ERR_NULLPTR;
  if (!al16(qkv) || !al16(o) || !al16(dout) || !al16(dqkv)) return MC_ERR_ALIGN;
  return d == 64 ? bwd_launch<64>(qkv, o, lse, dout, dqkv, delta, b, s, H, st)
                 : bwd_launch<128>(qkv, o, lse, dout, dqkv, delta, b, s, H, st);
}

// ---------------------------------------------------------------- no-alloc
// Fixed device scratch of the allocation-free attention backward: the
// delta = rowsum(dO * O) vector, kNoAllocDeltaFloats floats (4 MiB), enough
// for micro_batch * heads * seq_len <= 1,048,576.  It lives in this module's
// global memory on every device that loads the library, until the process
// exits.  All calls share it (it keeps the last call's values); the backward
// overwrites every element it reads, so nothing has to be cleared.  Calls
// whose kernels overlap on the GPU (different streams) race on it.
namespace {
constexpr int64_t kNoAllocDeltaFloats = int64_t(1) << 20;
__device__ __align__(256) float g_noalloc_delta[kNoAllocDeltaFloats];

std::mutex g_noalloc_mu;
std::vector<float*> g_noalloc_ptr;  // per device ordinal

// Device address of g_noalloc_delta on the current device; looked up once per
// device (the symbol's host-side name is only a stand-in, not an address).
int noalloc_scratch(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MC_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (static_cast<int>(g_noalloc_ptr.size()) <= dev) g_noalloc_ptr.resize(dev + 1, nullptr);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_delta) != cudaSuccess || !p) return MC_ERR_CUDA;
    g_noalloc_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return MC_OK;
}
}  // namespace

}  // namespace mc

extern "C" int mc_attention_backward_noalloc(const uint16_t* qkv, const uint16_t* o,
                                             const float* lse, const uint16_t* dout,
                                             uint16_t* dqkv, int32_t micro_batch,
                                             int32_t seq_len, int32_t heads, int32_t head_dim,
                                             int* status, void* stream) {
  if (micro_batch < 1 || seq_len < 1 || heads < 1) return MC_ERR_SHAPE;
  if (static_cast<int64_t>(micro_batch) * heads * seq_len > mc::kNoAllocDeltaFloats)
    return MC_ERR_SCRATCH_LIMIT;
  float* delta = nullptr;
  const int rc = mc::noalloc_scratch(&delta);
  if (rc != MC_OK) return rc;
  return mc::launch_attention_backward(qkv, o, lse, dout, dqkv, delta, micro_batch, seq_len, heads,
                                       head_dim, status, static_cast<cudaStream_t>(stream));
}
