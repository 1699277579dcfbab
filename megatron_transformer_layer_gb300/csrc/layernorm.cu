// LayerNorm forward/backward and column sums (bias gradients).
//
// These kernels are HBM-bound: every row is read with 128-bit loads (float4 of
// fp32, 4 x bf16 of gamma/beta), reduced with warp shuffles plus one
// cross-warp step in shared memory, and written once.  Column sums over rows
// (dgamma, dbeta, bias gradients) are accumulated per CTA and reduced by a
// second, deterministic pass -- no floating-point atomics.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "mc_layer_internal.h"
#include "ptx.cuh"

namespace mc {
namespace {

constexpr float kLnEps = 1e-5f;
constexpr int kLnThreads = 128;     // forward: one CTA per row
constexpr int kLnBwdThreads = 256;  // backward: grid-strided rows

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum over the block (THREADS threads); `red` has 2 * (THREADS/32) floats.
template <int THREADS = kLnThreads>
__device__ __forceinline__ float2 block_sum2(float a, float b, float* red) {
  a = warp_sum(a);
  b = warp_sum(b);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  constexpr int W = THREADS / 32;
  __syncthreads();  // red may still be read by a previous call
  if (l == 0) {
    red[w] = a;
    red[W + w] = b;
  }
  __syncthreads();
  float2 r = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < W; ++i) {
    r.x += red[i];
    r.y += red[W + i];
  }
  return r;
}

__device__ __forceinline__ float4 load_bf16x4(const uint16_t* p) {
  const uint2 w = *reinterpret_cast<const uint2*>(p);
  return make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
}

__device__ __forceinline__ void store_bf16x4(uint16_t* p, float4 v) {
  uint2 w;
  w.x = pack_bf16x2(v.x, v.y);
  w.y = pack_bf16x2(v.z, v.w);
  *reinterpret_cast<uint2*>(p) = w;
}

// One CTA per row; thread t owns float4 columns t, t + 128, ... (VPT of them).
template <int VPT>
__global__ void __launch_bounds__(kLnThreads) ln_fwd_kernel(const float* __restrict__ x,
                                                            const uint16_t* __restrict__ gamma,
                                                            const uint16_t* __restrict__ beta,
                                                            uint16_t* __restrict__ out,
                                                            float* __restrict__ mean_out,
                                                            float* __restrict__ rstd_out, int h,
                                                            int64_t rows, int* status) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_launch();
  __shared__ float red[2 * kLnThreads / 32];
  const int64_t row = blockIdx.x;
  const int n4 = h >> 2;
  const float4* xr = reinterpret_cast<const float4*>(x + row * h);
  float4 v[VPT];
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int c = threadIdx.x + i * kLnThreads;
    v[i] = c < n4 ? xr[c] : make_float4(0.f, 0.f, 0.f, 0.f);
    s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
  }
  const float mean = block_sum2(s, 0.f, red).x / h;
  float q = 0.f;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int c = threadIdx.x + i * kLnThreads;
    if (c < n4) {
      const float a = v[i].x - mean, b = v[i].y - mean, cc = v[i].z - mean, d = v[i].w - mean;
      q += (a * a + b * b) + (cc * cc + d * d);
    }
  }
  const float var = block_sum2(q, 0.f, red).x / h;
  const float rstd = rsqrtf(var + kLnEps);
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int c = threadIdx.x + i * kLnThreads;
    if (c < n4) {
      const float4 g = load_bf16x4(gamma + 4 * c);
      const float4 b = load_bf16x4(beta + 4 * c);
      float4 o;
      o.x = (v[i].x - mean) * rstd * g.x + b.x;
      o.y = (v[i].y - mean) * rstd * g.y + b.y;
      o.z = (v[i].z - mean) * rstd * g.z + b.z;
      o.w = (v[i].w - mean) * rstd * g.w + b.w;
      if (MC_DCHECK(row < rows && 4 * c + 4 <= h, status, kSiteLayerNorm))
        store_bf16x4(out + row * h + 4 * c, o);
    }
  }
  if (threadIdx.x == 0) {
    if (mean_out) mean_out[row] = mean;
    if (rstd_out) rstd_out[row] = rstd;
  }
}

// Grid-strided over rows.  Per-column partial sums of (dout * xhat, dout, dx)
// for this CTA's rows live in shared memory (3 * h floats; each thread owns
// its columns, so no synchronisation is needed) and are written to
// partials[blockIdx.x][3][h] at the end.  All three input rows (dout, x,
// resid) are requested before the row's reductions so one DRAM round trip
// covers the row.
template <int VPT>
__global__ void __launch_bounds__(kLnBwdThreads) ln_bwd_kernel(
    const float* __restrict__ dout, const float* __restrict__ x, const float* __restrict__ mean,
    const float* __restrict__ rstd, const uint16_t* __restrict__ gamma,
    const float* resid, float* dx, uint16_t* __restrict__ dx_bf16,
    float* __restrict__ partials, int64_t rows, int h, int want_colsum_dx, int* status) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_launch();
  extern __shared__ float colacc[];  // [3][h]
  __shared__ float red[2 * kLnBwdThreads / 32];
  const int n4 = h >> 2;
  float4 gam[VPT];
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int c = threadIdx.x + i * kLnBwdThreads;
    gam[i] = c < n4 ? load_bf16x4(gamma + 4 * c) : make_float4(0.f, 0.f, 0.f, 0.f);
    if (c < n4) {
      reinterpret_cast<float4*>(colacc)[c] = make_float4(0.f, 0.f, 0.f, 0.f);
      reinterpret_cast<float4*>(colacc + h)[c] = make_float4(0.f, 0.f, 0.f, 0.f);
      reinterpret_cast<float4*>(colacc + 2 * h)[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const float mu = mean[row], rs = rstd[row];
    const float4* dr = reinterpret_cast<const float4*>(dout + row * h);
    const float4* xr = reinterpret_cast<const float4*>(x + row * h);
    const float4* rr = resid ? reinterpret_cast<const float4*>(resid + row * h) : nullptr;
    float4 dy[VPT], xh[VPT], rv[VPT];
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int c = threadIdx.x + i * kLnBwdThreads;
      const bool ok = c < n4;
      dy[i] = ok ? dr[c] : make_float4(0.f, 0.f, 0.f, 0.f);
      xh[i] = ok ? xr[c] : make_float4(0.f, 0.f, 0.f, 0.f);
      rv[i] = (ok && rr) ? rr[c] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float s1 = 0.f, s2 = 0.f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      xh[i] = make_float4((xh[i].x - mu) * rs, (xh[i].y - mu) * rs, (xh[i].z - mu) * rs,
                          (xh[i].w - mu) * rs);
      const float4 gg = make_float4(dy[i].x * gam[i].x, dy[i].y * gam[i].y, dy[i].z * gam[i].z,
                                    dy[i].w * gam[i].w);
      s1 += (gg.x + gg.y) + (gg.z + gg.w);
      s2 += (gg.x * xh[i].x + gg.y * xh[i].y) + (gg.z * xh[i].z + gg.w * xh[i].w);
    }
    const float2 r = block_sum2<kLnBwdThreads>(s1, s2, red);
    const float m1 = r.x / h, m2 = r.y / h;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int c = threadIdx.x + i * kLnBwdThreads;
      if (c < n4) {
        const float4 gg = make_float4(dy[i].x * gam[i].x, dy[i].y * gam[i].y, dy[i].z * gam[i].z,
                                      dy[i].w * gam[i].w);
        float4 o;
        o.x = rs * (gg.x - m1 - xh[i].x * m2) + rv[i].x;
        o.y = rs * (gg.y - m1 - xh[i].y * m2) + rv[i].y;
        o.z = rs * (gg.z - m1 - xh[i].z * m2) + rv[i].z;
        o.w = rs * (gg.w - m1 - xh[i].w * m2) + rv[i].w;
        if (MC_DCHECK(row < rows && 4 * c + 4 <= h, status, kSiteLayerNorm)) {
          reinterpret_cast<float4*>(dx + row * h)[c] = o;
          if (dx_bf16) store_bf16x4(dx_bf16 + row * h + 4 * c, o);
        }
        float4* cg = reinterpret_cast<float4*>(colacc) + c;
        float4* cb = reinterpret_cast<float4*>(colacc + h) + c;
        float4 a = *cg, b = *cb;
        a.x += dy[i].x * xh[i].x;
        a.y += dy[i].y * xh[i].y;
        a.z += dy[i].z * xh[i].z;
        a.w += dy[i].w * xh[i].w;
        b.x += dy[i].x;
        b.y += dy[i].y;
        b.z += dy[i].z;
        b.w += dy[i].w;
        *cg = a;
        *cb = b;
        if (want_colsum_dx) {
          float4* cx = reinterpret_cast<float4*>(colacc + 2 * h) + c;
          float4 e = *cx;
          e.x += o.x;
          e.y += o.y;
          e.z += o.z;
          e.w += o.w;
          *cx = e;
        }
      }
    }
  }
  float4* dst = reinterpret_cast<float4*>(partials + static_cast<int64_t>(blockIdx.x) * 3 * h);
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int c = threadIdx.x + i * kLnBwdThreads;
    if (c < n4) {
      dst[c] = reinterpret_cast<float4*>(colacc)[c];
      dst[n4 + c] = reinterpret_cast<float4*>(colacc + h)[c];
      dst[2 * n4 + c] = reinterpret_cast<float4*>(colacc + 2 * h)[c];
    }
  }
}

// out_j[c] = (accumulate ? out_j[c] : 0) + sum_b partials[b][j][c], j < nsum.
// A CTA of 256 threads owns 32 columns of one sum j: thread (c, r) adds the
// partial rows r, r + 8, ... of column c, then the 8 row-group sums are
// combined in a fixed order through shared memory (deterministic).
__global__ void __launch_bounds__(256) reduce_partials_kernel(const float* __restrict__ partials,
                                                              int nblocks, int nsum, int64_t n,
                                                              float* out0, float* out1, float* out2,
                                                              int accumulate) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_launch();
  __shared__ float part[8][33];
  const int cl = threadIdx.x & 31, rg = threadIdx.x >> 5;
  const int64_t c = blockIdx.x * 32 + cl;
  const int j = blockIdx.y;
  float s = 0.f;
  if (c < n && j < nsum)
    for (int b = rg; b < nblocks; b += 8) s += partials[(static_cast<int64_t>(b) * nsum + j) * n + c];
  part[rg][cl] = s;
  __syncthreads();
  if (rg == 0 && c < n && j < nsum) {
    float* out = j == 0 ? out0 : (j == 1 ? out1 : out2);
    if (!out) return;
    float t = 0.f;
#pragma unroll
    for (int r = 0; r < 8; ++r) t += part[r][cl];
    out[c] = accumulate ? out[c] + t : t;
  }
}

// Column partial sums of a [rows, n] matrix over gridDim.y row ranges; a
// thread owns 8 consecutive columns and walks its rows four at a time (four
// loads in flight).  Optionally writes a bf16 copy of an fp32 input.
template <bool IN_BF16>
__global__ void colsum_partial_kernel(const void* __restrict__ in, int64_t rows, int64_t n,
                                      float* __restrict__ partials, uint16_t* __restrict__ copy) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_launch();
  const int64_t c8 = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) * 8;
  if (c8 >= n) return;
  const int split = blockIdx.y;
  const int64_t per = (rows + gridDim.y - 1) / gridDim.y;
  const int64_t r0 = split * per;
  const int64_t r1 = r0 + per < rows ? r0 + per : rows;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
  for (int64_t r = r0; r < r1; ++r) {
    if constexpr (IN_BF16) {
      const uint4 w = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(in) + r * n + c8);
      acc[0] += bf16_lo(w.x);
      acc[1] += bf16_hi(w.x);
      acc[2] += bf16_lo(w.y);
      acc[3] += bf16_hi(w.y);
      acc[4] += bf16_lo(w.z);
      acc[5] += bf16_hi(w.z);
      acc[6] += bf16_lo(w.w);
      acc[7] += bf16_hi(w.w);
    } else {
      const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(in) + r * n + c8);
      const float4 a = p[0], b = p[1];
      acc[0] += a.x;
      acc[1] += a.y;
      acc[2] += a.z;
      acc[3] += a.w;
      acc[4] += b.x;
      acc[5] += b.y;
      acc[6] += b.z;
      acc[7] += b.w;
      if (copy) {
        uint4 w;
        w.x = pack_bf16x2(a.x, a.y);
        w.y = pack_bf16x2(a.z, a.w);
        w.z = pack_bf16x2(b.x, b.y);
        w.w = pack_bf16x2(b.z, b.w);
        *reinterpret_cast<uint4*>(copy + r * n + c8) = w;
      }
    }
  }
  float4* dst = reinterpret_cast<float4*>(partials + split * n + c8);
  dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

template <int VPT>
int ln_fwd_launch(const float* x, const uint16_t* g, const uint16_t* b, uint16_t* out,
                  float* mean, float* rstd, int64_t rows, int h, int* status, cudaStream_t st) {
  launch_kernel(ln_fwd_kernel<VPT>, dim3(static_cast<unsigned>(rows)), dim3(kLnThreads), 0, st, 1,
                x, g, b, out, mean, rstd, h, rows, status);
  return cudaGetLastError() == cudaSuccess ? MC_OK : MC_ERR_CUDA;
}

// Launches the backward over min(rows, kLnBwdMaxBlocks, CTAs resident at once)
// CTAs -- one wave: at large h registers and the [3][h] column partials allow
// only one or two CTAs per SM, and further, partly occupied waves cost more
// than longer row loops -- and returns that count in *grid_out.
template <int VPT>
int ln_bwd_launch(const float* dout, const float* x, const float* mean, const float* rstd,
                  const uint16_t* gamma, const float* resid, float* dx, uint16_t* dx_bf16,
                  float* partials, int64_t rows, int h, int want_colsum_dx, int* grid_out,
                  int* status, cudaStream_t st) {
  const size_t smem = 3 * static_cast<size_t>(h) * sizeof(float);
  auto kern = ln_bwd_kernel<VPT>;
  // Opt in once per device to the largest column-partial buffer (h = kMaxLayerNormHidden);
  // 48 KB of dynamic memory plus the kernel's static reduction buffer already
  // exceeds the default limit at h = 4096.
  static PerDeviceInit init;
  const cudaError_t attr = once_per_device(init, [&](long long*) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                3 * kMaxLayerNormHidden * static_cast<int>(sizeof(float)));
  });
  if (attr != cudaSuccess) return MC_ERR_CUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kLnBwdThreads, smem) !=
          cudaSuccess ||
      per_sm < 1)
    return MC_ERR_CUDA;
  int64_t grid = rows < kLnBwdMaxBlocks ? rows : kLnBwdMaxBlocks;
  const int64_t resident = static_cast<int64_t>(per_sm) * num_sms();
  if (resident > 0 && grid > resident) grid = resident;
  *grid_out = static_cast<int>(grid);
  launch_kernel(kern, dim3(static_cast<unsigned>(grid)), dim3(kLnBwdThreads), smem, st, 1, dout, x,
                mean, rstd, gamma, resid, dx, dx_bf16, partials, rows, h, want_colsum_dx, status);
  return cudaGetLastError() == cudaSuccess ? MC_OK : MC_ERR_CUDA;
}

int vpt_for(int h, int threads = kLnThreads) {
  const int n4 = h / 4;
  int vpt = 1;
  while (vpt * threads < n4) vpt *= 2;
  return vpt;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

int launch_layernorm_forward(const float* x, const uint16_t* gamma, const uint16_t* beta,
                             uint16_t* out, float* mean, float* rstd, int64_t rows, int h,
                             int* status, cudaStream_t st) {
  if (rows < 1 || h < 8 || h % 8 || h > kMaxLayerNormHidden) return MC_ERR_UNSUPPORTED;
  if (rows > 0x7fffffff) return MC_ERR_UNSUPPORTED;
  if (!x || !gamma || !beta || !out) return MC_ERR_NULLPTR;
  if (!al16(x) || !al16(out) || (reinterpret_cast<uintptr_t>(gamma) & 7u) ||
      (reinterpret_cast<uintptr_t>(beta) & 7u))
    return MC_ERR_ALIGN;
  switch (vpt_for(h)) {
    case 1: return ln_fwd_launch<1>(x, gamma, beta, out, mean, rstd, rows, h, status, st);
    case 2: return ln_fwd_launch<2>(x, gamma, beta, out, mean, rstd, rows, h, status, st);
    case 4: return ln_fwd_launch<4>(x, gamma, beta, out, mean, rstd, rows, h, status, st);
    case 8: return ln_fwd_launch<8>(x, gamma, beta, out, mean, rstd, rows, h, status, st);
    case 16: return ln_fwd_launch<16>(x, gamma, beta, out, mean, rstd, rows, h, status, st);
    case 32: return ln_fwd_launch<32>(x, gamma, beta, out, mean, rstd, rows, h, status, st);
    default: return MC_ERR_UNSUPPORTED;
  }
}

size_t layernorm_backward_scratch_floats(int64_t rows, int h) {
  const int64_t grid = rows < kLnBwdMaxBlocks ? rows : kLnBwdMaxBlocks;
  return static_cast<size_t>(grid) * 3 * static_cast<size_t>(h);
}

int launch_layernorm_backward(const float* dout, const float* x, const float* mean,
                              const float* rstd, const uint16_t* gamma, const float* resid,
                              float* dx, uint16_t* dx_bf16, float* dgamma, float* dbeta,
                              float* colsum_dx, int accumulate, float* partials, int64_t rows,
                              int h, int* status, cudaStream_t st) {
  if (rows < 1 || h < 8 || h % 8 || h > kMaxLayerNormHidden) return MC_ERR_UNSUPPORTED;
  if (!dout || !x || !mean || !rstd || !gamma || !dx || !partials || !dgamma || !dbeta)
    return MC_ERR_NULLPTR;
  if (!al16(dout) || !al16(x) || !al16(dx) || !al16(partials) || (resid && !al16(resid)) ||
      (dx_bf16 && (reinterpret_cast<uintptr_t>(dx_bf16) & 7u)) ||
      (reinterpret_cast<uintptr_t>(gamma) & 7u))
    return MC_ERR_ALIGN;
  int grid = 0;  // set by the launch: the CTAs (and partial rows) used
  const int want = colsum_dx != nullptr;
  int rc;
  switch (vpt_for(h, kLnBwdThreads)) {
    case 1: rc = ln_bwd_launch<1>(dout, x, mean, rstd, gamma, resid, dx, dx_bf16, partials, rows, h, want, &grid, status, st); break;
    case 2: rc = ln_bwd_launch<2>(dout, x, mean, rstd, gamma, resid, dx, dx_bf16, partials, rows, h, want, &grid, status, st); break;
    case 4: rc = ln_bwd_launch<4>(dout, x, mean, rstd, gamma, resid, dx, dx_bf16, partials, rows, h, want, &grid, status, st); break;
    case 8: rc = ln_bwd_launch<8>(dout, x, mean, rstd, gamma, resid, dx, dx_bf16, partials, rows, h, want, &grid, status, st); break;
    case 16: rc = ln_bwd_launch<16>(dout, x, mean, rstd, gamma, resid, dx, dx_bf16, partials, rows, h, want, &grid, status, st); break;
    default: return MC_ERR_UNSUPPORTED;
  }
  if (rc != MC_OK) return rc;
  dim3 rgrid(static_cast<unsigned>((h + 31) / 32), want ? 3 : 2);
  launch_kernel(reduce_partials_kernel, dim3(rgrid), dim3(256), 0, st, 1, partials, grid, 3, h,
                dgamma, dbeta, colsum_dx, accumulate);
  return cudaGetLastError() == cudaSuccess ? MC_OK : MC_ERR_CUDA;
}

int launch_colsum(const void* in, bool in_bf16, int64_t rows, int64_t n, float* out,
                  int accumulate, uint16_t* bf16_copy, float* partials, int* status,
                  cudaStream_t st) {
  (void)status;
  if (rows < 1 || n < 8 || n % 8) return MC_ERR_UNSUPPORTED;
  if (!in || !out || !partials) return MC_ERR_NULLPTR;
  if (!al16(in) || !al16(partials) || (bf16_copy && !al16(bf16_copy))) return MC_ERR_ALIGN;
  const int64_t threads_needed = n / 8;
  const int64_t col_blocks = (threads_needed + 127) / 128;
  int64_t want = (4 * static_cast<int64_t>(num_sms()) + col_blocks - 1) / col_blocks;
  want = want < kColsumMinSplits ? kColsumMinSplits : want;
  want = want > kColsumMaxSplits ? kColsumMaxSplits : want;
  const int splits = static_cast<int>(rows < want ? rows : want);
  dim3 grid(static_cast<unsigned>(col_blocks), splits);
  if (in_bf16)
    launch_kernel(colsum_partial_kernel<true>, dim3(grid), dim3(128), 0, st, 1, in, rows, n,
                  partials, nullptr);
  else
    launch_kernel(colsum_partial_kernel<false>, dim3(grid), dim3(128), 0, st, 1, in, rows, n,
                  partials, bf16_copy);
  if (cudaGetLastError() != cudaSuccess) return MC_ERR_CUDA;
  dim3 rgrid(static_cast<unsigned>((n + 31) / 32), 1);
  launch_kernel(reduce_partials_kernel, dim3(rgrid), dim3(256), 0, st, 1, partials, splits, 1, n,
                out, nullptr, nullptr, accumulate);
  return cudaGetLastError() == cudaSuccess ? MC_OK : MC_ERR_CUDA;
}

}  // namespace mc
