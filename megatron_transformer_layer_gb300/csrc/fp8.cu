// Per-tensor current scaling to 8-bit floats for the FP8 GEMM path.
//
// The Megatron-Core listing (混合精度; --fp8-format hybrid: E4M3 forward,
// E5M2 gradients) names the formats and no recipe; the reading taken is the
// plainest one: amax = max |x| (fp32), scale = fmax / amax (fp32 division,
// 1 when amax is 0), q = round-to-nearest-even of x * scale (fp32 product),
// saturated to +-fmax (E4M3: 448, E5M2: 57344), and scale_inv = 1 / scale for
// the GEMM epilogue.
//   amax_partial_kernel  grid-stride |x| maxima (16-byte loads), one per block
//   fp8_scale_kernel     one block: the maximum of the partials, scale, scale_inv
//   fp8_cast_kernel      x * scale -> 8-bit, 8 elements per thread step
// The maximum is order-independent, so the result is deterministic.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "mc_layer_internal.h"
#include "ptx.cuh"

namespace mc {
namespace {

constexpr int kAmaxBlocks = 1024;
constexpr int kThreadsPerBlock = 256;

__device__ __forceinline__ float load_elem(const void* in, bool bf16, int64_t i) {
  return bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(in)[i])
              : static_cast<const float*>(in)[i];
}

// |x| maximum of one 16-byte vector: 8 bf16 or 4 fp32 values.
template <bool BF16>
__device__ __forceinline__ float vec_absmax(uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float m = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if constexpr (BF16) {
      m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[k])), fabsf(bf16_hi(w[k]))));
    } else {
      m = fmaxf(m, fabsf(__uint_as_float(w[k])));
    }
  }
  return m;
}

// Grid-stride |x| maxima, one per block: 16-byte loads, four in flight per
// thread, then the n % (elements per vector) tail element by element.
template <bool BF16>
__global__ void amax_partial_kernel(const void* __restrict__ in, int64_t n,
                                    float* __restrict__ partials) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_launch();
  constexpr int kPerVec = BF16 ? 8 : 4;
  const uint4* __restrict__ vin = static_cast<const uint4*>(in);
  const int64_t nv = n / kPerVec;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  float m = 0.f;
  for (; i + 3 * stride < nv; i += 4 * stride) {
    const uint4 a = __ldg(vin + i), b = __ldg(vin + i + stride), c = __ldg(vin + i + 2 * stride),
                d = __ldg(vin + i + 3 * stride);
    m = fmaxf(m, fmaxf(fmaxf(vec_absmax<BF16>(a), vec_absmax<BF16>(b)),
                       fmaxf(vec_absmax<BF16>(c), vec_absmax<BF16>(d))));
  }
  for (; i < nv; i += stride) m = fmaxf(m, vec_absmax<BF16>(__ldg(vin + i)));
  for (int64_t j = nv * kPerVec + blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
       j < n; j += stride)
    m = fmaxf(m, fabsf(load_elem(in, BF16, j)));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  __shared__ float wm[kThreadsPerBlock / 32];
  if ((threadIdx.x & 31) == 0) wm[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float r = wm[0];
    for (int w = 1; w < kThreadsPerBlock / 32; ++w) r = fmaxf(r, wm[w]);
    partials[blockIdx.x] = r;
  }
}

// One block of kAmaxBlocks threads.  state[0] = scale; scale_inv[0] = 1 / scale.
__global__ void fp8_scale_kernel(const float* __restrict__ partials, float fmax,
                                 float* __restrict__ state, float* __restrict__ scale_inv) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_launch();
  float m = partials[threadIdx.x];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  __shared__ float wm[kAmaxBlocks / 32];
  if ((threadIdx.x & 31) == 0) wm[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float amax = wm[0];
    for (int w = 1; w < kAmaxBlocks / 32; ++w) amax = fmaxf(amax, wm[w]);
    const float scale = amax > 0.f ? __fdiv_rn(fmax, amax) : 1.f;
    state[0] = scale;
    scale_inv[0] = __fdiv_rn(1.f, scale);
  }
}

template <bool BF16, int FMT>
__global__ void fp8_cast_kernel(const void* __restrict__ in, int64_t n,
                                const float* __restrict__ state, uint8_t* __restrict__ out) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_launch();
  const float sc = state[0];
  constexpr __nv_fp8_interpretation_t kInterp = FMT == 0 ? __NV_E4M3 : __NV_E5M2;
  const int64_t n8 = n / 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t v = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; v < n8; v += stride) {
    float x[8];
    if constexpr (BF16) {
      const uint4 w = reinterpret_cast<const uint4*>(in)[v];
      x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x); x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
      x[4] = bf16_lo(w.z); x[5] = bf16_hi(w.z); x[6] = bf16_lo(w.w); x[7] = bf16_hi(w.w);
    } else {
      const float4 a = reinterpret_cast<const float4*>(in)[2 * v];
      const float4 b = reinterpret_cast<const float4*>(in)[2 * v + 1];
      x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
      x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    }
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      lo |= static_cast<uint32_t>(__nv_cvt_float_to_fp8(__fmul_rn(x[e], sc), __NV_SATFINITE, kInterp))
            << (8 * e);
      hi |= static_cast<uint32_t>(
                __nv_cvt_float_to_fp8(__fmul_rn(x[4 + e], sc), __NV_SATFINITE, kInterp))
            << (8 * e);
    }
    reinterpret_cast<uint2*>(out)[v] = make_uint2(lo, hi);
  }
  // tail (n not a multiple of 8)
  for (int64_t i = n8 * 8 + blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += stride)
    out[i] = __nv_cvt_float_to_fp8(__fmul_rn(load_elem(in, BF16, i), sc), __NV_SATFINITE, kInterp);
}

// The same cast over a row-major [rows, cols] matrix, writing it as is
// (`out`, [rows, cols]) and/or transposed (`out_t`, [cols, rows]): the
// transposed copy is the K-major form of the matrix for products that
// contract over its rows (weight gradients, and the weight in an input
// gradient).  One 64 x 64 tile per block, staged through shared memory;
// cols and rows are multiples of 16.
constexpr int kTT = 64;  // tile edge
template <bool BF16, int FMT>
__global__ void __launch_bounds__(256)
    fp8_cast_2d_kernel(const void* __restrict__ in, int64_t rows, int64_t cols,
                       const float* __restrict__ state, uint8_t* __restrict__ out,
                       uint8_t* __restrict__ out_t) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_launch();
  __shared__ uint8_t tile[kTT][kTT + 4];
  const float sc = state[0];
  constexpr __nv_fp8_interpretation_t kInterp = FMT == 0 ? __NV_E4M3 : __NV_E5M2;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * kTT;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kTT;
  // load + cast: thread -> (row tid / 4, 16 columns at 16 (tid % 4))
  {
    const int lr = threadIdx.x >> 2, lc = (threadIdx.x & 3) * 16;
    const int64_t r = r0 + lr, c = c0 + lc;
    if (r < rows && c < cols) {
      float x[16];
      if constexpr (BF16) {
        const uint4* src = reinterpret_cast<const uint4*>(
            static_cast<const __nv_bfloat16*>(in) + r * cols + c);
#pragma unroll
        for (int v = 0; v < 2; ++v) {
          const uint4 w = src[v];
          x[8 * v + 0] = bf16_lo(w.x); x[8 * v + 1] = bf16_hi(w.x);
          x[8 * v + 2] = bf16_lo(w.y); x[8 * v + 3] = bf16_hi(w.y);
          x[8 * v + 4] = bf16_lo(w.z); x[8 * v + 5] = bf16_hi(w.z);
          x[8 * v + 6] = bf16_lo(w.w); x[8 * v + 7] = bf16_hi(w.w);
        }
      } else {
        const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(in) +
                                                            r * cols + c);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const float4 a = src[v];
          x[4 * v] = a.x; x[4 * v + 1] = a.y; x[4 * v + 2] = a.z; x[4 * v + 3] = a.w;
        }
      }
      uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const uint8_t b = __nv_cvt_float_to_fp8(__fmul_rn(x[e], sc), __NV_SATFINITE, kInterp);
        w[e >> 2] |= static_cast<uint32_t>(b) << (8 * (e & 3));
        tile[lr][lc + e] = b;
      }
      if (out) *reinterpret_cast<uint4*>(out + r * cols + c) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  if (!out_t) return;
  __syncthreads();
  // transposed store: thread -> (output row = column tid / 4, 16 source rows)
  {
    const int lc = threadIdx.x >> 2, lr = (threadIdx.x & 3) * 16;
    const int64_t c = c0 + lc, r = r0 + lr;
    if (c < cols && r < rows) {
      uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int e = 0; e < 16; ++e) w[e >> 2] |= static_cast<uint32_t>(tile[lr + e][lc]) << (8 * (e & 3));
      *reinterpret_cast<uint4*>(out_t + c * rows + r) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

}  // namespace

size_t fp8_scratch_floats() { return kAmaxBlocks + 1; }

int launch_fp8_quantize_2d(const void* in, bool in_bf16, int64_t rows, int64_t cols, int format,
                           uint8_t* out, uint8_t* out_t, float* scale_inv, float* scratch,
                           cudaStream_t st) {
  if (rows < 1 || cols < 1 || rows % 16 || cols % 16) return MC_ERR_SHAPE;
  if ((rows + kTT - 1) / kTT > 65535 || cols > (int64_t(1) << 31)) return MC_ERR_UNSUPPORTED;
  if (format < 0 || format > 1) return MC_ERR_ARGUMENT;
  if (!in || (!out && !out_t) || !scale_inv || !scratch) return MC_ERR_NULLPTR;
  if ((reinterpret_cast<uintptr_t>(in) & 15u) || (reinterpret_cast<uintptr_t>(out) & 15u) ||
      (reinterpret_cast<uintptr_t>(out_t) & 15u) || (reinterpret_cast<uintptr_t>(scratch) & 3u) ||
      (reinterpret_cast<uintptr_t>(scale_inv) & 3u))
    return MC_ERR_ALIGN;
  const int64_t n = rows * cols;
  const float fmax = format == 0 ? 448.f : 57344.f;
  float* partials = scratch;
  float* state = scratch + kAmaxBlocks;
  if (in_bf16)
    launch_kernel(amax_partial_kernel<true>, dim3(kAmaxBlocks), dim3(kThreadsPerBlock), 0, st, 1,
                  in, n, partials);
  else
    launch_kernel(amax_partial_kernel<false>, dim3(kAmaxBlocks), dim3(kThreadsPerBlock), 0, st, 1,
                  in, n, partials);
  launch_kernel(fp8_scale_kernel, dim3(1), dim3(kAmaxBlocks), 0, st, 1, partials, fmax, state,
                scale_inv);
  const dim3 grid(static_cast<unsigned>((cols + kTT - 1) / kTT),
                  static_cast<unsigned>((rows + kTT - 1) / kTT));
  auto kern = in_bf16 ? (format == 0 ? fp8_cast_2d_kernel<true, 0> : fp8_cast_2d_kernel<true, 1>)
                      : (format == 0 ? fp8_cast_2d_kernel<false, 0> : fp8_cast_2d_kernel<false, 1>);
  launch_kernel(kern, grid, dim3(256), 0, st, 1, in, rows, cols, state, out, out_t);
  return cudaGetLastError() == cudaSuccess ? MC_OK : MC_ERR_CUDA;
}

int launch_fp8_quantize(const void* in, bool in_bf16, int64_t n, int format, uint8_t* out,
                        float* scale_inv, float* scratch, cudaStream_t st) {
  if (n < 1) return MC_ERR_SHAPE;
  if (format < 0 || format > 1) return MC_ERR_ARGUMENT;
  if (!in || !out || !scale_inv || !scratch) return MC_ERR_NULLPTR;
  if ((reinterpret_cast<uintptr_t>(in) & 15u) || (reinterpret_cast<uintptr_t>(out) & 7u) ||
      (reinterpret_cast<uintptr_t>(scratch) & 3u) || (reinterpret_cast<uintptr_t>(scale_inv) & 3u))
    return MC_ERR_ALIGN;
  const float fmax = format == 0 ? 448.f : 57344.f;
  float* partials = scratch;
  float* state = scratch + kAmaxBlocks;
  const int64_t want = (n + kThreadsPerBlock - 1) / kThreadsPerBlock;
  // every partial is written: the grid is exactly kAmaxBlocks blocks
  if (in_bf16)
    launch_kernel(amax_partial_kernel<true>, dim3(kAmaxBlocks), dim3(kThreadsPerBlock), 0, st, 1,
                  in, n, partials);
  else
    launch_kernel(amax_partial_kernel<false>, dim3(kAmaxBlocks), dim3(kThreadsPerBlock), 0, st, 1,
                  in, n, partials);
  launch_kernel(fp8_scale_kernel, dim3(1), dim3(kAmaxBlocks), 0, st, 1, partials, fmax, state,
                scale_inv);
  const unsigned grid = static_cast<unsigned>(
      want / 8 + 1 < 4 * static_cast<int64_t>(num_sms()) ? want / 8 + 1 : 4 * num_sms());
  if (in_bf16 && format == 0)
    launch_kernel(fp8_cast_kernel<true, 0>, dim3(grid), dim3(kThreadsPerBlock), 0, st, 1, in, n,
                  state, out);
  else if (in_bf16)
    launch_kernel(fp8_cast_kernel<true, 1>, dim3(grid), dim3(kThreadsPerBlock), 0, st, 1, in, n,
                  state, out);
  else if (format == 0)
    launch_kernel(fp8_cast_kernel<false, 0>, dim3(grid), dim3(kThreadsPerBlock), 0, st, 1, in, n,
                  state, out);
  else
    launch_kernel(fp8_cast_kernel<false, 1>, dim3(grid), dim3(kThreadsPerBlock), 0, st, 1, in, n,
                  state, out);
  return cudaGetLastError() == cudaSuccess ? MC_OK : MC_ERR_CUDA;
}

}  // namespace mc

using namespace mc;

extern "C" {

size_t mc_fp8_scratch_floats(void) { return fp8_scratch_floats(); }

int mc_fp8_quantize(const void* in, int32_t in_bf16, int64_t n, int32_t format, uint8_t* out,
                    float* scale_inv, float* scratch, int* status, void* stream) {
  (void)status;
  return launch_fp8_quantize(in, in_bf16 != 0, n, format, out, scale_inv, scratch,
                             static_cast<cudaStream_t>(stream));
}

int mc_fp8_quantize_2d(const void* in, int32_t in_bf16, int64_t rows, int64_t cols,
                       int32_t format, uint8_t* out, uint8_t* out_t, float* scale_inv,
                       float* scratch, void* stream) {
  return launch_fp8_quantize_2d(in, in_bf16 != 0, rows, cols, format, out, out_t, scale_inv,
                                scratch, static_cast<cudaStream_t>(stream));
}

int mc_gemm_fp8(int64_t M, int64_t N, int64_t K, const uint8_t* A, int64_t lda, int32_t a_format,
                const uint8_t* B, int64_t ldb, int32_t b_format, const float* a_scale_inv,
                const float* b_scale_inv, void* out, int64_t ldc, int32_t epilogue,
                const uint16_t* bias, const void* aux, int64_t ldaux, int32_t accumulate,
                int32_t k_parts, int* status, void* stream) {
  return launch_gemm_fp8(M, N, K, A, lda, a_format, B, ldb, b_format, a_scale_inv, b_scale_inv,
                         out, ldc, epilogue, bias, aux, ldaux, accumulate, k_parts, status,
                         static_cast<cudaStream_t>(stream));
}

}  // extern "C"
