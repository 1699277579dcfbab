// Per-tensor current scaling to 8-bit floats for the FP8 GEMM path.
//
// The Megatron-Core listing (混合精度; --fp8-format hybrid: E4M3 forward,
// E5M2 gradients) names the formats and no recipe; the reading taken is the
// plainest one: amax = max |x| (fp32), scale = fmax / amax (fp32 division,
// 1 when amax is 0), q = round-to-nearest-even of x * scale (fp32 product),
// saturated to +-fmax (E4M3: 448, E5M2: 57344), and scale_inv = 1 / scale for
// the GEMM epilogue.
//   amax_partial_kernel  grid-stride |x| maxima, one per block
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

template <bool BF16>
__global__ void amax_partial_kernel(const void* __restrict__ in, int64_t n,
                                    float* __restrict__ partials) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_launch();
  float m = 0.f;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n; i += stride)
    m = fmaxf(m, fabsf(load_elem(in, BF16, i)));
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

}  // namespace

size_t fp8_scratch_floats() { return kAmaxBlocks + 1; }

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
