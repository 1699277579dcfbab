// Attention entry points: argument checks, the delta = rowsum(dO * O)
// pre-pass of the backward, and the allocation-free backward variant.  The
// forward and backward kernels themselves run on tcgen05 (attention_tc.cu).
//
// Layout: qkv [T, 3a] bf16 (token-major; Q | K | V blocks, head k at columns
// k*d of its block), o / dO [T, a] bf16, lse / delta [b, H, s] fp32.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "mc_layer_internal.h"
#include "ptx.cuh"

namespace mc {
namespace {

// ---------------------------------------------------------------- backward
// delta[b, h, i] = sum_c dO[i, h*D + c] * O[i, h*D + c].  D/8 threads share a
// (token, head) row, each loading 16 bytes of O and of dO; rows are taken
// token-major (head fastest), so row r starts at element r * D of both
// [T, a] arrays and a block streams one contiguous range of each (the
// scattered 4-byte delta stores are 1/(2D) of the traffic and merge in L2),
// and each thread handles kDeltaPasses rows with all their loads issued first.
constexpr int kDeltaThreads = 256;
constexpr int kDeltaPasses = 4;

template <int D>
__host__ __device__ constexpr int64_t delta_rows_per_block() {
  return static_cast<int64_t>(kDeltaThreads / (D / 8)) * kDeltaPasses;
}

template <int D>
__global__ void __launch_bounds__(kDeltaThreads)
    attn_bwd_pre_kernel(const uint16_t* __restrict__ o, const uint16_t* __restrict__ dout,
                        float* __restrict__ delta, int64_t T, int s, int H) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_launch();
  constexpr int TPR = D / 8;                  // threads per row: 16 (D = 128) or 8 (D = 64)
  constexpr int RPP = kDeltaThreads / TPR;    // rows per pass of the block
  const int sub = static_cast<int>(threadIdx.x) % TPR;
  const int64_t rows = T * H;
  const int64_t r0 = blockIdx.x * delta_rows_per_block<D>() + threadIdx.x / TPR;
  uint4 xo[kDeltaPasses], xd[kDeltaPasses];
#pragma unroll
  for (int p = 0; p < kDeltaPasses; ++p) {
    const int64_t r = r0 + p * RPP;  // r = token * H + head
    xo[p] = make_uint4(0u, 0u, 0u, 0u);
    xd[p] = make_uint4(0u, 0u, 0u, 0u);
    if (r < rows) {
      const int64_t off = r * D + sub * 8;  // = token * a + head * D + sub * 8
      xo[p] = __ldg(reinterpret_cast<const uint4*>(o + off));
      xd[p] = __ldg(reinterpret_cast<const uint4*>(dout + off));
    }
  }
#pragma unroll
  for (int p = 0; p < kDeltaPasses; ++p) {
    float acc = bf16_lo(xo[p].x) * bf16_lo(xd[p].x) + bf16_hi(xo[p].x) * bf16_hi(xd[p].x) +
                bf16_lo(xo[p].y) * bf16_lo(xd[p].y) + bf16_hi(xo[p].y) * bf16_hi(xd[p].y) +
                bf16_lo(xo[p].z) * bf16_lo(xd[p].z) + bf16_hi(xo[p].z) * bf16_hi(xd[p].z) +
                bf16_lo(xo[p].w) * bf16_lo(xd[p].w) + bf16_hi(xo[p].w) * bf16_hi(xd[p].w);
    // the TPR lanes of a row are consecutive and aligned within the warp
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    const int64_t r = r0 + p * RPP;
    if (sub == 0 && r < rows) {
      const int64_t hh = r % H, tok = r / H;
      const int64_t bi = tok / s, i = tok % s;
      delta[(bi * H + hh) * s + i] = acc;
    }
  }
}

template <int D>
int bwd_launch(const uint16_t* qkv, const uint16_t* o, const float* lse, const uint16_t* dout,
               uint16_t* dqkv, float* delta, int b, int s, int H, int* status, cudaStream_t st,
               uint8_t* ds_tiles) {
  const int64_t T = static_cast<int64_t>(b) * s;
  const int64_t blocks = (T * H + delta_rows_per_block<D>() - 1) / delta_rows_per_block<D>();
  launch_kernel(attn_bwd_pre_kernel<D>, dim3(static_cast<unsigned>(blocks)), dim3(kDeltaThreads),
                0, st, 1, o, dout, delta, T, s, H);
  if (cudaGetLastError() != cudaSuccess) return MC_ERR_CUDA;
  return launch_attention_backward_tc(qkv, lse, dout, dqkv, delta, b, s, H, D, status, st,
                                      ds_tiles);
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

int launch_attention_delta(const uint16_t* o, const uint16_t* dout, float* delta, int b, int s,
                           int H, int d, cudaStream_t st) {
  const int64_t T = static_cast<int64_t>(b) * s;
  if (d == 64)
    launch_kernel(attn_bwd_pre_kernel<64>,
                  dim3(static_cast<unsigned>((T * H + delta_rows_per_block<64>() - 1) /
                                             delta_rows_per_block<64>())),
                  dim3(kDeltaThreads), 0, st, 1, o, dout, delta, T, s, H);
  else
    launch_kernel(attn_bwd_pre_kernel<128>,
                  dim3(static_cast<unsigned>((T * H + delta_rows_per_block<128>() - 1) /
                                             delta_rows_per_block<128>())),
                  dim3(kDeltaThreads), 0, st, 1, o, dout, delta, T, s, H);
  return cudaGetLastError() == cudaSuccess ? MC_OK : MC_ERR_CUDA;
}

int launch_attention_forward(const uint16_t* qkv, uint16_t* o, float* lse, int b, int s, int H,
                             int d, int* status, cudaStream_t st) {
  (void)status;
  if (b < 1 || s < 1 || H < 1) return MC_ERR_SHAPE;
  if (d != 64 && d != 128) return MC_ERR_UNSUPPORTED;
  if (H > 65535 || b > 65535) return MC_ERR_UNSUPPORTED;
  if (!qkv || !o || !lse) return MC_ERR_NULLPTR;
  if (!al16(qkv) || !al16(o)) return MC_ERR_ALIGN;
  return launch_attention_forward_wide(qkv, o, lse, b, s, H, d, status, st);
}

int launch_attention_backward(const uint16_t* qkv, const uint16_t* o, const float* lse,
                              const uint16_t* dout, uint16_t* dqkv, float* delta, int b, int s,
                              int H, int d, int* status, cudaStream_t st, uint8_t* ds_tiles) {
  (void)status;
  if (b < 1 || s < 1 || H < 1) return MC_ERR_SHAPE;
  if (d != 64 && d != 128) return MC_ERR_UNSUPPORTED;
  if (H > 65535 || b > 65535) return MC_ERR_UNSUPPORTED;
  if (!qkv || !o || !lse || !dout || !dqkv || !delta) return MC_ERR_NULLPTR;
  if (!al16(qkv) || !al16(o) || !al16(dout) || !al16(dqkv) || !al16(ds_tiles))
    return MC_ERR_ALIGN;
  return d == 64 ? bwd_launch<64>(qkv, o, lse, dout, dqkv, delta, b, s, H, status, st, ds_tiles)
                 : bwd_launch<128>(qkv, o, lse, dout, dqkv, delta, b, s, H, status, st, ds_tiles);
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

PerDeviceInit g_noalloc_init;

// Device address of g_noalloc_delta on the current device, looked up with
// cudaGetSymbolAddress the first time for each device (again if the device's
// context was re-created); the symbol's host-side name is only a stand-in,
// not an address a kernel may be given.
int noalloc_scratch(float** out) {
  long long addr = 0;
  const cudaError_t e = once_per_device(g_noalloc_init, [](long long* value) {
    void* p = nullptr;
    const cudaError_t r = cudaGetSymbolAddress(&p, g_noalloc_delta);
    if (r != cudaSuccess) return r;
    if (!p) return cudaErrorInvalidSymbol;
    *value = static_cast<long long>(reinterpret_cast<uintptr_t>(p));
    return cudaSuccess;
  }, &addr);
  if (e != cudaSuccess || addr == 0) return MC_ERR_CUDA;
  *out = reinterpret_cast<float*>(static_cast<uintptr_t>(addr));
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
                                       head_dim, status, static_cast<cudaStream_t>(stream),
                                       nullptr);
}
