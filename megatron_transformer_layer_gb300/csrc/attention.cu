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
// delta[b, h, i] = sum_c dO[i, h*D + c] * O[i, h*D + c]; one warp per (token, head).
template <int D>
__global__ void attn_bwd_pre_kernel(const uint16_t* __restrict__ o, const uint16_t* __restrict__ dout,
                                    float* __restrict__ delta, int64_t T, int s, int H) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_launch();
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

template <int D>
int bwd_launch(const uint16_t* qkv, const uint16_t* o, const float* lse, const uint16_t* dout,
               uint16_t* dqkv, float* delta, int b, int s, int H, int* status, cudaStream_t st) {
  const int64_t T = static_cast<int64_t>(b) * s;
  const int64_t warps = T * H;
  launch_kernel(attn_bwd_pre_kernel<D>, dim3(static_cast<unsigned>((warps * 32 + 255) / 256)), dim3(256), 0, st, 1, 
      o, dout, delta, T, s, H);
  if (cudaGetLastError() != cudaSuccess) return MC_ERR_CUDA;
  return launch_attention_backward_tc(qkv, lse, dout, dqkv, delta, b, s, H, D, status, st);
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

int launch_attention_delta(const uint16_t* o, const uint16_t* dout, float* delta, int b, int s,
                           int H, int d, cudaStream_t st) {
  const int64_t T = static_cast<int64_t>(b) * s;
  const unsigned blocks = static_cast<unsigned>((T * H * 32 + 255) / 256);
  if (d == 64)
    launch_kernel(attn_bwd_pre_kernel<64>, dim3(blocks), dim3(256), 0, st, 1, o, dout, delta, T, s, H);
  else
    launch_kernel(attn_bwd_pre_kernel<128>, dim3(blocks), dim3(256), 0, st, 1, o, dout, delta, T, s, H);
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
  return d == 64 ? bwd_launch<64>(qkv, o, lse, dout, dqkv, delta, b, s, H, status, st)
                 : bwd_launch<128>(qkv, o, lse, dout, dqkv, delta, b, s, H, status, st);
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
