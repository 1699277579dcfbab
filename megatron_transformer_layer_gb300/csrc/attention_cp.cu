// Context-parallel causal attention as virtual CP partitions on one GPU.
//
// Megatron Core guide (parallelism table; proving semantics unchanged) and
// the Megatron-Core listing (dynamic context parallelism): context
// parallelism splits the sequence of inputs and activations across ranks,
// and attention still needs every earlier token's K and V from the others.
//
// Here each micro-batch's sequence is cut into C = 2 cp chunks of c tokens;
// virtual rank r owns chunks r and C - 1 - r, which evens out the causal
// work (every rank computes 2 cp - 1 full chunk pairs and 2 diagonal ones).
// In ring step t rank r holds the K/V chunks of rank (r - t) mod cp and
// computes the partial attention of each of its query chunks i over each
// held key chunk j <= i.  The partial (i, j) lands in fp32 slot
// i (i + 1) / 2 + j of the workspace:
//   forward  O_ij normalised over chunk j's keys and lse_ij, merged per query
//            chunk with the log-sum-exp rule (cp_merge_kernel);
//   backward dQ_ij, dK_ij, dV_ij from the merged lse and delta; a chunk's dQ
//            sums its pairs over j, its dK, dV over i (cp_reduce_kernel), in
//            index order, in fp32.
// On one GPU the K/V exchange is the read of the other chunk's rows; the
// partial kernels are the fused kernels restricted to a rectangle of the
// score matrix (attention_tc.cu).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "mc_layer_internal.h"
#include "ptx.cuh"

namespace mc {
namespace {

__host__ __device__ inline int64_t pair_slot(int i, int j) {
  return static_cast<int64_t>(i) * (i + 1) / 2 + j;
}

int64_t num_pairs(int cp) {
  const int64_t C = 2 * static_cast<int64_t>(cp);
  return C * (C + 1) / 2;
}

// One warp per (token, head): merge the partials of the token's query chunk.
template <int D>
__global__ void cp_merge_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse,
                                uint16_t* __restrict__ o, float* __restrict__ lse, int b, int s,
                                int H, int c) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_launch();
  const int64_t wid = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= static_cast<int64_t>(b) * s * H) return;
  const int64_t tok = wid / H;
  const int hh = static_cast<int>(wid % H);
  const int bi = static_cast<int>(tok / s), pos = static_cast<int>(tok % s);
  const int i = pos / c, row = pos % c;
  const int64_t a = static_cast<int64_t>(H) * D;
  constexpr int PER = D / 32;
  auto lse_of = [&](int j) {
    return part_lse[((pair_slot(i, j) * b + bi) * H + hh) * c + row];
  };
  float mx = -INFINITY;
  for (int j = 0; j <= i; ++j) mx = fmaxf(mx, lse_of(j));
  float den = 0.f;
  for (int j = 0; j <= i; ++j) den += expf(lse_of(j) - mx);
  const float l = mx + logf(den);
  float acc[PER] = {};
  for (int j = 0; j <= i; ++j) {
    const float wgt = expf(lse_of(j) - l);
    const float* src = part_o + ((pair_slot(i, j) * b + bi) * c + row) * a + hh * D + lane * PER;
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] += wgt * src[e];
  }
  uint16_t* dst = o + tok * a + hh * D + lane * PER;
#pragma unroll
  for (int e = 0; e < PER; e += 2) *reinterpret_cast<uint32_t*>(dst + e) = pack_bf16x2(acc[e], acc[e + 1]);
  if (lane == 0) lse[(static_cast<int64_t>(bi) * H + hh) * s + pos] = l;
}

// One thread per 4 consecutive columns of a token's dQ | dK | dV row.
__global__ void cp_reduce_kernel(const float* __restrict__ part_dq, const float* __restrict__ part_dkv,
                                 uint16_t* __restrict__ dqkv, int b, int s, int a, int c, int C) {
  pdl_wait();  // the previous kernel on the stream has completed
  pdl_launch();
  const int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  const int64_t per_tok = 3 * static_cast<int64_t>(a) / 4;
  if (idx >= static_cast<int64_t>(b) * s * per_tok) return;
  const int64_t tok = idx / per_tok;
  const int col = static_cast<int>(idx % per_tok) * 4;
  const int bi = static_cast<int>(tok / s), pos = static_cast<int>(tok % s);
  const int chunk = pos / c, row = pos % c;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  auto add = [&](const float* p) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  };
  if (col < a) {  // dQ of query chunk `chunk`: its pairs over key chunks j <= chunk
    for (int j = 0; j <= chunk; ++j)
      add(part_dq + ((pair_slot(chunk, j) * b + bi) * c + row) * a + col);
  } else {        // dK | dV of key chunk `chunk`: the query chunks i >= chunk that saw it
    for (int i = chunk; i < C; ++i)
      add(part_dkv + ((pair_slot(i, chunk) * b + bi) * c + row) * 2 * a + (col - a));
  }
  uint2 w;
  w.x = pack_bf16x2(acc.x, acc.y);
  w.y = pack_bf16x2(acc.z, acc.w);
  *reinterpret_cast<uint2*>(dqkv + tok * 3 * a + col) = w;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_cp(int b, int s, int H, int d, int cp) {
  if (b < 1 || s < 1 || H < 1 || cp < 1) return MC_ERR_SHAPE;
  if (d != 64 && d != 128) return MC_ERR_UNSUPPORTED;
  if (H > 65535 || b > 65535) return MC_ERR_UNSUPPORTED;
  if (s % (256 * cp) != 0) return MC_ERR_SHAPE;  // chunks of a whole number of 128-token tiles
  return MC_OK;
}

size_t cp_workspace_bytes(int b, int s, int H, int d, int cp) {
  const int64_t c = s / (2 * cp), a = static_cast<int64_t>(H) * d;
  // region A: O or dQ partials (a per row); region B: lse (H per row) or dK | dV (2a per row)
  return static_cast<size_t>(num_pairs(cp) * b * c * (a + 2 * a)) * sizeof(float);
}

}  // namespace
}  // namespace mc

using namespace mc;

extern "C" {

int mc_cp_schedule(int32_t cp_parts, int32_t rank, int32_t step, int32_t* pairs) {
  if (cp_parts < 1 || rank < 0 || rank >= cp_parts || step < 0 || step >= cp_parts || !pairs)
    return MC_ERR_ARGUMENT;
  const int C = 2 * cp_parts;
  const int src = (rank - step + cp_parts) % cp_parts;  // whose K/V this rank holds in `step`
  const int q[2] = {rank, C - 1 - rank}, k[2] = {src, C - 1 - src};
  int n = 0;
  for (int qi : q)
    for (int kj : k)
      if (kj <= qi) {
        pairs[2 * n] = qi;
        pairs[2 * n + 1] = kj;
        ++n;
      }
  return n;
}

size_t mc_attention_cp_workspace_bytes(int32_t micro_batch, int32_t seq_len, int32_t heads,
                                       int32_t head_dim, int32_t cp_parts) {
  if (check_cp(micro_batch, seq_len, heads, head_dim, cp_parts) != MC_OK) return 0;
  return cp_workspace_bytes(micro_batch, seq_len, heads, head_dim, cp_parts);
}

int mc_attention_forward_cp(const uint16_t* qkv, uint16_t* o, float* lse, int32_t micro_batch,
                            int32_t seq_len, int32_t heads, int32_t head_dim, int32_t cp_parts,
                            void* workspace, size_t workspace_bytes, int* status, void* stream) {
  const int b = micro_batch, s = seq_len, H = heads, d = head_dim, cp = cp_parts;
  int rc = check_cp(b, s, H, d, cp);
  if (rc != MC_OK) return rc;
  if (!qkv || !o || !lse || !workspace) return MC_ERR_NULLPTR;
  if (!al16(qkv) || !al16(o) || !al16(workspace)) return MC_ERR_ALIGN;
  if (workspace_bytes < cp_workspace_bytes(b, s, H, d, cp)) return MC_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int c = s / (2 * cp), cb = c / 128;
  const int64_t a = static_cast<int64_t>(H) * d;
  float* part_o = static_cast<float*>(workspace);
  float* part_lse = part_o + num_pairs(cp) * b * c * a;
  for (int t = 0; t < cp; ++t)
    for (int r = 0; r < cp; ++r) {
      int32_t pairs[8];
      const int n = mc_cp_schedule(cp, r, t, pairs);
      for (int k = 0; k < n; ++k) {
        const int i = pairs[2 * k], j = pairs[2 * k + 1];
        const int64_t sl = pair_slot(i, j);
        rc = launch_attention_forward_part(qkv, b, s, H, d, i * c, c, j * cb, (j + 1) * cb,
                                           part_o + sl * b * c * a, part_lse + sl * b * H * c,
                                           status, st);
        if (rc != MC_OK) return rc;
      }
    }
  const int64_t warps = static_cast<int64_t>(b) * s * H;
  const unsigned blocks = static_cast<unsigned>((warps * 32 + 255) / 256);
  if (d == 64)
    launch_kernel(cp_merge_kernel<64>, dim3(blocks), dim3(256), 0, st, 1, part_o, part_lse, o, lse,
                  b, s, H, c);
  else
    launch_kernel(cp_merge_kernel<128>, dim3(blocks), dim3(256), 0, st, 1, part_o, part_lse, o, lse,
                  b, s, H, c);
  return cudaGetLastError() == cudaSuccess ? MC_OK : MC_ERR_CUDA;
}

int mc_attention_backward_cp(const uint16_t* qkv, const uint16_t* o, const float* lse,
                             const uint16_t* dout, uint16_t* dqkv, float* delta,
                             int32_t micro_batch, int32_t seq_len, int32_t heads,
                             int32_t head_dim, int32_t cp_parts, void* workspace,
                             size_t workspace_bytes, int* status, void* stream) {
  const int b = micro_batch, s = seq_len, H = heads, d = head_dim, cp = cp_parts;
  int rc = check_cp(b, s, H, d, cp);
  if (rc != MC_OK) return rc;
  if (!qkv || !o || !lse || !dout || !dqkv || !delta || !workspace) return MC_ERR_NULLPTR;
  if (!al16(qkv) || !al16(o) || !al16(dout) || !al16(dqkv) || !al16(workspace))
    return MC_ERR_ALIGN;
  if (workspace_bytes < cp_workspace_bytes(b, s, H, d, cp)) return MC_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int c = s / (2 * cp), cb = c / 128, C = 2 * cp;
  const int64_t a = static_cast<int64_t>(H) * d;
  float* part_dq = static_cast<float*>(workspace);
  float* part_dkv = part_dq + num_pairs(cp) * b * c * a;
  rc = launch_attention_delta(o, dout, delta, b, s, H, d, st);
  if (rc != MC_OK) return rc;
  for (int t = 0; t < cp; ++t)
    for (int r = 0; r < cp; ++r) {
      int32_t pairs[8];
      const int n = mc_cp_schedule(cp, r, t, pairs);
      for (int k = 0; k < n; ++k) {
        const int i = pairs[2 * k], j = pairs[2 * k + 1];
        const int64_t sl = pair_slot(i, j);
        rc = launch_attention_dq_part(qkv, lse, dout, delta, b, s, H, d, i * c, c, j * cb,
                                      (j + 1) * cb, part_dq + sl * b * c * a, status, st);
        if (rc != MC_OK) return rc;
        rc = launch_attention_dkdv_part(qkv, lse, dout, delta, b, s, H, d, j * c, c, i * cb,
                                        (i + 1) * cb, part_dkv + sl * b * c * 2 * a, status, st);
        if (rc != MC_OK) return rc;
      }
    }
  const int64_t threads = static_cast<int64_t>(b) * s * (3 * a / 4);
  launch_kernel(cp_reduce_kernel, dim3(static_cast<unsigned>((threads + 255) / 256)), dim3(256), 0,
                st, 1, part_dq, part_dkv, dqkv, b, s, static_cast<int>(a), c, C);
  return cudaGetLastError() == cudaSuccess ? MC_OK : MC_ERR_CUDA;
}

}  // extern "C"
