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
// held key chunk j <= i.  The ranks of a ring step run together: sub-step k
// of step t is one launch of every rank's k-th pair (no two of which share a
// query chunk or a key chunk).  As a ring implementation does, each partial
// is folded into running fp32 results at once, in schedule order:
//   forward  chunk i's O and log-sum-exp merged with the pair's by the
//            log-sum-exp rule;
//   backward the pair's dK, dV added to key chunk j's sums (the ones a ring
//            sends back to the owner of j) and its dQ = dS K_j to query
//            chunk i's, from the merged lse and delta; dS goes through a
//            tile workspace between the dK/dV kernel and the dQ kernel.
// A chunk's last pair writes the bf16 result.  On one GPU the K/V exchange
// is the read of the other chunk's rows; the partial kernels are the fused
// kernels restricted to a rectangle of the score matrix.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mc_layer_internal.h"

namespace mc {
namespace {

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kCpMaxParts = 256;  // the launch plan's fixed arrays

int check_cp(int b, int s, int H, int d, int cp) {
  if (b < 1 || s < 1 || H < 1 || cp < 1) return MC_ERR_SHAPE;
  if (cp > kCpMaxParts) return MC_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return MC_ERR_UNSUPPORTED;
  if (H > 65535 || b > 65535) return MC_ERR_UNSUPPORTED;
  if (s % (256 * cp) != 0) return MC_ERR_SHAPE;  // chunks of a whole number of 128-token tiles
  return MC_OK;
}

// The launches in order: ring step t, sub-step k = the k-th pair of every
// rank in step t (ranks in order, at most kCpMaxRects to a launch).  Each
// pair is the rectangle of its query chunk i and key chunk j (chunks of c
// rows) with the accumulation modes of both: chunk i has i + 1 pairs, key
// chunk j has C - j.  A rank's pairs of a step keep their order in the
// sub-steps, and a chunk's pairs all come from one rank within a step, so
// every chunk sees its pairs in schedule order.  Calls f(rects, n) for each
// launch and stops at the first code other than MC_OK that f returns; no
// heap memory (cp <= kCpMaxParts).
template <typename F>
int for_each_cp_launch(int cp, int c, F&& f) {
  const int C = 2 * cp;
  int seen_q[2 * kCpMaxParts] = {}, seen_k[2 * kCpMaxParts] = {};
  int32_t pairs[kCpMaxParts][8];
  int np[kCpMaxParts];
  for (int t = 0; t < cp; ++t) {
    int kmax = 0;
    for (int r = 0; r < cp; ++r) {
      np[r] = mc_cp_schedule(cp, r, t, pairs[r]);
      if (np[r] < 0) return np[r];
      kmax = np[r] > kmax ? np[r] : kmax;
    }
    for (int k = 0; k < kmax; ++k) {
      CpRect launch[kCpMaxRects];
      int n = 0;
      for (int r = 0; r < cp; ++r) {
        if (k >= np[r]) continue;
        const int i = pairs[r][2 * k], j = pairs[r][2 * k + 1];
        CpRect p = {i * c, c, j * c, c, 0, 0};
        p.mode_q = (seen_q[i] > 0 ? kCpAccMerge : 0) | (seen_q[i] == i ? kCpAccFinal : 0);
        p.mode_k = (seen_k[j] > 0 ? kCpAccMerge : 0) | (seen_k[j] == C - 1 - j ? kCpAccFinal : 0);
        ++seen_q[i];
        ++seen_k[j];
        launch[n++] = p;
        if (n == kCpMaxRects) {
          const int rc = f(launch, n);
          if (rc != MC_OK) return rc;
          n = 0;
        }
      }
      if (n > 0) {
        const int rc = f(launch, n);
        if (rc != MC_OK) return rc;
      }
    }
  }
  return MC_OK;
}

// Workspace: the running sums, [b, s, 3a] fp32 (forward: O at [0, a) per
// row and the log2-sum-exp [b, H, s] after it; backward: dQ [b, s, a] then
// dK | dV [b, s, 2a]), followed by the dS^T tiles of the largest launch
// (at most cp pairs).
size_t cp_workspace_bytes(int b, int s, int H, int d, int cp) {
  const int64_t a = static_cast<int64_t>(H) * d;
  int64_t tiles = 0;
  for_each_cp_launch(cp, s / (2 * cp), [&](const CpRect* rects, int n) {
    const int64_t t = attention_cp_tile_bytes(rects, n, b, H);
    tiles = t > tiles ? t : tiles;
    return MC_OK;
  });
  return static_cast<size_t>(static_cast<int64_t>(b) * s * 3 * a * 4 + tiles);
}

}  // namespace

int check_cp_rects(const CpRect* rects, int n, int s) {
  if (!rects || n < 1 || n > kCpMaxRects) return MC_ERR_ARGUMENT;
  for (int i = 0; i < n; ++i) {
    const CpRect& r = rects[i];
    // whole 128-row blocks inside the sequence; every query block sees at
    // least one key block and every key block at least one query block
    if (r.q_base < 0 || r.k_base < 0 || r.q_len < 128 || r.k_len < 128 || r.q_base % 128 ||
        r.k_base % 128 || r.q_len % 128 || r.k_len % 128 ||
        static_cast<int64_t>(r.q_base) + r.q_len > s ||
        static_cast<int64_t>(r.k_base) + r.k_len > s || r.k_base > r.q_base ||
        r.k_base + r.k_len > r.q_base + r.q_len)
      return MC_ERR_ARGUMENT;
    for (int j = 0; j < i; ++j) {  // no running sum touched twice in one launch
      const CpRect& o = rects[j];
      if (r.q_base < o.q_base + o.q_len && o.q_base < r.q_base + r.q_len) return MC_ERR_ARGUMENT;
      if (r.k_base < o.k_base + o.k_len && o.k_base < r.k_base + r.k_len) return MC_ERR_ARGUMENT;
    }
  }
  return MC_OK;
}

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

int mc_cp_launch_plan(int32_t cp_parts, int32_t* entries, int32_t max_pairs) {
  if (cp_parts < 1 || cp_parts > kCpMaxParts || !entries) return MC_ERR_ARGUMENT;
  const int64_t pairs = static_cast<int64_t>(cp_parts) * (2 * cp_parts + 1);
  if (max_pairs < pairs) return MC_ERR_WORKSPACE;
  int launch = 0, k = 0;
  const int rc = for_each_cp_launch(cp_parts, 1, [&](const CpRect* rects, int n) {
    for (int i = 0; i < n; ++i, ++k) {
      int32_t* e = entries + 5 * static_cast<int64_t>(k);
      e[0] = launch;
      e[1] = rects[i].q_base;  // chunks of one row: the chunk index
      e[2] = rects[i].k_base;
      e[3] = rects[i].mode_q;
      e[4] = rects[i].mode_k;
    }
    ++launch;
    return MC_OK;
  });
  return rc != MC_OK ? rc : k;
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
  const int c = s / (2 * cp);
  const int64_t a = static_cast<int64_t>(H) * d;
  float* acc_o = static_cast<float*>(workspace);
  float* acc_lse2 = acc_o + static_cast<int64_t>(b) * s * a;
  return for_each_cp_launch(cp, c, [&](const CpRect* rects, int n) {
    return launch_attention_forward_parts(qkv, o, lse, b, s, H, d, rects, n, acc_o, acc_lse2,
                                          status, st);
  });
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
  const int c = s / (2 * cp);
  const int64_t a = static_cast<int64_t>(H) * d;
  float* acc_dq = static_cast<float*>(workspace);
  float* acc_dkv = acc_dq + static_cast<int64_t>(b) * s * a;
  uint8_t* tiles = reinterpret_cast<uint8_t*>(acc_dkv + static_cast<int64_t>(b) * s * 2 * a);
  rc = launch_attention_delta(o, dout, delta, b, s, H, d, st);
  if (rc != MC_OK) return rc;
  return for_each_cp_launch(cp, c, [&](const CpRect* rects, int n) {
    // key rows of chunk j against the query blocks of chunk i: dK, dV and dS^T
    const int r = launch_attention_dkdv_parts(qkv, lse, dout, delta, dqkv, b, s, H, d, rects, n,
                                              acc_dkv, tiles, status, st);
    if (r != MC_OK) return r;
    // dQ of chunk i from those tiles and K of chunk j
    return launch_attention_dq_parts(qkv, tiles, dqkv, b, s, H, d, rects, n, acc_dq, status, st);
  });
}

}  // extern "C"
