// C ABI: shape checks, the `saved` / `ws` buffer plans and the launch
// sequences of one layer's forward and backward pass.  All launches go to the
// caller's stream; nothing here allocates or synchronises (except
// mc_layer_device_status).
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "mc_layer_internal.h"

namespace mc {

cudaError_t current_context(int* dev, unsigned long long* ctx_id) {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;  // driver entry points are process-wide
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(p);
  });
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return e;
  if (!get_current || !get_id) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  if (!ctx) {
    // No context current on this thread yet: cudaSetDevice initialises the
    // device's primary context and makes it current.
    e = cudaSetDevice(*dev);
    if (e != cudaSuccess) return e;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorDeviceUninitialized;
  }
  unsigned long long id = 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  *ctx_id = id + 1;  // never 0, which marks "not set up"
  return cudaSuccess;
}

int num_sms() {
  static std::mutex mu;
  static std::vector<int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  std::lock_guard<std::mutex> lock(mu);
  if (static_cast<int>(cache.size()) <= dev) cache.resize(dev + 1, 0);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
      n = 1;
    cache[dev] = n;
  }
  return cache[dev];
}

namespace {

struct Dims {
  int64_t b, s, T, h, H, d, a, f, t;
  bool fp8;       // MC_FP8_HYBRID
  bool ds_tiles;  // the attention backward's dS tiles (not MC_ATTN_DQ_RECOMPUTE)
};

Dims dims_of(const mc_layer_shape& sh) {
  Dims D;
  D.b = sh.micro_batch;
  D.s = sh.seq_len;
  D.T = D.b * D.s;
  D.h = sh.hidden;
  D.H = sh.heads;
  D.d = sh.head_dim ? sh.head_dim : (sh.heads ? sh.hidden / sh.heads : 0);
  D.a = D.H * D.d;
  D.f = sh.ffn_hidden;
  D.t = sh.tp_parts;
  D.fp8 = (sh.flags & MC_FP8_HYBRID) != 0;
  D.ds_tiles = (sh.flags & MC_ATTN_DQ_RECOMPUTE) == 0;
  return D;
}

int check_shape(const mc_layer_shape* sh) {
  if (!sh) return MC_ERR_NULLPTR;
  if (sh->micro_batch <= 0 || sh->seq_len <= 0 || sh->hidden <= 0 || sh->heads <= 0 ||
      sh->ffn_hidden <= 0 || sh->tp_parts <= 0 || sh->head_dim < 0)
    return MC_ERR_SHAPE;
  if ((sh->flags & ~(MC_ACCUMULATE_GRADS | MC_RECOMPUTE_ACTIVATIONS | MC_SEQUENCE_PARALLEL |
                     MC_FP8_HYBRID | MC_ATTN_DQ_RECOMPUTE)) != 0)
    return MC_ERR_ARGUMENT;
  if ((sh->flags & MC_FP8_HYBRID) && (sh->flags & MC_SEQUENCE_PARALLEL)) return MC_ERR_ARGUMENT;
  const int t = sh->tp_parts;
  // Sequence-parallel contract: the tokens split evenly into t shards.
  if ((sh->flags & MC_SEQUENCE_PARALLEL) &&
      (static_cast<int64_t>(sh->micro_batch) * sh->seq_len) % t != 0)
    return MC_ERR_SHAPE;
  // Divisibility: hidden size and heads (and the ffn slice of the column
  // split) must divide by the tensor-parallel degree.
  if (sh->hidden % t || sh->heads % t || sh->ffn_hidden % t) return MC_ERR_SHAPE;
  if (sh->head_dim == 0 && sh->hidden % sh->heads) return MC_ERR_SHAPE;
  const Dims D = dims_of(*sh);
  if (D.d != 64 && D.d != 128) return MC_ERR_UNSUPPORTED;
  if (D.h % 64 || (D.a / t) % 64 || (D.f / t) % 64) return MC_ERR_UNSUPPORTED;
  if (D.h > kMaxLayerNormHidden) return MC_ERR_UNSUPPORTED;
  if (D.T > (1 << 24) || D.f > (1 << 20) || 3 * D.a > (1 << 20) || D.H > 65535 || D.b > 65535)
    return MC_ERR_UNSUPPORTED;
  // FP8 products contract over tokens in the weight gradients (K = T).
  // (and the 8-bit casts tile the token dimension in at most 65535 x 64 rows)
  if (D.fp8 && (D.T % 16 || D.T > 65535 * 64)) return MC_ERR_UNSUPPORTED;
  return MC_OK;
}

// Sequential 256-byte-aligned carving of a buffer.
struct Carver {
  uint8_t* base;
  size_t off = 0;
  explicit Carver(void* p) : base(static_cast<uint8_t*>(p)) {}
  template <typename T>
  T* take(size_t count) {
    off = (off + 255) & ~static_cast<size_t>(255);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += count * sizeof(T);
    return p;
  }
};

struct Saved {
  uint16_t *ln1, *qkv, *o, *ln2, *hp, *g;
  float *mu1, *rs1, *lse, *x1, *mu2, *rs2;
  // MC_FP8_HYBRID: what the backward reads of the forward's 8-bit operands --
  // the transposed (K-major over tokens) activations for the weight
  // gradients, the transposed weights for the input gradients -- and the
  // inverse scales [ln1, o, ln2, g, w_qkv, w_o, w_fc1, w_fc2].
  uint8_t *ln1_t, *o_t, *ln2_t, *g_t, *wqkv_t, *wo_t, *w1_t, *w2_t;
  float* scale_inv;
};

Saved plan_saved(const Dims& D, void* p, size_t* bytes) {  // NOLINT
  Carver c(p);
  Saved S;
  S.ln1 = c.take<uint16_t>(D.T * D.h);
  S.mu1 = c.take<float>(D.T);
  S.rs1 = c.take<float>(D.T);
  S.qkv = c.take<uint16_t>(D.T * 3 * D.a);
  S.o = c.take<uint16_t>(D.T * D.a);
  S.lse = c.take<float>(D.b * D.H * D.s);
  S.x1 = c.take<float>(D.T * D.h);
  S.ln2 = c.take<uint16_t>(D.T * D.h);
  S.mu2 = c.take<float>(D.T);
  S.rs2 = c.take<float>(D.T);
  S.hp = c.take<uint16_t>(D.T * D.f);
  S.g = c.take<uint16_t>(D.T * D.f);
  S.ln1_t = S.o_t = S.ln2_t = S.g_t = S.wqkv_t = S.wo_t = S.w1_t = S.w2_t = nullptr;
  S.scale_inv = nullptr;
  if (D.fp8) {
    S.ln1_t = c.take<uint8_t>(D.h * D.T);
    S.o_t = c.take<uint8_t>(D.a * D.T);
    S.ln2_t = c.take<uint8_t>(D.h * D.T);
    S.g_t = c.take<uint8_t>(D.f * D.T);
    S.wqkv_t = c.take<uint8_t>(D.h * 3 * D.a);
    S.wo_t = c.take<uint8_t>(D.a * D.h);
    S.w1_t = c.take<uint8_t>(D.h * D.f);
    S.w2_t = c.take<uint8_t>(D.f * D.h);
    S.scale_inv = c.take<float>(8);
  }
  if (bytes) *bytes = (c.off + 255) & ~static_cast<size_t>(255);
  return S;
}

struct Work {
  int* status;
  uint16_t *dy16, *dhp, *dx1_16, *dO, *dqkv;
  float *dln, *dx1, *delta, *partials;
  uint8_t* ds;  // the attention backward's dS^T tiles
  void* recompute_saved;  // activations region when they are recomputed
  // MC_FP8_HYBRID: the row-major 8-bit operands (forward: ln1, o, ln2, g and
  // the weights; backward: dy, dhp, dx1, dqkv), the backward operands'
  // transposed copies and their inverse scales [dy, dhp, dx1, dqkv].
  uint8_t *ln1_q, *o_q, *ln2_q, *g_q, *wqkv_q, *wo_q, *w1_q, *w2_q;
  uint8_t *dy_q, *dy_t, *dhp_q, *dhp_t, *dx1_q, *dx1_t, *dqkv_q, *dqkv_t;
  float* scale_inv;
};

Saved plan_saved(const Dims& D, void* p, size_t* bytes);

bool recompute(const mc_layer_shape& sh) { return (sh.flags & MC_RECOMPUTE_ACTIVATIONS) != 0; }

Work plan_ws(const Dims& D, bool with_saved, void* p, size_t* bytes) {
  Carver c(p);
  Work W;
  W.status = c.take<int>(kStatusBytes / sizeof(int));
  W.dy16 = c.take<uint16_t>(D.T * D.h);
  W.dhp = c.take<uint16_t>(D.T * D.f);
  W.dln = c.take<float>(D.T * D.h);
  W.dx1 = c.take<float>(D.T * D.h);
  W.dx1_16 = c.take<uint16_t>(D.T * D.h);
  W.dO = c.take<uint16_t>(D.T * D.a);
  W.delta = c.take<float>(D.b * D.H * D.s);
  W.dqkv = c.take<uint16_t>(D.T * 3 * D.a);
  W.ds = D.ds_tiles ? c.take<uint8_t>(attention_ds_workspace_bytes(D.b, D.s, D.H)) : nullptr;
  const size_t ln_part = layernorm_backward_scratch_floats(D.T, static_cast<int>(D.h));
  int64_t widest = D.f > 3 * D.a ? D.f : 3 * D.a;
  if (D.h > widest) widest = D.h;
  const size_t col_part = static_cast<size_t>(kColsumMaxSplits) * widest;
  size_t part = ln_part > col_part ? ln_part : col_part;
  if (part < fp8_scratch_floats()) part = fp8_scratch_floats();
  W.partials = c.take<float>(part);
  W.ln1_q = W.o_q = W.ln2_q = W.g_q = W.wqkv_q = W.wo_q = W.w1_q = W.w2_q = nullptr;
  W.dy_q = W.dy_t = W.dhp_q = W.dhp_t = W.dx1_q = W.dx1_t = W.dqkv_q = W.dqkv_t = nullptr;
  W.scale_inv = nullptr;
  if (D.fp8) {
    W.ln1_q = c.take<uint8_t>(D.T * D.h);
    W.o_q = c.take<uint8_t>(D.T * D.a);
    W.ln2_q = c.take<uint8_t>(D.T * D.h);
    W.g_q = c.take<uint8_t>(D.T * D.f);
    W.wqkv_q = c.take<uint8_t>(3 * D.a * D.h);
    W.wo_q = c.take<uint8_t>(D.h * D.a);
    W.w1_q = c.take<uint8_t>(D.f * D.h);
    W.w2_q = c.take<uint8_t>(D.h * D.f);
    W.dy_q = c.take<uint8_t>(D.T * D.h);
    W.dy_t = c.take<uint8_t>(D.h * D.T);
    W.dhp_q = c.take<uint8_t>(D.T * D.f);
    W.dhp_t = c.take<uint8_t>(D.f * D.T);
    W.dx1_q = c.take<uint8_t>(D.T * D.h);
    W.dx1_t = c.take<uint8_t>(D.h * D.T);
    W.dqkv_q = c.take<uint8_t>(D.T * 3 * D.a);
    W.dqkv_t = c.take<uint8_t>(3 * D.a * D.T);
    W.scale_inv = c.take<float>(4);
  }
  W.recompute_saved = nullptr;
  if (with_saved) {
    size_t sb = 0;
    plan_saved(D, nullptr, &sb);
    W.recompute_saved = c.take<uint8_t>(sb);
  }
  if (bytes) *bytes = (c.off + 255) & ~static_cast<size_t>(255);
  return W;
}

bool al(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0; }

int check_weights(const mc_layer_weights* w) {
  if (!w) return MC_ERR_NULLPTR;
  const uint16_t* ptrs[12] = {w->ln1_g, w->ln1_b, w->w_qkv, w->b_qkv, w->w_o,   w->b_o,
                              w->ln2_g, w->ln2_b, w->w_fc1, w->b_fc1, w->w_fc2, w->b_fc2};
  for (auto p : ptrs) {
    if (!p) return MC_ERR_NULLPTR;
    if (!al(p, 16)) return MC_ERR_ALIGN;
  }
  return MC_OK;
}

int check_grads(const mc_layer_grads* g) {
  if (!g) return MC_ERR_NULLPTR;
  float* ptrs[12] = {g->ln1_g, g->ln1_b, g->w_qkv, g->b_qkv, g->w_o,   g->b_o,
                     g->ln2_g, g->ln2_b, g->w_fc1, g->b_fc1, g->w_fc2, g->b_fc2};
  for (auto p : ptrs) {
    if (!p) return MC_ERR_NULLPTR;
    if (!al(p, 16)) return MC_ERR_ALIGN;
  }
  return MC_OK;
}

#define MC_TRY(expr)           \
  do {                         \
    const int rc_ = (expr);    \
    if (rc_ != MC_OK) return rc_; \
  } while (0)

}  // namespace
}  // namespace mc

using namespace mc;

extern "C" {

int mc_layer_check_shape(const mc_layer_shape* shape) { return check_shape(shape); }

size_t mc_layer_saved_bytes(const mc_layer_shape* shape) {
  if (check_shape(shape) != MC_OK) return 0;
  if (recompute(*shape)) return 0;  // nothing is kept between the passes
  size_t n = 0;
  plan_saved(dims_of(*shape), nullptr, &n);
  return n;
}

size_t mc_layer_workspace_bytes(const mc_layer_shape* shape) {
  if (check_shape(shape) != MC_OK) return 0;
  size_t n = 0;
  plan_ws(dims_of(*shape), recompute(*shape), nullptr, &n);
  return n;
}

namespace mc {
namespace {
bool seq_parallel(const mc_layer_shape& sh) { return (sh.flags & MC_SEQUENCE_PARALLEL) != 0; }

// Sequence shards of the sequence-parallel mode: `shards` (t, else 1) runs
// of Ts = T / shards consecutive tokens.  A per-token kernel (LayerNorm, the
// residual epilogue of a row-parallel GEMM) is launched once per shard on
// its rows -- the work one tensor-parallel rank does on its sequence shard.
struct Shards {
  int64_t n, rows;
};

Shards shards_of(const Dims& D, bool sp) { return sp ? Shards{D.t, D.T / D.t} : Shards{1, D.T}; }

// F1..F7: the forward launch sequence into the activations `S`.
// Sequence-parallel mode: LN1, LN2 and the two row-parallel GEMMs run per
// sequence shard.  Each row-parallel launch covers one shard's rows and sums
// every partition's K slice in its accumulator: the reduce-scatter of the
// partial sums.  QKV and fc1 read all shards' LayerNorm output, which lie
// side by side in one buffer: the all-gather.
constexpr int kE4M3 = 0, kE5M2 = 1;

// F1..F7 with FP8 GEMMs (MC_FP8_HYBRID): every GEMM operand is quantised to
// E4M3 first (per-tensor current scaling) -- into a row-major copy for this
// product and, with the same scale, a transposed copy kept for the backward
// pass -- and the GEMM's epilogue multiplies by the two inverse scales.
int enqueue_forward_fp8(const Dims& D, const mc_layer_weights* w, const float* x, float* y,
                        const Saved& S, const Work& W, cudaStream_t st) {
  StageRanges R("mc_layer_forward (fp8)");
  const int t = static_cast<int>(D.t);
  const int h = static_cast<int>(D.h);
  float* si = S.scale_inv;  // [ln1, o, ln2, g, w_qkv, w_o, w_fc1, w_fc2]
  auto quant = [&](const void* in, bool bf16, int64_t rows, int64_t cols, uint8_t* out,
                   uint8_t* out_t, float* sinv) {
    return launch_fp8_quantize_2d(in, bf16, rows, cols, kE4M3, out, out_t, sinv, W.partials, st);
  };
  // the weights, [out, in] as stored and transposed for the input gradients
  R.next("F0 weights to E4M3");
  MC_TRY(quant(w->w_qkv, true, 3 * D.a, D.h, W.wqkv_q, S.wqkv_t, si + 4));
  MC_TRY(quant(w->w_o, true, D.h, D.a, W.wo_q, S.wo_t, si + 5));
  MC_TRY(quant(w->w_fc1, true, D.f, D.h, W.w1_q, S.w1_t, si + 6));
  MC_TRY(quant(w->w_fc2, true, D.h, D.f, W.w2_q, S.w2_t, si + 7));
  // F1  LN1, quantised
  R.next("F1 LN1");
  MC_TRY(launch_layernorm_forward(x, w->ln1_g, w->ln1_b, S.ln1, S.mu1, S.rs1, D.T, h, W.status, st));
  MC_TRY(quant(S.ln1, true, D.T, D.h, W.ln1_q, S.ln1_t, si + 0));
  // F2  QKV
  R.next("F2 QKV");
  MC_TRY(launch_gemm_fp8(D.T, 3 * D.a, D.h, W.ln1_q, D.h, kE4M3, W.wqkv_q, D.h, kE4M3, si + 0,
                         si + 4, S.qkv, 3 * D.a, MC_EPI_BIAS_BF16, w->b_qkv, nullptr, 0, 0, 1,
                         W.status, st));
  // F3  causal attention (bf16), O quantised
  R.next("F3 causal attention");
  MC_TRY(launch_attention_forward(S.qkv, S.o, S.lse, static_cast<int>(D.b), static_cast<int>(D.s),
                                  static_cast<int>(D.H), static_cast<int>(D.d), W.status, st));
  MC_TRY(quant(S.o, true, D.T, D.a, W.o_q, S.o_t, si + 1));
  // F4  out-projection: partition partials summed in the accumulator, + b_o + x
  R.next("F4 out-projection");
  MC_TRY(launch_gemm_fp8(D.T, D.h, D.a, W.o_q, D.a, kE4M3, W.wo_q, D.a, kE4M3, si + 1, si + 5,
                         S.x1, D.h, MC_EPI_BIAS_RESID_F32, w->b_o, x, D.h, 0, t, W.status, st));
  // F5  LN2, quantised
  R.next("F5 LN2");
  MC_TRY(launch_layernorm_forward(S.x1, w->ln2_g, w->ln2_b, S.ln2, S.mu2, S.rs2, D.T, h, W.status,
                                  st));
  MC_TRY(quant(S.ln2, true, D.T, D.h, W.ln2_q, S.ln2_t, si + 2));
  // F6  fc1 + bias + GeLU; g quantised
  R.next("F6 fc1");
  MC_TRY(launch_gemm_fp8(D.T, D.f, D.h, W.ln2_q, D.h, kE4M3, W.w1_q, D.h, kE4M3, si + 2, si + 6,
                         S.g, D.f, MC_EPI_BIAS_GELU, w->b_fc1, S.hp, D.f, 0, 1, W.status, st));
  MC_TRY(quant(S.g, true, D.T, D.f, W.g_q, S.g_t, si + 3));
  // F7  fc2: partials summed, + b_fc2 + x1
  R.next("F7 fc2");
  MC_TRY(launch_gemm_fp8(D.T, D.h, D.f, W.g_q, D.f, kE4M3, W.w2_q, D.f, kE4M3, si + 3, si + 7, y,
                         D.h, MC_EPI_BIAS_RESID_F32, w->b_fc2, S.x1, D.h, 0, t, W.status, st));
  return MC_OK;
}

int enqueue_forward(const Dims& D, const mc_layer_weights* w, const float* x, float* y,
                    const Saved& S, const Work& W, bool sp, cudaStream_t st) {
  if (D.fp8) return enqueue_forward_fp8(D, w, x, y, S, W, st);
  StageRanges R("mc_layer_forward");
  const int t = static_cast<int>(D.t);
  const int h = static_cast<int>(D.h);
  const Shards sh = shards_of(D, sp);
  // F1  LN1 (per shard)
  R.next("F1 LN1");
  for (int64_t p = 0; p < sh.n; ++p) {
    const int64_t r0 = p * sh.rows;
    MC_TRY(launch_layernorm_forward(x + r0 * D.h, w->ln1_g, w->ln1_b, S.ln1 + r0 * D.h, S.mu1 + r0,
                                    S.rs1 + r0, sh.rows, h, W.status, st));
  }
  // F2  QKV (column-parallel: every partition's heads are output columns)
  R.next("F2 QKV");
  MC_TRY(launch_gemm(D.T, 3 * D.a, D.h, S.ln1, D.h, 0, w->w_qkv, D.h, 0, S.qkv, 3 * D.a,
                     MC_EPI_BIAS_BF16, w->b_qkv, nullptr, 0, 0, 1, W.status, st));
  // F3  causal attention, local per head
  R.next("F3 causal attention");
  MC_TRY(launch_attention_forward(S.qkv, S.o, S.lse, static_cast<int>(D.b), static_cast<int>(D.s),
                                  static_cast<int>(D.H), static_cast<int>(D.d), W.status, st));
  // F4  out-projection, row-parallel: partition partials summed in the
  R.next("F4 out-projection");
  //     accumulator, then + b_o + x (per shard)
  for (int64_t p = 0; p < sh.n; ++p) {
    const int64_t r0 = p * sh.rows;
    MC_TRY(launch_gemm(sh.rows, D.h, D.a, S.o + r0 * D.a, D.a, 0, w->w_o, D.a, 0, S.x1 + r0 * D.h,
                       D.h, MC_EPI_BIAS_RESID_F32, w->b_o, x + r0 * D.h, D.h, 0, t, W.status, st));
  }
  // F5  LN2 (per shard)
  R.next("F5 LN2");
  for (int64_t p = 0; p < sh.n; ++p) {
    const int64_t r0 = p * sh.rows;
    MC_TRY(launch_layernorm_forward(S.x1 + r0 * D.h, w->ln2_g, w->ln2_b, S.ln2 + r0 * D.h,
                                    S.mu2 + r0, S.rs2 + r0, sh.rows, h, W.status, st));
  }
  // F6  fc1 + bias + GeLU (column-parallel)
  R.next("F6 fc1");
  MC_TRY(launch_gemm(D.T, D.f, D.h, S.ln2, D.h, 0, w->w_fc1, D.h, 0, S.g, D.f, MC_EPI_BIAS_GELU,
                     w->b_fc1, S.hp, D.f, 0, 1, W.status, st));
  // F7  fc2, row-parallel: partials summed, + b_fc2 + x1 (per shard)
  R.next("F7 fc2");
  for (int64_t p = 0; p < sh.n; ++p) {
    const int64_t r0 = p * sh.rows;
    MC_TRY(launch_gemm(sh.rows, D.h, D.f, S.g + r0 * D.f, D.f, 0, w->w_fc2, D.f, 0, y + r0 * D.h,
                       D.h, MC_EPI_BIAS_RESID_F32, w->b_fc2, S.x1 + r0 * D.h, D.h, 0, t, W.status,
                       st));
  }
  return MC_OK;
}
// B1..B7 with FP8 GEMMs (MC_FP8_HYBRID): the gradient operands dy, dhp, dx1
// and dQ|dK|dV are quantised to E5M2 (row-major and transposed, one scale);
// weight gradients contract over tokens with the transposed copies of both
// operands, input gradients read the forward's transposed E4M3 weights.
int enqueue_backward_fp8(const Dims& D, const mc_layer_weights* w, const float* x,
                         const float* dy, float* dx, const mc_layer_grads& G, const Saved& S,
                         const Work& W, int acc, cudaStream_t st) {
  StageRanges R("mc_layer_backward (fp8)");
  const int t = static_cast<int>(D.t);
  const int h = static_cast<int>(D.h);
  const float* sf = S.scale_inv;  // [ln1, o, ln2, g, w_qkv, w_o, w_fc1, w_fc2]
  float* sb = W.scale_inv;        // [dy, dhp, dx1, dqkv]
  auto quant = [&](const void* in, bool bf16, int64_t rows, int64_t cols, uint8_t* out,
                   uint8_t* out_t, float* sinv) {
    return launch_fp8_quantize_2d(in, bf16, rows, cols, kE5M2, out, out_t, sinv, W.partials, st);
  };
  // B1  fc2: db2 = colsum(dy); dW2 = dy^T g; dhp = (dy W2) * gelu'(hp)
  R.next("B1 fc2");
  MC_TRY(launch_colsum(dy, false, D.T, D.h, G.b_fc2, acc, nullptr, W.partials, W.status, st));
  MC_TRY(quant(dy, false, D.T, D.h, W.dy_q, W.dy_t, sb + 0));
  MC_TRY(launch_gemm_fp8(D.h, D.f, D.T, W.dy_t, D.T, kE5M2, S.g_t, D.T, kE4M3, sb + 0, sf + 3,
                         G.w_fc2, D.f, MC_EPI_STORE_F32, nullptr, nullptr, 0, acc, 1, W.status,
                         st));
  MC_TRY(launch_gemm_fp8(D.T, D.f, D.h, W.dy_q, D.h, kE5M2, S.w2_t, D.h, kE4M3, sb + 0, sf + 7,
                         W.dhp, D.f, MC_EPI_GELU_BWD, nullptr, S.hp, D.f, 0, 1, W.status, st));
  // B2  fc1: db1; dW1 = dhp^T ln2; dln2 = sum_p dhp_p W1_p
  R.next("B2 fc1");
  MC_TRY(launch_colsum(W.dhp, true, D.T, D.f, G.b_fc1, acc, nullptr, W.partials, W.status, st));
  MC_TRY(quant(W.dhp, true, D.T, D.f, W.dhp_q, W.dhp_t, sb + 1));
  MC_TRY(launch_gemm_fp8(D.f, D.h, D.T, W.dhp_t, D.T, kE5M2, S.ln2_t, D.T, kE4M3, sb + 1, sf + 2,
                         G.w_fc1, D.h, MC_EPI_STORE_F32, nullptr, nullptr, 0, acc, 1, W.status,
                         st));
  MC_TRY(launch_gemm_fp8(D.T, D.h, D.f, W.dhp_q, D.f, kE5M2, S.w1_t, D.f, kE4M3, sb + 1, sf + 6,
                         W.dln, D.h, MC_EPI_STORE_F32, nullptr, nullptr, 0, 0, t, W.status, st));
  // B3  LN2 backward: dx1 = dy + LN2^T(dln2); dgamma2, dbeta2; db_o
  R.next("B3 LN2 backward");
  MC_TRY(launch_layernorm_backward(W.dln, S.x1, S.mu2, S.rs2, w->ln2_g, dy, W.dx1, nullptr,
                                   G.ln2_g, G.ln2_b, G.b_o, acc, W.partials, D.T, h, W.status, st));
  MC_TRY(quant(W.dx1, false, D.T, D.h, W.dx1_q, W.dx1_t, sb + 2));
  // B4  out-projection: dWo = dx1^T O; dO = dx1 Wo
  R.next("B4 out-projection");
  MC_TRY(launch_gemm_fp8(D.h, D.a, D.T, W.dx1_t, D.T, kE5M2, S.o_t, D.T, kE4M3, sb + 2, sf + 1,
                         G.w_o, D.a, MC_EPI_STORE_F32, nullptr, nullptr, 0, acc, 1, W.status, st));
  MC_TRY(launch_gemm_fp8(D.T, D.a, D.h, W.dx1_q, D.h, kE5M2, S.wo_t, D.h, kE4M3, sb + 2, sf + 5,
                         W.dO, D.a, MC_EPI_STORE_BF16, nullptr, nullptr, 0, 0, 1, W.status, st));
  // B5  attention backward (bf16) -> dQ | dK | dV
  R.next("B5 attention backward");
  MC_TRY(launch_attention_backward(S.qkv, S.o, S.lse, W.dO, W.dqkv, W.delta, static_cast<int>(D.b),
                                   static_cast<int>(D.s), static_cast<int>(D.H),
                                   static_cast<int>(D.d), W.status, st, W.ds));
  // B6  QKV: db_qkv; dWqkv = dqkv^T ln1; dln1 = sum_p dqkv_p Wqkv_p
  R.next("B6 QKV");
  MC_TRY(launch_colsum(W.dqkv, true, D.T, 3 * D.a, G.b_qkv, acc, nullptr, W.partials, W.status, st));
  MC_TRY(quant(W.dqkv, true, D.T, 3 * D.a, W.dqkv_q, W.dqkv_t, sb + 3));
  MC_TRY(launch_gemm_fp8(3 * D.a, D.h, D.T, W.dqkv_t, D.T, kE5M2, S.ln1_t, D.T, kE4M3, sb + 3,
                         sf + 0, G.w_qkv, D.h, MC_EPI_STORE_F32, nullptr, nullptr, 0, acc, 1,
                         W.status, st));
  MC_TRY(launch_gemm_fp8(D.T, D.h, 3 * D.a, W.dqkv_q, 3 * D.a, kE5M2, S.wqkv_t, 3 * D.a, kE4M3,
                         sb + 3, sf + 4, W.dln, D.h, MC_EPI_STORE_F32, nullptr, nullptr, 0, 0, t,
                         W.status, st));
  // B7  LN1 backward: dx = dx1 + LN1^T(dln1); dgamma1, dbeta1
  R.next("B7 LN1 backward");
  MC_TRY(launch_layernorm_backward(W.dln, x, S.mu1, S.rs1, w->ln1_g, W.dx1, dx, nullptr, G.ln1_g,
                                   G.ln1_b, nullptr, acc, W.partials, D.T, h, W.status, st));
  return MC_OK;
}

}  // namespace
}  // namespace mc

int mc_layer_forward(const mc_layer_shape* shape, const mc_layer_weights* w, const float* x,
                     float* y, void* saved, void* ws, size_t ws_bytes, void* stream) {
  MC_TRY(check_shape(shape));
  MC_TRY(check_weights(w));
  const bool rc_mode = recompute(*shape);
  if (!x || !y || (!saved && !rc_mode) || !ws) return MC_ERR_NULLPTR;
  if (!al(x, 16) || !al(y, 16) || (saved && !al(saved, 256)) || !al(ws, 256)) return MC_ERR_ALIGN;
  const Dims D = dims_of(*shape);
  size_t need = 0;
  plan_ws(D, rc_mode, nullptr, &need);
  if (ws_bytes < need) return MC_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const Work W = plan_ws(D, rc_mode, ws, nullptr);
  const Saved S = plan_saved(D, rc_mode ? W.recompute_saved : saved, nullptr);
  if (cudaMemsetAsync(W.status, 0, kStatusBytes, st) != cudaSuccess) return MC_ERR_CUDA;
  return enqueue_forward(D, w, x, y, S, W, seq_parallel(*shape), st);
}

int mc_layer_backward(const mc_layer_shape* shape, const mc_layer_weights* w, const float* x,
                      const float* dy, const void* saved, float* dx, const mc_layer_grads* grads,
                      void* ws, size_t ws_bytes, void* stream) {
  MC_TRY(check_shape(shape));
  MC_TRY(check_weights(w));
  MC_TRY(check_grads(grads));
  const bool rc_mode = recompute(*shape);
  if (!x || !dy || (!saved && !rc_mode) || !dx || !ws) return MC_ERR_NULLPTR;
  if (!al(x, 16) || !al(dy, 16) || !al(dx, 16) || (saved && !al(saved, 256)) || !al(ws, 256))
    return MC_ERR_ALIGN;
  const Dims D = dims_of(*shape);
  size_t need = 0;
  plan_ws(D, rc_mode, nullptr, &need);
  if (ws_bytes < need) return MC_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const Work W = plan_ws(D, rc_mode, ws, nullptr);
  const Saved S = plan_saved(D, rc_mode ? W.recompute_saved : const_cast<void*>(saved), nullptr);
  if (rc_mode) {
    // Activation recomputation: rebuild F1..F7's activations from x.  The
    // recomputed y lands in dx1's buffer, which B3 overwrites later.
    MC_TRY(enqueue_forward(D, w, x, W.dx1, S, W, seq_parallel(*shape), st));
  }
  const int acc = (shape->flags & MC_ACCUMULATE_GRADS) ? 1 : 0;
  const int t = static_cast<int>(D.t);
  const int h = static_cast<int>(D.h);
  const mc_layer_grads& G = *grads;
  // Sequence-parallel mode: the per-token steps (the column sum of dy, both
  // LayerNorm backwards) and the two column-parallel input gradients (dln2,
  // dln1: a reduce-scatter of the partitions' partial sums) run per sequence
  // shard; the gradients of the sequence-sharded parameters (LayerNorm
  // gamma / beta, the row-parallel biases) are the shards' partial sums,
  // added in shard order (the first shard honours MC_ACCUMULATE_GRADS, the
  // rest add).  Weight gradients and the column-parallel products read all
  // shards' rows, which lie side by side: the all-gather.
  if (D.fp8) return enqueue_backward_fp8(D, w, x, dy, dx, G, S, W, acc, st);
  StageRanges R("mc_layer_backward");
  const Shards sh = shards_of(D, seq_parallel(*shape));
  auto shard_acc = [&](int64_t p) { return p == 0 ? acc : 1; };

  // B1  fc2: db2 = colsum(dy) (+ bf16 copy of dy as a GEMM operand),
  R.next("B1 fc2");
  //     dW2 = dy^T g, dhp = (dy W2) * gelu'(hp)
  for (int64_t p = 0; p < sh.n; ++p) {
    const int64_t r0 = p * sh.rows;
    MC_TRY(launch_colsum(dy + r0 * D.h, false, sh.rows, D.h, G.b_fc2, shard_acc(p),
                         W.dy16 + r0 * D.h, W.partials, W.status, st));
  }
  MC_TRY(launch_gemm(D.h, D.f, D.T, W.dy16, D.h, 1, S.g, D.f, 1, G.w_fc2, D.f, MC_EPI_STORE_F32,
                     nullptr, nullptr, 0, acc, 1, W.status, st));
  MC_TRY(launch_gemm(D.T, D.f, D.h, W.dy16, D.h, 0, w->w_fc2, D.f, 1, W.dhp, D.f, MC_EPI_GELU_BWD,
                     nullptr, S.hp, D.f, 0, 1, W.status, st));
  // B2  fc1: db1, dW1 = dhp^T ln2, dln2 = sum_p dhp_p W1_p (partition sum in
  R.next("B2 fc1");
  //     the accumulator; per shard in sequence-parallel mode)
  MC_TRY(launch_colsum(W.dhp, true, D.T, D.f, G.b_fc1, acc, nullptr, W.partials, W.status, st));
  MC_TRY(launch_gemm(D.f, D.h, D.T, W.dhp, D.f, 1, S.ln2, D.h, 1, G.w_fc1, D.h, MC_EPI_STORE_F32,
                     nullptr, nullptr, 0, acc, 1, W.status, st));
  for (int64_t p = 0; p < sh.n; ++p) {
    const int64_t r0 = p * sh.rows;
    MC_TRY(launch_gemm(sh.rows, D.h, D.f, W.dhp + r0 * D.f, D.f, 0, w->w_fc1, D.h, 1,
                       W.dln + r0 * D.h, D.h, MC_EPI_STORE_F32, nullptr, nullptr, 0, 0, t, W.status,
                       st));
  }
  // B3  LN2 backward: dx1 = dy + LN2^T(dln2); dgamma2, dbeta2; db_o = colsum(dx1)
  R.next("B3 LN2 backward");
  for (int64_t p = 0; p < sh.n; ++p) {
    const int64_t r0 = p * sh.rows;
    MC_TRY(launch_layernorm_backward(W.dln + r0 * D.h, S.x1 + r0 * D.h, S.mu2 + r0, S.rs2 + r0,
                                     w->ln2_g, dy + r0 * D.h, W.dx1 + r0 * D.h,
                                     W.dx1_16 + r0 * D.h, G.ln2_g, G.ln2_b, G.b_o, shard_acc(p),
                                     W.partials, sh.rows, h, W.status, st));
  }
  // B4  out-projection: dWo = dx1^T O, dO = dx1 Wo
  R.next("B4 out-projection");
  MC_TRY(launch_gemm(D.h, D.a, D.T, W.dx1_16, D.h, 1, S.o, D.a, 1, G.w_o, D.a, MC_EPI_STORE_F32,
                     nullptr, nullptr, 0, acc, 1, W.status, st));
  MC_TRY(launch_gemm(D.T, D.a, D.h, W.dx1_16, D.h, 0, w->w_o, D.a, 1, W.dO, D.a, MC_EPI_STORE_BF16,
                     nullptr, nullptr, 0, 0, 1, W.status, st));
  // B5  attention backward -> dQ | dK | dV
  R.next("B5 attention backward");
  MC_TRY(launch_attention_backward(S.qkv, S.o, S.lse, W.dO, W.dqkv, W.delta, static_cast<int>(D.b),
                                   static_cast<int>(D.s), static_cast<int>(D.H),
                                   static_cast<int>(D.d), W.status, st, W.ds));
  // B6  QKV: db_qkv, dWqkv = dqkv^T ln1, dln1 = sum_p dqkv_p Wqkv_p (per
  R.next("B6 QKV");
  //     shard in sequence-parallel mode)
  MC_TRY(launch_colsum(W.dqkv, true, D.T, 3 * D.a, G.b_qkv, acc, nullptr, W.partials, W.status, st));
  MC_TRY(launch_gemm(3 * D.a, D.h, D.T, W.dqkv, 3 * D.a, 1, S.ln1, D.h, 1, G.w_qkv, D.h,
                     MC_EPI_STORE_F32, nullptr, nullptr, 0, acc, 1, W.status, st));
  for (int64_t p = 0; p < sh.n; ++p) {
    const int64_t r0 = p * sh.rows;
    MC_TRY(launch_gemm(sh.rows, D.h, 3 * D.a, W.dqkv + r0 * 3 * D.a, 3 * D.a, 0, w->w_qkv, D.h, 1,
                       W.dln + r0 * D.h, D.h, MC_EPI_STORE_F32, nullptr, nullptr, 0, 0, t,
                       W.status, st));
  }
  // B7  LN1 backward: dx = dx1 + LN1^T(dln1); dgamma1, dbeta1
  R.next("B7 LN1 backward");
  for (int64_t p = 0; p < sh.n; ++p) {
    const int64_t r0 = p * sh.rows;
    MC_TRY(launch_layernorm_backward(W.dln + r0 * D.h, x + r0 * D.h, S.mu1 + r0, S.rs1 + r0,
                                     w->ln1_g, W.dx1 + r0 * D.h, dx + r0 * D.h, nullptr, G.ln1_g,
                                     G.ln1_b, nullptr, shard_acc(p), W.partials, sh.rows, h,
                                     W.status, st));
  }
  return MC_OK;
}

int mc_layer_device_status(const void* ws, void* stream) {
  if (!ws) return MC_ERR_NULLPTR;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int host[2] = {0, 0};
  if (cudaMemcpyAsync(host, ws, sizeof(host), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MC_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MC_ERR_CUDA;
  return host[0];
}

const char* mc_strerror(int code) {
  switch (code) {
    case MC_OK: return "ok";
    case MC_ERR_SHAPE: return "illegal shape (non-positive field or divisibility rule broken)";
    case MC_ERR_UNSUPPORTED: return "shape not supported by this build";
    case MC_ERR_NULLPTR: return "required pointer is NULL";
    case MC_ERR_ALIGN: return "pointer or leading dimension not aligned as required";
    case MC_ERR_WORKSPACE: return "workspace smaller than mc_layer_workspace_bytes()";
    case MC_ERR_CUDA: return "CUDA runtime error";
    case MC_ERR_DEVICE_TIMEOUT: return "device: bounded wait gave up";
    case MC_ERR_DEVICE_BOUNDS: return "device: index check failed";
    case MC_ERR_ARGUMENT: return "invalid argument";
    case MC_ERR_SCRATCH_LIMIT:
      return "problem exceeds the fixed device scratch of the allocation-free entry point";
    default: return "unknown status code";
  }
}

// ---- stage entry points -------------------------------------------------
int mc_layernorm_forward(const float* x, const uint16_t* gamma, const uint16_t* beta,
                         uint16_t* out, float* mean, float* rstd, int64_t rows, int32_t h,
                         int* status, void* stream) {
  return launch_layernorm_forward(x, gamma, beta, out, mean, rstd, rows, h, status,
                                  static_cast<cudaStream_t>(stream));
}

int mc_layernorm_backward(const float* dout, const float* x, const float* mean, const float* rstd,
                          const uint16_t* gamma, const float* resid, float* dx, uint16_t* dx_bf16,
                          float* dgamma, float* dbeta, float* colsum_dx, int accumulate,
                          float* partials, int64_t rows, int32_t h, int* status, void* stream) {
  return launch_layernorm_backward(dout, x, mean, rstd, gamma, resid, dx, dx_bf16, dgamma, dbeta,
                                   colsum_dx, accumulate, partials, rows, h, status,
                                   static_cast<cudaStream_t>(stream));
}

size_t mc_layernorm_backward_scratch_floats(int64_t rows, int32_t h) {
  return layernorm_backward_scratch_floats(rows, h);
}

int mc_gemm(int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda, int a_layout,
            const uint16_t* B, int64_t ldb, int b_layout, void* out, int64_t ldc, int epilogue,
            const uint16_t* bias, const void* aux, int64_t ldaux, int accumulate, int k_parts,
            int* status, void* stream) {
  return launch_gemm(M, N, K, A, lda, a_layout, B, ldb, b_layout, out, ldc, epilogue, bias, aux,
                     ldaux, accumulate, k_parts, status, static_cast<cudaStream_t>(stream));
}

int mc_attention_forward(const uint16_t* qkv, uint16_t* o, float* lse, int32_t micro_batch,
                         int32_t seq_len, int32_t heads, int32_t head_dim, int* status,
                         void* stream) {
  return launch_attention_forward(qkv, o, lse, micro_batch, seq_len, heads, head_dim, status,
                                  static_cast<cudaStream_t>(stream));
}

int mc_attention_backward(const uint16_t* qkv, const uint16_t* o, const float* lse,
                          const uint16_t* dout, uint16_t* dqkv, float* delta, int32_t micro_batch,
                          int32_t seq_len, int32_t heads, int32_t head_dim, int* status,
                          void* stream) {
  return launch_attention_backward(qkv, o, lse, dout, dqkv, delta, micro_batch, seq_len, heads,
                                   head_dim, status, static_cast<cudaStream_t>(stream));
}

int mc_build_features(void) {
  int f = 0;
#ifdef MC_DEBUG
  f |= MC_BUILD_DEBUG;
#endif
#ifdef MC_NVTX
  f |= MC_BUILD_NVTX;
#endif
  return f;
}

size_t mc_attention_backward_ws_bytes(int32_t micro_batch, int32_t seq_len, int32_t heads,
                                      int32_t head_dim) {
  if (micro_batch < 1 || seq_len < 1 || heads < 1 || (head_dim != 64 && head_dim != 128))
    return 0;
  return static_cast<size_t>(attention_ds_workspace_bytes(micro_batch, seq_len, heads));
}

int mc_attention_backward_ws(const uint16_t* qkv, const uint16_t* o, const float* lse,
                             const uint16_t* dout, uint16_t* dqkv, float* delta,
                             int32_t micro_batch, int32_t seq_len, int32_t heads,
                             int32_t head_dim, void* ds_workspace, size_t ds_workspace_bytes,
                             int* status, void* stream) {
  if (micro_batch < 1 || seq_len < 1 || heads < 1) return MC_ERR_SHAPE;
  if (!ds_workspace) return MC_ERR_NULLPTR;
  if (ds_workspace_bytes <
      static_cast<size_t>(attention_ds_workspace_bytes(micro_batch, seq_len, heads)))
    return MC_ERR_WORKSPACE;
  return launch_attention_backward(qkv, o, lse, dout, dqkv, delta, micro_batch, seq_len, heads,
                                   head_dim, status, static_cast<cudaStream_t>(stream),
                                   static_cast<uint8_t*>(ds_workspace));
}

}  // extern "C"
