// Internal declarations shared by the library's translation units.
#pragma once
#include <cstddef>
#include <cstdint>

#include "../../include/mc_layer.h"

#ifdef __CUDACC__
#include <cuda.h>
#include <cuda_runtime.h>
#endif

#include <mutex>
#ifdef MC_NVTX
#include <nvtx3/nvToolsExt.h>
#endif

namespace mc {

#ifdef __CUDACC__
// Launches `kern` on `st` with programmatic stream serialisation, and in
// clusters of cluster_x CTAs along x when cluster_x > 1.  The kernel may then
// start (run its prologue) while the previous kernel on the stream finishes;
// every kernel of this library calls pdl_wait() before touching global memory.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t st, unsigned cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[2];
  unsigned n = 0;
  at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    at[n].id = cudaLaunchAttributeClusterDimension;
    at[n].val.clusterDim.x = cluster_x;
    at[n].val.clusterDim.y = 1;
    at[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = at;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}
#endif

// Status block at the start of a workspace: int[64] (256 bytes).
// status[0] = first error code recorded on the device, status[1] = where.
constexpr size_t kStatusBytes = 256;

// Where a device error was recorded (status[1]).
enum ErrorSite : int {
  kSiteGemmProducer = 1,
  kSiteGemmMma = 2,
  kSiteGemmEpilogue = 3,
  kSiteGemmDrain = 4,
  kSiteLayerNorm = 10,
  kSiteAttention = 20,
  kSiteSelfTest = 30,
};

// Row-major bf16 leading dimension bound used by the shape checks.
constexpr int kMaxLayerNormHidden = 16384;

// Grid cap of the LayerNorm-backward kernel; its column partial sums take
// 3 * min(rows, kLnBwdMaxBlocks) * h floats of scratch.
constexpr int kLnBwdMaxBlocks = 456;

// Row splits of the column-sum (bias gradient) kernel: enough for four
// blocks per SM, at least 64, at most kColsumMaxSplits.
constexpr int kColsumMinSplits = 64;
constexpr int kColsumMaxSplits = 512;

int num_sms();  // SM count of the current device (cached per device)

// Whole-matrix attention grids of at most four waves (tiles x heads x batch
// CTAs against the SMs) take every head's heaviest tiles first
// (attention_cta in ptx.cuh); the grid for either order.
inline bool attention_head_major(int64_t tiles, int64_t H, int64_t b) {
  return tiles * H * b <= 4ll * num_sms();
}
inline dim3 attention_grid(bool head_major, int tiles, int H, int b) {
  return head_major ? dim3(static_cast<unsigned>(H * b), static_cast<unsigned>(tiles), 1u)
                    : dim3(static_cast<unsigned>(tiles), static_cast<unsigned>(H),
                           static_cast<unsigned>(b));
}

#ifdef __CUDACC__
// Identity of the current device's context: (device ordinal, context id).
// The context id changes when the context is destroyed and re-created (e.g.
// by cudaDeviceReset), so set-up that belongs to a context is redone then.
cudaError_t current_context(int* dev, unsigned long long* ctx_id);

// One-time set-up that belongs to a device's context -- a kernel attribute,
// an occupancy figure, a symbol's device address: run with that device
// current, once per device and context, its status and value cached.
constexpr int kMaxDevices = 64;
struct PerDeviceInit {
  std::mutex mu;
  unsigned long long ctx[kMaxDevices] = {};  // 0: not set up yet
  cudaError_t err[kMaxDevices] = {};
  long long value[kMaxDevices] = {};
};

// Runs init(&value) the first time it is called for the current device's
// context; returns its status (and value) then and on every later call.
template <class F>
inline cudaError_t once_per_device(PerDeviceInit& s, F&& init, long long* value = nullptr) {
  int dev = 0;
  unsigned long long id = 0;
  cudaError_t e = current_context(&dev, &id);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(s.mu);
  if (s.ctx[dev] != id) {
    s.value[dev] = 0;
    s.err[dev] = init(&s.value[dev]);
    s.ctx[dev] = id;
  }
  if (value) *value = s.value[dev];
  return s.err[dev];
}
#endif

// NVTX ranges of the layer's launch sequence (compiled in with -DMC_NVTX):
// one range for the call and, inside it, one per stage, each closing when
// the next opens.  Host-side only; no effect on what is enqueued.
class StageRanges {
 public:
  explicit StageRanges(const char* call) {
#ifdef MC_NVTX
    nvtxRangePushA(call);
#else
    (void)call;
#endif
  }
  void next(const char* stage) {
#ifdef MC_NVTX
    if (open_) nvtxRangePop();
    nvtxRangePushA(stage);
    open_ = true;
#else
    (void)stage;
#endif
  }
  ~StageRanges() {
#ifdef MC_NVTX
    if (open_) nvtxRangePop();
    nvtxRangePop();
#endif
  }
  StageRanges(const StageRanges&) = delete;
  StageRanges& operator=(const StageRanges&) = delete;

 private:
  bool open_ = false;
};

#ifdef __CUDACC__
// bf16 tensor map with 128-byte swizzle and zero fill; strides_bytes has
// rank - 1 entries (dimension 0 is contiguous).
bool make_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box);

// Launchers (enqueue on `stream`; return MC_OK or MC_ERR_*).
int launch_layernorm_forward(const float* x, const uint16_t* gamma, const uint16_t* beta,
                             uint16_t* out, float* mean, float* rstd, int64_t rows, int h,
                             int* status, cudaStream_t stream);
int launch_layernorm_backward(const float* dout, const float* x, const float* mean,
                              const float* rstd, const uint16_t* gamma, const float* resid,
                              float* dx, uint16_t* dx_bf16, float* dgamma, float* dbeta,
                              float* colsum_dx, int accumulate, float* partials, int64_t rows,
                              int h, int* status, cudaStream_t stream);
size_t layernorm_backward_scratch_floats(int64_t rows, int h);

// Column sums over rows of a [rows, n] matrix (bf16 if in_bf16 else fp32);
// optionally writes a bf16 copy of an fp32 input.  out[n] = (accumulate ?
// out : 0) + sum.  `partials` holds kColsumMaxSplits * n floats.
int launch_colsum(const void* in, bool in_bf16, int64_t rows, int64_t n, float* out,
                  int accumulate, uint16_t* bf16_copy, float* partials, int* status,
                  cudaStream_t stream);

int launch_gemm(int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda, int a_layout,
                const uint16_t* B, int64_t ldb, int b_layout, void* out, int64_t ldc, int epi,
                const uint16_t* bias, const void* aux, int64_t ldaux, int accumulate, int k_parts,
                int* status, cudaStream_t stream);

// 8-bit floating-point GEMM: A [M, K], B [N, K] K-major bytes (format 0 =
// E4M3, 1 = E5M2), fp32 accumulation scaled by *a_scale_inv * *b_scale_inv,
// then the same fused epilogues as launch_gemm.
int launch_gemm_fp8(int64_t M, int64_t N, int64_t K, const uint8_t* A, int64_t lda, int a_format,
                    const uint8_t* B, int64_t ldb, int b_format, const float* a_scale_inv,
                    const float* b_scale_inv, void* out, int64_t ldc, int epi,
                    const uint16_t* bias, const void* aux, int64_t ldaux, int accumulate,
                    int k_parts, int* status, cudaStream_t stream);

// Per-tensor current scaling to 8-bit floats: amax of n fp32 (in_bf16 =
// false) or bf16 values, scale = fmax / amax, out = RNE_satfinite(x * scale);
// writes scale_inv[0] = 1 / scale.  `scratch` holds fp8_scratch_floats().
size_t fp8_scratch_floats();
int launch_fp8_quantize(const void* in, bool in_bf16, int64_t n, int format, uint8_t* out,
                        float* scale_inv, float* scratch, cudaStream_t stream);
// The same over a row-major [rows, cols] matrix (both multiples of 16),
// writing it as is (`out`) and/or transposed (`out_t`, [cols, rows]); either
// output may be NULL.
int launch_fp8_quantize_2d(const void* in, bool in_bf16, int64_t rows, int64_t cols, int format,
                           uint8_t* out, uint8_t* out_t, float* scale_inv, float* scratch,
                           cudaStream_t stream);

int launch_attention_forward(const uint16_t* qkv, uint16_t* o, float* lse, int b, int s, int H,
                             int d, int* status, cudaStream_t stream);
// The whole-sequence causal forward with 256-key blocks (one 128-query tile
// per CTA, 320 threads).
int launch_attention_forward_wide(const uint16_t* qkv, uint16_t* o, float* lse, int b, int s,
                                  int H, int d, int* status, cudaStream_t stream);
// Bytes of the dS^T tile workspace of the attention backward: one 32 KB
// bf16 tile per (query block, key block <= it) pair, per head and batch.
int64_t attention_ds_workspace_bytes(int64_t b, int64_t s, int64_t H);
// `ds_tiles` (16-byte aligned, attention_ds_workspace_bytes) selects the
// backward whose dK/dV kernel writes dS^T and whose dQ is dS K; NULL selects
// the one whose dQ kernel forms S and dP again.
int launch_attention_backward_tc(const uint16_t* qkv, const float* lse, const uint16_t* dout,
                                 uint16_t* dqkv, const float* delta, int b, int s, int H, int d,
                                 int* status, cudaStream_t stream, uint8_t* ds_tiles);
int launch_attention_backward(const uint16_t* qkv, const uint16_t* o, const float* lse,
                              const uint16_t* dout, uint16_t* dqkv, float* delta, int b, int s,
                              int H, int d, int* status, cudaStream_t stream,
                              uint8_t* ds_tiles = nullptr);

// delta[b, h, i] = rowsum(dO * O) for head h of token i (the backward's pre-pass).
int launch_attention_delta(const uint16_t* o, const uint16_t* dout, float* delta, int b, int s,
                           int H, int d, cudaStream_t stream);

// Rectangles of the causal score matrix for the context-parallel path: one
// chunk pair (query rows [q_base, q_base + q_len) against key rows
// [k_base, k_base + k_len), all multiples of 128, k_base <= q_base), and the
// accumulation modes of its query chunk (mode_q) and key chunk (mode_k).
// Each rectangle adds its share to running fp32 sums indexed by the
// absolute row; a mode says whether an earlier rectangle left one
// (kCpAccMerge) and whether this is the rows' last rectangle (kCpAccFinal),
// which writes the bf16 result instead.  One launch takes up to
// kCpMaxRects rectangles, no two of which share a query chunk (forward, dQ)
// or a key chunk (dK/dV), so that no running sum is touched twice:
//   forward: O [b, s, a] over the keys seen so far and its log2-sum-exp
//            [b, H, s], merged by the log-sum-exp rule; final: o and the
//            natural-log lse;
//   dkdv:    dK | dV [b, s, 2a] (dK scaled by 1/sqrt(d)) using the full lse
//            and delta; final: the dK, dV columns of dqkv.  It also writes
//            each rectangle's dS^T tiles to `ds_tiles`, rectangle after
//            rectangle in the order given, [b, H, nq, nk] x 32 KB each (nq
//            query blocks, nk key blocks), for
//   dq:      dQ [b, s, a] += dS K_j / sqrt(d) over those tiles (the same
//            rectangles in the same order); final: the dQ columns of dqkv.
constexpr int kCpAccMerge = 1;
constexpr int kCpAccFinal = 2;
constexpr int kCpMaxRects = 16;
struct CpRect {
  int q_base, q_len, k_base, k_len;
  int mode_q, mode_k;
};
// The dS^T tile bytes of rectangles[0, n).
int64_t attention_cp_tile_bytes(const CpRect* rects, int n, int64_t b, int64_t H);
int launch_attention_forward_parts(const uint16_t* qkv, uint16_t* o, float* lse, int b, int s,
                                   int H, int d, const CpRect* rects, int n, float* acc_o,
                                   float* acc_lse2, int* status, cudaStream_t stream);
int launch_attention_dkdv_parts(const uint16_t* qkv, const float* lse, const uint16_t* dout,
                                const float* delta, uint16_t* dqkv, int b, int s, int H, int d,
                                const CpRect* rects, int n, float* acc_dkv, uint8_t* ds_tiles,
                                int* status, cudaStream_t stream);
int launch_attention_dq_parts(const uint16_t* qkv, const uint8_t* ds_tiles, uint16_t* dqkv, int b,
                              int s, int H, int d, const CpRect* rects, int n, float* acc_dq,
                              int* status, cudaStream_t stream);
// Checks a launch's rectangles against the sequence (MC_OK or MC_ERR_ARGUMENT).
int check_cp_rects(const CpRect* rects, int n, int s);
#endif

}  // namespace mc
