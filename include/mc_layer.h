/*
 * mc_layer.h -- C ABI of a GB300 (sm_103a) library that runs one GPT pre-LN
 * transformer layer, forward and backward, in BF16 with FP32 accumulation.
 *
 * What is computed
 * ----------------
 *   x1 = x + OutProj(CausalAttention(LN1(x)))        (attention sub-block)
 *   y  = x1 + FC2(GeLU_tanh(FC1(LN2(x1))))            (MLP sub-block)
 * and, for an upstream gradient dy, dx and the gradients of all twelve
 * parameters.  LayerNorm uses the biased variance and eps = 1e-5; attention is
 * softmax(q k^T / sqrt(d)) v with key j visible to query i iff j <= i; no
 * dropout.
 *
 * Tensor-parallel split (Megatron tutorial cf-1.com/news/5344657, section 2.2
 * "张量并行：把一个大矩阵劈开"): the QKV projection is split across tp_parts
 * partitions by heads, the first MLP linear by columns and the second by
 * rows, so the out-projection and fc2 each produce one partial product per
 * partition that has to be summed (on a TP group of GPUs, an all-reduce).
 * Here the partitions are virtual and live on one GPU: each partition's
 * K-slice of a row-parallel GEMM accumulates into the same FP32 tensor-memory
 * accumulator, in partition order, and the epilogue adds the bias once after
 * the sum plus the residual.  The backward pass sums the column-parallel
 * input gradients (QKV and fc1 dgrad) the same way.
 * Divisibility (ai.lansai.wang/82226.html, section 并行度先做整数校验; tutorial
 * section 2.2): hidden, heads and ffn_hidden must divide by tp_parts.
 *
 * Layouts (all row-major, all pointers are device pointers unless stated)
 * -------------------------------------------------------------------------
 *   T = micro_batch * seq_len tokens, h = hidden, H = heads,
 *   d = head_dim (0 => h / H), a = H * d, f = ffn_hidden.
 *   x, y, dy, dx      float32 [T, h]  (token-major; token = b * seq_len + s)
 *   Weights (bf16 bit patterns, nn.Linear layout out x in, y = x W^T + b):
 *     w_qkv [3a, h] = [Wq; Wk; Wv], each block head-major (head k owns rows
 *     [k d, (k+1) d) of its block); b_qkv [3a]; w_o [h, a]; b_o [h];
 *     w_fc1 [f, h]; b_fc1 [f]; w_fc2 [h, f]; b_fc2 [h];
 *     ln{1,2}_g, ln{1,2}_b [h].
 *   Gradients: float32, same shapes as the weights.
 *
 * Ownership and ordering
 * ----------------------
 *   All memory is owned by the caller.  The library never allocates, frees or
 *   synchronises (except mc_layer_device_status, which synchronises `stream`).
 *   Every call enqueues kernels on `stream` (a cudaStream_t; NULL = legacy
 *   default stream) and returns without waiting.  `saved` is written by
 *   mc_layer_forward and read by mc_layer_backward; `x` and `saved` must not
 *   change in between.  `ws` is scratch; concurrent calls need distinct
 *   `saved`/`ws` buffers.  All pointers must be 16-byte aligned; `saved` and
 *   `ws` 256-byte aligned.
 *   Kernels are launched with programmatic stream serialisation: a library
 *   kernel may become resident while the kernel before it on `stream` is
 *   still running, but it touches no global memory until that kernel has
 *   completed and its writes are visible, so stream order holds for the
 *   caller's own kernels, copies and events as for ordinary launches.
 *
 * Errors
 * ------
 *   Every entry point returns MC_OK (0) or a negative code.  Shape, pointer,
 *   alignment and workspace-size errors are detected on the host before any
 *   launch and nothing is enqueued.  MC_ERR_CUDA reports a launch error.
 *   Device-side errors (a bounded wait that ran out, an out-of-range index
 *   caught by a kernel's own check) are recorded in a status word inside `ws`
 *   and read with mc_layer_device_status.
 */
#ifndef MC_LAYER_H_
#define MC_LAYER_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------- */
#define MC_OK 0
#define MC_ERR_SHAPE (-1)          /* a field <= 0, or a divisibility rule broken  */
#define MC_ERR_UNSUPPORTED (-2)    /* legal shape this build does not run          */
#define MC_ERR_NULLPTR (-3)        /* a required pointer is NULL                   */
#define MC_ERR_ALIGN (-4)          /* a pointer is not aligned as documented       */
#define MC_ERR_WORKSPACE (-5)      /* ws_bytes smaller than mc_layer_workspace_bytes */
#define MC_ERR_CUDA (-6)           /* a CUDA runtime call or launch failed         */
#define MC_ERR_DEVICE_TIMEOUT (-7) /* device: a bounded wait gave up               */
#define MC_ERR_DEVICE_BOUNDS (-8)  /* device: an index check of a debug build
                                      (-DMC_DEBUG) failed; the store is skipped */
#define MC_ERR_ARGUMENT (-9)       /* another invalid argument (e.g. an enum)      */
#define MC_ERR_SCRATCH_LIMIT (-10) /* problem larger than the fixed scratch of an
                                      allocation-free entry point                 */

/* shape flags */
#define MC_ACCUMULATE_GRADS 1u /* backward adds into the gradient buffers (+=)    */
/* Activation recomputation (the Megatron tutorial cf-1.com/news/5344657,
 * section 6.2, and its --recompute-method block): nothing is kept between
 * forward and backward -- mc_layer_saved_bytes() is 0 and `saved` may be
 * NULL; the forward's intermediates live in `ws` (which grows by the size of
 * the activations) and mc_layer_backward first re-runs the forward kernels
 * from x.  Results are identical to the default mode.  One `ws` can then be
 * shared by every layer of a stack run in sequence. */
#define MC_RECOMPUTE_ACTIVATIONS 2u
/* Sequence-parallel tensor parallelism (named with TP and EP in the Megatron
 * Core guide's record card and parallelism table): the tokens are cut into
 * tp_parts sequence shards of T / tp_parts consecutive tokens, and the
 * per-token work each tensor-parallel rank does on its own shard is launched
 * once per shard: LayerNorm forward and backward, the residual epilogues of
 * the out-projection and fc2, the column sum of dy.  The sum of the
 * row-parallel partials becomes a reduce-scatter: one out-projection / fc2
 * launch per shard writes that shard's rows, its accumulator summing every
 * partition's K slice; in the backward pass the QKV and fc1 input gradients
 * are reduce-scattered the same way.  QKV and fc1 (and every weight
 * gradient) read all shards' rows, which lie side by side in one buffer: the
 * all-gather.  Gradients of the sequence-sharded parameters (LayerNorm gamma
 * and beta, b_o, b_fc2) are the shards' partial sums added in shard order.
 * Contract: micro_batch * seq_len divides by tp_parts (MC_ERR_SHAPE
 * otherwise).  Results equal the default mode up to the order of those
 * fp32 sums. */
#define MC_SEQUENCE_PARALLEL 4u
/* FP8 "hybrid" GEMMs (the Megatron-Core listing, 混合精度: FP8 training on
 * Blackwell Ultra with E4M3 in the forward pass and E5M2 for gradients):
 * all twelve GEMMs of the layer run on 8-bit operands with fp32
 * accumulation (tcgen05 kind::f8f6f4).  Forward operands -- ln1, O, ln2, g
 * and the four weight matrices -- are E4M3; the gradient operands dy, dhp,
 * dx1 and dQ|dK|dV are E5M2.  Each operand tensor is quantised with
 * per-tensor current scaling (amax of the tensor as it stands, scale =
 * fmax / amax, as mc_fp8_quantize), once, into a row-major copy and, where a
 * product contracts over its rows, a transposed copy with the same scale;
 * the GEMM epilogue multiplies by the two inverse scales.  Everything else
 * (LayerNorm, attention, GeLU, bias and residual, the stored activations and
 * all gradients) is as in the default mode.  Requires micro_batch * seq_len
 * to be a multiple of 16 (MC_ERR_UNSUPPORTED otherwise) and is not combined
 * with MC_SEQUENCE_PARALLEL (MC_ERR_ARGUMENT).  mc_layer_saved_bytes and
 * mc_layer_workspace_bytes include the 8-bit copies. */
#define MC_FP8_HYBRID 8u

/* Attention backward without the dS tile workspace: the dQ kernel forms S
 * and dP a second time (seven 128 x 128 products per causal block pair
 * instead of five) and mc_layer_workspace_bytes leaves out the
 * mc_attention_backward_ws_bytes tiles, which grow as seq_len^2 (34.5 GB at
 * s = 32768 with 32 heads; ~550 GB at s = 131072).  For long sequences whose
 * tiles do not fit.  Results as the default mode up to the summation order
 * of S and dP inside the tensor core. */
#define MC_ATTN_DQ_RECOMPUTE 16u

typedef struct mc_layer_shape {
  int32_t micro_batch; /* b  (--micro-batch-size)               */
  int32_t seq_len;     /* s  (--seq-length), any value >= 1      */
  int32_t hidden;      /* h  (--hidden-size)                     */
  int32_t heads;       /* H  (--num-attention-heads)             */
  int32_t ffn_hidden;  /* f  (--ffn-hidden-size)                 */
  int32_t tp_parts;    /* t  (--tensor-model-parallel-size)      */
  int32_t head_dim;    /* 0 => hidden / heads; > 0 decouples a = heads * head_dim
                          from hidden (one tensor-parallel rank's shard run alone) */
  uint32_t flags;      /* MC_ACCUMULATE_GRADS | MC_RECOMPUTE_ACTIVATIONS |
                          MC_SEQUENCE_PARALLEL | MC_FP8_HYBRID |
                          MC_ATTN_DQ_RECOMPUTE, or 0 */
} mc_layer_shape;

/* bf16 parameters (uint16_t bit patterns), device pointers. */
typedef struct mc_layer_weights {
  const uint16_t *ln1_g, *ln1_b, *w_qkv, *b_qkv, *w_o, *b_o;
  const uint16_t *ln2_g, *ln2_b, *w_fc1, *b_fc1, *w_fc2, *b_fc2;
} mc_layer_weights;

/* fp32 parameter gradients, device pointers. */
typedef struct mc_layer_grads {
  float *ln1_g, *ln1_b, *w_qkv, *b_qkv, *w_o, *b_o;
  float *ln2_g, *ln2_b, *w_fc1, *b_fc1, *w_fc2, *b_fc2;
} mc_layer_grads;

/* Returns MC_OK when the shape is legal and runnable, MC_ERR_SHAPE when a
 * field is <= 0 or hidden/heads/ffn_hidden do not divide by tp_parts (or
 * hidden by heads when head_dim = 0), MC_ERR_UNSUPPORTED when head_dim is not
 * 64 or 128, or hidden, a / tp_parts or ffn_hidden / tp_parts is not a
 * multiple of 64.  Pure host function; needs no GPU. */
int mc_layer_check_shape(const mc_layer_shape* shape);

/* Bytes of the `saved` buffer (activations kept from forward to backward):
 * LN1/LN2 outputs and statistics, Q|K|V, attention output and log-sum-exp,
 * x1, fc1 pre-activation and GeLU output.  0 for an illegal shape and with
 * MC_RECOMPUTE_ACTIVATIONS. */
size_t mc_layer_saved_bytes(const mc_layer_shape* shape);

/* Bytes of the `ws` scratch buffer, including the 256-byte device status
 * block at its start and (unless MC_ATTN_DQ_RECOMPUTE) the attention
 * backward's dS tiles (mc_attention_backward_ws_bytes).  0 for an illegal
 * shape. */
size_t mc_layer_workspace_bytes(const mc_layer_shape* shape);

/* Forward pass.  x [T, h] fp32 in, y [T, h] fp32 out; fills `saved`.
 * Clears the device status word in `ws` first. */
int mc_layer_forward(const mc_layer_shape* shape, const mc_layer_weights* w, const float* x,
                     float* y, void* saved, void* ws, size_t ws_bytes, void* stream);

/* Backward pass.  dy [T, h] fp32 in; dx [T, h] fp32 out; parameter
 * gradients written (or accumulated with MC_ACCUMULATE_GRADS) into `grads`.
 * Reads `saved` from the matching forward call.  dx may alias dy. */
int mc_layer_backward(const mc_layer_shape* shape, const mc_layer_weights* w, const float* x,
                      const float* dy, const void* saved, float* dx, const mc_layer_grads* grads,
                      void* ws, size_t ws_bytes, void* stream);

/* Synchronises `stream` and returns the device status recorded in `ws` by
 * the kernels since the last forward call: MC_OK, MC_ERR_DEVICE_TIMEOUT or
 * MC_ERR_DEVICE_BOUNDS (or MC_ERR_CUDA if the synchronisation fails). */
int mc_layer_device_status(const void* ws, void* stream);

/* What this build of the library was compiled with, a bit mask:
 * MC_BUILD_DEBUG (1) -- the -DMC_DEBUG index checks before every global
 * store; MC_BUILD_NVTX (2) -- NVTX ranges around the layer's calls and
 * each of their stages (F1..F7, B1..B7), for a profiler's timeline or its
 * range filters. */
#define MC_BUILD_DEBUG 1
#define MC_BUILD_NVTX 2
int mc_build_features(void);

/* Static, human-readable text for a status code. */
const char* mc_strerror(int code);

/* ---- stage entry points ---------------------------------------------------
 * The same kernels the layer calls use, exposed one stage at a time so each
 * can be checked alone.  `status` is a device int[64] (256 bytes) that the
 * kernels record device-side errors into; it may be NULL. */

/* LayerNorm forward over rows of x [rows, h] fp32: out = (x - mean) * rstd *
 * gamma + beta as bf16 [rows, h]; mean and rstd fp32 [rows] (may be NULL).
 * Biased variance, eps = 1e-5.  h must be a multiple of 8 and <= 16384. */
int mc_layernorm_forward(const float* x, const uint16_t* gamma, const uint16_t* beta,
                         uint16_t* out, float* mean, float* rstd, int64_t rows, int32_t h,
                         int* status, void* stream);

/* LayerNorm backward: dx = resid + rstd * (g - mean(g) - xhat * mean(g * xhat))
 * with g = dout * gamma and xhat = (x - mean) * rstd; dx fp32 [rows, h]
 * (resid may be NULL, dx may alias resid).  If dx_bf16 is not NULL, a bf16
 * copy of dx is written too.  Column sums over rows of dout * xhat, dout and
 * (if colsum_dx is not NULL) dx are written to dgamma, dbeta, colsum_dx
 * (fp32 [h]; added to their contents when `accumulate` is non-zero).
 * `partials` is fp32 scratch of mc_layernorm_backward_scratch_floats(rows, h)
 * floats. */
int mc_layernorm_backward(const float* dout, const float* x, const float* mean, const float* rstd,
                          const uint16_t* gamma, const float* resid, float* dx, uint16_t* dx_bf16,
                          float* dgamma, float* dbeta, float* colsum_dx, int accumulate,
                          float* partials, int64_t rows, int32_t h, int* status, void* stream);
size_t mc_layernorm_backward_scratch_floats(int64_t rows, int32_t h);

/* GEMM on the tcgen05 tensor cores: C[M, N] = sum_k A[m, k] B[n, k] (fp32
 * accumulation), then an epilogue.
 *   a_layout 0: A stored [M, K] (row stride lda); 1: A stored [K, M] (lda).
 *   b_layout 0: B stored [N, K] (row stride ldb); 1: B stored [K, N] (ldb).
 * Epilogues (out row stride ldc, aux row stride ldaux):
 *   MC_EPI_STORE_F32        out fp32  = acc (+ out if accumulate)
 *   MC_EPI_STORE_BF16       out bf16  = acc
 *   MC_EPI_BIAS_BF16        out bf16  = acc + bias[n]
 *   MC_EPI_BIAS_GELU        aux bf16  = acc + bias[n];  out bf16 = gelu_tanh(acc + bias[n])
 *   MC_EPI_BIAS_RESID_F32   out fp32  = acc + bias[n] + resid[m, n] (resid fp32, ldaux)
 *   MC_EPI_GELU_BWD         out bf16  = acc * gelu_tanh'(aux[m, n]) (aux bf16)
 * `k_parts` states that the K range is k_parts equal partitions (a
 * row-parallel product: partition p owns k in [p K/k_parts, (p+1) K/k_parts)).
 * It is only checked (k_parts >= 1 and dividing K, else MC_ERR_ARGUMENT):
 * the MMAs walk K in order into one fp32 tensor-memory accumulator, so
 * partition p's K slice is the p-th contiguous run of that walk and the
 * epilogue sees the partitions' sum, taken in partition order.  The sum of
 * partials is this in-accumulator accumulation, not a separate pass.
 * Requirements: M >= 1, N and K multiples of 64 (K >= 64 unless a_layout = 1,
 * where K is the token count and may be any value >= 1), 16-byte aligned
 * pointers and leading dimensions that are multiples of 8 elements. */
#define MC_EPI_STORE_F32 0
#define MC_EPI_STORE_BF16 1
#define MC_EPI_BIAS_BF16 2
#define MC_EPI_BIAS_GELU 3
#define MC_EPI_BIAS_RESID_F32 4
#define MC_EPI_GELU_BWD 5
int mc_gemm(int64_t M, int64_t N, int64_t K, const uint16_t* A, int64_t lda, int a_layout,
            const uint16_t* B, int64_t ldb, int b_layout, void* out, int64_t ldc, int epilogue,
            const uint16_t* bias, const void* aux, int64_t ldaux, int accumulate, int k_parts,
            int* status, void* stream);

/* Causal flash attention forward over a packed Q|K|V tensor qkv [T, 3a] bf16
 * (token-major; head k of Q at columns [k d, (k+1) d), of K at a + k d, of V
 * at 2a + k d).  Writes o [T, a] bf16 (heads in order) and lse [b, H, s]
 * fp32 (natural log of the softmax denominator, scores scaled by 1/sqrt(d)).
 * head_dim must be 64 or 128. */
int mc_attention_forward(const uint16_t* qkv, uint16_t* o, float* lse, int32_t micro_batch,
                         int32_t seq_len, int32_t heads, int32_t head_dim, int* status,
                         void* stream);

/* Causal flash attention backward: from qkv, o, lse and dO [T, a] bf16 writes
 * dqkv [T, 3a] bf16 (dQ | dK | dV in the qkv layout).  `delta` is fp32
 * scratch [b, H, s] (receives rowsum(dO * O)). */
int mc_attention_backward(const uint16_t* qkv, const uint16_t* o, const float* lse,
                          const uint16_t* dout, uint16_t* dqkv, float* delta, int32_t micro_batch,
                          int32_t seq_len, int32_t heads, int32_t head_dim, int* status,
                          void* stream);

/* Bytes of the dS workspace of mc_attention_backward_ws: one 32 KB bf16
 * tile per pair (query block i, key block j <= i) of 128 rows each, per head
 * and batch: micro_batch * heads * n (n + 1) / 2 * 32768 with n =
 * ceil(seq_len / 128) (1.1 GB at s = 4096 with 64 heads, 34.5 GB at
 * s = 32768 with 32 heads).  0 for an invalid shape. */
size_t mc_attention_backward_ws_bytes(int32_t micro_batch, int32_t seq_len, int32_t heads,
                                      int32_t head_dim);

/* mc_attention_backward with a dS workspace (device memory of
 * mc_attention_backward_ws_bytes, 16-byte aligned; too small ->
 * MC_ERR_WORKSPACE): the dK/dV kernel writes dS^T = P^T (dP^T - delta) as
 * bf16 tiles there and dQ = dS K / sqrt(d) is a product over those tiles,
 * instead of a kernel that forms S and dP a second time.  The backward the
 * layer calls.  Same results as mc_attention_backward up to the summation
 * order of S and dP inside the tensor core (dQ is formed from the dK/dV
 * kernel's dS). */
int mc_attention_backward_ws(const uint16_t* qkv, const uint16_t* o, const float* lse,
                             const uint16_t* dout, uint16_t* dqkv, float* delta,
                             int32_t micro_batch, int32_t seq_len, int32_t heads,
                             int32_t head_dim, void* ds_workspace, size_t ds_workspace_bytes,
                             int* status, void* stream);

/* Allocation-free variant of mc_attention_backward.  The pages have no
 * counterpart to this entry point; it exists for callers that cannot allocate
 * device memory themselves -- for example a plugin whose host framework
 * forbids cudaMalloc while it runs, or a process whose device memory is
 * already fully reserved by another allocator -- and so cannot supply the
 * `delta` scratch buffer.  Same arguments and results as
 * mc_attention_backward without `delta`: the rowsum(dO * O) scratch is a fixed
 * 4 MiB array inside the library (micro_batch * heads * seq_len <= 1,048,576;
 * larger problems return MC_ERR_SCRATCH_LIMIT before anything is enqueued).
 * That array is held on every GPU that loads the library until the process
 * exits.  The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current, and looks it up again if
 * the device's context was re-created (cudaDeviceReset); make that first call
 * before any stream capture.  This entry point calls no cudaMalloc, cudaFree
 * or allocating library routine.  All calls share the array and it keeps the
 * last call's contents (each call overwrites every element it reads); calls
 * whose kernels overlap on the GPU, e.g. on different streams, race on it. */
int mc_attention_backward_noalloc(const uint16_t* qkv, const uint16_t* o, const float* lse,
                                  const uint16_t* dout, uint16_t* dqkv, int32_t micro_batch,
                                  int32_t seq_len, int32_t heads, int32_t head_dim, int* status,
                                  void* stream);

/* Failure-detection self-test: one kernel waits on an mbarrier that nothing
 * arrives on, bounded by timeout_ns (1 us to 100 ms, else MC_ERR_ARGUMENT),
 * exactly as every wait of the library is bounded.  When the limit passes it
 * records MC_ERR_DEVICE_TIMEOUT in status[0] and the site code 30 in
 * status[1] (status: int[64] device memory, zeroed by the caller) and
 * returns; the context stays usable.  No fault, trap or hang is involved. */
int mc_selftest_wait_timeout(int64_t timeout_ns, int* status, void* stream);

/* Index-check self-test: one thread checks 0 <= index < extent with the
 * check a debug build of this library (compiled with -DMC_DEBUG) runs before
 * every global store of its kernels, and writes buf[index] = 1 only if the
 * check passes; otherwise it records MC_ERR_DEVICE_BOUNDS in status[0] and
 * the site code 30 in status[1], and touches nothing.  buf: int device
 * memory of `extent` elements (NULL -> MC_ERR_NULLPTR; extent < 1 ->
 * MC_ERR_ARGUMENT).  No fault is involved: an out-of-range index is never
 * dereferenced. */
int mc_selftest_bounds_check(int64_t index, int64_t extent, int* buf, int* status, void* stream);

/* ---- 8-bit floating-point GEMMs (the Megatron-Core listing, 混合精度:
 * FP8 / FP4 training on Blackwell Ultra, --fp8-format hybrid = E4M3 forward,
 * E5M2 gradients).  Formats: 0 = E4M3 (largest finite 448), 1 = E5M2
 * (57344), OCP 8-bit floating point.  The pages give no scaling recipe; the
 * one implemented is per-tensor current scaling (below). */

/* Floats of device scratch that mc_fp8_quantize needs. */
size_t mc_fp8_scratch_floats(void);

/* Quantises n values of `in` (fp32, or bf16 when in_bf16 != 0; 16-byte
 * aligned) to `out` (n bytes, 8-byte aligned): amax = max |x|, scale =
 * fmax / amax (fp32 division; 1 when amax is 0), out = round-to-nearest-even
 * of x * scale (fp32 product) saturated to +-fmax; writes the device scalar
 * *scale_inv = 1 / scale.  Enqueued on `stream`; deterministic. */
int mc_fp8_quantize(const void* in, int32_t in_bf16, int64_t n, int32_t format, uint8_t* out,
                    float* scale_inv, float* scratch, int* status, void* stream);

/* The same quantisation of a row-major [rows, cols] matrix (in: fp32, or
 * bf16 when in_bf16 != 0; rows and cols multiples of 16, pointers 16-byte
 * aligned), writing the bytes as is to `out` ([rows, cols]) and/or
 * transposed to `out_t` ([cols, rows]); either output may be NULL.  One
 * scale for both.  The transposed copy is the K-major operand of a product
 * that contracts over the matrix's rows (a weight gradient contracts over
 * tokens; an input gradient reads the weight transposed).  `scratch` as for
 * mc_fp8_quantize; MC_ERR_SHAPE for dimensions that are not multiples of
 * 16. */
int mc_fp8_quantize_2d(const void* in, int32_t in_bf16, int64_t rows, int64_t cols,
                       int32_t format, uint8_t* out, uint8_t* out_t, float* scale_inv,
                       float* scratch, void* stream);

/* out = epilogue((A B^T) * *a_scale_inv * *b_scale_inv) with A [M, K] and
 * B [N, K] row-major 8-bit floats (K contiguous; lda, ldb multiples of 16),
 * fp32 accumulation on the tensor cores (tcgen05 kind::f8f6f4, SM pairs for
 * large problems).  Epilogues, bias / aux / accumulate / k_parts and errors as
 * mc_gemm; K a multiple of 16 (a ragged last 128-wide block reads zeros). */
int mc_gemm_fp8(int64_t M, int64_t N, int64_t K, const uint8_t* A, int64_t lda, int32_t a_format,
                const uint8_t* B, int64_t ldb, int32_t b_format, const float* a_scale_inv,
                const float* b_scale_inv, void* out, int64_t ldc, int32_t epilogue,
                const uint16_t* bias, const void* aux, int64_t ldaux, int32_t accumulate,
                int32_t k_parts, int* status, void* stream);

/* ---- Context-parallel causal attention (virtual CP partitions on one GPU).
 *
 * The pages (the Megatron Core guide: parallelism table and the section on
 * proving semantics unchanged; the Megatron-Core listing: dynamic context
 * parallelism) describe context parallelism as splitting the sequence
 * dimension of inputs and activations across ranks, attention still needing
 * every earlier token's K and V from the other ranks, and masks checked
 * across sequence lengths.  Here the sequence of every micro-batch is cut
 * into 2 * cp_parts chunks of c = seq_len / (2 cp_parts) tokens; virtual rank
 * r owns chunks r and 2 cp_parts - 1 - r (queries, keys and values), which
 * gives every rank the same causal work.  In ring step t rank r holds the K/V
 * chunks of rank (r - t) mod cp_parts and computes, for each of its query
 * chunks i and each held key chunk j <= i, the partial attention of chunk i
 * over chunk j (causal mask inside the diagonal pair).  Each partial is
 * folded into running fp32 results as soon as it is computed: a query
 * chunk's O and log-sum-exp by the log-sum-exp rule, its dQ and a key
 * chunk's dK, dV by addition; a chunk's last pair writes the bf16 result.
 * On one GPU the K/V exchange is the read of the other chunk's rows, and
 * the ranks of a ring step run together: one launch per sub-step (every
 * rank's k-th pair of the step), on `stream`, in schedule order.  Results equal mc_attention_forward / _backward up to the fp32
 * rounding of the merges and sums (to the bit for a chunk with one pair:
 * O, lse and dQ of chunk 0, dK and dV of the last chunk).
 *
 * Requirements: 1 <= cp_parts <= 256 (MC_ERR_UNSUPPORTED above), seq_len a
 * multiple of 256 * cp_parts,
 * head_dim 64 or 128; the caller-owned workspace of
 * mc_attention_cp_workspace_bytes bytes (16-byte aligned) holds the running
 * sums (micro_batch x seq_len x 3a floats) and the bf16 dS^T tiles of one
 * sub-step (up to cp_parts chunk pairs of micro_batch x heads x (c / 128)^2
 * tiles of 128 x 128); its size does not grow with cp_parts.  Forward and backward may share it; it must
 * not be shared with a concurrent call.  Errors as mc_attention_forward,
 * plus MC_ERR_SHAPE for an unsupported seq_len / cp_parts pair and
 * MC_ERR_WORKSPACE for a short workspace. */

/* The pairs (query chunk, key chunk) that virtual rank `rank` computes in
 * ring step `step`: writes up to 4 pairs as pairs[2k] = query chunk,
 * pairs[2k + 1] = key chunk and returns their number, or MC_ERR_ARGUMENT.
 * Host only; every pair j <= i of the 2 cp_parts chunks occurs exactly once
 * over all ranks and steps. */
int mc_cp_schedule(int32_t cp_parts, int32_t rank, int32_t step, int32_t* pairs);

/* The launch plan of mc_attention_forward_cp / _backward_cp.  Host only.
 * Every chunk pair of the schedule in launch order: sub-step k of ring
 * step t is one launch of every rank's k-th pair of that step.  Each pair
 * writes five entries: the index of its launch, its query chunk i, its key
 * chunk j, and the accumulation modes of i and j (bit 0: add to a running
 * sum left by an earlier pair of that chunk; bit 1: the chunk's last pair,
 * which writes the result).  No launch holds two pairs of one query chunk
 * or of one key chunk.  Returns the number of pairs, cp_parts (2 cp_parts
 * + 1); MC_ERR_ARGUMENT for cp_parts outside [1, 256] or a null `entries`;
 * MC_ERR_WORKSPACE when max_pairs is smaller. */
int mc_cp_launch_plan(int32_t cp_parts, int32_t* entries, int32_t max_pairs);

size_t mc_attention_cp_workspace_bytes(int32_t micro_batch, int32_t seq_len, int32_t heads,
                                       int32_t head_dim, int32_t cp_parts);

/* Same results and layouts as mc_attention_forward (o bf16, lse fp32). */
int mc_attention_forward_cp(const uint16_t* qkv, uint16_t* o, float* lse, int32_t micro_batch,
                            int32_t seq_len, int32_t heads, int32_t head_dim, int32_t cp_parts,
                            void* workspace, size_t workspace_bytes, int* status, void* stream);

/* Same results and layouts as mc_attention_backward: each pair's dQ, dK, dV
 * use the merged lse and delta = rowsum(dO * O); a chunk's dQ is the sum of
 * its pairs', a chunk's dK and dV the sum over the query chunks that saw it,
 * each summed in fp32 in schedule order (deterministic). */
int mc_attention_backward_cp(const uint16_t* qkv, const uint16_t* o, const float* lse,
                             const uint16_t* dout, uint16_t* dqkv, float* delta,
                             int32_t micro_batch, int32_t seq_len, int32_t heads,
                             int32_t head_dim, int32_t cp_parts, void* workspace,
                             size_t workspace_bytes, int* status, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MC_LAYER_H_ */
