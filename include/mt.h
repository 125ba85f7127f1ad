/* mt.h — C ABI of the layer-streamed training library (libmt.so).
 *
 * One training step of a Llama-style decoder on ONE GPU whose parameters all
 * live in pinned host memory ("MegaTrain: Full Precision Training of 100B+
 * Parameter Large Language Models on a Single GPU"):
 *  - the host owns parameters and gradients; the GPU holds an empty layer
 *    template bound to whatever weights stream in (section 核心方法);
 *  - forward: each layer's packed weights are copied H2D into one of two
 *    ping-pong device buffers while the previous layer computes; the residual
 *    stream is checkpointed every K layers (section 方法步骤详情, stage 1);
 *  - loss anchor: final norm, LM head and cross-entropy, head gradients
 *    offloaded (stage 2);
 *  - backward: per block of K layers, top block first, restore the block's
 *    checkpoint, recompute its forward, then back-propagate it layer by
 *    layer, copying each layer's gradients D2H on a separate stream
 *    (stage 3);
 *  - three CUDA streams (compute, weight-in, grad-out) ordered only by CUDA
 *    events: weight-ready, backward-done, buffer-free (section 技术新颖性).
 *
 * Conventions for every function below:
 *  - integer status returns: MT_OK (0) or a negative mt_status; no function
 *    aborts the process or lets a C++ exception cross this boundary;
 *  - a context is not thread-safe; use one per thread and per GPU;
 *  - pointers documented as "host" are CPU addresses, "device" are CUDA
 *    device addresses on the context's device; the caller keeps ownership of
 *    every buffer it passes in.
 */
#ifndef MT_H
#define MT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MT_ABI_VERSION 1

typedef enum {
  MT_OK = 0,
  MT_ERR_ARG = -1,         /* bad argument (null pointer, size out of range, token id >= vocab, ...) */
  MT_ERR_BUDGET = -2,      /* the device budget cannot hold the buffers this call needs */
  MT_ERR_NOT_PINNED = -3,  /* a host buffer is not page-locked CUDA host memory */
  MT_ERR_ALIGN = -4,       /* a host buffer is not 4096-byte aligned */
  MT_ERR_CUDA = -5,        /* a CUDA runtime/driver call failed (text in mt_last_error) */
  MT_ERR_TIMEOUT = -6,     /* a bounded wait (host event poll or device barrier) ran out */
  MT_ERR_STATE = -7,       /* call out of order (e.g. forward_backward before bind) */
  MT_ERR_UNSUPPORTED = -8, /* configuration outside what the kernels implement */
  MT_ERR_DEVICE = -9       /* a kernel reported an internal error through the device error word */
} mt_status;

typedef enum { MT_F32 = 0, MT_BF16 = 1, MT_FP8 = 2 } mt_dtype;

/* Model and capacity description.
 * Shapes: hidden h, n_heads query heads and n_kv_heads key/value heads of
 * head_dim d (n_heads % n_kv_heads == 0; query head j reads KV head
 * j / (n_heads / n_kv_heads)), SwiGLU FFN width ffn_dim, untied vocab.
 * Supported: h % 64 == 0, d in {16, 32, 64, 128}, for MT_BF16 params
 * ffn_dim % 8 == 0; any ffn_dim >= 1 for MT_F32 params; for MT_FP8 params
 * ffn_dim % 16 == 0.
 * max_batch * max_seq bounds the tokens of one call; max_K bounds the
 * checkpoint interval. param_dtype is the dtype of the host parameters that
 * will be bound. n_experts = top_k = expert_ffn = 0: dense SwiGLU FFN.
 * n_experts > 0: every layer's FFN is a mixture of experts (the MoE layer of
 * the streamed workloads, Qwen3-MoE style, e.g. Qwen3-235B: 128 experts,
 * top-8, expert width 1536; the pages name the model and its routing, not
 * the formulas): router logits r = m Wr^T from the FFN-norm output m,
 * p = softmax(r); the top_k experts of largest logit (equal: lower index)
 * with weights p_j / sum of the chosen p; each a SwiGLU MLP of width
 * expert_ffn; out = sum_j w_j y_j. No shared expert, no auxiliary loss.
 * Then ffn_dim = 0, n_experts a multiple of 8 in [8, 1024], top_k in
 * [1, min(32, n_experts)], expert_ffn % 32 == 0, and MT_BF16 or MT_FP8
 * params. */
typedef struct {
  int32_t n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn_dim, vocab;
  float rope_theta, norm_eps;
  int32_t max_batch, max_seq, max_K;
  int32_t param_dtype; /* mt_dtype */
  int32_t n_experts, top_k, expert_ffn;
  /* dtype of the host gradient buffer (same packed layout with that element
   * size): MT_F32 (0, the default) or MT_BF16 (gradients rounded to nearest
   * even on the device before they stream back: half the D2H bytes; the host
   * optimizer entry points take MT_F32 gradients only). */
  int32_t grad_dtype;
} mt_layer_cfg;

typedef struct mt_ctx mt_ctx;

/* Packed host parameter layout ("each layer's state packed into one
 * contiguous block aligned to a 4 KB page", MegaTrain, section 技术新颖性):
 *  unit 0        : embedding E[vocab, h]                       (tensor 0)
 *  unit 1..L     : one decoder layer each, tensors in order
 *                  0 w_attn_norm[h], 1 Wq[n_heads*d, h], 2 Wk[n_kv_heads*d, h],
 *                  3 Wv[n_kv_heads*d, h], 4 Wo[h, n_heads*d], 5 w_ffn_norm[h],
 *                  6 Wg[ffn, h], 7 Wu[ffn, h], 8 Wd[h, ffn]
 *                  (mixture of experts: 6 Wr[E, h], 7 Wgu[E, 2*Fe, h] with
 *                  each expert's gate rows then up rows, 8 Wd[E, h, Fe];
 *                  E = n_experts, Fe = expert_ffn)
 *  unit L+1      : 0 w_final_norm[h], 1 W_out[vocab, h]
 * Matrices are row-major [out, in] (y = x W^T). Every tensor starts on a
 * 256-byte boundary, every unit on a 4096-byte boundary. The gradient buffer
 * uses the same layout with grad_dtype elements (fp32 by default).
 *
 * MT_FP8 (opt-in weight-streaming variant, "use lower precision formats such
 * as FP8 to further reduce the PCIe bandwidth pressure", MegaTrain, section
 * 未来方向): every matrix tensor is its FP8 E4M3 codes, row-major [rows,
 * cols] (one byte each), followed at the next 16-byte boundary by one fp32
 * scale per row; the RMSNorm gains are fp32. The weight the step computes
 * with is bf16(e4m3(code) * scale) (fp32 product, then round to nearest
 * even), formed on the device for layers and head slices and on the host
 * for the embedding rows. Half the streamed bytes of bf16. Gradients stay
 * fp32 (or bf16) in their own layout; the host optimizer does not publish
 * FP8 (MT_ERR_UNSUPPORTED). */
size_t mt_packed_bytes(const mt_layer_cfg* cfg, mt_dtype dtype);

/* Byte offset and byte size of tensor `tensor` of unit `unit` in the packed
 * layout of `dtype`. Returns MT_ERR_ARG for an unknown unit/tensor. */
int mt_tensor_offset(const mt_layer_cfg* cfg, mt_dtype dtype, int unit, int tensor, size_t* off, size_t* bytes);

/* Quantise a packed model (layout of src_dtype, MT_F32 or MT_BF16) into the
 * MT_FP8 layout: per matrix row, scale = max|w| / 448 (1 for an all-zero
 * row) and each code the E4M3 value nearest to w / scale (ties to even,
 * saturating at 448); gains copied as fp32. dst: mt_packed_bytes(cfg,
 * MT_FP8) bytes. Host threads (0 = one per core); needs no GPU.
 * MT_ERR_ARG for a non-finite weight or bad arguments, MT_ERR_UNSUPPORTED for
 * mixture-of-experts layers. */
int mt_quantize_params_fp8(const mt_layer_cfg* cfg, const void* src, mt_dtype src_dtype, void* dst,
                           int32_t n_threads);

/* Device bytes a context needs for cfg (all K in [1, max_K], batches up to
 * max_batch x max_seq): two weight buffers, two gradient staging buffers,
 * checkpoints, one K-block of saved activations and fixed workspace.
 * Returns 0 if cfg is invalid. */
size_t mt_required_budget(const mt_layer_cfg* cfg);

/* Create a context on the current CUDA device. Allocates one device arena of
 * mt_required_budget(cfg) bytes (MT_ERR_BUDGET if that exceeds
 * device_budget_bytes) and three streams. *out is set only on MT_OK. */
int mt_create(const mt_layer_cfg* cfg, size_t device_budget_bytes, mt_ctx** out);

/* Same, but adopt a caller-owned device arena of device_budget_bytes
 * (256-byte aligned; e.g. a PyTorch tensor) and, if streams is non-null,
 * three caller-owned cudaStream_t values {compute, weight-in, grad-out}.
 * The caller keeps them alive until mt_destroy. */
int mt_create_ex(const mt_layer_cfg* cfg, size_t device_budget_bytes, void* device_arena, void* const* streams,
                 mt_ctx** out);

/* Bind the packed host parameters (layout above, dtype == cfg.param_dtype).
 * host_params must be page-locked CUDA host memory (MT_ERR_NOT_PINNED),
 * 4096-byte aligned (MT_ERR_ALIGN), at least mt_packed_bytes bytes, and stay
 * valid and unmodified during every mt_forward_backward call. No copy is
 * made; re-binding replaces the pointer. */
int mt_bind_host_params(mt_ctx* ctx, const void* host_params, mt_dtype dtype);

/* One training step: forward, loss, backward, all gradients to host.
 *  tokens, labels : host int32 [B, S], values in [0, vocab) (MT_ERR_ARG otherwise)
 *  B, S           : 1 <= B*S, B <= max_batch, S <= max_seq
 *  K              : checkpoint interval, 1 <= K <= min(n_layers, max_K); n_layers % K
 *                   may be nonzero (the top block is then partial)
 *  host_grad_out  : pinned host buffer of grad_dtype elements (fp32 by default),
 *                   mt_packed_bytes(cfg, grad_dtype) bytes,
 *                   4096-byte aligned; OVERWRITTEN with dLoss/dtheta in the
 *                   packed layout (embedding rows of unused tokens are 0; the
 *                   padding bytes between tensors are written as 0)
 *  loss_out       : host; Loss = mean over the B*S positions of
 *                   logsumexp(z_t) - z_t[label_t]
 * Synchronous: on return every gradient has landed. Results are bitwise
 * independent of K. */
int mt_forward_backward(mt_ctx* ctx, const int32_t* tokens, const int32_t* labels, int B, int S, int K,
                        float* host_grad_out, float* loss_out);

/* Per-step measurements of the last mt_forward_backward call (CUDA events). */
typedef struct {
  double step_ms;          /* first H2D issue to last D2H completion */
  double compute_busy_ms;  /* sum of compute-stream segment times */
  double h2d_ms, d2h_ms;   /* sum of copy durations on the weight-in / grad-out streams */
  double h2d_bytes, d2h_bytes;
  double h2d_hidden_frac;  /* fraction of H2D copy time overlapped by compute segments */
  double d2h_hidden_frac;
  int32_t n_h2d, n_d2h, n_units;
  int32_t timing_enabled;  /* 0: MT_TRACE=0 (no events); 1: per-unit events; 2: also per-kernel events */
  /* With MT_TRACE=2: summed device time and algorithmic work of a sample of
   * the GEMM launches (2*M*N*K flop each) and of the attention launches
   * (causal lower-triangle flop), one launch in MT_TRACE_SAMPLE (default 16)
   * bracketed with CUDA events on the compute stream; n_gemm/n_attn count the
   * sampled launches. */
  double gemm_ms, gemm_flop, attn_ms, attn_flop;
  int32_t n_gemm, n_attn;
  int32_t n_launches;      /* kernels launched by this step (all trace levels) */
  int32_t reserved;
  /* mt_train_step only: host wall time spent applying AdamW (summed over the
   * units, measured on the optimizer thread) and the part of it after the
   * step's last device work had finished (not hidden behind the step). */
  double optimizer_ms, optimizer_exposed_ms;
  /* Trace level >= 1: the weight copies (H2D) and gradient copies (D2H) of
   * the step by phase, [0] forward, [1] LM head (both passes), [2] block
   * recompute, [3] backward (the embedding rows are not counted): bytes and
   * summed copy durations. */
  double h2d_phase_bytes[4], h2d_phase_ms[4], d2h_phase_bytes[4], d2h_phase_ms[4];
  /* Trace level >= 1: rates of the step's individual weight copies (GB/s),
   * minimum, 10th, 50th and 90th percentile. */
  double h2d_copy_gbs_min, h2d_copy_gbs_p10, h2d_copy_gbs_p50, h2d_copy_gbs_p90;
  /* Host page toucher (env MT_PAGE_TOUCH = number of host threads, default
   * 4, 0 = off): before each weight copy, host threads read one byte of
   * every 4 KB page of its host range, two copies ahead of the copy stream,
   * so that pages whose host-side mapping lapsed are restored by the CPU
   * instead of stalling the copy engine page by page. Busiest thread's
   * reading time in the step (ms). */
  double page_touch_ms;
} mt_stats;
int mt_get_stats(const mt_ctx* ctx, mt_stats* out);

/* Mixture of experts: the experts chosen in the last completed step,
 * host_out[l][t][j] = the j-th choice (descending router logit) of layer l+1
 * for token t, n = n_layers * B*S * top_k int32 (else MT_ERR_ARG).
 * MT_ERR_STATE for a dense model or before the first step. Synchronous. */
int mt_get_routing(const mt_ctx* ctx, int32_t* host_out, size_t n);

/* Tracing of the following mt_forward_backward calls: level 0 none, 1
 * per-unit and per-copy events (overlap statistics; the default, also set
 * by env MT_TRACE), 2 additionally one GEMM/attention launch in `sample`
 * bracketed by events (kernel durations; this perturbs the step's own
 * timing, so measure step time at level 1). sample >= 1. */
int mt_set_tracing(mt_ctx* ctx, int level, int sample);

/* Copy-only replay of a step's weight stream: the host-to-device copies
 * mt_forward_backward issues for checkpoint interval K (every layer's packed
 * weights and every LM-head vocab slice, in the step's order, from the bound
 * host parameters into the two device weight buffers), issued back to back
 * on the weight-in stream with no kernels and no gradient copies beside
 * them. flags: 0 = no host threads either; MT_REPLAY_TOUCH = with the host
 * page toucher the step runs (one byte of every 4 KB page of each copy's
 * host range read by host threads two copies ahead of the copy stream).
 * Each copy is timed with CUDA events; copy_gbs_out (optional, max_copies
 * floats) receives the rate of each copy in GB/s, in order. A diagnostic of
 * the host link as the bound buffer sees it, apart from the step (MegaTrain,
 * section 技术新颖性: the transfer must keep up with the compute it hides
 * under). Synchronous; the weight buffers' contents are overwritten (the
 * next step reloads them anyway). MT_ERR_STATE without bound parameters;
 * MT_ERR_ARG for K outside [1, min(L, max_K)]. */
#define MT_REPLAY_TOUCH 1
typedef struct {
  int32_t n_copies, reserved;
  double bytes, ms;        /* total bytes and summed copy durations */
  int32_t host_numa_node;  /* cudaDevAttrHostNumaId of the context's device (-1: none) */
  int32_t reserved2;
  double touch_ms;         /* MT_REPLAY_TOUCH: busiest toucher thread's time spent reading */
} mt_replay_result;
int mt_replay_weight_stream(mt_ctx* ctx, int K, int flags, float* copy_gbs_out, int max_copies,
                            mt_replay_result* out);

/* Arena partition of a context (bytes). */
typedef struct {
  size_t total, weight_buffers, grad_buffers, checkpoints, block_activations, workspace;
} mt_memory_plan;
int mt_get_memory_plan(const mt_ctx* ctx, mt_memory_plan* out);

/* ---------------------------------------------------------------------------
 * Optimizer step on the host (MegaTrain, section 方法步骤详情, stage 4: the CPU
 * applies theta <- AdamUpdate(theta, grad, m, v) to the host-resident master
 * weights once their gradients have streamed back). The update is AdamW:
 *   m = beta1 m + (1 - beta1) g;  v = beta2 v + (1 - beta2) g^2
 *   theta -= lr (m / (1 - beta1^t) / (sqrt(v / (1 - beta2^t)) + eps) + weight_decay theta)
 * in fp32, on an fp32 master copy with fp32 moments (all three in the packed
 * layout of mt_packed_bytes(cfg, MT_F32)); the parameters the GPU streams
 * (bf16 or fp32 packed layout) receive the updated master rounded to their
 * type (bf16: round to nearest even). Padding between tensors is untouched.
 * ------------------------------------------------------------------------- */
typedef struct {
  float lr, beta1, beta2, eps, weight_decay;
} mt_adamw_cfg;

/* One AdamW update (step number `step` >= 1) of the packed units
 * [unit_begin, unit_end) (0 = embedding, 1..n_layers = layers, n_layers+1 =
 * final norm + head). master, m, v: host fp32 packed; grads: host fp32 packed
 * (the layout mt_forward_backward fills); params: host, dtype params_dtype.
 * n_threads host threads (0 = one per core). Pure host work: needs no GPU.
 * Errors: MT_ERR_ARG for null pointers, bad units or step < 1. */
int mt_adamw_update(const mt_layer_cfg* cfg, const mt_adamw_cfg* opt, int64_t step, int32_t unit_begin,
                    int32_t unit_end, float* master, float* m, float* v, const float* grads, void* params,
                    mt_dtype params_dtype, int32_t n_threads);

/* Attach optimizer state to ctx (host fp32 packed arrays as above; the caller
 * initialises master = the bound parameters in fp32 and m = v = 0, and keeps
 * them alive). The step counter starts at 1. */
int mt_bind_optimizer(mt_ctx* ctx, const mt_adamw_cfg* opt, float* master, float* m, float* v, int32_t n_threads);

/* mt_forward_backward followed by the AdamW update of every unit, each unit
 * updated by host threads as soon as its gradients have landed in
 * host_grad_out (head first, layers top-down as the backward produces them,
 * embedding last), overlapping the rest of the step. The GPU reads no unit's
 * parameters again in a step after its gradients land, so the next call sees
 * every unit updated (synchronous semantics: staleness 0). Returns when all
 * updates are applied. Device errors detected before a unit's update leave
 * that unit and the later ones untouched (MT_ERR_DEVICE). */
int mt_train_step(mt_ctx* ctx, const int32_t* tokens, const int32_t* labels, int B, int S, int K,
                  float* host_grad_out, float* loss_out);

/* Asynchronous form (RoundPipe's staleness-1 optimizer, one GPU): call k runs
 * step k on the GPU with the parameters updated through step k-2 while host
 * threads compute the update from step k-1's gradients (the previous call's
 * host_grad_out) into the fp32 master and moments; each unit's streamed copy
 * is rewritten only after step k's gradients of that unit have landed, when
 * the GPU reads that unit no more in step k (per-unit ordering instead of a
 * whole-model barrier). So after call k the streamed parameters hold the
 * update through step k-1. host_grad_out must not be the previous call's
 * buffer (alternate two pinned buffers): that one is still being read. The
 * first call applies no update. mt_optimizer_flush applies the pending
 * update (after the last call); mt_train_step refuses while one is pending.
 * A call that fails part-way leaves the pending update pending and records,
 * per unit, whether its update was already computed into the master and
 * moments and whether it was already published; the next call (or the
 * flush) completes each unit's update exactly once, never applying it
 * twice. */
int mt_train_step_async(mt_ctx* ctx, const int32_t* tokens, const int32_t* labels, int B, int S, int K,
                        float* host_grad_out, float* loss_out);
int mt_optimizer_flush(mt_ctx* ctx);

/* Text of the last error on ctx (never null; "" if none). */
const char* mt_last_error(const mt_ctx* ctx);

/* Destroy streams/events it created and free the arena it allocated. Null is ignored. */
void mt_destroy(mt_ctx* ctx);

/* Page-locked, 4096-byte aligned host memory (cudaHostAlloc); null on failure. */
void* mt_host_alloc(size_t bytes);
void mt_host_free(void* p);

/* Test hook: make the n-th (1-based) weight copy issue or host event wait of
 * the next mt_forward_backward calls on ctx fail as if the CUDA call had
 * failed (kind 1 = copy issue -> MT_ERR_CUDA) or timed out (kind 2 = wait ->
 * MT_ERR_TIMEOUT). kind 0 clears it. Host-side only: nothing is injected
 * into the GPU. */
int mt_debug_inject_fault(mt_ctx* ctx, int kind, int nth);

/* ---------------------------------------------------------------------------
 * Kernel-level entry points (the layer template's operations, exposed for
 * testing and measurement). All tensor pointers are DEVICE pointers on the
 * current device; `stream` is a cudaStream_t (null = legacy default stream).
 * Calls are asynchronous; errors in launch configuration are returned, and
 * device-side barrier timeouts are reported by mt_op_device_error.
 * bf16 tensors are raw 16-bit bfloat16 storage.
 * ------------------------------------------------------------------------- */

/* GEMM on the tensor cores, bf16 operands, fp32 accumulation.
 *  mode MT_GEMM_NT: C[M,N] = A[M,K] * B[N,K]^T   (forward: y = x W^T)
 *  mode MT_GEMM_NN: C[M,N] = A[M,K] * B[K,N]     (input gradient: dx = dy W)
 *  mode MT_GEMM_TN: C[M,N] = A[K,M]^T * B[K,N]   (weight gradient: dW = dy^T x)
 * lda/ldb are the row strides (elements) of A and B as stored; they must be
 * multiples of 8 and the base pointers 16-byte aligned.
 *  epi MT_EPI_BF16  : C bf16 = round(acc)
 *  epi MT_EPI_F32   : C fp32 = acc
 *  epi MT_EPI_F32_ADD: C fp32 = addend + acc (addend may equal C; row stride ldc)
 * ldc is C's row stride in elements. */
enum { MT_GEMM_NT = 0, MT_GEMM_NN = 1, MT_GEMM_TN = 2 };
enum { MT_EPI_BF16 = 0, MT_EPI_F32 = 1, MT_EPI_F32_ADD = 2 };
int mt_op_gemm(int mode, int epi, const void* A, const void* B, void* C, const void* addend, int M, int N, int K,
               int lda, int ldb, int ldc, void* stream);

/* RMSNorm forward: y[t] = bf16(x[t] * w * rstd[t]), rstd[t] = 1/sqrt(mean(x[t]^2) + eps).
 * x fp32 [T,h], w fp32 [h], y bf16 [T,h], rstd fp32 [T]. */
int mt_op_rmsnorm_fwd(const float* x, const float* w, void* y, float* rstd, int T, int h, float eps, void* stream);

/* RMSNorm backward with residual: dx = resid + rstd*(dy*w - xhat*mean(dy*w*xhat)),
 * xhat = x*rstd; dx fp32 (and bf16 copy dx_bf16 if non-null); dw fp32 [h] = sum_t dy*xhat
 * (fixed-order reduction; workspace fp32 of mt_op_rmsnorm_bwd_workspace(T,h) floats).
 * resid may be null (treated as 0) or equal dx. */
size_t mt_op_rmsnorm_bwd_workspace(int T, int h);
int mt_op_rmsnorm_bwd(const float* x, const float* w, const float* rstd, const float* dy, const float* resid,
                      float* dx, void* dx_bf16, float* dw, float* workspace, int T, int h, void* stream);

/* Allocation-free variant of mt_op_rmsnorm_bwd (same arguments and results,
 * minus the workspace). The paper has no counterpart: this entry point serves
 * callers that cannot allocate device memory where they call us, for example
 * code whose device memory is owned by another component's allocator, or
 * code that must not risk the implicit device synchronisation that
 * cudaMalloc/cudaFree can cause. Instead of a caller buffer it uses a
 * fixed 4 MiB array (1,048,576 floats) compiled into the library, which
 * every GPU that loads libmt.so holds until the process exits.
 *  - Limit: ceil(T/32) * h must be <= 1,048,576 (e.g. T = 8192 tokens at
 *    h = 4096); larger sizes return MT_ERR_BUDGET before anything runs.
 *  - The first call in each CUDA context (per device) looks up the array's
 *    device address (cudaGetSymbolAddress, with that device current) and
 *    caches it for that context; make that first call before any stream
 *    capture begins. A device reset or a new context gets a fresh lookup.
 *  - All calls share the one array and it keeps the last call's contents:
 *    calls whose executions overlap on the GPU (e.g. on two streams without
 *    ordering between them) race on it and give wrong results. The
 *    array needs no clearing: each call writes every entry it reads.
 *  - It calls no cudaMalloc, cudaFree or other allocating routine. */
int mt_op_rmsnorm_bwd_noalloc(const float* x, const float* w, const float* rstd, const float* dy, const float* resid,
                              float* dx, void* dx_bf16, float* dw, int T, int h, void* stream);

/* RoPE in place on bf16 x laid out [B*S, row_stride] where heads
 * [head0, head0 + n_heads) of width d start at column head0*d; dir +1
 * rotates by +pos*theta^(-2i/d) on the half-split pairs (i, i+d/2), -1 by the
 * opposite angle (the backward). table: device fp32 workspace of S*d floats
 * (overwritten with the cos/sin table). d must be a multiple of 8. */
int mt_op_rope(void* x, float* table, int B, int S, int row_stride, int head0, int n_heads, int d, float theta,
               int dir, void* stream);

/* The q|k|v projection with RoPE fused into the GEMM epilogue:
 * C[M,N] bf16 = A[M,K] W[N,K]^T where columns [0, rope_cols) (whole heads of
 * width d in {16,32,64,128}) are rotated by RoPE at position row % S before
 * the single rounding to bf16 (theta as in mt_op_rope). table: device fp32
 * workspace of S*d floats, overwritten. rope_cols must be a multiple of d. */
int mt_op_gemm_rope(const void* A, const void* W, void* C, int M, int N, int K, int lda, int ldb, int ldc,
                    float* table, int S, int d, float theta, int rope_cols, void* stream);

/* Gate-up projection with SwiGLU fused into the epilogue. W holds the gate
 * rows [0, F) and the up rows [u_off, u_off + F) of one [u_off + F, K]
 * matrix (bf16, row stride ldb). For X[M,K] (row stride lda) it writes
 *   gu[m, f] = bf16(g), gu[m, u_off + f] = bf16(u)   (gu row stride 2*u_off),
 *   act[m, f] = bf16(silu(g) * u)                     (act row stride u_off),
 * g = X Wg^T and u = X Wu^T in fp32; u_off must be a multiple of 8, >= F. */
int mt_op_gemm_swiglu(const void* X, const void* W, void* gu, void* act, int M, int F, int K, int lda, int ldb,
                      int u_off, void* stream);

/* Down-projection input gradient with the SwiGLU backward fused: dact =
 * dY[M,K] Wd where Wd is stored [K, F] (row stride ldb); with g, u read from
 * gu (layout as above), gu is overwritten in place by
 * dg = dact*u*silu'(g), du = dact*silu(g) (dact is never stored). */
int mt_op_gemm_swiglu_bwd(const void* dY, const void* Wd, void* gu, int M, int F, int K, int lda, int ldb, int u_off,
                          void* stream);

/* Causal GQA attention forward on bf16 q/k/v/o with row strides (elements):
 * q [B*S, ldq] heads at columns j*d, k/v [B*S, ldkv], o [B*S, ldo];
 * lse fp32 [B, n_heads, S] (natural-log logsumexp of the scaled scores). */
int mt_op_attention_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int S, int n_heads,
                        int n_kv_heads, int d, int ldq, int ldkv, int ldo, void* stream);

/* Attention backward: dq [B*S, ldq], dk/dv [B*S, ldkv] bf16 outputs
 * (overwritten); do_ bf16 [B*S, ldo]; workspace fp32 of
 * mt_op_attention_bwd_workspace(B,S,n_heads) floats, 16-byte aligned (it
 * receives per-row delta = rowsum(dO * O) and the log-sum-exp in log2 units,
 * S padded to a multiple of 128). Deterministic. */
size_t mt_op_attention_bwd_workspace(int B, int S, int n_heads);
int mt_op_attention_bwd(const void* q, const void* k, const void* v, const void* o, const void* do_, const float* lse,
                        void* dq, void* dk, void* dv, float* workspace, int B, int S, int n_heads, int n_kv_heads,
                        int d, int ldq, int ldkv, int ldo, void* stream);

/* mt_op_attention_bwd for q and k that were rotated by RoPE after the
 * projection: dq and dk are returned rotated back (the gradient w.r.t. the
 * unrotated projections), fused into the output stage. table: device fp32
 * workspace of S*d floats, overwritten. */
int mt_op_attention_bwd_rope(const void* q, const void* k, const void* v, const void* o, const void* do_,
                             const float* lse, void* dq, void* dk, void* dv, float* workspace, int B, int S,
                             int n_heads, int n_kv_heads, int d, int ldq, int ldkv, int ldo, float* table, float theta,
                             void* stream);

/* SwiGLU on gu bf16 [T, 2*ld] (gate columns [0,F), up columns [ld, ld+F)):
 * forward act bf16 [T, ld] = silu(g)*u (padding columns F..ld-1 written 0);
 * backward in place: gu <- (dact*u*silu'(g), dact*silu(g)). */
int mt_op_swiglu_fwd(const void* gu, void* act, int T, int F, int ld, void* stream);
int mt_op_swiglu_bwd(void* gu, const void* dact, int T, int F, int ld, void* stream);

/* Cross-entropy loss over logits produced by an NT product with a vocab
 * slice (never materialising [T, vocab]): see mt_op_lmhead_ce. Computes
 * loss = scale * sum_t (lse_t - z_t[label_t]) and dX [T,h] fp32 =
 * dz W_out, dW_out fp32 [V,h] = dz^T X, dz = scale*(softmax - onehot),
 * for X bf16 [T,h], W_out bf16 [V,h]; labels device int32 [T].
 * loss_dev is a device float. workspace bytes: mt_op_lmhead_ce_workspace. */
size_t mt_op_lmhead_ce_workspace(int T, int V, int h);
int mt_op_lmhead_ce(const void* X, const void* W, const int32_t* labels, float scale, float* dX, float* dW,
                    float* loss_dev, void* workspace, int T, int V, int h, void* stream);

/* Mixture-of-experts FFN forward on device buffers (the routed part of a
 * MoE layer, as the streamed step runs it): router logits r = m Wr^T, top_k
 * experts of largest logit per token (equal: lower index), weights
 * renormalised over the k, grouped SwiGLU expert GEMMs, and
 * out[t] = resid[t] + sum_j w_tj y_{e_tj}(m_t).
 *  m bf16 [T, h]; Wr bf16 [E, h]; Wgu bf16 [E, 2*Fe, h] (each expert's gate
 *  rows then up rows); Wd bf16 [E, h, Fe]; resid fp32 [T, h]; out fp32
 *  [T, h] (not aliasing resid); route int32 [T, top_k] receives the experts
 *  (descending logit). workspace: mt_op_moe_workspace(T, h, E, top_k, Fe)
 *  bytes of device memory, 256-byte aligned, owned by the caller.
 * Same limits as the MoE layer (h % 64 == 0, E % 8 == 0 and <= 1024,
 * top_k <= min(32, E), Fe % 32 == 0); MT_ERR_ARG otherwise. */
size_t mt_op_moe_workspace(int T, int h, int E, int top_k, int Fe);
int mt_op_moe_ffn_fwd(const void* m, const void* Wr, const void* Wgu, const void* Wd, const float* resid,
                      float* out, int32_t* route, void* workspace, int T, int h, int E, int top_k, int Fe,
                      void* stream);

/* Its backward: runs the forward of mt_op_moe_ffn_fwd on the same inputs
 * (same routing, written to route) and then, for dout = dLoss/d(out) fp32
 * [T, h]: dm fp32 [T, h] (gradient of m, the router's path included),
 * dWr fp32 [E, h], dWgu fp32 [E, 2*Fe, h], dWd fp32 [E, h, Fe] (all written;
 * zero for experts that received no token). workspace:
 * mt_op_moe_bwd_workspace(T, h, E, top_k, Fe) bytes, 256-byte aligned. */
size_t mt_op_moe_bwd_workspace(int T, int h, int E, int top_k, int Fe);
int mt_op_moe_ffn_bwd(const void* m, const void* Wr, const void* Wgu, const void* Wd, const float* dout, float* dm,
                      float* dWr, float* dWgu, float* dWd, int32_t* route, void* workspace, int T, int h, int E,
                      int top_k, int Fe, void* stream);

/* Device error word of the kernels (barrier timeouts etc.): returns and
 * clears it (0 = none). Synchronizes the device. */
int mt_op_device_error(void);

#ifdef __cplusplus
}
#endif
#endif /* MT_H */
