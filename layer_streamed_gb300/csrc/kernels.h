// Internal launch interface of the layer-template kernels (host side).
// Every launcher returns 0 on success and -1 on a bad argument or a failed
// launch; none allocates memory.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mt {

// Number of kernels launched by the launchers below (host-side counter,
// read by the runtime to report launches per step).
extern long g_kernel_launches;
inline void count_launches(int n) { g_kernel_launches += n; }

enum { GEMM_NT = 0, GEMM_NN = 1, GEMM_TN = 2 };
enum { EPI_BF16 = 0, EPI_F32 = 1, EPI_F32_ADD = 2 };

struct GemmParams {
  int M, N, K;
  int epi;
  void* C;
  const void* addend;  // EPI_F32_ADD: C = addend + acc (same row stride)
  int ldc;
  int vec;      // set by gemm_bf16: 1 if C rows allow 16-byte stores
  int group_m;  // set by gemm_bf16: row-blocks per tile group (L2 reuse)
  // Optional RoPE in the bf16 epilogue: columns [0, rope_cols) form heads of
  // width rope_d rotated by the (cos, sin) table [rope_S][rope_d/2] at
  // position row % rope_S before the single rounding to bf16.
  const float2* rope_tab = nullptr;
  int rope_S = 0, rope_d = 0, rope_cols = 0;
  // Gated (SwiGLU) forward, mode NT only: each 256-wide tile is rows
  // [f0, f0+128) of B (gate) and rows [u_off + f0, u_off + f0 + 128) (up);
  // N counts features. The epilogue writes g to C column f, u to C column
  // u_col + f (bf16) and act = silu(g) * u to act[row * ld_act + f].
  int gated = 0, u_off = 0, u_col = 0, ld_act = 0;
  uint16_t* act = nullptr;
  // SwiGLU backward epilogue (mode NN, bf16 C unused): the accumulator is
  // dact; g, u are read from gu (row stride ld_gu, up at column u_col) and
  // replaced in place by dg = dact*u*silu'(g), du = dact*silu(g).
  int swiglu_bwd = 0, ld_gu = 0;
  uint16_t* gu = nullptr;
  // Grouped form (mixture-of-experts products; one launch for all experts,
  // single-CTA kernel). grp_seg[0..grp_E] (device): expert e owns rows
  // [grp_seg[e], grp_seg[e+1]) of the routed-row operands, each segment a
  // multiple of 128 rows (padding rows hold zeros).
  //  NT, NN: M counts all padded rows; grp_tile_e[m / 128] (device) is the
  //   expert owning 128-row block m (-1: unused, skipped); expert e's B starts
  //   e * grp_b_rows rows further (NT: rows of B, NN: K rows of B).
  //  TN: expert e's M x N output is rows [e*M, (e+1)*M) of C, its reduction
  //   runs over its own segment (K = all padded rows); an empty segment
  //   gives zeros.
  const int* grp_seg = nullptr;
  const int* grp_tile_e = nullptr;
  int grp_E = 0, grp_b_rows = 0;
  // set by gemm_bf16: fp32 results go through shared memory so that stores
  // are whole 128-byte row segments (when the epilogue, not the mainloop,
  // bounds the tile: short reductions)
  int stage_f32 = 0;
};

// C[M,N] = op(A) op(B) with bf16 operands, fp32 accumulation (see gemm.cu).
int gemm_bf16(int mode, const GemmParams& p, const void* A, const void* B, int lda, int ldb, cudaStream_t st);

// RMSNorm (elementwise.cu)
int rmsnorm_fwd(const float* x, const float* w, uint16_t* y, float* rstd, int T, int h, float eps, cudaStream_t st);
size_t rmsnorm_bwd_partials(int T, int h);  // floats of workspace
int rmsnorm_bwd(const float* x, const float* w, const float* rstd, const float* dy, const float* resid, float* dx,
                uint16_t* dx_bf16, float* dw, float* work, int T, int h, cudaStream_t st);

// The same backward with its partial sums in a fixed device array of the
// library (no allocation, no workspace argument). Returns -2 when
// ceil(T/32) * h exceeds rmsnorm_bwd_noalloc_capacity() floats.
size_t rmsnorm_bwd_noalloc_capacity();
int rmsnorm_bwd_noalloc(const float* x, const float* w, const float* rstd, const float* dy, const float* resid,
                        float* dx, uint16_t* dx_bf16, float* dw, int T, int h, cudaStream_t st);

// RoPE table [S, d/2] of (cos, sin) and in-place rotation of bf16 heads.
int rope_table(float2* tab, int S, int d, float theta, cudaStream_t st);
int rope_apply(uint16_t* x, const float2* tab, int B, int S, int row_stride, int head0, int n_heads, int d, int dir,
               cudaStream_t st);

// SwiGLU on gu [T, 2*ld] (gate [0,F), up [ld, ld+F)).
int swiglu_fwd(const uint16_t* gu, uint16_t* act, int T, int F, int ld, cudaStream_t st);
int swiglu_bwd(uint16_t* gu, const uint16_t* dact, int T, int F, int ld, cudaStream_t st);

// Mixture-of-experts routing (moe.cu). Slot t*k + j is token t's j-th
// choice; rows are the slots grouped by expert in ascending slot order.
// moe_route: top-k of router logits r [T,E] (ties: lower index), sel/w [T*k]
// (descending logit, weights renormalised over the k), counts[E] (zeroed
// here), log (optional) = a copy of sel.
int moe_route(const float* r, int T, int E, int k, int32_t* sel, float* w, int32_t* counts, int32_t* log,
              cudaStream_t st);
// seg[0..E]: expert e's rows start at seg[e], each segment its count rounded
// up to 128 rows; tile_e[b] (b < n_blocks): expert of 128-row block b, or -1.
int moe_segments(const int32_t* counts, int E, int n_blocks, int32_t* seg, int32_t* tile_e, cudaStream_t st);
// spos[slot] = row for the n = T*k slots (expert e's rows from seg[e], in
// ascending slot order).
int moe_permute(const int32_t* sel, int n, int E, const int32_t* seg, int32_t* spos, cudaStream_t st);
// xp[spos[s]] = m[s / k] for the n slots (bf16 rows of h).
int moe_gather(const uint16_t* m, const int32_t* spos, int n, int k, int h, uint16_t* xp, cudaStream_t st);
// y[t] = hmid[t] + sum_j w[t,j] yp[spos[t,j]] (fp32).
int moe_combine(const float* hmid, const float* yp, const int32_t* spos, const float* w, int T, int k, int h,
                float* y, cudaStream_t st);
// dyp[spos[t,j]] = bf16(w[t,j] dh[t]), dw[t,j] = <dh[t], yp[spos[t,j]]>.
int moe_combine_bwd(const float* dh, const float* yp, const int32_t* spos, const float* w, int T, int k, int h,
                    uint16_t* dyp, float* dw, cudaStream_t st);
// dm[t] = sum_j dxp[spos[t,j]] (fp32).
int moe_unpermute(const float* dxp, const int32_t* spos, int T, int k, int h, float* dm, cudaStream_t st);
// dr [T,E] bf16: w_j (dw_j - sum_i w_i dw_i) at the selected experts, 0 elsewhere.
int moe_router_bwd(const float* w, const float* dw, const int32_t* sel, int T, int k, int E, uint16_t* dr,
                   cudaStream_t st);


// Compact form over the n_ids distinct token ids: rows[u] = sum over the
// positions perm[start[u] .. start[u+1]) of dh0 ([n_ids, h] fp32 output).
int embed_scatter_rows(const int32_t* perm, const int32_t* start, int n_ids, const float* dh0, float* rows, int h,
                       cudaStream_t st);
int cast_bf16_f32(const uint16_t* src, float* dst, size_t n, cudaStream_t st);

// Weight preparation: fp32 [rows_src, cols] -> bf16 [rows_dst, ld_dst]
// (rows >= rows_src and columns >= cols are zero); bf16/fp32 gains -> fp32.
int cast_rows_f32_bf16(const float* src, uint16_t* dst, int rows_src, int rows_dst, int cols, int ld_dst,
                       cudaStream_t st);
int gains_to_f32(const void* src, bool bf16, float* dst, int n, cudaStream_t st);
// FP8 e4m3 rows with one fp32 scale per row to bf16 (dst row stride ld_dst):
// dst[r][c] = bf16(float(q[r][c]) * scales[r]); cols % 16 == 0, q and dst
// 16-byte aligned.
int dequant_fp8_rows(const uint8_t* q, const float* scales, int rows, int cols, uint16_t* dst, int ld_dst,
                     cudaStream_t st);

// Cross-entropy over vocab slices of materialised fp32 logits [T, R] (row
// stride ld): per-row (max, sum exp) partials, merged in slice order.
int ce_slice_stats(const float* logits, int T, int R, int ld, int row0, const int32_t* labels, float2* part,
                   float* zlab, cudaStream_t st);
int ce_finalize(const float2* part, int nslices, const float* zlab, float* lse, float* loss_terms, float* loss,
                int T, float scale, cudaStream_t st);
int ce_slice_grad(const float* logits, int T, int R, int ld, int row0, const int32_t* labels, const float* lse,
                  float scale, uint16_t* dz, cudaStream_t st);

// Read and clear the device error words of the kernels that wait on
// barriers (0 = no error). Synchronous with respect to the device.
uint32_t gemm_take_device_error();
uint32_t attention_tc_take_device_error();
uint32_t gemm_peek_device_error();  // the same words, not cleared
uint32_t attention_tc_peek_device_error();

// Tensor-core flash attention (attention_tc.cu); head_dim in {16,32,64,128},
// row strides multiples of 8. work: attention_bwd_workspace(B, S, nq) floats
// (per row delta and the log-sum-exp in log2 units, S padded to 64).
size_t attention_bwd_workspace(int B, int S, int nq);
int attention_fwd_tc(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* o, float* lse, int B, int S,
                     int nq, int nkv, int d, int ldq, int ldkv, int ldo, cudaStream_t st);
// rope_tab (nullable, [S][d/2] (cos, sin)): q and k were rotated after
// projection; dq and dk are then rotated back (inverse RoPE) before rounding.
int attention_bwd_tc(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* o, const uint16_t* dout,
                     const float* lse, uint16_t* dq, uint16_t* dk, uint16_t* dv, float* work, int B, int S, int nq,
                     int nkv, int d, int ldq, int ldkv, int ldo, cudaStream_t st, const float2* rope_tab = nullptr);

// fp32 -> bf16 copy of a dense buffer.
int cast_f32_bf16(const float* src, uint16_t* dst, size_t n, cudaStream_t st);

}  // namespace mt
