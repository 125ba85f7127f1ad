// Kernel-level C entry points (declared in include/mt.h): thin argument
// checks in front of the layer-template launchers, for tests and
// measurement. They allocate nothing.
#include <algorithm>

#include "../../include/mt.h"
#include "common.cuh"
#include "kernels.h"

using namespace mt;

namespace {
inline cudaStream_t S(void* s) { return (cudaStream_t)s; }
inline int rc(int r) {
  if (r == 0) return MT_OK;
  return cudaPeekAtLastError() != cudaSuccess ? MT_ERR_CUDA : MT_ERR_ARG;
}
size_t rup(size_t x, size_t a) { return (x + a - 1) / a * a; }
// Carving of the mixture-of-experts workspace (byte offsets, 256-aligned).
struct MoeWs {
  size_t r, sel, w, spos, counts, seg, tile_e, xp, gup, actp, yp, total;
  size_t dyp, dw, dr, total_bwd;  // backward only
  int n_pad;
};
MoeWs moe_ws(int T, int h, int E, int k, int Fe) {
  MoeWs o;
  const size_t n = (size_t)T * k;
  o.n_pad = (int)rup(n + (size_t)E * 127, 128);
  size_t a = 0;
  auto take = [&](size_t b) {
    const size_t r = a;
    a += rup(b, 256);
    return r;
  };
  o.r = take((size_t)T * E * 4);
  o.sel = take(n * 4);
  o.w = take(n * 4);
  o.spos = take(n * 4);
  o.counts = take(((size_t)E + 1) * 4);
  o.seg = take(((size_t)E + 1) * 4);
  o.tile_e = take((size_t)o.n_pad / 128 * 4);
  o.xp = take((size_t)o.n_pad * h * 2);
  o.gup = take((size_t)o.n_pad * 2 * Fe * 2);
  o.actp = take((size_t)o.n_pad * Fe * 2);
  o.yp = take((size_t)o.n_pad * h * 4);
  o.total = a;
  o.dyp = take((size_t)o.n_pad * h * 2);
  o.dw = take(n * 4);
  o.dr = take((size_t)T * E * 2);
  o.total_bwd = a;
  return o;
}

// Device pointers of the carved workspace.
struct MoeBufs {
  float *r, *w, *yp;
  int32_t *sel, *spos, *counts, *seg, *tile_e;
  uint16_t *xp, *gup, *actp, *dyp, *dr;
  float* dw;
};
MoeBufs moe_bufs(const MoeWs& o, void* workspace) {
  uint8_t* ws = (uint8_t*)workspace;
  MoeBufs b;
  b.r = (float*)(ws + o.r);
  b.sel = (int32_t*)(ws + o.sel);
  b.w = (float*)(ws + o.w);
  b.spos = (int32_t*)(ws + o.spos);
  b.counts = (int32_t*)(ws + o.counts);
  b.seg = (int32_t*)(ws + o.seg);
  b.tile_e = (int32_t*)(ws + o.tile_e);
  b.xp = (uint16_t*)(ws + o.xp);
  b.gup = (uint16_t*)(ws + o.gup);
  b.actp = (uint16_t*)(ws + o.actp);
  b.yp = (float*)(ws + o.yp);
  b.dyp = (uint16_t*)(ws + o.dyp);
  b.dw = (float*)(ws + o.dw);
  b.dr = (uint16_t*)(ws + o.dr);
  return b;
}

// The routed part of the forward up to the experts' outputs y (rows in
// expert order): router, routing, segments, gather, grouped gate|up (SwiGLU
// epilogue) and grouped down products.
int moe_fwd_core(const void* m, const void* Wr, const void* Wgu, const void* Wd, int32_t* route, const MoeWs& o,
                 const MoeBufs& b, int T, int h, int E, int k, int Fe, cudaStream_t st) {
  const int n = T * k;
  {
    GemmParams gp{T, E, h, EPI_F32, b.r, nullptr, E, 0, 1};
    if (gemm_bf16(GEMM_NT, gp, m, Wr, h, h, st)) return -1;
  }
  if (moe_route(b.r, T, E, k, b.sel, b.w, b.counts, route, st) ||
      moe_segments(b.counts, E, o.n_pad / 128, b.seg, b.tile_e, st) || moe_permute(b.sel, n, E, b.seg, b.spos, st))
    return -1;
  if (cudaMemsetAsync(b.xp, 0, (size_t)o.n_pad * h * 2, st) != cudaSuccess) return -1;
  if (moe_gather((const uint16_t*)m, b.spos, n, k, h, b.xp, st)) return -1;
  {
    GemmParams gp{o.n_pad, Fe, h, EPI_BF16, b.gup, nullptr, 2 * Fe, 0, 1};
    gp.gated = 1;
    gp.u_off = Fe;
    gp.u_col = Fe;
    gp.act = b.actp;
    gp.ld_act = Fe;
    gp.grp_seg = b.seg;
    gp.grp_tile_e = b.tile_e;
    gp.grp_E = E;
    gp.grp_b_rows = 2 * Fe;
    if (gemm_bf16(GEMM_NT, gp, b.xp, Wgu, h, h, st)) return -1;
  }
  GemmParams gp{o.n_pad, h, Fe, EPI_F32, b.yp, nullptr, h, 0, 1};
  gp.grp_seg = b.seg;
  gp.grp_tile_e = b.tile_e;
  gp.grp_E = E;
  gp.grp_b_rows = h;
  return gemm_bf16(GEMM_NT, gp, b.actp, Wd, Fe, Fe, st);
}
bool moe_dims_ok(int T, int h, int E, int k, int Fe) {
  return T >= 1 && h >= 64 && h % 64 == 0 && E >= 8 && E <= 1024 && E % 8 == 0 && k >= 1 && k <= 32 && k <= E &&
         Fe >= 32 && Fe % 32 == 0 && (double)T * k * std::max(h, 2 * Fe) < 2147483647.0 * 4;
}
}  // namespace

extern "C" {

size_t mt_op_moe_workspace(int T, int h, int E, int top_k, int Fe) {
  if (!moe_dims_ok(T, h, E, top_k, Fe)) return 0;
  return moe_ws(T, h, E, top_k, Fe).total;
}

int mt_op_moe_ffn_fwd(const void* m, const void* Wr, const void* Wgu, const void* Wd, const float* resid,
                      float* out, int32_t* route, void* workspace, int T, int h, int E, int top_k, int Fe,
                      void* stream) {
  if (!m || !Wr || !Wgu || !Wd || !resid || !out || !route || !workspace) return MT_ERR_ARG;
  if (!moe_dims_ok(T, h, E, top_k, Fe) || ((uintptr_t)workspace & 255)) return MT_ERR_ARG;
  const MoeWs o = moe_ws(T, h, E, top_k, Fe);
  const MoeBufs b = moe_bufs(o, workspace);
  cudaStream_t st = S(stream);
  if (moe_fwd_core(m, Wr, Wgu, Wd, route, o, b, T, h, E, top_k, Fe, st)) return rc(-1);
  return rc(moe_combine(resid, b.yp, b.spos, b.w, T, top_k, h, out, st));
}

size_t mt_op_moe_bwd_workspace(int T, int h, int E, int top_k, int Fe) {
  if (!moe_dims_ok(T, h, E, top_k, Fe)) return 0;
  return moe_ws(T, h, E, top_k, Fe).total_bwd;
}

int mt_op_moe_ffn_bwd(const void* m, const void* Wr, const void* Wgu, const void* Wd, const float* dout, float* dm,
                      float* dWr, float* dWgu, float* dWd, int32_t* route, void* workspace, int T, int h, int E,
                      int top_k, int Fe, void* stream) {
  if (!m || !Wr || !Wgu || !Wd || !dout || !dm || !dWr || !dWgu || !dWd || !route || !workspace) return MT_ERR_ARG;
  if (!moe_dims_ok(T, h, E, top_k, Fe) || ((uintptr_t)workspace & 255)) return MT_ERR_ARG;
  const MoeWs o = moe_ws(T, h, E, top_k, Fe);
  const MoeBufs b = moe_bufs(o, workspace);
  const int k = top_k;
  cudaStream_t st = S(stream);
  if (moe_fwd_core(m, Wr, Wgu, Wd, route, o, b, T, h, E, k, Fe, st)) return rc(-1);
  if (cudaMemsetAsync(b.dyp, 0, (size_t)o.n_pad * h * 2, st) != cudaSuccess) return MT_ERR_CUDA;
  if (moe_combine_bwd(dout, b.yp, b.spos, b.w, T, k, h, b.dyp, b.dw, st)) return rc(-1);
  auto grouped = [&](GemmParams& gp, bool tn, int b_rows) {
    gp.grp_seg = b.seg;
    gp.grp_tile_e = tn ? nullptr : b.tile_e;
    gp.grp_E = E;
    gp.grp_b_rows = b_rows;
  };
  {  // dWd_e = dY_e^T act_e
    GemmParams gp{h, Fe, o.n_pad, EPI_F32, dWd, nullptr, Fe, 0, 1};
    grouped(gp, true, 0);
    if (gemm_bf16(GEMM_TN, gp, b.dyp, b.actp, h, Fe, st)) return rc(-1);
  }
  {  // dact = dY Wd_e -> (dg, du) in place over (g, u)
    GemmParams gp{o.n_pad, Fe, h, EPI_BF16, b.gup, nullptr, 2 * Fe, 0, 1};
    gp.swiglu_bwd = 1;
    gp.gu = b.gup;
    gp.ld_gu = 2 * Fe;
    gp.u_col = Fe;
    grouped(gp, false, h);
    if (gemm_bf16(GEMM_NN, gp, b.dyp, Wd, h, Fe, st)) return rc(-1);
  }
  {  // dWgu_e = d(g|u)_e^T x_e
    GemmParams gp{2 * Fe, h, o.n_pad, EPI_F32, dWgu, nullptr, h, 0, 1};
    grouped(gp, true, 0);
    if (gemm_bf16(GEMM_TN, gp, b.gup, b.xp, 2 * Fe, h, st)) return rc(-1);
  }
  {  // d x (routed rows, over y's rows) = d(g|u) Wgu_e
    GemmParams gp{o.n_pad, h, 2 * Fe, EPI_F32, b.yp, nullptr, h, 0, 1};
    grouped(gp, false, 2 * Fe);
    if (gemm_bf16(GEMM_NN, gp, b.gup, Wgu, 2 * Fe, h, st)) return rc(-1);
  }
  if (moe_unpermute(b.yp, b.spos, T, k, h, dm, st) || moe_router_bwd(b.w, b.dw, b.sel, T, k, E, b.dr, st))
    return rc(-1);
  {  // dm += dr Wr
    GemmParams gp{T, h, E, EPI_F32_ADD, dm, dm, h, 0, 1};
    if (gemm_bf16(GEMM_NN, gp, b.dr, Wr, E, h, st)) return rc(-1);
  }
  GemmParams gp{E, h, T, EPI_F32, dWr, nullptr, h, 0, 1};  // dWr = dr^T m
  return rc(gemm_bf16(GEMM_TN, gp, b.dr, m, E, h, st));
}


int mt_op_gemm(int mode, int epi, const void* A, const void* B, void* C, const void* addend, int M, int N, int K,
               int lda, int ldb, int ldc, void* stream) {
  if (!A || !B || !C) return MT_ERR_ARG;
  GemmParams p{M, N, K, epi, C, addend, ldc, 0, 1};
  return rc(gemm_bf16(mode, p, A, B, lda, ldb, S(stream)));
}

int mt_op_rmsnorm_fwd(const float* x, const float* w, void* y, float* rstd, int T, int h, float eps, void* stream) {
  if (!x || !w || !y || !rstd) return MT_ERR_ARG;
  return rc(rmsnorm_fwd(x, w, (uint16_t*)y, rstd, T, h, eps, S(stream)));
}

size_t mt_op_rmsnorm_bwd_workspace(int T, int h) { return rmsnorm_bwd_partials(T, h); }

int mt_op_rmsnorm_bwd(const float* x, const float* w, const float* rstd, const float* dy, const float* resid,
                      float* dx, void* dx_bf16, float* dw, float* workspace, int T, int h, void* stream) {
  if (!x || !w || !rstd || !dy || !dx || !dw || !workspace) return MT_ERR_ARG;
  return rc(rmsnorm_bwd(x, w, rstd, dy, resid, dx, (uint16_t*)dx_bf16, dw, workspace, T, h, S(stream)));
}

int mt_op_rmsnorm_bwd_noalloc(const float* x, const float* w, const float* rstd, const float* dy, const float* resid,
                              float* dx, void* dx_bf16, float* dw, int T, int h, void* stream) {
  if (!x || !w || !rstd || !dy || !dx || !dw) return MT_ERR_ARG;
  const int r = rmsnorm_bwd_noalloc(x, w, rstd, dy, resid, dx, (uint16_t*)dx_bf16, dw, T, h, S(stream));
  if (r == -2) return MT_ERR_BUDGET;
  if (r != 0) return cudaPeekAtLastError() != cudaSuccess ? MT_ERR_CUDA : MT_ERR_ARG;
  return MT_OK;
}

int mt_op_rope(void* x, float* table, int B, int S_, int row_stride, int head0, int n_heads, int d, float theta,
               int dir, void* stream) {
  if (!x || !table || B < 1 || S_ < 1 || d < 8 || (dir != 1 && dir != -1)) return MT_ERR_ARG;
  float2* tab = (float2*)table;
  if (rope_table(tab, S_, d, theta, S(stream))) return rc(-1);
  return rc(rope_apply((uint16_t*)x, tab, B, S_, row_stride, head0, n_heads, d, dir, S(stream)));
}

int mt_op_gemm_rope(const void* A, const void* W, void* C, int M, int N, int K, int lda, int ldb, int ldc,
                    float* table, int S_, int d, float theta, int rope_cols, void* stream) {
  if (!A || !W || !C || !table || S_ < 1 || d < 16 || rope_cols < 0) return MT_ERR_ARG;
  if (rope_table((float2*)table, S_, d, theta, S(stream))) return rc(-1);
  GemmParams p{M, N, K, EPI_BF16, C, nullptr, ldc, 0, 1};
  p.rope_tab = (const float2*)table;
  p.rope_S = S_;
  p.rope_d = d;
  p.rope_cols = rope_cols;
  return rc(gemm_bf16(GEMM_NT, p, A, W, lda, ldb, S(stream)));
}

int mt_op_gemm_swiglu(const void* X, const void* W, void* gu, void* act, int M, int F, int K, int lda, int ldb,
                      int u_off, void* stream) {
  if (!X || !W || !gu || !act || u_off < F) return MT_ERR_ARG;
  GemmParams p{M, F, K, EPI_BF16, gu, nullptr, 2 * u_off, 0, 1};
  p.gated = 1;
  p.u_off = u_off;
  p.u_col = u_off;
  p.act = (uint16_t*)act;
  p.ld_act = u_off;
  return rc(gemm_bf16(GEMM_NT, p, X, W, lda, ldb, S(stream)));
}

int mt_op_gemm_swiglu_bwd(const void* dY, const void* Wd, void* gu, int M, int F, int K, int lda, int ldb, int u_off,
                          void* stream) {
  if (!dY || !Wd || !gu || u_off < F) return MT_ERR_ARG;
  GemmParams p{M, F, K, EPI_BF16, gu, nullptr, 2 * u_off, 0, 1};
  p.swiglu_bwd = 1;
  p.gu = (uint16_t*)gu;
  p.ld_gu = 2 * u_off;
  p.u_col = u_off;
  return rc(gemm_bf16(GEMM_NN, p, dY, Wd, lda, ldb, S(stream)));
}

int mt_op_attention_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int S_, int n_heads,
                        int n_kv_heads, int d, int ldq, int ldkv, int ldo, void* stream) {
  if (!q || !k || !v || !o || !lse) return MT_ERR_ARG;
  return rc(attention_fwd_tc((const uint16_t*)q, (const uint16_t*)k, (const uint16_t*)v, (uint16_t*)o, lse, B, S_,
                          n_heads, n_kv_heads, d, ldq, ldkv, ldo, S(stream)));
}

size_t mt_op_attention_bwd_workspace(int B, int S_, int n_heads) { return attention_bwd_workspace(B, S_, n_heads); }

int mt_op_attention_bwd(const void* q, const void* k, const void* v, const void* o, const void* do_, const float* lse,
                        void* dq, void* dk, void* dv, float* workspace, int B, int S_, int n_heads, int n_kv_heads,
                        int d, int ldq, int ldkv, int ldo, void* stream) {
  if (!q || !k || !v || !o || !do_ || !lse || !dq || !dk || !dv || !workspace) return MT_ERR_ARG;
  return rc(attention_bwd_tc((const uint16_t*)q, (const uint16_t*)k, (const uint16_t*)v, (const uint16_t*)o,
                          (const uint16_t*)do_, lse, (uint16_t*)dq, (uint16_t*)dk, (uint16_t*)dv, workspace, B, S_,
                          n_heads, n_kv_heads, d, ldq, ldkv, ldo, S(stream)));
}

int mt_op_attention_bwd_rope(const void* q, const void* k, const void* v, const void* o, const void* do_,
                             const float* lse, void* dq, void* dk, void* dv, float* workspace, int B, int S_,
                             int n_heads, int n_kv_heads, int d, int ldq, int ldkv, int ldo, float* table, float theta,
                             void* stream) {
  if (!q || !k || !v || !o || !do_ || !lse || !dq || !dk || !dv || !workspace || !table) return MT_ERR_ARG;
  if (rope_table((float2*)table, S_, d, theta, S(stream))) return rc(-1);
  return rc(attention_bwd_tc((const uint16_t*)q, (const uint16_t*)k, (const uint16_t*)v, (const uint16_t*)o,
                             (const uint16_t*)do_, lse, (uint16_t*)dq, (uint16_t*)dk, (uint16_t*)dv, workspace, B, S_,
                             n_heads, n_kv_heads, d, ldq, ldkv, ldo, S(stream), (const float2*)table));
}

int mt_op_swiglu_fwd(const void* gu, void* act, int T, int F, int ld, void* stream) {
  if (!gu || !act) return MT_ERR_ARG;
  return rc(swiglu_fwd((const uint16_t*)gu, (uint16_t*)act, T, F, ld, S(stream)));
}

int mt_op_swiglu_bwd(void* gu, const void* dact, int T, int F, int ld, void* stream) {
  if (!gu || !dact) return MT_ERR_ARG;
  return rc(swiglu_bwd((uint16_t*)gu, (const uint16_t*)dact, T, F, ld, S(stream)));
}

size_t mt_op_lmhead_ce_workspace(int T, int V, int h) {
  (void)h;
  const size_t ld = rup((size_t)V, 8);
  return rup((size_t)T * ld * 4, 256) + rup((size_t)T * ld * 2, 256) + rup((size_t)T * 8, 256) +
         3 * rup((size_t)T * 4, 256);
}

int mt_op_lmhead_ce(const void* X, const void* W, const int32_t* labels, float scale, float* dX, float* dW,
                    float* loss_dev, void* workspace, int T, int V, int h, void* stream) {
  if (!X || !W || !labels || !dX || !dW || !loss_dev || !workspace || T < 1 || V < 1 || h < 1) return MT_ERR_ARG;
  const int ld = (int)rup((size_t)V, 8);
  uint8_t* w = (uint8_t*)workspace;
  float* logits = (float*)w;
  w += rup((size_t)T * ld * 4, 256);
  uint16_t* dz = (uint16_t*)w;
  w += rup((size_t)T * ld * 2, 256);
  float2* part = (float2*)w;
  w += rup((size_t)T * 8, 256);
  float* zlab = (float*)w;
  w += rup((size_t)T * 4, 256);
  float* lse = (float*)w;
  w += rup((size_t)T * 4, 256);
  float* terms = (float*)w;
  cudaStream_t st = S(stream);
  GemmParams p1{T, V, h, EPI_F32, logits, nullptr, ld, 0, 1};
  if (gemm_bf16(GEMM_NT, p1, X, W, h, h, st)) return rc(-1);
  if (ce_slice_stats(logits, T, V, ld, 0, labels, part, zlab, st)) return rc(-1);
  if (ce_finalize(part, 1, zlab, lse, terms, loss_dev, T, scale, st)) return rc(-1);
  if (ce_slice_grad(logits, T, V, ld, 0, labels, lse, scale, dz, st)) return rc(-1);
  GemmParams p2{T, h, V, EPI_F32, dX, nullptr, h, 0, 1};
  if (gemm_bf16(GEMM_NN, p2, dz, W, ld, h, st)) return rc(-1);
  GemmParams p3{V, h, T, EPI_F32, dW, nullptr, h, 0, 1};
  if (gemm_bf16(GEMM_TN, p3, dz, X, ld, h, st)) return rc(-1);
  return MT_OK;
}

int mt_op_device_error(void) {
  cudaDeviceSynchronize();
  return (int)(gemm_take_device_error() | attention_tc_take_device_error());
}

}  // extern "C"
