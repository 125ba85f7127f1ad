// Causal GQA attention, forward and backward, with online softmax.
// o_t = sum_{s<=t} softmax_s(q_t . k_s / sqrt(d)) v_s, query head j reading
// KV head j / (n_q / n_kv). The forward saves the natural-log logsumexp of
// each row's scaled scores; the backward recomputes the probabilities from
// it (no [S, S] matrix is ever stored) and produces dK/dV per KV row and dQ
// per query row in separate passes, each summing in a fixed order, so the
// result is deterministic.
//
// This file holds the warp-per-row formulation (any head_dim up to 128).
#include "common.cuh"
#include "kernels.h"

namespace mt {

MT_DEVICE_ERROR_READER(attention_take_device_error)

namespace {

constexpr int kWarps = 4;

template <int E>
__device__ __forceinline__ void load_row(const uint16_t* p, int d, float (&r)[E]) {
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = lane_id() + 32 * e;
    r[e] = i < d ? bf2f(p[i]) : 0.f;
  }
}

template <int E>
__device__ __forceinline__ float dot_row(const float (&a)[E], const uint16_t* p, int d) {
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = lane_id() + 32 * e;
    if (i < d) s += a[e] * bf2f(p[i]);
  }
  return warp_sum(s);
}

template <int E>
__global__ void __launch_bounds__(32 * kWarps) attn_fwd_rows_kernel(const uint16_t* __restrict__ q,
                                                                    const uint16_t* __restrict__ k,
                                                                    const uint16_t* __restrict__ v, uint16_t* o,
                                                                    float* lse, int B, int S, int nq, int nkv, int d,
                                                                    int ldq, int ldkv, int ldo, float scale) {
  const size_t wid = (size_t)blockIdx.x * kWarps + warp_id();
  if (wid >= (size_t)B * S * nq) return;
  const int j = (int)(wid % nq);
  const int t = (int)((wid / nq) % S);
  const int b = (int)(wid / ((size_t)nq * S));
  const int g = j / (nq / nkv);
  float qv[E], acc[E];
  load_row<E>(q + ((size_t)b * S + t) * ldq + (size_t)j * d, d, qv);
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float m = -INFINITY, l = 0.f;
  for (int s = 0; s <= t; ++s) {
    const size_t rs = (size_t)b * S + s;
    const float sc = dot_row<E>(qv, k + rs * ldkv + (size_t)g * d, d) * scale;
    const float mn = fmaxf(m, sc);
    const float corr = __expf(m - mn), p = __expf(sc - mn);
    l = l * corr + p;
    const uint16_t* vr = v + rs * ldkv + (size_t)g * d;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int i = lane_id() + 32 * e;
      acc[e] = acc[e] * corr + (i < d ? p * bf2f(vr[i]) : 0.f);
    }
    m = mn;
  }
  const float inv = 1.f / l;
  uint16_t* orow = o + ((size_t)b * S + t) * ldo + (size_t)j * d;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = lane_id() + 32 * e;
    if (i < d) orow[i] = f2bf(acc[e] * inv);
  }
  if (lane_id() == 0) lse[((size_t)b * nq + j) * S + t] = m + logf(l);
}

// delta[b, j, t] = sum_e dO[t, j, e] * O[t, j, e]
template <int E>
__global__ void __launch_bounds__(32 * kWarps) attn_delta_kernel(const uint16_t* __restrict__ o,
                                                                 const uint16_t* __restrict__ dout, float* delta,
                                                                 int B, int S, int nq, int d, int ldo) {
  const size_t wid = (size_t)blockIdx.x * kWarps + warp_id();
  if (wid >= (size_t)B * S * nq) return;
  const int j = (int)(wid % nq);
  const int t = (int)((wid / nq) % S);
  const int b = (int)(wid / ((size_t)nq * S));
  float ov[E];
  const size_t off = ((size_t)b * S + t) * ldo + (size_t)j * d;
  load_row<E>(o + off, d, ov);
  const float dl = dot_row<E>(ov, dout + off, d);
  if (lane_id() == 0) delta[((size_t)b * nq + j) * S + t] = dl;
}

// dq_t = scale * sum_{s<=t} P_ts (dP_ts - delta_t) k_s
template <int E>
__global__ void __launch_bounds__(32 * kWarps) attn_dq_kernel(const uint16_t* __restrict__ q,
                                                              const uint16_t* __restrict__ k,
                                                              const uint16_t* __restrict__ v,
                                                              const uint16_t* __restrict__ dout,
                                                              const float* __restrict__ lse,
                                                              const float* __restrict__ delta, uint16_t* dq, int B,
                                                              int S, int nq, int nkv, int d, int ldq, int ldkv,
                                                              int ldo, float scale) {
  const size_t wid = (size_t)blockIdx.x * kWarps + warp_id();
  if (wid >= (size_t)B * S * nq) return;
  const int j = (int)(wid % nq);
  const int t = (int)((wid / nq) % S);
  const int b = (int)(wid / ((size_t)nq * S));
  const int g = j / (nq / nkv);
  float qv[E], gv[E], acc[E];
  load_row<E>(q + ((size_t)b * S + t) * ldq + (size_t)j * d, d, qv);
  load_row<E>(dout + ((size_t)b * S + t) * ldo + (size_t)j * d, d, gv);
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  const size_t ri = ((size_t)b * nq + j) * S + t;
  const float L = lse[ri], D = delta[ri];
  for (int s = 0; s <= t; ++s) {
    const size_t rs = (size_t)b * S + s;
    const uint16_t* kr = k + rs * ldkv + (size_t)g * d;
    const float p = __expf(dot_row<E>(qv, kr, d) * scale - L);
    const float dp = dot_row<E>(gv, v + rs * ldkv + (size_t)g * d, d);
    const float ds = p * (dp - D) * scale;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int i = lane_id() + 32 * e;
      if (i < d) acc[e] += ds * bf2f(kr[i]);
    }
  }
  uint16_t* out = dq + ((size_t)b * S + t) * ldq + (size_t)j * d;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = lane_id() + 32 * e;
    if (i < d) out[i] = f2bf(acc[e]);
  }
}

// For KV row s of head g: dv_s = sum_j sum_{t>=s} P_ts dO_t, dk_s = scale * sum P_ts (dP_ts - delta_t) q_t.
template <int E>
__global__ void __launch_bounds__(32 * kWarps) attn_dkv_kernel(const uint16_t* __restrict__ q,
                                                               const uint16_t* __restrict__ k,
                                                               const uint16_t* __restrict__ v,
                                                               const uint16_t* __restrict__ dout,
                                                               const float* __restrict__ lse,
                                                               const float* __restrict__ delta, uint16_t* dk,
                                                               uint16_t* dv, int B, int S, int nq, int nkv, int d,
                                                               int ldq, int ldkv, int ldo, float scale) {
  const size_t wid = (size_t)blockIdx.x * kWarps + warp_id();
  if (wid >= (size_t)B * S * nkv) return;
  const int g = (int)(wid % nkv);
  const int s = (int)((wid / nkv) % S);
  const int b = (int)(wid / ((size_t)nkv * S));
  const int grp = nq / nkv;
  float kv[E], vv[E], adk[E], adv[E];
  const size_t rs = (size_t)b * S + s;
  load_row<E>(k + rs * ldkv + (size_t)g * d, d, kv);
  load_row<E>(v + rs * ldkv + (size_t)g * d, d, vv);
#pragma unroll
  for (int e = 0; e < E; ++e) adk[e] = adv[e] = 0.f;
  for (int jj = 0; jj < grp; ++jj) {
    const int j = g * grp + jj;
    for (int t = s; t < S; ++t) {
      const size_t rt = (size_t)b * S + t;
      const uint16_t* qr = q + rt * ldq + (size_t)j * d;
      const uint16_t* gr = dout + rt * ldo + (size_t)j * d;
      const size_t ri = ((size_t)b * nq + j) * S + t;
      const float p = __expf(dot_row<E>(kv, qr, d) * scale - lse[ri]);
      const float dp = dot_row<E>(vv, gr, d);
      const float ds = p * (dp - delta[ri]) * scale;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int i = lane_id() + 32 * e;
        if (i < d) {
          adv[e] += p * bf2f(gr[i]);
          adk[e] += ds * bf2f(qr[i]);
        }
      }
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = lane_id() + 32 * e;
    if (i < d) {
      dk[rs * ldkv + (size_t)g * d + i] = f2bf(adk[e]);
      dv[rs * ldkv + (size_t)g * d + i] = f2bf(adv[e]);
    }
  }
}

inline unsigned warps_grid(size_t n) { return (unsigned)((n + kWarps - 1) / kWarps); }

bool check(int B, int S, int nq, int nkv, int d) {
  return B > 0 && S > 0 && nq > 0 && nkv > 0 && nq % nkv == 0 && d > 0 && d <= 128;
}

}  // namespace

int attention_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* o, float* lse, int B, int S,
                  int nq, int nkv, int d, int ldq, int ldkv, int ldo, cudaStream_t st) {
  if (!check(B, S, nq, nkv, d)) return -1;
  const float scale = 1.f / sqrtf((float)d);
  const unsigned grid = warps_grid((size_t)B * S * nq);
  if (d <= 32)
    attn_fwd_rows_kernel<1><<<grid, 32 * kWarps, 0, st>>>(q, k, v, o, lse, B, S, nq, nkv, d, ldq, ldkv, ldo, scale);
  else if (d <= 64)
    attn_fwd_rows_kernel<2><<<grid, 32 * kWarps, 0, st>>>(q, k, v, o, lse, B, S, nq, nkv, d, ldq, ldkv, ldo, scale);
  else
    attn_fwd_rows_kernel<4><<<grid, 32 * kWarps, 0, st>>>(q, k, v, o, lse, B, S, nq, nkv, d, ldq, ldkv, ldo, scale);
  count_launches(1);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

size_t attention_bwd_workspace(int B, int S, int nq) { return (size_t)B * S * nq; }

int attention_bwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* o, const uint16_t* dout,
                  const float* lse, uint16_t* dq, uint16_t* dk, uint16_t* dv, float* work, int B, int S, int nq,
                  int nkv, int d, int ldq, int ldkv, int ldo, cudaStream_t st) {
  if (!check(B, S, nq, nkv, d)) return -1;
  const float scale = 1.f / sqrtf((float)d);
  const unsigned gq = warps_grid((size_t)B * S * nq), gk = warps_grid((size_t)B * S * nkv);
  float* delta = work;
#define MT_ATTN_BWD(E)                                                                                          \
  attn_delta_kernel<E><<<gq, 32 * kWarps, 0, st>>>(o, dout, delta, B, S, nq, d, ldo);                          \
  attn_dq_kernel<E><<<gq, 32 * kWarps, 0, st>>>(q, k, v, dout, lse, delta, dq, B, S, nq, nkv, d, ldq, ldkv, ldo, \
                                                scale);                                                         \
  attn_dkv_kernel<E><<<gk, 32 * kWarps, 0, st>>>(q, k, v, dout, lse, delta, dk, dv, B, S, nq, nkv, d, ldq, ldkv,  \
                                                 ldo, scale);
  if (d <= 32) {
    MT_ATTN_BWD(1)
  } else if (d <= 64) {
    MT_ATTN_BWD(2)
  } else {
    MT_ATTN_BWD(4)
  }
#undef MT_ATTN_BWD
  count_launches(3);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace mt
