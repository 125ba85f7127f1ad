// Routing kernels of the mixture-of-experts FFN (the MoE layer template of the
// streamed workloads, Qwen3-MoE style: softmax router, top-k experts with
// renormalised weights, SwiGLU experts). The expert products themselves run
// on the grouped form of the tcgen05 GEMM of gemm.cu (one launch per product
// for all experts); these kernels move rows between token order and expert
// order and carry the router's forward and backward.
//
// Slots: token t's j-th choice is slot t*k + j. The rows of all slots are
// grouped by expert in ascending slot order; expert e's segment starts at
// sum_{f<e} roundup(count_f, 128), so every 128-row GEMM tile belongs to one
// expert (the padding rows are zero). The grouping, and every sum below, is
// the same in every run: results are bitwise reproducible.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace mt {
namespace {

constexpr int kMaxExpertsPerLane = 32;  // E <= 1024

// One warp per token: logits r[t, 0..E) -> the k experts of largest logit
// (equal logits: lower index first), in descending order, and their weights
// renormalised over the k, w_j = exp(r_j) / sum_i exp(r_i) (= p_j / sum_i p_i
// with p = softmax(r) over all E). counts[e] += 1 for every choice.
__global__ void moe_route_kernel(const float* __restrict__ r, int T, int E, int k, int32_t* __restrict__ sel,
                                 float* __restrict__ w, int32_t* __restrict__ counts, int32_t* __restrict__ log) {
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;  // whole warps leave together
  float v[kMaxExpertsPerLane];
  const float* rt = r + (size_t)t * E;
#pragma unroll
  for (int i = 0; i < kMaxExpertsPerLane; ++i) {
    const int e = lane + 32 * i;
    const float x = e < E ? rt[e] : -INFINITY;
    v[i] = x == x ? x : -INFINITY;  // a NaN logit ranks last
  }
  // Experts already chosen (bit i: expert lane + 32 i). Every round has an
  // untaken expert left (k <= E), so the winner is always a valid index.
  uint32_t taken = 0;
  float top = 0.f, wsum = 0.f, my_logit = 0.f;
  int my_e = 0;
  for (int j = 0; j < k; ++j) {
    float best = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < kMaxExpertsPerLane; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u) && (v[i] > best || (v[i] == best && e < bi))) {
        best = v[i];
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ob > best || (ob == best && oi < bi)) {
        best = ob;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);  // the owner lane marks the winner
    if (j == 0) top = best;
    const float ex = expf(best - top);
    wsum += ex;
    if (lane == j) {
      my_e = bi;
      my_logit = best;
    }
  }
  if (lane < k) {
    const size_t s = (size_t)t * k + lane;
    sel[s] = my_e;
    if (log) log[s] = my_e;
    w[s] = expf(my_logit - top) / wsum;
    atomicAdd(&counts[my_e], 1);
  }
}

// Segments of the routed rows: expert e owns rows [seg[e], seg[e+1]), its
// count rounded up to a multiple of 128 (whole tiles of the grouped GEMM);
// tile_e[b] = the expert owning 128-row block b, -1 past the last segment.
__global__ void __launch_bounds__(1024) moe_segments_kernel(const int32_t* __restrict__ counts, int E, int n_blocks,
                                                            int32_t* __restrict__ seg, int32_t* __restrict__ tile_e) {
  __shared__ int s_seg[1025];
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int e = 0; e < E; ++e) {
      s_seg[e] = acc;
      acc += (counts[e] + 127) & ~127;
    }
    s_seg[E] = acc;
  }
  __syncthreads();
  for (int i = threadIdx.x; i <= E; i += blockDim.x) seg[i] = s_seg[i];
  for (int b = threadIdx.x; b < n_blocks; b += blockDim.x) {
    const int row = b * 128;
    int e = -1;
    if (row < s_seg[E]) {  // the last e with s_seg[e] <= row: its segment is non-empty and holds row
      int lo = 0, hi = E - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_seg[mid] <= row) lo = mid;
        else hi = mid - 1;
      }
      e = lo;
    }
    tile_e[b] = e;
  }
}

// One block per expert: the rows of expert e in ascending slot order from
// the start of its segment, spos[slot] = row.
__global__ void __launch_bounds__(1024) moe_permute_kernel(const int32_t* __restrict__ sel, int n, int E,
                                                           const int32_t* __restrict__ seg,
                                                           int32_t* __restrict__ spos) {
  __shared__ int warp_tot[32];
  const int e = blockIdx.x;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int running = seg[e];
  for (int c0 = 0; c0 < n; c0 += blockDim.x) {
    const int s = c0 + threadIdx.x;
    const bool hit = s < n && sel[s] == e;
    const unsigned bal = __ballot_sync(0xffffffffu, hit);
    if (lane == 0) warp_tot[wid] = __popc(bal);
    __syncthreads();
    int before = 0, total = 0;
    for (int i = 0; i < nw; ++i) {
      const int c = warp_tot[i];
      before += i < wid ? c : 0;
      total += c;
    }
    if (hit) {
      const int row = running + before + __popc(bal & ((1u << lane) - 1u));
      spos[s] = row;
    }
    running += total;
    __syncthreads();
  }
}

// One block per slot s: xp[spos[s]] = m[s / k] (bf16 rows of h, 16-byte
// copies; the padding rows of the segments are not touched).
__global__ void moe_gather_kernel(const uint16_t* __restrict__ m, const int32_t* __restrict__ spos, int k, int h,
                                  uint16_t* __restrict__ xp) {
  const int s = blockIdx.x;
  const int t = s / k;
  const int row = spos[s];
  const uint4* src = (const uint4*)(m + (size_t)t * h);
  uint4* dst = (uint4*)(xp + (size_t)row * h);
  for (int i = threadIdx.x; i < h / 8; i += blockDim.x) dst[i] = src[i];
}

// y[t] = hmid[t] + sum_j w[t,j] yp[spos[t,j]], j ascending (fp32 rows).
__global__ void moe_combine_kernel(const float* __restrict__ hmid, const float* __restrict__ yp,
                                   const int32_t* __restrict__ spos, const float* __restrict__ w, int k, int h,
                                   float* __restrict__ y) {
  const int t = blockIdx.x;
  for (int i = threadIdx.x; i < h / 4; i += blockDim.x) {
    float4 acc = ((const float4*)(hmid + (size_t)t * h))[i];
    for (int j = 0; j < k; ++j) {
      const float wj = w[(size_t)t * k + j];
      const float4 v = ((const float4*)(yp + (size_t)spos[(size_t)t * k + j] * h))[i];
      acc.x = fmaf(wj, v.x, acc.x);
      acc.y = fmaf(wj, v.y, acc.y);
      acc.z = fmaf(wj, v.z, acc.z);
      acc.w = fmaf(wj, v.w, acc.w);
    }
    ((float4*)(y + (size_t)t * h))[i] = acc;
  }
}

__device__ __forceinline__ float block_sum_fixed(float v, float* red) {
  v = warp_sum(v);
  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  float s = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) s += red[i];  // same order in every thread
  return s;
}

// Backward of the combine, one block per token: dyp[spos[t,j]] = bf16(w_j dh[t])
// and dw[t,j] = <dh[t], yp[spos[t,j]]>.
__global__ void moe_combine_bwd_kernel(const float* __restrict__ dh, const float* __restrict__ yp,
                                       const int32_t* __restrict__ spos, const float* __restrict__ w, int k, int h,
                                       uint16_t* __restrict__ dyp, float* __restrict__ dw) {
  __shared__ float red[32];
  const int t = blockIdx.x;
  const float4* g = (const float4*)(dh + (size_t)t * h);
  for (int j = 0; j < k; ++j) {
    const size_t s = (size_t)t * k + j;
    const size_t row = (size_t)spos[s];
    const float wj = w[s];
    const float4* yr = (const float4*)(yp + row * h);
    uint2* dr = (uint2*)(dyp + row * h);
    float dot = 0.f;
    for (int i = threadIdx.x; i < h / 4; i += blockDim.x) {
      const float4 a = g[i], b = yr[i];
      dot = fmaf(a.x, b.x, dot);
      dot = fmaf(a.y, b.y, dot);
      dot = fmaf(a.z, b.z, dot);
      dot = fmaf(a.w, b.w, dot);
      uint2 o;
      o.x = pack_bf2(wj * a.x, wj * a.y);
      o.y = pack_bf2(wj * a.z, wj * a.w);
      dr[i] = o;
    }
    dot = block_sum_fixed(dot, red);
    if (threadIdx.x == 0) dw[s] = dot;
  }
}

// dm[t] = sum_j dxp[spos[t,j]], j ascending (fp32 rows).
__global__ void moe_unpermute_kernel(const float* __restrict__ dxp, const int32_t* __restrict__ spos, int k, int h,
                                     float* __restrict__ dm) {
  const int t = blockIdx.x;
  for (int i = threadIdx.x; i < h / 4; i += blockDim.x) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
      const float4 v = ((const float4*)(dxp + (size_t)spos[(size_t)t * k + j] * h))[i];
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    ((float4*)(dm + (size_t)t * h))[i] = acc;
  }
}

// Router backward: with w_j = p_{e_j} / sum_i p_{e_i} and p = softmax(r),
// dr[t, e_j] = w_j (dw_j - sum_i w_i dw_i) and dr = 0 for unselected experts
// (the softmax Jacobian's centring term sum_f p_f dp_f vanishes because the
// renormalised weights sum to one). Written as bf16, one thread per entry.
__global__ void moe_router_bwd_kernel(const float* __restrict__ w, const float* __restrict__ dw,
                                      const int32_t* __restrict__ sel, int T, int k, int E,
                                      uint16_t* __restrict__ dr) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (size_t)T * E) return;
  const int t = (int)(i / E), e = (int)(i % E);
  const size_t s0 = (size_t)t * k;
  float wdw = 0.f, out = 0.f;
  int hit = -1;
  for (int j = 0; j < k; ++j) {
    wdw = fmaf(w[s0 + j], dw[s0 + j], wdw);
    if (sel[s0 + j] == e) hit = j;
  }
  if (hit >= 0) out = w[s0 + hit] * (dw[s0 + hit] - wdw);
  dr[i] = f2bf(out);
}

bool launched() { return cudaGetLastError() == cudaSuccess; }

}  // namespace

int moe_route(const float* r, int T, int E, int k, int32_t* sel, float* w, int32_t* counts, int32_t* log,
              cudaStream_t st) {
  if (T < 1 || E < 1 || E > 32 * kMaxExpertsPerLane || k < 1 || k > 32 || k > E) return -1;
  if (cudaMemsetAsync(counts, 0, (size_t)E * 4, st) != cudaSuccess) return -1;
  const int warps = 8;
  moe_route_kernel<<<(T + warps - 1) / warps, warps * 32, 0, st>>>(r, T, E, k, sel, w, counts, log);
  count_launches(1);
  return launched() ? 0 : -1;
}

int moe_segments(const int32_t* counts, int E, int n_blocks, int32_t* seg, int32_t* tile_e, cudaStream_t st) {
  if (E < 1 || E > 1024 || n_blocks < 1) return -1;
  moe_segments_kernel<<<1, 1024, 0, st>>>(counts, E, n_blocks, seg, tile_e);
  count_launches(1);
  return launched() ? 0 : -1;
}

int moe_permute(const int32_t* sel, int n, int E, const int32_t* seg, int32_t* spos, cudaStream_t st) {
  if (n < 1 || E < 1) return -1;
  moe_permute_kernel<<<E, 1024, 0, st>>>(sel, n, E, seg, spos);
  count_launches(1);
  return launched() ? 0 : -1;
}

int moe_gather(const uint16_t* m, const int32_t* spos, int n, int k, int h, uint16_t* xp, cudaStream_t st) {
  if (n < 1 || h % 8) return -1;
  moe_gather_kernel<<<n, std::min(256, h / 8), 0, st>>>(m, spos, k, h, xp);
  count_launches(1);
  return launched() ? 0 : -1;
}

int moe_combine(const float* hmid, const float* yp, const int32_t* spos, const float* w, int T, int k, int h,
                float* y, cudaStream_t st) {
  if (T < 1 || h % 4) return -1;
  moe_combine_kernel<<<T, std::min(256, h / 4), 0, st>>>(hmid, yp, spos, w, k, h, y);
  count_launches(1);
  return launched() ? 0 : -1;
}

int moe_combine_bwd(const float* dh, const float* yp, const int32_t* spos, const float* w, int T, int k, int h,
                    uint16_t* dyp, float* dw, cudaStream_t st) {
  if (T < 1 || h % 4) return -1;
  // whole warps (the block sum shuffles over full warps); idle threads add 0
  moe_combine_bwd_kernel<<<T, h / 4 >= 256 ? 256 : 128, 0, st>>>(dh, yp, spos, w, k, h, dyp, dw);
  count_launches(1);
  return launched() ? 0 : -1;
}

int moe_unpermute(const float* dxp, const int32_t* spos, int T, int k, int h, float* dm, cudaStream_t st) {
  if (T < 1 || h % 4) return -1;
  moe_unpermute_kernel<<<T, std::min(256, h / 4), 0, st>>>(dxp, spos, k, h, dm);
  count_launches(1);
  return launched() ? 0 : -1;
}

int moe_router_bwd(const float* w, const float* dw, const int32_t* sel, int T, int k, int E, uint16_t* dr,
                   cudaStream_t st) {
  if (T < 1 || E < 1) return -1;
  const size_t n = (size_t)T * E;
  moe_router_bwd_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(w, dw, sel, T, k, E, dr);
  count_launches(1);
  return launched() ? 0 : -1;
}

}  // namespace mt
