// Host runtime of the layer-streamed step: packed layout, device arena
// partition, and the StreamIn-Bind-Compute-Offload schedule over three CUDA
// streams ordered by events ("MegaTrain: Full Precision Training of 100B+
// Parameter Large Language Models on a Single GPU", sections 核心方法,
// 方法步骤详情 and 技术新颖性).
//
//  - Host memory is the parameter and gradient store; the device holds two
//    weight buffers (ping-pong: the copy of unit i+1 runs while unit i
//    computes), two gradient staging buffers (the D2H copy of layer i's
//    gradients runs while layer i-1 back-propagates), the residual-stream
//    checkpoints h_0, h_K, h_2K, ... and the saved activations of one block
//    of K layers.
//  - The weight stream waits "buffer-free" before overwriting a buffer and
//    records "weight-ready"; the compute stream waits "weight-ready", and
//    "gradient-buffer-free" before writing a staging buffer, then records
//    "backward-done"; the grad stream waits "backward-done", copies, records
//    "gradient-buffer-free". No host barrier inside the step; no CUDA graph
//    (the bound weights change every unit).
//  - Block loop (the pages' loop bounds overrun L when L is a multiple of K;
//    the reading taken here): blocks b = ceil(L/K)-1 .. 0 cover layers
//    bK+1 .. min((b+1)K, L); the top block's activations are still in the
//    block arena after the forward pass, so it is not recomputed (the
//    result is identical; RoundPipe's "fused stage" observation).
#include <algorithm>
#include <chrono>
#include <memory>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <atomic>
#include <thread>
#include <type_traits>
#include <vector>

#include <sys/syscall.h>
#include <unistd.h>

#include "../../include/mt.h"
#include "common.cuh"
#include "kernels.h"

#include <nvtx3/nvToolsExt.h>

using namespace mt;

namespace mt {
long g_kernel_launches = 0;
}

namespace {

size_t rup(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---------------------------------------------------------------------------
// Packed layout
// ---------------------------------------------------------------------------
int tensors_in_unit(const mt_layer_cfg& c, int u) {
  if (u == 0) return 1;
  if (u >= 1 && u <= c.n_layers) return 9;
  if (u == c.n_layers + 1) return 2;
  return 0;
}

size_t tensor_numel(const mt_layer_cfg& c, int u, int t) {
  const size_t h = c.hidden, qd = (size_t)c.n_heads * c.head_dim, kd = (size_t)c.n_kv_heads * c.head_dim,
               F = c.ffn_dim, V = c.vocab;
  if (u == 0) return V * h;
  if (u == c.n_layers + 1) return t == 0 ? h : V * h;
  if (c.n_experts > 0 && t >= 6) {  // router Wr[E,h], experts' Wgu[E,2Fe,h], Wd[E,h,Fe]
    const size_t E = c.n_experts, Fe = c.expert_ffn;
    return t == 6 ? E * h : t == 7 ? E * 2 * Fe * h : E * h * Fe;
  }
  static const int kind[9] = {0, 1, 2, 2, 3, 0, 4, 4, 4};
  switch (kind[t]) {
    case 0: return h;
    case 1: return qd * h;
    case 2: return kd * h;
    case 3: return h * qd;
    default: return F * h;
  }
}

bool is_gain(const mt_layer_cfg& c, int u, int t) {
  return (u >= 1 && u <= c.n_layers && (t == 0 || t == 5)) || (u == c.n_layers + 1 && t == 0);
}

// Columns (the reduction width) of a matrix tensor of a dense model.
size_t tensor_cols(const mt_layer_cfg& c, int u, int t) {
  if (u >= 1 && u <= c.n_layers && t == 4) return (size_t)c.n_heads * c.head_dim;  // Wo[h, qd]
  if (u >= 1 && u <= c.n_layers && t == 8)  // Wd[h, F], or every expert's Wd[h, Fe]
    return (size_t)(c.n_experts ? c.expert_ffn : c.ffn_dim);
  return (size_t)c.hidden;  // mixture of experts: Wr[E, h] and Wgu[E * 2Fe, h] rows
}

// Bytes of one packed tensor. esz 4 / 2: fp32 / bf16 elements. esz 1: the
// FP8 layout: every matrix is its e4m3 codes, row-major [rows, cols], then
// (at the next 16-byte boundary) one fp32 scale per row; the RMSNorm gains
// stay fp32.
size_t tensor_bytes(const mt_layer_cfg& c, int u, int t, size_t esz) {
  const size_t n = tensor_numel(c, u, t);
  if (esz != 1) return n * esz;
  if (is_gain(c, u, t)) return n * 4;
  return rup(n, 16) + n / tensor_cols(c, u, t) * 4;
}

// offsets[u][t] in bytes for element size esz (1: FP8 with row scales);
// returns total bytes.
size_t build_layout(const mt_layer_cfg& c, size_t esz, std::vector<std::vector<size_t>>* offs) {
  size_t pos = 0;
  if (offs) offs->assign(c.n_layers + 2, {});
  for (int u = 0; u <= c.n_layers + 1; ++u) {
    pos = rup(pos, 4096);
    for (int t = 0; t < tensors_in_unit(c, u); ++t) {
      pos = rup(pos, 256);
      if (offs) (*offs)[u].push_back(pos);
      pos += tensor_bytes(c, u, t, esz);
    }
  }
  return rup(pos, 4096);
}

size_t dtype_esz(int dtype) { return dtype == MT_BF16 ? 2 : dtype == MT_FP8 ? 1 : 4; }

// ---------------------------------------------------------------------------
// FP8 e4m3 (the OCP 8-bit format E4M3: sign, 4 exponent bits with bias 7, 3
// mantissa bits; no infinities; S.1111.111 is NaN; largest finite 448) and
// the row-scaled weight encoding of the FP8 packed layout.
// ---------------------------------------------------------------------------
float e4m3_decode(uint8_t code) {
  const int e = (code >> 3) & 15, m = code & 7;
  float v;
  if (e == 15 && m == 7) v = NAN;
  else if (e == 0) v = std::ldexp((float)m, -9);
  else v = std::ldexp(1.f + m / 8.f, e - 7);
  return (code & 0x80) ? -v : v;
}

// Nearest e4m3 value (ties to even mantissa), saturating at +-448. x finite.
uint8_t e4m3_encode(float x) {
  const uint8_t sign = std::signbit(x) ? 0x80 : 0;
  const float a = std::fabs(x);
  if (a >= 448.f) return sign | 0x7E;
  if (a < 0.015625f) {  // below 2^-6: subnormal steps of 2^-9 (8 steps reach the smallest normal)
    const int m = (int)std::nearbyint(a * 512.f);  // exact scaling, then round half to even
    return sign | (uint8_t)m;                          // m == 8 is exactly the code of 2^-6
  }
  int e;
  std::frexp(a, &e);  // a = f 2^e, f in [0.5, 1)
  e -= 1;             // a in [2^e, 2^(e+1)), e in [-6, 8]
  int m = (int)std::nearbyint((std::ldexp(a, -e) - 1.f) * 8.f);
  if (m == 8) {
    m = 0;
    e += 1;
  }
  if (e > 8 || (e == 8 && m > 6)) return sign | 0x7E;
  return sign | (uint8_t)(((e + 7) << 3) | m);
}

// bf16 bits of the dequantised weight: bf16(float(code) * scale).
inline uint16_t host_bf16_rne(float f);
uint16_t e4m3_dequant_bf16(uint8_t code, float scale) { return host_bf16_rne(e4m3_decode(code) * scale); }

// ---------------------------------------------------------------------------
// AdamW on the host (MegaTrain stage 4), fp32, over packed units.
// ---------------------------------------------------------------------------
struct AdamCoef {
  float lr, b1, omb1, b2, omb2, bc1, bc2, eps, wd;
};

AdamCoef adam_coef(const mt_adamw_cfg& o, int64_t step) {
  AdamCoef c;
  c.lr = o.lr;
  c.b1 = o.beta1;
  c.omb1 = 1.f - o.beta1;
  c.b2 = o.beta2;
  c.omb2 = 1.f - o.beta2;
  c.bc1 = (float)(1.0 / (1.0 - std::pow((double)o.beta1, (double)step)));
  c.bc2 = (float)(1.0 / (1.0 - std::pow((double)o.beta2, (double)step)));
  c.eps = o.eps;
  c.wd = o.weight_decay;
  return c;
}

inline uint16_t host_bf16_rne(float f) {  // round to nearest even
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x7fffffu)) return (uint16_t)((u >> 16) | 0x40);  // quiet NaN
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

// n elements of one tensor: master w, moments m, v, gradient g; the streamed
// copy p is bf16 (OutT = uint16_t), fp32 (float) or not written (void).
// Non-aliasing arrays and no per-element branches, so the loop vectorizes.
template <typename OutT>
void adamw_span_t(const AdamCoef c, float* __restrict__ w, float* __restrict__ m, float* __restrict__ v,
                  const float* __restrict__ g, OutT* __restrict__ p, size_t n) {
  for (size_t i = 0; i < n; ++i) {
    const float gi = g[i];
    const float mi = c.b1 * m[i] + c.omb1 * gi;
    const float vi = c.b2 * v[i] + c.omb2 * (gi * gi);
    m[i] = mi;
    v[i] = vi;
    const float wi = w[i];
    const float nw = wi - c.lr * ((mi * c.bc1) / (std::sqrt(vi * c.bc2) + c.eps) + c.wd * wi);
    w[i] = nw;
    if constexpr (std::is_same<OutT, uint16_t>::value) {
      uint32_t u;
      std::memcpy(&u, &nw, 4);
      p[i] = (uint16_t)((u + 0x7fffu + ((u >> 16) & 1u)) >> 16);  // round to nearest even (finite values)
    } else if constexpr (std::is_same<OutT, float>::value) {
      p[i] = nw;
    }
  }
}
void adamw_span(const AdamCoef& c, float* w, float* m, float* v, const float* g, uint16_t* pb, float* pf, size_t n) {
  if (pb) adamw_span_t<uint16_t>(c, w, m, v, g, pb, n);
  else if (pf) adamw_span_t<float>(c, w, m, v, g, pf, n);
  else adamw_span_t<void>(c, w, m, v, g, (void*)nullptr, n);
}

// Rewrite the streamed copy of units [u0, u1) from the fp32 master.
void publish_units(const mt_layer_cfg& cfg, const std::vector<std::vector<size_t>>& off32,
                   const std::vector<std::vector<size_t>>& offp, size_t esz, int u0, int u1, const float* master,
                   void* params, int nthr) {
  std::vector<std::thread> th;
  for (int u = u0; u < u1; ++u)
    for (int t = 0; t < tensors_in_unit(cfg, u); ++t) {
      const size_t n = tensor_numel(cfg, u, t);
      const float* src = master + off32[u][t] / 4;
      const size_t per = std::max<size_t>((n + nthr - 1) / nthr, 1 << 16);
      for (size_t lo = 0; lo < n; lo += per) {
        const size_t hi = std::min(n, lo + per);
        if (esz == 2) {
          uint16_t* dst = (uint16_t*)params + offp[u][t] / 2;
          th.emplace_back([=] {
            for (size_t i = lo; i < hi; ++i) dst[i] = host_bf16_rne(src[i]);
          });
        } else {
          float* dst = (float*)params + offp[u][t] / 4;
          th.emplace_back([=] { std::memcpy(dst + lo, src + lo, (hi - lo) * 4); });
        }
      }
      if (th.size() >= (size_t)nthr) {
        for (auto& x : th) x.join();
        th.clear();
      }
    }
  for (auto& x : th) x.join();
}

// Update units [u0, u1) with nthr threads splitting the elements evenly.
void adamw_units(const mt_layer_cfg& cfg, const std::vector<std::vector<size_t>>& off32,
                 const std::vector<std::vector<size_t>>& offp, size_t esz, const AdamCoef& c, int u0, int u1,
                 float* master, float* m, float* v, const float* grads, void* params, int nthr) {
  struct Span {
    size_t o32, op, n;
  };
  std::vector<Span> spans;
  size_t total = 0;
  for (int u = u0; u < u1; ++u)
    for (int t = 0; t < tensors_in_unit(cfg, u); ++t) {
      const size_t n = tensor_numel(cfg, u, t);
      spans.push_back({off32[u][t] / 4, offp[u][t] / esz, n});
      total += n;
    }
  if (!total) return;
  auto run = [&](size_t lo, size_t hi) {  // element range [lo, hi) of the concatenated spans
    size_t base = 0;
    for (const Span& sp : spans) {
      const size_t a = std::max(lo, base), b = std::min(hi, base + sp.n);
      if (a < b) {
        const size_t k = sp.o32 + (a - base), kp = sp.op + (a - base);
        adamw_span(c, master + k, m + k, v + k, grads + k, params && esz == 2 ? (uint16_t*)params + kp : nullptr,
                   params && esz == 4 ? (float*)params + kp : nullptr, b - a);
      }
      base += sp.n;
      if (base >= hi) break;
    }
  };
  const size_t per = std::max<size_t>((total + nthr - 1) / nthr, 1 << 16);
  std::vector<std::thread> th;
  for (size_t lo = per; lo < total; lo += per) th.emplace_back(run, lo, std::min(total, lo + per));
  run(0, std::min(total, per));
  for (auto& x : th) x.join();
}

bool cfg_valid(const mt_layer_cfg& c, std::string* why) {
  auto fail = [&](const char* m) {
    if (why) *why = m;
    return false;
  };
  const bool moe = c.n_experts != 0 || c.top_k != 0 || c.expert_ffn != 0;
  if (c.n_layers < 1 || c.hidden < 64 || c.n_heads < 1 || c.n_kv_heads < 1 || (!moe && c.ffn_dim < 1) ||
      c.vocab < 1)
    return fail("non-positive dimension");
  if (moe) {
    if (c.ffn_dim != 0) return fail("mixture-of-experts layers take ffn_dim = 0");
    if (c.n_experts < 8 || c.n_experts > 1024 || c.n_experts % 8)
      return fail("n_experts must be a multiple of 8 in [8, 1024]");
    if (c.top_k < 1 || c.top_k > 32 || c.top_k > c.n_experts) return fail("top_k must be in [1, min(32, n_experts)]");
    if (c.expert_ffn < 32 || c.expert_ffn % 32) return fail("expert_ffn must be a positive multiple of 32");
    if (c.param_dtype != MT_BF16 && c.param_dtype != MT_FP8)
      return fail("mixture-of-experts layers need bf16 or FP8 params");
  }
  if (c.hidden % 64) return fail("hidden must be a multiple of 64");
  if (c.hidden > 8192) return fail("hidden above 8192 is not supported");
  if (c.n_heads % c.n_kv_heads) return fail("n_heads must be a multiple of n_kv_heads");
  if (c.head_dim != 16 && c.head_dim != 32 && c.head_dim != 64 && c.head_dim != 128)
    return fail("head_dim must be 16, 32, 64 or 128");
  if (c.param_dtype != MT_F32 && c.param_dtype != MT_BF16 && c.param_dtype != MT_FP8)
    return fail("param_dtype must be MT_F32, MT_BF16 or MT_FP8");
  if (c.param_dtype == MT_FP8 && c.ffn_dim % 16) return fail("FP8 params need ffn_dim % 16 == 0");
  if (c.grad_dtype != MT_F32 && c.grad_dtype != MT_BF16) return fail("grad_dtype must be MT_F32 or MT_BF16");
  if (c.param_dtype == MT_BF16 && c.ffn_dim % 8) return fail("bf16 params need ffn_dim % 8 == 0");
  if (c.max_batch < 1 || c.max_seq < 1 || c.max_K < 1) return fail("max_batch, max_seq, max_K must be >= 1");
  if (!(c.rope_theta > 0.f) || !(c.norm_eps > 0.f)) return fail("rope_theta and norm_eps must be positive");
  if ((double)c.max_batch * c.max_seq > 2147483647.0 / 4) return fail("too many tokens");
  if (moe && (double)c.max_batch * c.max_seq * c.top_k * std::max(c.hidden, 2 * c.expert_ffn) > 2147483647.0 * 4)
    return fail("too many routed rows");
  return true;
}

// ---------------------------------------------------------------------------
// Arena plan
// ---------------------------------------------------------------------------
struct Plan {
  // dims
  int L, h, nq, nkv, d, F, Fp, V, qd, kd, qkv, Tmax;
  int E, topk, Fe;  // mixture-of-experts FFN when E > 0 (F = Fp = 0)
  int n_pad;        // routed rows incl. padding of every expert segment to 128 rows
  size_t esz;
  size_t gesz;  // element size of the streamed gradients (4: fp32, 2: bf16)
  int gepi;     // GEMM epilogue that writes a weight gradient
  // slicing of vocab-sized units
  int head_rows, n_head_slices;
  // sizes
  size_t wbuf, wcast, gbuf, ckpt_one, act_layer, fixed_ws, dyn_max, total;
  // activation layout inside one block-arena slot (byte offsets)
  size_t o_x, o_a, o_rstd1, o_qkv, o_o, o_lse, o_hmid, o_m, o_rstd2, o_gu, o_act;
  // mixture-of-experts slot: router logits, selection, weights, slot <-> row
  // maps, and the routed rows (grouped by expert) with their activations
  size_t o_r, o_sel, o_w, o_spos, o_seg, o_tile_e, o_xp, o_gup, o_actp, o_yp;
};

// Bytes of a head vocab slice of `rows` rows in a weight buffer (FP8: the
// codes, then the row scales at the next 256-byte boundary).
size_t head_slice_bytes(const Plan& p, int rows) {
  if (p.esz == 1) return rup((size_t)rows * p.h, 256) + (size_t)rows * 4;
  return (size_t)rows * p.h * p.esz;
}

size_t layer_cast_bytes(const Plan& p) {  // device bf16 view of one layer (fp32 or FP8 params)
  const size_t attn = rup((size_t)p.qkv * p.h * 2, 256) + rup((size_t)p.h * p.qd * 2, 256);
  if (p.E > 0)  // router, every expert's gate|up and down
    return attn + rup((size_t)p.E * p.h * 2, 256) + rup((size_t)p.E * 2 * p.Fe * p.h * 2, 256) +
           rup((size_t)p.E * p.h * p.Fe * 2, 256);
  return attn + rup((size_t)2 * p.Fp * p.h * 2, 256) + rup((size_t)p.h * p.Fp * 2, 256);
}

bool make_plan(const mt_layer_cfg& c, Plan* P) {
  Plan& p = *P;
  p.L = c.n_layers;
  p.h = c.hidden;
  p.nq = c.n_heads;
  p.nkv = c.n_kv_heads;
  p.d = c.head_dim;
  p.F = c.ffn_dim;
  p.Fp = c.param_dtype == MT_F32 ? (int)rup(c.ffn_dim, 8) : c.ffn_dim;
  p.V = c.vocab;
  p.qd = p.nq * p.d;
  p.kd = p.nkv * p.d;
  p.qkv = p.qd + 2 * p.kd;
  p.Tmax = c.max_batch * c.max_seq;
  p.esz = dtype_esz(c.param_dtype);
  p.gesz = c.grad_dtype == MT_BF16 ? 2 : 4;
  p.gepi = p.gesz == 2 ? EPI_BF16 : EPI_F32;
  p.E = c.n_experts;
  p.topk = c.top_k;
  p.Fe = c.expert_ffn;
  p.n_pad = p.E ? (int)rup((size_t)p.Tmax * p.topk + (size_t)p.E * 127, 128) : 0;
  std::vector<std::vector<size_t>> o;
  build_layout(c, p.esz, &o);
  const size_t layer_bytes = (o[1][8] + tensor_bytes(c, 1, 8, p.esz)) - o[1][0];
  // vocab slices: the fewest equal slices (multiples of 256 rows) that fit a layer buffer
  // (FP8: a slice's codes, then its row scales at the next 256-byte boundary)
  auto slices = [&](size_t row_bytes, size_t cap, int* rows, int* n) {
    int ns = (int)std::max<size_t>(1, (p.V * row_bytes + cap - 1) / cap);
    while (true) {
      int r = (int)rup((p.V + ns - 1) / ns, 256);
      if (r > p.V) r = p.V;
      if ((size_t)r * row_bytes <= cap || r <= 256) {
        *rows = r;
        *n = (p.V + r - 1) / r;
        return;
      }
      ++ns;
    }
  };
  if (p.esz == 1) slices((size_t)p.h + 4, layer_bytes - 256, &p.head_rows, &p.n_head_slices);
  else slices((size_t)p.h * p.esz, layer_bytes, &p.head_rows, &p.n_head_slices);
  std::vector<std::vector<size_t>> og;
  build_layout(c, p.gesz, &og);
  const size_t layer_grad_bytes = (og[1][8] + tensor_numel(c, 1, 8) * p.gesz) - og[1][0];
  p.wbuf = rup(std::max(layer_bytes, head_slice_bytes(p, p.head_rows)), 4096);
  // fp32 and FP8 host params are turned into a bf16 view on the device
  p.wcast = p.esz != 2 ? rup(std::max(layer_cast_bytes(p), (size_t)p.head_rows * p.h * 2), 4096) : 0;
  p.gbuf = rup(std::max({layer_grad_bytes, (size_t)p.head_rows * p.h * p.gesz, (size_t)p.h * p.gesz}), 4096);
  const size_t T = p.Tmax, h = p.h;
  p.ckpt_one = rup(T * h * 4, 256);
  size_t a = 0;
  auto take = [&](size_t bytes) {
    size_t r = a;
    a += rup(bytes, 256);
    return r;
  };
  p.o_x = take(T * h * 4);
  p.o_a = take(T * h * 2);
  p.o_rstd1 = take(T * 4);
  p.o_qkv = take(T * p.qkv * 2);
  p.o_o = take(T * p.qd * 2);
  p.o_lse = take(T * p.nq * 4);
  p.o_hmid = take(T * h * 4);
  p.o_m = take(T * h * 2);
  p.o_rstd2 = take(T * 4);
  p.o_gu = take(T * 2 * p.Fp * 2);
  p.o_act = take(T * p.Fp * 2);
  {
    const size_t E = p.E, R = T * p.topk, Rp = p.n_pad, Fe = p.Fe;  // all zero for dense layers
    p.o_r = take(T * E * 4);
    p.o_sel = take(R * 4);
    p.o_w = take(R * 4);
    p.o_spos = take(R * 4);
    p.o_seg = take((E + 1) * 4);
    p.o_tile_e = take(Rp / 128 * 4);
    p.o_xp = take(Rp * h * 2);
    p.o_gup = take(Rp * 2 * Fe * 2);
    p.o_actp = take(Rp * Fe * 2);
    p.o_yp = take(Rp * h * 4);
  }
  p.act_layer = rup(a, 4096);
  // fixed workspace (see Ctx::carve)
  size_t w = 0;
  auto ws = [&](size_t bytes) { w += rup(bytes, 256); };
  ws(T * h * 4);                                   // h_top (h_L)
  ws(T * h * 4);                                   // dh
  ws(T * h * 2);                                   // dh bf16
  ws(T * h * 4);                                   // dm / da / dxf
  ws(T * h * 2);                                   // dhmid bf16
  ws(T * p.qd * 2);                                // do
  ws(T * p.qkv * 2);                               // dqkv
  ws(attention_bwd_workspace(c.max_batch, c.max_seq, p.nq) * 4);
  ws(rmsnorm_bwd_partials((int)T, p.h) * 4);
  ws(T * h * 2);                                   // xf bf16
  ws(T * 4);                                       // rstd_f
  ws(T * (size_t)p.head_rows * 4);                 // logits slice fp32
  ws(T * (size_t)p.head_rows * 2);                 // dz slice bf16
  ws((size_t)p.n_head_slices * T * 8);             // CE partials
  ws(T * 4 * 3);                                   // zlab, lse, terms
  ws(256);                                         // loss
  ws((T * 5 + 1) * 4);                             // tokens, labels, perm, used ids, id ranges
  ws((size_t)c.max_seq * p.d / 2 * 8);             // rope table
  ws(2 * 2 * (size_t)p.h * 4);                     // gains of the two weight slots
  ws((size_t)p.h * 4 * 2);                         // final norm gain (raw + fp32)
  ws((size_t)p.n_pad * p.h * 2);                   // MoE: d(routed outputs) bf16
  ws(T * p.topk * 4);                              // MoE: d(weights)
  ws(T * (size_t)p.E * 2);                         // MoE: d(router logits) bf16
  ws(((size_t)p.E + 1) * 4);                       // MoE: expert counts
  ws((size_t)p.h * 4);                             // a gain gradient before its bf16 rounding
  ws((size_t)p.L * T * p.topk * 4);                // MoE: routing of every layer
  p.fixed_ws = w;
  // dynamic part: checkpoints for ceil(L/K) blocks + K activation slots
  p.dyn_max = 0;
  for (int K = 1; K <= std::min(c.max_K, p.L); ++K) {
    const size_t nb = (p.L + K - 1) / K;
    p.dyn_max = std::max(p.dyn_max, nb * p.ckpt_one + (size_t)K * p.act_layer);
  }
  p.total = 2 * p.wbuf + 2 * p.wcast + 2 * p.gbuf + p.fixed_ws + p.dyn_max + 4096;
  return true;
}

// One use of a streamed weight unit (or vocab slice) by the compute stream.
enum ItemKind { IT_LAYER = 1, IT_HEAD = 2 };
struct Item {
  int kind, index;  // layer index 1..L, or slice index
  bool operator==(const Item& o) const { return kind == o.kind && index == o.index; }
};

// Pool of timing events.
struct Seg {
  int stream;  // 0 compute, 1 h2d, 2 d2h
  cudaEvent_t a, b;
  double bytes;
  int unit;    // position in the step's unit sequence (-1: none)
};
// Per-kernel timing (trace level 2): category 0 GEMM, 1 attention.
struct OpSeg {
  int cat;
  cudaEvent_t a, b;
  double flop;
};

// Host page toucher. Reads one byte of every 4 KB of the host ranges the
// step's copies are about to read (weights) or write (gradients), from a few
// host threads, a fixed number of weight copies ahead of the weight stream
// (paced on per-copy completion events). Measured on the GB300 machines: pinned
// host pages that only the GPU accesses lose their mapping on the host side
// after some idle time (in 4 KB units), and the copy engines then stall on
// every such page (4-13 GB/s instead of 211 GB/s for weight copies, 28 GB/s
// for gradient copies); a CPU read of each 4 KB page restores the mapping
// cheaply, so the copy that follows runs at the link rate. The touches are
// reads only: no byte of either buffer is changed.
class PageToucher {
 public:
  struct Range {
    const uint8_t* p;
    size_t bytes;
    int wait;  // touch once weight copy `wait` has completed (-1: at once)
  };
  PageToucher() = default;
  PageToucher(const PageToucher&) = delete;
  PageToucher& operator=(const PageToucher&) = delete;
  ~PageToucher() { stop(); }

  // Touch ranges[0..] in order with nthreads threads (each a contiguous part
  // of every range); range r waits for weight copy r.wait (of n_copies) to
  // complete.
  void start(std::vector<Range> ranges, size_t n_copies, int nthreads, int device) {
    r_ = std::move(ranges);
    ev_.assign(n_copies, nullptr);
    touched_.reset(new std::atomic<int>[r_.size() + 1]);
    for (size_t j = 0; j <= r_.size(); ++j) touched_[j] = 0;
    n_ = std::max(1, nthreads);
    busy_.assign(n_, 0.0);
    for (int w = 0; w < n_; ++w) th_.emplace_back([this, w, device] { run(w, device); });
  }
  // Weight copy j has been issued; `done` completes with it (copies are
  // published in order).
  void published(size_t j, cudaEvent_t done) {
    if (j >= ev_.size()) return;
    ev_[j] = done;
    published_.store(j + 1, std::memory_order_release);
  }
  // Wait (bounded) until every thread has touched range j.
  bool wait_touched(size_t j, double seconds) {
    if (th_.empty() || j >= r_.size()) return true;
    const auto t0 = std::chrono::steady_clock::now();
    while (touched_[j].load(std::memory_order_acquire) < n_) {
      if (std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count() > seconds) return false;
      std::this_thread::sleep_for(std::chrono::microseconds(20));
    }
    return true;
  }
  void stop() {
    stop_ = true;
    for (auto& t : th_)
      if (t.joinable()) t.join();
    th_.clear();
  }
  double busy_ms() const {
    double b = 0;
    for (double x : busy_) b = std::max(b, x);
    return b;
  }

 private:
  void run(int w, int device) {
    cudaSetDevice(device);
    double busy = 0;
    uint64_t acc = 0;
    for (size_t j = 0; j < r_.size() && !stop_; ++j) {
      if (r_[j].wait >= 0 && (size_t)r_[j].wait < ev_.size()) {
        const size_t k = (size_t)r_[j].wait;
        while (published_.load(std::memory_order_acquire) <= k) {
          if (stop_) return;
          std::this_thread::sleep_for(std::chrono::microseconds(20));
        }
        while (cudaEventQuery(ev_[k]) == cudaErrorNotReady) {
          if (stop_) return;
          std::this_thread::sleep_for(std::chrono::microseconds(50));
        }
      }
      const auto t0 = std::chrono::steady_clock::now();
      const size_t pages = (r_[j].bytes + 4095) / 4096;
      const size_t per = (pages + n_ - 1) / n_;
      const volatile uint8_t* q = r_[j].p;
      for (size_t pg = (size_t)w * per; pg < std::min(pages, (size_t)(w + 1) * per); ++pg) acc += q[pg * 4096];
      busy += std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
      touched_[j].fetch_add(1, std::memory_order_release);
    }
    cudaGetLastError();
    busy_[w] = busy;
    sink_ += acc;
  }
  std::vector<Range> r_;
  std::vector<cudaEvent_t> ev_;
  std::unique_ptr<std::atomic<int>[]> touched_;
  std::atomic<size_t> published_{0};
  std::atomic<bool> stop_{false};
  std::atomic<uint64_t> sink_{0};
  std::vector<std::thread> th_;
  std::vector<double> busy_;
  int n_ = 1;
};

}  // namespace

struct mt_ctx {
  mt_layer_cfg cfg;
  Plan P;
  std::vector<std::vector<size_t>> off_p, off_g;  // host param layout, host gradient layout (grad_dtype)
  int device = 0;
  cudaStream_t s_comp = nullptr, s_h2d = nullptr, s_d2h = nullptr;
  bool own_streams = false;
  // optimizer state (mt_bind_optimizer)
  bool opt_bound = false;
  mt_adamw_cfg opt{};
  float *opt_master = nullptr, *opt_m = nullptr, *opt_v = nullptr;
  int opt_threads = 0;
  int64_t opt_step = 1;
  // asynchronous form (mt_train_step_async): gradients of the previous call,
  // whose update is applied during the next call, and per unit how far that
  // update has gone (0 not computed, 1 computed into the master and
  // moments, 2 also published to the streamed copy), so that a call that
  // fails part-way is completed by the next call or mt_optimizer_flush
  // without applying any unit's update twice
  const float* opt_pending = nullptr;
  std::vector<uint8_t> opt_state;
  cudaEvent_t ev_wready[2], ev_wfree[2], ev_bwd_done[2], ev_gfree[2], ev_done = nullptr;
  uint8_t* arena = nullptr;
  size_t arena_bytes = 0;
  bool own_arena = false;
  // carved regions
  uint8_t* wbuf[2];
  uint16_t* wcast[2];
  float* gbuf[2];
  uint8_t* dyn = nullptr;
  float *h_top, *dh, *dm, *attn_ws, *norm_ws, *rstd_f, *logits, *zlab, *lse, *terms, *loss_dev, *gains[2], *wf32;
  uint16_t *dh_b, *dhmid_b, *do_b, *dqkv, *xf_b, *dz;
  float2 *ce_part, *rope_tab;
  int32_t *tok_d, *lab_d, *perm_d, *ids_d, *ids_start_d;
  // mixture-of-experts: d(routed outputs), d(weights), d(router logits),
  // expert counts, the routing of every layer
  uint16_t *moe_dyp = nullptr, *moe_dr = nullptr;
  float* moe_dw = nullptr;
  int32_t *moe_counts = nullptr, *moe_route = nullptr;
  float* gain_grad = nullptr;  // bf16 gradients: an RMSNorm gain's fp32 gradient before rounding
  const void* host_params_dev = nullptr;  // device-side address of the bound host parameters
  void* wf_raw;
  int32_t* host_stage = nullptr;  // pinned: tokens, labels, perm, used ids, id ranges, loss
  uint8_t* host_rows = nullptr;   // pinned staging: embedding rows of the tokens [T, h] (param dtype)
  float* host_grad_rows = nullptr;  // pinned staging: embedding gradient rows of the used ids [T, h]
  int rope_S = -1;
  int last_T = 0;  // tokens of the last step that ran to completion
  std::vector<int32_t> csr;  // token-id counting sort (vocab + 1)
  const void* host_params = nullptr;
  std::string err;
  mt_stats stats{};
  int trace = 1;
  bool fuse_top = true;
  bool debug_sync = false;  // MT_DEBUG_SYNC=1: wait for every unit, report progress on stderr
  bool serial = false;      // MT_SERIAL=1: no copy/compute overlap (ablation)
  bool nvtx = false;        // MT_NVTX=1: an NVTX range around the issue of every unit (for nsys)
  std::string timeline;     // MT_TIMELINE=path: write the step's segments as CSV
  std::vector<Seg> segs;
  std::vector<OpSeg> opsegs;
  long launches_at_start = 0;
  int trace_sample = 16;    // MT_TRACE_SAMPLE: time 1 in N GEMM/attention launches at trace level 2
  long op_counter = 0;
  std::vector<cudaEvent_t> ev_pool;
  size_t ev_used = 0;
  cudaEvent_t ev_base = nullptr;
  int fault_kind = 0, fault_nth = 0, fault_count = 0;
  int gslot = 0;
  // phase of every position of the step's unit sequence (0 forward, 1 LM
  // head, 2 recompute, 3 backward) and the position being issued, for the
  // per-phase copy statistics
  std::vector<int8_t> unit_phase;
  int cur_unit = -1;
  int touch_threads = 4;  // host page toucher threads (MT_PAGE_TOUCH; 0: off)
};

namespace {

int set_err(mt_ctx* c, int code, const std::string& m) {
  if (c) c->err = m;
  return code;
}

#define CK(call)                                                                               \
  do {                                                                                         \
    cudaError_t e_ = (call);                                                                   \
    if (e_ != cudaSuccess)                                                                     \
      return set_err(ctx, MT_ERR_CUDA, std::string(#call) + ": " + cudaGetErrorString(e_));  \
  } while (0)
#define CKL(call)                                                                \
  do {                                                                           \
    if ((call) != 0) {                                                           \
      cudaError_t e_ = cudaGetLastError();                                       \
      return set_err(ctx, e_ != cudaSuccess ? MT_ERR_CUDA : MT_ERR_ARG,          \
                     std::string(#call) + " failed: " + cudaGetErrorString(e_)); \
    }                                                                            \
  } while (0)

int carve(mt_ctx* ctx) {
  const Plan& p = ctx->P;
  uint8_t* cur = (uint8_t*)rup((uintptr_t)ctx->arena, 4096);
  auto take = [&](size_t bytes) {
    uint8_t* r = cur;
    cur += rup(bytes, 256);
    return r;
  };
  for (int i = 0; i < 2; ++i) ctx->wbuf[i] = take(p.wbuf);
  for (int i = 0; i < 2; ++i) ctx->wcast[i] = p.wcast ? (uint16_t*)take(p.wcast) : nullptr;
  for (int i = 0; i < 2; ++i) ctx->gbuf[i] = (float*)take(p.gbuf);
  const size_t T = p.Tmax, h = p.h;
  ctx->h_top = (float*)take(T * h * 4);
  ctx->dh = (float*)take(T * h * 4);
  ctx->dh_b = (uint16_t*)take(T * h * 2);
  ctx->dm = (float*)take(T * h * 4);
  ctx->dhmid_b = (uint16_t*)take(T * h * 2);
  ctx->do_b = (uint16_t*)take(T * p.qd * 2);
  ctx->dqkv = (uint16_t*)take(T * p.qkv * 2);
  ctx->attn_ws = (float*)take(attention_bwd_workspace(ctx->cfg.max_batch, ctx->cfg.max_seq, p.nq) * 4);
  ctx->norm_ws = (float*)take(rmsnorm_bwd_partials((int)T, p.h) * 4);
  ctx->xf_b = (uint16_t*)take(T * h * 2);
  ctx->rstd_f = (float*)take(T * 4);
  ctx->logits = (float*)take(T * (size_t)p.head_rows * 4);
  ctx->dz = (uint16_t*)take(T * (size_t)p.head_rows * 2);
  ctx->ce_part = (float2*)take((size_t)p.n_head_slices * T * 8);
  ctx->zlab = (float*)take(T * 4);
  ctx->lse = (float*)take(T * 4);
  ctx->terms = (float*)take(T * 4);
  ctx->loss_dev = (float*)take(256);
  int32_t* ints = (int32_t*)take((T * 5 + 1) * 4);
  ctx->tok_d = ints;
  ctx->lab_d = ints + T;
  ctx->perm_d = ints + 2 * T;
  ctx->ids_d = ints + 3 * T;
  ctx->ids_start_d = ints + 4 * T;
  ctx->rope_tab = (float2*)take((size_t)ctx->cfg.max_seq * p.d / 2 * 8);
  ctx->gains[0] = (float*)take(2 * (size_t)p.h * 4);
  ctx->gains[1] = (float*)take(2 * (size_t)p.h * 4);
  ctx->wf_raw = take((size_t)p.h * 4);
  ctx->wf32 = (float*)take((size_t)p.h * 4);
  ctx->moe_dyp = (uint16_t*)take((size_t)p.n_pad * h * 2);
  ctx->moe_dw = (float*)take(T * p.topk * 4);
  ctx->moe_dr = (uint16_t*)take(T * (size_t)p.E * 2);
  ctx->moe_counts = (int32_t*)take(((size_t)p.E + 1) * 4);
  ctx->gain_grad = (float*)take((size_t)p.h * 4);
  ctx->moe_route = (int32_t*)take((size_t)p.L * T * p.topk * 4);
  ctx->dyn = cur;
  cur += p.dyn_max;
  if ((size_t)(cur - ctx->arena) > ctx->arena_bytes) return set_err(ctx, MT_ERR_BUDGET, "arena too small for plan");
  return MT_OK;
}

// Bounded host wait on an event: polls with a deadline instead of blocking.
int wait_event(mt_ctx* ctx, cudaEvent_t ev, double seconds) {
  if (ctx->fault_kind == 2 && ++ctx->fault_count == ctx->fault_nth)
    return set_err(ctx, MT_ERR_TIMEOUT, "injected wait timeout");
  const auto t0 = std::chrono::steady_clock::now();
  while (true) {
    cudaError_t e = cudaEventQuery(ev);
    if (e == cudaSuccess) return MT_OK;
    if (e != cudaErrorNotReady) return set_err(ctx, MT_ERR_CUDA, std::string("event: ") + cudaGetErrorString(e));
    const double el = std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
    if (el > seconds) return set_err(ctx, MT_ERR_TIMEOUT, "step did not finish in time");
    std::this_thread::sleep_for(std::chrono::microseconds(el < 0.01 ? 20 : 200));
  }
}

cudaEvent_t next_event(mt_ctx* ctx) {
  if (ctx->ev_used >= ctx->ev_pool.size()) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    ctx->ev_pool.push_back(e);
  }
  return ctx->ev_pool[ctx->ev_used++];
}

// Timing segment helpers (only when tracing).
struct SegScope {
  mt_ctx* ctx;
  int idx = -1;
  cudaStream_t st;
  SegScope(mt_ctx* c, int stream_id, cudaStream_t s, double bytes, int unit = -1) : ctx(c), st(s) {
    if (!c->trace) return;
    cudaEvent_t a = next_event(c), b = next_event(c);
    if (!a || !b) return;
    cudaEventRecord(a, s);
    c->segs.push_back(Seg{stream_id, a, b, bytes, unit});
    idx = (int)c->segs.size() - 1;
  }
  ~SegScope() {
    if (idx >= 0) cudaEventRecord(ctx->segs[idx].b, st);
  }
};

struct LayerView {  // bf16 matrices and fp32 gains of one bound layer
  const uint16_t *wqkv, *wo, *wgu, *wd;
  const uint16_t* wr;  // mixture-of-experts router (wgu, wd then hold all experts)
  int ldd;  // row stride of Wd
  const float *w1, *w2;
};

struct ActSlot {
  float *x, *rstd1, *lse, *hmid, *rstd2;
  uint16_t *a, *qkv, *o, *m, *gu, *act;
  // mixture-of-experts
  float *r, *w, *yp;
  int32_t *sel, *spos, *seg, *tile_e;
  uint16_t *xp, *gup, *actp;
};

ActSlot act_slot(mt_ctx* ctx, int K, int nb, int j) {
  const Plan& p = ctx->P;
  uint8_t* base = ctx->dyn + (size_t)nb * p.ckpt_one + (size_t)j * p.act_layer;
  ActSlot s;
  s.x = (float*)(base + p.o_x);
  s.a = (uint16_t*)(base + p.o_a);
  s.rstd1 = (float*)(base + p.o_rstd1);
  s.qkv = (uint16_t*)(base + p.o_qkv);
  s.o = (uint16_t*)(base + p.o_o);
  s.lse = (float*)(base + p.o_lse);
  s.hmid = (float*)(base + p.o_hmid);
  s.m = (uint16_t*)(base + p.o_m);
  s.rstd2 = (float*)(base + p.o_rstd2);
  s.gu = (uint16_t*)(base + p.o_gu);
  s.act = (uint16_t*)(base + p.o_act);
  s.r = (float*)(base + p.o_r);
  s.sel = (int32_t*)(base + p.o_sel);
  s.w = (float*)(base + p.o_w);
  s.spos = (int32_t*)(base + p.o_spos);
  s.seg = (int32_t*)(base + p.o_seg);
  s.tile_e = (int32_t*)(base + p.o_tile_e);
  s.xp = (uint16_t*)(base + p.o_xp);
  s.gup = (uint16_t*)(base + p.o_gup);
  s.actp = (uint16_t*)(base + p.o_actp);
  s.yp = (float*)(base + p.o_yp);
  (void)K;
  return s;
}

float* ckpt(mt_ctx* ctx, int b) { return (float*)(ctx->dyn + (size_t)b * ctx->P.ckpt_one); }

// Brackets one kernel launch with events when per-kernel tracing is on.
struct OpTimer {
  mt_ctx* ctx;
  int idx = -1;
  OpTimer(mt_ctx* c, int cat, double flop) : ctx(c) {
    // Events around every launch would serialise the stream far more than
    // they measure, so only one launch in trace_sample is bracketed.
    if (c->trace < 2 || (c->op_counter++ % c->trace_sample) != 0) return;
    cudaEvent_t a = next_event(c), b = next_event(c);
    if (!a || !b) return;
    cudaEventRecord(a, c->s_comp);
    c->opsegs.push_back(OpSeg{cat, a, b, flop});
    idx = (int)c->opsegs.size() - 1;
  }
  ~OpTimer() {
    if (idx >= 0) cudaEventRecord(ctx->opsegs[idx].b, ctx->s_comp);
  }
};

int gemm_p(mt_ctx* ctx, int mode, const GemmParams& p, const void* A, const void* B, int lda, int ldb,
           double flop) {
  OpTimer timer(ctx, 0, flop);
  if (gemm_bf16(mode, p, A, B, lda, ldb, ctx->s_comp) != 0) {
    cudaError_t e = cudaGetLastError();
    char buf[256];
    snprintf(buf, sizeof buf, "gemm mode %d M=%d N=%d K=%d lda=%d ldb=%d ldc=%d failed: %s", mode, p.M, p.N, p.K, lda,
             ldb, p.ldc, cudaGetErrorString(e));
    return set_err(ctx, e != cudaSuccess ? MT_ERR_CUDA : MT_ERR_ARG, buf);
  }
  return MT_OK;
}

int gemm(mt_ctx* ctx, int mode, int epi, const void* A, const void* B, void* C, const void* add, int M, int N, int K,
         int lda, int ldb, int ldc, int rope_S = 0, int rope_cols = 0) {
  GemmParams p{M, N, K, epi, C, add, ldc, 0, 1};
  if (rope_cols > 0) {
    p.rope_tab = ctx->rope_tab;
    p.rope_S = rope_S;
    p.rope_d = ctx->P.d;
    p.rope_cols = rope_cols;
  }
  return gemm_p(ctx, mode, p, A, B, lda, ldb, 2.0 * M * N * K);
}

#define CKR(x)              \
  do {                      \
    int r_ = (x);           \
    if (r_ != MT_OK) return r_; \
  } while (0)

}  // namespace

// ===========================================================================
// The step
// ===========================================================================
namespace {

// An NVTX range (host side) around the issue of one unit, so that a
// system profiler attributes the unit's copies and kernels to it; a no-op
// unless enabled (and nearly free when no tool is attached).
struct NvtxRange {
  bool on;
  NvtxRange(bool enable, const char* name) : on(enable) {
    if (on) nvtxRangePushA(name);
  }
  ~NvtxRange() {
    if (on) nvtxRangePop();
  }
};

struct Step {
  mt_ctx* ctx;
  int B, S, T, K, nb;
  float* host_grad;
  std::vector<Item> seq;        // compute-stream consumption order
  std::vector<int> slot_of;     // slot per step
  std::vector<char> needs_load; // load before step
  bool train = false;                 // apply the optimizer as gradients land
  bool async = false;                 // apply the previous step's update, publishing units as they land
  std::vector<cudaEvent_t> landed;    // per unit (train steps): its gradients are on the host
  std::vector<int> load_index;        // per position of seq: index among the step's weight copies (-1: none)
  PageToucher* toucher = nullptr;
};

void plan_sequence(Step& st) {
  mt_ctx* ctx = st.ctx;
  const Plan& p = ctx->P;
  auto& q = st.seq;
  for (int l = 1; l <= p.L; ++l) q.push_back({IT_LAYER, l});
  for (int s = 0; s < p.n_head_slices; ++s) q.push_back({IT_HEAD, s});
  for (int s = p.n_head_slices - 1; s >= 0; --s) q.push_back({IT_HEAD, s});
  for (int b = st.nb - 1; b >= 0; --b) {
    const int lo = b * st.K + 1, hi = std::min((b + 1) * st.K, p.L);
    const bool recompute = !(b == st.nb - 1 && ctx->fuse_top);
    if (recompute)
      for (int l = lo; l <= hi; ++l) q.push_back({IT_LAYER, l});
    for (int l = hi; l >= lo; --l) q.push_back({IT_LAYER, -l});  // negative: backward use
  }
  // slots: a step reuses a slot that already holds its unit, otherwise loads
  // into the slot the previous step did not use.
  Item held[2] = {{-1, 0}, {-1, 0}};
  int prev = 1;
  for (size_t i = 0; i < q.size(); ++i) {
    Item key{q[i].kind, std::abs(q[i].index)};
    int s = -1;
    for (int k = 0; k < 2; ++k)
      if (held[k] == key) s = k;
    if (s >= 0) {
      st.slot_of.push_back(s);
      st.needs_load.push_back(0);
    } else {
      s = 1 - prev;
      held[s] = key;
      st.slot_of.push_back(s);
      st.needs_load.push_back(1);
    }
    prev = s;
  }
}

// Host byte range (offset into the bound parameters, bytes) that one use of
// a streamed unit copies: a layer's packed weights, or an LM-head vocab slice.
// FP8 head slices have a second range, their row scales (*scale_bytes > 0),
// copied to the weight buffer at head_scale_dst(rows).
void load_range(const mt_ctx* ctx, const Item& it, size_t* src_off, size_t* bytes, size_t* scale_off = nullptr,
                size_t* scale_bytes = nullptr) {
  const Plan& p = ctx->P;
  if (scale_bytes) *scale_bytes = 0;
  if (it.kind == IT_LAYER) {
    const int l = std::abs(it.index);
    *src_off = ctx->off_p[l][0];
    *bytes = ctx->off_p[l][8] + tensor_bytes(ctx->cfg, l, 8, p.esz) - *src_off;
  } else {
    const int r0 = it.index * p.head_rows, rows = std::min(p.head_rows, p.V - r0);
    if (p.esz == 1) {
      *src_off = ctx->off_p[p.L + 1][1] + (size_t)r0 * p.h;
      *bytes = (size_t)rows * p.h;
      if (scale_off && scale_bytes) {
        *scale_off = ctx->off_p[p.L + 1][1] + rup((size_t)p.V * p.h, 16) + (size_t)r0 * 4;
        *scale_bytes = (size_t)rows * 4;
      }
    } else {
      *src_off = ctx->off_p[p.L + 1][1] + (size_t)r0 * p.h * p.esz;
      *bytes = (size_t)rows * p.h * p.esz;
    }
  }
}
// Where an FP8 head slice's row scales sit in its weight buffer.
size_t head_scale_dst(const Plan& p, int rows) { return rup((size_t)rows * p.h, 256); }
int head_slice_rows(const Plan& p, int s) { return std::min(p.head_rows, p.V - s * p.head_rows); }

// Host ranges to touch ahead of the step's copies, in the order the copies
// use them: each weight copy's source, paced two weight copies ahead of it,
// and (when grad_out is given) each gradient copy's destination next to the
// weight copy that precedes the unit producing it. index receives, per
// position of the unit sequence, its weight copy's index (-1: none);
// *n_copies the number of weight copies.
std::vector<PageToucher::Range> touch_plan(const mt_ctx* ctx, const Step& st, const uint8_t* grad_out,
                                           std::vector<int>* index, size_t* n_copies) {
  const Plan& p = ctx->P;
  std::vector<PageToucher::Range> r;
  index->assign(st.seq.size(), -1);
  int copies = 0, last = -1;
  for (size_t i = 0; i < st.seq.size(); ++i) {
    const Item& it = st.seq[i];
    if (st.needs_load[i]) {
      size_t off, bytes, soff = 0, sbytes = 0;
      load_range(ctx, it, &off, &bytes, &soff, &sbytes);
      last = copies++;
      (*index)[i] = last;
      r.push_back({(const uint8_t*)ctx->host_params + off, bytes, last - 2});
      if (sbytes) r.push_back({(const uint8_t*)ctx->host_params + soff, sbytes, last - 2});
    }
    if (!grad_out) continue;
    const bool pass2 = it.kind == IT_HEAD && (int)i >= p.L + p.n_head_slices;
    if (it.kind == IT_LAYER && it.index < 0) {  // a layer's backward: its whole gradient unit
      const int l = -it.index;
      const size_t g0 = ctx->off_g[l][0], g1 = ctx->off_g[l][8] + tensor_numel(ctx->cfg, l, 8) * p.gesz;
      r.push_back({grad_out + g0, g1 - g0, last - 2});
    } else if (pass2) {  // a head slice's weight gradient
      const int r0 = it.index * p.head_rows, rows = std::min(p.head_rows, p.V - r0);
      r.push_back({grad_out + ctx->off_g[p.L + 1][1] + (size_t)r0 * p.h * p.gesz, (size_t)rows * p.h * p.gesz,
                   last - 2});
    }
  }
  *n_copies = (size_t)copies;
  return r;
}

// H2D copy of step i's weights into its slot (weight stream).
int issue_load(Step& st, size_t i) {
  mt_ctx* ctx = st.ctx;
  const int slot = st.slot_of[i];
  const uint8_t* hp = (const uint8_t*)ctx->host_params;
  size_t src_off = 0, bytes = 0, scale_off = 0, scale_bytes = 0;
  load_range(ctx, st.seq[i], &src_off, &bytes, &scale_off, &scale_bytes);
  if (ctx->fault_kind == 1 && ++ctx->fault_count == ctx->fault_nth)
    return set_err(ctx, MT_ERR_CUDA, "injected copy-issue failure");
  CK(cudaStreamWaitEvent(ctx->s_h2d, ctx->ev_wfree[slot], 0));
  if (ctx->serial && i > 0) CK(cudaStreamWaitEvent(ctx->s_h2d, ctx->ev_wfree[st.slot_of[i - 1]], 0));
  {
    SegScope sg(ctx, 1, ctx->s_h2d, (double)(bytes + scale_bytes), (int)i);
    CK(cudaMemcpyAsync(ctx->wbuf[slot], hp + src_off, bytes, cudaMemcpyHostToDevice, ctx->s_h2d));
    if (scale_bytes)
      CK(cudaMemcpyAsync(ctx->wbuf[slot] + head_scale_dst(ctx->P, head_slice_rows(ctx->P, st.seq[i].index)),
                         hp + scale_off, scale_bytes, cudaMemcpyHostToDevice, ctx->s_h2d));
  }
  bytes += scale_bytes;
  CK(cudaEventRecord(ctx->ev_wready[slot], ctx->s_h2d));
  if (st.toucher && st.load_index[i] >= 0) {
    cudaEvent_t done = next_event(ctx);
    if (!done) return set_err(ctx, MT_ERR_CUDA, "event pool");
    CK(cudaEventRecord(done, ctx->s_h2d));
    st.toucher->published((size_t)st.load_index[i], done);
  }
  ctx->stats.h2d_bytes += (double)bytes;
  ctx->stats.n_h2d += 1;
  return MT_OK;
}

// Bind a loaded layer: fp32 params are cast into the slot's bf16 view.
int bind_layer(Step& st, int l, int slot, bool fresh, LayerView* v) {
  mt_ctx* ctx = st.ctx;
  const Plan& p = ctx->P;
  const uint8_t* base = ctx->wbuf[slot];
  const size_t u0 = ctx->off_p[l][0];
  auto at = [&](int t) { return base + (ctx->off_p[l][t] - u0); };
  float* g = ctx->gains[slot];
  v->wr = nullptr;
  if (p.esz == 2) {
    v->wqkv = (const uint16_t*)at(1);
    v->wo = (const uint16_t*)at(4);
    v->wgu = (const uint16_t*)at(6);
    v->wd = (const uint16_t*)at(8);
    v->ldd = p.F;
    if (p.E > 0) {  // router, then all experts' gate|up and down matrices
      v->wr = (const uint16_t*)at(6);
      v->wgu = (const uint16_t*)at(7);
      v->ldd = p.Fe;
    }
    if (fresh) {
      CKL(gains_to_f32(at(0), true, g, p.h, ctx->s_comp));
      CKL(gains_to_f32(at(5), true, g + p.h, p.h, ctx->s_comp));
    }
  } else {
    uint16_t* c = ctx->wcast[slot];
    uint16_t* cqkv = c;
    uint16_t* co = cqkv + rup((size_t)p.qkv * p.h * 2, 256) / 2;
    uint16_t* cgu = co + rup((size_t)p.h * p.qd * 2, 256) / 2;
    uint16_t* cd = cgu + rup((size_t)2 * p.Fp * p.h * 2, 256) / 2;
    if (p.esz == 1 && p.E > 0) {
      // mixture of experts: router, every expert's gate|up rows and down
      // matrices, expert by expert as in the packed layout
      uint16_t* cr = co + rup((size_t)p.h * p.qd * 2, 256) / 2;
      uint16_t* cegu = cr + rup((size_t)p.E * p.h * 2, 256) / 2;
      uint16_t* ced = cegu + rup((size_t)p.E * 2 * p.Fe * p.h * 2, 256) / 2;
      if (fresh) {
        auto deq = [&](int t, size_t rows, int cols, uint16_t* dst) {
          const uint8_t* q = at(t);
          return dequant_fp8_rows(q, (const float*)(q + rup(rows * cols, 16)), (int)rows, cols, dst, cols,
                                  ctx->s_comp);
        };
        CKL(deq(1, p.qd, p.h, cqkv));
        CKL(deq(2, p.kd, p.h, cqkv + (size_t)p.qd * p.h));
        CKL(deq(3, p.kd, p.h, cqkv + (size_t)(p.qd + p.kd) * p.h));
        CKL(deq(4, p.h, p.qd, co));
        CKL(deq(6, p.E, p.h, cr));
        CKL(deq(7, (size_t)p.E * 2 * p.Fe, p.h, cegu));
        CKL(deq(8, (size_t)p.E * p.h, p.Fe, ced));
        CKL(gains_to_f32(at(0), false, g, p.h, ctx->s_comp));
        CKL(gains_to_f32(at(5), false, g + p.h, p.h, ctx->s_comp));
      }
      v->wqkv = cqkv;
      v->wo = co;
      v->wr = cr;
      v->wgu = cegu;
      v->wd = ced;
      v->ldd = p.Fe;
      v->w1 = g;
      v->w2 = g + p.h;
      return MT_OK;
    }
    if (fresh && p.esz == 1) {
      // FP8 codes with row scales -> the bf16 view (Wq, Wk, Wv stacked as one
      // q|k|v matrix; Wg then Wu; Fp == F for FP8)
      auto deq = [&](int t, int rows, int cols, uint16_t* dst, int ld) {
        const uint8_t* q = at(t);
        return dequant_fp8_rows(q, (const float*)(q + rup((size_t)rows * cols, 16)), rows, cols, dst, ld, ctx->s_comp);
      };
      CKL(deq(1, p.qd, p.h, cqkv, p.h));
      CKL(deq(2, p.kd, p.h, cqkv + (size_t)p.qd * p.h, p.h));
      CKL(deq(3, p.kd, p.h, cqkv + (size_t)(p.qd + p.kd) * p.h, p.h));
      CKL(deq(4, p.h, p.qd, co, p.qd));
      CKL(deq(6, p.F, p.h, cgu, p.h));
      CKL(deq(7, p.F, p.h, cgu + (size_t)p.Fp * p.h, p.h));
      CKL(deq(8, p.h, p.F, cd, p.Fp));
      CKL(gains_to_f32(at(0), false, g, p.h, ctx->s_comp));
      CKL(gains_to_f32(at(5), false, g + p.h, p.h, ctx->s_comp));
    } else if (fresh) {
      // Wq, Wk, Wv are contiguous in the packed layout (hidden % 64 == 0)
      CKL(cast_rows_f32_bf16((const float*)at(1), cqkv, p.qkv, p.qkv, p.h, p.h, ctx->s_comp));
      CKL(cast_rows_f32_bf16((const float*)at(4), co, p.h, p.h, p.qd, p.qd, ctx->s_comp));
      CKL(cast_rows_f32_bf16((const float*)at(6), cgu, p.F, p.Fp, p.h, p.h, ctx->s_comp));
      CKL(cast_rows_f32_bf16((const float*)at(7), cgu + (size_t)p.Fp * p.h, p.F, p.Fp, p.h, p.h, ctx->s_comp));
      CKL(cast_rows_f32_bf16((const float*)at(8), cd, p.h, p.h, p.F, p.Fp, ctx->s_comp));
      CKL(gains_to_f32(at(0), false, g, p.h, ctx->s_comp));
      CKL(gains_to_f32(at(5), false, g + p.h, p.h, ctx->s_comp));
    }
    v->wqkv = cqkv;
    v->wo = co;
    v->wgu = cgu;
    v->wd = cd;
    v->ldd = p.Fp;
  }
  v->w1 = g;
  v->w2 = g + p.h;
  return MT_OK;
}

const uint16_t* bind_head(Step& st, int s, int slot, bool fresh, int* rows) {
  mt_ctx* ctx = st.ctx;
  const Plan& p = ctx->P;
  const int r0 = s * p.head_rows;
  *rows = std::min(p.head_rows, p.V - r0);
  if (p.esz == 2) return (const uint16_t*)ctx->wbuf[slot];
  if (fresh && p.esz == 1) {
    const uint8_t* q = ctx->wbuf[slot];
    if (dequant_fp8_rows(q, (const float*)(q + head_scale_dst(p, *rows)), *rows, p.h, ctx->wcast[slot], p.h,
                         ctx->s_comp))
      return nullptr;
  } else if (fresh) {
    if (cast_rows_f32_bf16((const float*)ctx->wbuf[slot], ctx->wcast[slot], *rows, *rows, p.h, p.h, ctx->s_comp))
      return nullptr;
  }
  return ctx->wcast[slot];
}

// x_in / x_out of layer l (1-based) for checkpoint interval K.
float* layer_input(Step& st, int l) {
  const int i = l - 1;  // index of the input residual h_{l-1}
  if (i % st.K == 0) return ckpt(st.ctx, i / st.K);
  return act_slot(st.ctx, st.K, st.nb, i % st.K).x;
}
float* layer_output(Step& st, int l) {
  if (l == st.ctx->P.L) return st.ctx->h_top;
  return layer_input(st, l + 1);
}

// Causal attention forward work: Q K^T and P V over the lower triangle,
// 2 * (2 * B * n_q * d * S(S+1)/2) flop; the backward is 2.5 times that.
double attn_flop(const Step& st, const Plan& p) {
  return 2.0 * st.B * p.nq * (double)p.d * st.S * (st.S + 1.0);
}

// Mixture-of-experts FFN forward of layer l: router logits, top-k routing,
// rows grouped by expert in segments of whole 128-row tiles, one grouped
// gate|up GEMM for all experts (SwiGLU in the epilogue) and one grouped down
// GEMM, then the weighted combine into the residual stream,
// y = h_mid + sum_j w_j y_j. Everything stays on the device: the tile
// schedule of the grouped GEMMs is read from the segment table.
int moe_ffn_forward(Step& st, int l, const LayerView& w, const ActSlot& a, float* y) {
  mt_ctx* ctx = st.ctx;
  const Plan& p = ctx->P;
  const int T = st.T, h = p.h, E = p.E, k = p.topk, Fe = p.Fe, n = T * k;
  cudaStream_t s = ctx->s_comp;
  CKR(gemm(ctx, GEMM_NT, EPI_F32, a.m, w.wr, a.r, nullptr, T, E, h, h, h, E));
  CKL(moe_route(a.r, T, E, k, a.sel, a.w, ctx->moe_counts, ctx->moe_route + (size_t)(l - 1) * T * k, s));
  CKL(moe_segments(ctx->moe_counts, E, p.n_pad / 128, a.seg, a.tile_e, s));
  CKL(moe_permute(a.sel, n, E, a.seg, a.spos, s));
  CK(cudaMemsetAsync(a.xp, 0, (size_t)p.n_pad * h * 2, s));  // padding rows are zero
  CKL(moe_gather(a.m, a.spos, n, k, h, a.xp, s));
  {
    GemmParams gp{p.n_pad, Fe, h, EPI_BF16, a.gup, nullptr, 2 * Fe, 0, 1};
    gp.gated = 1;
    gp.u_off = Fe;
    gp.u_col = Fe;
    gp.act = a.actp;
    gp.ld_act = Fe;
    gp.grp_seg = a.seg;
    gp.grp_tile_e = a.tile_e;
    gp.grp_E = E;
    gp.grp_b_rows = 2 * Fe;
    CKR(gemm_p(ctx, GEMM_NT, gp, a.xp, w.wgu, h, h, 2.0 * n * 2 * Fe * h));
  }
  {
    GemmParams gp{p.n_pad, h, Fe, EPI_F32, a.yp, nullptr, h, 0, 1};
    gp.grp_seg = a.seg;
    gp.grp_tile_e = a.tile_e;
    gp.grp_E = E;
    gp.grp_b_rows = h;
    CKR(gemm_p(ctx, GEMM_NT, gp, a.actp, w.wd, Fe, Fe, 2.0 * n * h * Fe));
  }
  CKL(moe_combine(a.hmid, a.yp, a.spos, a.w, T, k, h, y, s));
  return MT_OK;
}

int layer_forward(Step& st, int l, const LayerView& w) {
  mt_ctx* ctx = st.ctx;
  const Plan& p = ctx->P;
  const int T = st.T, h = p.h;
  ActSlot a = act_slot(ctx, st.K, st.nb, (l - 1) % st.K);
  float* x = layer_input(st, l);
  float* y = layer_output(st, l);
  cudaStream_t s = ctx->s_comp;
  CKL(rmsnorm_fwd(x, w.w1, a.a, a.rstd1, T, h, ctx->cfg.norm_eps, s));
  // q|k|v projection with RoPE applied to the q and k heads in the epilogue
  CKR(gemm(ctx, GEMM_NT, EPI_BF16, a.a, w.wqkv, a.qkv, nullptr, T, p.qkv, h, h, h, p.qkv, st.S, p.qd + p.kd));
  {
    OpTimer timer(ctx, 1, attn_flop(st, p));
    CKL(attention_fwd_tc(a.qkv, a.qkv + p.qd, a.qkv + p.qd + p.kd, a.o, a.lse, st.B, st.S, p.nq, p.nkv, p.d, p.qkv,
                      p.qkv, p.qd, s));
  }
  CKR(gemm(ctx, GEMM_NT, EPI_F32_ADD, a.o, w.wo, a.hmid, x, T, h, p.qd, p.qd, p.qd, h));
  CKL(rmsnorm_fwd(a.hmid, w.w2, a.m, a.rstd2, T, h, ctx->cfg.norm_eps, s));
  if (p.E > 0) return moe_ffn_forward(st, l, w, a, y);
  {  // gate-up projection with SwiGLU fused: g, u (kept for the backward) and act = silu(g) u
    GemmParams gp{T, p.Fp, h, EPI_BF16, a.gu, nullptr, 2 * p.Fp, 0, 1};
    gp.gated = 1;
    gp.u_off = p.Fp;
    gp.u_col = p.Fp;
    gp.act = a.act;
    gp.ld_act = p.Fp;
    CKR(gemm_p(ctx, GEMM_NT, gp, a.m, w.wgu, h, h, 2.0 * T * 2 * p.Fp * h));
  }
  CKR(gemm(ctx, GEMM_NT, EPI_F32_ADD, a.act, w.wd, y, a.hmid, T, h, p.Fp, p.Fp, w.ldd, h));
  return MT_OK;
}

// Gradient staging slot handshake.
int grad_slot_begin(Step& st, int* g) {
  mt_ctx* ctx = st.ctx;
  *g = ctx->gslot;
  ctx->gslot ^= 1;
  CK(cudaStreamWaitEvent(ctx->s_comp, ctx->ev_gfree[*g], 0));
  return MT_OK;
}
int grad_slot_end(Step& st, int g, size_t host_off, size_t bytes) {
  mt_ctx* ctx = st.ctx;
  CK(cudaEventRecord(ctx->ev_bwd_done[g], ctx->s_comp));
  CK(cudaStreamWaitEvent(ctx->s_d2h, ctx->ev_bwd_done[g], 0));
  {
    SegScope sg(ctx, 2, ctx->s_d2h, (double)bytes, ctx->cur_unit);
    CK(cudaMemcpyAsync((uint8_t*)st.host_grad + host_off, ctx->gbuf[g], bytes, cudaMemcpyDeviceToHost, ctx->s_d2h));
  }
  CK(cudaEventRecord(ctx->ev_gfree[g], ctx->s_d2h));
  if (ctx->serial) CK(cudaStreamWaitEvent(ctx->s_comp, ctx->ev_gfree[g], 0));
  ctx->stats.d2h_bytes += (double)bytes;
  ctx->stats.n_d2h += 1;
  return MT_OK;
}

// Copy one finished range of a layer's gradients (packed offsets [off0,
// off1) of the unit starting at u0) from gradient buffer g to the host, as
// soon as the compute stream has produced it.
// Tensors t0..t1 of unit l, copied tensor by tensor (the padding between
// them in the device buffer holds no gradient and is not copied).
int grad_piece(Step& st, int g, int l, int t0, int t1) {
  mt_ctx* ctx = st.ctx;
  const size_t u0 = ctx->off_g[l][0];
  cudaEvent_t ready = next_event(ctx);
  if (!ready) return set_err(ctx, MT_ERR_CUDA, "event pool");
  CK(cudaEventRecord(ready, ctx->s_comp));
  CK(cudaStreamWaitEvent(ctx->s_d2h, ready, 0));
  const size_t gesz = ctx->P.gesz;
  const size_t span = ctx->off_g[l][t1] + tensor_numel(ctx->cfg, l, t1) * gesz - ctx->off_g[l][t0];
  SegScope sg(ctx, 2, ctx->s_d2h, (double)span, ctx->cur_unit);
  for (int t = t0; t <= t1; ++t) {
    const size_t off = ctx->off_g[l][t], nb = tensor_numel(ctx->cfg, l, t) * gesz;
    CK(cudaMemcpyAsync((uint8_t*)st.host_grad + off, (const uint8_t*)ctx->gbuf[g] + (off - u0), nb,
                       cudaMemcpyDeviceToHost, ctx->s_d2h));
    ctx->stats.d2h_bytes += (double)nb;
  }
  ctx->stats.n_d2h += 1;
  return MT_OK;
}
// After the last piece of gradient buffer g: it is free once the copies drain.
int grad_slot_release(Step& st, int g) {
  mt_ctx* ctx = st.ctx;
  CK(cudaEventRecord(ctx->ev_gfree[g], ctx->s_d2h));
  if (ctx->serial) CK(cudaStreamWaitEvent(ctx->s_comp, ctx->ev_gfree[g], 0));
  return MT_OK;
}

// Mixture-of-experts FFN backward of layer l, from dh (the gradient of the
// layer output) to ctx->dm (the gradient of the FFN input m); writes the
// experts' and the router's gradients and sends them to the host. The four
// expert products are grouped launches over the segment table of the
// forward (or recompute) that filled this activation slot.
int moe_ffn_backward(Step& st, int l, const LayerView& w, const ActSlot& a, int g, float* g_router,
                     float* g_gu, float* g_down) {
  mt_ctx* ctx = st.ctx;
  const Plan& p = ctx->P;
  const int T = st.T, h = p.h, E = p.E, k = p.topk, Fe = p.Fe, n = T * k;
  cudaStream_t s = ctx->s_comp;
  CK(cudaMemsetAsync(ctx->moe_dyp, 0, (size_t)p.n_pad * h * 2, s));  // padding rows are zero
  CKL(moe_combine_bwd(ctx->dh, a.yp, a.spos, a.w, T, k, h, ctx->moe_dyp, ctx->moe_dw, s));
  float* dxp = a.yp;  // the routed outputs are consumed: their rows take d(routed inputs)
  auto grouped = [&](GemmParams& gp, bool tn, int b_rows) {
    gp.grp_seg = a.seg;
    gp.grp_tile_e = tn ? nullptr : a.tile_e;
    gp.grp_E = E;
    gp.grp_b_rows = b_rows;
  };
  {  // y_e = act Wd_e^T: dWd_e = dY_e^T act_e (each expert's [h, Fe])
    GemmParams gp{h, Fe, p.n_pad, p.gepi, g_down, nullptr, Fe, 0, 1};
    grouped(gp, true, 0);
    CKR(gemm_p(ctx, GEMM_TN, gp, ctx->moe_dyp, a.actp, h, Fe, 2.0 * n * h * Fe));
  }
  {  // dact = dY Wd_e, turned into (dg, du) in place over (g, u) by the epilogue
    GemmParams bp{p.n_pad, Fe, h, EPI_BF16, a.gup, nullptr, 2 * Fe, 0, 1};
    bp.swiglu_bwd = 1;
    bp.gu = a.gup;
    bp.ld_gu = 2 * Fe;
    bp.u_col = Fe;
    grouped(bp, false, h);
    CKR(gemm_p(ctx, GEMM_NN, bp, ctx->moe_dyp, w.wd, h, Fe, 2.0 * n * Fe * h));
  }
  {  // g|u = x Wgu_e^T: dWgu_e = d(g|u)_e^T x_e (each expert's [2Fe, h])
    GemmParams gp{2 * Fe, h, p.n_pad, p.gepi, g_gu, nullptr, h, 0, 1};
    grouped(gp, true, 0);
    CKR(gemm_p(ctx, GEMM_TN, gp, a.gup, a.xp, 2 * Fe, h, 2.0 * n * 2 * Fe * h));
  }
  {  // dx = d(g|u) Wgu_e
    GemmParams gp{p.n_pad, h, 2 * Fe, EPI_F32, dxp, nullptr, h, 0, 1};
    grouped(gp, false, 2 * Fe);
    CKR(gemm_p(ctx, GEMM_NN, gp, a.gup, w.wgu, 2 * Fe, h, 2.0 * n * 2 * Fe * h));
  }
  CKR(grad_piece(st, g, l, 7, 8));
  CKL(moe_unpermute(dxp, a.spos, T, k, h, ctx->dm, s));
  // router: dr, then dm += dr Wr and dWr = dr^T m
  CKL(moe_router_bwd(a.w, ctx->moe_dw, a.sel, T, k, E, ctx->moe_dr, s));
  CKR(gemm(ctx, GEMM_NN, EPI_F32_ADD, ctx->moe_dr, w.wr, ctx->dm, ctx->dm, T, h, E, E, h, h));
  CKR(gemm(ctx, GEMM_TN, p.gepi, ctx->moe_dr, a.m, g_router, nullptr, E, h, T, E, h, h));
  return grad_piece(st, g, l, 6, 6);
}

int layer_backward(Step& st, int l, const LayerView& w) {
  mt_ctx* ctx = st.ctx;
  const Plan& p = ctx->P;
  const int T = st.T, h = p.h, Fp = p.Fp, F = p.F;
  ActSlot a = act_slot(ctx, st.K, st.nb, (l - 1) % st.K);
  float* x = layer_input(st, l);
  cudaStream_t s = ctx->s_comp;
  int g;
  CKR(grad_slot_begin(st, &g));
  float* G = ctx->gbuf[g];
  const size_t u0 = ctx->off_g[l][0];
  auto GT = [&](int t) { return (float*)((uint8_t*)G + (ctx->off_g[l][t] - u0)); };
  // RMSNorm gain gradients come out in fp32; with bf16 gradients they are
  // rounded into the staging buffer afterwards.
  auto GGAIN = [&](int t) { return p.gesz == 2 ? ctx->gain_grad : GT(t); };
  auto gain_grad_out = [&](int t) -> int {
    if (p.gesz == 2) CKL(cast_f32_bf16(ctx->gain_grad, (uint16_t*)GT(t), (size_t)h, s));
    return MT_OK;
  };
  // Gradient tensors go to the host in four groups, each as soon as it is
  // complete: [Wd], [Wg Wu], [Wo w_ffn], [w_attn Wq Wk Wv] (mixture of
  // experts: [experts' Wgu Wd], [router], then the same two).
  if (p.E > 0) {
    CKR(moe_ffn_backward(st, l, w, a, g, GT(6), GT(7), GT(8)));
  } else {
    // h_out = h_mid + act Wd^T
    CKR(gemm(ctx, GEMM_TN, p.gepi, ctx->dh_b, a.act, GT(8), nullptr, h, F, T, h, Fp, F));
    CKR(grad_piece(st, g, l, 8, 8));
    {  // dact = dh Wd, turned into (dg, du) in place over (g, u) by the epilogue
      GemmParams bp{T, Fp, h, EPI_BF16, a.gu, nullptr, 2 * Fp, 0, 1};
      bp.swiglu_bwd = 1;
      bp.gu = a.gu;
      bp.ld_gu = 2 * Fp;
      bp.u_col = Fp;
      CKR(gemm_p(ctx, GEMM_NN, bp, ctx->dh_b, w.wd, h, w.ldd, 2.0 * T * Fp * h));
    }
    if (Fp == F) {
      CKR(gemm(ctx, GEMM_TN, p.gepi, a.gu, a.m, GT(6), nullptr, 2 * F, h, T, 2 * Fp, h, h));
    } else {
      CKR(gemm(ctx, GEMM_TN, p.gepi, a.gu, a.m, GT(6), nullptr, F, h, T, 2 * Fp, h, h));
      CKR(gemm(ctx, GEMM_TN, p.gepi, a.gu + Fp, a.m, GT(7), nullptr, F, h, T, 2 * Fp, h, h));
    }
    CKR(grad_piece(st, g, l, 6, 7));
    CKR(gemm(ctx, GEMM_NN, EPI_F32, a.gu, w.wgu, ctx->dm, nullptr, T, h, 2 * Fp, 2 * Fp, h, h));
  }
  // RMSNorm 2 (+ residual): dh_mid written over h_mid (row-local, in place)
  CKL(rmsnorm_bwd(a.hmid, w.w2, a.rstd2, ctx->dm, ctx->dh, a.hmid, ctx->dhmid_b, GGAIN(5), ctx->norm_ws, T, h, s));
  CKR(gain_grad_out(5));
  // h_mid = x + o Wo^T
  CKR(gemm(ctx, GEMM_TN, p.gepi, ctx->dhmid_b, a.o, GT(4), nullptr, h, p.qd, T, h, p.qd, p.qd));
  CKR(grad_piece(st, g, l, 4, 5));
  CKR(gemm(ctx, GEMM_NN, EPI_BF16, ctx->dhmid_b, w.wo, ctx->do_b, nullptr, T, p.qd, h, h, p.qd, p.qd));
  {
    OpTimer timer(ctx, 1, 2.5 * attn_flop(st, p));
    // dq and dk come out rotated back by RoPE (the forward rotated q and k)
    CKL(attention_bwd_tc(a.qkv, a.qkv + p.qd, a.qkv + p.qd + p.kd, a.o, ctx->do_b, a.lse, ctx->dqkv,
                      ctx->dqkv + p.qd, ctx->dqkv + p.qd + p.kd, ctx->attn_ws, st.B, st.S, p.nq, p.nkv, p.d, p.qkv,
                      p.qkv, p.qd, s, ctx->rope_tab));
  }
  CKR(gemm(ctx, GEMM_TN, p.gepi, ctx->dqkv, a.a, GT(1), nullptr, p.qkv, h, T, p.qkv, h, h));
  CKR(gemm(ctx, GEMM_NN, EPI_F32, ctx->dqkv, w.wqkv, ctx->dm, nullptr, T, h, p.qkv, p.qkv, h, h));
  // RMSNorm 1 (+ residual): new dh
  CKL(rmsnorm_bwd(x, w.w1, a.rstd1, ctx->dm, a.hmid, ctx->dh, ctx->dh_b, GGAIN(0), ctx->norm_ws, T, h, s));
  CKR(gain_grad_out(0));
  CKR(grad_piece(st, g, l, 0, 3));
  if (st.train || st.async) {
    st.landed[l] = next_event(ctx);
    if (!st.landed[l]) return set_err(ctx, MT_ERR_CUDA, "event pool");
    CK(cudaEventRecord(st.landed[l], ctx->s_d2h));
  }
  return grad_slot_release(st, g);
}

// Debug aid: wait (bounded) for the compute stream after a unit and report
// which stream is still busy if it does not finish.
int debug_wait(mt_ctx* ctx, size_t i, Item it, int slot, int loaded) {
  const auto t0 = std::chrono::steady_clock::now();
  while (true) {
    cudaError_t e = cudaStreamQuery(ctx->s_comp);
    const double el = std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
    if (e == cudaSuccess) {
      fprintf(stderr, "[mt] unit %zu kind %d index %d slot %d loaded %d: compute idle after %.3f s\n", i, it.kind,
              it.index, slot, loaded, el);
      return MT_OK;
    }
    if (e != cudaErrorNotReady) return set_err(ctx, MT_ERR_CUDA, cudaGetErrorString(e));
    if (el > 60.0) {
      fprintf(stderr, "[mt] unit %zu kind %d index %d STUCK: compute %s, weight-in %s, grad-out %s\n", i, it.kind,
              it.index, cudaStreamQuery(ctx->s_comp) == cudaSuccess ? "idle" : "busy",
              cudaStreamQuery(ctx->s_h2d) == cudaSuccess ? "idle" : "busy",
              cudaStreamQuery(ctx->s_d2h) == cudaSuccess ? "idle" : "busy");
      return set_err(ctx, MT_ERR_TIMEOUT, "debug: unit did not finish");
    }
    std::this_thread::sleep_for(std::chrono::microseconds(200));
  }
}

int run_step(Step& st, const int32_t* tokens, const int32_t* labels, float* loss_out) {
  mt_ctx* ctx = st.ctx;
  const Plan& p = ctx->P;
  const int T = st.T, h = p.h, L = p.L;
  cudaStream_t s = ctx->s_comp;

  // The embedding gradient region of the host buffer is cleared by CPU
  // threads while the GPU works; the rows of used tokens are written into it
  // after the step has drained.
  // (Started right after the embedding rows are gathered, so that the two
  // do not compete for the host cores while the first layer waits.)
  std::vector<std::thread> zeroers;
  // The bytes between tensors (and after each unit) of the gradient buffer
  // hold no gradient: written as zeros, so the whole buffer is defined.
  {
    uint8_t* gb = (uint8_t*)st.host_grad;
    size_t pos = 0;
    for (int u = 0; u <= L + 1; ++u)
      for (int t = 0; t < tensors_in_unit(ctx->cfg, u); ++t) {
        const size_t off = ctx->off_g[u][t];
        if (off > pos) std::memset(gb + pos, 0, off - pos);
        pos = off + tensor_numel(ctx->cfg, u, t) * p.gesz;
      }
    const size_t total = build_layout(ctx->cfg, p.gesz, nullptr);
    if (total > pos) std::memset(gb + pos, 0, total - pos);
  }
  auto start_zeroers = [&] {
    uint8_t* eg = (uint8_t*)st.host_grad + ctx->off_g[0][0];
    const size_t nbytes = (size_t)p.V * h * p.gesz;
    const unsigned hw = std::max(1u, std::thread::hardware_concurrency());
    const size_t nthr = std::min<size_t>(std::max(1u, hw / 2), std::max<size_t>(1, nbytes >> 26));
    const size_t chunk = (nbytes / nthr + 4095) & ~(size_t)4095;
    for (size_t i = 0; i < nthr; ++i) {
      const size_t b = i * chunk;
      if (b >= nbytes) break;
      const size_t n = std::min(chunk, nbytes - b);
      zeroers.emplace_back([eg, b, n] { std::memset(eg + b, 0, n); });
    }
  };
  struct Joiner {
    std::vector<std::thread>& t;
    ~Joiner() {
      for (auto& x : t)
        if (x.joinable()) x.join();
    }
  } joiner{zeroers};

  // Asynchronous optimizer: the previous call's gradients are complete, so
  // host threads compute that update (fp32 master and moments only) while
  // this step runs; each unit's streamed copy is rewritten (published) only
  // once this step has read that unit for the last time (see below).
  struct AsyncRun {
    std::vector<std::atomic<int>> done;
    std::atomic<bool> abort{false};
    double busy_ms = 0;
    std::thread th;
    explicit AsyncRun(int n) : done(n) {
      for (auto& d : done) d = 0;
    }
    ~AsyncRun() {
      abort = true;
      if (th.joinable()) th.join();
    }
  } arun(L + 2);
  const bool have_pending = st.async && ctx->opt_pending;
  if (have_pending) {
    arun.th = std::thread([ctx, &arun, &p, L] {
      const AdamCoef coef = adam_coef(ctx->opt, ctx->opt_step);
      const int nthr = ctx->opt_threads > 0 ? ctx->opt_threads
                                            : (int)std::max(1u, std::thread::hardware_concurrency());
      const auto t0 = std::chrono::steady_clock::now();
      for (int u = L + 1; u >= 0; --u) {  // the order in which this step's units become publishable
        if (arun.abort) return;
        if (ctx->opt_state[u] == 0) {  // not yet computed (by an earlier call that failed part-way)
          adamw_units(ctx->cfg, ctx->off_g, ctx->off_p, p.esz, coef, u, u + 1, ctx->opt_master, ctx->opt_m,
                      ctx->opt_v, ctx->opt_pending, nullptr, nthr);
          ctx->opt_state[u] = 1;
        }
        arun.done[u] = 1;
      }
      arun.busy_ms = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
    });
  }

  // Host preparation: stable counting sort of token ids (positions grouped
  // by id in ascending position order) and the list of distinct ids with
  // their ranges, for the deterministic embedding gradient.
  int32_t* hs = ctx->host_stage;
  std::memcpy(hs, tokens, (size_t)T * 4);
  std::memcpy(hs + T, labels, (size_t)T * 4);
  int32_t* perm = hs + 2 * T;
  int32_t* ids = hs + 3 * T;
  int32_t* ranges = hs + 4 * T;
  std::vector<int32_t>& start = ctx->csr;
  start.assign((size_t)p.V + 1, 0);
  for (int t = 0; t < T; ++t) start[tokens[t] + 1]++;
  for (int v = 0; v < p.V; ++v) start[v + 1] += start[v];
  int n_ids = 0;
  for (int v = 0; v < p.V; ++v)
    if (start[v + 1] > start[v]) {
      ids[n_ids] = v;
      ranges[n_ids] = start[v];
      ++n_ids;
    }
  ranges[n_ids] = T;
  {
    std::vector<int32_t> fill(start.begin(), start.end() - 1);
    for (int t = 0; t < T; ++t) perm[fill[tokens[t]]++] = t;
  }
  ctx->segs.clear();
  ctx->opsegs.clear();
  ctx->ev_used = 0;
  ctx->stats = mt_stats{};
  ctx->stats.timing_enabled = ctx->trace;
  ctx->launches_at_start = g_kernel_launches;
  ctx->gslot = 0;
  ctx->fault_count = 0;
  // Fresh step: the previous step fully drained, so every buffer is free.
  if (ctx->trace) CK(cudaEventRecord(ctx->ev_base, s));
  cudaGetLastError();
  CK(cudaMemcpyAsync(ctx->tok_d, hs, (size_t)(5 * T + 1) * 4, cudaMemcpyHostToDevice, s));
  // The copy streams wait for the step start so that their timestamps are
  // ordered after the base event and no buffer of the previous step is live.
  cudaEvent_t ev_start = next_event(ctx);
  CK(cudaEventRecord(ev_start, s));
  CK(cudaStreamWaitEvent(ctx->s_h2d, ev_start, 0));
  CK(cudaStreamWaitEvent(ctx->s_d2h, ev_start, 0));
  if (ctx->rope_S != st.S) {
    CKL(rope_table(ctx->rope_tab, st.S, p.d, ctx->cfg.rope_theta, s));
    ctx->rope_S = st.S;
  }
  // Final-norm gain: tiny copy on the weight stream.
  {
    const size_t wf_bytes = (size_t)h * (p.esz == 2 ? 2 : 4);  // FP8 layouts keep the gains fp32
    CK(cudaMemcpyAsync(ctx->wf_raw, (const uint8_t*)ctx->host_params + ctx->off_p[L + 1][0], wf_bytes,
                       cudaMemcpyHostToDevice, ctx->s_h2d));
    cudaEvent_t e = next_event(ctx);
    CK(cudaEventRecord(e, ctx->s_h2d));
    CK(cudaStreamWaitEvent(s, e, 0));
    CKL(gains_to_f32(ctx->wf_raw, p.esz == 2, ctx->wf32, h, s));
  }

  plan_sequence(st);
  const size_t n = st.seq.size();
  ctx->stats.n_units = (int)n;
  ctx->unit_phase.assign(n + 1, 3);  // position n: the embedding gradient (backward)
  for (size_t i = 0; i < n; ++i) {
    const Item& it = st.seq[i];
    ctx->unit_phase[i] = it.kind == IT_HEAD ? 1 : it.index < 0 ? 3 : (int)i < L ? 0 : 2;
  }
  ctx->cur_unit = -1;
  // Host pages of the weight copies are touched two copies ahead of the
  // copy stream; the first copy waits (bounded) for its own pages.
  PageToucher toucher;
  if (ctx->touch_threads > 0) {
    size_t n_copies = 0;
    std::vector<PageToucher::Range> plan = touch_plan(ctx, st, (const uint8_t*)st.host_grad, &st.load_index, &n_copies);
    // the embedding gradient rows land in the context's own pinned staging
    plan.push_back({(const uint8_t*)ctx->host_grad_rows, (size_t)n_ids * h * 4, (int)n_copies - 2});
    toucher.start(std::move(plan), n_copies, ctx->touch_threads, ctx->device);
    st.toucher = &toucher;
    toucher.wait_touched(0, 2.0);
  }
  if (st.needs_load[0]) CKR(issue_load(st, 0));

  // Embedding: h_0 = E[tok]. CPU threads gather the T rows from the host
  // table into a contiguous pinned buffer (the first layer's weights are
  // already streaming), then one copy brings them to the device.
  {
    // staged rows: fp32 for fp32 params, bf16 otherwise (FP8 rows are
    // dequantised by the gathering threads: bf16(code * row scale))
    const size_t row_bytes = (size_t)h * (p.esz == 4 ? 4 : 2);
    const uint8_t* E = (const uint8_t*)ctx->host_params + ctx->off_p[0][0];
    const float* E_scale = (const float*)(E + rup((size_t)p.V * h, 16));
    const bool fp8 = p.esz == 1;
    uint8_t* dst = ctx->host_rows;
    const int nthr = (int)std::min<unsigned>(16, std::max(1u, std::thread::hardware_concurrency()));
    std::vector<std::thread> gth;
    const int per = (T + nthr - 1) / nthr;
    for (int i = 0; i < nthr; ++i) {
      const int t0 = i * per, t1 = std::min(T, t0 + per);
      if (t0 >= t1) break;
      gth.emplace_back([=] {
        for (int t = t0; t < t1; ++t) {
          if (fp8) {
            const uint8_t* src = E + (size_t)tokens[t] * h;
            const float sc = E_scale[tokens[t]];
            uint16_t* out = (uint16_t*)(dst + (size_t)t * row_bytes);
            for (int c = 0; c < h; ++c) out[c] = e4m3_dequant_bf16(src[c], sc);
          } else {
            std::memcpy(dst + (size_t)t * row_bytes, E + (size_t)tokens[t] * row_bytes, row_bytes);
          }
        }
      });
    }
    for (auto& x : gth) x.join();
    start_zeroers();
    // On the weight stream, queued right behind the first layer's copy (the
    // copy engine serves one H2D stream at a time, so issuing it from the
    // compute stream would put it behind the second layer's copy too).
    void* land = p.esz == 4 ? (void*)ckpt(ctx, 0) : (void*)ctx->xf_b;
    cudaEvent_t rows_in = next_event(ctx);
    {
      SegScope sg(ctx, 1, ctx->s_h2d, (double)T * row_bytes, -1);
      CK(cudaMemcpyAsync(land, dst, (size_t)T * row_bytes, cudaMemcpyHostToDevice, ctx->s_h2d));
    }
    CK(cudaEventRecord(rows_in, ctx->s_h2d));
    CK(cudaStreamWaitEvent(s, rows_in, 0));
    if (p.esz != 4) {
      SegScope sg(ctx, 0, s, 0, -1);
      CKL(cast_bf16_f32(ctx->xf_b, ckpt(ctx, 0), (size_t)T * h, s));
    }
  }
  ctx->stats.h2d_bytes += (double)T * h * (p.esz == 4 ? 4 : 2);
  int head_pass2_count = 0;
  bool first_dxf = true;
  for (size_t i = 0; i < n; ++i) {
    // Ping-pong: the copy of the next unit is issued before this unit's
    // compute (it overlaps it); in the serial ablation it waits for it.
    if (!ctx->serial && i + 1 < n && st.needs_load[i + 1]) CKR(issue_load(st, i + 1));
    const Item it = st.seq[i];
    const int slot = st.slot_of[i];
    const bool fresh = st.needs_load[i];
    ctx->cur_unit = (int)i;
    if (fresh) CK(cudaStreamWaitEvent(s, ctx->ev_wready[slot], 0));
    char label[48] = "";
    if (ctx->nvtx) {
      if (it.kind == IT_LAYER)
        snprintf(label, sizeof label, "layer %d %s", std::abs(it.index), it.index > 0 ? "forward" : "backward");
      else
        snprintf(label, sizeof label, "head slice %d pass %d", it.index, (int)i >= L + p.n_head_slices ? 2 : 1);
    }
    NvtxRange nr(ctx->nvtx, label);
    {
      SegScope sg(ctx, 0, s, 0, (int)i);
      if (it.kind == IT_LAYER) {
        const int l = std::abs(it.index);
        LayerView w;
        CKR(bind_layer(st, l, slot, fresh, &w));
        if (it.index > 0) {
          CKR(layer_forward(st, l, w));
        } else {
          CKR(layer_backward(st, l, w));
        }
      } else {  // head slice
        int rows;
        const uint16_t* W = bind_head(st, it.index, slot, fresh, &rows);
        if (!W) return set_err(ctx, MT_ERR_CUDA, "head cast failed");
        const int r0 = it.index * p.head_rows;
        const bool pass2 = (int)i >= L + p.n_head_slices;
        if (!pass2) {
          if (it.index == 0) CKL(rmsnorm_fwd(ctx->h_top, ctx->wf32, ctx->xf_b, ctx->rstd_f, T, h, ctx->cfg.norm_eps, s));
          CKR(gemm(ctx, GEMM_NT, EPI_F32, ctx->xf_b, W, ctx->logits, nullptr, T, rows, h, h, h, p.head_rows));
          CKL(ce_slice_stats(ctx->logits, T, rows, p.head_rows, r0, ctx->lab_d, ctx->ce_part + (size_t)it.index * T,
                             ctx->zlab, s));
          if (it.index == p.n_head_slices - 1)
            CKL(ce_finalize(ctx->ce_part, p.n_head_slices, ctx->zlab, ctx->lse, ctx->terms, ctx->loss_dev, T,
                            1.f / (float)T, s));
        } else {
          CKR(gemm(ctx, GEMM_NT, EPI_F32, ctx->xf_b, W, ctx->logits, nullptr, T, rows, h, h, h, p.head_rows));
          CKL(ce_slice_grad(ctx->logits, T, rows, p.head_rows, r0, ctx->lab_d, ctx->lse, 1.f / (float)T, ctx->dz, s));
          CKR(gemm(ctx, GEMM_NN, first_dxf ? EPI_F32 : EPI_F32_ADD, ctx->dz, W, ctx->dm, ctx->dm, T, h, rows,
                   p.head_rows, h, h));
          first_dxf = false;
          int g;
          CKR(grad_slot_begin(st, &g));
          CKR(gemm(ctx, GEMM_TN, p.gepi, ctx->dz, ctx->xf_b, ctx->gbuf[g], nullptr, rows, h, T, p.head_rows, h, h));
          CKR(grad_slot_end(st, g, ctx->off_g[L + 1][1] + (size_t)r0 * h * p.gesz, (size_t)rows * h * p.gesz));
          if (++head_pass2_count == p.n_head_slices) {
            // final norm backward -> dh_L, and its gain gradient
            CKR(grad_slot_begin(st, &g));
            CKL(rmsnorm_bwd(ctx->h_top, ctx->wf32, ctx->rstd_f, ctx->dm, nullptr, ctx->dh, ctx->dh_b,
                            p.gesz == 2 ? ctx->gain_grad : ctx->gbuf[g], ctx->norm_ws, T, h, s));
            if (p.gesz == 2) CKL(cast_f32_bf16(ctx->gain_grad, (uint16_t*)ctx->gbuf[g], (size_t)h, s));
            CKR(grad_slot_end(st, g, ctx->off_g[L + 1][0], (size_t)h * p.gesz));
            if (st.train || st.async) {
              st.landed[L + 1] = next_event(ctx);
              if (!st.landed[L + 1]) return set_err(ctx, MT_ERR_CUDA, "event pool");
              CK(cudaEventRecord(st.landed[L + 1], ctx->s_d2h));
            }
          }
        }
      }
    }
    CK(cudaEventRecord(ctx->ev_wfree[slot], s));
    if (ctx->serial && i + 1 < n && st.needs_load[i + 1]) CKR(issue_load(st, i + 1));
    if (ctx->debug_sync) CKR(debug_wait(ctx, i, it, slot, st.needs_load[i]));
  }
  // Train steps: host threads apply AdamW to each unit as soon as its
  // gradients have landed (head first, then the layers top-down, the
  // embedding after its scatter below). Every landed event is recorded by
  // now, so they can be waited on from another thread.
  struct OptRun {
    std::atomic<int> emb_ready{0};
    std::atomic<bool> abort{false};
    std::atomic<int> status{MT_OK};
    double busy_ms = 0;
    std::thread th;
    ~OptRun() {
      abort = true;
      if (th.joinable()) th.join();
    }
  } opt;
  if (have_pending) {  // publisher: unit u once this step's gradients of u have landed and its update is computed
    opt.th = std::thread([ctx, &st, &opt, &arun, &p, L] {
      const int nthr = ctx->opt_threads > 0 ? ctx->opt_threads
                                            : (int)std::max(1u, std::thread::hardware_concurrency());
      const auto deadline = std::chrono::steady_clock::now() + std::chrono::seconds(3600);
      auto wait_until = [&](auto ready) {
        while (!ready()) {
          if (opt.abort || std::chrono::steady_clock::now() > deadline) return false;
          std::this_thread::sleep_for(std::chrono::microseconds(100));
        }
        return true;
      };
      for (int u = L + 1; u >= 0; --u) {
        if (ctx->opt_state[u] == 2) continue;  // published by an earlier call that failed part-way
        bool ok = true;
        if (u >= 1) {
          ok = wait_until([&] {
            const cudaError_t e = cudaEventQuery(st.landed[u]);
            if (e != cudaSuccess && e != cudaErrorNotReady) opt.status = MT_ERR_CUDA;
            return e != cudaErrorNotReady;
          });
          if (opt.status != MT_OK) return;
        }
        // the embedding (u = 0) was gathered at the start of the step
        if (!ok || !wait_until([&] { return arun.done[u].load() == 1; })) {
          opt.status = MT_ERR_TIMEOUT;
          return;
        }
        if (gemm_peek_device_error() | attention_tc_peek_device_error()) {
          opt.status = MT_ERR_DEVICE;
          return;
        }
        publish_units(ctx->cfg, ctx->off_g, ctx->off_p, p.esz, u, u + 1, ctx->opt_master,
                      const_cast<void*>(ctx->host_params), nthr);
        ctx->opt_state[u] = 2;
      }
    });
  }
  if (st.train) {
    opt.th = std::thread([ctx, &st, &opt, &p, L] {
      const AdamCoef coef = adam_coef(ctx->opt, ctx->opt_step);
      const int nthr = ctx->opt_threads > 0 ? ctx->opt_threads
                                            : (int)std::max(1u, std::thread::hardware_concurrency());
      auto update = [&](int u) {
        if (gemm_peek_device_error() | attention_tc_peek_device_error()) {  // garbage gradients: apply nothing
          opt.status = MT_ERR_DEVICE;
          return false;
        }
        const auto t0 = std::chrono::steady_clock::now();
        adamw_units(ctx->cfg, ctx->off_g, ctx->off_p, p.esz, coef, u, u + 1, ctx->opt_master, ctx->opt_m,
                    ctx->opt_v, st.host_grad, const_cast<void*>(ctx->host_params), nthr);
        opt.busy_ms += std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
        return true;
      };
      const auto deadline = std::chrono::steady_clock::now() + std::chrono::seconds(3600);
      for (int u = L + 1; u >= 1; --u) {
        while (true) {  // bounded poll of the unit's landed event
          if (opt.abort || std::chrono::steady_clock::now() > deadline) {
            opt.status = MT_ERR_TIMEOUT;
            return;
          }
          const cudaError_t e = cudaEventQuery(st.landed[u]);
          if (e == cudaSuccess) break;
          if (e != cudaErrorNotReady) {
            opt.status = MT_ERR_CUDA;
            return;
          }
          std::this_thread::sleep_for(std::chrono::microseconds(100));
        }
        if (!update(u)) return;
      }
      while (!opt.emb_ready) {
        if (opt.abort || std::chrono::steady_clock::now() > deadline) {
          opt.status = MT_ERR_TIMEOUT;
          return;
        }
        std::this_thread::sleep_for(std::chrono::microseconds(100));
      }
      update(0);
    });
  }
  // Embedding backward: the gradient rows of the used ids (summed in
  // position order) are packed densely, copied to a pinned staging buffer,
  // and scattered into the cleared host gradient after the step drains.
  {
    SegScope sg(ctx, 0, s, 0, (int)n);
    CKL(embed_scatter_rows(ctx->perm_d, ctx->ids_start_d, n_ids, ctx->dh, ctx->dm, h, s));
  }
  cudaEvent_t emb_done = next_event(ctx);
  CK(cudaEventRecord(emb_done, s));
  CK(cudaStreamWaitEvent(ctx->s_d2h, emb_done, 0));
  {
    SegScope sg(ctx, 2, ctx->s_d2h, (double)n_ids * h * 4, (int)n);
    CK(cudaMemcpyAsync(ctx->host_grad_rows, ctx->dm, (size_t)n_ids * h * 4, cudaMemcpyDeviceToHost, ctx->s_d2h));
  }
  ctx->stats.d2h_bytes += (double)n_ids * h * 4;
  // Completion: the grad stream's last copy, and the loss.
  float* loss_host = (float*)(ctx->host_stage + 5 * (size_t)p.Tmax + 1);
  CK(cudaStreamWaitEvent(ctx->s_d2h, ctx->ev_wfree[0], 0));
  CK(cudaStreamWaitEvent(ctx->s_d2h, ctx->ev_wfree[1], 0));
  CK(cudaMemcpyAsync(loss_host, ctx->loss_dev, 4, cudaMemcpyDeviceToHost, ctx->s_d2h));
  cudaEvent_t h2d_end = next_event(ctx);
  CK(cudaEventRecord(h2d_end, ctx->s_h2d));
  CK(cudaStreamWaitEvent(ctx->s_d2h, h2d_end, 0));
  CK(cudaEventRecord(ctx->ev_done, ctx->s_d2h));
  CKR(wait_event(ctx, ctx->ev_done, 3600.0));
  *loss_out = *loss_host;
  toucher.stop();
  ctx->stats.page_touch_ms = toucher.busy_ms();
  // Scatter the embedding gradient rows into the (now cleared) host buffer.
  for (auto& x : zeroers) x.join();
  {
    uint8_t* eg = (uint8_t*)st.host_grad + ctx->off_g[0][0];
    const float* src = ctx->host_grad_rows;
    const size_t gesz = p.gesz;
    const int nthr = (int)std::min<unsigned>(8, std::max(1u, std::thread::hardware_concurrency() / 2));
    std::vector<std::thread> sth;
    const int per = (n_ids + nthr - 1) / nthr;
    for (int i = 0; i < nthr; ++i) {
      const int u0 = i * per, u1 = std::min(n_ids, u0 + per);
      if (u0 >= u1) break;
      sth.emplace_back([=] {
        for (int u = u0; u < u1; ++u) {
          const float* row = src + (size_t)u * h;
          if (gesz == 4) {
            std::memcpy(eg + (size_t)ids[u] * h * 4, row, (size_t)h * 4);
          } else {
            uint16_t* dst = (uint16_t*)eg + (size_t)ids[u] * h;
            for (int c = 0; c < h; ++c) dst[c] = host_bf16_rne(row[c]);
          }
        }
      });
    }
    for (auto& x : sth) x.join();
  }
  if (have_pending) {
    const auto t_drained = std::chrono::steady_clock::now();
    opt.th.join();
    arun.th.join();
    ctx->stats.optimizer_ms = arun.busy_ms;
    ctx->stats.optimizer_exposed_ms =
        std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t_drained).count();
    if (opt.status != MT_OK)
      return set_err(ctx, opt.status, opt.status == MT_ERR_DEVICE ? "device error before publishing an update"
                                                                  : "optimizer did not finish");
  }
  if (st.train) {
    const auto t_drained = std::chrono::steady_clock::now();
    opt.emb_ready = 1;
    opt.th.join();
    ctx->stats.optimizer_ms = opt.busy_ms;
    ctx->stats.optimizer_exposed_ms =
        std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t_drained).count();
    if (opt.status != MT_OK)
      return set_err(ctx, opt.status, opt.status == MT_ERR_DEVICE ? "device error before an optimizer update"
                                                                  : "optimizer did not finish");
  }
  return MT_OK;
}

void compute_stats(mt_ctx* ctx) {
  ctx->stats.n_launches = (int32_t)(g_kernel_launches - ctx->launches_at_start);
  for (auto& o : ctx->opsegs) {
    float ms = 0;
    if (cudaEventElapsedTime(&ms, o.a, o.b) != cudaSuccess) continue;
    if (o.cat == 0) {
      ctx->stats.gemm_ms += ms;
      ctx->stats.gemm_flop += o.flop;
      ctx->stats.n_gemm += 1;
    } else {
      ctx->stats.attn_ms += ms;
      ctx->stats.attn_flop += o.flop;
      ctx->stats.n_attn += 1;
    }
  }
  if (!ctx->trace || ctx->segs.empty()) return;
  struct Iv {
    double a, b;
  };
  std::vector<Iv> comp, h2d, d2h;
  std::vector<double> rates;  // GB/s of each weight copy
  double end = 0;
  for (auto& sg : ctx->segs) {
    float ta = 0, tb = 0;
    if (cudaEventElapsedTime(&ta, ctx->ev_base, sg.a) != cudaSuccess) continue;
    if (cudaEventElapsedTime(&tb, ctx->ev_base, sg.b) != cudaSuccess) continue;
    Iv v{ta, tb};
    end = std::max(end, (double)tb);
    if (sg.stream == 0) comp.push_back(v);
    else if (sg.stream == 1) h2d.push_back(v);
    else d2h.push_back(v);
    if (sg.stream != 0 && sg.unit >= 0 && sg.unit < (int)ctx->unit_phase.size()) {
      const int ph = ctx->unit_phase[sg.unit];
      (sg.stream == 1 ? ctx->stats.h2d_phase_bytes : ctx->stats.d2h_phase_bytes)[ph] += sg.bytes;
      (sg.stream == 1 ? ctx->stats.h2d_phase_ms : ctx->stats.d2h_phase_ms)[ph] += tb - ta;
      if (sg.stream == 1 && tb > ta) rates.push_back(sg.bytes / ((tb - ta) * 1e6));
    }
  }
  if (!rates.empty()) {
    std::sort(rates.begin(), rates.end());
    auto pct = [&](double q) { return rates[std::min(rates.size() - 1, (size_t)(q * (rates.size() - 1) + 0.5))]; };
    ctx->stats.h2d_copy_gbs_min = rates.front();
    ctx->stats.h2d_copy_gbs_p10 = pct(0.1);
    ctx->stats.h2d_copy_gbs_p50 = pct(0.5);
    ctx->stats.h2d_copy_gbs_p90 = pct(0.9);
  }
  if (!ctx->timeline.empty()) {
    FILE* f = fopen(ctx->timeline.c_str(), "w");
    if (f) {
      fprintf(f, "stream,unit,start_ms,end_ms,bytes\n");
      for (auto& sg : ctx->segs) {
        float ta = 0, tb = 0;
        if (cudaEventElapsedTime(&ta, ctx->ev_base, sg.a) != cudaSuccess) continue;
        if (cudaEventElapsedTime(&tb, ctx->ev_base, sg.b) != cudaSuccess) continue;
        fprintf(f, "%s,%d,%.4f,%.4f,%.0f\n", sg.stream == 0 ? "compute" : sg.stream == 1 ? "h2d" : "d2h", sg.unit, ta,
                tb, sg.bytes);
      }
      fclose(f);
    }
  }
  std::sort(comp.begin(), comp.end(), [](const Iv& x, const Iv& y) { return x.a < y.a; });
  std::vector<Iv> uni;
  for (auto& v : comp) {
    if (!uni.empty() && v.a <= uni.back().b) uni.back().b = std::max(uni.back().b, v.b);
    else uni.push_back(v);
  }
  double busy = 0;
  for (auto& v : uni) busy += v.b - v.a;
  auto hidden = [&](const std::vector<Iv>& cps, double* total) {
    double tot = 0, hid = 0;
    for (auto& c : cps) {
      tot += c.b - c.a;
      for (auto& u : uni) {
        const double lo = std::max(c.a, u.a), hi = std::min(c.b, u.b);
        if (hi > lo) hid += hi - lo;
      }
    }
    *total = tot;
    return tot > 0 ? hid / tot : 1.0;
  };
  ctx->stats.compute_busy_ms = busy;
  ctx->stats.h2d_hidden_frac = hidden(h2d, &ctx->stats.h2d_ms);
  ctx->stats.d2h_hidden_frac = hidden(d2h, &ctx->stats.d2h_ms);
  ctx->stats.step_ms = end;
}

}  // namespace

// ===========================================================================
// C ABI
// ===========================================================================
extern "C" {

size_t mt_packed_bytes(const mt_layer_cfg* cfg, mt_dtype dtype) {
  if (!cfg || cfg->n_layers < 1) return 0;
  return build_layout(*cfg, dtype_esz(dtype), nullptr);
}

int mt_tensor_offset(const mt_layer_cfg* cfg, mt_dtype dtype, int unit, int tensor, size_t* off, size_t* bytes) {
  if (!cfg || !off || !bytes || unit < 0 || unit > cfg->n_layers + 1 || tensor < 0 ||
      tensor >= tensors_in_unit(*cfg, unit))
    return MT_ERR_ARG;
  std::vector<std::vector<size_t>> o;
  const size_t esz = dtype_esz(dtype);
  build_layout(*cfg, esz, &o);
  *off = o[unit][tensor];
  *bytes = tensor_bytes(*cfg, unit, tensor, esz);
  return MT_OK;
}

int mt_quantize_params_fp8(const mt_layer_cfg* cfg, const void* src, mt_dtype src_dtype, void* dst,
                           int32_t n_threads) {
  if (!cfg || !src || !dst || n_threads < 0 || cfg->n_layers < 1) return MT_ERR_ARG;
  if (src_dtype != MT_F32 && src_dtype != MT_BF16) return MT_ERR_ARG;
  const mt_layer_cfg& c = *cfg;
  std::vector<std::vector<size_t>> os, od;
  const size_t es = dtype_esz(src_dtype);
  build_layout(c, es, &os);
  build_layout(c, 1, &od);
  const uint8_t* S = (const uint8_t*)src;
  uint8_t* Dp = (uint8_t*)dst;
  auto val = [&](const uint8_t* base, size_t i) -> float {
    if (es == 4) return ((const float*)base)[i];
    uint32_t u = (uint32_t)((const uint16_t*)base)[i] << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return f;
  };
  // one task per tensor row block; every row is quantised independently
  struct Job {
    const uint8_t* s;
    uint8_t* d;
    size_t rows, cols;
    bool gain;
  };
  std::vector<Job> jobs;
  for (int u = 0; u <= c.n_layers + 1; ++u)
    for (int t = 0; t < tensors_in_unit(c, u); ++t) {
      const size_t n = tensor_numel(c, u, t);
      if (is_gain(c, u, t)) {
        jobs.push_back({S + os[u][t], Dp + od[u][t], 1, n, true});
      } else {
        const size_t cols = tensor_cols(c, u, t);
        jobs.push_back({S + os[u][t], Dp + od[u][t], n / cols, cols, false});
      }
    }
  std::atomic<int> bad{0};
  auto run_rows = [&](const Job& j, size_t r0, size_t r1) {
    if (j.gain) {
      for (size_t i = 0; i < j.cols; ++i) ((float*)j.d)[i] = val(j.s, i);
      return;
    }
    float* scales = (float*)(j.d + rup(j.rows * j.cols, 16));
    for (size_t r = r0; r < r1; ++r) {
      float amax = 0.f;
      for (size_t cc = 0; cc < j.cols; ++cc) {
        const float v = val(j.s, r * j.cols + cc);
        if (!std::isfinite(v)) bad = 1;
        amax = std::max(amax, std::fabs(v));
      }
      const float sc = amax > 0.f ? amax / 448.f : 1.f;
      scales[r] = sc;
      for (size_t cc = 0; cc < j.cols; ++cc) j.d[r * j.cols + cc] = e4m3_encode(val(j.s, r * j.cols + cc) / sc);
    }
  };
  const int nthr = n_threads > 0 ? n_threads : (int)std::max(1u, std::thread::hardware_concurrency());
  std::vector<std::thread> th;
  for (int w = 0; w < nthr; ++w)
    th.emplace_back([&, w] {
      for (const Job& j : jobs) {
        const size_t per = (j.rows + nthr - 1) / nthr;
        const size_t r0 = (size_t)w * per, r1 = std::min(j.rows, r0 + per);
        if (j.gain ? w == 0 : r0 < r1) run_rows(j, r0, r1);
      }
    });
  for (auto& x : th) x.join();
  return bad ? MT_ERR_ARG : MT_OK;
}

size_t mt_required_budget(const mt_layer_cfg* cfg) {
  if (!cfg || !cfg_valid(*cfg, nullptr)) return 0;
  Plan p;
  make_plan(*cfg, &p);
  return p.total;
}

static int create_impl(const mt_layer_cfg* cfg, size_t budget, void* arena, void* const* streams, mt_ctx** out) {
  if (!cfg || !out) return MT_ERR_ARG;
  *out = nullptr;
  std::string why;
  if (!cfg_valid(*cfg, &why)) {
    fprintf(stderr, "mt_create: %s\n", why.c_str());
    return ((cfg->n_experts && cfg->param_dtype != MT_BF16 && cfg->param_dtype != MT_FP8) || cfg->hidden % 64 ||
            (cfg->param_dtype == MT_FP8 && cfg->ffn_dim % 16) ||
            (cfg->head_dim != 16 && cfg->head_dim != 32 && cfg->head_dim != 64 && cfg->head_dim != 128))
               ? MT_ERR_UNSUPPORTED
               : MT_ERR_ARG;
  }
  mt_ctx* ctx = new (std::nothrow) mt_ctx();
  if (!ctx) return MT_ERR_CUDA;
  ctx->cfg = *cfg;
  make_plan(*cfg, &ctx->P);
  if (ctx->P.total > budget) {
    delete ctx;
    return MT_ERR_BUDGET;
  }
  build_layout(*cfg, ctx->P.esz, &ctx->off_p);
  build_layout(*cfg, ctx->P.gesz, &ctx->off_g);
  const char* tr = getenv("MT_TRACE");
  ctx->trace = tr ? atoi(tr) : 1;
  if (ctx->trace < 0 || ctx->trace > 2) ctx->trace = 1;
  const char* ft = getenv("MT_FUSE_TOP_BLOCK");
  ctx->fuse_top = !(ft && ft[0] == '0');
  const char* ds = getenv("MT_DEBUG_SYNC");
  ctx->debug_sync = ds && ds[0] == '1';
  const char* ts = getenv("MT_TRACE_SAMPLE");
  if (ts && atoi(ts) > 0) ctx->trace_sample = atoi(ts);
  const char* se = getenv("MT_SERIAL");
  ctx->serial = se && se[0] == '1';
  const char* nv = getenv("MT_NVTX");
  ctx->nvtx = nv && nv[0] == '1';
  const char* tl = getenv("MT_TIMELINE");
  if (tl) ctx->timeline = tl;
  const char* pt = getenv("MT_PAGE_TOUCH");
  if (pt) ctx->touch_threads = std::max(0, std::min(64, atoi(pt)));
  auto fail = [&](int code, const char* m, cudaError_t e) {
    fprintf(stderr, "mt_create: %s: %s\n", m, cudaGetErrorString(e));
    mt_destroy(ctx);
    return code;
  };
  cudaError_t e;
  if ((e = cudaGetDevice(&ctx->device)) != cudaSuccess) return fail(MT_ERR_CUDA, "cudaGetDevice", e);
  if (arena) {
    if ((uintptr_t)arena & 255) {
      mt_destroy(ctx);
      return MT_ERR_ALIGN;
    }
    ctx->arena = (uint8_t*)arena;
    ctx->arena_bytes = budget;
    ctx->own_arena = false;
  } else {
    ctx->arena_bytes = ctx->P.total;
    if ((e = cudaMalloc(&ctx->arena, ctx->arena_bytes)) != cudaSuccess) return fail(MT_ERR_BUDGET, "cudaMalloc", e);
    ctx->own_arena = true;
  }
  if (streams) {
    ctx->s_comp = (cudaStream_t)streams[0];
    ctx->s_h2d = (cudaStream_t)streams[1];
    ctx->s_d2h = (cudaStream_t)streams[2];
    ctx->own_streams = false;
  } else {
    if ((e = cudaStreamCreateWithFlags(&ctx->s_comp, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&ctx->s_h2d, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&ctx->s_d2h, cudaStreamNonBlocking)) != cudaSuccess)
      return fail(MT_ERR_CUDA, "stream create", e);
    ctx->own_streams = true;
  }
  for (int i = 0; i < 2; ++i) {
    if ((e = cudaEventCreateWithFlags(&ctx->ev_wready[i], cudaEventDisableTiming)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&ctx->ev_wfree[i], cudaEventDisableTiming)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&ctx->ev_bwd_done[i], cudaEventDisableTiming)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&ctx->ev_gfree[i], cudaEventDisableTiming)) != cudaSuccess)
      return fail(MT_ERR_CUDA, "event create", e);
  }
  if ((e = cudaEventCreateWithFlags(&ctx->ev_done, cudaEventDisableTiming)) != cudaSuccess ||
      (e = cudaEventCreate(&ctx->ev_base)) != cudaSuccess)
    return fail(MT_ERR_CUDA, "event create", e);
  const size_t stage_ints = 5 * (size_t)ctx->P.Tmax + 1 + 64;
  if ((e = cudaHostAlloc((void**)&ctx->host_stage, stage_ints * 4, cudaHostAllocDefault)) != cudaSuccess ||
      (e = cudaHostAlloc((void**)&ctx->host_rows, (size_t)ctx->P.Tmax * ctx->P.h * (ctx->P.esz == 4 ? 4 : 2),
                         cudaHostAllocDefault)) !=
          cudaSuccess ||
      (e = cudaHostAlloc((void**)&ctx->host_grad_rows, (size_t)ctx->P.Tmax * ctx->P.h * 4, cudaHostAllocDefault)) !=
          cudaSuccess)
    return fail(MT_ERR_CUDA, "cudaHostAlloc", e);
  if (carve(ctx) != MT_OK) {
    mt_destroy(ctx);
    return MT_ERR_BUDGET;
  }
  *out = ctx;
  return MT_OK;
}

int mt_create(const mt_layer_cfg* cfg, size_t device_budget_bytes, mt_ctx** out) {
  return create_impl(cfg, device_budget_bytes, nullptr, nullptr, out);
}

int mt_create_ex(const mt_layer_cfg* cfg, size_t device_budget_bytes, void* device_arena, void* const* streams,
                 mt_ctx** out) {
  if (!device_arena) return MT_ERR_ARG;
  return create_impl(cfg, device_budget_bytes, device_arena, streams, out);
}

int mt_bind_host_params(mt_ctx* ctx, const void* host_params, mt_dtype dtype) {
  if (!ctx || !host_params) return set_err(ctx, MT_ERR_ARG, "null argument");
  if ((int)dtype != ctx->cfg.param_dtype) return set_err(ctx, MT_ERR_ARG, "dtype differs from cfg.param_dtype");
  if ((uintptr_t)host_params & 4095) return set_err(ctx, MT_ERR_ALIGN, "host params not 4096-byte aligned");
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, host_params) != cudaSuccess || at.type != cudaMemoryTypeHost) {
    cudaGetLastError();
    return set_err(ctx, MT_ERR_NOT_PINNED, "host params are not page-locked CUDA host memory");
  }
  void* dev = nullptr;
  if (cudaHostGetDevicePointer(&dev, const_cast<void*>(host_params), 0) != cudaSuccess || !dev) {
    cudaGetLastError();
    return set_err(ctx, MT_ERR_NOT_PINNED, "host params are not mapped into the device address space");
  }
  ctx->host_params = host_params;
  ctx->host_params_dev = dev;
  return MT_OK;
}

int step_common(mt_ctx* ctx, const int32_t* tokens, const int32_t* labels, int B, int S, int K, float* host_grad_out,
                float* loss_out, bool train, bool async_ = false);

int mt_forward_backward(mt_ctx* ctx, const int32_t* tokens, const int32_t* labels, int B, int S, int K,
                        float* host_grad_out, float* loss_out) {
  return step_common(ctx, tokens, labels, B, S, K, host_grad_out, loss_out, false);
}

int mt_train_step(mt_ctx* ctx, const int32_t* tokens, const int32_t* labels, int B, int S, int K,
                  float* host_grad_out, float* loss_out) {
  if (!ctx) return MT_ERR_ARG;
  if (!ctx->opt_bound) return set_err(ctx, MT_ERR_STATE, "no optimizer bound");
  if (ctx->opt_pending) return set_err(ctx, MT_ERR_STATE, "an asynchronous update is pending; call mt_optimizer_flush");
  const int rc = step_common(ctx, tokens, labels, B, S, K, host_grad_out, loss_out, true);
  if (rc == MT_OK) ctx->opt_step += 1;
  return rc;
}

int mt_train_step_async(mt_ctx* ctx, const int32_t* tokens, const int32_t* labels, int B, int S, int K,
                        float* host_grad_out, float* loss_out) {
  if (!ctx) return MT_ERR_ARG;
  if (!ctx->opt_bound) return set_err(ctx, MT_ERR_STATE, "no optimizer bound");
  if (host_grad_out && host_grad_out == ctx->opt_pending)
    return set_err(ctx, MT_ERR_ARG, "the previous call's gradient buffer is still being read; alternate two buffers");
  const bool pending = ctx->opt_pending != nullptr;
  const int rc = step_common(ctx, tokens, labels, B, S, K, host_grad_out, loss_out, false, true);
  // On failure the pending update stays pending: opt_state records the units
  // already computed or published, which the next call or the flush skips.
  if (rc != MT_OK) return rc;
  if (pending) ctx->opt_step += 1;
  ctx->opt_pending = host_grad_out;
  ctx->opt_state.assign((size_t)ctx->cfg.n_layers + 2, 0);
  return MT_OK;
}

int mt_optimizer_flush(mt_ctx* ctx) {
  if (!ctx) return MT_ERR_ARG;
  if (!ctx->opt_bound) return set_err(ctx, MT_ERR_STATE, "no optimizer bound");
  if (!ctx->opt_pending) return MT_OK;
  const int nthr = ctx->opt_threads > 0 ? ctx->opt_threads : (int)std::max(1u, std::thread::hardware_concurrency());
  const int L = ctx->cfg.n_layers;
  const AdamCoef coef = adam_coef(ctx->opt, ctx->opt_step);
  for (int u = 0; u < L + 2; ++u) {
    if (ctx->opt_state[u] == 0)  // compute and publish
      adamw_units(ctx->cfg, ctx->off_g, ctx->off_p, ctx->P.esz, coef, u, u + 1, ctx->opt_master, ctx->opt_m,
                  ctx->opt_v, ctx->opt_pending, const_cast<void*>(ctx->host_params), nthr);
    else if (ctx->opt_state[u] == 1)  // computed by a call that failed before publishing it
      publish_units(ctx->cfg, ctx->off_g, ctx->off_p, ctx->P.esz, u, u + 1, ctx->opt_master,
                    const_cast<void*>(ctx->host_params), nthr);
  }
  ctx->opt_step += 1;
  ctx->opt_pending = nullptr;
  ctx->opt_state.assign((size_t)L + 2, 0);
  return MT_OK;
}

int mt_bind_optimizer(mt_ctx* ctx, const mt_adamw_cfg* opt, float* master, float* m, float* v, int32_t n_threads) {
  if (!ctx || !opt || !master || !m || !v || n_threads < 0) return set_err(ctx, MT_ERR_ARG, "null argument");
  if (!(opt->lr >= 0.f) || !(opt->beta1 >= 0.f && opt->beta1 < 1.f) || !(opt->beta2 >= 0.f && opt->beta2 < 1.f) ||
      !(opt->eps > 0.f) || !(opt->weight_decay >= 0.f))
    return set_err(ctx, MT_ERR_ARG, "AdamW hyper-parameters out of range");
  if (ctx->cfg.grad_dtype != MT_F32)
    return set_err(ctx, MT_ERR_UNSUPPORTED, "the host optimizer takes fp32 gradients (grad_dtype = MT_F32)");
  if (ctx->cfg.param_dtype == MT_FP8)
    return set_err(ctx, MT_ERR_UNSUPPORTED, "the host optimizer publishes fp32 or bf16 parameters, not FP8");
  ctx->opt = *opt;
  ctx->opt_master = master;
  ctx->opt_m = m;
  ctx->opt_v = v;
  ctx->opt_threads = n_threads;
  ctx->opt_step = 1;
  ctx->opt_pending = nullptr;
  ctx->opt_state.assign((size_t)ctx->cfg.n_layers + 2, 0);
  ctx->opt_bound = true;
  return MT_OK;
}

int mt_adamw_update(const mt_layer_cfg* cfg, const mt_adamw_cfg* opt, int64_t step, int32_t unit_begin,
                    int32_t unit_end, float* master, float* m, float* v, const float* grads, void* params,
                    mt_dtype params_dtype, int32_t n_threads) {
  if (!cfg || !opt || !master || !m || !v || !grads || !params || step < 1 || n_threads < 0) return MT_ERR_ARG;
  if (params_dtype == MT_FP8) return MT_ERR_UNSUPPORTED;
  if (params_dtype != MT_F32 && params_dtype != MT_BF16) return MT_ERR_ARG;
  if (unit_begin < 0 || unit_end > cfg->n_layers + 2 || unit_begin > unit_end) return MT_ERR_ARG;
  std::string why;
  if (!cfg_valid(*cfg, &why)) return MT_ERR_ARG;
  if (cfg->grad_dtype != MT_F32) return MT_ERR_UNSUPPORTED;
  std::vector<std::vector<size_t>> off32, offp;
  const size_t esz = params_dtype == MT_BF16 ? 2 : 4;
  build_layout(*cfg, 4, &off32);
  build_layout(*cfg, esz, &offp);
  const int nthr = n_threads > 0 ? n_threads : (int)std::max(1u, std::thread::hardware_concurrency());
  adamw_units(*cfg, off32, offp, esz, adam_coef(*opt, step), unit_begin, unit_end, master, m, v, grads, params, nthr);
  return MT_OK;
}

int step_common(mt_ctx* ctx, const int32_t* tokens, const int32_t* labels, int B, int S, int K, float* host_grad_out,
                float* loss_out, bool train, bool async_) {
  if (!ctx) return MT_ERR_ARG;
  ctx->err.clear();
  if (!ctx->host_params) return set_err(ctx, MT_ERR_STATE, "no parameters bound");
  if (!tokens || !labels || !host_grad_out || !loss_out) return set_err(ctx, MT_ERR_ARG, "null argument");
  if (B < 1 || S < 1 || B > ctx->cfg.max_batch || S > ctx->cfg.max_seq)
    return set_err(ctx, MT_ERR_ARG, "B or S outside [1, max]");
  if (K < 1 || K > ctx->cfg.max_K || K > ctx->cfg.n_layers) return set_err(ctx, MT_ERR_ARG, "K outside [1, min(L, max_K)]");
  const int T = B * S;
  for (int t = 0; t < T; ++t)
    if (tokens[t] < 0 || tokens[t] >= ctx->cfg.vocab || labels[t] < 0 || labels[t] >= ctx->cfg.vocab)
      return set_err(ctx, MT_ERR_ARG, "token or label id outside [0, vocab)");
  if ((uintptr_t)host_grad_out & 4095) return set_err(ctx, MT_ERR_ALIGN, "grad buffer not 4096-byte aligned");
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, host_grad_out) != cudaSuccess || at.type != cudaMemoryTypeHost) {
    cudaGetLastError();
    return set_err(ctx, MT_ERR_NOT_PINNED, "grad buffer is not page-locked CUDA host memory");
  }
  int cur = 0;
  cudaGetDevice(&cur);
  if (cur != ctx->device) cudaSetDevice(ctx->device);
  Step st{ctx, B, S, T, K, (ctx->cfg.n_layers + K - 1) / K, host_grad_out, {}, {}, {}, false, false, {}};
  st.train = train;
  if (train || async_) st.landed.assign(ctx->cfg.n_layers + 2, nullptr);
  st.async = async_;
  const auto t0 = std::chrono::steady_clock::now();
  int rc = run_step(st, tokens, labels, loss_out);
  if (rc != MT_OK) {
    // Drain whatever was enqueued so the context stays usable/destroyable.
    const std::string msg = ctx->err;
    cudaEventRecord(ctx->ev_done, ctx->s_comp);
    ctx->fault_kind = 0;
    wait_event(ctx, ctx->ev_done, 600.0);
    cudaStreamSynchronize(ctx->s_h2d);
    cudaStreamSynchronize(ctx->s_d2h);
    cudaGetLastError();
    ctx->err = msg;
  } else {
    const uint32_t derr = gemm_take_device_error() | attention_tc_take_device_error();
    if (derr) {
      char b[96];
      snprintf(b, sizeof b, "device error word 0x%x (barrier timeout inside a kernel)", derr);
      rc = set_err(ctx, MT_ERR_DEVICE, b);
    } else {
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) rc = set_err(ctx, MT_ERR_CUDA, cudaGetErrorString(e));
    }
    if (rc == MT_OK) ctx->last_T = T;
    compute_stats(ctx);
    if (!ctx->trace)
      ctx->stats.step_ms = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
  }
  if (cur != ctx->device) cudaSetDevice(cur);
  return rc;
}

int mt_get_routing(const mt_ctx* ctx, int32_t* host_out, size_t n) {
  if (!ctx || !host_out) return MT_ERR_ARG;
  if (ctx->cfg.n_experts == 0 || ctx->last_T == 0) return MT_ERR_STATE;
  const size_t need = (size_t)ctx->cfg.n_layers * ctx->last_T * ctx->cfg.top_k;
  if (n != need) return MT_ERR_ARG;
  if (cudaMemcpy(host_out, ctx->moe_route, need * 4, cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return MT_ERR_CUDA;
  }
  return MT_OK;
}

int mt_get_stats(const mt_ctx* ctx, mt_stats* out) {
  if (!ctx || !out) return MT_ERR_ARG;
  *out = ctx->stats;
  return MT_OK;
}

int mt_replay_weight_stream(mt_ctx* ctx, int K, int flags, float* copy_gbs_out, int max_copies,
                            mt_replay_result* out) {
  if (!ctx || !out || max_copies < 0) return set_err(ctx, MT_ERR_ARG, "null argument");
  if (!ctx->host_params) return set_err(ctx, MT_ERR_STATE, "no parameters bound");
  if (K < 1 || K > ctx->cfg.max_K || K > ctx->cfg.n_layers) return set_err(ctx, MT_ERR_ARG, "K outside [1, min(L, max_K)]");
  *out = mt_replay_result{};
  int node = -1;
  if (cudaDeviceGetAttribute(&node, cudaDevAttrHostNumaId, ctx->device) != cudaSuccess) node = -1;
  cudaGetLastError();
  out->host_numa_node = node;
  int cur = 0;
  cudaGetDevice(&cur);
  if (cur != ctx->device) cudaSetDevice(ctx->device);
  Step st{ctx, 1, 1, 1, K, (ctx->cfg.n_layers + K - 1) / K, nullptr, {}, {}, {}, false, false, {}};
  plan_sequence(st);
  const uint8_t* hp = (const uint8_t*)ctx->host_params;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> ev;
  std::vector<double> bytes;
  PageToucher toucher;
  std::vector<int> load_index;
  if (flags & MT_REPLAY_TOUCH) {
    size_t n_copies = 0;
    std::vector<PageToucher::Range> plan = touch_plan(ctx, st, nullptr, &load_index, &n_copies);
    toucher.start(std::move(plan), n_copies, std::max(1, ctx->touch_threads), ctx->device);
    toucher.wait_touched(0, 2.0);
  }
  int rc = MT_OK;
  for (size_t i = 0; i < st.seq.size() && rc == MT_OK; ++i) {
    if (!st.needs_load[i]) continue;
    size_t src_off, nb, soff = 0, sbytes = 0;
    load_range(ctx, st.seq[i], &src_off, &nb, &soff, &sbytes);
    cudaEvent_t a = nullptr, b = nullptr;
    if (cudaEventCreate(&a) != cudaSuccess || cudaEventCreate(&b) != cudaSuccess) {
      if (a) cudaEventDestroy(a);
      rc = set_err(ctx, MT_ERR_CUDA, "event create");
      break;
    }
    ev.push_back({a, b});
    bytes.push_back((double)(nb + sbytes));
    uint8_t* dst = ctx->wbuf[st.slot_of[i]];
    if (cudaEventRecord(a, ctx->s_h2d) != cudaSuccess ||
        cudaMemcpyAsync(dst, hp + src_off, nb, cudaMemcpyHostToDevice, ctx->s_h2d) != cudaSuccess ||
        (sbytes && cudaMemcpyAsync(dst + head_scale_dst(ctx->P, head_slice_rows(ctx->P, st.seq[i].index)),
                                   hp + soff, sbytes, cudaMemcpyHostToDevice, ctx->s_h2d) != cudaSuccess) ||
        cudaEventRecord(b, ctx->s_h2d) != cudaSuccess)
      rc = set_err(ctx, MT_ERR_CUDA, std::string("replay copy: ") + cudaGetErrorString(cudaGetLastError()));
    if (flags & MT_REPLAY_TOUCH) toucher.published((size_t)load_index[i], b);
  }
  if (cudaStreamSynchronize(ctx->s_h2d) != cudaSuccess && rc == MT_OK)
    rc = set_err(ctx, MT_ERR_CUDA, std::string("replay: ") + cudaGetErrorString(cudaGetLastError()));
  for (size_t i = 0; i < ev.size(); ++i) {
    float ms = 0;
    if (rc == MT_OK && cudaEventElapsedTime(&ms, ev[i].first, ev[i].second) == cudaSuccess) {
      out->bytes += bytes[i];
      out->ms += ms;
      if (copy_gbs_out && (int)i < max_copies) copy_gbs_out[i] = ms > 0 ? (float)(bytes[i] / (ms * 1e6)) : 0.f;
    }
    cudaEventDestroy(ev[i].first);
    cudaEventDestroy(ev[i].second);
  }
  toucher.stop();
  out->n_copies = (int32_t)ev.size();
  out->touch_ms = toucher.busy_ms();
  if (cur != ctx->device) cudaSetDevice(cur);
  return rc;
}

int mt_set_tracing(mt_ctx* ctx, int level, int sample) {
  if (!ctx || level < 0 || level > 2 || sample < 1) return MT_ERR_ARG;
  ctx->trace = level;
  ctx->trace_sample = sample;
  ctx->op_counter = 0;
  return MT_OK;
}

int mt_get_memory_plan(const mt_ctx* ctx, mt_memory_plan* out) {
  if (!ctx || !out) return MT_ERR_ARG;
  const Plan& p = ctx->P;
  out->total = p.total;
  out->weight_buffers = 2 * p.wbuf + 2 * p.wcast;
  out->grad_buffers = 2 * p.gbuf;
  out->workspace = p.fixed_ws;
  size_t ck = 0, ac = 0;
  for (int K = 1; K <= std::min(ctx->cfg.max_K, p.L); ++K) {
    const size_t nb = (p.L + K - 1) / K;
    if (nb * p.ckpt_one + (size_t)K * p.act_layer == p.dyn_max) {
      ck = nb * p.ckpt_one;
      ac = (size_t)K * p.act_layer;
    }
  }
  out->checkpoints = ck;
  out->block_activations = ac;
  return MT_OK;
}

const char* mt_last_error(const mt_ctx* ctx) { return ctx ? ctx->err.c_str() : "null context"; }

void mt_destroy(mt_ctx* ctx) {
  if (!ctx) return;
  if (ctx->s_comp) cudaStreamSynchronize(ctx->s_comp);
  if (ctx->s_h2d) cudaStreamSynchronize(ctx->s_h2d);
  if (ctx->s_d2h) cudaStreamSynchronize(ctx->s_d2h);
  for (int i = 0; i < 2; ++i) {
    if (ctx->ev_wready[i]) cudaEventDestroy(ctx->ev_wready[i]);
    if (ctx->ev_wfree[i]) cudaEventDestroy(ctx->ev_wfree[i]);
    if (ctx->ev_bwd_done[i]) cudaEventDestroy(ctx->ev_bwd_done[i]);
    if (ctx->ev_gfree[i]) cudaEventDestroy(ctx->ev_gfree[i]);
  }
  if (ctx->ev_done) cudaEventDestroy(ctx->ev_done);
  if (ctx->ev_base) cudaEventDestroy(ctx->ev_base);
  for (auto e : ctx->ev_pool) cudaEventDestroy(e);
  if (ctx->own_streams) {
    if (ctx->s_comp) cudaStreamDestroy(ctx->s_comp);
    if (ctx->s_h2d) cudaStreamDestroy(ctx->s_h2d);
    if (ctx->s_d2h) cudaStreamDestroy(ctx->s_d2h);
  }
  if (ctx->own_arena && ctx->arena) cudaFree(ctx->arena);
  if (ctx->host_stage) cudaFreeHost(ctx->host_stage);
  if (ctx->host_rows) cudaFreeHost(ctx->host_rows);
  if (ctx->host_grad_rows) cudaFreeHost(ctx->host_grad_rows);
  delete ctx;
}

// Pinned host memory from cudaHostAlloc (driver-allocated page-locked memory:
// on this platform the copy engines stream it at the link rate, whereas
// cudaHostRegister'ed anonymous memory of the same size streamed an order of
// magnitude slower in measurements). The calling thread's memory policy is
// set to prefer the host NUMA node nearest the current GPU for the duration
// of the allocation, so that the pages land next to the GPU's link on
// multi-node hosts. A small header just below the returned (4096-aligned)
// pointer keeps the original allocation for mt_host_free.
namespace {
struct HostBlock {
  void* base;
  size_t bytes;
};
}  // namespace

void* mt_host_alloc(size_t bytes) {
  const size_t total = (bytes ? bytes : 1) + 4096 + sizeof(HostBlock);
  int dev = 0, node = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&node, cudaDevAttrHostNumaId, dev) != cudaSuccess)
    node = -1;
  cudaGetLastError();
  bool policy_set = false;
  if (node >= 0 && node < 1024) {
    unsigned long mask[16] = {0};
    mask[node / 64] |= 1ul << (node % 64);
    policy_set = syscall(SYS_set_mempolicy, 1 /* MPOL_PREFERRED */, mask, 1025ul) == 0;
  }
  void* p = nullptr;
  const cudaError_t e = cudaHostAlloc(&p, total, cudaHostAllocDefault);
  if (policy_set) syscall(SYS_set_mempolicy, 0 /* MPOL_DEFAULT */, nullptr, 0ul);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  const uintptr_t a = ((uintptr_t)p + sizeof(HostBlock) + 4095) & ~(uintptr_t)4095;
  *((HostBlock*)a - 1) = HostBlock{p, total};
  return (void*)a;
}

void mt_host_free(void* p) {
  if (p) cudaFreeHost(((const HostBlock*)p - 1)->base);
}

int mt_debug_inject_fault(mt_ctx* ctx, int kind, int nth) {
  if (!ctx || kind < 0 || kind > 2 || (kind && nth < 1)) return MT_ERR_ARG;
  ctx->fault_kind = kind;
  ctx->fault_nth = nth;
  return MT_OK;
}

}  // extern "C"
