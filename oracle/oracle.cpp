// CPU oracle for layer-streamed decoder training.
//
// TEST INFRASTRUCTURE ONLY. Nothing in the product path links, loads or calls
// this file; only the tests, the smoke check and the CPU-baseline leg of the
// benchmark do. It shares no code, header, table or helper with the CUDA
// library: the packed-parameter layout below is written out again from its
// definition, and every operation is a plain loop in the scalar type S
// (float for the reference, double for the finite-difference pins).
//
// What it computes is the plain definition of one training step of a
// Llama-style decoder ("MegaTrain: Full Precision Training of 100B+ Parameter
// Large Language Models on a Single GPU", section 方法步骤详情, stages 1-3):
//   h_0 = Embed(x); h_i = f_i(h_{i-1}, theta_i) for i = 1..L;
//   loss = L(h_L); then the gradient of every parameter.
// The streamed method reaches exactly this result (up to rounding order):
// streaming, checkpointing every K layers and block-wise recompute change
// where values live and when they are made, not what they are (same page,
// 核心方法 and 实验结果: the system matches native full-GPU training).
// Here everything is materialised and there is no recompute.
//
// Readings where the pages are silent (each listed in the design notes):
//  - layer f_i: pre-norm RMSNorm -> q,k,v projections -> RoPE on q,k (half-
//    split pairs (i, i+d/2), angle = pos * theta^(-2i/d), pos = index within
//    the sequence) -> causal softmax attention with scale 1/sqrt(d), query
//    head j reading KV head floor(j / (n_q/n_kv)) -> h += o Wo^T ->
//    RMSNorm -> SwiGLU MLP silu(m Wg^T) * (m Wu^T) -> h += a Wd^T;
//  - final RMSNorm before the untied LM head; loss = scale * sum_t CE_t with
//    scale = 1/T by default (mean over the B*S tokens);
//  - RoPE angles are formed in double precision in both instantiations (the
//    angle is a definition, not part of the arithmetic under test), then
//    cos/sin are rounded to S;
//  - no biases, no dropout.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

struct Dims {
  int L, h, nq, nkv, d, F, V;
  double theta, eps;
  int E, topk, Fe;  // mixture-of-experts FFN when E > 0 (F unused then)
};

// ---------------------------------------------------------------------------
// Packed layout (the library's documented host format, restated here):
// unit 0 = embedding E[V,h]; units 1..L = one decoder layer each, holding
// w_attn_norm[h], Wq[nq*d,h], Wk[nkv*d,h], Wv[nkv*d,h], Wo[h,nq*d],
// w_ffn_norm[h], Wg[F,h], Wu[F,h], Wd[h,F] (mixture-of-experts layers hold
// instead the router Wr[E,h], the experts' gate and up rows Wgu[E,2Fe,h]
// (rows [0,Fe) gate, [Fe,2Fe) up) and their down matrices Wd[E,h,Fe], in
// the same three places); unit L+1 = final norm w_f[h] and
// the head W_out[V,h]. Matrices are row-major [out,in]. Every tensor starts
// on a 256-byte boundary and every unit on a 4096-byte boundary ("layer
// contiguous tiling ... aligned to 4KB pages", same page, 技术新颖性).
// ---------------------------------------------------------------------------
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int unit_tensor_count(const Dims& D, int unit) {
  if (unit == 0) return 1;
  if (unit >= 1 && unit <= D.L) return 9;
  if (unit == D.L + 1) return 2;
  return 0;
}

size_t tensor_elems(const Dims& D, int unit, int t) {
  const size_t h = D.h, qd = (size_t)D.nq * D.d, kd = (size_t)D.nkv * D.d, F = D.F, V = D.V;
  if (unit == 0) return V * h;
  if (unit == D.L + 1) return t == 0 ? h : V * h;
  if (D.E > 0 && t >= 6) {
    const size_t E = D.E, Fe = D.Fe;
    return t == 6 ? E * h : t == 7 ? E * 2 * Fe * h : E * h * Fe;
  }
  switch (t) {
    case 0: return h;       // w_attn_norm
    case 1: return qd * h;  // Wq
    case 2: return kd * h;  // Wk
    case 3: return kd * h;  // Wv
    case 4: return h * qd;  // Wo
    case 5: return h;       // w_ffn_norm
    case 6: return F * h;   // Wg
    case 7: return F * h;   // Wu
    case 8: return h * F;   // Wd
  }
  return 0;
}

// Byte offset of (unit, tensor) for element size esz; returns the total
// packed size when unit == L+2.
size_t layout_offset(const Dims& D, size_t esz, int unit, int tensor) {
  size_t pos = 0;
  for (int u = 0; u <= D.L + 1; ++u) {
    pos = round_up(pos, 4096);
    const int nt = unit_tensor_count(D, u);
    for (int t = 0; t < nt; ++t) {
      pos = round_up(pos, 256);
      if (u == unit && t == tensor) return pos;
      pos += tensor_elems(D, u, t) * esz;
    }
  }
  return round_up(pos, 4096);
}

// ---------------------------------------------------------------------------
// Plain dense linear algebra. Every output element is a sum taken in
// ascending order of the reduction index; the loops are ordered so that the
// innermost one runs over contiguous memory (transpose once, then axpy).
// ---------------------------------------------------------------------------

// Y[M,N] = X[M,K] * W[N,K]^T
template <class S>
void mm_nt(const S* X, const S* W, S* Y, int M, int N, int K) {
  std::vector<S> WT((size_t)K * N);
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < K; ++k) WT[(size_t)k * N + n] = W[(size_t)n * K + k];
  for (int m = 0; m < M; ++m) {
    S* y = Y + (size_t)m * N;
    for (int n = 0; n < N; ++n) y[n] = S(0);
    for (int k = 0; k < K; ++k) {
      const S xv = X[(size_t)m * K + k];
      const S* w = &WT[(size_t)k * N];
      for (int n = 0; n < N; ++n) y[n] += xv * w[n];
    }
  }
}

// Y[M,N] = X[M,K] * W[K,N]
template <class S>
void mm_nn(const S* X, const S* W, S* Y, int M, int N, int K) {
  for (int m = 0; m < M; ++m) {
    S* y = Y + (size_t)m * N;
    for (int n = 0; n < N; ++n) y[n] = S(0);
    for (int k = 0; k < K; ++k) {
      const S xv = X[(size_t)m * K + k];
      const S* w = W + (size_t)k * N;
      for (int n = 0; n < N; ++n) y[n] += xv * w[n];
    }
  }
}

// Y[M,N] = A[K,M]^T * B[K,N]   (sum over the K rows, e.g. tokens)
template <class S>
void mm_tn(const S* A, const S* B, S* Y, int M, int N, int K) {
  for (size_t i = 0; i < (size_t)M * N; ++i) Y[i] = S(0);
  for (int k = 0; k < K; ++k) {
    const S* b = B + (size_t)k * N;
    for (int m = 0; m < M; ++m) {
      const S av = A[(size_t)k * M + m];
      S* y = Y + (size_t)m * N;
      for (int n = 0; n < N; ++n) y[n] += av * b[n];
    }
  }
}

// ---------------------------------------------------------------------------
// RMSNorm: y = x * w / sqrt(mean(x^2) + eps), per row of length h.
// ---------------------------------------------------------------------------
template <class S>
void rmsnorm_fwd(const S* x, const S* w, int T, int h, double eps, S* y, S* rstd) {
  for (int t = 0; t < T; ++t) {
    const S* xr = x + (size_t)t * h;
    S ss = 0;
    for (int j = 0; j < h; ++j) ss += xr[j] * xr[j];
    const S r = S(1) / std::sqrt(ss / S(h) + S(eps));
    rstd[t] = r;
    for (int j = 0; j < h; ++j) y[(size_t)t * h + j] = xr[j] * r * w[j];
  }
}

// With xhat = x*r and y = xhat*w:
//   dxhat = dy*w;  dx = r * (dxhat - xhat * mean(dxhat*xhat));  dw = sum_t dy*xhat.
// dx is written (not accumulated); dw is accumulated.
template <class S>
void rmsnorm_bwd(const S* x, const S* w, const S* rstd, const S* dy, int T, int h, S* dx, S* dw) {
  for (int t = 0; t < T; ++t) {
    const S* xr = x + (size_t)t * h;
    const S* g = dy + (size_t)t * h;
    const S r = rstd[t];
    S dot = 0;
    for (int j = 0; j < h; ++j) dot += g[j] * w[j] * xr[j] * r;
    const S mean = dot / S(h);
    for (int j = 0; j < h; ++j) {
      const S xh = xr[j] * r;
      dx[(size_t)t * h + j] = r * (g[j] * w[j] - xh * mean);
      dw[j] += g[j] * xh;
    }
  }
}

// ---------------------------------------------------------------------------
// RoPE on a [B*S, nh, d] tensor, half-split pairs (i, i + d/2).
// dir = +1 rotates by +angle (forward), -1 by -angle (the backward, which is
// the transpose of a rotation, i.e. its inverse).
// ---------------------------------------------------------------------------
template <class S>
void rope(S* x, int B, int Sq, int nh, int d, double theta, int dir) {
  const int half = d / 2;
  for (int b = 0; b < B; ++b)
    for (int s = 0; s < Sq; ++s)
      for (int i = 0; i < half; ++i) {
        const double freq = std::pow(theta, -2.0 * i / d);
        const double ang = (double)s * freq;
        const S c = S(std::cos(ang)), sn = S(dir * std::sin(ang));
        for (int j = 0; j < nh; ++j) {
          S* v = x + (((size_t)b * Sq + s) * nh + j) * d;
          const S x1 = v[i], x2 = v[i + half];
          v[i] = x1 * c - x2 * sn;
          v[i + half] = x1 * sn + x2 * c;
        }
      }
}

// ---------------------------------------------------------------------------
// Causal GQA attention. q [B*S, nq, d], k/v [B*S, nkv, d], o [B*S, nq, d].
// P (probabilities) stored as [B, nq, S, S] (upper triangle zero).
// ---------------------------------------------------------------------------
template <class S>
void attn_fwd(const S* q, const S* k, const S* v, int B, int Sq, int nq, int nkv, int d, S* o, S* P, S* lse) {
  const int grp = nq / nkv;
  const S scale = S(1) / std::sqrt(S(d));
  std::vector<S> sc(Sq);
  for (int b = 0; b < B; ++b)
    for (int j = 0; j < nq; ++j) {
      const int kvh = j / grp;
      for (int t = 0; t < Sq; ++t) {
        const S* qr = q + (((size_t)b * Sq + t) * nq + j) * d;
        S mx = -INFINITY;
        for (int s = 0; s <= t; ++s) {
          const S* kr = k + (((size_t)b * Sq + s) * nkv + kvh) * d;
          S dot = 0;
          for (int e = 0; e < d; ++e) dot += qr[e] * kr[e];
          sc[s] = dot * scale;
          mx = std::max(mx, sc[s]);
        }
        S sum = 0;
        for (int s = 0; s <= t; ++s) {
          sc[s] = std::exp(sc[s] - mx);
          sum += sc[s];
        }
        S* prow = P + (((size_t)b * nq + j) * Sq + t) * Sq;
        for (int s = 0; s < Sq; ++s) prow[s] = s <= t ? sc[s] / sum : S(0);
        if (lse) lse[((size_t)b * nq + j) * Sq + t] = mx + std::log(sum);
        S* orow = o + (((size_t)b * Sq + t) * nq + j) * d;
        for (int e = 0; e < d; ++e) orow[e] = 0;
        for (int s = 0; s <= t; ++s) {
          const S* vr = v + (((size_t)b * Sq + s) * nkv + kvh) * d;
          for (int e = 0; e < d; ++e) orow[e] += prow[s] * vr[e];
        }
      }
    }
}

// Backward of attn_fwd given P. dq written; dk, dv written (zeroed here).
template <class S>
void attn_bwd(const S* q, const S* k, const S* v, const S* P, const S* dout, int B, int Sq, int nq, int nkv, int d,
              S* dq, S* dk, S* dv) {
  const int grp = nq / nkv;
  const S scale = S(1) / std::sqrt(S(d));
  const size_t nqel = (size_t)B * Sq * nq * d, nkel = (size_t)B * Sq * nkv * d;
  for (size_t i = 0; i < nqel; ++i) dq[i] = 0;
  for (size_t i = 0; i < nkel; ++i) dk[i] = dv[i] = 0;
  std::vector<S> dP(Sq);
  for (int b = 0; b < B; ++b)
    for (int j = 0; j < nq; ++j) {
      const int kvh = j / grp;
      for (int t = 0; t < Sq; ++t) {
        const S* prow = P + (((size_t)b * nq + j) * Sq + t) * Sq;
        const S* g = dout + (((size_t)b * Sq + t) * nq + j) * d;
        // dV[s] += P[t,s] * dO[t];  dP[t,s] = dO[t] . V[s]
        S rowdot = 0;
        for (int s = 0; s <= t; ++s) {
          const S* vr = v + (((size_t)b * Sq + s) * nkv + kvh) * d;
          S* dvr = dv + (((size_t)b * Sq + s) * nkv + kvh) * d;
          S dot = 0;
          for (int e = 0; e < d; ++e) {
            dvr[e] += prow[s] * g[e];
            dot += g[e] * vr[e];
          }
          dP[s] = dot;
          rowdot += prow[s] * dot;
        }
        // dS = P * (dP - sum_s P dP); scores = q.k * scale
        const S* qr = q + (((size_t)b * Sq + t) * nq + j) * d;
        S* dqr = dq + (((size_t)b * Sq + t) * nq + j) * d;
        for (int s = 0; s <= t; ++s) {
          const S ds = prow[s] * (dP[s] - rowdot) * scale;
          const S* kr = k + (((size_t)b * Sq + s) * nkv + kvh) * d;
          S* dkr = dk + (((size_t)b * Sq + s) * nkv + kvh) * d;
          for (int e = 0; e < d; ++e) {
            dqr[e] += ds * kr[e];
            dkr[e] += ds * qr[e];
          }
        }
      }
    }
}

// silu(g) = g * sigmoid(g)
template <class S>
S sigmoid(S g) { return S(1) / (S(1) + std::exp(-g)); }

template <class S>
void swiglu_fwd(const S* g, const S* u, size_t n, S* a) {
  for (size_t i = 0; i < n; ++i) a[i] = g[i] * sigmoid(g[i]) * u[i];
}

// d silu(g)/dg = sig(g) * (1 + g * (1 - sig(g)))
template <class S>
void swiglu_bwd(const S* g, const S* u, const S* da, size_t n, S* dg, S* du) {
  for (size_t i = 0; i < n; ++i) {
    const S sg = sigmoid(g[i]);
    dg[i] = da[i] * u[i] * sg * (S(1) + g[i] * (S(1) - sg));
    du[i] = da[i] * g[i] * sg;
  }
}

// Cross-entropy over logits z [T,V]: loss = scale * sum_t (lse_t - z[t,label_t]);
// dz = scale * (softmax(z_t) - onehot(label_t)).
template <class S>
S ce_fwd_bwd(const S* z, const int32_t* labels, int T, int V, S scale, S* dz, float* tok_loss = nullptr) {
  S loss = 0;
  for (int t = 0; t < T; ++t) {
    const S* zr = z + (size_t)t * V;
    S mx = -INFINITY;
    for (int v = 0; v < V; ++v) mx = std::max(mx, zr[v]);
    S sum = 0;
    for (int v = 0; v < V; ++v) sum += std::exp(zr[v] - mx);
    const S lse = mx + std::log(sum);
    loss += lse - zr[labels[t]];
    if (tok_loss) tok_loss[t] = (float)(lse - zr[labels[t]]);
    if (dz) {
      S* dr = dz + (size_t)t * V;
      for (int v = 0; v < V; ++v) dr[v] = scale * std::exp(zr[v] - lse);
      dr[labels[t]] -= scale;
    }
  }
  return loss * scale;
}

// ---------------------------------------------------------------------------
// Mixture-of-experts FFN (the MoE layer of the streamed workloads, in the
// style of Qwen3's MoE blocks; the pages name the model and its 128 experts
// with top-8 routing, not the formulas, so this is the plain reading):
//   router logits r = m Wr^T, p = softmax(r) over the E experts;
//   the k experts of largest p are selected (equal p: lower index first);
//   their weights are renormalised, w_j = p_{e_j} / sum_i p_{e_i};
//   expert e is a SwiGLU MLP y_e(x) = (silu(x Wg_e^T) * (x Wu_e^T)) Wd_e^T;
//   out_t = sum_j w_j y_{e_j}(m_t), summed over j = 0..k-1.
// No shared expert, no load-balancing loss. The selection is a function of
// the logits, so its derivative is zero almost everywhere: gradients flow
// into Wr only through the weights w.
// ---------------------------------------------------------------------------
template <class S>
struct MoeAct {
  std::vector<S> p;                     // [T, E] router probabilities
  std::vector<int32_t> sel;             // [T, k] selected experts
  std::vector<S> w;                     // [T, k] renormalised weights
  std::vector<std::vector<int>> rows;   // per expert, the slots t*k+j routed to it, ascending
  std::vector<S> g, u, act, y;          // per slot: [T*k, Fe] (g, u, act), [T*k, h] (y)
};

// Writes out [T, h]. route_in (optional, [T, k]) replaces the selection by the
// given experts (validated by the caller); route_out (optional) receives it;
// logits_out (optional, [T, E]) receives the router logits r.
template <class S>
void moe_fwd(const Dims& D, const S* m, const S* Wr, const S* Wgu, const S* Wd, int T, const int32_t* route_in,
             int32_t* route_out, MoeAct<S>& A, S* out, float* logits_out = nullptr) {
  const int E = D.E, k = D.topk, Fe = D.Fe, h = D.h;
  std::vector<S> r((size_t)T * E);
  mm_nt(m, Wr, r.data(), T, E, h);
  if (logits_out)
    for (size_t i = 0; i < r.size(); ++i) logits_out[i] = (float)r[i];
  A.p.assign((size_t)T * E, S(0));
  A.sel.assign((size_t)T * k, 0);
  A.w.assign((size_t)T * k, S(0));
  std::vector<int> order(E);
  for (int t = 0; t < T; ++t) {
    const S* rt = &r[(size_t)t * E];
    S* pt = &A.p[(size_t)t * E];
    S mx = -INFINITY;
    for (int e = 0; e < E; ++e) mx = std::max(mx, rt[e]);
    S sum = 0;
    for (int e = 0; e < E; ++e) {
      pt[e] = std::exp(rt[e] - mx);
      sum += pt[e];
    }
    for (int e = 0; e < E; ++e) pt[e] /= sum;
    int32_t* st = &A.sel[(size_t)t * k];
    if (route_in) {
      for (int j = 0; j < k; ++j) st[j] = route_in[(size_t)t * k + j];
    } else {
      for (int e = 0; e < E; ++e) order[e] = e;
      std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return pt[a] > pt[b]; });
      for (int j = 0; j < k; ++j) st[j] = order[j];
    }
    if (route_out)
      for (int j = 0; j < k; ++j) route_out[(size_t)t * k + j] = st[j];
    S psel = 0;
    for (int j = 0; j < k; ++j) psel += pt[st[j]];
    for (int j = 0; j < k; ++j) A.w[(size_t)t * k + j] = pt[st[j]] / psel;
  }
  A.rows.assign(E, std::vector<int>());
  for (int t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) A.rows[A.sel[(size_t)t * k + j]].push_back(t * k + j);
  const size_t slots = (size_t)T * k;
  A.g.assign(slots * Fe, S(0));
  A.u.assign(slots * Fe, S(0));
  A.act.assign(slots * Fe, S(0));
  A.y.assign(slots * h, S(0));
  for (int e = 0; e < E; ++e) {
    const std::vector<int>& R = A.rows[e];
    const int n = (int)R.size();
    if (n == 0) continue;
    std::vector<S> X((size_t)n * h), G((size_t)n * Fe), U((size_t)n * Fe), Act((size_t)n * Fe), Y((size_t)n * h);
    for (int i = 0; i < n; ++i)
      for (int c = 0; c < h; ++c) X[(size_t)i * h + c] = m[(size_t)(R[i] / k) * h + c];
    const S* wg = Wgu + (size_t)e * 2 * Fe * h;
    mm_nt(X.data(), wg, G.data(), n, Fe, h);
    mm_nt(X.data(), wg + (size_t)Fe * h, U.data(), n, Fe, h);
    swiglu_fwd(G.data(), U.data(), (size_t)n * Fe, Act.data());
    mm_nt(Act.data(), Wd + (size_t)e * h * Fe, Y.data(), n, h, Fe);
    for (int i = 0; i < n; ++i) {
      for (int c = 0; c < Fe; ++c) {
        A.g[(size_t)R[i] * Fe + c] = G[(size_t)i * Fe + c];
        A.u[(size_t)R[i] * Fe + c] = U[(size_t)i * Fe + c];
        A.act[(size_t)R[i] * Fe + c] = Act[(size_t)i * Fe + c];
      }
      for (int c = 0; c < h; ++c) A.y[(size_t)R[i] * h + c] = Y[(size_t)i * h + c];
    }
  }
  for (int t = 0; t < T; ++t) {
    S* o = out + (size_t)t * h;
    for (int c = 0; c < h; ++c) o[c] = 0;
    for (int j = 0; j < k; ++j) {
      const S wj = A.w[(size_t)t * k + j];
      const S* y = &A.y[((size_t)t * k + j) * h];
      for (int c = 0; c < h; ++c) o[c] += wj * y[c];
    }
  }
}

// Backward of moe_fwd given dout [T, h]: dm [T, h] written; dWr, dWgu, dWd
// written for every expert (zero where no slot was routed).
template <class S>
void moe_bwd(const Dims& D, const S* m, const S* Wr, const S* Wgu, const S* Wd, int T, const MoeAct<S>& A,
             const S* dout, S* dm, S* dWr, S* dWgu, S* dWd) {
  const int E = D.E, k = D.topk, Fe = D.Fe, h = D.h;
  for (size_t i = 0; i < (size_t)E * h; ++i) dWr[i] = 0;
  for (size_t i = 0; i < (size_t)E * 2 * Fe * h; ++i) dWgu[i] = 0;
  for (size_t i = 0; i < (size_t)E * h * Fe; ++i) dWd[i] = 0;
  for (size_t i = 0; i < (size_t)T * h; ++i) dm[i] = 0;
  // out_t = sum_j w_tj y_tj:  dw_tj = <dout_t, y_tj>,  dy_tj = w_tj dout_t
  std::vector<S> dw((size_t)T * k);
  for (int t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) {
      const S* y = &A.y[((size_t)t * k + j) * h];
      S dot = 0;
      for (int c = 0; c < h; ++c) dot += dout[(size_t)t * h + c] * y[c];
      dw[(size_t)t * k + j] = dot;
    }
  for (int e = 0; e < E; ++e) {
    const std::vector<int>& R = A.rows[e];
    const int n = (int)R.size();
    if (n == 0) continue;
    std::vector<S> X((size_t)n * h), dY((size_t)n * h), G((size_t)n * Fe), U((size_t)n * Fe), Act((size_t)n * Fe);
    for (int i = 0; i < n; ++i) {
      const int t = R[i] / k;
      const S wj = A.w[R[i]];
      for (int c = 0; c < h; ++c) {
        X[(size_t)i * h + c] = m[(size_t)t * h + c];
        dY[(size_t)i * h + c] = wj * dout[(size_t)t * h + c];
      }
      for (int c = 0; c < Fe; ++c) {
        G[(size_t)i * Fe + c] = A.g[(size_t)R[i] * Fe + c];
        U[(size_t)i * Fe + c] = A.u[(size_t)R[i] * Fe + c];
        Act[(size_t)i * Fe + c] = A.act[(size_t)R[i] * Fe + c];
      }
    }
    const S* wg = Wgu + (size_t)e * 2 * Fe * h;
    const S* wd = Wd + (size_t)e * h * Fe;
    std::vector<S> dAct((size_t)n * Fe), dG((size_t)n * Fe), dU((size_t)n * Fe), dX((size_t)n * h),
        tmp((size_t)n * h);
    mm_nn(dY.data(), wd, dAct.data(), n, Fe, h);                 // dact = dY Wd_e
    mm_tn(dY.data(), Act.data(), dWd + (size_t)e * h * Fe, h, Fe, n);  // dWd_e = dY^T act
    swiglu_bwd(G.data(), U.data(), dAct.data(), (size_t)n * Fe, dG.data(), dU.data());
    mm_nn(dG.data(), wg, dX.data(), n, h, Fe);                   // dX = dG Wg_e + dU Wu_e
    mm_nn(dU.data(), wg + (size_t)Fe * h, tmp.data(), n, h, Fe);
    for (size_t i = 0; i < (size_t)n * h; ++i) dX[i] += tmp[i];
    S* dwg = dWgu + (size_t)e * 2 * Fe * h;
    mm_tn(dG.data(), X.data(), dwg, Fe, h, n);                   // dWg_e = dG^T X
    mm_tn(dU.data(), X.data(), dwg + (size_t)Fe * h, Fe, h, n);  // dWu_e = dU^T X
    for (int i = 0; i < n; ++i)
      for (int c = 0; c < h; ++c) dm[(size_t)(R[i] / k) * h + c] += dX[(size_t)i * h + c];
  }
  // w_j = p_{e_j} / P with P = sum_i p_{e_i}:  dL/dp_{e_i} = (dw_i - sum_j w_j dw_j) / P
  // for selected experts, 0 for the rest; then through the softmax,
  // dr_e = p_e (dp_e - sum_f p_f dp_f).
  std::vector<S> dr((size_t)T * E), dp(E);
  for (int t = 0; t < T; ++t) {
    const S* pt = &A.p[(size_t)t * E];
    const int32_t* st = &A.sel[(size_t)t * k];
    const S* wt = &A.w[(size_t)t * k];
    const S* dwt = &dw[(size_t)t * k];
    S psel = 0, wdw = 0;
    for (int j = 0; j < k; ++j) {
      psel += pt[st[j]];
      wdw += wt[j] * dwt[j];
    }
    for (int e = 0; e < E; ++e) dp[e] = 0;
    for (int j = 0; j < k; ++j) dp[st[j]] = (dwt[j] - wdw) / psel;
    S pdp = 0;
    for (int e = 0; e < E; ++e) pdp += pt[e] * dp[e];
    for (int e = 0; e < E; ++e) dr[(size_t)t * E + e] = pt[e] * (dp[e] - pdp);
  }
  std::vector<S> dmr((size_t)T * h);
  mm_nn(dr.data(), Wr, dmr.data(), T, h, E);  // dm += dr Wr
  for (size_t i = 0; i < (size_t)T * h; ++i) dm[i] += dmr[i];
  mm_tn(dr.data(), m, dWr, E, h, T);          // dWr = dr^T m
}

// ---------------------------------------------------------------------------
// The whole step. P and G index the packed fp32 layout in elements
// (byte offset / 4). G is fully written.
// ---------------------------------------------------------------------------
template <class S>
struct LayerAct {
  std::vector<S> x, a, rstd1, q, k, v, P, o, hmid, m, rstd2, g, u, act;
  MoeAct<S> moe;
};

template <class S>
S forward_backward(const Dims& D, const S* P, const int32_t* tok, const int32_t* lab, int B, int Sq, S scale,
                   S* G, float* tok_loss = nullptr, const int32_t* route_in = nullptr,
                   int32_t* route_out = nullptr, float* logits_out = nullptr) {
  const int T = B * Sq, h = D.h, qd = D.nq * D.d, kd = D.nkv * D.d, F = D.F, V = D.V;
  auto off = [&](int unit, int t) { return layout_offset(D, 4, unit, t) / 4; };
  const size_t total = layout_offset(D, 4, D.L + 2, 0) / 4;
  for (size_t i = 0; i < total; ++i) G[i] = 0;

  // Stage 1: h_0 = Embed(x)
  std::vector<S> hcur((size_t)T * h);
  const S* E = P + off(0, 0);
  for (int t = 0; t < T; ++t)
    for (int j = 0; j < h; ++j) hcur[(size_t)t * h + j] = E[(size_t)tok[t] * h + j];

  std::vector<LayerAct<S>> acts(D.L);
  std::vector<S> tmp((size_t)T * std::max(h, F));
  for (int l = 0; l < D.L; ++l) {
    const int u = l + 1;
    LayerAct<S>& A = acts[l];
    A.x = hcur;
    A.a.resize((size_t)T * h); A.rstd1.resize(T);
    rmsnorm_fwd(A.x.data(), P + off(u, 0), T, h, D.eps, A.a.data(), A.rstd1.data());
    A.q.resize((size_t)T * qd); A.k.resize((size_t)T * kd); A.v.resize((size_t)T * kd);
    mm_nt(A.a.data(), P + off(u, 1), A.q.data(), T, qd, h);
    mm_nt(A.a.data(), P + off(u, 2), A.k.data(), T, kd, h);
    mm_nt(A.a.data(), P + off(u, 3), A.v.data(), T, kd, h);
    rope(A.q.data(), B, Sq, D.nq, D.d, D.theta, +1);
    rope(A.k.data(), B, Sq, D.nkv, D.d, D.theta, +1);
    A.P.resize((size_t)B * D.nq * Sq * Sq); A.o.resize((size_t)T * qd);
    attn_fwd(A.q.data(), A.k.data(), A.v.data(), B, Sq, D.nq, D.nkv, D.d, A.o.data(), A.P.data(), (S*)nullptr);
    A.hmid = A.x;
    mm_nt(A.o.data(), P + off(u, 4), tmp.data(), T, h, qd);
    for (size_t i = 0; i < (size_t)T * h; ++i) A.hmid[i] += tmp[i];
    A.m.resize((size_t)T * h); A.rstd2.resize(T);
    rmsnorm_fwd(A.hmid.data(), P + off(u, 5), T, h, D.eps, A.m.data(), A.rstd2.data());
    if (D.E > 0) {
      const size_t rs = (size_t)T * D.topk;
      moe_fwd(D, A.m.data(), P + off(u, 6), P + off(u, 7), P + off(u, 8), T, route_in ? route_in + l * rs : nullptr,
              route_out ? route_out + l * rs : nullptr, A.moe, tmp.data(),
              logits_out ? logits_out + (size_t)l * T * D.E : nullptr);
      hcur = A.hmid;
      for (size_t i = 0; i < (size_t)T * h; ++i) hcur[i] += tmp[i];
      continue;
    }
    A.g.resize((size_t)T * F); A.u.resize((size_t)T * F); A.act.resize((size_t)T * F);
    mm_nt(A.m.data(), P + off(u, 6), A.g.data(), T, F, h);
    mm_nt(A.m.data(), P + off(u, 7), A.u.data(), T, F, h);
    swiglu_fwd(A.g.data(), A.u.data(), (size_t)T * F, A.act.data());
    hcur = A.hmid;
    mm_nt(A.act.data(), P + off(u, 8), tmp.data(), T, h, F);
    for (size_t i = 0; i < (size_t)T * h; ++i) hcur[i] += tmp[i];
  }

  // Stage 2: loss anchor. z_in = RMSNorm(h_L; w_f); logits = z_in W_out^T.
  const int hu = D.L + 1;
  std::vector<S> zin((size_t)T * h), rstdf(T), logits((size_t)T * V), dz((size_t)T * V);
  rmsnorm_fwd(hcur.data(), P + off(hu, 0), T, h, D.eps, zin.data(), rstdf.data());
  mm_nt(zin.data(), P + off(hu, 1), logits.data(), T, V, h);
  const S loss = ce_fwd_bwd(logits.data(), lab, T, V, scale, dz.data(), tok_loss);
  mm_tn(dz.data(), zin.data(), G + off(hu, 1), V, h, T);  // dW_out = dz^T z_in
  std::vector<S> dzin((size_t)T * h), dh((size_t)T * h);
  mm_nn(dz.data(), P + off(hu, 1), dzin.data(), T, h, V);  // dz_in = dz W_out
  rmsnorm_bwd(hcur.data(), P + off(hu, 0), rstdf.data(), dzin.data(), T, h, dh.data(), G + off(hu, 0));

  // Stage 3: layer backward, top to bottom.
  std::vector<S> dact((size_t)T * F), dg((size_t)T * F), du((size_t)T * F), dm((size_t)T * h), dhmid((size_t)T * h);
  std::vector<S> dout((size_t)T * qd), dq((size_t)T * qd), dk((size_t)T * kd), dv((size_t)T * kd), da((size_t)T * h);
  for (int l = D.L - 1; l >= 0; --l) {
    const int u = l + 1;
    LayerAct<S>& A = acts[l];
    if (D.E > 0) {
      moe_bwd(D, A.m.data(), P + off(u, 6), P + off(u, 7), P + off(u, 8), T, A.moe, dh.data(), dm.data(),
              G + off(u, 6), G + off(u, 7), G + off(u, 8));
    } else {
      // h_out = h_mid + act Wd^T
      mm_nn(dh.data(), P + off(u, 8), dact.data(), T, F, h);
      mm_tn(dh.data(), A.act.data(), G + off(u, 8), h, F, T);
      swiglu_bwd(A.g.data(), A.u.data(), dact.data(), (size_t)T * F, dg.data(), du.data());
      mm_nn(dg.data(), P + off(u, 6), dm.data(), T, h, F);
      mm_nn(du.data(), P + off(u, 7), tmp.data(), T, h, F);
      for (size_t i = 0; i < (size_t)T * h; ++i) dm[i] += tmp[i];
      mm_tn(dg.data(), A.m.data(), G + off(u, 6), F, h, T);
      mm_tn(du.data(), A.m.data(), G + off(u, 7), F, h, T);
    }
    rmsnorm_bwd(A.hmid.data(), P + off(u, 5), A.rstd2.data(), dm.data(), T, h, dhmid.data(), G + off(u, 5));
    for (size_t i = 0; i < (size_t)T * h; ++i) dhmid[i] += dh[i];
    // h_mid = x + o Wo^T
    mm_nn(dhmid.data(), P + off(u, 4), dout.data(), T, qd, h);
    mm_tn(dhmid.data(), A.o.data(), G + off(u, 4), h, qd, T);
    attn_bwd(A.q.data(), A.k.data(), A.v.data(), A.P.data(), dout.data(), B, Sq, D.nq, D.nkv, D.d, dq.data(),
             dk.data(), dv.data());
    rope(dq.data(), B, Sq, D.nq, D.d, D.theta, -1);
    rope(dk.data(), B, Sq, D.nkv, D.d, D.theta, -1);
    mm_nn(dq.data(), P + off(u, 1), da.data(), T, h, qd);
    mm_nn(dk.data(), P + off(u, 2), tmp.data(), T, h, kd);
    for (size_t i = 0; i < (size_t)T * h; ++i) da[i] += tmp[i];
    mm_nn(dv.data(), P + off(u, 3), tmp.data(), T, h, kd);
    for (size_t i = 0; i < (size_t)T * h; ++i) da[i] += tmp[i];
    mm_tn(dq.data(), A.a.data(), G + off(u, 1), qd, h, T);
    mm_tn(dk.data(), A.a.data(), G + off(u, 2), kd, h, T);
    mm_tn(dv.data(), A.a.data(), G + off(u, 3), kd, h, T);
    rmsnorm_bwd(A.x.data(), P + off(u, 0), A.rstd1.data(), da.data(), T, h, dh.data(), G + off(u, 0));
    for (size_t i = 0; i < (size_t)T * h; ++i) dh[i] += dhmid[i];
    acts[l] = LayerAct<S>();  // release
  }
  // Embedding: dE[tok[t]] += dh_0[t]
  S* dE = G + off(0, 0);
  for (int t = 0; t < T; ++t)
    for (int j = 0; j < h; ++j) dE[(size_t)tok[t] * h + j] += dh[(size_t)t * h + j];
  return loss;
}

float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

bool valid_dims(const Dims& D) {
  const bool ffn = D.E == 0 ? (D.F >= 1 && D.topk == 0 && D.Fe == 0)
                            : (D.E >= 1 && D.topk >= 1 && D.topk <= D.E && D.Fe >= 1);
  return D.L >= 1 && D.h >= 1 && D.nq >= 1 && D.nkv >= 1 && D.nq % D.nkv == 0 && D.d >= 2 && D.d % 2 == 0 &&
         D.V >= 1 && D.E >= 0 && ffn;
}

// A forced routing [L][T][k] must name k distinct experts per position.
bool valid_routing(const Dims& D, const int32_t* route, int T) {
  if (!route) return true;
  if (D.E == 0) return false;
  for (size_t r = 0; r < (size_t)D.L * T; ++r) {
    const int32_t* st = route + r * D.topk;
    for (int j = 0; j < D.topk; ++j) {
      if (st[j] < 0 || st[j] >= D.E) return false;
      for (int i = 0; i < j; ++i)
        if (st[i] == st[j]) return false;
    }
  }
  return true;
}

}  // namespace

// ===========================================================================
// C interface (ctypes). Status: 0 ok, -1 bad argument.
// ===========================================================================
extern "C" {

typedef struct {
  int32_t n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn_dim, vocab;
  double rope_theta, norm_eps;
  int32_t n_experts, top_k, expert_ffn;  // all 0: dense SwiGLU FFN
} oracle_cfg;

static Dims to_dims(const oracle_cfg* c) {
  return Dims{c->n_layers, c->hidden, c->n_heads,   c->n_kv_heads, c->head_dim,  c->ffn_dim,
              c->vocab,    c->rope_theta, c->norm_eps, c->n_experts, c->top_k, c->expert_ffn};
}

// dtype: 0 = fp32, 1 = bf16
size_t oracle_packed_bytes(const oracle_cfg* c, int dtype) {
  const Dims D = to_dims(c);
  return layout_offset(D, dtype == 1 ? 2 : 4, D.L + 2, 0);
}

int oracle_tensor_offset(const oracle_cfg* c, int dtype, int unit, int tensor, size_t* off, size_t* bytes) {
  const Dims D = to_dims(c);
  if (unit < 0 || unit > D.L + 1 || tensor < 0 || tensor >= unit_tensor_count(D, unit)) return -1;
  const size_t esz = dtype == 1 ? 2 : 4;
  *off = layout_offset(D, esz, unit, tensor);
  *bytes = tensor_elems(D, unit, tensor) * esz;
  return 0;
}

static int check_tokens(const Dims& D, const int32_t* tok, const int32_t* lab, int T) {
  for (int t = 0; t < T; ++t)
    if (tok[t] < 0 || tok[t] >= D.V || lab[t] < 0 || lab[t] >= D.V) return -1;
  return 0;
}

// One step in fp32. params: packed host layout of dtype (0 fp32, 1 bf16).
// grads: packed fp32 layout, fully overwritten. loss: scale * sum_t CE_t.
// token_losses (optional, [B*S]): the unscaled CE term of every position.
// Mixture-of-experts layers: route_in (optional, [L][B*S][top_k]) forces the
// selected experts of every layer and position; route_out (optional, same
// shape) receives the selection used; router_logits (optional,
// [L][B*S][n_experts]) receives every layer's router logits.
int oracle_forward_backward_f32(const oracle_cfg* c, const void* params, int dtype, const int32_t* tokens,
                                const int32_t* labels, int B, int S, double scale, float* grads, double* loss,
                                float* token_losses, const int32_t* route_in, int32_t* route_out,
                                float* router_logits) {
  const Dims D = to_dims(c);
  if (!valid_dims(D) || B < 1 || S < 1 || check_tokens(D, tokens, labels, B * S)) return -1;
  if (!valid_routing(D, route_in, B * S) || ((route_out || router_logits) && D.E == 0)) return -1;
  const size_t n32 = layout_offset(D, 4, D.L + 2, 0) / 4;
  std::vector<float> P(n32, 0.f);
  if (dtype == 0) {
    std::memcpy(P.data(), params, n32 * 4);
  } else {
    // Same tensors in the bf16 layout, widened exactly to fp32.
    const uint8_t* src = (const uint8_t*)params;
    for (int u = 0; u <= D.L + 1; ++u)
      for (int t = 0; t < unit_tensor_count(D, u); ++t) {
        const size_t o16 = layout_offset(D, 2, u, t), o32 = layout_offset(D, 4, u, t) / 4;
        const uint16_t* s = (const uint16_t*)(src + o16);
        for (size_t i = 0; i < tensor_elems(D, u, t); ++i) P[o32 + i] = bf16_to_f32(s[i]);
      }
  }
  *loss = forward_backward<float>(D, P.data(), tokens, labels, B, S, (float)scale, grads, token_losses, route_in,
                                  route_out, router_logits);
  return 0;
}

// One step in fp64; params and grads are doubles at the fp32 layout's element
// offsets (byte offset / 4).
int oracle_forward_backward_f64(const oracle_cfg* c, const double* params, const int32_t* tokens,
                                const int32_t* labels, int B, int S, double scale, double* grads, double* loss,
                                const int32_t* route_in, int32_t* route_out) {
  const Dims D = to_dims(c);
  if (!valid_dims(D) || B < 1 || S < 1 || check_tokens(D, tokens, labels, B * S)) return -1;
  if (!valid_routing(D, route_in, B * S) || (route_out && D.E == 0)) return -1;
  *loss = forward_backward<double>(D, params, tokens, labels, B, S, scale, grads, nullptr, route_in, route_out);
  return 0;
}

}  // extern "C"

// ---- single operations (float in/out; acc selects float or double math) ----
#define ORACLE_DISPATCH(acc, FN_F, FN_D) \
  do {                                    \
    if (acc) { FN_D; } else { FN_F; }     \
  } while (0)

template <class S>
static std::vector<S> widen(const float* p, size_t n) {
  return std::vector<S>(p, p + n);
}
template <class S>
static void narrow(const std::vector<S>& v, float* p) {
  for (size_t i = 0; i < v.size(); ++i) p[i] = (float)v[i];
}
template <class S>
static void op_matmul(int mode, const float* A, const float* Bm, float* Y, int M, int N, int K) {
  // mode 0: Y = A[M,K] B[N,K]^T; 1: Y = A[M,K] B[K,N]; 2: Y = A[K,M]^T B[K,N]
  const size_t na = (size_t)M * K, nb = (size_t)N * K;
  auto a = widen<S>(A, na), b = widen<S>(Bm, nb);
  std::vector<S> y((size_t)M * N);
  if (mode == 0) mm_nt(a.data(), b.data(), y.data(), M, N, K);
  else if (mode == 1) mm_nn(a.data(), b.data(), y.data(), M, N, K);
  else mm_tn(a.data(), b.data(), y.data(), M, N, K);
  narrow(y, Y);
}
extern "C" {

int oracle_matmul(int mode, int use_f64, const float* A, const float* B, float* Y, int M, int N, int K) {
  if (mode < 0 || mode > 2 || M < 0 || N < 0 || K < 0) return -1;
  ORACLE_DISPATCH(use_f64, (op_matmul<float>(mode, A, B, Y, M, N, K)), (op_matmul<double>(mode, A, B, Y, M, N, K)));
  return 0;
}

// Selected elements of Y = A[M,K] B[N,K]^T (or mode 1/2 as above), one dot
// product each in double: for checking large products element by element.
int oracle_matmul_sampled(int mode, const float* A, const float* Bm, int M, int N, int K, const int64_t* rows,
                          const int64_t* cols, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) {
    const int64_t r = rows[i], c = cols[i];
    if (r < 0 || r >= M || c < 0 || c >= N) return -1;
    double s = 0;
    for (int k = 0; k < K; ++k) {
      double a, b;
      if (mode == 0) { a = A[(size_t)r * K + k]; b = Bm[(size_t)c * K + k]; }
      else if (mode == 1) { a = A[(size_t)r * K + k]; b = Bm[(size_t)k * N + c]; }
      else { a = A[(size_t)k * M + r]; b = Bm[(size_t)k * N + c]; }
      s += a * b;
    }
    out[i] = s;
  }
  return 0;
}

}  // extern "C"
template <class S>
static void op_rmsnorm_fwd(const float* x, const float* w, int T, int h, double eps, float* y, float* rstd) {
  auto X = widen<S>(x, (size_t)T * h), W = widen<S>(w, h);
  std::vector<S> Y((size_t)T * h), R(T);
  rmsnorm_fwd(X.data(), W.data(), T, h, eps, Y.data(), R.data());
  narrow(Y, y);
  if (rstd) narrow(R, rstd);
}
extern "C" {
int oracle_rmsnorm_fwd(int use_f64, const float* x, const float* w, int T, int h, double eps, float* y, float* rstd) {
  ORACLE_DISPATCH(use_f64, (op_rmsnorm_fwd<float>(x, w, T, h, eps, y, rstd)),
                  (op_rmsnorm_fwd<double>(x, w, T, h, eps, y, rstd)));
  return 0;
}

}  // extern "C"
template <class S>
static void op_rmsnorm_bwd(const float* x, const float* w, const float* dy, int T, int h, double eps, float* dx,
                           float* dw) {
  auto X = widen<S>(x, (size_t)T * h), W = widen<S>(w, h), DY = widen<S>(dy, (size_t)T * h);
  std::vector<S> Y((size_t)T * h), R(T), DX((size_t)T * h), DW(h, S(0));
  rmsnorm_fwd(X.data(), W.data(), T, h, eps, Y.data(), R.data());
  rmsnorm_bwd(X.data(), W.data(), R.data(), DY.data(), T, h, DX.data(), DW.data());
  narrow(DX, dx);
  narrow(DW, dw);
}
extern "C" {
int oracle_rmsnorm_bwd(int use_f64, const float* x, const float* w, const float* dy, int T, int h, double eps,
                       float* dx, float* dw) {
  ORACLE_DISPATCH(use_f64, (op_rmsnorm_bwd<float>(x, w, dy, T, h, eps, dx, dw)),
                  (op_rmsnorm_bwd<double>(x, w, dy, T, h, eps, dx, dw)));
  return 0;
}

// In-place RoPE on x [B*S, nh, d]; dir +1 forward, -1 backward.
int oracle_rope(int use_f64, float* x, int B, int S, int nh, int d, double theta, int dir) {
  if (d % 2 || (dir != 1 && dir != -1)) return -1;
  const size_t n = (size_t)B * S * nh * d;
  if (use_f64) {
    auto X = widen<double>(x, n);
    rope(X.data(), B, S, nh, d, theta, dir);
    narrow(X, x);
  } else {
    rope(x, B, S, nh, d, theta, dir);
  }
  return 0;
}

}  // extern "C"
template <class S>
static void op_attn(const float* q, const float* k, const float* v, const float* dout, int B, int Sq, int nq, int nkv,
                    int d, float* o, float* lse, float* dq, float* dk, float* dv) {
  const size_t nqe = (size_t)B * Sq * nq * d, nke = (size_t)B * Sq * nkv * d;
  auto Q = widen<S>(q, nqe), K = widen<S>(k, nke), V = widen<S>(v, nke);
  std::vector<S> O(nqe), P((size_t)B * nq * Sq * Sq), L((size_t)B * nq * Sq);
  attn_fwd(Q.data(), K.data(), V.data(), B, Sq, nq, nkv, d, O.data(), P.data(), L.data());
  if (o) narrow(O, o);
  if (lse) narrow(L, lse);
  if (dout) {
    auto DO = widen<S>(dout, nqe);
    std::vector<S> DQ(nqe), DK(nke), DV(nke);
    attn_bwd(Q.data(), K.data(), V.data(), P.data(), DO.data(), B, Sq, nq, nkv, d, DQ.data(), DK.data(), DV.data());
    narrow(DQ, dq);
    narrow(DK, dk);
    narrow(DV, dv);
  }
}
extern "C" {
// Causal GQA attention on q [B*S,nq,d], k/v [B*S,nkv,d]. o, lse ([B,nq,S]) optional;
// if dout is given, dq/dk/dv are written.
int oracle_attention(int use_f64, const float* q, const float* k, const float* v, const float* dout, int B, int S,
                     int nq, int nkv, int d, float* o, float* lse, float* dq, float* dk, float* dv) {
  if (nq % nkv) return -1;
  ORACLE_DISPATCH(use_f64, (op_attn<float>(q, k, v, dout, B, S, nq, nkv, d, o, lse, dq, dk, dv)),
                  (op_attn<double>(q, k, v, dout, B, S, nq, nkv, d, o, lse, dq, dk, dv)));
  return 0;
}

int oracle_swiglu(int use_f64, const float* g, const float* u, const float* da, size_t n, float* a, float* dg,
                  float* du) {
  if (use_f64) {
    auto G = widen<double>(g, n), U = widen<double>(u, n);
    std::vector<double> A(n);
    swiglu_fwd(G.data(), U.data(), n, A.data());
    if (a) narrow(A, a);
    if (da) {
      auto DA = widen<double>(da, n);
      std::vector<double> DG(n), DU(n);
      swiglu_bwd(G.data(), U.data(), DA.data(), n, DG.data(), DU.data());
      narrow(DG, dg);
      narrow(DU, du);
    }
  } else {
    if (a) swiglu_fwd(g, u, n, a);
    if (da) swiglu_bwd(g, u, da, n, dg, du);
  }
  return 0;
}

}  // extern "C"
template <class S>
static void op_moe(const float* m, const float* Wr, const float* Wgu, const float* Wd, int T, const Dims& D,
                   const int32_t* route_in, int32_t* route_out, float* out, const float* dout, float* dm, float* dWr,
                   float* dWgu, float* dWd) {
  const size_t h = D.h, E = D.E, Fe = D.Fe;
  auto M = widen<S>(m, T * h), R = widen<S>(Wr, E * h), GU = widen<S>(Wgu, E * 2 * Fe * h),
       WD = widen<S>(Wd, E * h * Fe);
  MoeAct<S> A;
  std::vector<S> O(T * h);
  moe_fwd(D, M.data(), R.data(), GU.data(), WD.data(), T, route_in, route_out, A, O.data());
  narrow(O, out);
  if (dout) {
    auto DO = widen<S>(dout, T * h);
    std::vector<S> DM(T * h), DR(E * h), DGU(E * 2 * Fe * h), DD(E * h * Fe);
    moe_bwd(D, M.data(), R.data(), GU.data(), WD.data(), T, A, DO.data(), DM.data(), DR.data(), DGU.data(),
            DD.data());
    narrow(DM, dm);
    narrow(DR, dWr);
    narrow(DGU, dWgu);
    narrow(DD, dWd);
  }
}
extern "C" {
// Mixture-of-experts FFN on m [T,h] with router Wr [E,h], experts' gate|up
// Wgu [E,2Fe,h] and down Wd [E,h,Fe]: out [T,h]; route_in (optional, [T,k])
// forces the selection, route_out (optional) receives it; if dout is given,
// dm, dWr, dWgu, dWd are written.
int oracle_moe_ffn(int use_f64, const float* m, const float* Wr, const float* Wgu, const float* Wd, int T, int h,
                   int E, int k, int Fe, const int32_t* route_in, int32_t* route_out, float* out, const float* dout,
                   float* dm, float* dWr, float* dWgu, float* dWd) {
  Dims D{1, h, 1, 1, 2, 0, 1, 1e4, 1e-5, E, k, Fe};
  if (T < 0 || h < 1 || !valid_dims(D) || !valid_routing(D, route_in, T)) return -1;
  ORACLE_DISPATCH(use_f64,
                  (op_moe<float>(m, Wr, Wgu, Wd, T, D, route_in, route_out, out, dout, dm, dWr, dWgu, dWd)),
                  (op_moe<double>(m, Wr, Wgu, Wd, T, D, route_in, route_out, out, dout, dm, dWr, dWgu, dWd)));
  return 0;
}

// Cross-entropy on logits [T,V]; returns the loss in *loss, dz optional.
int oracle_cross_entropy(int use_f64, const float* z, const int32_t* labels, int T, int V, double scale,
                         double* loss, float* dz) {
  for (int t = 0; t < T; ++t)
    if (labels[t] < 0 || labels[t] >= V) return -1;
  if (use_f64) {
    auto Z = widen<double>(z, (size_t)T * V);
    std::vector<double> DZ(dz ? (size_t)T * V : 0);
    *loss = ce_fwd_bwd(Z.data(), labels, T, V, scale, dz ? DZ.data() : nullptr);
    if (dz) narrow(DZ, dz);
  } else {
    *loss = ce_fwd_bwd(z, labels, T, V, (float)scale, dz);
  }
  return 0;
}

}  // extern "C"
