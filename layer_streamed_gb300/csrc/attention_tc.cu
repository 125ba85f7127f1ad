// Causal GQA flash attention on the 5th-generation tensor cores.
//
// Forward (one CTA per (128-row query tile, query head, sequence)): Q stays
// in shared memory, K/V tiles stream through a two-stage TMA ring;
// S = Q K^T lands in tensor memory (two S buffers so the next product
// overlaps this tile's softmax), the softmax warps (one thread per query
// row) apply the causal mask and the online-softmax update, write P as bf16
// into shared memory in the MMA operand layout, and O += P V accumulates in
// tensor memory. The running maximum is only moved (and O rescaled) when it
// grows by more than 2^8, which keeps every exponent bounded while skipping
// most rescales; the final O / l and log-sum-exp use the same reference, so
// the result is exact up to rounding.
//
// Backward: delta = rowsum(dO * O) first; then one pass per 128-row KV tile
// (all query heads of its group, all query tiles at or after it) computes
// S^T = K Q^T and dP^T = V dO^T, P^T = exp(S^T - lse), dS^T = P^T (dP^T -
// delta), and accumulates dV += P^T dO, dK += dS^T Q in tensor memory; a
// separate pass per query tile accumulates dQ += dS K. Each output row is
// produced by one CTA with a fixed loop order: deterministic.
//
// Operand layouts (128-byte swizzle, 1024-byte aligned tiles):
//  Q/K/V/dO tiles come from TMA as [128 rows][64 head-dim] boxes (head dims
//  below 64 are zero-filled by TMA), which is K-major for Q K^T-type
//  products and MN-major for P V-type products. P / dS tiles are written by
//  the softmax threads as [128 rows][128] K-major (two 64-column blocks).
#include "common.cuh"
#include "kernels.h"

namespace mt {

MT_DEVICE_ERROR_READER(attention_tc_take_device_error)
MT_DEVICE_ERROR_PEEKER(attention_tc_peek_device_error)

namespace {

constexpr int TILE = 128;
constexpr int BOX = 128 * 64 * 2;  // one [128 rows][64] bf16 box = 16 KB

// ---- small device helpers --------------------------------------------------
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z,
                                            int w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];" ::"r"(smem_u32(dst)),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
      : "memory");
}

// Load a [128 rows][D] tile of one head (D/64 boxes, at least one).
template <int D>
__device__ __forceinline__ void load_head_tile(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int head,
                                               int row0, int b) {
#pragma unroll
  for (int i = 0; i < (D + 63) / 64; ++i) tma_load_4d(dst + i * BOX, map, bar, i * 64, head, row0, b);
}
template <int D>
constexpr uint32_t tile_bytes() {
  return ((D + 63) / 64) * BOX;
}

// K-major A/B descriptor of the k-th 16-wide step of a [128][64*n] tile.
__device__ __forceinline__ uint64_t kmaj_desc(const uint8_t* tile, int kk) {
  return make_sdesc(smem_u32(tile) + (kk >> 2) * BOX + (kk & 3) * 32, 16, 1024);
}
// MN-major B descriptor (N = head dim, K = rows) of the k-th 16-row step.
__device__ __forceinline__ uint64_t mnmaj_desc(const uint8_t* tile, int kk) {
  return make_sdesc(smem_u32(tile) + kk * 2048, BOX, 1024);
}

__device__ __forceinline__ void store_row_bf16(uint16_t* dst, const uint32_t (&r)[32], int n, float mul) {
  // n valid columns (<= 32); dst 16-byte aligned when n == 32
  if (n == 32) {
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      uint4 w;
      w.x = pack_bf2(__uint_as_float(r[8 * v + 0]) * mul, __uint_as_float(r[8 * v + 1]) * mul);
      w.y = pack_bf2(__uint_as_float(r[8 * v + 2]) * mul, __uint_as_float(r[8 * v + 3]) * mul);
      w.z = pack_bf2(__uint_as_float(r[8 * v + 4]) * mul, __uint_as_float(r[8 * v + 5]) * mul);
      w.w = pack_bf2(__uint_as_float(r[8 * v + 6]) * mul, __uint_as_float(r[8 * v + 7]) * mul);
      ((uint4*)dst)[v] = w;
    }
  } else {
#pragma unroll
    for (int v = 0; v < 2; ++v) {  // n == 16
      uint4 w;
      w.x = pack_bf2(__uint_as_float(r[8 * v + 0]) * mul, __uint_as_float(r[8 * v + 1]) * mul);
      w.y = pack_bf2(__uint_as_float(r[8 * v + 2]) * mul, __uint_as_float(r[8 * v + 3]) * mul);
      w.z = pack_bf2(__uint_as_float(r[8 * v + 4]) * mul, __uint_as_float(r[8 * v + 5]) * mul);
      w.w = pack_bf2(__uint_as_float(r[8 * v + 6]) * mul, __uint_as_float(r[8 * v + 7]) * mul);
      ((uint4*)dst)[v] = w;
    }
  }
}

struct AttnArgs {
  uint16_t* o;       // fwd output / unused
  float* lse;        // [B, nq, S] natural log
  const float* lse_in;
  const float* delta;  // backward: [B, nq, pad128(S)] (see the delta kernel)
  const float* lse2;   // backward: [B, nq, pad128(S)] log-sum-exp in log2 units
  uint16_t *dq, *dk, *dv;
  int B, S, nq, nkv, ldq, ldkv, ldo;
  float scale_log2;  // log2(e) / sqrt(d)
  float scale;       // 1 / sqrt(d)
  const float2* rope_tab;  // backward: rotate dq/dk back by RoPE (nullable), [S][d/2] (cos, sin)
};

// Store one row of a head-dim gradient (dq or dk) held in TMEM columns
// [tcol, tcol + D), scaled by mul, optionally rotated back by RoPE (the
// transpose of the forward rotation: (x1, x2) -> (x1 c + x2 s, -x1 s + x2 c)).
// part/nparts split the work between warpgroups (each call is warp-collective).
template <int D>
__device__ __forceinline__ void store_grad_row(uint16_t* orow, uint32_t tcol, bool row_ok, float mul,
                                               const float2* tab, int part, int nparts) {
  constexpr int NCH = (D + 31) / 32;
  if (!tab) {
#pragma unroll 1
    for (int c = part; c < NCH; c += nparts) {
      uint32_t v[32];
      __syncwarp();
      tmem_ld32(tcol + c * 32, v);
      tmem_ld_wait();
      if (row_ok) store_row_bf16(orow + c * 32, v, D < 32 ? D : 32, mul);
    }
    return;
  }
  if (D >= 64) {
    constexpr int P = D / 64;  // chunk distance between the halves of the head
#pragma unroll 1
    for (int c = part; c < P; c += nparts) {
      uint32_t va[32], vb[32];
      __syncwarp();
      tmem_ld32(tcol + c * 32, va);
      tmem_ld32(tcol + (c + P) * 32, vb);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float2 cs = tab[c * 32 + i];
        const float x1 = __uint_as_float(va[i]) * mul, x2 = __uint_as_float(vb[i]) * mul;
        va[i] = __float_as_uint(x1 * cs.x + x2 * cs.y);
        vb[i] = __float_as_uint(-x1 * cs.y + x2 * cs.x);
      }
      if (row_ok) {
        store_row_bf16(orow + c * 32, va, 32, 1.f);
        store_row_bf16(orow + (c + P) * 32, vb, 32, 1.f);
      }
    }
  } else if (part == 0) {  // D in {16, 32}: both halves in the first chunk
    uint32_t v[32];
    __syncwarp();
    tmem_ld32(tcol, v);
    tmem_ld_wait();
    constexpr int H = D / 2;
#pragma unroll
    for (int i = 0; i < H; ++i) {
      const float2 cs = tab[i];
      const float x1 = __uint_as_float(v[i]) * mul, x2 = __uint_as_float(v[i + H]) * mul;
      v[i] = __float_as_uint(x1 * cs.x + x2 * cs.y);
      v[i + H] = __float_as_uint(-x1 * cs.y + x2 * cs.x);
    }
    if (row_ok) store_row_bf16(orow, v, D, 1.f);
  }
}

constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// ===========================================================================
// Forward. CTA = two consecutive 128-row query tiles (A = 2m, B = 2m+1) of
// one query head and sequence; 12 warps: warp 0 TMA, warp 1 MMA issue,
// warps 4-7 softmax of tile A, warps 8-11 softmax of tile B (warps 2-3 idle).
// The MMA thread alternates between the tiles (PV_A(t), S_A(t+1), PV_B(t),
// S_B(t+1)), so each softmax warpgroup works while the tensor core serves
// the other tile. TMEM: S_A +0, S_B +128, O_A +256, O_B +384; the softmax
// writes P (bf16 pairs) over the first 64 columns of its S, and the PV
// product reads it from there as its A operand (the next S product of that
// tile is issued after the PV product, and tensor-core operations of one
// thread run in issue order). Shared: Q_A, Q_B, K and V in two stages each.
// ===========================================================================
template <int D>
struct FwdSmem {
  static constexpr int QA = 0;
  static constexpr int QB = QA + tile_bytes<D>();
  static constexpr int K0 = QB + tile_bytes<D>();
  static constexpr int V0 = K0 + 2 * tile_bytes<D>();
  static constexpr int BAR = V0 + 2 * tile_bytes<D>();
  static constexpr int TOTAL = BAR + 256;
  static constexpr int ALLOC = (TOTAL + 1024 > 118 * 1024) ? TOTAL + 1024 : 118 * 1024;  // one CTA per SM
};

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D>
__global__ void __launch_bounds__(384, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                       const __grid_constant__ CUtensorMap tv, AttnArgs a) {
  using L = FwdSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(sm + L::BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;   // [2]
  uint64_t* k_empty = bars + 3;  // [2]
  uint64_t* v_full = bars + 5;   // [2]
  uint64_t* v_empty = bars + 7;  // [2]
  uint64_t* s_full = bars + 9;   // [2]: tile A, tile B
  uint64_t* p_full = bars + 11;  // [2]
  uint64_t* o_done = bars + 13;  // [2]
  uint32_t* tmem_slot = (uint32_t*)(bars + 15);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

  const int nqt = (a.S + TILE - 1) / TILE;
  const int npairs = (nqt + 1) / 2;
  // Blocks start roughly in linear order: the pair index is the slowest
  // coordinate, so every head's longest pairs start first (longest first
  // over the whole grid, which keeps the tail short).
  const int lin = (int)(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
  const int hb = lin % (a.nq * a.B);
  const int m = npairs - 1 - lin / (a.nq * a.B);
  const int j = hb % a.nq, b = hb / a.nq;
  const int g = j / (a.nq / a.nkv);
  const int tA = 2 * m + 1, tB = 2 * m + 2;  // KV tiles seen by tile A / tile B
  const uint32_t warp = warp_id(), lane = lane_id();

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);
      mbar_init(&o_done[i], 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      mbar_arrive_expect_tx(q_full, 2 * tile_bytes<D>());
      load_head_tile<D>(sm + L::QA, &tq, q_full, j, (2 * m) * TILE, b);
      load_head_tile<D>(sm + L::QB, &tq, q_full, j, (2 * m + 1) * TILE, b);
      for (int t = 0; t < tB; ++t) {
        const int st = t & 1;
        const uint32_t free_par = ((t >> 1) & 1) ^ 1;
        mbar_wait(&k_empty[st], free_par, abort_flag, kErrTimeoutAttn);
        mbar_arrive_expect_tx(&k_full[st], tile_bytes<D>());
        load_head_tile<D>(sm + L::K0 + st * tile_bytes<D>(), &tk, &k_full[st], g, t * TILE, b);
        mbar_wait(&v_empty[st], free_par, abort_flag, kErrTimeoutAttn);
        mbar_arrive_expect_tx(&v_full[st], tile_bytes<D>());
        load_head_tile<D>(sm + L::V0 + st * tile_bytes<D>(), &tv, &v_full[st], g, t * TILE, b);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t IDESC_S = make_idesc(128, 128, false, false);
      constexpr uint32_t IDESC_O = make_idesc(128, D < 64 ? 64 : D, false, true);  // padded head dims read zeros
      constexpr int KS = D / 16;
      auto issue_s = [&](int side, int t) {  // S_side(t) = Q_side K_t^T
        const uint8_t* q = sm + (side ? L::QB : L::QA);
        const uint8_t* kt = sm + L::K0 + (t & 1) * tile_bytes<D>();
#pragma unroll
        for (int kk = 0; kk < KS; ++kk)
          tc_mma(tmem + side * 128, kmaj_desc(q, kk), kmaj_desc(kt, kk), IDESC_S, kk > 0 ? 1u : 0u);
        tc_commit(&s_full[side]);
      };
      auto issue_pv = [&](int side, int t) {  // O_side += P_side(t) V_t, P from tensor memory
        const uint8_t* vt = sm + L::V0 + (t & 1) * tile_bytes<D>();
#pragma unroll
        for (int kk = 0; kk < TILE / 16; ++kk)
          tc_mma_ts(tmem + 256 + side * 128, tmem + side * 128 + kk * 8, mnmaj_desc(vt, kk), IDESC_O,
                    (t > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&o_done[side]);
      };
      mbar_wait(q_full, 0, abort_flag, kErrTimeoutAttn);
      mbar_wait(&k_full[0], 0, abort_flag, kErrTimeoutAttn);
      tc_fence_after();
      issue_s(0, 0);
      issue_s(1, 0);
      tc_commit(&k_empty[0]);
      for (int t = 0; t < tB; ++t) {
        const bool next = t + 1 < tB;
        // V(t) and K(t+1) are waited for here, while the softmax of tile A
        // still runs: between the products of one tile a wait would leave
        // the tensor core idle (its issue queue holds little work).
        mbar_wait(&v_full[t & 1], (t >> 1) & 1, abort_flag, kErrTimeoutAttn);
        if (next) mbar_wait(&k_full[(t + 1) & 1], ((t + 1) >> 1) & 1, abort_flag, kErrTimeoutAttn);
        if (t < tA) {
          mbar_wait(&p_full[0], t & 1, abort_flag, kErrTimeoutAttn);
          tc_fence_after();
          issue_pv(0, t);
          if (t + 1 < tA) issue_s(0, t + 1);
        }
        mbar_wait(&p_full[1], t & 1, abort_flag, kErrTimeoutAttn);
        tc_fence_after();
        issue_pv(1, t);
        tc_commit(&v_empty[t & 1]);
        if (next) {
          issue_s(1, t + 1);
          tc_commit(&k_empty[(t + 1) & 1]);
        }
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    // softmax / epilogue of one tile: thread owns query row r
    const int side = warp >= 8 ? 1 : 0;
    const int nt = side ? tB : tA;
    const uint32_t q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const int trow = (2 * m + side) * TILE + r;  // position in the sequence
    const uint32_t lane_base = (q4 * 32) << 16;
    const uint32_t s_col = tmem + lane_base + side * 128;
    const uint32_t o_col = tmem + lane_base + 256 + side * 128;
    float m_ref = -INFINITY, l = 0.f;
    for (int t = 0; t < nt; ++t) {
      mbar_wait(&s_full[side], t & 1, abort_flag, kErrTimeoutAttn);
      tc_fence_after();
      float sv[128];
      {
        uint32_t v0[32], v1[32], v2[32], v3[32];
        __syncwarp();
        tmem_ld32(s_col + 0, v0);
        tmem_ld32(s_col + 32, v1);
        tmem_ld32(s_col + 64, v2);
        tmem_ld32(s_col + 96, v3);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          sv[i] = __uint_as_float(v0[i]);
          sv[32 + i] = __uint_as_float(v1[i]);
          sv[64 + i] = __uint_as_float(v2[i]);
          sv[96 + i] = __uint_as_float(v3[i]);
        }
      }
      const int kv0 = t * TILE;
      if (t == nt - 1 || kv0 + TILE > a.S) {  // diagonal or sequence tail: mask
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (kv0 + i > trow || kv0 + i >= a.S) sv[i] = -INFINITY;
      }
      float mx8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx8[i] = sv[i];
#pragma unroll
      for (int i = 8; i < 128; ++i) mx8[i & 7] = fmaxf(mx8[i & 7], sv[i]);
      const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      const float m_new = mx * a.scale_log2;
      // The rescale touches O through warp-collective tensor-memory loads and
      // stores, so the decision is taken per warp: if any row of the warp
      // needs a new reference maximum, every row of the warp moves its
      // reference to max(m_new, m_ref) (alpha = 1 where nothing changes).
      if (__any_sync(0xffffffffu, m_new > m_ref + kRescaleThreshold) || t == 0) {
        const float m_use = fmaxf(m_new, m_ref);
        const float alpha = (m_ref == -INFINITY) ? 0.f : ex2_approx(m_ref - m_use);
        l *= alpha;
        if (t > 0) {
          // O may be touched only once the previous P V product is complete.
          // P needs no such wait: S(t) was issued after that product and the
          // tensor core runs one thread's operations in order.
          mbar_wait(&o_done[side], (t - 1) & 1, abort_flag, kErrTimeoutAttn);
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < (D + 31) / 32; ++c) {
            uint32_t v[32];
            __syncwarp();
            tmem_ld32(o_col + c * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
            tmem_st32(o_col + c * 32, v);
          }
        }
        m_ref = m_use;
      }
      // probabilities relative to m_ref (masked entries give 0), row sum,
      // and P as bf16 pairs over the first 64 columns of S
      float l8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float p0 = ex2_approx(fmaf(sv[64 * c + 2 * i], a.scale_log2, -m_ref));
          const float p1 = ex2_approx(fmaf(sv[64 * c + 2 * i + 1], a.scale_log2, -m_ref));
          l8[(2 * i) & 7] += p0;
          l8[(2 * i + 1) & 7] += p1;
          pk[i] = pack_bf2(p0, p1);
        }
        __syncwarp();
        tmem_st32(s_col + 32 * c, pk);
      }
      l += ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[side]);
    }
    // epilogue: O / l and the log-sum-exp
    mbar_wait(&o_done[side], (nt - 1) & 1, abort_flag, kErrTimeoutAttn);
    tc_fence_after();
    const bool row_ok = trow < a.S;
    const float inv_l = 1.f / l;
    uint16_t* orow = a.o + ((size_t)b * a.S + trow) * a.ldo + (size_t)j * D;
#pragma unroll 1
    for (int c = 0; c < (D + 31) / 32; ++c) {
      uint32_t v[32];
      __syncwarp();
      tmem_ld32(o_col + c * 32, v);
      tmem_ld_wait();
      if (row_ok) store_row_bf16(orow + c * 32, v, D < 32 ? D : 32, inv_l);
    }
    if (row_ok) a.lse[((size_t)b * a.nq + j) * a.S + trow] = (m_ref + log2f(l)) * kLn2;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ===========================================================================
// Backward. Both passes work on 128-row tiles of queries and keys, so every
// product is 128 wide (narrower tcgen05 products run well below the tensor
// core's rate). 12 warps: warp 0 TMA, warp 1 MMA issue, warps 4-7 and 8-11
// are two elementwise warpgroups that split the 128 columns of a tile
// (warpgroup A columns 0-63, B 64-127); thread = row of the 128-row tile.
// The elementwise warps write P^T and dS^T (or dS) as bf16 pairs over
// columns of their S and dP buffers that they have already read (see
// packed_col128), and the gradient products read them from tensor memory as
// their A operand; tensor-core operations of one thread run in issue order,
// so a later score product that overwrites those buffers follows the
// gradient products that read them.
//
// The delta kernel also writes, per (sequence, query head), the log-sum-exp
// in log2 units over S padded to a multiple of 128 (+inf on the padding, so
// padded query rows get probability 0) beside delta (0 on the padding).
// ===========================================================================
constexpr int kDkvStages = 2;  // Q / dO tiles in flight in the dK/dV pass

__host__ __device__ constexpr int pad128(int S) { return (S + 127) & ~127; }

// Untiled bulk copy global -> shared; both addresses 16-byte aligned, size a
// multiple of 16.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// 32 values of one row as 16 bf16 pairs into tensor-memory columns [col, col+16).
__device__ __forceinline__ void tmem_st_bf16x32(uint32_t col, const float (&v)[32]) {
  uint32_t pk[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) pk[i] = pack_bf2(v[2 * i], v[2 * i + 1]);
  tmem_st16(col, pk);
}

// K step kk (16 rows of the 128-wide loop dimension) of a packed bf16
// operand: warpgroup kk / 4 wrote its 64 columns as 32 pairs at the start of
// its own 64-column range (dQ pass).
__device__ __forceinline__ uint32_t packed_col128(int kk) { return (kk >> 2) * 64 + (kk & 3) * 8; }
// The same for the dK/dV pass, whose 32-column chunks alternate between the
// warpgroups: K step kk sits in chunk kk / 2, at +8 for its second 16 rows.
__device__ __forceinline__ uint32_t packed_col_dkv(int kk) { return (kk >> 1) * 32 + (kk & 1) * 8; }

// dK/dV pass: CTA = (128-row KV tile kt, KV head g, sequence b); loop over the
// query heads of the group and the 128-row query tiles at or after kt. Per
// step: S^T = K Q^T and dP^T = V dO^T, then P^T = exp2(S^T - lse), dS^T =
// P^T (dP^T - delta) by the elementwise warps, then dV += P^T dO and dK +=
// dS^T Q. TMEM: S^T +0 (P^T packed over it), dP^T +128 (dS^T packed over
// it), dV +256, dK +384: full, so the score products of step i+1 follow the
// gradient products of step i. The elementwise warps do the first 64
// queries of a step first (warpgroup w: columns 32w..32w+31), then the last
// 64 (64+32w..), and signal each half, so the gradient products of the first
// half run while the second is computed. Pairs of chunk (c, w) go over the
// first 16 of its own 32 columns: K step kk at packed_col_dkv(kk).
template <int D>
struct DkvSmem {
  static constexpr int K = 0;
  static constexpr int V = K + tile_bytes<D>();
  static constexpr int Q0 = V + tile_bytes<D>();                      // [kDkvStages] Q tiles
  static constexpr int DO0 = Q0 + kDkvStages * tile_bytes<D>();       // [kDkvStages] dO tiles
  static constexpr int LD0 = DO0 + kDkvStages * tile_bytes<D>();      // [kDkvStages] lse2[128], delta[128]
  static constexpr int BAR = LD0 + kDkvStages * 1024;
  static constexpr int TOTAL = BAR + 256;
  static constexpr int ALLOC = (TOTAL + 1024 > 118 * 1024) ? TOTAL + 1024 : 118 * 1024;
};

template <int D>
__global__ void __launch_bounds__(384, 1)
    attn_bwd_dkv_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                           const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                           AttnArgs a) {
  using L = DkvSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(sm + L::BAR);
  uint64_t* kv_full = bars + 0;
  uint64_t* qdo_full = bars + 1;                  // [kDkvStages]
  uint64_t* qdo_empty = bars + 1 + kDkvStages;    // [kDkvStages]
  uint64_t* s_full = bars + 1 + 2 * kDkvStages;   // S^T and dP^T of this step are in tensor memory
  uint64_t* p_full = bars + 2 + 2 * kDkvStages;   // [2] P^T and dS^T of the first / last 64 queries written
  uint64_t* pd_done = bars + 4 + 2 * kDkvStages;  // the last gradient products are complete
  uint32_t* tmem_slot = (uint32_t*)(bars + 5 + 2 * kDkvStages);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

  const int nqt = (a.S + TILE - 1) / TILE;
  // longest tiles (the first KV tiles see the most queries) first over the
  // whole grid: the tile index is the slowest coordinate of the linear order
  const int lin = (int)(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
  const int gb = lin % (a.nkv * a.B);
  const int kt = lin / (a.nkv * a.B);
  const int g = gb % a.nkv, b = gb / a.nkv;
  const int grp = a.nq / a.nkv;
  const int per_head = nqt - kt;  // query tiles at or after the KV tile
  const int iters = grp * per_head;
  const int Sp = pad128(a.S);
  const uint32_t warp = warp_id(), lane = lane_id();

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int i = 0; i < kDkvStages; ++i) {
      mbar_init(&qdo_full[i], 1);
      mbar_init(&qdo_empty[i], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(&p_full[0], 8);
    mbar_init(&p_full[1], 8);
    mbar_init(pd_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      prefetch_tmap(&tdo);
      mbar_arrive_expect_tx(kv_full, 2 * tile_bytes<D>());
      load_head_tile<D>(sm + L::K, &tk, kv_full, g, kt * TILE, b);
      load_head_tile<D>(sm + L::V, &tv, kv_full, g, kt * TILE, b);
      for (int it = 0; it < iters; ++it) {
        const int j = g * grp + it / per_head;
        const int qt = kt + it % per_head;
        const int st = it % kDkvStages;
        mbar_wait(&qdo_empty[st], ((it / kDkvStages) & 1) ^ 1, abort_flag, kErrTimeoutAttn);
        mbar_arrive_expect_tx(&qdo_full[st], 2 * tile_bytes<D>() + 1024);
        load_head_tile<D>(sm + L::Q0 + st * tile_bytes<D>(), &tq, &qdo_full[st], j, qt * TILE, b);
        load_head_tile<D>(sm + L::DO0 + st * tile_bytes<D>(), &tdo, &qdo_full[st], j, qt * TILE, b);
        const size_t ro = ((size_t)b * a.nq + j) * Sp + (size_t)qt * TILE;
        bulk_load(sm + L::LD0 + st * 1024, a.lse2 + ro, 512, &qdo_full[st]);
        bulk_load(sm + L::LD0 + st * 1024 + 512, a.delta + ro, 512, &qdo_full[st]);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t IDESC_S = make_idesc(128, 128, false, false);
      constexpr uint32_t IDESC_G = make_idesc(128, D < 64 ? 64 : D, false, true);
      constexpr int KS = D / 16;
      mbar_wait(kv_full, 0, abort_flag, kErrTimeoutAttn);
      for (int it = 0; it < iters; ++it) {
        const int st = it % kDkvStages;
        const uint8_t* q = sm + L::Q0 + st * tile_bytes<D>();
        const uint8_t* dout = sm + L::DO0 + st * tile_bytes<D>();
        mbar_wait(&qdo_full[st], (it / kDkvStages) & 1, abort_flag, kErrTimeoutAttn);
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < KS; ++kk)  // S^T = K Q^T
          tc_mma(tmem, kmaj_desc(sm + L::K, kk), kmaj_desc(q, kk), IDESC_S, kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < KS; ++kk)  // dP^T = V dO^T
          tc_mma(tmem + 128, kmaj_desc(sm + L::V, kk), kmaj_desc(dout, kk), IDESC_S, kk > 0 ? 1u : 0u);
        tc_commit(s_full);
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // the two 64-query halves, as the elementwise warps finish them
          mbar_wait(&p_full[h], it & 1, abort_flag, kErrTimeoutAttn);
          tc_fence_after();
#pragma unroll
          for (int kk = 4 * h; kk < 4 * h + 4; ++kk) {  // dV += P^T dO ; dK += dS^T Q  (A operands in TMEM)
            const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
            tc_mma_ts(tmem + 256, tmem + packed_col_dkv(kk), mnmaj_desc(dout, kk), IDESC_G, acc);
            tc_mma_ts(tmem + 384, tmem + 128 + packed_col_dkv(kk), mnmaj_desc(q, kk), IDESC_G, acc);
          }
        }
        tc_commit(&qdo_empty[st]);
      }
      tc_commit(pd_done);
    }
    __syncwarp();
  } else if (warp >= 4) {
    const int half = warp >= 8 ? 1 : 0;  // warpgroup: columns 32 * half + 64 * c of chunk c
    const uint32_t q4 = warp & 3;
    const int r = q4 * 32 + lane;        // KV row of the tile
    const int srow = kt * TILE + r;      // KV position
    const uint32_t lane_base = (q4 * 32) << 16;
    for (int it = 0; it < iters; ++it) {
      const int st = it % kDkvStages;
      const int q0 = (kt + it % per_head) * TILE;
      const float* s_lse = (const float*)(sm + L::LD0 + st * 1024);
      const float* s_delta = s_lse + 128;
      mbar_wait(s_full, it & 1, abort_flag, kErrTimeoutAttn);
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 2; ++c) {  // the first 64 queries, then the last 64
        const int col = 64 * c + 32 * half;
        const bool need_mask = q0 + col < srow + 1;  // padded query rows have lse2 = +inf
        uint32_t sv[32], dv[32];
        __syncwarp();
        tmem_ld32(tmem + lane_base + col, sv);
        tmem_ld32(tmem + lane_base + 128 + col, dv);
        tmem_ld_wait();
        float p[32], ds[32];
        float lse_c[32], del_c[32];  // 16-byte loads (the stage is 1024-byte aligned)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 l4 = ((const float4*)(s_lse + col))[i], d4 = ((const float4*)(s_delta + col))[i];
          lse_c[4 * i] = l4.x, lse_c[4 * i + 1] = l4.y, lse_c[4 * i + 2] = l4.z, lse_c[4 * i + 3] = l4.w;
          del_c[4 * i] = d4.x, del_c[4 * i + 1] = d4.y, del_c[4 * i + 2] = d4.z, del_c[4 * i + 3] = d4.w;
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float pv = ex2_approx(fmaf(__uint_as_float(sv[i]), a.scale_log2, -lse_c[i]));
          if (need_mask && q0 + col + i < srow) pv = 0.f;  // query must be at or after the key
          p[i] = pv;
          ds[i] = pv * (__uint_as_float(dv[i]) - del_c[i]);
        }
        // pairs over the first 16 of this chunk's columns, already read
        __syncwarp();
        tmem_st_bf16x32(tmem + lane_base + col, p);
        tmem_st_bf16x32(tmem + lane_base + 128 + col, ds);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[c]);
      }
    }
    mbar_wait(pd_done, 0, abort_flag, kErrTimeoutAttn);
    tc_fence_after();
    // epilogue: warpgroup A writes dV, warpgroup B writes dK (rotated back by RoPE if requested)
    const bool row_ok = srow < a.S;
    const size_t orow = ((size_t)b * a.S + srow) * a.ldkv + (size_t)g * D;
    const float2* tab = a.rope_tab ? a.rope_tab + (size_t)(row_ok ? srow : 0) * (D / 2) : nullptr;
    if (half == 0)
      store_grad_row<D>(a.dv + orow, tmem + lane_base + 256, row_ok, 1.f, nullptr, 0, 1);
    else
      store_grad_row<D>(a.dk + orow, tmem + lane_base + 384, row_ok, a.scale, tab, 0, 1);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// dQ pass: CTA = (128-row query tile qt, query head j, sequence b); loop over
// the 128-row KV tiles 0..qt (every product is 128 wide: narrower tcgen05
// products run well below the tensor core's rate). TMEM: S [2 x 128] +0
// (dS packed over each warpgroup's own first 32 columns), dP [128] +256,
// dQ +384. Once both warpgroups have read dP(t), the MMA thread issues
// S(t+1) and dP(t+1), so they run while the elementwise warps work on t;
// dQ += dS(t) K(t) follows when dS(t) is written. K has three stages (it is
// held until its dQ product), V two (released after its dP product).
constexpr int kDqKStages = 3;  // K is held until its dQ product; V only until its dP product

template <int D>
struct DqSmem {
  static constexpr int Q = 0;
  static constexpr int DO = Q + tile_bytes<D>();
  static constexpr int K0 = DO + tile_bytes<D>();                   // [3] 128-row K tiles
  static constexpr int V0 = K0 + kDqKStages * tile_bytes<D>();      // [2] 128-row V tiles
  static constexpr int BAR = V0 + 2 * tile_bytes<D>();
  static constexpr int TOTAL = BAR + 256;
  static constexpr int ALLOC = (TOTAL + 1024 > 118 * 1024) ? TOTAL + 1024 : 118 * 1024;
};


template <int D>
__global__ void __launch_bounds__(384, 1)
    attn_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                          const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                          AttnArgs a) {
  using L = DqSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(sm + L::BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;   // [3]
  uint64_t* k_empty = bars + 4;  // [3]
  uint64_t* v_full = bars + 7;   // [2]
  uint64_t* v_empty = bars + 9;  // [2]
  uint64_t* s_full = bars + 11;  // [2]: S(t) and dP(t) ready
  uint64_t* dp_free = bars + 13;
  uint64_t* p_full = bars + 14;
  uint64_t* g_done = bars + 15;
  uint32_t* tmem_slot = (uint32_t*)(bars + 16);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

  const int nqt = (a.S + TILE - 1) / TILE;
  // longest tiles first over the whole grid (the tile index is the slowest
  // coordinate of the linear block order)
  const int lin = (int)(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
  const int hb = lin % (a.nq * a.B);
  const int qt = nqt - 1 - lin / (a.nq * a.B);
  const int j = hb % a.nq, b = hb / a.nq;
  const int g = j / (a.nq / a.nkv);
  const int iters = qt + 1;  // KV tiles at or before the query tile
  const uint32_t warp = warp_id(), lane = lane_id();

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < kDqKStages; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
      mbar_init(&s_full[i], 1);
    }
    mbar_init(dp_free, 8);
    mbar_init(p_full, 8);
    mbar_init(g_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      prefetch_tmap(&tdo);
      mbar_arrive_expect_tx(q_full, 2 * tile_bytes<D>());
      load_head_tile<D>(sm + L::Q, &tq, q_full, j, qt * TILE, b);
      load_head_tile<D>(sm + L::DO, &tdo, q_full, j, qt * TILE, b);
      for (int it = 0; it < iters; ++it) {
        const int sv = it & 1, sk = it % kDqKStages;
        mbar_wait(&v_empty[sv], ((it >> 1) & 1) ^ 1, abort_flag, kErrTimeoutAttn);  // V frees first (after dP)
        mbar_arrive_expect_tx(&v_full[sv], tile_bytes<D>());
        load_head_tile<D>(sm + L::V0 + sv * tile_bytes<D>(), &tv, &v_full[sv], g, it * TILE, b);
        mbar_wait(&k_empty[sk], ((it / kDqKStages) & 1) ^ 1, abort_flag, kErrTimeoutAttn);
        mbar_arrive_expect_tx(&k_full[sk], tile_bytes<D>());
        load_head_tile<D>(sm + L::K0 + sk * tile_bytes<D>(), &tk, &k_full[sk], g, it * TILE, b);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t IDESC_S = make_idesc(128, 128, false, false);
      constexpr uint32_t IDESC_G = make_idesc(128, D < 64 ? 64 : D, false, true);
      constexpr int KS = D / 16;
      auto issue_scores = [&](int t) {  // S(t) = Q K_t^T into S[t & 1]; dP(t) = dO V_t^T
        const int st = t & 1;
        const uint8_t* kt = sm + L::K0 + (t % kDqKStages) * tile_bytes<D>();
        const uint8_t* vt = sm + L::V0 + st * tile_bytes<D>();
#pragma unroll
        for (int kk = 0; kk < KS; ++kk)
          tc_mma(tmem + st * 128, kmaj_desc(sm + L::Q, kk), kmaj_desc(kt, kk), IDESC_S, kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < KS; ++kk)
          tc_mma(tmem + 256, kmaj_desc(sm + L::DO, kk), kmaj_desc(vt, kk), IDESC_S, kk > 0 ? 1u : 0u);
        tc_commit(&s_full[st]);
        tc_commit(&v_empty[st]);
      };
      mbar_wait(q_full, 0, abort_flag, kErrTimeoutAttn);
      mbar_wait(&k_full[0], 0, abort_flag, kErrTimeoutAttn);
      mbar_wait(&v_full[0], 0, abort_flag, kErrTimeoutAttn);
      tc_fence_after();
      issue_scores(0);
      for (int it = 0; it < iters; ++it) {
        if (it + 1 < iters) {
          const int t1 = it + 1;
          mbar_wait(&k_full[t1 % kDqKStages], (t1 / kDqKStages) & 1, abort_flag, kErrTimeoutAttn);
          mbar_wait(&v_full[t1 & 1], (t1 >> 1) & 1, abort_flag, kErrTimeoutAttn);
          mbar_wait(dp_free, it & 1, abort_flag, kErrTimeoutAttn);  // both warpgroups have read dP(it)
          tc_fence_after();
          issue_scores(it + 1);  // S[(it+1)&1] held dS(it-1), consumed by dQ products issued before
        }
        mbar_wait(p_full, it & 1, abort_flag, kErrTimeoutAttn);
        tc_fence_after();
        const uint8_t* kt = sm + L::K0 + (it % kDqKStages) * tile_bytes<D>();
#pragma unroll
        for (int kk = 0; kk < TILE / 16; ++kk)  // dQ += dS K  (dS in TMEM)
          tc_mma_ts(tmem + 384, tmem + (it & 1) * 128 + packed_col128(kk), mnmaj_desc(kt, kk), IDESC_G,
                    (it > 0 || kk > 0) ? 1u : 0u);
        tc_commit(g_done);
        tc_commit(&k_empty[it % kDqKStages]);
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    const int half = warp >= 8 ? 1 : 0;  // which 64 of the 128 KV columns
    const uint32_t q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const int trow = qt * TILE + r;
    const uint32_t lane_base = (q4 * 32) << 16;
    const bool row_ok = trow < a.S;
    const size_t ri = ((size_t)b * a.nq + j) * pad128(a.S) + (row_ok ? trow : 0);
    const float lse2 = row_ok ? a.lse2[ri] : INFINITY;  // rows past S get probability 0
    const float dl = row_ok ? a.delta[ri] : 0.f;
    for (int it = 0; it < iters; ++it) {
      const int buf = it & 1;
      const uint32_t s_col = tmem + lane_base + buf * 128 + half * 64;
      const uint32_t dp_col = tmem + lane_base + 256 + half * 64;
      mbar_wait(&s_full[buf], (it >> 1) & 1, abort_flag, kErrTimeoutAttn);
      tc_fence_after();
      uint32_t dv0[32], dv1[32], sv0[32], sv1[32];
      __syncwarp();
      tmem_ld32(dp_col, dv0);
      tmem_ld32(dp_col + 32, dv1);
      tmem_ld32(s_col, sv0);
      tmem_ld32(s_col + 32, sv1);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dp_free);  // dP(it+1) may now be written
      const int kv0 = it * TILE + half * 64;
      const bool need_mask = it == qt;  // the diagonal tile (also holds the sequence tail)
      float ds0[32], ds1[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float p0 = ex2_approx(fmaf(__uint_as_float(sv0[i]), a.scale_log2, -lse2));
        float p1 = ex2_approx(fmaf(__uint_as_float(sv1[i]), a.scale_log2, -lse2));
        if (need_mask) {
          if (kv0 + i > trow || kv0 + i >= a.S) p0 = 0.f;
          if (kv0 + 32 + i > trow || kv0 + 32 + i >= a.S) p1 = 0.f;
        }
        ds0[i] = p0 * (__uint_as_float(dv0[i]) - dl);
        ds1[i] = p1 * (__uint_as_float(dv1[i]) - dl);
      }
      __syncwarp();
      tmem_st_bf16x32(s_col, ds0);       // packed over this warpgroup's own S columns, already read
      tmem_st_bf16x32(s_col + 16, ds1);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    mbar_wait(g_done, (iters - 1) & 1, abort_flag, kErrTimeoutAttn);
    tc_fence_after();
    // epilogue: the two warpgroups share the head-dim columns
    uint16_t* orow = a.dq + ((size_t)b * a.S + trow) * a.ldq + (size_t)j * D;
    const float2* tab = a.rope_tab ? a.rope_tab + (size_t)(row_ok ? trow : 0) * (D / 2) : nullptr;
    store_grad_row<D>(orow, tmem + lane_base + 384, row_ok, a.scale, tab, half, 2);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Per (sequence b, query head j, position t < Sp): delta = sum_e dO O over
// the head's columns and lse2 = lse * log2(e); padding rows t >= S get delta
// 0 and lse2 +inf. Layout [B][nq][Sp] each. Sixteen lanes per row, 16-byte
// loads (head dims of 64 and 128; narrower heads use 4-byte loads).
__global__ void attn_delta_tc_kernel(const uint16_t* __restrict__ o, const uint16_t* __restrict__ dout,
                                     const float* __restrict__ lse, float* __restrict__ delta,
                                     float* __restrict__ lse2, int B, int S, int Sp, int nq, int d, int ldo) {
  const size_t row = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) >> 4;
  const int sub = threadIdx.x & 15;
  const bool valid = row < (size_t)B * Sp * nq;  // every lane reaches the shuffles below
  const int j = (int)(row % nq);
  const int t = (int)((row / nq) % Sp);
  const int b = (int)(row / ((size_t)nq * Sp));
  const size_t ri = ((size_t)b * nq + j) * Sp + t;
  float s = 0.f;
  if (valid && t < S) {
    const size_t off = ((size_t)b * S + t) * ldo + (size_t)j * d;
    if ((d & 63) == 0 && (ldo & 7) == 0) {
      for (int e = sub * 8; e < d; e += 128) {
        const uint4 ov = *(const uint4*)(o + off + e), gv = *(const uint4*)(dout + off + e);
        const uint32_t oa[4] = {ov.x, ov.y, ov.z, ov.w}, ga[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
          s += bf2f(oa[k] & 0xffff) * bf2f(ga[k] & 0xffff) + bf2f(oa[k] >> 16) * bf2f(ga[k] >> 16);
      }
    } else {
      for (int e = sub * 2; e < d; e += 32) {
        const uint32_t ov = *(const uint32_t*)(o + off + e), gv = *(const uint32_t*)(dout + off + e);
        s += bf2f(ov & 0xffff) * bf2f(gv & 0xffff) + bf2f(ov >> 16) * bf2f(gv >> 16);
      }
    }
  }
#pragma unroll
  for (int m = 8; m >= 1; m >>= 1) s += __shfl_xor_sync(0xffffffffu, s, m);
  if (valid && sub == 0) {
    delta[ri] = s;
    lse2[ri] = t < S ? lse[((size_t)b * nq + j) * S + t] * 1.4426950408889634f : INFINITY;
  }
}

// 4D map over a [B, S, heads, d] view with row stride ld (elements); boxes
// of [rows][64] (one head).
int head_map(CUtensorMap* m, const void* base, int d, int heads, int S, int B, int ld, int rows = 128) {
  const uint64_t gdim[4] = {(uint64_t)d, (uint64_t)heads, (uint64_t)S, (uint64_t)B};
  const uint64_t gstride[3] = {(uint64_t)d * 2, (uint64_t)ld * 2, (uint64_t)S * ld * 2};
  const uint32_t box[4] = {64, 1, (uint32_t)rows, 1};
  return mt_host::encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, gdim, gstride, box,
                               CU_TENSOR_MAP_SWIZZLE_128B) == CUDA_SUCCESS
             ? 0
             : -1;
}

template <typename K>
bool set_smem(K kern, int bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) == cudaSuccess;
}

template <int D>
int fwd_launch(const uint16_t* q, const uint16_t* k, const uint16_t* v, AttnArgs& a, cudaStream_t st) {
  CUtensorMap tq, tk, tv;
  if (head_map(&tq, q, D, a.nq, a.S, a.B, a.ldq) || head_map(&tk, k, D, a.nkv, a.S, a.B, a.ldkv) ||
      head_map(&tv, v, D, a.nkv, a.S, a.B, a.ldkv))
    return -1;
  static bool init = false;
  if (!init) {
    if (!set_smem(attn_fwd_tc_kernel<D>, FwdSmem<D>::ALLOC)) return -1;
    init = true;
  }
  const int nqt = (a.S + TILE - 1) / TILE;
  dim3 grid((nqt + 1) / 2, a.nq, a.B);
  attn_fwd_tc_kernel<D><<<grid, 384, FwdSmem<D>::ALLOC, st>>>(tq, tk, tv, a);
  count_launches(1);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

template <int D>
int bwd_launch(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* o, const uint16_t* dout,
               AttnArgs& a, float* delta, cudaStream_t st) {
  // both passes: everything in 128-row tiles
  CUtensorMap tk128, tv128, tq128, tdo128;
  if (head_map(&tk128, k, D, a.nkv, a.S, a.B, a.ldkv) || head_map(&tv128, v, D, a.nkv, a.S, a.B, a.ldkv) ||
      head_map(&tq128, q, D, a.nq, a.S, a.B, a.ldq) || head_map(&tdo128, dout, D, a.nq, a.S, a.B, a.ldo))
    return -1;
  static bool init = false;
  if (!init) {
    if (!set_smem(attn_bwd_dkv_tc_kernel<D>, DkvSmem<D>::ALLOC) || !set_smem(attn_bwd_dq_tc_kernel<D>, DqSmem<D>::ALLOC))
      return -1;
    init = true;
  }
  const int Sp = pad128(a.S);
  const size_t rows = (size_t)a.B * Sp * a.nq;
  float* lse2 = delta + rows;
  attn_delta_tc_kernel<<<(unsigned)((rows * 16 + 255) / 256), 256, 0, st>>>(o, dout, a.lse_in, delta, lse2, a.B, a.S,
                                                                            Sp, a.nq, D, a.ldo);
  a.delta = delta;
  a.lse2 = lse2;
  const int nt = (a.S + TILE - 1) / TILE;
  attn_bwd_dkv_tc_kernel<D><<<dim3(nt, a.nkv, a.B), 384, DkvSmem<D>::ALLOC, st>>>(tq128, tk128, tv128, tdo128, a);
  attn_bwd_dq_tc_kernel<D><<<dim3(nt, a.nq, a.B), 384, DqSmem<D>::ALLOC, st>>>(tq128, tk128, tv128, tdo128, a);
  count_launches(3);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

size_t attention_bwd_workspace(int B, int S, int nq) { return 2 * (size_t)B * nq * pad128(S); }

namespace {

bool tc_ok(int B, int S, int nq, int nkv, int d, int ldq, int ldkv, int ldo, const void* q, const void* k,
           const void* v) {
  if (B <= 0 || S <= 0 || nq <= 0 || nkv <= 0 || nq % nkv) return false;
  if (d != 16 && d != 32 && d != 64 && d != 128) return false;
  if ((ldq & 7) || (ldkv & 7) || (ldo & 7)) return false;
  if (((uintptr_t)q & 15) || ((uintptr_t)k & 15) || ((uintptr_t)v & 15)) return false;
  return true;
}

}  // namespace

int attention_fwd_tc(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* o, float* lse, int B, int S,
                     int nq, int nkv, int d, int ldq, int ldkv, int ldo, cudaStream_t st) {
  if (!tc_ok(B, S, nq, nkv, d, ldq, ldkv, ldo, q, k, v)) return -1;
  AttnArgs a{o, lse, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, B, S, nq, nkv, ldq, ldkv, ldo,
             1.4426950408889634f / sqrtf((float)d), 1.f / sqrtf((float)d), nullptr};
  switch (d) {
    case 16: return fwd_launch<16>(q, k, v, a, st);
    case 32: return fwd_launch<32>(q, k, v, a, st);
    case 64: return fwd_launch<64>(q, k, v, a, st);
    default: return fwd_launch<128>(q, k, v, a, st);
  }
}

int attention_bwd_tc(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* o, const uint16_t* dout,
                     const float* lse, uint16_t* dq, uint16_t* dk, uint16_t* dv, float* work, int B, int S, int nq,
                     int nkv, int d, int ldq, int ldkv, int ldo, cudaStream_t st, const float2* rope_tab) {
  if (!tc_ok(B, S, nq, nkv, d, ldq, ldkv, ldo, q, k, v) || ((uintptr_t)work & 15)) return -1;
  AttnArgs a{nullptr, nullptr, lse, nullptr, nullptr, dq, dk, dv, B, S, nq, nkv, ldq, ldkv, ldo,
             1.4426950408889634f / sqrtf((float)d), 1.f / sqrtf((float)d), rope_tab};
  switch (d) {
    case 16: return bwd_launch<16>(q, k, v, o, dout, a, work, st);
    case 32: return bwd_launch<32>(q, k, v, o, dout, a, work, st);
    case 64: return bwd_launch<64>(q, k, v, o, dout, a, work, st);
    default: return bwd_launch<128>(q, k, v, o, dout, a, work, st);
  }
}

}  // namespace mt
