// Dense bf16 GEMM on the 5th-generation tensor cores (tcgen05), fp32
// accumulation in tensor memory, operands staged by TMA.
//
// The layer template's linear maps (QKV, O, gate-up, down, LM head) in their
// three forms: forward y = x W^T (both operands K-major), input gradient
// dx = dy W (B stored [K, N], MN-major), weight gradient dW = dy^T x (both
// operands MN-major, the reduction runs over tokens). MegaTrain (section
// 核心方法) describes the template as CUDA kernels for the attention and MLP
// blocks bound to streamed weights; here weights arrive as plain device
// pointers per launch, so the kernel holds no persistent weight state.
//
// Structure: persistent CTAs (one per SM), 128 x BN output tiles, K in steps
// of 64 (one 128-byte swizzle row), STAGES-deep TMA ring; warp 0 issues TMA,
// warp 1 issues tcgen05.mma from one thread, warps 2-5 drain the two TMEM
// accumulators (2 x BN columns) so the epilogue of tile i overlaps the
// mainloop of tile i+1. Each output tile is produced by one CTA with a fixed
// K order, so results do not depend on the grid size (deterministic).
#include <algorithm>
#include <cstdio>
#include <cstdlib>

#include "common.cuh"
#include "kernels.h"

namespace mt {

MT_DEVICE_ERROR_READER(gemm_take_device_error)
MT_DEVICE_ERROR_PEEKER(gemm_peek_device_error)

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB
// fp32 epilogue staging: per epilogue warp 32 rows x 32 columns, row stride
// 36 floats (conflict-free 16-byte accesses both ways)
constexpr int kStgStride = 36;
constexpr int kStagingBytes = 4 * 32 * kStgStride * 4;  // 18 KB

template <int BN>
struct GemmCfg {
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = (BN == 256) ? 4 : 6;
  static constexpr int SMEM = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/ + kStagingBytes;
  static constexpr int TMEM_COLS = 2 * BN;
};

// Tile order: groups of GROUP_M row-blocks, row-block fastest inside a group,
// so a wave of CTAs shares a band of A rows and a few B column-blocks in L2.
// GROUP_M is chosen on the host so that the band of A fits comfortably in L2
// (the whole of M when it does), which makes B stream from DRAM once per group.
__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int GROUP_M, int& m_blk, int& n_blk) {
  const int per_group = GROUP_M * num_n;
  const int g = tile / per_group;
  const int first_m = g * GROUP_M;
  const int gsize = min(num_m - first_m, GROUP_M);
  const int r = tile - g * per_group;
  m_blk = first_m + r % gsize;
  n_blk = r / gsize;
}

// One output tile of the (possibly grouped) product: its row/column origin,
// K range and operand offsets.
struct TileInfo {
  int m0, n0, nb;
  int crow;        // row of C holding the tile's first row
  int a_k0, b_k0;  // added to the K coordinate of A / of B
  int b_n0;        // added to the row (NT) coordinate of B
  int nkb;         // K steps
  bool skip;
};

// A_MN marks the weight-gradient form (TN); B_MN without A_MN is NN.
template <bool A_MN, bool B_MN>
__device__ __forceinline__ TileInfo decode_tile(const GemmParams& p, int tile, int num_m, int num_n, int tile_n,
                                                int num_kb) {
  TileInfo t;
  const bool grouped = p.grp_seg != nullptr;
  int e = 0, local = tile;
  if (grouped && A_MN) {
    e = tile / (num_m * num_n);
    local = tile - e * num_m * num_n;
  }
  int mb, nb;
  tile_coords(local, num_m, num_n, p.group_m, mb, nb);
  t.m0 = mb * BM;
  t.n0 = nb * tile_n;
  t.nb = nb;
  t.crow = t.m0;
  t.a_k0 = t.b_k0 = t.b_n0 = 0;
  t.nkb = num_kb;
  t.skip = false;
  if (grouped) {
    if (A_MN) {  // TN: this expert's segment is the reduction
      const int s0 = p.grp_seg[e], s1 = p.grp_seg[e + 1];
      t.a_k0 = t.b_k0 = s0;
      t.nkb = (s1 - s0) / BK;
      t.crow = e * p.M + t.m0;
    } else {
      e = p.grp_tile_e[mb];
      t.skip = e < 0;
      if (!t.skip) {
        if (B_MN) t.b_k0 = e * p.grp_b_rows;  // NN: the expert's K rows of B
        else t.b_n0 = e * p.grp_b_rows;       // NT: the expert's rows of B
      }
    }
  }
  return t;
}

// Zeros over columns [n0, n0 + BN) of row `row` (an expert that received
// no rows: its weight gradient is zero).
template <int BN>
__device__ __forceinline__ void zero_tile_row(const GemmParams& p, int row, bool row_ok, int n0) {
  if (!row_ok) return;
  if (p.epi == EPI_BF16) {
    uint16_t* out = (uint16_t*)p.C + (size_t)row * p.ldc;
    for (int j = n0; j < n0 + BN && j < p.N; ++j) out[j] = 0;
  } else {
    float* out = (float*)p.C + (size_t)row * p.ldc;
    for (int j = n0; j < n0 + BN && j < p.N; ++j) out[j] = 0.f;
  }
}

// Store 32 fp32 values as bf16 at columns [col0, col0+32) of a row (partial
// at the right edge).
__device__ __forceinline__ void store_bf16_32(uint16_t* out, const float (&v)[32], int col0, int N, bool vec) {
  if (vec && col0 + 32 <= N) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint4 w;
      w.x = pack_bf2(v[8 * k + 0], v[8 * k + 1]);
      w.y = pack_bf2(v[8 * k + 2], v[8 * k + 3]);
      w.z = pack_bf2(v[8 * k + 4], v[8 * k + 5]);
      w.w = pack_bf2(v[8 * k + 6], v[8 * k + 7]);
      ((uint4*)out)[k] = w;
    }
  } else {
    for (int j = 0; j < 32 && col0 + j < N; ++j) out[j] = f2bf(v[j]);
  }
}

// bf16 epilogue with RoPE on the head columns (half-split pairs (i, i+d/2)):
// for d >= 64 the two halves of a head are chunk pairs (c, c + d/64); for
// d < 64 both halves sit in one 32-column chunk. Tiles are head-aligned
// (BN is a multiple of d).
template <int BN>
__device__ __forceinline__ void rope_epilogue(const GemmParams& p, uint32_t tbase, int row, bool row_ok, int n0) {
  const int d = p.rope_d, half = d >> 1;
  const float2* tab = p.rope_tab + (size_t)(row_ok ? row % p.rope_S : 0) * half;
  uint16_t* out = (uint16_t*)p.C + (size_t)row * p.ldc;
  if (d >= 64) {
    const int P = d >> 6;  // chunk distance between the halves
#pragma unroll 1
    for (int ca = 0; ca < BN / 32; ++ca) {
      if ((ca % (2 * P)) >= P) continue;  // second half: handled with its partner
      const int cb = ca + P;
      uint32_t ra[32], rb[32];
      __syncwarp();
      tmem_ld32(tbase + ca * 32, ra);
      tmem_ld32(tbase + cb * 32, rb);
      tmem_ld_wait();
      const int cola = n0 + ca * 32, colb = n0 + cb * 32;
      if (!row_ok || cola >= p.N) continue;
      const bool rot = cola < p.rope_cols;
      const int i0 = (ca % P) * 32;  // pair index of the chunk's first column within the head
      float fa[32], fb[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float x1 = __uint_as_float(ra[i]), x2 = __uint_as_float(rb[i]);
        if (rot) {
          const float2 cs = tab[i0 + i];
          fa[i] = x1 * cs.x - x2 * cs.y;
          fb[i] = x1 * cs.y + x2 * cs.x;
        } else {
          fa[i] = x1;
          fb[i] = x2;
        }
      }
      store_bf16_32(out + cola, fa, cola, p.N, p.vec);
      if (colb < p.N) store_bf16_32(out + colb, fb, colb, p.N, p.vec);
    }
  } else {
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t r[32];
      __syncwarp();
      tmem_ld32(tbase + c * 32, r);
      tmem_ld_wait();
      const int col0 = n0 + c * 32;
      if (!row_ok || col0 >= p.N) continue;
      float f[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int li = i % d;  // d in {16, 32}: divides 32
        const bool rot = col0 + i - li < p.rope_cols;
        if (rot && li < half) {
          const float x1 = __uint_as_float(r[i]), x2 = __uint_as_float(r[i + half]);
          const float2 cs = tab[li];
          f[i] = x1 * cs.x - x2 * cs.y;
          f[i + half] = x1 * cs.y + x2 * cs.x;
        } else if (!rot) {
          f[i] = __uint_as_float(r[i]);
        }
      }
      store_bf16_32(out + col0, f, col0, p.N, p.vec);
    }
  }
}

// sigmoid(g) = 1 / (1 + e^-g), the reciprocal by the hardware's approximate
// reciprocal (1 ulp; +0 for an infinite denominator).
__device__ __forceinline__ float silu_sig(float g) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.f + __expf(-g)));
  return r;
}

__device__ __forceinline__ void load_bf16_32(const uint16_t* src, float (&v)[32], int col0, int N, bool vec) {
  if (vec && col0 + 32 <= N) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 w = ((const uint4*)src)[k];
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v[8 * k + 2 * e] = bf2f(ws[e] & 0xffff);
        v[8 * k + 2 * e + 1] = bf2f(ws[e] >> 16);
      }
    }
  } else {
    for (int j = 0; j < 32; ++j) v[j] = col0 + j < N ? bf2f(src[j]) : 0.f;
  }
}

// Gated epilogue: TMEM columns [0, BN/2) hold g, [BN/2, BN) hold u for the
// features [f0, f0 + BN/2); act = silu(g) * u is formed from the fp32
// accumulators before rounding.
template <int BN>
__device__ __forceinline__ void gated_epilogue(const GemmParams& p, uint32_t tbase, int row, bool row_ok, int f0) {
  uint16_t* grow = (uint16_t*)p.C + (size_t)row * p.ldc;
  uint16_t* arow = p.act + (size_t)row * p.ld_act;
#pragma unroll 1
  for (int c = 0; c < BN / 64; ++c) {
    uint32_t rg[32], ru[32];
    __syncwarp();
    tmem_ld32(tbase + c * 32, rg);
    tmem_ld32(tbase + BN / 2 + c * 32, ru);
    tmem_ld_wait();
    const int col0 = f0 + c * 32;
    if (!row_ok || col0 >= p.N) continue;
    float g[32], u[32], a[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      g[i] = __uint_as_float(rg[i]);
      u[i] = __uint_as_float(ru[i]);
      a[i] = g[i] * silu_sig(g[i]) * u[i];
    }
    store_bf16_32(grow + col0, g, col0, p.N, p.vec);
    store_bf16_32(grow + p.u_col + col0, u, col0, p.N, p.vec);
    store_bf16_32(arow + col0, a, col0, p.N, p.vec);
  }
}

// SwiGLU backward epilogue: the accumulator is dact for features
// [n0, n0 + BN); g and u are read from gu and replaced by dg and du. Where
// the whole tile is in range and 16-byte aligned, the next chunk's g and u
// are loaded before this chunk is computed (their latency then overlaps the
// work; the addresses differ from this chunk's stores).
__device__ __forceinline__ void swiglu_bwd_32(const uint32_t (&rd)[32], float (&g)[32], float (&u)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float d = __uint_as_float(rd[i]);
    const float sg = silu_sig(g[i]);
    const float dg = d * u[i] * sg * (1.f + g[i] * (1.f - sg));
    u[i] = d * g[i] * sg;  // du
    g[i] = dg;
  }
}
__device__ __forceinline__ void unpack_bf16x8(const uint4 (&w)[4], float (&v)[32]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t ws[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[8 * k + 2 * e] = bf2f(ws[e] & 0xffff);
      v[8 * k + 2 * e + 1] = bf2f(ws[e] >> 16);
    }
  }
}
template <int BN>
__device__ __forceinline__ void swiglu_bwd_epilogue(const GemmParams& p, uint32_t tbase, int row, bool row_ok,
                                                    int n0) {
  uint16_t* gurow = p.gu + (size_t)row * p.ld_gu;
  if (p.vec && n0 + BN <= p.N) {  // the same in every lane
    uint4 gn[4], un[4];
    auto fetch = [&](int c) {
      if (!row_ok) return;
      const uint4* gp = (const uint4*)(gurow + n0 + 32 * c);
      const uint4* up = (const uint4*)(gurow + p.u_col + n0 + 32 * c);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        gn[k] = gp[k];
        un[k] = up[k];
      }
    };
    fetch(0);
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      uint4 gc[4], uc[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        gc[k] = gn[k];
        uc[k] = un[k];
      }
      if (c + 1 < BN / 32) fetch(c + 1);
      uint32_t rd[32];
      __syncwarp();
      tmem_ld32(tbase + c * 32, rd);
      tmem_ld_wait();
      if (!row_ok) continue;
      float g[32], u[32];
      unpack_bf16x8(gc, g);
      unpack_bf16x8(uc, u);
      swiglu_bwd_32(rd, g, u);
      const int col0 = n0 + c * 32;
      store_bf16_32(gurow + col0, g, col0, p.N, true);
      store_bf16_32(gurow + p.u_col + col0, u, col0, p.N, true);
    }
    return;
  }
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    uint32_t rd[32];
    __syncwarp();
    tmem_ld32(tbase + c * 32, rd);
    tmem_ld_wait();
    const int col0 = n0 + c * 32;
    if (!row_ok || col0 >= p.N) continue;
    float g[32], u[32];
    load_bf16_32(gurow + col0, g, col0, p.N, p.vec);
    load_bf16_32(gurow + p.u_col + col0, u, col0, p.N, p.vec);
    swiglu_bwd_32(rd, g, u);
    store_bf16_32(gurow + col0, g, col0, p.N, p.vec);
    store_bf16_32(gurow + p.u_col + col0, u, col0, p.N, p.vec);
  }
}

// g and u of the SwiGLU backward for one row of a tile, pulled into L2 while
// the tile's products still run, so that the epilogue's loads hit L2. Only
// addresses inside the row's valid columns are touched. (The fp32 residual
// of the add epilogue is not prefetched: its loads are issued ahead of the
// accumulator read already, and an L2 prefetch measured slower there.)
template <int BN>
__device__ __forceinline__ void prefetch_epilogue_inputs(const GemmParams& p, int row, bool row_ok, int n0) {
  if (!p.swiglu_bwd || !row_ok || n0 >= p.N) return;
  const int ncols = min(BN, p.N - n0);
  const char* g = (const char*)(p.gu + (size_t)row * p.ld_gu + n0);
  const char* u = (const char*)(p.gu + (size_t)row * p.ld_gu + p.u_col + n0);
  for (int off = 0; off < ncols * 2; off += 128) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(g + off));
    asm volatile("prefetch.global.L2 [%0];" ::"l"(u + off));
  }
}

// Epilogue of one output tile for one warp: TMEM lanes of `tb` hold row
// `row` (the warp's rows are consecutive); columns [nb * BN, nb * BN + BN) of
// C (gated tiles: tile_n features). fp32 results of whole 32-column chunks go
// through the warp's staging rows `stg` so that each group of 8 lanes stores
// 128 contiguous bytes of one row.
template <int BN>
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, uint32_t tb, int row, bool row_ok, int nb,
                                              int tile_n, float* stg) {
  if (p.rope_tab || p.gated || p.swiglu_bwd) {
    if (p.rope_tab) rope_epilogue<BN>(p, tb, row, row_ok, nb * BN);
    else if (p.gated) gated_epilogue<BN>(p, tb, row, row_ok, nb * tile_n);
    else swiglu_bwd_epilogue<BN>(p, tb, row, row_ok, nb * BN);
    return;
  }
  // The addend may be C itself (a residual added in place), so the compiler
  // keeps each addend load behind the previous store; the loads of a chunk
  // are therefore all issued up front, before its accumulator is read.
  const unsigned valid = __ballot_sync(0xffffffffu, row_ok);
  const int lane = threadIdx.x & 31;
  const int wrow0 = row - lane;
  const int sub = lane >> 3, c4 = (lane & 7) * 4;
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    uint32_t r[32];
    const int col0 = nb * BN + c * 32;
    const bool full_cols = p.vec && col0 + 32 <= p.N;  // the same in every lane
    const bool staged = p.epi != EPI_BF16 && full_cols && p.stage_f32;
    float4 a[8];
    if (p.epi == EPI_F32_ADD && full_cols) {
      const float* add = (const float*)p.addend;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        a[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (staged) {
          const int rr = 4 * i + sub;
          if ((valid >> rr) & 1u) a[i] = *(const float4*)(add + (size_t)(wrow0 + rr) * p.ldc + col0 + c4);
        } else if (row_ok) {
          a[i] = *(const float4*)(add + (size_t)row * p.ldc + col0 + 4 * i);
        }
      }
    }
    __syncwarp();
    tmem_ld32(tb + c * 32, r);
    tmem_ld_wait();
    if (staged) {
      __syncwarp();
      float* srow = stg + lane * kStgStride;
#pragma unroll
      for (int v = 0; v < 8; ++v)
        ((float4*)srow)[v] = make_float4(__uint_as_float(r[4 * v + 0]), __uint_as_float(r[4 * v + 1]),
                                         __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int rr = 4 * i + sub;
        if ((valid >> rr) & 1u) {
          float4 w = *(const float4*)(stg + rr * kStgStride + c4);
          if (p.epi == EPI_F32_ADD) {
            w.x += a[i].x;
            w.y += a[i].y;
            w.z += a[i].z;
            w.w += a[i].w;
          }
          *(float4*)((float*)p.C + (size_t)(wrow0 + rr) * p.ldc + col0 + c4) = w;
        }
      }
      continue;
    }
    if (!row_ok || col0 >= p.N) continue;
    if (p.epi == EPI_BF16) {
      uint16_t* out = (uint16_t*)p.C + (size_t)row * p.ldc + col0;
      if (full_cols) {
        uint4* o4 = (uint4*)out;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 w;
          w.x = pack_bf2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
          w.y = pack_bf2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
          w.z = pack_bf2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
          w.w = pack_bf2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
          o4[v] = w;
        }
      } else {
        for (int j = 0; j < 32 && col0 + j < p.N; ++j) out[j] = f2bf(__uint_as_float(r[j]));
      }
    } else {
      float* out = (float*)p.C + (size_t)row * p.ldc + col0;
      const float* add = p.epi == EPI_F32_ADD ? (const float*)p.addend + (size_t)row * p.ldc + col0 : nullptr;
      if (full_cols) {
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          float4 w = make_float4(__uint_as_float(r[4 * v + 0]), __uint_as_float(r[4 * v + 1]),
                                 __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
          if (add) {
            w.x += a[v].x;
            w.y += a[v].y;
            w.z += a[v].z;
            w.w += a[v].w;
          }
          ((float4*)out)[v] = w;
        }
      } else {
        for (int j = 0; j < 32 && col0 + j < p.N; ++j) out[j] = __uint_as_float(r[j]) + (add ? add[j] : 0.f);
      }
    }
  }
}

template <int BN, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(192, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, GemmParams p) {
  using C = GemmCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem;
  uint8_t* sB = smem + C::STAGES * A_BYTES;
  uint64_t* full = (uint64_t*)(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = (uint32_t*)(tempty + 2);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
  float* staging = (float*)(smem + C::STAGES * C::STAGE_BYTES + 256);  // after the barriers

  const uint32_t warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int tile_n = p.gated ? BN / 2 : BN;  // gated tiles cover BN/2 features (gate + up halves)
  const int num_m = (p.M + BM - 1) / BM, num_n = (p.N + tile_n - 1) / tile_n;
  // grouped weight gradients: one M x N output per expert
  const int num_tiles = num_m * num_n * ((p.grp_seg && A_MN) ? p.grp_E : 1);
  const int num_kb = (p.K + BK - 1) / BK;

  if (warp == 0) {
    if (lane == 0) {  // TMA producer
      int stage = 0;
      uint32_t phase = 0;
      for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
        const TileInfo ti = decode_tile<A_MN, B_MN>(p, tile, num_m, num_n, tile_n, num_kb);
        if (ti.skip) continue;
        const int m0 = ti.m0, n0 = ti.n0;
        for (int kb = 0; kb < ti.nkb; ++kb) {
          mbar_wait(&empty[stage], phase ^ 1, abort_flag, kErrTimeoutTma);
          mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
          uint8_t* a_dst = sA + stage * A_BYTES;
          uint8_t* b_dst = sB + stage * C::B_BYTES;
          const int ka = ti.a_k0 + kb * BK, kb_ = ti.b_k0 + kb * BK;
          if (!A_MN) {
            tma_load_2d(a_dst, &tmA, &full[stage], ka, m0);
          } else {
#pragma unroll
            for (int j = 0; j < BM / 64; ++j) tma_load_2d(a_dst + j * 8192, &tmA, &full[stage], m0 + 64 * j, ka);
          }
          if (!B_MN && p.gated) {  // gate rows then the matching up rows
            tma_load_2d(b_dst, &tmB, &full[stage], kb_, ti.b_n0 + n0);
            tma_load_2d(b_dst + (BN / 2) * 128, &tmB, &full[stage], kb_, ti.b_n0 + p.u_off + n0);
          } else if (!B_MN) {
            tma_load_2d(b_dst, &tmB, &full[stage], kb_, ti.b_n0 + n0);
          } else {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j) tma_load_2d(b_dst + j * 8192, &tmB, &full[stage], n0 + 64 * j, kb_);
          }
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      constexpr uint32_t IDESC = make_idesc(BM, BN, A_MN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
        const TileInfo ti = decode_tile<A_MN, B_MN>(p, tile, num_m, num_n, tile_n, num_kb);
        if (ti.skip) continue;
        const int acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        ++local;
        mbar_wait(&tempty[acc], acc_phase ^ 1, abort_flag, kErrTimeoutMma);
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < ti.nkb; ++kb) {
          mbar_wait(&full[stage], phase, abort_flag, kErrTimeoutMma);
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + stage * A_BYTES);
          const uint32_t b_base = smem_u32(sB + stage * C::B_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = A_MN ? make_sdesc(a_base + kk * 2048, 8192, 1024) : make_sdesc(a_base + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? make_sdesc(b_base + kk * 2048, 8192, 1024) : make_sdesc(b_base + kk * 32, 16, 1024);
            tc_mma(d_tmem, ad, bd, IDESC, (kb | kk) != 0);
          }
          tc_commit(&empty[stage]);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        tc_commit(&tfull[acc]);  // with no K steps: arrives once earlier work is done
      }
    }
    __syncwarp();
  } else {  // epilogue warps 2..5; warp w reads TMEM lanes 32*(w%4) .. +31
    const uint32_t q = warp & 3;
    int local = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      const TileInfo ti = decode_tile<A_MN, B_MN>(p, tile, num_m, num_n, tile_n, num_kb);
      if (ti.skip) continue;
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      ++local;
      const int r = ti.m0 + q * 32 + lane;  // row within this product's M
      if (ti.nkb > 0) prefetch_epilogue_inputs<BN>(p, ti.crow + q * 32 + lane, r < p.M, ti.nb * BN);
      mbar_wait(&tfull[acc], acc_phase, abort_flag, kErrTimeoutEpi);
      tc_fence_after();
      if (ti.nkb == 0) {
        zero_tile_row<BN>(p, ti.crow + q * 32 + lane, r < p.M, ti.n0);
      } else {
        epilogue_tile<BN>(p, tmem_base + ((q * 32) << 16) + acc * BN, ti.crow + q * 32 + lane, r < p.M, ti.nb,
                          tile_n, staging + q * 32 * kStgStride);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Paired-SM form for wide tiles: a cluster of two CTAs computes 256 x 256
// output tiles with tcgen05.mma.cta_group::2. Each CTA stages its own 128
// rows of A and its half (128 rows of N) of B, so every SM feeds the tensor
// core from 32 KB of shared memory per 64-deep K step instead of 48 KB, and
// the ring holds six stages. The even CTA issues the MMAs; its accumulator
// rows [0, 128) land in its tensor memory and rows [128, 256) in the odd
// CTA's. Both CTAs' TMA loads complete on the even CTA's stage barrier, the
// even CTA's commits arrive on both CTAs' stage-free and accumulator-ready
// barriers, and both CTAs' epilogue warps report a drained accumulator to
// the even CTA. Gated tiles put the gate rows in the even CTA's half of B and
// the matching up rows in the odd CTA's, which gives the same accumulator
// column layout as the single-CTA kernel.
// ---------------------------------------------------------------------------
struct PairCfg {
  static constexpr int BN = 256;
  static constexpr int B_BYTES = 128 * BK * 2;            // this CTA's half of B: 16 KB
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 32 KB
  static constexpr int STAGES = 6;
  static constexpr int SMEM = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/ + kStagingBytes;
};

template <bool A_MN, bool B_MN>
__global__ void __launch_bounds__(192, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, GemmParams p) {
  using C = PairCfg;
  constexpr int BN = C::BN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem;
  uint8_t* sB = smem + C::STAGES * A_BYTES;
  uint64_t* full = (uint64_t*)(smem + C::STAGES * C::STAGE_BYTES);  // even CTA: both halves landed
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 2;             // even CTA: both CTAs drained the accumulator
  uint32_t* tmem_slot = (uint32_t*)(tempty + 2);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
  float* staging = (float*)(smem + C::STAGES * C::STAGE_BYTES + 256);  // after the barriers

  const uint32_t warp = warp_id(), lane = lane_id();
  const uint32_t rank = cluster_rank();
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 8);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc2(tmem_slot, 2 * BN);
    tmem_relinquish2();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // barriers of both CTAs initialised, tensor memory allocated
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int tile_n = p.gated ? BN / 2 : BN;
  const int num_m = (p.M + 2 * BM - 1) / (2 * BM), num_n = (p.N + tile_n - 1) / tile_n;
  const int num_tiles = num_m * num_n;
  const int num_kb = (p.K + BK - 1) / BK;
  const int cl = (int)(blockIdx.x >> 1), ncl = (int)(gridDim.x >> 1);

  if (warp == 0) {
    if (lane == 0) {  // TMA producer (both CTAs)
      const uint32_t full0 = mapa_shared(full, 0);
      int stage = 0;
      uint32_t phase = 0;
      for (int tile = cl; tile < num_tiles; tile += ncl) {
        int mb, nb;
        tile_coords(tile, num_m, num_n, p.group_m, mb, nb);
        const int m0 = mb * 2 * BM + (int)rank * BM;
        const int nrow0 = p.gated ? (rank ? p.u_off : 0) + nb * tile_n : nb * BN + (int)rank * 128;
        for (int kb = 0; kb < num_kb; ++kb) {
          mbar_wait<true>(&empty[stage], phase ^ 1, abort_flag, kErrTimeoutTma);
          if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * C::STAGE_BYTES);
          const uint32_t bar = full0 + stage * 8;
          uint8_t* a_dst = sA + stage * A_BYTES;
          uint8_t* b_dst = sB + stage * C::B_BYTES;
          if (!A_MN) {
            tma_load_2d_pair(a_dst, &tmA, bar, kb * BK, m0);
          } else {
#pragma unroll
            for (int j = 0; j < BM / 64; ++j) tma_load_2d_pair(a_dst + j * 8192, &tmA, bar, m0 + 64 * j, kb * BK);
          }
          if (!B_MN) {
            tma_load_2d_pair(b_dst, &tmB, bar, kb * BK, nrow0);
          } else {
#pragma unroll
            for (int j = 0; j < 2; ++j) tma_load_2d_pair(b_dst + j * 8192, &tmB, bar, nrow0 + 64 * j, kb * BK);
          }
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {  // MMA issuer (even CTA)
      constexpr uint32_t IDESC = make_idesc(2 * BM, BN, A_MN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      for (int tile = cl; tile < num_tiles; tile += ncl, ++local) {
        const int acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        mbar_wait<true>(&tempty[acc], acc_phase ^ 1, abort_flag, kErrTimeoutMma);
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < num_kb; ++kb) {
          mbar_wait(&full[stage], phase, abort_flag, kErrTimeoutMma);
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + stage * A_BYTES);
          const uint32_t b_base = smem_u32(sB + stage * C::B_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = A_MN ? make_sdesc(a_base + kk * 2048, 8192, 1024) : make_sdesc(a_base + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? make_sdesc(b_base + kk * 2048, 8192, 1024) : make_sdesc(b_base + kk * 32, 16, 1024);
            tc_mma2(d_tmem, ad, bd, IDESC, (kb | kk) != 0);
          }
          tc_commit2(&empty[stage], 0x3);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        tc_commit2(&tfull[acc], 0x3);
      }
    }
    __syncwarp();
  } else {  // epilogue warps 2..5 of both CTAs; warp w reads TMEM lanes 32*(w%4) .. +31
    const uint32_t q = warp & 3;
    const uint32_t tempty0 = mapa_shared(tempty, 0);
    int local = 0;
    for (int tile = cl; tile < num_tiles; tile += ncl, ++local) {
      int mb, nb;
      tile_coords(tile, num_m, num_n, p.group_m, mb, nb);
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      const int row = mb * 2 * BM + (int)rank * BM + q * 32 + lane;
      prefetch_epilogue_inputs<BN>(p, row, row < p.M, nb * BN);
      mbar_wait<true>(&tfull[acc], acc_phase, abort_flag, kErrTimeoutEpi);
      tc_fence_after();
      epilogue_tile<BN>(p, tmem_base + ((q * 32) << 16) + acc * BN, row, row < p.M, nb, tile_n,
                        staging + q * 32 * kStgStride);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty0 + acc * 8);
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still address its barriers or tensor memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc2(tmem_base, 2 * BN);
  }
}

template <bool A_MN, bool B_MN>
int launch_pair(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p, cudaStream_t st) {
  auto kern = gemm_pair_kernel<A_MN, B_MN>;
  // shared memory without the fp32 staging rows unless this launch stages
  const int smem = p.stage_f32 ? PairCfg::SMEM : PairCfg::SMEM - kStagingBytes;
  static int max_clusters_v[2] = {0, 0};
  int& max_clusters = max_clusters_v[p.stage_f32 ? 1 : 0];
  static bool attr_set = false;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (!attr_set) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PairCfg::SMEM) != cudaSuccess)
      return -1;
    attr_set = true;
  }
  if (!max_clusters) {
    cfg.gridDim = dim3(2 * (mt_host::num_sms() / 2));
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (const void*)kern, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = mt_host::num_sms() / 2;
    }
    const char* fc = getenv("MT_GEMM_PAIR_CLUSTERS");
    if (fc && atoi(fc) > 0) n = atoi(fc);
    const char* dbg = getenv("MT_GEMM_DEBUG");
    if (dbg && dbg[0] == '1') fprintf(stderr, "gemm pair kernel: %d co-resident clusters\n", n);
    max_clusters = n;
  }
  const int tile_n = p.gated ? PairCfg::BN / 2 : PairCfg::BN;
  const int tiles = ((p.M + 2 * BM - 1) / (2 * BM)) * ((p.N + tile_n - 1) / tile_n);
  const int clusters = tiles < max_clusters ? tiles : max_clusters;
  cfg.gridDim = dim3(2 * clusters);
  if (cudaLaunchKernelEx(&cfg, kern, ta, tb, p) != cudaSuccess) return -1;
  count_launches(1);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

template <int BN, bool A_MN, bool B_MN>
int launch(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p, cudaStream_t st) {
  using C = GemmCfg<BN>;
  static bool attr_set = false;
  auto kern = gemm_kernel<BN, A_MN, B_MN>;
  if (!attr_set) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess) return -1;
    attr_set = true;
  }
  const int tile_n = p.gated ? BN / 2 : BN;
  const int tiles =
      ((p.M + BM - 1) / BM) * ((p.N + tile_n - 1) / tile_n) * ((p.grp_seg && A_MN) ? p.grp_E : 1);
  const int grid = tiles < mt_host::num_sms() ? tiles : mt_host::num_sms();
  const int smem = p.stage_f32 ? C::SMEM : C::SMEM - kStagingBytes;  // staging rows only when used
  kern<<<grid, 192, smem, st>>>(ta, tb, p);
  count_launches(1);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

// Tensor map of a bf16 matrix stored row-major with `rows` rows of `cols`
// valid elements and row stride `ld` (elements). box_inner is along cols.
int make_map(CUtensorMap* m, const void* base, int rows, int cols, int ld, int box_inner, int box_outer) {
  const uint64_t gdim[2] = {(uint64_t)cols, (uint64_t)rows};
  const uint64_t gstride[1] = {(uint64_t)ld * 2};
  const uint32_t box[2] = {(uint32_t)box_inner, (uint32_t)box_outer};
  return mt_host::encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, gdim, gstride, box,
                               CU_TENSOR_MAP_SWIZZLE_128B) == CUDA_SUCCESS
             ? 0
             : -1;
}

}  // namespace

int gemm_bf16(int mode, const GemmParams& pin, const void* A, const void* B, int lda, int ldb, cudaStream_t st) {
  GemmParams p = pin;
  if (p.M <= 0 || p.N <= 0 || p.K <= 0 || !p.C || p.epi < EPI_BF16 || p.epi > EPI_F32_ADD) return -1;
  if ((lda & 7) || (ldb & 7) || ((uintptr_t)A & 15) || ((uintptr_t)B & 15)) return -1;
  if (p.epi == EPI_F32_ADD && !p.addend) return -1;
  if (p.rope_tab && (p.epi != EPI_BF16 || p.rope_S <= 0 || (p.rope_d != 16 && p.rope_d != 32 && p.rope_d != 64 &&
                                                             p.rope_d != 128) || p.rope_cols % p.rope_d))
    return -1;
  // 16-byte stores need 16-byte aligned rows; otherwise the epilogue stores element by element.
  const int esz = p.epi == EPI_BF16 ? 2 : 4;
  p.vec = (((uintptr_t)p.C & 15) == 0 && ((size_t)p.ldc * esz) % 16 == 0 &&
           (p.epi != EPI_F32_ADD || ((uintptr_t)p.addend & 15) == 0))
              ? 1
              : 0;
  {
    // Band of A rows shared by one tile group: MT_GEMM_BAND_MB (default 32 MB).
    static size_t band_budget = 0;
    if (!band_budget) {
      const char* e = getenv("MT_GEMM_BAND_MB");
      const long mb = e ? atol(e) : 32;
      band_budget = (size_t)(mb > 0 ? mb : 32) << 20;
    }
    const int num_m = (p.M + BM - 1) / BM;
    const size_t band = (size_t)BM * p.K * 2;  // bytes of A per row-block
    const int gm = (int)std::max<size_t>(1, band_budget / band);
    p.group_m = gm < num_m ? gm : num_m;
  }
  if (p.gated && (mode != GEMM_NT || !p.act || (p.ld_act & 7) || (p.u_col & 7) || p.epi != EPI_BF16)) return -1;
  const bool grouped = p.grp_seg != nullptr;
  // fp32 outputs go through the shared-memory staging rows (coalesced
  // 128-byte row segments); bf16 outputs are stored straight from registers.
  p.stage_f32 = p.epi != EPI_BF16 ? 1 : 0;
  if (grouped) {
    if (p.grp_E < 1 || p.rope_tab) return -1;
    if (mode == GEMM_TN) {
      if (p.gated || p.swiglu_bwd || p.epi == EPI_F32_ADD || (p.K % BM)) return -1;
    } else if (!p.grp_tile_e || p.grp_b_rows < 1 || (p.M % BM)) {
      return -1;
    }
    if (mode == GEMM_NN && (p.grp_b_rows % BK || p.K != p.grp_b_rows)) return -1;  // K tiles stay in one expert
  }
  if (p.swiglu_bwd && (mode != GEMM_NN || !p.gu || (p.ld_gu & 7) || (p.u_col & 7))) return -1;
  if (p.swiglu_bwd) p.vec = (((uintptr_t)p.gu & 15) == 0) ? 1 : 0;
  if (p.gated) p.vec = p.vec && (((uintptr_t)p.act & 15) == 0);
  // BN = 256 unless that leaves most SMs idle (gated tiles are always 256 wide).
  const int tiles256 = ((p.M + BM - 1) / BM) * ((p.N + 255) / 256);
  const bool wide = tiles256 >= mt_host::num_sms() || p.gated || grouped;
  const int BN = wide ? 256 : 128;
  // Wide tiles run on SM pairs (MT_GEMM_PAIR=0 keeps them on single SMs).
  static int pair_mode = -1;
  if (pair_mode < 0) {
    const char* e = getenv("MT_GEMM_PAIR");
    pair_mode = (e && e[0] == '0') ? 0 : 1;
  }
  const bool pair = wide && pair_mode && !grouped;  // grouped products run on single SMs
  if (pair) {  // tile groups in units of 256-row blocks
    const int num_m2 = (p.M + 2 * BM - 1) / (2 * BM);
    const int gm = std::max(1, p.group_m / 2);
    p.group_m = gm < num_m2 ? gm : num_m2;
  }
  const int b_rows = pair ? 128 : BN;  // K-major B box height
  CUtensorMap ta, tb;
  int rc = 0;
  if (mode == GEMM_NT) {  // A [M,K] K-major, B [N,K] K-major
    rc |= make_map(&ta, A, p.M, p.K, lda, 64, BM);
    const int b_all = grouped ? p.grp_E * p.grp_b_rows : 0;  // every expert's rows
    if (p.gated)  // gate and up rows of one combined matrix, 128-row boxes
      rc |= make_map(&tb, B, grouped ? b_all : p.u_off + p.N, p.K, ldb, 64, 128);
    else
      rc |= make_map(&tb, B, grouped ? b_all : p.N, p.K, ldb, 64, b_rows);
    if (rc) return -1;
    if (pair) return launch_pair<false, false>(ta, tb, p, st);
    return wide ? launch<256, false, false>(ta, tb, p, st) : launch<128, false, false>(ta, tb, p, st);
  }
  if (mode == GEMM_NN) {  // A [M,K] K-major, B stored [K,N]: MN-major
    rc |= make_map(&ta, A, p.M, p.K, lda, 64, BM);
    rc |= make_map(&tb, B, grouped ? p.grp_E * p.grp_b_rows : p.K, p.N, ldb, 64, 64);
    if (rc) return -1;
    if (pair) return launch_pair<false, true>(ta, tb, p, st);
    return wide ? launch<256, false, true>(ta, tb, p, st) : launch<128, false, true>(ta, tb, p, st);
  }
  if (mode == GEMM_TN) {  // A stored [K,M], B stored [K,N]: both MN-major
    rc |= make_map(&ta, A, p.K, p.M, lda, 64, 64);
    rc |= make_map(&tb, B, p.K, p.N, ldb, 64, 64);
    if (rc) return -1;
    if (pair) return launch_pair<true, true>(ta, tb, p, st);
    return wide ? launch<256, true, true>(ta, tb, p, st) : launch<128, true, true>(ta, tb, p, st);
  }
  (void)BN;
  return -1;
}

}  // namespace mt

namespace mt_host {

CUresult encode_tiled(CUtensorMap* map, CUtensorMapDataType dt, uint32_t rank, const void* gaddr,
                      const uint64_t* gdim, const uint64_t* gstride_bytes, const uint32_t* box,
                      CUtensorMapSwizzle swz) {
  typedef CUresult (*Fn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*, const cuuint64_t*,
                         const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                         CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static Fn fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !f)
      return CUDA_ERROR_NOT_FOUND;
    fn = (Fn)f;
  }
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(map, dt, rank, const_cast<void*>(gaddr), (const cuuint64_t*)gdim, (const cuuint64_t*)gstride_bytes,
            (const cuuint32_t*)box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

}  // namespace mt_host
