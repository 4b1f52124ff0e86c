// Persistent tcgen05 GEMM for the layer templates: forward (activation x weight^T),
// dgrad (gradient x weight) and wgrad (gradient^T x activation) of the QKV, O,
// gate-up, down and LM-head projections. The three share one kernel: the operands'
// storage order is expressed in the shared-memory descriptors (K-major or MN-major),
// so no operand is ever transposed in memory.
//
// Per CTA (one per SM, persistent over output tiles of 128 x 256):
//   warp 0      TMA producer: 64-wide K slices of A and B into a 4-stage smem ring
//   warp 1      MMA issuer: one elected lane issues tcgen05.mma 128x256x16, accumulator in TMEM
//   warps 2..9  epilogue (two warps per TMEM lane quarter, each half of the tile's columns):
//               tcgen05.ld of the accumulator, convert, store to global; the
//               fused epilogues apply RoPE (QKV projection), SwiGLU (gate-up projection:
//               gate and up rows share one 256-row B tile) or the SwiGLU backward (down
//               projection's data gradient) on the fp32 accumulator before the store
// TMEM holds two 256-column fp32 accumulators so the epilogue of one tile overlaps the
// MMAs of the next.
//
// Last wave split over K. When the tile count is not a multiple of the grid, the tiles of
// the last, partial wave would leave SMs idle. Given a workspace, those tiles' K ranges are
// cut into one contiguous run of k-blocks per CTA (every CTA gets the same share of the
// wave's work). A CTA whose run ends a tile owns that tile; the other CTAs on the tile
// write their fp32 partial sums to their own workspace slot and raise a per-warp flag
// (the launch's epoch); the owner waits for the flags, adds the partials to its
// accumulator in CTA order and runs the tile's epilogue. Every CTA computes its
// contributions before the tile it owns, and contributors have lower indices than the
// owner, so no wait depends on a CTA that is itself waiting on a later one. The split
// depends only on the shape and the SM count, and partials are added in a fixed order:
// results are deterministic and identical between runs.
#include <cuda.h>

#include <atomic>
#include <mutex>

#include "kernels.h"
#include "ptx.cuh"
#include "tma.h"

namespace mt {

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int A_TILE_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_TILE_BYTES = BN * BK * 2;  // 32 KB
constexpr int STAGE_BYTES = A_TILE_BYTES + B_TILE_BYTES;
constexpr int UMMA_K = 16;
constexpr int NUM_THREADS = 320;  // TMA warp, MMA warp, 8 epilogue warps
constexpr int EPI_WARPS = 8;
constexpr int TMEM_COLS = 2 * BN;  // two accumulators
constexpr size_t SMEM_BYTES = 1024 /*align slack*/ + STAGES * STAGE_BYTES + 256 /*barriers*/;
// last-wave split: at most kMaxSplitCtas CTAs, each with one partial slot and one flag per
// epilogue warp; a CTA's run is at least a quarter of a tile's k-blocks, so at most four
// CTAs contribute to a tile besides its owner (which bounds the owner's added reads)
constexpr int kMaxSplitCtas = 256;
constexpr size_t kSplitFlagBytes = kMaxSplitCtas * EPI_WARPS * sizeof(unsigned);
constexpr size_t kSplitSlotFloats = static_cast<size_t>(BM) * BN;
static_assert(kSplitFlagBytes == kGemmFlagBytes, "flag area size shared with the workspace users");
enum { kRoleWhole = 0, kRoleContrib = 1, kRoleOwner = 2 };

struct Params {
  int M, N, K;
  void* C;
  int64_t ldc;
  const float* R;
  int64_t ldr;
  int epi;
  int tiles_m, tiles_n;
  int n_fastest;  // tile order: column tiles vary fastest (else row tiles)
  int bn_out;     // output columns per tile: BN, or BN / 2 when gate and up rows are paired
  int pair_rows;  // paired B tile: rows [n0, n0 + 128) and [pair_rows + n0, ...) (SwiGLU)
  void* C2;
  int64_t ldc2;
  const bf16* G;
  int64_t ldg;
  const float* cs;
  int rope_cols, hd, seq;
  int* err;
  // last-wave split (sk_w == 0: none): tiles [0, dp_tiles) run whole, one CTA each; the
  // remaining tiles' sk_total k-blocks are cut into runs of sk_w per CTA
  int dp_tiles, sk_w, sk_total;
  unsigned* flags;  // [CTA][epilogue warp]
  float* slots;     // [CTA][BM * BN] fp32 partial sums
  unsigned epoch;   // value a flag takes when this launch's partial is in place
};

// One unit of a CTA's work: tile `tile`, k-blocks [k0, k1), and what to do with the sum.
struct Work {
  int tile, k0, k1, role;
};

// The i-th unit of this CTA (tile < 0: none left). Whole tiles first (blockIdx.x, + gridDim.x,
// ...), then the CTA's run of the split wave: its piece of a later tile (a contribution) before
// its piece of an earlier tile (which ends that tile, so the CTA owns it).
template <bool SPLIT>
__device__ __forceinline__ Work work_item(const Params& p, int i, int num_kb) {
  const int G = gridDim.x, b = blockIdx.x;
  const Work none{-1, 0, 0, 0};
  if constexpr (!SPLIT) {
    const int tile = b + i * G;
    return tile < p.tiles_m * p.tiles_n ? Work{tile, 0, num_kb, kRoleWhole} : none;
  }
  const int n_whole = b < p.dp_tiles ? (p.dp_tiles - 1 - b) / G + 1 : 0;
  if (i < n_whole) return {b + i * G, 0, num_kb, kRoleWhole};
  const int s = b * p.sk_w, e = min(s + p.sk_w, p.sk_total);
  if (s >= e) return none;
  const int ta = s / num_kb, tb = (e - 1) / num_kb, j = i - n_whole;
  if (ta == tb) {
    if (j > 0) return none;
    return {p.dp_tiles + ta, s - ta * num_kb, e - ta * num_kb, e == (ta + 1) * num_kb ? kRoleOwner : kRoleContrib};
  }
  if (j == 0) return {p.dp_tiles + tb, 0, e - tb * num_kb, kRoleContrib};
  if (j == 1) return {p.dp_tiles + ta, s - ta * num_kb, num_kb, kRoleOwner};
  return none;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* ptr) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(unsigned* ptr, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(ptr), "r"(v) : "memory");
}

// Partial sums an owner adds to its accumulator: the slots of n consecutive CTAs from `base`,
// in CTA order.
struct SplitSrc {
  const float* base;
  int n;
};

// Owner side: wait (bounded) until every contributing CTA's warp that wrote this warp's rows
// and columns has raised its flag. On a timeout the error flag is set (the launch's result is
// then invalid) and the wait ends.
__device__ __forceinline__ void split_sources(const Params& p, int tile, int num_kb, int epi_warp, SplitSrc& src) {
  const int t = tile - p.dp_tiles;
  const int c_first = (t * num_kb) / p.sk_w, c_last = ((t + 1) * num_kb - 1) / p.sk_w;
  src.base = p.slots + static_cast<size_t>(c_first) * kSplitSlotFloats;
  src.n = c_last - c_first;
  for (int c = c_first; c < c_last; ++c) {
    const unsigned* f = p.flags + c * EPI_WARPS + epi_warp;
    if (ld_acquire_u32(f) == p.epoch) continue;
    const unsigned long long t0 = global_ns();
    for (uint32_t it = 1;; ++it) {
      __nanosleep(64);
      if (ld_acquire_u32(f) == p.epoch) break;
      if ((it & 63u) == 0) {
        if (*reinterpret_cast<volatile int*>(p.err) != 0) break;
        if (global_ns() - t0 > kWaitLimitNs) {
          atomicCAS(p.err, 0, kErrTimeoutSplit);
          break;
        }
      }
    }
  }
  __syncwarp();
}

// Slot layout, in float4 units: [32-column chunk][group of 4 columns][tile row], so the 32 lanes
// of a warp (32 consecutive rows) move 512 contiguous bytes per access.
__device__ __forceinline__ size_t slot_f4(int chunk, int v, int row) {
  return (static_cast<size_t>(chunk) * 8 + v) * BM + row;
}

__device__ __forceinline__ void add_partials(const SplitSrc* src, int chunk, int row, uint32_t (&r)[32]) {
  if (!src) return;
  for (int i = 0; i < src->n; ++i) {
    const float4* q = reinterpret_cast<const float4*>(src->base + static_cast<size_t>(i) * kSplitSlotFloats);
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      const float4 x = __ldcg(q + slot_f4(chunk, v, row));
      r[4 * v + 0] = __float_as_uint(__uint_as_float(r[4 * v + 0]) + x.x);
      r[4 * v + 1] = __float_as_uint(__uint_as_float(r[4 * v + 1]) + x.y);
      r[4 * v + 2] = __float_as_uint(__uint_as_float(r[4 * v + 2]) + x.z);
      r[4 * v + 3] = __float_as_uint(__uint_as_float(r[4 * v + 3]) + x.w);
    }
  }
}

// The i-th (of BN / 64) 32-column accumulator chunk that the epilogue warps of column half
// `half` read: the lower or upper half of the tile, except in the SwiGLU epilogue, whose warps
// take matching gate and up chunks (two from each half).
__device__ __forceinline__ int epi_chunk(const Params& p, int half, int i) {
  if (p.epi == kEpiSwigluBf16) return i < 2 ? half * 2 + i : BN / 64 + half * 2 + (i - 2);
  return half * (BN / 64) + i;
}

// Contributor side: the accumulator chunks the owner's warp of the same rows and column half
// will read, raw fp32, into the CTA's slot; then every lane fences its stores and lane 0
// raises the warp's flag.
__device__ __forceinline__ void epilogue_contrib(const Params& p, uint32_t t_row, int row, int half, int epi_warp) {
  float* slot = p.slots + static_cast<size_t>(blockIdx.x) * kSplitSlotFloats;
#pragma unroll 1
  for (int i = 0; i < BN / 64; ++i) {
    const int c = epi_chunk(p, half, i);
    uint32_t r[32];
    __syncwarp();
    tmem_ld_32cols(t_row + c * 32, r);
    tmem_ld_wait();
    float4* q = reinterpret_cast<float4*>(slot);
#pragma unroll
    for (int v = 0; v < 8; ++v)
      __stcg(q + slot_f4(c, v, row), make_float4(__uint_as_float(r[4 * v + 0]), __uint_as_float(r[4 * v + 1]),
                                __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3])));
  }
  __threadfence();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) st_release_u32(p.flags + blockIdx.x * EPI_WARPS + epi_warp, p.epoch);
}

// Output tile of linear index `tile`. Tiles are visited in groups of kGroup tiles along the
// "fast" dimension (rows, or columns when n_fastest): inside a group the fast index varies
// first, then the slow one. A wave of CTAs in flight then covers kGroup fast tiles x a few slow
// tiles, so the group's slice of the fast-dimension operand stays in L2 while the other operand
// is streamed once per group (instead of the whole fast-dimension operand once per wave).
constexpr int kGroup = 8;
__device__ __forceinline__ void tile_coords(const Params& p, int tile, int& m0, int& n0) {
  const int n_fast = p.n_fastest ? p.tiles_n : p.tiles_m;  // tiles along the fast dimension
  const int n_slow = p.n_fastest ? p.tiles_m : p.tiles_n;
  const int per_group = kGroup * n_slow;
  const int g = tile / per_group;
  const int in_group = tile - g * per_group;
  const int width = min(kGroup, n_fast - g * kGroup);  // the last group may be narrower
  const int fast = g * kGroup + in_group % width;
  const int slow = in_group / width;
  if (p.n_fastest) {
    m0 = slow * BM;
    n0 = fast * p.bn_out;
  } else {
    m0 = fast * BM;
    n0 = slow * p.bn_out;
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void store_bf16x32(bf16* dst, const float (&v)[32]) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 u;
    u.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
    u.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
    u.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
    u.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
    d[q] = u;
  }
}

__device__ __forceinline__ float bf16_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// Plain epilogues: C = acc (bf16 or fp32), or C = R + acc (fp32).
__device__ __forceinline__ void epilogue_store(const Params& p, uint32_t t_row, int m, int n_base, int half,
                                               const SplitSrc* src, int row) {
#pragma unroll 1
  for (int c = half * (BN / 64); c < (half + 1) * (BN / 64); ++c) {
    uint32_t r[32];
    __syncwarp();
    tmem_ld_32cols(t_row + c * 32, r);
    tmem_ld_wait();
    add_partials(src, c, row, r);
    const int n = n_base + c * 32;
    const bool in_range = (m < p.M) && (n < p.N);
    const bool full_chunk = (n + 32 <= p.N);
    if (!in_range) continue;  // rows/columns past the edge of C: nothing to store
    if (p.epi == kEpiStoreBf16) {
      bf16* crow = reinterpret_cast<bf16*>(p.C) + static_cast<int64_t>(m) * p.ldc + n;
      if (full_chunk) {
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
        store_bf16x32(crow, v);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (n + j < p.N) crow[j] = __float2bfloat16_rn(__uint_as_float(r[j]));
      }
    } else {
      float* crow = reinterpret_cast<float*>(p.C) + static_cast<int64_t>(m) * p.ldc + n;
      const float* rrow = (p.epi == kEpiAddF32) ? p.R + static_cast<int64_t>(m) * p.ldr + n : nullptr;
      if (full_chunk) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float4 v = make_float4(__uint_as_float(r[4 * q + 0]), __uint_as_float(r[4 * q + 1]),
                                 __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
          if (rrow) {
            const float4 rv = reinterpret_cast<const float4*>(rrow)[q];
            v.x += rv.x;
            v.y += rv.y;
            v.z += rv.z;
            v.w += rv.w;
          }
          reinterpret_cast<float4*>(crow)[q] = v;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (n + j < p.N) {
            float v = __uint_as_float(r[j]);
            if (rrow) v += rrow[j];
            crow[j] = v;
          }
        }
      }
    }
  }
}

// RoPE on the accumulator (rotate-half): within each head, column i < hd/2 pairs with
// column i + hd/2; a 256-column tile holds whole heads (hd = 64 or 128 divides 256), so both
// halves of a pair are in the same thread's TMEM row. The tile is walked as 4 pairs of
// 32-column chunks (lo, lo + hd/64 chunks).
__device__ __forceinline__ void epilogue_rope(const Params& p, uint32_t t_row, int m, int n_base, int half_tile,
                                              const SplitSrc* src, int row) {
  const int hc = p.hd >> 6;  // 32-column chunks per half head
  const int half = p.hd >> 1;
  const int pos = m % p.seq;
#pragma unroll 1
  for (int pi = half_tile * (BN / 128); pi < (half_tile + 1) * (BN / 128); ++pi) {
    const int lo = (pi / hc) * 2 * hc + (pi % hc), hi = lo + hc;
    uint32_t ra[32], rb[32];
    __syncwarp();
    tmem_ld_32cols(t_row + lo * 32, ra);
    tmem_ld_32cols(t_row + hi * 32, rb);
    tmem_ld_wait();
    add_partials(src, lo, row, ra);
    add_partials(src, hi, row, rb);
    const int n_lo = n_base + lo * 32;
    if (m >= p.M || n_lo >= p.N) continue;  // N is a multiple of hd: a pair is in or out whole
    float a[32], b[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      a[j] = __uint_as_float(ra[j]);
      b[j] = __uint_as_float(rb[j]);
    }
    if (n_lo < p.rope_cols) {
      const int i0 = n_lo % p.hd;  // rotation index of column j is i0 + j (< hd/2)
      const float4* c4 = reinterpret_cast<const float4*>(p.cs + (static_cast<int64_t>(pos) * half + i0) * 2);
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const float4 c = __ldg(c4 + j / 2);  // cos_i, sin_i, cos_{i+1}, sin_{i+1}
        const float a0 = a[j] * c.x - b[j] * c.y, b0 = b[j] * c.x + a[j] * c.y;
        const float a1 = a[j + 1] * c.z - b[j + 1] * c.w, b1 = b[j + 1] * c.z + a[j + 1] * c.w;
        a[j] = a0;
        b[j] = b0;
        a[j + 1] = a1;
        b[j + 1] = b1;
      }
    }
    bf16* crow = reinterpret_cast<bf16*>(p.C) + static_cast<int64_t>(m) * p.ldc;
    store_bf16x32(crow + n_lo, a);
    store_bf16x32(crow + n_lo + (hi - lo) * 32, b);
  }
}

// silu(g) = g sigmoid(g) with the fast exponential and division: both are exact to a few
// ulp of fp32, far below the bf16 rounding of the result; for g < -87 the denominator
// overflows to +inf and the quotient is 0, the limit of silu.
__device__ __forceinline__ float sigmoid_of(float g) { return __fdividef(1.f, 1.f + __expf(-g)); }
__device__ __forceinline__ float silu_of(float g) { return __fdividef(g, 1.f + __expf(-g)); }

// SwiGLU forward: accumulator columns [0, 128) are the gate projection of output columns
// n_base + [0, 128), columns [128, 256) the up projection of the same columns.
__device__ __forceinline__ void epilogue_swiglu(const Params& p, uint32_t t_row, int m, int n_base, int half,
                                                const SplitSrc* src, int row) {
#pragma unroll 1
  for (int c = half * (BN / 128); c < (half + 1) * (BN / 128); ++c) {
    uint32_t rg[32], ru[32];
    __syncwarp();
    tmem_ld_32cols(t_row + c * 32, rg);
    tmem_ld_32cols(t_row + BN / 2 + c * 32, ru);
    tmem_ld_wait();
    add_partials(src, c, row, rg);
    add_partials(src, BN / 64 + c, row, ru);
    const int n = n_base + c * 32;
    if (m >= p.M || n >= p.N) continue;
    float g[32], u[32], o[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      g[j] = bf16_round(__uint_as_float(rg[j]));
      u[j] = bf16_round(__uint_as_float(ru[j]));
      o[j] = silu_of(g[j]) * u[j];
    }
    bf16* arow = reinterpret_cast<bf16*>(p.C) + static_cast<int64_t>(m) * p.ldc + n;
    bf16* grow = p.C2 ? reinterpret_cast<bf16*>(p.C2) + static_cast<int64_t>(m) * p.ldc2 + n : nullptr;
    if (n + 32 <= p.N) {
      store_bf16x32(arow, o);
      if (grow) {
        store_bf16x32(grow, g);
        store_bf16x32(grow + p.N, u);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (n + j < p.N) {
          arow[j] = __float2bfloat16_rn(o[j]);
          if (grow) {
            grow[j] = __float2bfloat16_rn(g[j]);
            grow[p.N + j] = __float2bfloat16_rn(u[j]);
          }
        }
      }
    }
  }
}

// [g | u] of one 32-column chunk, as raw bf16 pairs, fetched ahead of its use.
struct GuChunk {
  uint4 g[4], u[4];
};

__device__ __forceinline__ void fetch_gu(const Params& p, int m, int n, GuChunk& r) {
  if (m < p.M && n + 32 <= p.N) {
    const uint4* gp = reinterpret_cast<const uint4*>(p.G + static_cast<int64_t>(m) * p.ldg + n);
    const uint4* up = reinterpret_cast<const uint4*>(p.G + static_cast<int64_t>(m) * p.ldg + p.N + n);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      r.g[q] = __ldg(gp + q);
      r.u[q] = __ldg(up + q);
    }
  }
}

__device__ __forceinline__ void unpack_bf16x32(const uint4 (&w)[4], float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t x[4] = {w[q].x, w[q].y, w[q].z, w[q].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[8 * q + 2 * j] = __uint_as_float(x[j] << 16);
      v[8 * q + 2 * j + 1] = __uint_as_float(x[j] & 0xffff0000u);
    }
  }
}

// SwiGLU backward on dact = the accumulator: dg = dact * u * s (1 + g (1 - s)), du = dact * g * s
// with s = sigmoid(g), written to C = [dg | du]. `next` holds the [g | u] of this warp's first
// chunk (fetched before the accumulator was ready); each chunk fetches the next one's.
__device__ __forceinline__ void epilogue_swiglu_bwd(const Params& p, uint32_t t_row, int m, int n_base, int half,
                                                    GuChunk& next, const SplitSrc* src, int row) {
  const int c0 = half * (BN / 64), c1 = c0 + BN / 64;
#pragma unroll 1
  for (int c = c0; c < c1; ++c) {
    const GuChunk cur = next;
    const int n = n_base + c * 32;
    if (c + 1 < c1) fetch_gu(p, m, n + 32, next);
    uint32_t r[32];
    __syncwarp();
    tmem_ld_32cols(t_row + c * 32, r);
    tmem_ld_wait();
    add_partials(src, c, row, r);
    if (m >= p.M || n >= p.N) continue;
    const bf16* grow = p.G + static_cast<int64_t>(m) * p.ldg + n;
    bf16* drow = reinterpret_cast<bf16*>(p.C) + static_cast<int64_t>(m) * p.ldc + n;
    float g[32], u[32];
    const bool full_chunk = n + 32 <= p.N;
    if (full_chunk) {
      unpack_bf16x32(cur.g, g);
      unpack_bf16x32(cur.u, u);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        g[j] = n + j < p.N ? __bfloat162float(grow[j]) : 0.f;
        u[j] = n + j < p.N ? __bfloat162float(grow[p.N + j]) : 0.f;
      }
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float d = __uint_as_float(r[j]);
      const float sg = sigmoid_of(g[j]);
      const float dg = d * u[j] * sg * (1.f + g[j] * (1.f - sg));
      u[j] = d * g[j] * sg;
      g[j] = dg;
    }
    if (full_chunk) {
      store_bf16x32(drow, g);
      store_bf16x32(drow + p.N, u);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (n + j < p.N) {
          drow[j] = __float2bfloat16_rn(g[j]);
          drow[p.N + j] = __float2bfloat16_rn(u[j]);
        }
      }
    }
  }
}

template <bool A_MN, bool B_MN, bool SPLIT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b, Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* full = bars;                 // [STAGES]  TMA -> MMA
  uint64_t* empty = bars + STAGES;       // [STAGES]  MMA -> TMA
  uint64_t* acc_full = bars + 2 * STAGES;   // [2]   MMA -> epilogue
  uint64_t* acc_empty = bars + 2 * STAGES + 2;  // [2] epilogue -> MMA
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_kb = (p.K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], EPI_WARPS);
    }
    fence_mbar_init();
    tma_prefetch_map(&map_a);
    tma_prefetch_map(&map_b);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int i = 0; ok; ++i) {
        const Work w = work_item<SPLIT>(p, i, num_kb);
        if (w.tile < 0) break;
        int m0, n0;
        tile_coords(p, w.tile, m0, n0);
        for (int kb = w.k0; kb < w.k1; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, p.err, kErrTimeoutSmemFree)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * STAGE_BYTES;
          uint8_t* sb = sa + A_TILE_BYTES;
          mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
          const int k0 = kb * BK;
          if (A_MN) {
            tma_load_2d(sa, &map_a, &full[stage], m0, k0);
            tma_load_2d(sa + 8192, &map_a, &full[stage], m0 + 64, k0);
          } else {
            tma_load_2d(sa, &map_a, &full[stage], k0, m0);
          }
          if (B_MN) {
#pragma unroll
            for (int j = 0; j < 4; ++j) tma_load_2d(sb + j * 8192, &map_b, &full[stage], n0 + 64 * j, k0);
          } else if (p.pair_rows) {  // 128-row boxes: gate rows, then the matching up rows
            tma_load_2d(sb, &map_b, &full[stage], k0, n0);
            tma_load_2d(sb + B_TILE_BYTES / 2, &map_b, &full[stage], k0, p.pair_rows + n0);
          } else {
            tma_load_2d(sb, &map_b, &full[stage], k0, n0);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop with warp-uniform descriptors; one elected lane issues
    // each MMA and commit (a lone thread in a lane-0 branch issues measurably slower while the
    // epilogue warps load TMEM).
    {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, A_MN, B_MN);
      // K step inside a 64-wide slice: +32 B along a K-major row, +16 rows (2048 B) for MN-major.
      constexpr uint32_t a_kstep = A_MN ? 2048u : 32u;
      constexpr uint32_t b_kstep = B_MN ? 2048u : 32u;
      constexpr uint32_t a_lbo = A_MN ? 8192u : 16u;
      constexpr uint32_t b_lbo = B_MN ? 8192u : 16u;
      const uint64_t a_desc0 = smem_desc_sw128(smem_addr(smem), a_lbo, 1024);
      const uint64_t b_desc0 = smem_desc_sw128(smem_addr(smem + A_TILE_BYTES), b_lbo, 1024);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int iter = 0; ok; ++iter) {
        const Work w = work_item<SPLIT>(p, iter, num_kb);
        if (w.tile < 0) break;
        const int acc = iter & 1;
        const uint32_t acc_phase = (iter >> 1) & 1;
        if (!mbar_wait_warp(&acc_empty[acc], acc_phase ^ 1u, p.err, kErrTimeoutAccFree)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = w.k0; kb < w.k1; ++kb) {
          if (!mbar_wait_warp(&full[stage], phase, p.err, kErrTimeoutTmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = desc_advance(a_desc0, stage * STAGE_BYTES);
          const uint64_t bd = desc_advance(b_desc0, stage * STAGE_BYTES);
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k)
            umma_bf16_warp(d_tmem, desc_advance(ad, k * a_kstep), desc_advance(bd, k * b_kstep), idesc,
                           (kb > (SPLIT ? w.k0 : 0) || k > 0) ? 1u : 0u);
          umma_commit_warp(&empty[stage]);  // frees the smem stage once these MMAs finish
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) umma_commit_warp(&acc_full[acc]);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..9)
    const int sub = warp & 3;          // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;  // which half of the tile's columns it takes
    const int row_in_tile = sub * 32 + lane;
    const int epi_warp = warp - 2;
    for (int iter = 0;; ++iter) {
      const Work w = work_item<SPLIT>(p, iter, num_kb);
      if (w.tile < 0) break;
      const int acc = iter & 1;
      const uint32_t acc_phase = (iter >> 1) & 1;
      int m_base, n_base;
      tile_coords(p, w.tile, m_base, n_base);
      const int m = m_base + row_in_tile;
      GuChunk gu_next;  // the SwiGLU backward reads [g | u]: start before the accumulator is ready
      if (p.epi == kEpiSwigluBwdBf16 && (!SPLIT || w.role != kRoleContrib)) fetch_gu(p, m, n_base + half * (BN / 2), gu_next);
      SplitSrc src;
      const SplitSrc* sp = nullptr;
      if constexpr (SPLIT) {
        if (w.role == kRoleOwner) {
          split_sources(p, w.tile, num_kb, epi_warp, src);
          sp = &src;
        }
      }
      if (!mbar_wait_warp(&acc_full[acc], acc_phase, p.err, kErrTimeoutAccFull)) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(sub * 32) << 16) + acc * BN;
      if (SPLIT && w.role == kRoleContrib) {
        epilogue_contrib(p, t_row, row_in_tile, half, epi_warp);
      } else if (p.epi == kEpiRopeBf16) {
        epilogue_rope(p, t_row, m, n_base, half, sp, row_in_tile);
      } else if (p.epi == kEpiSwigluBf16) {
        epilogue_swiglu(p, t_row, m, n_base, half, sp, row_in_tile);
      } else if (p.epi == kEpiSwigluBwdBf16) {
        epilogue_swiglu_bwd(p, t_row, m, n_base, half, gu_next, sp, row_in_tile);
      } else {
        epilogue_store(p, t_row, m, n_base, half, sp, row_in_tile);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

// ------------------------------------------------------------------ host side
int g_num_sms = 0;
std::atomic<unsigned> g_epoch{0};  // launch epochs of split GEMMs: unique per process
std::once_flag g_once;
cudaError_t g_init_err = cudaSuccess;

void init_once() {
  cudaError_t e = tma_init();
  if (e != cudaSuccess) {
    g_init_err = e;
    return;
  }
  int dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
  const void* ks[8] = {reinterpret_cast<const void*>(&gemm_kernel<false, false, false>),
                       reinterpret_cast<const void*>(&gemm_kernel<false, true, false>),
                       reinterpret_cast<const void*>(&gemm_kernel<true, false, false>),
                       reinterpret_cast<const void*>(&gemm_kernel<true, true, false>),
                       reinterpret_cast<const void*>(&gemm_kernel<false, false, true>),
                       reinterpret_cast<const void*>(&gemm_kernel<false, true, true>),
                       reinterpret_cast<const void*>(&gemm_kernel<true, false, true>),
                       reinterpret_cast<const void*>(&gemm_kernel<true, true, true>)};
  for (const void* k : ks) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(SMEM_BYTES));
    if (e != cudaSuccess) {
      g_init_err = e;
      return;
    }
  }
}

}  // namespace

uint64_t gemm_workspace_bytes() { return kSplitFlagBytes + static_cast<uint64_t>(kMaxSplitCtas) * kSplitSlotFloats * 4; }

int gemm_num_sms() {
  std::call_once(g_once, init_once);
  return g_num_sms;
}

cudaError_t gemm(const GemmArgs& g, int* err_flag, cudaStream_t stream) {
  std::call_once(g_once, init_once);
  if (g_init_err != cudaSuccess) return g_init_err;
  if (g.M <= 0 || g.N <= 0 || g.K <= 0) return cudaErrorInvalidValue;
  if ((g.lda % 8) || (g.ldb % 8) || (g.ldc % 8) || (g.epi == kEpiAddF32 && (g.ldr % 4))) return cudaErrorInvalidValue;
  if ((reinterpret_cast<uintptr_t>(g.A) | reinterpret_cast<uintptr_t>(g.B) | reinterpret_cast<uintptr_t>(g.C)) & 15)
    return cudaErrorMisalignedAddress;
  CUtensorMap ma, mb;
  bool ok;
  if (g.a_mn)  // stored [K][M]
    ok = tma_map_2d(&ma, g.A, g.M, g.K, g.lda, 64, 64);
  else  // stored [M][K]
    ok = tma_map_2d(&ma, g.A, g.K, g.M, g.lda, 64, BM);
  if (!ok) return cudaErrorInvalidValue;
  const bool paired = g.epi == kEpiSwigluBf16;
  if (g.epi == kEpiRopeBf16) {
    if ((g.hd != 64 && g.hd != 128) || g.N % g.hd || g.rope_cols % g.hd || g.rope_cols < 0 || g.rope_cols > g.N ||
        g.seq <= 0 || !g.cs || (reinterpret_cast<uintptr_t>(g.cs) & 15))
      return cudaErrorInvalidValue;
  } else if (paired) {
    if (g.a_mn || g.b_mn || g.N % 8 || (g.C2 && (g.ldc2 % 8 || g.ldc2 < 2 * static_cast<int64_t>(g.N) ||
                                                 (reinterpret_cast<uintptr_t>(g.C2) & 15))))
      return cudaErrorInvalidValue;
  } else if (g.epi == kEpiSwigluBwdBf16) {
    if (!g.G || g.N % 8 || g.ldg % 8 || g.ldg < 2 * static_cast<int64_t>(g.N) || g.ldc < 2 * static_cast<int64_t>(g.N) ||
        (reinterpret_cast<uintptr_t>(g.G) & 15))
      return cudaErrorInvalidValue;
  } else if (g.epi < kEpiStoreBf16 || g.epi > kEpiAddF32) {
    return cudaErrorInvalidValue;
  }
  if (g.b_mn)  // stored [K][N]
    ok = tma_map_2d(&mb, g.B, g.N, g.K, g.ldb, 64, 64);
  else if (paired)  // stored [2N][K]: gate rows [0, N), up rows [N, 2N); 128-row boxes
    ok = tma_map_2d(&mb, g.B, g.K, 2 * static_cast<int64_t>(g.N), g.ldb, 64, BN / 2);
  else  // stored [N][K]
    ok = tma_map_2d(&mb, g.B, g.K, g.N, g.ldb, 64, BN);
  if (!ok) return cudaErrorInvalidValue;

  Params p;
  p.M = g.M;
  p.N = g.N;
  p.K = g.K;
  p.C = g.C;
  p.ldc = g.ldc;
  p.R = g.R;
  p.ldr = g.ldr;
  p.epi = g.epi;
  p.bn_out = paired ? BN / 2 : BN;
  p.pair_rows = paired ? g.N : 0;
  p.C2 = g.C2;
  p.ldc2 = g.ldc2;
  p.G = g.G;
  p.ldg = g.ldg;
  p.cs = g.cs;
  p.rope_cols = g.rope_cols;
  p.hd = g.hd;
  p.seq = g.seq;
  p.tiles_m = (g.M + BM - 1) / BM;
  p.tiles_n = (g.N + p.bn_out - 1) / p.bn_out;
  // tile order (see tile_coords): the fast-dimension operand is read about once, the other once
  // per group of kGroup fast tiles; pick the orientation with the smaller estimated traffic
  {
    const double a_bytes = 2.0 * g.M * g.K, b_bytes = 2.0 * (paired ? 2.0 * g.N : g.N) * g.K;
    const double groups_m = (p.tiles_m + kGroup - 1) / kGroup, groups_n = (p.tiles_n + kGroup - 1) / kGroup;
    const double rows_fast = a_bytes + groups_m * b_bytes, cols_fast = b_bytes + groups_n * a_bytes;
    p.n_fastest = cols_fast < rows_fast ? 1 : 0;
  }
  p.err = err_flag;
  const int tiles = p.tiles_m * p.tiles_n;
  int grid = tiles < g_num_sms ? tiles : g_num_sms;
  p.dp_tiles = tiles;
  p.sk_w = p.sk_total = 0;
  p.flags = nullptr;
  p.slots = nullptr;
  p.epoch = 0;
  const int kb = (g.K + BK - 1) / BK;
  const int split_grid = g_num_sms < kMaxSplitCtas ? g_num_sms : kMaxSplitCtas;
  const int rem = tiles % split_grid;
  // Split the last wave only where it was measured to pay on GB300: a tile of at least 128
  // k-blocks and a last wave at most half full. The owner's epilogue runs after its own previous
  // tile's epilogue, so with shorter tiles the exposed epilogues cost what the split saves
  // (7B layer shapes, K = 4096: 0.3-2.8 % slower split; weight gradients with K = 8192 and a
  // last wave of 8-56 tiles: 1.3-4.4 % faster).
  if (g.ws && rem != 0 && 2 * rem <= split_grid && kb >= 128) {
    p.dp_tiles = tiles - rem;
    p.sk_total = rem * kb;
    const int even = (p.sk_total + split_grid - 1) / split_grid, quarter = (kb + 3) / 4;
    p.sk_w = even > quarter ? even : quarter;
    p.flags = static_cast<unsigned*>(g.ws);
    p.slots = reinterpret_cast<float*>(static_cast<uint8_t*>(g.ws) + kSplitFlagBytes);
    p.epoch = g_epoch.fetch_add(1u) + 1u;
    if (p.epoch == 0) p.epoch = g_epoch.fetch_add(1u) + 1u;  // 0 is the cleared value
    grid = split_grid;
  }
  const bool split = p.sk_w > 0;
  if (!g.a_mn && !g.b_mn)
    (split ? gemm_kernel<false, false, true> : gemm_kernel<false, false, false>)<<<grid, NUM_THREADS, SMEM_BYTES,
                                                                                     stream>>>(ma, mb, p);
  else if (!g.a_mn && g.b_mn)
    (split ? gemm_kernel<false, true, true> : gemm_kernel<false, true, false>)<<<grid, NUM_THREADS, SMEM_BYTES,
                                                                                   stream>>>(ma, mb, p);
  else if (g.a_mn && !g.b_mn)
    (split ? gemm_kernel<true, false, true> : gemm_kernel<true, false, false>)<<<grid, NUM_THREADS, SMEM_BYTES,
                                                                                   stream>>>(ma, mb, p);
  else
    (split ? gemm_kernel<true, true, true> : gemm_kernel<true, true, false>)<<<grid, NUM_THREADS, SMEM_BYTES,
                                                                                 stream>>>(ma, mb, p);
  return cudaGetLastError();
}

}  // namespace mt
