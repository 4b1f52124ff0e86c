// Persistent tcgen05 GEMM for the layer templates: forward (activation x weight^T),
// dgrad (gradient x weight) and wgrad (gradient^T x activation) of the QKV, O,
// gate-up, down and LM-head projections. The three share one kernel: the operands'
// storage order is expressed in the shared-memory descriptors (K-major or MN-major),
// so no operand is ever transposed in memory.
//
// Per CTA (one per SM, persistent over output tiles of 128 x 256):
//   warp 0      TMA producer: 64-wide K slices of A and B into a 4-stage smem ring
//   warp 1      MMA issuer: one thread issues tcgen05.mma 128x256x16, accumulator in TMEM
//   warps 2..5  epilogue: tcgen05.ld of the accumulator, convert, store to global
// TMEM holds two 256-column fp32 accumulators so the epilogue of one tile overlaps the
// MMAs of the next. The K loop runs in a fixed order and there is no split-K, so every
// output element is produced by one CTA in one order: results are deterministic.
#include <cuda.h>

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
constexpr int NUM_THREADS = 192;
constexpr int TMEM_COLS = 2 * BN;  // two accumulators
constexpr size_t SMEM_BYTES = 1024 /*align slack*/ + STAGES * STAGE_BYTES + 256 /*barriers*/;

struct Params {
  int M, N, K;
  void* C;
  int64_t ldc;
  const float* R;
  int64_t ldr;
  int epi;
  int tiles_m, tiles_n;
  int n_fastest;  // tile order: column tiles vary fastest (else row tiles)
  int* err;
};

// Output tile of linear index `tile`. The wave of CTAs in flight covers consecutive tiles, so
// the operand along the slow dimension is shared by the wave and the one along the fast
// dimension is swept; sweeping the smaller operand keeps it in L2 (see gemm()).
__device__ __forceinline__ void tile_coords(const Params& p, int tile, int& m0, int& n0) {
  if (p.n_fastest) {
    m0 = (tile / p.tiles_n) * BM;
    n0 = (tile % p.tiles_n) * BN;
  } else {
    m0 = (tile % p.tiles_m) * BM;
    n0 = (tile / p.tiles_m) * BN;
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

template <bool A_MN, bool B_MN>
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
  const int num_tiles = p.tiles_m * p.tiles_n;
  const int num_kb = (p.K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 4 * 32);
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
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        int m0, n0;
        tile_coords(p, tile, m0, n0);
        for (int kb = 0; kb < num_kb; ++kb) {
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
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, A_MN, B_MN);
      // K step inside a 64-wide slice: +32 B along a K-major row, +16 rows (2048 B) for MN-major.
      constexpr uint32_t a_kstep = A_MN ? 2048u : 32u;
      constexpr uint32_t b_kstep = B_MN ? 2048u : 32u;
      constexpr uint32_t a_lbo = A_MN ? 8192u : 16u;
      constexpr uint32_t b_lbo = B_MN ? 8192u : 16u;
      int stage = 0;
      uint32_t phase = 0;
      int iter = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++iter) {
        const int acc = iter & 1;
        const uint32_t acc_phase = (iter >> 1) & 1;
        if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1u, p.err, kErrTimeoutAccFree)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&full[stage], phase, p.err, kErrTimeoutTmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_addr(smem + stage * STAGE_BYTES);
          const uint32_t sb = sa + A_TILE_BYTES;
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k) {
            const uint64_t ad = smem_desc_sw128(sa + k * a_kstep, a_lbo, 1024);
            const uint64_t bd = smem_desc_sw128(sb + k * b_kstep, b_lbo, 1024);
            umma_bf16(d_tmem, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
          }
          umma_commit(&empty[stage]);  // frees the smem stage once these MMAs finish
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) umma_commit(&acc_full[acc]);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const int sub = warp & 3;  // TMEM lane quarter this warp may access
    const int row_in_tile = sub * 32 + lane;
    int iter = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++iter) {
      const int acc = iter & 1;
      const uint32_t acc_phase = (iter >> 1) & 1;
      if (!mbar_wait_warp(&acc_full[acc], acc_phase, p.err, kErrTimeoutAccFull)) break;
      tc_fence_after();
      int m_base, n_base;
      tile_coords(p, tile, m_base, n_base);
      const int m = m_base + row_in_tile;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(sub * 32) << 16) + acc * BN;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        __syncwarp();
        tmem_ld_32cols(t_row + c * 32, r);
        tmem_ld_wait();
        const int n = n_base + c * 32;
        const bool in_range = (m < p.M) && (n < p.N);
        const bool full_chunk = (n + 32 <= p.N);
        if (!in_range) {
          // rows/columns past the edge of C: nothing to store
        } else if (p.epi == kEpiStoreBf16) {
          bf16* crow = reinterpret_cast<bf16*>(p.C) + static_cast<int64_t>(m) * p.ldc + n;
          if (full_chunk) {
            uint4* dst = reinterpret_cast<uint4*>(crow);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 v;
              v.x = pack_bf16x2(__uint_as_float(r[8 * q + 0]), __uint_as_float(r[8 * q + 1]));
              v.y = pack_bf16x2(__uint_as_float(r[8 * q + 2]), __uint_as_float(r[8 * q + 3]));
              v.z = pack_bf16x2(__uint_as_float(r[8 * q + 4]), __uint_as_float(r[8 * q + 5]));
              v.w = pack_bf16x2(__uint_as_float(r[8 * q + 6]), __uint_as_float(r[8 * q + 7]));
              dst[q] = v;
            }
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
      tc_fence_before();
      mbar_arrive(&acc_empty[acc]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

// ------------------------------------------------------------------ host side
int g_num_sms = 0;
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
  const void* ks[4] = {reinterpret_cast<const void*>(&gemm_kernel<false, false>),
                       reinterpret_cast<const void*>(&gemm_kernel<false, true>),
                       reinterpret_cast<const void*>(&gemm_kernel<true, false>),
                       reinterpret_cast<const void*>(&gemm_kernel<true, true>)};
  for (const void* k : ks) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(SMEM_BYTES));
    if (e != cudaSuccess) {
      g_init_err = e;
      return;
    }
  }
}

}  // namespace

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
  if (g.b_mn)  // stored [K][N]
    ok = tma_map_2d(&mb, g.B, g.N, g.K, g.ldb, 64, 64);
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
  p.tiles_m = (g.M + BM - 1) / BM;
  p.tiles_n = (g.N + BN - 1) / BN;
  // sweep the smaller operand: with row tiles fastest the wave shares a column tile of B and
  // sweeps A (M x K); with column tiles fastest it shares a row tile of A and sweeps B (N x K)
  p.n_fastest = g.M > g.N ? 1 : 0;
  p.err = err_flag;
  const int tiles = p.tiles_m * p.tiles_n;
  const int grid = tiles < g_num_sms ? tiles : g_num_sms;
  if (!g.a_mn && !g.b_mn)
    gemm_kernel<false, false><<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(ma, mb, p);
  else if (!g.a_mn && g.b_mn)
    gemm_kernel<false, true><<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(ma, mb, p);
  else if (g.a_mn && !g.b_mn)
    gemm_kernel<true, false><<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(ma, mb, p);
  else
    gemm_kernel<true, true><<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(ma, mb, p);
  return cudaGetLastError();
}

}  // namespace mt
