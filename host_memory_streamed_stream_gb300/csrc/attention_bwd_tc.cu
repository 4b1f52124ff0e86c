// Causal grouped-query flash attention backward on the tcgen05 tensor cores.
//
// Deterministic, no atomics:
//  * lsd[b, n, i] = (-lse2[b, n, i], -delta[b, n, i]), delta = sum_d dO[i, n, d] O[i, n, d]
//    (HD/8 lanes per row), padded to a multiple of 128 rows with (-inf, -0): past the end of
//    the sequence every probability is then exactly 0 with no mask, and the causal mask is
//    only evaluated on tiles that straddle the diagonal. Stored negated, the pairs enter the
//    elementwise step as addends of packed fp32x2 operations (2^(S scale - lse2) as one fused
//    multiply-add per pair of scores, dP - delta as one add)
//  * dK/dV, KV-outer: one CTA per (128-key tile, kv head, sequence) walks every 128-query
//    tile of every query head of its group in a fixed order:
//        S^T  = K Q^T,  dP^T = V dO^T                         (TMEM, 128 x 128 each)
//        P^T  = exp2(S^T log2(e)/sqrt(hd) - lse2),  dS^T = P^T (dP^T - delta)
//        dV  += P^T dO,  dK += dS^T Q                         (TMEM accumulators)
//  * dQ, Q-outer: one CTA per (128-query tile, query head, sequence) walks the 128-key tiles:
//        S = Q K^T,  dP = dO V^T,  dS = P (dP - delta),  dQ += dS K
// Every tile is 128 x 128: the score MMAs have N = 128 (at N = 64 the two shared-memory
// operands of each MMA need more bytes per cycle than shared memory gives; only dK/dV's dP^T is
// issued as two N = 64 halves, for the schedule described with that kernel), and every TMA box
// is 128 rows high (the TMA issues far more bytes per cycle with tall boxes).
// Roles per CTA: warp 0 TMA, warp 1 MMA issuer (all 32 lanes, one elected), warps 2..9 the
// elementwise step: each TMEM lane (one key row, resp. one query row) is shared by two warps,
// and each warp takes 32 of the first 64 score columns and then 32 of the last 64 (the step
// needs no row reductions: lse2 and delta are precomputed). Eight warps rather than sixteen:
// every hand-off between the MMA issuer and these warps waits for all of them, and with half as
// many warps each doing twice the work the hand-offs are shorter (7B shapes 763 -> 786 TFLOP/s). They write P^T / dS^T (dQ kernel: dS) as bf16 pairs back
// into TMEM over the scores they came from, where the accumulating MMAs read them as their A
// operand. The tile's accumulating MMAs over its first 64 columns start as soon as every warp
// has finished those columns, while the warps work on the last 64. TMEM (512 columns) holds two
// score slots next to the two accumulators, so the next tile's score MMAs overlap this tile's
// elementwise step (the kernels below say how each one reuses its slots; MMAs of one thread run
// in issue order). The MMA warp issues as a whole warp with one elected lane. Every wait is
// bounded (error flag on timeout).
#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"
#include "tile_order.cuh"
#include "tma.h"

namespace mt {

namespace {

constexpr int kThreads = 320;       // TMA warp, MMA warp, 8 elementwise warps
constexpr int kElem = 256;          // elementwise threads
constexpr int kCols = 32;           // score columns an elementwise warp takes per half tile
constexpr int kParts = kElem / 128;  // elementwise warps on each TMEM lane quadrant
constexpr int kElemWarps = kElem / 32;  // arrivals per barrier phase (one elected lane per warp)
constexpr int kSlice128 = 128 * 128;  // bytes of a [128 rows][64 bf16] swizzle-atom-wide slice

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float ex2(float x) {  // hardware 2^x (ex2.approx, flush to zero)
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Pack the 16 values v[o .. o + 15] into 8 bf16 pairs and store them to 8 TMEM columns of this
// thread's lane (the A-operand layout: element k of a row in column k/2, even k in the low half).
__device__ __forceinline__ void store_pairs16(uint32_t taddr, const float (&v)[kCols], int o) {
  uint32_t w[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) w[c] = pack_bf16(v[o + 2 * c], v[o + 2 * c + 1]);
  tmem_st_8cols(taddr, w);
}

// Two 32-column TMEM loads (S and dP of one row) behind a single wait.
__device__ __forceinline__ void tmem_ld_2x32f(uint32_t ta, uint32_t tb, float (&a)[kCols], float (&b)[kCols]) {
  uint32_t ra[32], rb[32];
  tmem_ld_32cols(ta, ra);
  tmem_ld_32cols(tb, rb);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    a[i] = __uint_as_float(ra[i]);
    b[i] = __uint_as_float(rb[i]);
  }
}

template <int W>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[W]) {
  uint32_t r[W];
  if constexpr (W == 16) tmem_ld_16cols(taddr, r);
  else tmem_ld_8cols(taddr, r);
#pragma unroll
  for (int i = 0; i < W; ++i) v[i] = __uint_as_float(r[i]);
}

template <int W>
__device__ __forceinline__ void store_bf16_cols(bf16* dst, const float (&v)[W]) {
#pragma unroll
  for (int q = 0; q < W / 8; ++q) {
    uint4 u;
    u.x = pack_bf16(v[8 * q + 0], v[8 * q + 1]);
    u.y = pack_bf16(v[8 * q + 2], v[8 * q + 3]);
    u.z = pack_bf16(v[8 * q + 4], v[8 * q + 5]);
    u.w = pack_bf16(v[8 * q + 6], v[8 * q + 7]);
    reinterpret_cast<uint4*>(dst)[q] = u;
  }
}

// (cos, sin) of the HD/8 rotation indices [part*HD/8, +HD/8) at position `pos`, from the table
// fp32 [seq][HD/2][2], as HD/16 float4 = two pairs each. Issued before the final accumulator
// wait so the loads overlap the last MMAs.
template <int HD>
__device__ __forceinline__ void load_rotation(const float* cs, int pos, int part, float4 (&rot)[HD / 16]) {
  const float4* r = reinterpret_cast<const float4*>(cs + static_cast<int64_t>(pos) * HD + 2 * part * (HD / 8));
#pragma unroll
  for (int k = 0; k < HD / 16; ++k) rot[k] = __ldg(r + k);
}

// Store one TMEM lane's fp32 row (HD columns), times `scale`, as bf16 to dst (if `store`). Part
// `part` (0..3; each of the lane's warps takes two) is columns [part*HD/8, +HD/8) and the same
// HD/2 further on, which are the rotation pairs of rotate-half RoPE: with `rot` (from load_rotation) the
// transpose rotation is applied on the way out (the backward of the RoPE that the forward
// applied to q and k).
template <int HD>
__device__ __forceinline__ void tmem_row_out(uint32_t taddr, int part, float scale, bf16* dst, bool store,
                                             const float4 (*rot)[HD / 16]) {
  constexpr int W = HD / 8;
  const int c0 = part * W;
  float a[W], b[W];
  tmem_ld_cols<W>(taddr + c0, a);
  tmem_ld_cols<W>(taddr + HD / 2 + c0, b);
  tmem_ld_wait();
  if (!store) return;
#pragma unroll
  for (int i = 0; i < W; ++i) {
    a[i] *= scale;
    b[i] *= scale;
  }
  if (rot) {
#pragma unroll
    for (int i = 0; i < W; ++i) {
      const float4 t = (*rot)[i / 2];
      const float c = (i & 1) ? t.z : t.x, sn = (i & 1) ? t.w : t.y;
      const float na = a[i] * c + b[i] * sn, nb = b[i] * c - a[i] * sn;
      a[i] = na;
      b[i] = nb;
    }
  }
  store_bf16_cols<W>(dst + c0, a);
  store_bf16_cols<W>(dst + HD / 2 + c0, b);
}

// ------------------------------------------------------------------ delta
__host__ __device__ __forceinline__ int pad128(int s) { return (s + 127) & ~127; }

// One row per HD/8 lanes (16-byte loads of 8 bf16 each): a warp covers 256 / HD rows.
template <int HD>
__global__ void attn_delta_kernel(const bf16* __restrict__ o, const bf16* __restrict__ dout,
                                  const float* __restrict__ lse, float2* __restrict__ lsd, int B, int s, int nh) {
  constexpr int kLanes = HD / 8;  // lanes per row
  const int64_t rid = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) / kLanes;
  const int sub = threadIdx.x % kLanes;
  const int sp = pad128(s);
  const bool live = rid < static_cast<int64_t>(B) * sp * nh;
  const int i = live ? static_cast<int>(rid % sp) : 0;
  const int64_t bh = live ? rid / sp : 0;  // b * nh + head
  float acc = 0.f;
  if (live && i < s) {
    const int head = static_cast<int>(bh % nh);
    const int64_t t = (bh / nh) * s + i;
    const uint4 a = reinterpret_cast<const uint4*>(o + t * nh * HD + static_cast<int64_t>(head) * HD)[sub];
    const uint4 d = reinterpret_cast<const uint4*>(dout + t * nh * HD + static_cast<int64_t>(head) * HD)[sub];
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, dv[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      acc += __uint_as_float(av[k] << 16) * __uint_as_float(dv[k] << 16) +
             __uint_as_float(av[k] & 0xffff0000u) * __uint_as_float(dv[k] & 0xffff0000u);
    }
  }
#pragma unroll
  for (int off = kLanes / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (live && sub == 0)
    lsd[bh * sp + i] = i < s ? make_float2(-lse[bh * s + i], -acc) : make_float2(-__int_as_float(0x7f800000), -0.f);
}

// ------------------------------------------------------------------ dK, dV (KV-outer)
// TMEM: two 128-column score slots that swap roles every tile (S^T in one, dP^T in the other),
// then dV and dK. The elementwise warps load their S^T and dP^T columns, tell the MMA issuer
// once every dP^T column of the tile is in registers (the dP^T slot is then free and the next
// tile's S^T goes there), and write P^T and dS^T as bf16 pairs side by side over their own
// S^T columns (per 16 score columns: 8 columns of P^T pairs, then 8 of dS^T pairs), where the
// accumulating MMAs read them as their A operand; the next tile's dP^T goes into that slot in two
// 64-query halves (N = 64 MMAs), each right after the accumulating MMAs that read the pairs
// under it (MMAs of one thread run in issue order). Each half has its own barrier, so the warps
// start the next tile's first half while this tile's last accumulating MMAs still run (with one
// whole-tile dP^T they waited for those MMAs and the whole dP^T). Q and dO come in two rings (Q three
// tiles deep, since the next tile's S^T starts while this tile is converted; dO two deep, with
// the tile's 128 (lse2, delta) pairs), so the next tile's operands are in place when its
// score MMAs are issued.
template <int HD>
struct SmemKV {
  static constexpr int NSL = HD / 64;
  static constexpr int QS = 3, DS = 2;                  // Q ring and dO ring depths
  static constexpr int TILE = NSL * kSlice128;          // one 128-row tile: NSL x [128][64]
  static constexpr int K = 0;
  static constexpr int V = K + TILE;
  static constexpr int Q = V + TILE;                    // QS tiles
  static constexpr int DO = Q + QS * TILE;              // DS x (tile, then 128 (lse2, delta) pairs)
  static constexpr int DSTAGE = TILE + 1024;
  static constexpr int BAR = DO + DS * DSTAGE;
  static constexpr int BYTES = BAR + 256;               // the dynamic window is 1024-aligned (checked)
  static_assert(BYTES <= 232448, "dK/dV shared memory above the 227 KB per-CTA limit");
};

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap map_kv, const __grid_constant__ CUtensorMap map_q,
                            const __grid_constant__ CUtensorMap map_do, const float2* __restrict__ lsd,
                            const float* __restrict__ rope_cs, bf16* __restrict__ dqkv, int s, int nh, int nkv,
                            float scale_log2, float scale, int* err) {
  using L = SmemKV<HD>;
  constexpr int QS = L::QS, DS = L::DS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  if (smem_addr(sm) & 1023) {  // the swizzled layouts need a 1024-byte aligned base
    if (threadIdx.x == 0) atomicCAS(err, 0, kErrTimeoutAttn);
    return;
  }
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::BAR);
  uint64_t* kv_full = bar + 0;
  uint64_t* q_full = bar + 1;            // [QS]
  uint64_t* q_empty = bar + 4;           // [QS]
  uint64_t* d_full = bar + 7;            // [DS]
  uint64_t* d_empty = bar + 9;           // [DS]
  uint64_t* sdp_full = bar + 11;         // [2]: the tile's S^T and that half of its dP^T are complete
  uint64_t* dp_free = bar + 13;          // every warp holds its dP^T columns in registers
  uint64_t* p_half = bar + 14;           // [2]: every warp has written P^T/dS^T of that half
  uint64_t* acc_done = bar + 16;         // the last tile's accumulating MMAs have completed
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 17);

  const int n_t = (s + 127) / 128;
  const TileSlot slot = heavy_first_slot(static_cast<int>(blockIdx.x), n_t, static_cast<int>(gridDim.x) / n_t);
  const int kt = slot.rank;  // the first key tile is seen by the most queries
  const int kvh = slot.hb % nkv, b = slot.hb / nkv;
  const int group = nh / nkv;
  const int k0 = kt * 128;
  const int per_head = n_t - kt;  // query tiles kt .. n_t - 1
  const int total = group * per_head;
  const int sp = pad128(s);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int i = 0; i < QS; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
    }
    for (int i = 0; i < DS; ++i) {
      mbar_init(&d_full[i], 1);
      mbar_init(&d_empty[i], 1);
    }
    mbar_init(&sdp_full[0], 1);
    mbar_init(&sdp_full[1], 1);
    mbar_init(dp_free, kElemWarps);
    mbar_init(&p_half[0], kElemWarps);
    mbar_init(&p_half[1], kElemWarps);
    mbar_init(acc_done, 1);
    fence_mbar_init();
    tma_prefetch_map(&map_kv);
    tma_prefetch_map(&map_q);
    tma_prefetch_map(&map_do);
  }
  if (warp == 1) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const uint32_t tdV = tbase + 256, tdK = tbase + 256 + HD;
  auto s_slot = [&](int i) { return tbase + (i & 1) * 128; };        // S^T, then P^T | dS^T pairs
  auto d_slot = [&](int i) { return tbase + ((i & 1) ^ 1) * 128; };  // dP^T

  if (warp == 0) {
    // lane 0: K and V once, then the Q ring; lane 1: the dO ring with the (lse2, delta) pairs
    if (lane == 0) {
      mbar_arrive_expect_tx(kv_full, 2 * L::TILE);
      tma_load_4d(sm + L::K, &map_kv, kv_full, 0, k0, (nh + kvh) * (HD / 64), b);
      tma_load_4d(sm + L::V, &map_kv, kv_full, 0, k0, (nh + nkv + kvh) * (HD / 64), b);
      for (int i = 0; i < total; ++i) {
        const int st = i % QS;
        const int hq = kvh * group + i / per_head;
        const int q0 = (kt + i % per_head) * 128;
        if (!mbar_wait(&q_empty[st], ((i / QS) & 1) ^ 1u, err, kErrTimeoutAttn)) break;
        mbar_arrive_expect_tx(&q_full[st], L::TILE);
        tma_load_4d(sm + L::Q + st * L::TILE, &map_q, &q_full[st], 0, q0, hq * (HD / 64), b);
      }
    } else if (lane == 1) {
      for (int i = 0; i < total; ++i) {
        const int st = i % DS;
        const int hq = kvh * group + i / per_head;
        const int q0 = (kt + i % per_head) * 128;
        if (!mbar_wait(&d_empty[st], ((i / DS) & 1) ^ 1u, err, kErrTimeoutAttn)) break;
        mbar_arrive_expect_tx(&d_full[st], L::TILE + 1024);
        uint8_t* base = sm + L::DO + st * L::DSTAGE;
        tma_load_4d(base, &map_do, &d_full[st], 0, q0, hq * (HD / 64), b);
        bulk_load_1d(base + L::TILE, lsd + (static_cast<int64_t>(b) * nh + hq) * sp + q0, 1024, &d_full[st]);
      }
    }
  } else if (warp == 1) {
    // the whole warp runs the issuing loop; elect.sync picks the lane that issues each MMA
    constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t idesc_dh = idesc_bf16_f32(128, 64, false, false);
    constexpr uint32_t idesc_acc = idesc_bf16_f32(128, HD, false, true);
    const uint64_t kd = smem_desc_sw128(smem_addr(sm + L::K), 16, 1024);
    const uint64_t vd = smem_desc_sw128(smem_addr(sm + L::V), 16, 1024);
    bool ok = mbar_wait_warp(kv_full, 0, err, kErrTimeoutAttn);
    // S^T = K Q^T of tile i into TMEM slot t, once its Q tile is in
    auto s_scores = [&](int i, uint32_t t) -> bool {
      if (!mbar_wait_warp(&q_full[i % QS], (i / QS) & 1, err, kErrTimeoutAttn)) return false;
      tc_fence_after();
      const uint64_t bd = smem_desc_sw128(smem_addr(sm + L::Q + (i % QS) * L::TILE), 16, 1024);
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        const uint32_t off = (kk >> 2) * kSlice128 + (kk & 3) * 32;
        umma_bf16_warp(t, desc_advance(kd, off), desc_advance(bd, off), idesc_s, kk > 0 ? 1u : 0u);
      }
      return true;
    };
    // half h of dP^T = V dO^T of tile i (queries [64 h, 64 h + 64): dO rows from 8 KB into each
    // slice, a whole number of swizzle atoms) into columns [64 h, 64 h + 64) of TMEM slot t
    auto dp_half = [&](int i, int h, uint32_t t) -> bool {
      if (!mbar_wait_warp(&d_full[i % DS], (i / DS) & 1, err, kErrTimeoutAttn)) return false;
      tc_fence_after();
      const uint64_t bd = smem_desc_sw128(smem_addr(sm + L::DO + (i % DS) * L::DSTAGE), 16, 1024);
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        const uint32_t off = (kk >> 2) * kSlice128 + (kk & 3) * 32;
        umma_bf16_warp(t + h * 64, desc_advance(vd, off), desc_advance(bd, off + h * 8192), idesc_dh,
                       kk > 0 ? 1u : 0u);
      }
      return true;
    };
    if (ok && total > 0) ok = s_scores(0, s_slot(0)) && dp_half(0, 0, d_slot(0)) && dp_half(0, 1, d_slot(0));
    if (ok && total > 0) {
      umma_commit_warp(&sdp_full[0]);
      umma_commit_warp(&sdp_full[1]);
    }
    for (int i = 0; i < total && ok; ++i) {
      // B operands of the accumulating MMAs: dO and Q tiles read MN-major (16 queries per step)
      const uint64_t qd = smem_desc_sw128(smem_addr(sm + L::Q + (i % QS) * L::TILE), kSlice128, 1024);
      const uint64_t dd = smem_desc_sw128(smem_addr(sm + L::DO + (i % DS) * L::DSTAGE), kSlice128, 1024);
      const uint32_t ts = s_slot(i);
      for (int h = 0; h < 2 && ok; ++h) {
        if (h == 1 && i + 1 < total) {
          // the next tile's first dP^T half over this tile's first P^T/dS^T pairs, after the
          // MMAs reading them; then the next S^T into the dP^T slot, free once every warp holds
          // its columns
          if (!(ok = dp_half(i + 1, 0, d_slot(i + 1)))) break;
          if (!(ok = mbar_wait_warp(dp_free, i & 1, err, kErrTimeoutAttn))) break;
          tc_fence_after();
          if (!(ok = s_scores(i + 1, s_slot(i + 1)))) break;
          umma_commit_warp(&sdp_full[0]);
        }
        if (!(ok = mbar_wait_warp(&p_half[h], i & 1, err, kErrTimeoutAttn))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 4 * h; kk < 4 * h + 4; ++kk) {  // 16 queries per step; A (P^T, dS^T) from TMEM
          const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
          umma_bf16_tmem_a_warp(tdV, ts + kk * 16, desc_advance(dd, kk * 2048), idesc_acc, acc);
          umma_bf16_tmem_a_warp(tdK, ts + kk * 16 + 8, desc_advance(qd, kk * 2048), idesc_acc, acc);
        }
      }
      if (!ok) break;
      umma_commit_warp(&q_empty[i % QS]);
      umma_commit_warp(&d_empty[i % DS]);
      if (i + 1 < total) {
        // the next tile's second dP^T half over this tile's last P^T/dS^T pairs
        if (!(ok = dp_half(i + 1, 1, d_slot(i + 1)))) break;
        umma_commit_warp(&sdp_full[1]);
      } else {
        umma_commit_warp(acc_done);
      }
    }
  } else {
    const int sub = warp & 3;
    const int part = (warp - 2) >> 2;  // which 32 of each 64 query columns this warp takes
    const int row = sub * 32 + lane;
    const int key = k0 + row;
    const uint32_t tl = static_cast<uint32_t>(sub * 32) << 16;
    bool ok = true;
    for (int i = 0; i < total && ok; ++i) {
      const int q0 = (kt + i % per_head) * 128;
      const float4* lsd_s = reinterpret_cast<const float4*>(sm + L::DO + (i % DS) * L::DSTAGE + L::TILE);
      // the pairs were copied with the tile's dO: observe that copy before reading them
      if (!(ok = mbar_wait_warp(&d_full[i % DS], (i / DS) & 1, err, kErrTimeoutAttn))) break;
      const uint32_t ts = s_slot(i) + tl, td = d_slot(i) + tl;
      for (int h = 0; h < 2 && ok; ++h) {
        if (!(ok = mbar_wait_warp(&sdp_full[h], i & 1, err, kErrTimeoutAttn))) break;
        tc_fence_after();
        const int cb = h * 64 + part * kCols;  // this warp's score columns [cb, cb + 32)
        const int qc = q0 + cb;
        float sv[kCols], dv[kCols];
        tmem_ld_2x32f(ts + cb, td + cb, sv, dv);
        if (h == 1) {  // every dP^T column of the tile is now in registers
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(dp_free);
        }
        const float2 sl = make_float2(scale_log2, scale_log2);
#pragma unroll
        for (int k = 0; k < kCols / 2; ++k) {  // columns 2k, 2k+1: queries with (-lse2, -delta) in lv
          const float4 lv = lsd_s[cb / 2 + k];
          const float2 e = __ffma2_rn(make_float2(sv[2 * k], sv[2 * k + 1]), sl, make_float2(lv.x, lv.z));
          const float2 p = make_float2(ex2(e.x), ex2(e.y));
          const float2 d = __fmul2_rn(p, __fadd2_rn(make_float2(dv[2 * k], dv[2 * k + 1]), make_float2(lv.y, lv.w)));
          sv[2 * k] = p.x;
          sv[2 * k + 1] = p.y;
          dv[2 * k] = d.x;
          dv[2 * k + 1] = d.y;
        }
        if (__any_sync(0xffffffffu, key > qc)) {  // the tile straddles the diagonal: keys after queries
#pragma unroll
          for (int c = 0; c < kCols; ++c) {
            const bool keep = key <= qc + c;
            sv[c] = keep ? sv[c] : 0.f;
            dv[c] = keep ? dv[c] : 0.f;
          }
        }
        // P^T pairs then dS^T pairs over this warp's own 16 S^T columns: the A operands of
        // K-step cb / 16 of the accumulating MMAs
#pragma unroll
        for (int o = 0; o < kCols; o += 16) {
          store_pairs16(ts + cb + o, sv, o);
          store_pairs16(ts + cb + o + 8, dv, o);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_half[h]);
      }
    }
    float4 rot[4 / kParts][HD / 16];
    const bool rotate = rope_cs != nullptr && key < s;
    if (rotate)
#pragma unroll
      for (int r = 0; r < 4 / kParts; ++r) load_rotation<HD>(rope_cs, key, part + r * kParts, rot[r]);
    if (ok && total > 0 && mbar_wait_warp(acc_done, 0, err, kErrTimeoutAttn)) {
      tc_fence_after();
      const int64_t ld = static_cast<int64_t>(nh + 2 * nkv) * HD;
      bf16* rowp = dqkv + (static_cast<int64_t>(b) * s + key) * ld;
#pragma unroll
      for (int r = 0; r < 4 / kParts; ++r) {
        tmem_row_out<HD>(tdK + tl, part + r * kParts, scale, rowp + static_cast<int64_t>(nh + kvh) * HD, key < s,
                         rotate ? &rot[r] : nullptr);
        tmem_row_out<HD>(tdV + tl, part + r * kParts, 1.f, rowp + static_cast<int64_t>(nh + nkv + kvh) * HD,
                         key < s, nullptr);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

// ------------------------------------------------------------------ dQ (Q-outer)
// TMEM: two 128-column S slots (tile j in slot j & 1), one dP slot, the dQ accumulator. The next
// tile's S is computed while the warps work on this one; its dP goes into the dP slot once every
// warp holds this tile's dP columns in registers. dS is written as bf16 pairs over its S columns.
// K and V come in separate rings: K three tiles deep (read by S and by dQ, and the next tile's S
// starts early), V two deep (read only by dP, released as soon as dP has run).
template <int HD>
struct SmemQ {
  static constexpr int NSL = HD / 64;
  static constexpr int KS = 3, VS = 2;               // K ring and V ring depths
  static constexpr int TILE = NSL * kSlice128;
  static constexpr int Q = 0;
  static constexpr int DO = Q + TILE;
  static constexpr int K = DO + TILE;                // KS tiles
  static constexpr int V = K + KS * TILE;            // VS tiles
  static constexpr int BAR = V + VS * TILE;
  static constexpr int BYTES = BAR + 256;            // the dynamic window is 1024-aligned (checked)
  static_assert(BYTES <= 232448, "dQ shared memory above the 227 KB per-CTA limit");
};

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_do,
                          const __grid_constant__ CUtensorMap map_kv, const float2* __restrict__ lsd,
                          const float* __restrict__ rope_cs, bf16* __restrict__ dqkv, int s, int nh, int nkv,
                          float scale_log2, float scale, int* err) {
  using L = SmemQ<HD>;
  constexpr int KS = L::KS, VS = L::VS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  if (smem_addr(sm) & 1023) {  // the swizzled layouts need a 1024-byte aligned base
    if (threadIdx.x == 0) atomicCAS(err, 0, kErrTimeoutAttn);
    return;
  }
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::BAR);
  uint64_t* q_full = bar + 0;
  uint64_t* k_full = bar + 1;            // [KS]
  uint64_t* k_empty = bar + 4;           // [KS]
  uint64_t* v_full = bar + 7;            // [VS]
  uint64_t* v_empty = bar + 9;           // [VS]
  uint64_t* sdp_full = bar + 11;         // the tile's S and dP are complete
  uint64_t* dp_free = bar + 12;          // every warp holds its dP columns in registers
  uint64_t* ds_half = bar + 13;          // [2]
  uint64_t* dq_done = bar + 15;          // the last tile's dQ MMAs have completed
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 16);

  const int n_t = (s + 127) / 128;
  const TileSlot slot = heavy_first_slot(static_cast<int>(blockIdx.x), n_t, static_cast<int>(gridDim.x) / n_t);
  const int qt = n_t - 1 - slot.rank;  // the last query tile sees the most keys
  const int head = slot.hb % nh, b = slot.hb / nh;
  const int kvh = head / (nh / nkv);
  const int q0 = qt * 128;
  const int n_kv = qt + 1;  // 128-key tiles up to the diagonal one
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < KS; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < VS; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    mbar_init(sdp_full, 1);
    mbar_init(dp_free, kElemWarps);
    mbar_init(&ds_half[0], kElemWarps);
    mbar_init(&ds_half[1], kElemWarps);
    mbar_init(dq_done, 1);
    fence_mbar_init();
    tma_prefetch_map(&map_q);
    tma_prefetch_map(&map_do);
    tma_prefetch_map(&map_kv);
  }
  if (warp == 1) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const uint32_t tdP = tbase + 256, tdQ = tbase + 384;
  auto s_slot = [&](int j) { return tbase + (j & 1) * 128; };

  if (warp == 0) {
    // lane 0: Q and dO once, then the K ring; lane 1: the V ring
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, 2 * L::TILE);
      tma_load_4d(sm + L::Q, &map_q, q_full, 0, q0, head * (HD / 64), b);
      tma_load_4d(sm + L::DO, &map_do, q_full, 0, q0, head * (HD / 64), b);
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % KS;
        if (!mbar_wait(&k_empty[st], ((j / KS) & 1) ^ 1u, err, kErrTimeoutAttn)) break;
        mbar_arrive_expect_tx(&k_full[st], L::TILE);
        tma_load_4d(sm + L::K + st * L::TILE, &map_kv, &k_full[st], 0, j * 128, (nh + kvh) * (HD / 64), b);
      }
    } else if (lane == 1) {
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % VS;
        if (!mbar_wait(&v_empty[st], ((j / VS) & 1) ^ 1u, err, kErrTimeoutAttn)) break;
        mbar_arrive_expect_tx(&v_full[st], L::TILE);
        tma_load_4d(sm + L::V + st * L::TILE, &map_kv, &v_full[st], 0, j * 128, (nh + nkv + kvh) * (HD / 64), b);
      }
    }
  } else if (warp == 1) {
    // the whole warp runs the issuing loop; elect.sync picks the lane that issues each MMA
    constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t idesc_acc = idesc_bf16_f32(128, HD, false, true);
    const uint64_t qd = smem_desc_sw128(smem_addr(sm + L::Q), 16, 1024);
    const uint64_t dd = smem_desc_sw128(smem_addr(sm + L::DO), 16, 1024);
    bool ok = mbar_wait_warp(q_full, 0, err, kErrTimeoutAttn);
    // S = Q K^T (dp = false) or dP = dO V^T of tile j into TMEM slot t, once its operand is in;
    // a V stage is released as soon as its dP has run
    auto scores = [&](int j, bool dp, uint32_t t) -> bool {
      uint64_t* full = dp ? &v_full[j % VS] : &k_full[j % KS];
      const uint32_t parity = dp ? (j / VS) & 1 : (j / KS) & 1;
      if (!mbar_wait_warp(full, parity, err, kErrTimeoutAttn)) return false;
      tc_fence_after();
      const uint64_t ad = dp ? dd : qd;
      const uint64_t bd =
          smem_desc_sw128(smem_addr(dp ? sm + L::V + (j % VS) * L::TILE : sm + L::K + (j % KS) * L::TILE), 16, 1024);
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        const uint32_t off = (kk >> 2) * kSlice128 + (kk & 3) * 32;
        umma_bf16_warp(t, desc_advance(ad, off), desc_advance(bd, off), idesc_s, kk > 0 ? 1u : 0u);
      }
      if (dp) umma_commit_warp(&v_empty[j % VS]);
      return true;
    };
    if (ok) ok = scores(0, false, s_slot(0)) && scores(0, true, tdP);
    if (ok) umma_commit_warp(sdp_full);
    for (int j = 0; j < n_kv && ok; ++j) {
      // B operand of the dQ MMAs: the K tile read MN-major (16 keys per step)
      const uint64_t kd = smem_desc_sw128(smem_addr(sm + L::K + (j % KS) * L::TILE), kSlice128, 1024);
      // the next tile's S into the other S slot, whose dS was read by MMAs issued earlier
      if (j + 1 < n_kv && !(ok = scores(j + 1, false, s_slot(j + 1)))) break;
      for (int h = 0; h < 2 && ok; ++h) {
        if (h == 1 && j + 1 < n_kv) {  // the dP slot is free once every warp holds its columns
          if (!(ok = mbar_wait_warp(dp_free, j & 1, err, kErrTimeoutAttn))) break;
          tc_fence_after();
          if (!(ok = scores(j + 1, true, tdP))) break;
          umma_commit_warp(sdp_full);
        }
        if (!(ok = mbar_wait_warp(&ds_half[h], j & 1, err, kErrTimeoutAttn))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 4 * h; kk < 4 * h + 4; ++kk)  // 16 keys per step; A (dS) from TMEM
          umma_bf16_tmem_a_warp(tdQ, s_slot(j) + kk * 16, desc_advance(kd, kk * 2048), idesc_acc,
                                (j > 0 || kk > 0) ? 1u : 0u);
      }
      if (!ok) break;
      umma_commit_warp(&k_empty[j % KS]);
      if (j == n_kv - 1) umma_commit_warp(dq_done);
    }
  } else {
    const int sub = warp & 3;
    const int part = (warp - 2) >> 2;  // which 32 of each 64 key columns this warp takes
    const int row = sub * 32 + lane;
    const int q = q0 + row;
    const uint32_t tl = static_cast<uint32_t>(sub * 32) << 16;
    const int sp = pad128(s);
    const float2 lq = lsd[(static_cast<int64_t>(b) * nh + head) * sp + q];  // q < sp: the tile lies in the padding
    const float2 nl2 = make_float2(lq.x, lq.x), ndl = make_float2(lq.y, lq.y), sl = make_float2(scale_log2, scale_log2);
    bool ok = true;
    for (int j = 0; j < n_kv && ok; ++j) {
      if (!(ok = mbar_wait_warp(sdp_full, j & 1, err, kErrTimeoutAttn))) break;
      tc_fence_after();
      const uint32_t ts = s_slot(j) + tl;
      for (int h = 0; h < 2; ++h) {
        const int cb = h * 64 + part * kCols;
        float sv[kCols], dv[kCols];
        tmem_ld_2x32f(ts + cb, tdP + tl + cb, sv, dv);
        if (h == 1) {  // every dP column of the tile is now in registers
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(dp_free);
        }
        const int key0 = j * 128 + cb;
#pragma unroll
        for (int k = 0; k < kCols / 2; ++k) {  // dS = 2^(S scale - lse2) (dP - delta), two columns at a time
          const float2 e = __ffma2_rn(make_float2(sv[2 * k], sv[2 * k + 1]), sl, nl2);
          const float2 d = __fmul2_rn(make_float2(ex2(e.x), ex2(e.y)),
                                      __fadd2_rn(make_float2(dv[2 * k], dv[2 * k + 1]), ndl));
          dv[2 * k] = d.x;
          dv[2 * k + 1] = d.y;
        }
        if (__any_sync(0xffffffffu, key0 + kCols - 1 > q)) {  // keys after some query of this warp
#pragma unroll
          for (int c = 0; c < kCols; ++c) dv[c] = key0 + c <= q ? dv[c] : 0.f;
        }
        // dS goes back into TMEM over this warp's S columns (A operand of K-step cb / 16)
#pragma unroll
        for (int o = 0; o < kCols; o += 16) store_pairs16(ts + cb + o, dv, o);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ds_half[h]);
      }
    }
    float4 rot[4 / kParts][HD / 16];
    const bool rotate = rope_cs != nullptr && q < s;
    if (rotate)
#pragma unroll
      for (int r = 0; r < 4 / kParts; ++r) load_rotation<HD>(rope_cs, q, part + r * kParts, rot[r]);
    if (ok && mbar_wait_warp(dq_done, 0, err, kErrTimeoutAttn)) {
      tc_fence_after();
      const int64_t ld = static_cast<int64_t>(nh + 2 * nkv) * HD;
#pragma unroll
      for (int r = 0; r < 4 / kParts; ++r)
        tmem_row_out<HD>(tdQ + tl, part + r * kParts, scale,
                         dqkv + (static_cast<int64_t>(b) * s + q) * ld + static_cast<int64_t>(head) * HD, q < s,
                         rotate ? &rot[r] : nullptr);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

template <int HD>
cudaError_t bwd_launch(const bf16* qkv, const bf16* o, const float* lse, const bf16* dout, bf16* dqkv, float* scratch,
                       const float* rope_cs, int B, int s, int nh, int nkv, int* err, cudaStream_t st) {
  const int64_t rows = static_cast<int64_t>(B) * pad128(s) * nh;
  float2* lsd = reinterpret_cast<float2*>(scratch);
  attn_delta_kernel<HD><<<static_cast<unsigned>((rows * (HD / 8) + 255) / 256), 256, 0, st>>>(o, dout, lse, lsd, B, s,
                                                                                               nh);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t ld = static_cast<int64_t>(nh + 2 * nkv) * HD, ldo = static_cast<int64_t>(nh) * HD;
  CUtensorMap kv128, do128;
  constexpr uint32_t nsl = HD / 64;  // one box carries every head_dim slice of a tile
  bool ok = tma_map_slices(&kv128, qkv, s, B, ld, s * ld, nsl, 128) &&
            tma_map_slices(&do128, dout, s, B, ldo, s * ldo, nsl, 128);
  if (!ok) return cudaErrorInvalidValue;
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(HD));
  const float scale = 1.f / sqrtf(static_cast<float>(HD));
  e = cudaFuncSetAttribute(attn_bwd_dq_tc_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, SmemQ<HD>::BYTES);
  if (e != cudaSuccess) return e;
  attn_bwd_dq_tc_kernel<HD><<<((s + 127) / 128) * nh * B, kThreads, SmemQ<HD>::BYTES, st>>>(
      kv128, do128, kv128, lsd, rope_cs, dqkv, s, nh, nkv, scale_log2, scale, err);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(attn_bwd_dkdv_tc_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           SmemKV<HD>::BYTES);
  if (e != cudaSuccess) return e;
  attn_bwd_dkdv_tc_kernel<HD><<<((s + 127) / 128) * nkv * B, kThreads, SmemKV<HD>::BYTES, st>>>(
      kv128, kv128, do128, lsd, rope_cs, dqkv, s, nh, nkv, scale_log2, scale, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t attn_bwd(const bf16* qkv, const bf16* o, const float* lse, const bf16* dout, bf16* dqkv, float* delta,
                     const float* rope_cs, int B, int s, int nh, int nkv, int hd, int* err, cudaStream_t st) {
  if (nkv <= 0 || nh % nkv || s <= 0 || B <= 0 || !err) return cudaErrorInvalidValue;
  if ((reinterpret_cast<uintptr_t>(qkv) | reinterpret_cast<uintptr_t>(o) | reinterpret_cast<uintptr_t>(dout) |
       reinterpret_cast<uintptr_t>(dqkv) | reinterpret_cast<uintptr_t>(delta)) & 15)
    return cudaErrorMisalignedAddress;
  if (hd == 64) return bwd_launch<64>(qkv, o, lse, dout, dqkv, delta, rope_cs, B, s, nh, nkv, err, st);
  if (hd == 128) return bwd_launch<128>(qkv, o, lse, dout, dqkv, delta, rope_cs, B, s, nh, nkv, err, st);
  return cudaErrorInvalidValue;
}

}  // namespace mt
