// Causal grouped-query flash attention backward on the tcgen05 tensor cores.
//
// Deterministic, no atomics:
//  * lsd[b, n, i] = (lse2[b, n, i], delta[b, n, i]), delta = sum_d dO[i, n, d] O[i, n, d]
//    (HD/8 lanes per row), padded to a multiple of 128 rows with (+inf, 0): past the end of
//    the sequence every probability is then exactly 0 with no mask, and the causal mask is
//    only evaluated on tiles that straddle the diagonal
//  * dK/dV, KV-outer: one CTA per (128-key tile, kv head, sequence) walks every 128-query
//    tile of every query head of its group in a fixed order:
//        S^T  = K Q^T,  dP^T = V dO^T                         (TMEM, 128 x 128 each)
//        P^T  = exp2(S^T log2(e)/sqrt(hd) - lse2),  dS^T = P^T (dP^T - delta)
//        dV  += P^T dO,  dK += dS^T Q                         (TMEM accumulators)
//  * dQ, Q-outer: one CTA per (128-query tile, query head, sequence) walks the 128-key tiles:
//        S = Q K^T,  dP = dO V^T,  dS = P (dP - delta),  dQ += dS K
// Every tile is 128 x 128: the score MMAs have N = 128 (at N = 64 the two shared-memory
// operands of each MMA need more bytes per cycle than shared memory gives), and every TMA box
// is 128 rows high (the TMA issues far more bytes per cycle with tall boxes).
// Roles per CTA: warp 0 TMA, warp 1 MMA issuer, warps 2..17 the elementwise step: each TMEM
// lane (one key row, resp. one query row) is shared by four warps, and each warp takes 16 of
// the first 64 score columns and then 16 of the last 64 (the step needs no row reductions:
// lse2 and delta are precomputed). They write P^T / dS^T (dQ kernel: dS) as bf16 pairs back
// into TMEM over the scores they came from, where the accumulating MMAs read them as their A
// operand. The tile's accumulating MMAs over its first 64 columns start as soon as every warp
// has finished those columns, while the warps work on the last 64. The score buffers are
// single (TMEM holds S, dP and both accumulators: 512 columns): the next tile's score MMAs,
// issued after this tile's accumulating MMAs, run after them (MMAs of one thread run in issue
// order). Every wait is bounded (error flag on timeout).
#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"
#include "tile_order.cuh"
#include "tma.h"

namespace mt {

namespace {

constexpr int kThreads = 576;       // TMA warp, MMA warp, 16 elementwise warps
constexpr int kElem = 512;          // elementwise threads
constexpr int kCols = 16;           // score columns an elementwise warp takes per half tile
constexpr int kElemWarps = kElem / 32;  // arrivals per barrier phase (one elected lane per warp)
constexpr int kSlice128 = 128 * 128;  // bytes of a [128 rows][64 bf16] swizzle-atom-wide slice
// Operand ring depth (streamed 128-row tiles of two tensors): as deep as shared memory allows.
template <int HD>
constexpr int ring_stages() { return HD == 64 ? 4 : 2; }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float ex2(float x) {  // hardware 2^x (ex2.approx, flush to zero)
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Pack 16 values into 8 bf16 pairs and store them to 8 TMEM columns of this thread's lane
// (the A-operand layout: element k of a row in column k/2, even k in the low half).
__device__ __forceinline__ void store_pairs_tmem(uint32_t taddr, const float (&v)[kCols]) {
  uint32_t w[kCols / 2];
#pragma unroll
  for (int c = 0; c < kCols / 2; ++c) w[c] = pack_bf16(v[2 * c], v[2 * c + 1]);
  tmem_st_8cols(taddr, w);
}

// Two 16-column TMEM loads (S and dP of one row) behind a single wait.
__device__ __forceinline__ void tmem_ld_2x16f(uint32_t ta, uint32_t tb, float (&a)[kCols], float (&b)[kCols]) {
  uint32_t ra[16], rb[16];
  tmem_ld_16cols(ta, ra);
  tmem_ld_16cols(tb, rb);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 16; ++i) {
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

// Store one TMEM lane's fp32 row (HD columns), times `scale`, as bf16 to dst (if `store`). Each
// of the four warps on the lane takes columns [part*HD/8, +HD/8) and the same HD/2 further on,
// which are the rotation pairs of rotate-half RoPE: with `rot` (from load_rotation) the
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
    lsd[bh * sp + i] = i < s ? make_float2(lse[bh * s + i], acc) : make_float2(__int_as_float(0x7f800000), 0.f);
}

// ------------------------------------------------------------------ dK, dV (KV-outer)
// Sub-tile n (64 queries) of the CTA's sequence is half n & 1 of ring stage (n / 2) % S; its
// S^T/dP^T live in TMEM buffer n & 1 (64 columns each), so the score MMAs of sub-tile n + 1 run
// while the elementwise warps convert sub-tile n.
template <int HD>
struct SmemKV {
  static constexpr int NSL = HD / 64;
  static constexpr int S = ring_stages<HD>();
  static constexpr int K = 0;                           // NSL x [128][64]
  static constexpr int V = K + NSL * kSlice128;         // NSL x [128][64]
  static constexpr int QD = V + NSL * kSlice128;        // S x (Q: NSL x [128][64], dO: same)
  static constexpr int STAGE = 2 * NSL * kSlice128;
  static constexpr int BAR = QD + S * STAGE;
  static constexpr int BYTES = BAR + 256 + 1024;
  static_assert(BYTES <= 232448, "dK/dV shared memory above the 227 KB per-CTA limit");
  static_assert(2 * S + 7 <= 30, "barriers and the TMEM slot fit the 256-byte barrier area");
};

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap map_kv, const __grid_constant__ CUtensorMap map_q,
                            const __grid_constant__ CUtensorMap map_do, const float2* __restrict__ lsd,
                            const float* __restrict__ rope_cs, bf16* __restrict__ dqkv, int s, int nh, int nkv,
                            float scale_log2, float scale, int* err) {
  using L = SmemKV<HD>;
  constexpr int S = L::S;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::BAR);
  uint64_t* kv_full = bar + 0;
  uint64_t* qd_full = bar + 1;           // [S]
  uint64_t* qd_empty = bar + 1 + S;      // [S]
  uint64_t* sdp_full = bar + 1 + 2 * S;  // [2]
  uint64_t* p_full = bar + 3 + 2 * S;    // [2]
  uint64_t* acc_done = bar + 5 + 2 * S;  // the last sub-tile's accumulating MMAs have completed
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 6 + 2 * S);

  const int n_t = (s + 127) / 128;
  const TileSlot slot = heavy_first_slot(static_cast<int>(blockIdx.x), n_t, static_cast<int>(gridDim.x) / n_t);
  const int kt = slot.rank;  // the first key tile is seen by the most queries
  const int kvh = slot.hb % nkv, b = slot.hb / nkv;
  const int group = nh / nkv;
  const int k0 = kt * 128;
  const int per_head = n_t - kt;  // query tiles kt .. n_t - 1
  const int total = group * per_head;  // 128-query tiles
  const int n_sub = 2 * total;         // 64-query sub-tiles
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int i = 0; i < S; ++i) {
      mbar_init(&qd_full[i], 1);
      mbar_init(&qd_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sdp_full[i], 1);
      mbar_init(&p_full[i], kElemWarps);
    }
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
  const uint32_t tS = tbase, tdP = tbase + 128, tdV = tbase + 256, tdK = tbase + 256 + HD;

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(kv_full, 2 * L::NSL * kSlice128);
      tma_load_4d(sm + L::K, &map_kv, kv_full, 0, k0, (nh + kvh) * (HD / 64), b);
      tma_load_4d(sm + L::V, &map_kv, kv_full, 0, k0, (nh + nkv + kvh) * (HD / 64), b);
      for (int i = 0; i < total; ++i) {
        const int st = i % S;
        const int hq = kvh * group + i / per_head;
        const int q0 = (kt + i % per_head) * 128;
        if (!mbar_wait(&qd_empty[st], ((i / S) & 1) ^ 1u, err, kErrTimeoutAttn)) break;
        mbar_arrive_expect_tx(&qd_full[st], 2 * L::NSL * kSlice128);
        uint8_t* base = sm + L::QD + st * L::STAGE;
        tma_load_4d(base, &map_q, &qd_full[st], 0, q0, hq * (HD / 64), b);
        tma_load_4d(base + L::NSL * kSlice128, &map_do, &qd_full[st], 0, q0, hq * (HD / 64), b);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 64, false, false);
      constexpr uint32_t idesc_acc = idesc_bf16_f32(128, HD, false, true);
      const uint32_t ka = smem_addr(sm + L::K), va = smem_addr(sm + L::V);
      bool ok = mbar_wait(kv_full, 0, err, kErrTimeoutAttn);
      // S^T/dP^T buffer n & 1 last held P^T/dS^T of sub-tile n - 2, read by that sub-tile's
      // accumulating MMAs, which were issued before these: MMAs run in issue order.
      auto issue_sdp = [&](int n) -> bool {
        const int i = n >> 1, st = i % S, half = n & 1, buf = n & 1;
        if (half == 0) {
          if (!mbar_wait(&qd_full[st], (i / S) & 1, err, kErrTimeoutAttn)) return false;
          tc_fence_after();
        }
        const uint32_t qa = smem_addr(sm + L::QD + st * L::STAGE) + half * 8192;  // 64 query rows in
        const uint32_t da = qa + L::NSL * kSlice128;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kSlice128 + (kk & 3) * 32;
          umma_bf16(tS + buf * 64, smem_desc_sw128(ka + off, 16, 1024), smem_desc_sw128(qa + off, 16, 1024),
                    idesc_s, kk > 0 ? 1u : 0u);
          umma_bf16(tdP + buf * 64, smem_desc_sw128(va + off, 16, 1024), smem_desc_sw128(da + off, 16, 1024),
                    idesc_s, kk > 0 ? 1u : 0u);
        }
        umma_commit(&sdp_full[buf]);
        return true;
      };
      if (ok && n_sub > 0) ok = issue_sdp(0);
      for (int n = 0; n < n_sub && ok; ++n) {
        if (n + 1 < n_sub && !(ok = issue_sdp(n + 1))) break;
        const int i = n >> 1, st = i % S, half = n & 1, buf = n & 1;
        if (!(ok = mbar_wait(&p_full[buf], (n >> 1) & 1, err, kErrTimeoutAttn))) break;
        tc_fence_after();
        const uint32_t qa = smem_addr(sm + L::QD + st * L::STAGE) + half * 8192;
        const uint32_t da = qa + L::NSL * kSlice128;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {  // 64 queries in steps of 16; A (P^T, dS^T) from TMEM
          const uint32_t acc = (n > 0 || kk > 0) ? 1u : 0u;
          umma_bf16_tmem_a(tdV, tS + buf * 64 + kk * kCols, smem_desc_sw128(da + kk * 2048, kSlice128, 1024),
                           idesc_acc, acc);
          umma_bf16_tmem_a(tdK, tdP + buf * 64 + kk * kCols, smem_desc_sw128(qa + kk * 2048, kSlice128, 1024),
                           idesc_acc, acc);
        }
        if (half == 1) umma_commit(&qd_empty[st]);
        if (n == n_sub - 1) umma_commit(acc_done);
      }
    }
  } else {
    const int sub = warp & 3;
    const int part = (warp - 2) >> 2;  // which 16 of the 64 query columns of a sub-tile this warp takes
    const int row = sub * 32 + lane;
    const int key = k0 + row;
    const uint32_t tl = static_cast<uint32_t>(sub * 32) << 16;
    const int sp = pad128(s);
    bool ok = true;
    for (int n = 0; n < n_sub && ok; ++n) {
      const int i = n >> 1, buf = n & 1;
      const int hq = kvh * group + i / per_head;
      const int qc = (kt + i % per_head) * 128 + (n & 1) * 64 + part * kCols;  // this warp's first query
      // the (lse2, delta) pairs of these 16 queries, fetched before the scores are ready
      const float4* lp = reinterpret_cast<const float4*>(lsd + (static_cast<int64_t>(b) * nh + hq) * sp + qc);
      float4 lv[kCols / 2];
#pragma unroll
      for (int k = 0; k < kCols / 2; ++k) lv[k] = __ldg(lp + k);
      if (!(ok = mbar_wait_warp(&sdp_full[buf], (n >> 1) & 1, err, kErrTimeoutAttn))) break;
      tc_fence_after();
      float sv[kCols], dv[kCols];
      tmem_ld_2x16f(tS + tl + buf * 64 + part * kCols, tdP + tl + buf * 64 + part * kCols, sv, dv);
#pragma unroll
      for (int c = 0; c < kCols; ++c) {
        const float l2 = (c & 1) ? lv[c / 2].z : lv[c / 2].x;
        const float dl = (c & 1) ? lv[c / 2].w : lv[c / 2].y;
        const float p = ex2(fmaf(sv[c], scale_log2, -l2));
        sv[c] = p;
        dv[c] = p * (dv[c] - dl);
      }
      if (__any_sync(0xffffffffu, key > qc)) {  // the sub-tile straddles the diagonal: keys after queries
#pragma unroll
        for (int c = 0; c < kCols; ++c) {
          const bool keep = key <= qc + c;
          sv[c] = keep ? sv[c] : 0.f;
          dv[c] = keep ? dv[c] : 0.f;
        }
      }
      // P^T and dS^T go back into TMEM over the scores they came from: this warp's 16 score
      // columns become 8 columns of bf16 pairs at their start, the A operand of K-step `part`
      // of the accumulating MMAs (no other warp reads or writes these columns).
      store_pairs_tmem(tS + tl + buf * 64 + part * kCols, sv);
      store_pairs_tmem(tdP + tl + buf * 64 + part * kCols, dv);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[buf]);
    }
    float4 rot[HD / 16];
    const bool rotate = rope_cs != nullptr && key < s;
    if (rotate) load_rotation<HD>(rope_cs, key, part, rot);
    if (ok && n_sub > 0 && mbar_wait_warp(acc_done, 0, err, kErrTimeoutAttn)) {
      tc_fence_after();
      const int64_t ld = static_cast<int64_t>(nh + 2 * nkv) * HD;
      bf16* rowp = dqkv + (static_cast<int64_t>(b) * s + key) * ld;
      tmem_row_out<HD>(tdK + tl, part, scale, rowp + static_cast<int64_t>(nh + kvh) * HD, key < s,
                       rotate ? &rot : nullptr);
      tmem_row_out<HD>(tdV + tl, part, 1.f, rowp + static_cast<int64_t>(nh + nkv + kvh) * HD, key < s, nullptr);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

// ------------------------------------------------------------------ dQ (Q-outer)
// Sub-tile n (64 keys) is half n & 1 of ring stage (n / 2) % S; its S/dP live in TMEM buffer
// n % 3 (128 columns: S then dP), three buffers next to the dQ accumulator.
template <int HD>
struct SmemQ {
  static constexpr int NSL = HD / 64;
  static constexpr int S = ring_stages<HD>();
  static constexpr int Q = 0;                        // NSL x [128][64]
  static constexpr int DO = Q + NSL * kSlice128;     // NSL x [128][64]
  static constexpr int KV = DO + NSL * kSlice128;    // S x (K: NSL x [128][64], V: same)
  static constexpr int STAGE = 2 * NSL * kSlice128;
  static constexpr int BAR = KV + S * STAGE;
  static constexpr int BYTES = BAR + 256 + 1024;
  static_assert(BYTES <= 232448, "dQ shared memory above the 227 KB per-CTA limit");
};

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_do,
                          const __grid_constant__ CUtensorMap map_kv, const float2* __restrict__ lsd,
                          const float* __restrict__ rope_cs, bf16* __restrict__ dqkv, int s, int nh, int nkv,
                          float scale_log2, float scale, int* err) {
  using L = SmemQ<HD>;
  constexpr int S = L::S;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::BAR);
  uint64_t* q_full = bar + 0;
  uint64_t* kv_full = bar + 1;           // [S]
  uint64_t* kv_empty = bar + 1 + S;      // [S]
  uint64_t* sdp_full = bar + 1 + 2 * S;  // [3]
  uint64_t* ds_full = bar + 4 + 2 * S;   // [3]
  uint64_t* dq_done = bar + 7 + 2 * S;   // the last sub-tile's dQ MMAs have completed
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 8 + 2 * S);

  const int n_t = (s + 127) / 128;
  const TileSlot slot = heavy_first_slot(static_cast<int>(blockIdx.x), n_t, static_cast<int>(gridDim.x) / n_t);
  const int qt = n_t - 1 - slot.rank;  // the last query tile sees the most keys
  const int head = slot.hb % nh, b = slot.hb / nh;
  const int kvh = head / (nh / nkv);
  const int q0 = qt * 128;
  const int n_kv = qt + 1;      // 128-key tiles up to the diagonal one
  const int n_sub = 2 * n_kv;   // 64-key sub-tiles
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < S; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < 3; ++i) {
      mbar_init(&sdp_full[i], 1);
      mbar_init(&ds_full[i], kElemWarps);
    }
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
  const uint32_t tdQ = tbase + 384;

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, 2 * L::NSL * kSlice128);
      tma_load_4d(sm + L::Q, &map_q, q_full, 0, q0, head * (HD / 64), b);
      tma_load_4d(sm + L::DO, &map_do, q_full, 0, q0, head * (HD / 64), b);
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % S;
        if (!mbar_wait(&kv_empty[st], ((j / S) & 1) ^ 1u, err, kErrTimeoutAttn)) break;
        mbar_arrive_expect_tx(&kv_full[st], 2 * L::NSL * kSlice128);
        uint8_t* base = sm + L::KV + st * L::STAGE;
        tma_load_4d(base, &map_kv, &kv_full[st], 0, j * 128, (nh + kvh) * (HD / 64), b);
        tma_load_4d(base + L::NSL * kSlice128, &map_kv, &kv_full[st], 0, j * 128, (nh + nkv + kvh) * (HD / 64), b);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 64, false, false);
      constexpr uint32_t idesc_acc = idesc_bf16_f32(128, HD, false, true);
      const uint32_t qa = smem_addr(sm + L::Q), da = smem_addr(sm + L::DO);
      bool ok = mbar_wait(q_full, 0, err, kErrTimeoutAttn);
      // S/dP buffer n % 3 last held dS of sub-tile n - 3, read by that sub-tile's dQ MMAs,
      // which were issued before these: MMAs run in issue order.
      auto issue_sdp = [&](int n) -> bool {
        const int j = n >> 1, ks = j % S, half = n & 1, buf = n % 3;
        if (half == 0) {
          if (!mbar_wait(&kv_full[ks], (j / S) & 1, err, kErrTimeoutAttn)) return false;
          tc_fence_after();
        }
        const uint32_t ka = smem_addr(sm + L::KV + ks * L::STAGE) + half * 8192;  // 64 key rows in
        const uint32_t va = ka + L::NSL * kSlice128;
        const uint32_t t = tbase + buf * 128;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kSlice128 + (kk & 3) * 32;
          umma_bf16(t, smem_desc_sw128(qa + off, 16, 1024), smem_desc_sw128(ka + off, 16, 1024), idesc_s,
                    kk > 0 ? 1u : 0u);
          umma_bf16(t + 64, smem_desc_sw128(da + off, 16, 1024), smem_desc_sw128(va + off, 16, 1024), idesc_s,
                    kk > 0 ? 1u : 0u);
        }
        umma_commit(&sdp_full[buf]);
        return true;
      };
      if (ok) ok = issue_sdp(0);
      if (ok && n_sub > 1) ok = issue_sdp(1);
      for (int n = 0; n < n_sub && ok; ++n) {
        if (n + 2 < n_sub && !(ok = issue_sdp(n + 2))) break;
        const int j = n >> 1, ks = j % S, half = n & 1, buf = n % 3;
        if (!(ok = mbar_wait(&ds_full[buf], (n / 3) & 1, err, kErrTimeoutAttn))) break;
        tc_fence_after();
        const uint32_t ka = smem_addr(sm + L::KV + ks * L::STAGE) + half * 8192;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // 64 keys in steps of 16; A (dS) from TMEM
          umma_bf16_tmem_a(tdQ, tbase + buf * 128 + kk * kCols, smem_desc_sw128(ka + kk * 2048, kSlice128, 1024),
                           idesc_acc, (n > 0 || kk > 0) ? 1u : 0u);
        if (half == 1) umma_commit(&kv_empty[ks]);
        if (n == n_sub - 1) umma_commit(dq_done);
      }
    }
  } else {
    const int sub = warp & 3;
    const int part = (warp - 2) >> 2;  // which 16 of the 64 key columns of a sub-tile this warp takes
    const int row = sub * 32 + lane;
    const int q = q0 + row;
    const uint32_t tl = static_cast<uint32_t>(sub * 32) << 16;
    const int sp = pad128(s);
    const float2 lq = lsd[(static_cast<int64_t>(b) * nh + head) * sp + q];  // q < sp: the tile lies in the padding
    const float l2 = lq.x, dl = lq.y;
    bool ok = true;
    for (int n = 0; n < n_sub && ok; ++n) {
      const int buf = n % 3;
      if (!(ok = mbar_wait_warp(&sdp_full[buf], (n / 3) & 1, err, kErrTimeoutAttn))) break;
      tc_fence_after();
      const uint32_t t = tbase + tl + buf * 128 + part * kCols;
      float sv[kCols], dv[kCols];
      tmem_ld_2x16f(t, t + 64, sv, dv);
      const int key0 = n * 64 + part * kCols;
#pragma unroll
      for (int c = 0; c < kCols; ++c) dv[c] = ex2(fmaf(sv[c], scale_log2, -l2)) * (dv[c] - dl);
      if (__any_sync(0xffffffffu, key0 + kCols - 1 > q)) {  // keys after some query of this warp
#pragma unroll
        for (int c = 0; c < kCols; ++c) dv[c] = key0 + c <= q ? dv[c] : 0.f;
      }
      // dS goes back into TMEM over this warp's score columns (A operand of K-step `part`)
      store_pairs_tmem(t, dv);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ds_full[buf]);
    }
    float4 rot[HD / 16];
    const bool rotate = rope_cs != nullptr && q < s;
    if (rotate) load_rotation<HD>(rope_cs, q, part, rot);
    if (ok && mbar_wait_warp(dq_done, 0, err, kErrTimeoutAttn)) {
      tc_fence_after();
      const int64_t ld = static_cast<int64_t>(nh + 2 * nkv) * HD;
      tmem_row_out<HD>(tdQ + tl, part, scale,
                       dqkv + (static_cast<int64_t>(b) * s + q) * ld + static_cast<int64_t>(head) * HD, q < s,
                       rotate ? &rot : nullptr);
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
