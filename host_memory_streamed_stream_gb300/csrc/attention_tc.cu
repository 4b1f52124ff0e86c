// Causal grouped-query flash attention forward on the tcgen05 tensor cores.
//
// One CTA per (128-query tile, query head, sequence), heaviest (most key tiles) first; two
// CTAs share an SM (at most 113 KB shared memory, 256 TMEM columns each), so each SM runs two
// softmax warpgroups against two MMA streams.
//   warp 0      TMA: Q once, then K and V tiles of 64 keys into two rings, one per tensor
//               (lane 0: K, 3 stages; lane 1: V, 2 stages), so a K stage is reloaded as soon
//               as S_j has read it instead of after O += P_j V_j (one load per tensor per
//               tile: every head_dim slice in one box)
//   warp 1      MMA: S_j = Q K_j^T into one of two TMEM score buffers (64 columns each),
//               then O += P_j V_j into the TMEM output accumulator (head_dim columns), with
//               P_j read from TMEM as the A operand
//   warps 2..5  softmax, one thread per query row: read S_j from TMEM, mask, running max,
//               P_j = exp2(S_j * log2(e)/sqrt(hd) - m) packed as bf16 pairs back into the
//               TMEM score buffer it came from, running row sum; at the end O / l to global
//               memory and lse2 = m + log2(l).
// S_{j+1} is computed while the softmax works on S_j. The running max is applied lazily:
// the output accumulator is rescaled only when a row's max grows by more than 2^8 (in
// probability units) over the max the exponentials were taken against, which keeps P <= 256
// and makes rescaling rare. Every wait is bounded (error flag on timeout).
#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"
#include "tile_order.cuh"
#include "tma.h"

namespace mt {

namespace {

constexpr int kThreads = 192;
constexpr int kKeys = 64;                // keys per tile
constexpr int kSlice128 = 128 * 128;     // [128 rows][64 bf16]: one 128-byte swizzle atom wide
constexpr int kSlice64 = 64 * 128;       // [64 rows][64 bf16]
constexpr float kLazyRescale = 8.f;      // log2 units
constexpr int kKStages = 3;              // K ring depth
constexpr int kVStages = 2;              // V ring depth

template <int HD>
struct Smem {
  static constexpr int NSL = HD / 64;               // 64-wide slices of head_dim
  static constexpr int Q = 0;                       // NSL x [128 queries][64]
  static constexpr int TILE = NSL * kSlice64;       // one K or V tile: NSL x [64 keys][64]
  static constexpr int K = Q + NSL * kSlice128;     // kKStages K tiles
  static constexpr int V = K + kKStages * TILE;     // kVStages V tiles
  static constexpr int BAR = V + kVStages * TILE;
  static constexpr int BYTES = BAR + 256;           // the dynamic window is 1024-aligned (checked)
  // two CTAs per SM: 228 KB per SM, 1 KB of it reserved per CTA
  static_assert(2 * (BYTES + 1024) <= 233472, "forward attention no longer fits two CTAs per SM");
};

__device__ __forceinline__ float ex2(float x) {  // hardware 2^x (ex2.approx, flush to zero)
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {  // three-input max (sm_100+)
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 2)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_kv,
                       bf16* __restrict__ o, float* __restrict__ lse, int s, int nh, int nkv, float scale_log2,
                       int* err) {
  using L = Smem<HD>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  if (smem_addr(sm) & 1023) {  // the swizzled layouts need a 1024-byte aligned base
    if (threadIdx.x == 0) atomicCAS(err, 0, kErrTimeoutAttn);
    return;
  }
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::BAR);
  uint64_t* q_full = bar + 0;
  uint64_t* k_full = bar + 1;    // [kKStages]  K ring: a stage is free again once S_j has read it
  uint64_t* k_empty = bar + 4;   // [kKStages]
  uint64_t* v_full = bar + 7;    // [kVStages]  V ring: free again once O += P_j V_j has read it
  uint64_t* v_empty = bar + 9;   // [kVStages]
  uint64_t* s_full = bar + 11;   // [2]
  uint64_t* p_full = bar + 13;   // [2]
  uint64_t* pv_done = bar + 15;  // one phase per O += P_j V_j (the lazy rescale waits on it)
  uint64_t* o_done = bar + 16;   // once: every O += P_j V_j of the tile has completed
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 17);

  const int n_qt = (s + 127) / 128;
  const TileSlot slot = heavy_first_slot(static_cast<int>(blockIdx.x), n_qt, static_cast<int>(gridDim.x) / n_qt);
  const int qt = n_qt - 1 - slot.rank;  // the last query tile sees the most keys
  const int head = slot.hb % nh, b = slot.hb / nh;
  const int kvh = head / (nh / nkv);
  const int q0 = qt * 128;
  const int n_kv = min((q0 + 127) / kKeys, (s - 1) / kKeys) + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
    }
    mbar_init(pv_done, 1);
    mbar_init(o_done, 1);
    fence_mbar_init();
    tma_prefetch_map(&map_q);
    tma_prefetch_map(&map_kv);
  }
  if (warp == 1) {
    tmem_alloc(tslot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const uint32_t tS0 = tbase, tO = tbase + 2 * kKeys;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producers
    // lane 0: Q, then the K ring; lane 1: the V ring. Two lanes, so a V stage that is still
    // in use never holds back the next K load.
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, L::NSL * kSlice128);
      tma_load_4d(sm + L::Q, &map_q, q_full, 0, q0, head * (HD / 64), b);  // all head_dim slices at once
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % kKStages;
        if (!mbar_wait(&k_empty[st], ((j / kKStages) & 1) ^ 1u, err, kErrTimeoutAttn)) break;
        mbar_arrive_expect_tx(&k_full[st], L::TILE);
        tma_load_4d(sm + L::K + st * L::TILE, &map_kv, &k_full[st], 0, j * kKeys, (nh + kvh) * (HD / 64), b);
      }
    } else if (lane == 1) {
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % kVStages;
        if (!mbar_wait(&v_empty[st], ((j / kVStages) & 1) ^ 1u, err, kErrTimeoutAttn)) break;
        mbar_arrive_expect_tx(&v_full[st], L::TILE);
        tma_load_4d(sm + L::V + st * L::TILE, &map_kv, &v_full[st], 0, j * kKeys, (nh + nkv + kvh) * (HD / 64), b);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // the whole warp runs the issuing loop; elect.sync picks the lane that issues each MMA
    constexpr uint32_t idesc_s = idesc_bf16_f32(128, kKeys, false, false);
    constexpr uint32_t idesc_o = idesc_bf16_f32(128, HD, false, true);
    const uint64_t qd = smem_desc_sw128(smem_addr(sm + L::Q), 16, 1024);
    bool ok = mbar_wait_warp(q_full, 0, err, kErrTimeoutAttn);
    // score buffer j&1 last held P_{j-2}, read by O += P_{j-2} V_{j-2}, which was issued
    // before S_j: MMAs run in issue order, so no wait is needed.
    auto issue_s = [&](int j) -> bool {
      const int st = j & 1, ks = j % kKStages;
      if (!mbar_wait_warp(&k_full[ks], (j / kKStages) & 1, err, kErrTimeoutAttn)) return false;
      tc_fence_after();
      const uint64_t kd = smem_desc_sw128(smem_addr(sm + L::K + ks * L::TILE), 16, 1024);
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        const uint32_t a_off = (kk >> 2) * kSlice128 + (kk & 3) * 32;
        const uint32_t b_off = (kk >> 2) * kSlice64 + (kk & 3) * 32;
        umma_bf16_warp(tS0 + st * kKeys, desc_advance(qd, a_off), desc_advance(kd, b_off), idesc_s, kk > 0 ? 1u : 0u);
      }
      umma_commit_warp(&s_full[st]);
      umma_commit_warp(&k_empty[ks]);
      return true;
    };
    if (ok) ok = issue_s(0);
    for (int j = 0; j < n_kv && ok; ++j) {
      if (j + 1 < n_kv && !(ok = issue_s(j + 1))) break;
      const int st = j & 1, vs = j % kVStages;
      if (!(ok = mbar_wait_warp(&p_full[st], (j >> 1) & 1, err, kErrTimeoutAttn))) break;
      if (!(ok = mbar_wait_warp(&v_full[vs], (j / kVStages) & 1, err, kErrTimeoutAttn))) break;
      tc_fence_after();
      const uint64_t vd = smem_desc_sw128(smem_addr(sm + L::V + vs * L::TILE), kSlice64, 1024);
#pragma unroll
      for (int kk = 0; kk < kKeys / 16; ++kk)  // A = P_j from TMEM: 16 keys = 8 columns per step
        umma_bf16_tmem_a_warp(tO, tS0 + st * kKeys + kk * 8, desc_advance(vd, kk * 2048), idesc_o,
                              (j > 0 || kk > 0) ? 1u : 0u);
      umma_commit_warp(&v_empty[vs]);
      umma_commit_warp(pv_done);
      if (j == n_kv - 1) umma_commit_warp(o_done);
    }
  } else {
    // ------------------------------------------------------------ softmax (warps 2..5)
    const int sub = warp & 3;
    const int row = sub * 32 + lane;
    const int q = q0 + row;
    const uint32_t tl = static_cast<uint32_t>(sub * 32) << 16;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int st = j & 1;
      if (!(ok = mbar_wait_warp(&s_full[st], (j >> 1) & 1, err, kErrTimeoutAttn))) break;
      tc_fence_after();
      float sc[kKeys];
#pragma unroll
      for (int c4 = 0; c4 < kKeys / 32; ++c4) {
        uint32_t r[32];
        tmem_ld_32cols(tS0 + tl + st * kKeys + c4 * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) sc[c4 * 32 + i] = __uint_as_float(r[i]);
      }
      const int key0 = j * kKeys;
      const bool mask_tile = (key0 + kKeys - 1 > q0) || (key0 + kKeys > s);
      if (mask_tile) {  // tiles on the diagonal or past the end: masked raw scores become -inf
#pragma unroll
        for (int c = 0; c < kKeys; ++c)
          if (key0 + c > q || key0 + c >= s) sc[c] = -INFINITY;
      }
      // the max of the raw scores, scaled once (scale > 0; -inf for a row with every key masked)
      float r = sc[0];
#pragma unroll
      for (int c = 1; c + 1 < kKeys; c += 2) r = fmax3(r, sc[c], sc[c + 1]);
      const float mx = fmaxf(r, sc[kKeys - 1]) * scale_log2;
      const bool need = mx > m_ref + kLazyRescale;
      const float m_new = need ? mx : m_ref;
      // rescale O only when a row's max grew past the lazy threshold; O += P_{j-1} V_{j-1} must
      // have finished first (P_j may be written before it has: it goes to the other buffer)
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        if (!(ok = mbar_wait_warp(pv_done, (j - 1) & 1, err, kErrTimeoutAttn))) break;
        tc_fence_after();
        {
          const float factor = need ? ex2(m_ref - m_new) : 1.f;
#pragma unroll
          for (int c4 = 0; c4 < HD / 32; ++c4) {
            uint32_t r[32];
            tmem_ld_32cols(tO + tl + c4 * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * factor);
            tmem_st_32cols(tO + tl + c4 * 32, r);
          }
          tmem_st_wait();
          l *= factor;
        }
      }
      m_ref = m_new;
      uint32_t pw[kKeys / 2];  // P_j as bf16 pairs: key 2c in the low half of column c
      // pairs of keys in the packed fp32x2 unit: one fused scale-and-shift, one add (a masked
      // score stays -inf and gives 0; m_ref is finite, every row seeing key 0 in its first tile)
      const float2 sl = make_float2(scale_log2, scale_log2), nm = make_float2(-m_ref, -m_ref);
      float2 acc = make_float2(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < kKeys / 2; ++c) {
        const float2 v = __ffma2_rn(make_float2(sc[2 * c], sc[2 * c + 1]), sl, nm);
        const float2 pp = make_float2(ex2(v.x), ex2(v.y));
        acc = __fadd2_rn(acc, pp);
        pw[c] = pack_bf16(pp.x, pp.y);
      }
      const float rs = acc.x + acc.y;
      tmem_st_32cols(tS0 + tl + st * kKeys, pw);
      tmem_st_wait();
      l += rs;
      tc_fence_before();
      mbar_arrive(&p_full[st]);
    }
    // the output waits on its own barrier: a parity wait on pv_done could not tell the last
    // product's phase from the one two before it (the softmax may finish its last tile while
    // O += P_{n-2} V_{n-2} has not completed yet)
    if (ok && mbar_wait_warp(o_done, 0, err, kErrTimeoutAttn)) {
      tc_fence_after();
      const float inv = 1.f / l;
      bf16* orow =
          o + (static_cast<int64_t>(b) * s + q) * (static_cast<int64_t>(nh) * HD) + static_cast<int64_t>(head) * HD;
#pragma unroll
      for (int c4 = 0; c4 < HD / 32; ++c4) {
        uint32_t r[32];
        tmem_ld_32cols(tO + tl + c4 * 32, r);
        tmem_ld_wait();
        if (q < s) {
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            uint4 v;
            v.x = pack_bf16(__uint_as_float(r[8 * v4 + 0]) * inv, __uint_as_float(r[8 * v4 + 1]) * inv);
            v.y = pack_bf16(__uint_as_float(r[8 * v4 + 2]) * inv, __uint_as_float(r[8 * v4 + 3]) * inv);
            v.z = pack_bf16(__uint_as_float(r[8 * v4 + 4]) * inv, __uint_as_float(r[8 * v4 + 5]) * inv);
            v.w = pack_bf16(__uint_as_float(r[8 * v4 + 6]) * inv, __uint_as_float(r[8 * v4 + 7]) * inv);
            reinterpret_cast<uint4*>(orow + c4 * 32)[v4] = v;
          }
        }
      }
      if (q < s) lse[(static_cast<int64_t>(b) * nh + head) * s + q] = m_ref + log2f(l);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, 256);
}

template <int HD>
cudaError_t launch(const bf16* qkv, bf16* o, float* lse, int B, int s, int nh, int nkv, int* err, cudaStream_t st) {
  using L = Smem<HD>;
  const int64_t ld = static_cast<int64_t>(nh + 2 * nkv) * HD;
  CUtensorMap map_q, map_kv;
  if (!tma_map_slices(&map_q, qkv, static_cast<uint64_t>(s), static_cast<uint64_t>(B), ld, static_cast<int64_t>(s) * ld,
                      L::NSL, 128) ||
      !tma_map_slices(&map_kv, qkv, static_cast<uint64_t>(s), static_cast<uint64_t>(B), ld,
                      static_cast<int64_t>(s) * ld, L::NSL, kKeys))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_tc_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::BYTES);
  if (e != cudaSuccess) return e;
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(HD));
  attn_fwd_tc_kernel<HD><<<((s + 127) / 128) * nh * B, kThreads, L::BYTES, st>>>(map_q, map_kv, o, lse, s, nh,
                                                                                      nkv, scale_log2, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t attn_fwd(const bf16* qkv, bf16* o, float* lse, int B, int s, int nh, int nkv, int hd, int* err,
                     cudaStream_t st) {
  if (nkv <= 0 || nh % nkv || s <= 0 || B <= 0 || !err) return cudaErrorInvalidValue;
  if ((reinterpret_cast<uintptr_t>(qkv) | reinterpret_cast<uintptr_t>(o)) & 15) return cudaErrorMisalignedAddress;
  if (hd == 64) return launch<64>(qkv, o, lse, B, s, nh, nkv, err, st);
  if (hd == 128) return launch<128>(qkv, o, lse, B, s, nh, nkv, err, st);
  return cudaErrorInvalidValue;
}

}  // namespace mt
