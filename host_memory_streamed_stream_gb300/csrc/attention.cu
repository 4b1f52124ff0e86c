// Causal grouped-query flash attention, forward and backward, for the layer templates.
//
// Forward: one CTA per (64-query tile, query head, sequence); four warps own 16 query
// rows each. K/V tiles of 64 keys stream through a double-buffered shared-memory ring
// (cp.async); scores and the running output stay in registers with an online softmax in
// base 2. Tiles above the diagonal are skipped (causal). The row statistics are saved as
// lse2 = max + log2(sum), in units of scores scaled by log2(e)/sqrt(hd).
//
// Backward, deterministic (no atomics): a KV-outer kernel accumulates dK and dV for 64
// keys over every query tile of every query head of the group, in a fixed order; a
// Q-outer kernel accumulates dQ over the key tiles. delta = rowsum(dO * O) comes first.
//
// Tensor-core work uses mma.sync m16n8k16 (bf16 in, fp32 accumulate) fed by ldmatrix
// from padded shared-memory rows (row pitch hd + 8 elements: conflict-free ldmatrix).
#include <cstdint>

#include "kernels.h"

namespace mt {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ uint32_t saddr(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(saddr(dst)), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Copy `rows` rows of HD bf16 (global row stride ld, first row `row0`, valid rows < nvalid)
// into shared memory with pitch HD + 8; invalid rows are zero-filled.
template <int HD>
__device__ __forceinline__ void load_tile(bf16* s, const bf16* g, int64_t ld, int row0, int rows, int nvalid) {
  constexpr int CH = HD / 8;  // 16-byte chunks per row
  for (int i = threadIdx.x; i < rows * CH; i += blockDim.x) {
    const int r = i / CH, c = i % CH;
    const bool ok = (row0 + r) < nvalid;
    const bf16* src = ok ? g + static_cast<int64_t>(row0 + r) * ld + c * 8 : g;
    cp_async16(s + r * (HD + 8) + c * 8, src, ok);
  }
}

// A fragments (16 x 16) of rows [r0, r0+16) and columns [k0, k0+16) of a padded tile.
template <int HD>
__device__ __forceinline__ void frag_a(const bf16* s, int r0, int k0, uint32_t (&a)[4]) {
  const int lane = threadIdx.x & 31;
  const bf16* p = s + (r0 + (lane & 15)) * (HD + 8) + k0 + (lane >> 4) * 8;
  ldsm_x4(saddr(p), a[0], a[1], a[2], a[3]);
}
// B fragments for two 8-column n-tiles [n0, n0+16) x k [k0, k0+16) from storage [n][k].
template <int HD>
__device__ __forceinline__ void frag_b_nk(const bf16* s, int n0, int k0, uint32_t (&b)[4]) {
  const int lane = threadIdx.x & 31;
  const bf16* p = s + (n0 + ((lane >> 4) << 3) + (lane & 7)) * (HD + 8) + k0 + ((lane >> 3) & 1) * 8;
  ldsm_x4(saddr(p), b[0], b[1], b[2], b[3]);
}
// B fragments for two n-tiles [n0, n0+16) x k [k0, k0+16) from storage [k][n] (transposing load).
template <int HD>
__device__ __forceinline__ void frag_b_kn(const bf16* s, int k0, int n0, uint32_t (&b)[4]) {
  const int lane = threadIdx.x & 31;
  const bf16* p = s + (k0 + ((lane >> 3) & 1) * 8 + (lane & 7)) * (HD + 8) + n0 + (lane >> 4) * 8;
  ldsm_x4_t(saddr(p), b[0], b[1], b[2], b[3]);
}

// ------------------------------------------------------------------ forward
template <int HD>
__global__ void __launch_bounds__(128) attn_fwd_kernel(const bf16* __restrict__ qkv, bf16* __restrict__ o,
                                                       float* __restrict__ lse, int s, int nh, int nkv,
                                                       float scale_log2) {
  constexpr int BQ = 64, BK = 64, P = HD + 8;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  bf16* Qs = reinterpret_cast<bf16*>(smem_raw);
  bf16* Ks = Qs + BQ * P;        // [2][BK][P]
  bf16* Vs = Ks + 2 * BK * P;    // [2][BK][P]

  const int qt = blockIdx.x, head = blockIdx.y, b = blockIdx.z;
  const int kvh = head / (nh / nkv);
  const int64_t ld = static_cast<int64_t>(nh + 2 * nkv) * HD;
  const bf16* base = qkv + static_cast<int64_t>(b) * s * ld;
  const bf16* qg = base + static_cast<int64_t>(head) * HD;
  const bf16* kg = base + static_cast<int64_t>(nh + kvh) * HD;
  const bf16* vg = base + static_cast<int64_t>(nh + nkv + kvh) * HD;
  const int q0 = qt * BQ;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;

  load_tile<HD>(Qs, qg, ld, q0, BQ, s);
  cp_commit();
  load_tile<HD>(Ks, kg, ld, 0, BK, s);
  load_tile<HD>(Vs, vg, ld, 0, BK, s);
  cp_commit();

  const int last_tile = min((q0 + BQ - 1) / BK, (s - 1) / BK);
  float m_i[2] = {-INFINITY, -INFINITY}, l_i[2] = {0.f, 0.f};
  float acc[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

  cp_wait<1>();
  __syncthreads();
  uint32_t qf[HD / 16][4];
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk) frag_a<HD>(Qs, warp * 16, kk * 16, qf[kk]);
  const int row_a = q0 + warp * 16 + g, row_b = row_a + 8;

  for (int j = 0; j <= last_tile; ++j) {
    if (j + 1 <= last_tile) {
      load_tile<HD>(Ks + ((j + 1) & 1) * BK * P, kg, ld, (j + 1) * BK, BK, s);
      load_tile<HD>(Vs + ((j + 1) & 1) * BK * P, vg, ld, (j + 1) * BK, BK, s);
    }
    cp_commit();
    cp_wait<1>();
    __syncthreads();
    const bf16* Kt = Ks + (j & 1) * BK * P;
    const bf16* Vt = Vs + (j & 1) * BK * P;
    float sc[BK / 8][4];
#pragma unroll
    for (int i = 0; i < BK / 8; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
#pragma unroll
      for (int np = 0; np < BK / 16; ++np) {
        uint32_t bb[4];
        frag_b_nk<HD>(Kt, np * 16, kk * 16, bb);
        mma16816(sc[2 * np], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], bb[0], bb[1]);
        mma16816(sc[2 * np + 1], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], bb[2], bb[3]);
      }
    }
    const bool need_mask = (j * BK + BK - 1 > q0) || (j * BK + BK > s);
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < BK / 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = j * BK + nt * 8 + 2 * c + (e & 1);
        const int row = (e < 2) ? row_a : row_b;
        float v = sc[nt][e] * scale_log2;
        if (need_mask && (key > row || key >= s)) v = -INFINITY;
        sc[nt][e] = v;
        mx[e >> 1] = fmaxf(mx[e >> 1], v);
      }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
    }
    float corr[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const float mn = fmaxf(m_i[r], mx[r]);
      corr[r] = (m_i[r] == -INFINITY) ? 0.f : exp2f(m_i[r] - mn);
      m_i[r] = mn;
      l_i[r] *= corr[r];
    }
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) {
      acc[i][0] *= corr[0];
      acc[i][1] *= corr[0];
      acc[i][2] *= corr[1];
      acc[i][3] *= corr[1];
    }
#pragma unroll
    for (int nt = 0; nt < BK / 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float mref = m_i[e >> 1];
        const float p = (sc[nt][e] == -INFINITY) ? 0.f : exp2f(sc[nt][e] - mref);
        sc[nt][e] = p;
        l_i[e >> 1] += p;
      }
    }
#pragma unroll
    for (int kk = 0; kk < BK / 16; ++kk) {
      const uint32_t a0 = pack2(sc[2 * kk][0], sc[2 * kk][1]);
      const uint32_t a1 = pack2(sc[2 * kk][2], sc[2 * kk][3]);
      const uint32_t a2 = pack2(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
      const uint32_t a3 = pack2(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
#pragma unroll
      for (int dp = 0; dp < HD / 16; ++dp) {
        uint32_t bb[4];
        frag_b_kn<HD>(Vt, kk * 16, dp * 16, bb);
        mma16816(acc[2 * dp], a0, a1, a2, a3, bb[0], bb[1]);
        mma16816(acc[2 * dp + 1], a0, a1, a2, a3, bb[2], bb[3]);
      }
    }
    __syncthreads();
  }
  cp_wait<0>();

#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l_i[r] += __shfl_xor_sync(0xffffffffu, l_i[r], 1);
    l_i[r] += __shfl_xor_sync(0xffffffffu, l_i[r], 2);
  }
  const float inv0 = 1.f / l_i[0], inv1 = 1.f / l_i[1];
  bf16* og = o + (static_cast<int64_t>(b) * s) * (static_cast<int64_t>(nh) * HD) + static_cast<int64_t>(head) * HD;
  const int64_t old = static_cast<int64_t>(nh) * HD;
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) {
    const int col = i * 8 + 2 * c;
    if (row_a < s)
      *reinterpret_cast<uint32_t*>(og + row_a * old + col) = pack2(acc[i][0] * inv0, acc[i][1] * inv0);
    if (row_b < s)
      *reinterpret_cast<uint32_t*>(og + row_b * old + col) = pack2(acc[i][2] * inv1, acc[i][3] * inv1);
  }
  if (c == 0) {
    float* lg = lse + (static_cast<int64_t>(b) * nh + head) * s;
    if (row_a < s) lg[row_a] = m_i[0] + log2f(l_i[0]);
    if (row_b < s) lg[row_b] = m_i[1] + log2f(l_i[1]);
  }
}

// ------------------------------------------------------------------ backward: delta
// delta[b, n, i] = sum_d dO[i, n, d] * O[i, n, d]; one warp per (token, head).
__global__ void attn_delta_kernel(const bf16* __restrict__ o, const bf16* __restrict__ dout,
                                  float* __restrict__ delta, int B, int s, int nh, int hd) {
  const int64_t wid = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= static_cast<int64_t>(B) * s * nh) return;
  const int head = static_cast<int>(wid % nh);
  const int64_t t = wid / nh;
  const bf16* op = o + t * nh * hd + static_cast<int64_t>(head) * hd;
  const bf16* dp = dout + t * nh * hd + static_cast<int64_t>(head) * hd;
  float acc = 0.f;
  for (int d = lane * 2; d < hd; d += 64) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(op + d));
    const float2 bb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(dp + d));
    acc += a.x * bb.x + a.y * bb.y;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) {
    const int b = static_cast<int>(t / s), i = static_cast<int>(t % s);
    delta[(static_cast<int64_t>(b) * nh + head) * s + i] = acc;
  }
}

// ------------------------------------------------------------------ backward: dQ
template <int HD>
__global__ void __launch_bounds__(128) attn_bwd_dq_kernel(const bf16* __restrict__ qkv, const float* __restrict__ lse,
                                                          const float* __restrict__ delta,
                                                          const bf16* __restrict__ dout, bf16* __restrict__ dqkv,
                                                          int s, int nh, int nkv, float scale_log2, float scale) {
  constexpr int BQ = 64, BK = 64, P = HD + 8;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  bf16* Qs = reinterpret_cast<bf16*>(smem_raw);  // [BQ][P]
  bf16* Ds = Qs + BQ * P;                        // dO [BQ][P]
  bf16* Ks = Ds + BQ * P;                        // [2][BK][P]
  bf16* Vs = Ks + 2 * BK * P;                    // [2][BK][P]

  const int qt = blockIdx.x, head = blockIdx.y, b = blockIdx.z;
  const int kvh = head / (nh / nkv);
  const int64_t ld = static_cast<int64_t>(nh + 2 * nkv) * HD;
  const int64_t ldo = static_cast<int64_t>(nh) * HD;
  const bf16* base = qkv + static_cast<int64_t>(b) * s * ld;
  const bf16* qg = base + static_cast<int64_t>(head) * HD;
  const bf16* kg = base + static_cast<int64_t>(nh + kvh) * HD;
  const bf16* vg = base + static_cast<int64_t>(nh + nkv + kvh) * HD;
  const bf16* dog = dout + static_cast<int64_t>(b) * s * ldo + static_cast<int64_t>(head) * HD;
  const int q0 = qt * BQ;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;

  load_tile<HD>(Qs, qg, ld, q0, BQ, s);
  load_tile<HD>(Ds, dog, ldo, q0, BQ, s);
  cp_commit();
  load_tile<HD>(Ks, kg, ld, 0, BK, s);
  load_tile<HD>(Vs, vg, ld, 0, BK, s);
  cp_commit();

  const int row_a = q0 + warp * 16 + g, row_b = row_a + 8;
  const float* lrow = lse + (static_cast<int64_t>(b) * nh + head) * s;
  const float* drow = delta + (static_cast<int64_t>(b) * nh + head) * s;
  const float lse_a = row_a < s ? lrow[row_a] : 0.f, lse_b = row_b < s ? lrow[row_b] : 0.f;
  const float del_a = row_a < s ? drow[row_a] : 0.f, del_b = row_b < s ? drow[row_b] : 0.f;

  cp_wait<1>();
  __syncthreads();
  uint32_t qf[HD / 16][4], df[HD / 16][4];
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk) {
    frag_a<HD>(Qs, warp * 16, kk * 16, qf[kk]);
    frag_a<HD>(Ds, warp * 16, kk * 16, df[kk]);
  }
  float acc[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

  const int last_tile = min((q0 + BQ - 1) / BK, (s - 1) / BK);
  for (int j = 0; j <= last_tile; ++j) {
    if (j + 1 <= last_tile) {
      load_tile<HD>(Ks + ((j + 1) & 1) * BK * P, kg, ld, (j + 1) * BK, BK, s);
      load_tile<HD>(Vs + ((j + 1) & 1) * BK * P, vg, ld, (j + 1) * BK, BK, s);
    }
    cp_commit();
    cp_wait<1>();
    __syncthreads();
    const bf16* Kt = Ks + (j & 1) * BK * P;
    const bf16* Vt = Vs + (j & 1) * BK * P;
    float sc[BK / 8][4], dp[BK / 8][4];
#pragma unroll
    for (int i = 0; i < BK / 8; ++i) {
      sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
      dp[i][0] = dp[i][1] = dp[i][2] = dp[i][3] = 0.f;
    }
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
#pragma unroll
      for (int np = 0; np < BK / 16; ++np) {
        uint32_t bb[4];
        frag_b_nk<HD>(Kt, np * 16, kk * 16, bb);
        mma16816(sc[2 * np], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], bb[0], bb[1]);
        mma16816(sc[2 * np + 1], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], bb[2], bb[3]);
        frag_b_nk<HD>(Vt, np * 16, kk * 16, bb);
        mma16816(dp[2 * np], df[kk][0], df[kk][1], df[kk][2], df[kk][3], bb[0], bb[1]);
        mma16816(dp[2 * np + 1], df[kk][0], df[kk][1], df[kk][2], df[kk][3], bb[2], bb[3]);
      }
    }
    // dS = P * (dP - delta), P = exp2(S * scale_log2 - lse2), masked entries 0
#pragma unroll
    for (int nt = 0; nt < BK / 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = j * BK + nt * 8 + 2 * c + (e & 1);
        const int row = (e < 2) ? row_a : row_b;
        const float l2 = (e < 2) ? lse_a : lse_b;
        const float dl = (e < 2) ? del_a : del_b;
        const bool valid = key <= row && key < s && row < s;
        const float p = valid ? exp2f(sc[nt][e] * scale_log2 - l2) : 0.f;
        sc[nt][e] = p * (dp[nt][e] - dl);
      }
    }
#pragma unroll
    for (int kk = 0; kk < BK / 16; ++kk) {
      const uint32_t a0 = pack2(sc[2 * kk][0], sc[2 * kk][1]);
      const uint32_t a1 = pack2(sc[2 * kk][2], sc[2 * kk][3]);
      const uint32_t a2 = pack2(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
      const uint32_t a3 = pack2(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
#pragma unroll
      for (int dpi = 0; dpi < HD / 16; ++dpi) {
        uint32_t bb[4];
        frag_b_kn<HD>(Kt, kk * 16, dpi * 16, bb);
        mma16816(acc[2 * dpi], a0, a1, a2, a3, bb[0], bb[1]);
        mma16816(acc[2 * dpi + 1], a0, a1, a2, a3, bb[2], bb[3]);
      }
    }
    __syncthreads();
  }
  cp_wait<0>();
  bf16* dqg = dqkv + static_cast<int64_t>(b) * s * ld + static_cast<int64_t>(head) * HD;
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) {
    const int col = i * 8 + 2 * c;
    if (row_a < s) *reinterpret_cast<uint32_t*>(dqg + row_a * ld + col) = pack2(acc[i][0] * scale, acc[i][1] * scale);
    if (row_b < s) *reinterpret_cast<uint32_t*>(dqg + row_b * ld + col) = pack2(acc[i][2] * scale, acc[i][3] * scale);
  }
}

// ------------------------------------------------------------------ backward: dK, dV
// One CTA per (64-key tile, kv head, sequence); warp w owns keys [16w, 16w+16) of the tile.
// Loops over the group's query heads, then over 32-query tiles, in ascending order.
template <int HD>
__global__ void __launch_bounds__(128) attn_bwd_dkdv_kernel(const bf16* __restrict__ qkv,
                                                            const float* __restrict__ lse,
                                                            const float* __restrict__ delta,
                                                            const bf16* __restrict__ dout, bf16* __restrict__ dqkv,
                                                            int s, int nh, int nkv, float scale_log2, float scale) {
  constexpr int BKV = 64, BQ = 32, P = HD + 8;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  bf16* Ks = reinterpret_cast<bf16*>(smem_raw);  // [BKV][P]
  bf16* Vs = Ks + BKV * P;                       // [BKV][P]
  bf16* Qs = Vs + BKV * P;                       // [2][BQ][P]
  bf16* Ds = Qs + 2 * BQ * P;                    // dO [2][BQ][P]
  float* Ls = reinterpret_cast<float*>(Ds + 2 * BQ * P);  // [2][BQ] lse
  float* Es = Ls + 2 * BQ;                                // [2][BQ] delta

  const int kt = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int group = nh / nkv;
  const int64_t ld = static_cast<int64_t>(nh + 2 * nkv) * HD;
  const int64_t ldo = static_cast<int64_t>(nh) * HD;
  const bf16* base = qkv + static_cast<int64_t>(b) * s * ld;
  const bf16* kg = base + static_cast<int64_t>(nh + kvh) * HD;
  const bf16* vg = base + static_cast<int64_t>(nh + nkv + kvh) * HD;
  const int k0 = kt * BKV;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int key_a = k0 + warp * 16 + g, key_b = key_a + 8;

  load_tile<HD>(Ks, kg, ld, k0, BKV, s);
  load_tile<HD>(Vs, vg, ld, k0, BKV, s);
  cp_commit();

  float dk[HD / 8][4], dv[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) {
    dk[i][0] = dk[i][1] = dk[i][2] = dk[i][3] = 0.f;
    dv[i][0] = dv[i][1] = dv[i][2] = dv[i][3] = 0.f;
  }

  const int first_qt = k0 / BQ;
  const int n_qt = (s + BQ - 1) / BQ;
  const int per_head = n_qt - first_qt;
  const int total = group * per_head;

  auto issue = [&](int it, int buf) {
    const int hq = kvh * group + it / per_head;
    const int qt = first_qt + it % per_head;
    const bf16* qg = base + static_cast<int64_t>(hq) * HD;
    const bf16* dog = dout + static_cast<int64_t>(b) * s * ldo + static_cast<int64_t>(hq) * HD;
    load_tile<HD>(Qs + buf * BQ * P, qg, ld, qt * BQ, BQ, s);
    load_tile<HD>(Ds + buf * BQ * P, dog, ldo, qt * BQ, BQ, s);
    if (threadIdx.x < BQ) {
      const int q = qt * BQ + threadIdx.x;
      const int64_t off = (static_cast<int64_t>(b) * nh + hq) * s + q;
      Ls[buf * BQ + threadIdx.x] = q < s ? lse[off] : 0.f;
      Es[buf * BQ + threadIdx.x] = q < s ? delta[off] : 0.f;
    }
  };
  if (total > 0) issue(0, 0);
  cp_commit();

  for (int it = 0; it < total; ++it) {
    const int buf = it & 1;
    const int q0 = (first_qt + it % per_head) * BQ;
    if (it + 1 < total) issue(it + 1, buf ^ 1);
    cp_commit();
    cp_wait<1>();
    __syncthreads();
    const bf16* Qt = Qs + buf * BQ * P;
    const bf16* Dt = Ds + buf * BQ * P;
    const float* Lt = Ls + buf * BQ;
    const float* Et = Es + buf * BQ;
    float st[BQ / 8][4], dpt[BQ / 8][4];
#pragma unroll
    for (int i = 0; i < BQ / 8; ++i) {
      st[i][0] = st[i][1] = st[i][2] = st[i][3] = 0.f;
      dpt[i][0] = dpt[i][1] = dpt[i][2] = dpt[i][3] = 0.f;
    }
    // S^T = K Q^T and dP^T = V dO^T for this warp's 16 keys x 32 queries
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
      uint32_t ka[4], va[4];
      frag_a<HD>(Ks, warp * 16, kk * 16, ka);
      frag_a<HD>(Vs, warp * 16, kk * 16, va);
#pragma unroll
      for (int np = 0; np < BQ / 16; ++np) {
        uint32_t bb[4];
        frag_b_nk<HD>(Qt, np * 16, kk * 16, bb);
        mma16816(st[2 * np], ka[0], ka[1], ka[2], ka[3], bb[0], bb[1]);
        mma16816(st[2 * np + 1], ka[0], ka[1], ka[2], ka[3], bb[2], bb[3]);
        frag_b_nk<HD>(Dt, np * 16, kk * 16, bb);
        mma16816(dpt[2 * np], va[0], va[1], va[2], va[3], bb[0], bb[1]);
        mma16816(dpt[2 * np + 1], va[0], va[1], va[2], va[3], bb[2], bb[3]);
      }
    }
    // P^T and dS^T (rows = keys, columns = queries)
#pragma unroll
    for (int nt = 0; nt < BQ / 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int ql = nt * 8 + 2 * c + (e & 1);
        const int q = q0 + ql;
        const int key = (e < 2) ? key_a : key_b;
        const bool valid = key <= q && q < s && key < s;
        const float p = valid ? exp2f(st[nt][e] * scale_log2 - Lt[ql]) : 0.f;
        st[nt][e] = p;
        dpt[nt][e] = p * (dpt[nt][e] - Et[ql]);
      }
    }
    // dV += P^T dO, dK += dS^T Q
#pragma unroll
    for (int kk = 0; kk < BQ / 16; ++kk) {
      const uint32_t p0 = pack2(st[2 * kk][0], st[2 * kk][1]);
      const uint32_t p1 = pack2(st[2 * kk][2], st[2 * kk][3]);
      const uint32_t p2 = pack2(st[2 * kk + 1][0], st[2 * kk + 1][1]);
      const uint32_t p3 = pack2(st[2 * kk + 1][2], st[2 * kk + 1][3]);
      const uint32_t d0 = pack2(dpt[2 * kk][0], dpt[2 * kk][1]);
      const uint32_t d1 = pack2(dpt[2 * kk][2], dpt[2 * kk][3]);
      const uint32_t d2 = pack2(dpt[2 * kk + 1][0], dpt[2 * kk + 1][1]);
      const uint32_t d3 = pack2(dpt[2 * kk + 1][2], dpt[2 * kk + 1][3]);
#pragma unroll
      for (int dpi = 0; dpi < HD / 16; ++dpi) {
        uint32_t bb[4];
        frag_b_kn<HD>(Dt, kk * 16, dpi * 16, bb);
        mma16816(dv[2 * dpi], p0, p1, p2, p3, bb[0], bb[1]);
        mma16816(dv[2 * dpi + 1], p0, p1, p2, p3, bb[2], bb[3]);
        frag_b_kn<HD>(Qt, kk * 16, dpi * 16, bb);
        mma16816(dk[2 * dpi], d0, d1, d2, d3, bb[0], bb[1]);
        mma16816(dk[2 * dpi + 1], d0, d1, d2, d3, bb[2], bb[3]);
      }
    }
    __syncthreads();
  }
  cp_wait<0>();
  bf16* dkg = dqkv + static_cast<int64_t>(b) * s * ld + static_cast<int64_t>(nh + kvh) * HD;
  bf16* dvg = dqkv + static_cast<int64_t>(b) * s * ld + static_cast<int64_t>(nh + nkv + kvh) * HD;
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) {
    const int col = i * 8 + 2 * c;
    if (key_a < s) {
      *reinterpret_cast<uint32_t*>(dkg + key_a * ld + col) = pack2(dk[i][0] * scale, dk[i][1] * scale);
      *reinterpret_cast<uint32_t*>(dvg + key_a * ld + col) = pack2(dv[i][0], dv[i][1]);
    }
    if (key_b < s) {
      *reinterpret_cast<uint32_t*>(dkg + key_b * ld + col) = pack2(dk[i][2] * scale, dk[i][3] * scale);
      *reinterpret_cast<uint32_t*>(dvg + key_b * ld + col) = pack2(dv[i][2], dv[i][3]);
    }
  }
}

template <int HD>
size_t fwd_smem() {
  return static_cast<size_t>(64 + 4 * 64) * (HD + 8) * 2;
}
template <int HD>
size_t dq_smem() {
  return static_cast<size_t>(2 * 64 + 4 * 64) * (HD + 8) * 2;
}
template <int HD>
size_t dkdv_smem() {
  return static_cast<size_t>(2 * 64 + 4 * 32) * (HD + 8) * 2 + 4 * 32 * sizeof(float);
}

template <int HD>
cudaError_t fwd_impl(const bf16* qkv, bf16* o, float* lse, int B, int s, int nh, int nkv, cudaStream_t st) {
  const size_t sm = fwd_smem<HD>();
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(sm));
  if (e != cudaSuccess) return e;
  dim3 grid((s + 63) / 64, nh, B);
  const float scale_log2 = kLog2e / sqrtf(static_cast<float>(HD));
  attn_fwd_kernel<HD><<<grid, 128, sm, st>>>(qkv, o, lse, s, nh, nkv, scale_log2);
  return cudaGetLastError();
}

template <int HD>
cudaError_t bwd_impl(const bf16* qkv, const bf16* o, const float* lse, const bf16* dout, bf16* dqkv, float* delta,
                     int B, int s, int nh, int nkv, cudaStream_t st) {
  const int64_t warps = static_cast<int64_t>(B) * s * nh;
  attn_delta_kernel<<<static_cast<unsigned>((warps * 32 + 255) / 256), 256, 0, st>>>(o, dout, delta, B, s, nh, HD);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const float scale_log2 = kLog2e / sqrtf(static_cast<float>(HD));
  const float scale = 1.f / sqrtf(static_cast<float>(HD));
  size_t sm = dq_smem<HD>();
  e = cudaFuncSetAttribute(attn_bwd_dq_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sm));
  if (e != cudaSuccess) return e;
  attn_bwd_dq_kernel<HD><<<dim3((s + 63) / 64, nh, B), 128, sm, st>>>(qkv, lse, delta, dout, dqkv, s, nh, nkv,
                                                                        scale_log2, scale);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  sm = dkdv_smem<HD>();
  e = cudaFuncSetAttribute(attn_bwd_dkdv_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(sm));
  if (e != cudaSuccess) return e;
  attn_bwd_dkdv_kernel<HD><<<dim3((s + 63) / 64, nkv, B), 128, sm, st>>>(qkv, lse, delta, dout, dqkv, s, nh, nkv,
                                                                           scale_log2, scale);
  return cudaGetLastError();
}

}  // namespace

cudaError_t attn_fwd(const bf16* qkv, bf16* o, float* lse, int B, int s, int nh, int nkv, int hd, cudaStream_t st) {
  if (nkv <= 0 || nh % nkv || s <= 0) return cudaErrorInvalidValue;
  if (hd == 64) return fwd_impl<64>(qkv, o, lse, B, s, nh, nkv, st);
  if (hd == 128) return fwd_impl<128>(qkv, o, lse, B, s, nh, nkv, st);
  return cudaErrorInvalidValue;
}

cudaError_t attn_bwd(const bf16* qkv, const bf16* o, const float* lse, const bf16* dout, bf16* dqkv, float* delta,
                     int B, int s, int nh, int nkv, int hd, cudaStream_t st) {
  if (nkv <= 0 || nh % nkv || s <= 0) return cudaErrorInvalidValue;
  if (hd == 64) return bwd_impl<64>(qkv, o, lse, dout, dqkv, delta, B, s, nh, nkv, st);
  if (hd == 128) return bwd_impl<128>(qkv, o, lse, dout, dqkv, delta, B, s, nh, nkv, st);
  return cudaErrorInvalidValue;
}

}  // namespace mt
