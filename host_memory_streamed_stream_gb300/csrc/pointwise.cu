// Memory-bound kernels of the layer templates: RMSNorm (forward, backward with a
// deterministic two-stage gain reduction), rotate-half RoPE, SwiGLU, embedding
// gather / ordered scatter, cross-entropy and small reductions. Each moves its
// bytes once with 16-byte (or 8-byte) vector accesses, coalesced along rows, and
// reduces with warp shuffles. None uses floating-point atomics, so every result
// is bit-reproducible.
#include <algorithm>
#include <cstdint>

#include "kernels.h"

namespace mt {

namespace {

constexpr int kMaxVec = 8;  // float4 chunks per thread kept in registers (h <= 8192 at 256 threads)

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
// Sum over the block (blockDim multiple of 32, <= 1024); every thread gets the result.
__device__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  float t = 0.f;
  for (int i = 0; i < nw; ++i) t += red[i];  // same order in every thread
  return t;
}

__device__ __forceinline__ float4 load_bf16x4(const bf16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&u.x);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&u.y);
  const float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
  return make_float4(fa.x, fa.y, fb.x, fb.y);
}
__device__ __forceinline__ void store_bf16x4(bf16* p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

int norm_threads(int h) {
  int t = h / 4 / 4;  // aim for ~4 float4 per thread
  t = (t + 31) / 32 * 32;
  if (t < 32) t = 32;
  if (t > 256) t = 256;
  return t;
}

// ------------------------------------------------------------------ RMSNorm
__global__ void rmsnorm_fwd_kernel(const float* __restrict__ x, const bf16* __restrict__ gamma, bf16* __restrict__ y,
                                   float* __restrict__ rstd, int h, float eps) {
  __shared__ float red[32];
  const int row = blockIdx.x;
  const int nv = h >> 2;
  const float4* xr = reinterpret_cast<const float4*>(x + static_cast<int64_t>(row) * h);
  float4 v[kMaxVec];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < kMaxVec; ++k) {
    const int i = threadIdx.x + k * blockDim.x;
    v[k] = (i < nv) ? xr[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    ss += v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z + v[k].w * v[k].w;
  }
  ss = block_sum(ss, red);
  const float r = rsqrtf(ss / static_cast<float>(h) + eps);
  if (threadIdx.x == 0) rstd[row] = r;
  bf16* yr = y + static_cast<int64_t>(row) * h;
#pragma unroll
  for (int k = 0; k < kMaxVec; ++k) {
    const int i = threadIdx.x + k * blockDim.x;
    if (i < nv) {
      const float4 g = load_bf16x4(gamma + 4 * i);
      store_bf16x4(yr + 4 * i, make_float4(v[k].x * r * g.x, v[k].y * r * g.y, v[k].z * r * g.z, v[k].w * r * g.w));
    }
  }
}

// cp.async (16 bytes, L1 bypassed) global -> shared, in commit groups.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most n of this thread's committed groups are still in flight (n < 4).
__device__ __forceinline__ void cp_async_wait(int n) {
  switch (n) {
    case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
    case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
    default: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
  }
}

// RMSNorm backward. One CTA per block of consecutive rows (two CTAs per SM), VPT float4
// columns per thread (h = 4 * VPT * blockDim), rows in order with the loads of the next
// `stages - 1` rows in flight: each thread copies its own columns of dy and x for a row into a
// shared-memory ring (cp.async) and reads back only what it copied, so the ring needs no
// barrier; the row reduction is the only block-wide step. dres is read straight from global
// memory at the start of the row, ahead of the reduction. Each CTA accumulates dy * xhat over
// its rows in row order into its own partial row (the first stage of the gain reduction).
template <int VPT>
__global__ void __launch_bounds__(256, 2)
    rmsnorm_bwd_async_kernel(const float* __restrict__ dy, const float* __restrict__ x, const bf16* __restrict__ gamma,
                             const float* __restrict__ rstd, const float* dres, float* dx, bf16* __restrict__ dx_bf16,
                             float* __restrict__ partial, int T, int h, int rows_per_part, int stages) {
  extern __shared__ float4 ring[];  // [stages][2][h / 4]: dy, x
  __shared__ float red[32];
  const int nv = h >> 2;
  const int r0 = blockIdx.x * rows_per_part;
  const int r1 = min(T, r0 + rows_per_part);
  float4 g[VPT], acc[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int i = threadIdx.x + k * blockDim.x;
    g[k] = load_bf16x4(gamma + 4 * i);
    acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  auto issue = [&](int row, int st) {
    if (row < r1) {
      const int64_t off = static_cast<int64_t>(row) * h;
      float4* sd = ring + static_cast<size_t>(st) * 2 * nv;
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int i = threadIdx.x + k * blockDim.x;
        cp_async16(sd + i, dy + off + 4 * i);
        cp_async16(sd + nv + i, x + off + 4 * i);
      }
    }
    cp_async_commit();  // one group per row slot, empty past the last row
  };
  for (int st = 0; st < stages; ++st) issue(r0 + st, st);
  const float inv_h = 1.f / static_cast<float>(h);
  int st = 0;
  for (int row = r0; row < r1; ++row) {
    const int64_t off = static_cast<int64_t>(row) * h;
    float4 d[VPT];
    if (dres) {
#pragma unroll
      for (int k = 0; k < VPT; ++k) d[k] = reinterpret_cast<const float4*>(dres + off)[threadIdx.x + k * blockDim.x];
    }
    const float r = rstd[row];
    cp_async_wait(stages - 1);  // this row's group has landed
    const float4* sd = ring + static_cast<size_t>(st) * 2 * nv;
    float4 dv[VPT], xa[VPT];
    float sa = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int i = threadIdx.x + k * blockDim.x;
      dv[k] = sd[i];
      const float4 v = sd[nv + i];
      xa[k] = make_float4(v.x * r, v.y * r, v.z * r, v.w * r);
      sa += dv[k].x * g[k].x * xa[k].x + dv[k].y * g[k].y * xa[k].y + dv[k].z * g[k].z * xa[k].z +
            dv[k].w * g[k].w * xa[k].w;
      acc[k].x += dv[k].x * xa[k].x;
      acc[k].y += dv[k].y * xa[k].y;
      acc[k].z += dv[k].z * xa[k].z;
      acc[k].w += dv[k].w * xa[k].w;
    }
    issue(row + stages, st);  // this thread's slots of the stage are read: refill them
    sa = block_sum(sa, red);
    const float m = sa * inv_h;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int i = threadIdx.x + k * blockDim.x;
      float4 o;
      o.x = r * (dv[k].x * g[k].x - xa[k].x * m);
      o.y = r * (dv[k].y * g[k].y - xa[k].y * m);
      o.z = r * (dv[k].z * g[k].z - xa[k].z * m);
      o.w = r * (dv[k].w * g[k].w - xa[k].w * m);
      if (dres) {
        o.x += d[k].x;
        o.y += d[k].y;
        o.z += d[k].z;
        o.w += d[k].w;
      }
      reinterpret_cast<float4*>(dx + off)[i] = o;
      if (dx_bf16) store_bf16x4(dx_bf16 + off + 4 * i, o);
    }
    st = st + 1 == stages ? 0 : st + 1;
  }
  cp_async_wait(0);
  float* pr = partial + static_cast<int64_t>(blockIdx.x) * h;
#pragma unroll
  for (int k = 0; k < VPT; ++k) reinterpret_cast<float4*>(pr)[threadIdx.x + k * blockDim.x] = acc[k];
}

// dgamma[j] = sum over parts of partial[p][j] in a fixed order: group g (0..7) sums parts
// g, g + 8, g + 16, ... in that order, then the eight group sums are added g = 0..7. One block
// covers 32 columns with 8 x 32 threads, so each thread walks parts / 8 rows instead of all.
constexpr int kReduceGroups = 8;
__global__ void reduce_parts_kernel(const float* __restrict__ partial, bf16* __restrict__ out, int parts, int h) {
  __shared__ float acc[kReduceGroups][32];
  const int c = threadIdx.x & 31, g = threadIdx.x >> 5;
  const int j = blockIdx.x * 32 + c;
  float sum = 0.f;
  if (j < h)
    for (int p = g; p < parts; p += kReduceGroups) sum += partial[static_cast<int64_t>(p) * h + j];
  acc[g][c] = sum;
  __syncthreads();
  if (g == 0 && j < h) {
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < kReduceGroups; ++k) t += acc[k][c];
    out[j] = __float2bfloat16_rn(t);
  }
}

// ------------------------------------------------------------------ RoPE
// One thread per (token, head, pair of rotation indices i, i+1 < hd/2).
__global__ void rope_kernel(bf16* __restrict__ qkv, int64_t ld, int T, int seq, int heads, int hd,
                            const float* __restrict__ cs, bool inverse) {
  const int half = hd >> 1;
  const int pairs = half >> 1;
  const int64_t total = static_cast<int64_t>(T) * heads * pairs;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int ip = static_cast<int>(idx % pairs);
    const int64_t th = idx / pairs;
    const int head = static_cast<int>(th % heads);
    const int t = static_cast<int>(th / heads);
    const int pos = t % seq;
    const int i = ip * 2;
    bf16* base = qkv + static_cast<int64_t>(t) * ld + static_cast<int64_t>(head) * hd;
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(base + i));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(base + half + i));
    const float4 c = *reinterpret_cast<const float4*>(cs + (static_cast<int64_t>(pos) * half + i) * 2);
    // c = (cos_i, sin_i, cos_{i+1}, sin_{i+1})
    const float sn0 = inverse ? -c.y : c.y;
    const float sn1 = inverse ? -c.w : c.w;
    const float a0 = a.x * c.x - b.x * sn0, b0 = b.x * c.x + a.x * sn0;
    const float a1 = a.y * c.z - b.y * sn1, b1 = b.y * c.z + a.y * sn1;
    *reinterpret_cast<__nv_bfloat162*>(base + i) = __floats2bfloat162_rn(a0, a1);
    *reinterpret_cast<__nv_bfloat162*>(base + half + i) = __floats2bfloat162_rn(b0, b1);
  }
}

// ------------------------------------------------------------------ SwiGLU
__device__ __forceinline__ float silu_f(float g) { return g / (1.f + expf(-g)); }

// Each thread handles 8 consecutive columns (16-byte vectors).
__global__ void swiglu_fwd_kernel(const bf16* __restrict__ gu, bf16* __restrict__ act, int T, int f) {
  const int per_row = f >> 3;
  const int64_t total = static_cast<int64_t>(T) * per_row;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = idx / per_row;
    const int c = static_cast<int>(idx % per_row) * 8;
    const bf16* g = gu + t * 2 * f + c;
    const bf16* u = g + f;
    uint4 gv = *reinterpret_cast<const uint4*>(g);
    uint4 uv = *reinterpret_cast<const uint4*>(u);
    const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gv);
    const __nv_bfloat162* u2 = reinterpret_cast<const __nv_bfloat162*>(&uv);
    uint4 ov;
    __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&ov);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 gf = __bfloat1622float2(g2[j]);
      const float2 uf = __bfloat1622float2(u2[j]);
      o2[j] = __floats2bfloat162_rn(silu_f(gf.x) * uf.x, silu_f(gf.y) * uf.y);
    }
    *reinterpret_cast<uint4*>(act + t * f + c) = ov;
  }
}

__global__ void swiglu_bwd_kernel(const bf16* __restrict__ gu, const bf16* __restrict__ dact, bf16* __restrict__ dgu,
                                  int T, int f) {
  const int per_row = f >> 3;
  const int64_t total = static_cast<int64_t>(T) * per_row;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = idx / per_row;
    const int c = static_cast<int>(idx % per_row) * 8;
    const uint4 gv = *reinterpret_cast<const uint4*>(gu + t * 2 * f + c);
    const uint4 uv = *reinterpret_cast<const uint4*>(gu + t * 2 * f + f + c);
    const uint4 dv = *reinterpret_cast<const uint4*>(dact + t * f + c);
    const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gv);
    const __nv_bfloat162* u2 = reinterpret_cast<const __nv_bfloat162*>(&uv);
    const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&dv);
    uint4 dgv, duv;
    __nv_bfloat162* dg2 = reinterpret_cast<__nv_bfloat162*>(&dgv);
    __nv_bfloat162* du2 = reinterpret_cast<__nv_bfloat162*>(&duv);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 g = __bfloat1622float2(g2[j]);
      const float2 u = __bfloat1622float2(u2[j]);
      const float2 d = __bfloat1622float2(d2[j]);
      const float s0 = 1.f / (1.f + expf(-g.x)), s1 = 1.f / (1.f + expf(-g.y));
      const float dg0 = d.x * u.x * s0 * (1.f + g.x * (1.f - s0));
      const float dg1 = d.y * u.y * s1 * (1.f + g.y * (1.f - s1));
      dg2[j] = __floats2bfloat162_rn(dg0, dg1);
      du2[j] = __floats2bfloat162_rn(d.x * g.x * s0, d.y * g.y * s1);
    }
    *reinterpret_cast<uint4*>(dgu + t * 2 * f + c) = dgv;
    *reinterpret_cast<uint4*>(dgu + t * 2 * f + f + c) = duv;
  }
}

// ------------------------------------------------------------------ embedding
__global__ void embed_fwd_kernel(const int32_t* __restrict__ tok, const bf16* __restrict__ E, float* __restrict__ x,
                                 int h) {
  const int t = blockIdx.x;
  const bf16* er = E + static_cast<int64_t>(tok[t]) * h;
  float4* xr = reinterpret_cast<float4*>(x + static_cast<int64_t>(t) * h);
  for (int i = threadIdx.x; i < (h >> 2); i += blockDim.x) xr[i] = load_bf16x4(er + 4 * i);
}

// dE[v] = sum of the dx rows at positions order[offsets[v] .. offsets[v+1]), visited in ascending
// order (one block per row; zero for a token id absent from the batch).
__device__ __forceinline__ void embed_row_grad(const int32_t* __restrict__ order, const int32_t* __restrict__ offsets,
                                               const float* __restrict__ dx, bf16* __restrict__ dE, int v, int h) {
  const int p0 = offsets[v], p1 = offsets[v + 1];
  bf16* out = dE + static_cast<int64_t>(v) * h;
  for (int i = threadIdx.x; i < (h >> 2); i += blockDim.x) {
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int p = p0; p < p1; ++p) {
      const float4 d = reinterpret_cast<const float4*>(dx + static_cast<int64_t>(order[p]) * h)[i];
      s.x += d.x;
      s.y += d.y;
      s.z += d.z;
      s.w += d.w;
    }
    store_bf16x4(out + 4 * i, s);
  }
}

// Every vocabulary row.
__global__ void embed_bwd_kernel(const int32_t* __restrict__ order, const int32_t* __restrict__ offsets,
                                 const float* __restrict__ dx, bf16* __restrict__ dE, int h) {
  embed_row_grad(order, offsets, dx, dE, blockIdx.x, h);
}

// Only the listed rows (same arithmetic, so the same bits, as embed_bwd_kernel for those rows).
__global__ void embed_bwd_rows_kernel(const int32_t* __restrict__ order, const int32_t* __restrict__ offsets,
                                      const int32_t* __restrict__ rows, const float* __restrict__ dx,
                                      bf16* __restrict__ dE, int h) {
  embed_row_grad(order, offsets, dx, dE, rows[blockIdx.x], h);
}

// ------------------------------------------------------------------ cross-entropy
__global__ void cross_entropy_kernel(const float* __restrict__ logits, const int32_t* __restrict__ labels,
                                     bf16* __restrict__ dlogits, float* __restrict__ row_loss, int V, float inv_T) {
  __shared__ float red_m[32], red_s[32];
  const int t = blockIdx.x;
  const float4* z = reinterpret_cast<const float4*>(logits + static_cast<int64_t>(t) * V);
  const int nv = V >> 2;
  // pass 1: running max and sum of exp(z - max) per thread, then merged over the block
  float m = -INFINITY, s = 0.f;
  for (int i = threadIdx.x; i < nv; i += blockDim.x) {
    const float4 q = z[i];
    const float mq = fmaxf(fmaxf(q.x, q.y), fmaxf(q.z, q.w));
    if (mq > m) {
      s *= expf(m - mq);
      m = mq;
    }
    s += expf(q.x - m) + expf(q.y - m) + expf(q.z - m) + expf(q.w - m);
  }
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float mo = __shfl_xor_sync(0xffffffffu, m, o);
    const float so = __shfl_xor_sync(0xffffffffu, s, o);
    const float mn = fmaxf(m, mo);
    s = (m == -INFINITY ? 0.f : s * expf(m - mn)) + (mo == -INFINITY ? 0.f : so * expf(mo - mn));
    m = mn;
  }
  if (lane == 0) {
    red_m[w] = m;
    red_s[w] = s;
  }
  __syncthreads();
  float M = -INFINITY;
  for (int i = 0; i < nw; ++i) M = fmaxf(M, red_m[i]);
  float S = 0.f;
  for (int i = 0; i < nw; ++i) S += red_s[i] * expf(red_m[i] - M);
  const float lse = M + logf(S);
  const int label = labels[t];
  if (threadIdx.x == 0) row_loss[t] = lse - logits[static_cast<int64_t>(t) * V + label];
  // pass 2: dlogits = (softmax - onehot) / T
  bf16* d = dlogits + static_cast<int64_t>(t) * V;
  for (int i = threadIdx.x; i < nv; i += blockDim.x) {
    const float4 q = z[i];
    float4 p = make_float4(expf(q.x - lse), expf(q.y - lse), expf(q.z - lse), expf(q.w - lse));
    const int c = 4 * i;
    if (label == c) p.x -= 1.f;
    if (label == c + 1) p.y -= 1.f;
    if (label == c + 2) p.z -= 1.f;
    if (label == c + 3) p.w -= 1.f;
    store_bf16x4(d + c, make_float4(p.x * inv_T, p.y * inv_T, p.z * inv_T, p.w * inv_T));
  }
}

// out = mean(v[0..n)) with a double accumulator, one block, fixed order.
__global__ void mean_reduce_kernel(const float* __restrict__ v, int n, float* __restrict__ out) {
  __shared__ double red[1024];
  double s = 0.0;
  for (int i = threadIdx.x; i < n; i += blockDim.x) s += static_cast<double>(v[i]);
  red[threadIdx.x] = s;
  __syncthreads();
  for (int w = blockDim.x >> 1; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) *out = static_cast<float>(red[0] / n);
}

__global__ void cast_kernel(const float* __restrict__ x, bf16* __restrict__ y, int64_t n4) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    store_bf16x4(y + 4 * i, reinterpret_cast<const float4*>(x)[i]);
}

int grid_for(int64_t work, int threads) {
  int64_t g = (work + threads - 1) / threads;
  const int64_t cap = 152 * 16;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return static_cast<int>(g);
}

}  // namespace

cudaError_t rmsnorm_fwd(const float* x, const bf16* gamma, bf16* y, float* rstd, int T, int h, float eps,
                        cudaStream_t s) {
  const int th = norm_threads(h);
  if (h % 8 || h / 4 > th * kMaxVec) return cudaErrorInvalidValue;
  // 16-byte loads of x, 8-byte accesses of gamma and y
  if ((reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(gamma) & 7) ||
      (reinterpret_cast<uintptr_t>(y) & 7))
    return cudaErrorInvalidValue;
  rmsnorm_fwd_kernel<<<T, th, 0, s>>>(x, gamma, y, rstd, h, eps);
  return cudaGetLastError();
}

int rmsnorm_bwd_parts(int T) { return T < 304 ? T : 304; }

bool rmsnorm_bwd_aligned(const float* dy, const float* x, const bf16* gamma, const float* dres, const float* dx,
                         const bf16* dx_bf16, const float* partial) {
  auto al = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; };
  return al(dy, 16) && al(x, 16) && al(dres, 16) && al(dx, 16) && al(partial, 16) && al(gamma, 8) &&
         al(dx_bf16, 8);
}

cudaError_t rmsnorm_bwd(const float* dy, const float* x, const bf16* gamma, const float* rstd, const float* dres,
                        float* dx, bf16* dx_bf16, float* partial, bf16* dgamma, int T, int h, cudaStream_t s) {
  // threads: a multiple of 32 dividing h/4 with at most 8 float4 per thread
  const int nv = h / 4;
  int th = 0;
  for (int t = 256; t >= 32; t -= 32)
    if (nv % t == 0 && nv / t <= 8) {
      th = t;
      break;
    }
  if (h % 8 || th == 0) return cudaErrorInvalidValue;
  // 16-byte vector accesses on the fp32 rows and the scratch, 8-byte ones on the bf16 gain and copy
  if (!rmsnorm_bwd_aligned(dy, x, gamma, dres, dx, dx_bf16, partial)) return cudaErrorInvalidValue;
  const int vpt = nv / th;
  const int parts = rmsnorm_bwd_parts(T);
  const int rpp = (T + parts - 1) / parts;
  const int used = (T + rpp - 1) / rpp;
  // ring stages of dy and x rows: up to 4, within ~110 KB so two CTAs share an SM
  const size_t stage_bytes = static_cast<size_t>(h) * 8;
  const int stages = static_cast<int>(std::max<size_t>(1, std::min<size_t>(4, (110u << 10) / stage_bytes)));
  const size_t smem = stages * stage_bytes;
  switch (vpt) {
#define MT_RMSBWD(V)                                                                                          \
  case V: {                                                                                                   \
    static bool attr = false;                                                                                 \
    if (!attr) {                                                                                              \
      cudaFuncSetAttribute(rmsnorm_bwd_async_kernel<V>, cudaFuncAttributeMaxDynamicSharedMemorySize, 112 << 10); \
      attr = true;                                                                                            \
    }                                                                                                         \
    rmsnorm_bwd_async_kernel<V><<<used, th, smem, s>>>(dy, x, gamma, rstd, dres, dx, dx_bf16, partial, T, h, rpp, \
                                                       stages);                                               \
    break;                                                                                                    \
  }
    MT_RMSBWD(1)
    MT_RMSBWD(2)
    MT_RMSBWD(3)
    MT_RMSBWD(4)
    MT_RMSBWD(5)
    MT_RMSBWD(6)
    MT_RMSBWD(7)
    MT_RMSBWD(8)
#undef MT_RMSBWD
    default:
      return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  reduce_parts_kernel<<<(h + 31) / 32, 32 * kReduceGroups, 0, s>>>(partial, dgamma, used, h);
  return cudaGetLastError();
}

cudaError_t rope(bf16* qkv, int64_t ld, int T, int seq, int n_heads, int n_kv_heads, int hd, const float* cs,
                 bool inverse, cudaStream_t s) {
  if (hd % 4 || ld % 2) return cudaErrorInvalidValue;
  const int heads = n_heads + n_kv_heads;  // q heads then k heads are contiguous columns
  const int64_t work = static_cast<int64_t>(T) * heads * (hd / 4);
  rope_kernel<<<grid_for(work, 256), 256, 0, s>>>(qkv, ld, T, seq, heads, hd, cs, inverse);
  return cudaGetLastError();
}

cudaError_t swiglu_fwd(const bf16* gu, bf16* act, int T, int f, cudaStream_t s) {
  if (f % 8) return cudaErrorInvalidValue;
  swiglu_fwd_kernel<<<grid_for(static_cast<int64_t>(T) * (f / 8), 256), 256, 0, s>>>(gu, act, T, f);
  return cudaGetLastError();
}

cudaError_t swiglu_bwd(const bf16* gu, const bf16* dact, bf16* dgu, int T, int f, cudaStream_t s) {
  if (f % 8) return cudaErrorInvalidValue;
  swiglu_bwd_kernel<<<grid_for(static_cast<int64_t>(T) * (f / 8), 256), 256, 0, s>>>(gu, dact, dgu, T, f);
  return cudaGetLastError();
}

cudaError_t embed_fwd(const int32_t* tok, const bf16* E, float* x, int T, int h, cudaStream_t s) {
  if (h % 4) return cudaErrorInvalidValue;
  embed_fwd_kernel<<<T, 128, 0, s>>>(tok, E, x, h);
  return cudaGetLastError();
}

cudaError_t embed_bwd(const int32_t* order, const int32_t* offsets, const float* dx, bf16* dE, int V, int h,
                      cudaStream_t s) {
  if (h % 4) return cudaErrorInvalidValue;
  embed_bwd_kernel<<<V, 128, 0, s>>>(order, offsets, dx, dE, h);
  return cudaGetLastError();
}

cudaError_t embed_bwd_rows(const int32_t* order, const int32_t* offsets, const int32_t* rows, int n_rows,
                           const float* dx, bf16* dE, int h, cudaStream_t s) {
  if (h % 4 || n_rows < 0) return cudaErrorInvalidValue;
  if (n_rows == 0) return cudaSuccess;
  embed_bwd_rows_kernel<<<n_rows, 128, 0, s>>>(order, offsets, rows, dx, dE, h);
  return cudaGetLastError();
}

cudaError_t cross_entropy(const float* logits, const int32_t* labels, bf16* dlogits, float* row_loss, int T, int V,
                          cudaStream_t s, int mean_over) {
  if (V % 4) return cudaErrorInvalidValue;
  const int n = mean_over > 0 ? mean_over : T;
  cross_entropy_kernel<<<T, 256, 0, s>>>(logits, labels, dlogits, row_loss, V, 1.f / static_cast<float>(n));
  return cudaGetLastError();
}

cudaError_t mean_reduce(const float* v, int n, float* out, cudaStream_t s) {
  mean_reduce_kernel<<<1, 1024, 0, s>>>(v, n, out);
  return cudaGetLastError();
}

cudaError_t cast_f32_bf16(const float* x, bf16* y, int64_t n, cudaStream_t s) {
  if (n % 4) return cudaErrorInvalidValue;
  cast_kernel<<<grid_for(n / 4, 256), 256, 0, s>>>(x, y, n / 4);
  return cudaGetLastError();
}

}  // namespace mt
