// Host-side Adam over the packed arena. The chestersoft digest (Methodik,
// "Layer-Contiguous Tiling") runs the optimizer step on the CPU with AVX-512; on a
// Grace host (aarch64) the same loop is vectorised by the compiler for NEON and spread
// over the cores with OpenMP. Per element, in fp32:
//   g = G (bf16 -> f32); m = b1 m + (1 - b1) g; v = b2 v + (1 - b2) g^2
//   w = W - lr * (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps), stored as bf16 (nearest even)
// With an fp32 master copy P (MT_FLAG_FP32_MASTER) the update is applied to P in fp32 and W
// becomes bf16(P): increments smaller than half a bf16 step then accumulate in P.
#include <omp.h>

#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <string>

#include "layout.h"

namespace mt {

static inline float bf16_to_f32(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}
// Round to nearest even; a NaN stays a (quiet) NaN. Branch-free so the loop vectorises.
static inline uint16_t f32_to_bf16(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  const uint32_t rounded = (u + 0x7fffu + ((u >> 16) & 1u)) >> 16;
  const uint32_t quiet_nan = (u >> 16) | 0x40u;
  const bool is_nan = (u & 0x7fffffffu) > 0x7f800000u;
  return static_cast<uint16_t>(is_nan ? quiet_nan : rounded);
}

// One tensor's update: n elements of W, G (bf16) and M, V (fp32). Called inside a parallel
// region: the threads share the elements (static schedule) and move on to the block's next tensor
// without waiting for one another.
static void adam_tensor(uint16_t* __restrict__ w, const uint16_t* __restrict__ g, float* __restrict__ m,
                        float* __restrict__ v, int64_t n, float lr, float b1, float b2, float ob1, float ob2,
                        float eps, float bc1, float bc2) {
#pragma omp for schedule(static) nowait
  for (int64_t i = 0; i < n; ++i) {
    const float gi = bf16_to_f32(g[i]);
    const float mi = b1 * m[i] + ob1 * gi;
    const float vi = b2 * v[i] + ob2 * gi * gi;
    m[i] = mi;
    v[i] = vi;
    const float mhat = mi / bc1;
    const float vhat = vi / bc2;
    w[i] = f32_to_bf16(bf16_to_f32(w[i]) - lr * mhat / (std::sqrt(vhat) + eps));
  }
}

// The same update with an fp32 master copy p: p -= lr * mhat / (sqrt(vhat) + eps); W = bf16(p).
static void adam_tensor_master(uint16_t* __restrict__ w, float* __restrict__ p, const uint16_t* __restrict__ g,
                               float* __restrict__ m, float* __restrict__ v, int64_t n, float lr, float b1, float b2,
                               float ob1, float ob2, float eps, float bc1, float bc2) {
#pragma omp for schedule(static) nowait
  for (int64_t i = 0; i < n; ++i) {
    const float gi = bf16_to_f32(g[i]);
    const float mi = b1 * m[i] + ob1 * gi;
    const float vi = b2 * v[i] + ob2 * gi * gi;
    m[i] = mi;
    v[i] = vi;
    const float mhat = mi / bc1;
    const float vhat = vi / bc2;
    const float pi = p[i] - lr * mhat / (std::sqrt(vhat) + eps);
    p[i] = pi;
    w[i] = f32_to_bf16(pi);
  }
}

// Adam on the tensors of one block.
void adam_block(const Layout& L, int block, uint8_t* arena, const mt_adam_cfg& hp) {
  const double t = static_cast<double>(hp.step);
  const float bc1 = static_cast<float>(1.0 - std::pow(hp.beta1, t));
  const float bc2 = static_cast<float>(1.0 - std::pow(hp.beta2, t));
  const float lr = static_cast<float>(hp.lr), b1 = static_cast<float>(hp.beta1), b2 = static_cast<float>(hp.beta2);
  const float ob1 = static_cast<float>(1.0 - hp.beta1), ob2 = static_cast<float>(1.0 - hp.beta2);
  const float eps = static_cast<float>(hp.eps);
  const auto& blk = L.blocks[block];
  // one parallel region per block (not per tensor: a decoder layer's two gain vectors are too
  // small to pay for opening one each)
#pragma omp parallel
  for (size_t k = 0; k < blk.shapes.size(); ++k) {
    const int64_t n = blk.shapes[k].numel();
    auto* w = reinterpret_cast<uint16_t*>(arena + blk.tensor_offset[MT_SEC_W][k]);
    const auto* g = reinterpret_cast<const uint16_t*>(arena + blk.tensor_offset[MT_SEC_G][k]);
    auto* m = reinterpret_cast<float*>(arena + blk.tensor_offset[MT_SEC_M][k]);
    auto* v = reinterpret_cast<float*>(arena + blk.tensor_offset[MT_SEC_V][k]);
    if (L.sections > MT_SEC_P)
      adam_tensor_master(w, reinterpret_cast<float*>(arena + blk.tensor_offset[MT_SEC_P][k]), g, m, v, n, lr, b1, b2,
                         ob1, ob2, eps, bc1, bc2);
    else
      adam_tensor(w, g, m, v, n, lr, b1, b2, ob1, ob2, eps, bc1, bc2);
  }
}

void adam_arena(const Layout& L, uint8_t* arena, const mt_adam_cfg& hp) {
  for (size_t b = 0; b < L.blocks.size(); ++b) adam_block(L, static_cast<int>(b), arena, hp);
}

// P = W (bf16 -> fp32, exact) for every tensor of every block.
void master_init(const Layout& L, uint8_t* arena) {
  for (const auto& blk : L.blocks) {
    for (size_t k = 0; k < blk.shapes.size(); ++k) {
      const int64_t n = blk.shapes[k].numel();
      const auto* w = reinterpret_cast<const uint16_t*>(arena + blk.tensor_offset[MT_SEC_W][k]);
      auto* p = reinterpret_cast<float*>(arena + blk.tensor_offset[MT_SEC_P][k]);
#pragma omp parallel for schedule(static)
      for (int64_t i = 0; i < n; ++i) p[i] = bf16_to_f32(w[i]);
    }
  }
}

// STREAM-style triad a = b + s c over three fp32 arrays of `bytes` / 12 elements each (first
// touched by the threads that use them), best of `reps` passes: the host memory bandwidth the
// host Adam (22 bytes moved per parameter) is measured against.
double host_triad_gbs(uint64_t bytes, int reps) {
  const int64_t n = static_cast<int64_t>(bytes / 12);
  if (n <= 0 || reps <= 0) return 0.0;
  float* a = static_cast<float*>(std::malloc(sizeof(float) * n));
  float* b = static_cast<float*>(std::malloc(sizeof(float) * n));
  float* c = static_cast<float*>(std::malloc(sizeof(float) * n));
  if (!a || !b || !c) {
    std::free(a);
    std::free(b);
    std::free(c);
    return 0.0;
  }
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    a[i] = 0.f;
    b[i] = 1.f;
    c[i] = 2.f;
  }
  double best = 0.0;
  for (int r = 0; r < reps; ++r) {
    const auto t0 = std::chrono::steady_clock::now();
    const float sc = 0.5f + static_cast<float>(r);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) a[i] = b[i] + sc * c[i];
    const double s = std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
    if (s > 0) best = std::max(best, 12.0 * static_cast<double>(n) / s / 1e9);
  }
  volatile float sink = a[n / 2];
  (void)sink;
  std::free(a);
  std::free(b);
  std::free(c);
  return best;
}

int host_threads() { return omp_get_max_threads(); }

bool adam_cfg_ok(const mt_adam_cfg& hp) {
  return hp.step >= 1 && hp.lr >= 0.0 && hp.beta1 >= 0.0 && hp.beta1 < 1.0 && hp.beta2 >= 0.0 && hp.beta2 < 1.0 &&
         hp.eps > 0.0;
}

}  // namespace mt
