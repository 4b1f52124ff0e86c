// Host-side Adam over the packed arena. The chestersoft digest (Methodik,
// "Layer-Contiguous Tiling") runs the optimizer step on the CPU with AVX-512; on a
// Grace host (aarch64) the same loop is vectorised by the compiler for NEON and spread
// over the cores with OpenMP. Per element, in fp32:
//   g = G (bf16 -> f32); m = b1 m + (1 - b1) g; v = b2 v + (1 - b2) g^2
//   w = W - lr * (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps), stored as bf16 (nearest even)
#include <cmath>
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

// One tensor's update: n elements of W, G (bf16) and M, V (fp32).
static void adam_tensor(uint16_t* __restrict__ w, const uint16_t* __restrict__ g, float* __restrict__ m,
                        float* __restrict__ v, int64_t n, float lr, float b1, float b2, float ob1, float ob2,
                        float eps, float bc1, float bc2) {
#pragma omp parallel for schedule(static)
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

// Adam on the tensors of one block.
void adam_block(const Layout& L, int block, uint8_t* arena, const mt_adam_cfg& hp) {
  const double t = static_cast<double>(hp.step);
  const float bc1 = static_cast<float>(1.0 - std::pow(hp.beta1, t));
  const float bc2 = static_cast<float>(1.0 - std::pow(hp.beta2, t));
  const auto& blk = L.blocks[block];
  for (size_t k = 0; k < blk.shapes.size(); ++k) {
    const int64_t n = blk.shapes[k].numel();
    adam_tensor(reinterpret_cast<uint16_t*>(arena + blk.tensor_offset[MT_SEC_W][k]),
                reinterpret_cast<const uint16_t*>(arena + blk.tensor_offset[MT_SEC_G][k]),
                reinterpret_cast<float*>(arena + blk.tensor_offset[MT_SEC_M][k]),
                reinterpret_cast<float*>(arena + blk.tensor_offset[MT_SEC_V][k]), n, static_cast<float>(hp.lr),
                static_cast<float>(hp.beta1), static_cast<float>(hp.beta2), static_cast<float>(1.0 - hp.beta1),
                static_cast<float>(1.0 - hp.beta2), static_cast<float>(hp.eps), bc1, bc2);
  }
}

void adam_arena(const Layout& L, uint8_t* arena, const mt_adam_cfg& hp) {
  const double t = static_cast<double>(hp.step);
  const float bc1 = static_cast<float>(1.0 - std::pow(hp.beta1, t));
  const float bc2 = static_cast<float>(1.0 - std::pow(hp.beta2, t));
  for (const auto& blk : L.blocks) {
    for (size_t k = 0; k < blk.shapes.size(); ++k) {
      const int64_t n = blk.shapes[k].numel();
      adam_tensor(reinterpret_cast<uint16_t*>(arena + blk.tensor_offset[MT_SEC_W][k]),
                  reinterpret_cast<const uint16_t*>(arena + blk.tensor_offset[MT_SEC_G][k]),
                  reinterpret_cast<float*>(arena + blk.tensor_offset[MT_SEC_M][k]),
                  reinterpret_cast<float*>(arena + blk.tensor_offset[MT_SEC_V][k]), n, static_cast<float>(hp.lr),
                  static_cast<float>(hp.beta1), static_cast<float>(hp.beta2), static_cast<float>(1.0 - hp.beta1),
                  static_cast<float>(1.0 - hp.beta2), static_cast<float>(hp.eps), bc1, bc2);
    }
  }
}

bool adam_cfg_ok(const mt_adam_cfg& hp) {
  return hp.step >= 1 && hp.lr >= 0.0 && hp.beta1 >= 0.0 && hp.beta1 < 1.0 && hp.beta2 >= 0.0 && hp.beta2 < 1.0 &&
         hp.eps > 0.0;
}

}  // namespace mt
