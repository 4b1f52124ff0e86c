// Packed layer-block layout of the host arena ("Layer-Contiguous Tiling", chestersoft
// digest, Methodik): per block, sections W (bf16), G (bf16), M (fp32), V (fp32), and with
// MT_FLAG_FP32_MASTER a fifth, P (fp32 master weights); every section and every tensor
// starts on a 4096-byte boundary.
#pragma once
#include <array>
#include <cstdint>
#include <string>
#include <vector>

#include "mt.h"

namespace mt {

constexpr uint64_t kAlign = 4096;
constexpr int kMaxSections = 5;

struct TensorShape {
  int64_t rows, cols;  // cols == 1 for a gain vector
  int64_t numel() const { return rows * cols; }
};

struct Layout {
  uint64_t total = 0;
  struct Block {
    uint64_t offset = 0, bytes = 0;
    std::vector<TensorShape> shapes;
    std::array<uint64_t, kMaxSections> sec_offset{}, sec_bytes{};
    std::array<std::vector<uint64_t>, kMaxSections> tensor_offset;  // absolute offsets per section
  };
  std::vector<Block> blocks;
  uint64_t max_wsec = 0;  // largest W (= G) section
  int sections = 4;       // 5 with the fp32 master section
};

// Checks the configuration; on failure returns false with a reason.
bool validate_cfg(const mt_model_cfg& c, std::string* why);
std::vector<TensorShape> block_shapes(const mt_model_cfg& c, int block);
Layout compute_layout(const mt_model_cfg& c);

}  // namespace mt
