// Host-arena layout arithmetic and its C ABI (mt_arena_bytes, mt_tensor_offset, ...).
#include "layout.h"

#include <algorithm>
#include <cstring>

namespace mt {

static uint64_t round_up(uint64_t n) { return (n + kAlign - 1) / kAlign * kAlign; }

bool validate_cfg(const mt_model_cfg& c, std::string* why) {
  auto fail = [&](const char* m) {
    if (why) *why = m;
    return false;
  };
  if (c.n_layers < 1) return fail("n_layers must be >= 1");
  if (c.hidden < 64 || c.hidden % 64) return fail("hidden must be a positive multiple of 64");
  if (c.n_heads < 1 || c.hidden % c.n_heads) return fail("n_heads must divide hidden");
  const int hd = c.hidden / c.n_heads;
  if (hd != 64 && hd != 128) return fail("head_dim = hidden / n_heads must be 64 or 128");
  if (c.n_kv_heads < 1 || c.n_heads % c.n_kv_heads) return fail("n_kv_heads must divide n_heads");
  if (c.ffn < 8 || c.ffn % 8) return fail("ffn must be a positive multiple of 8");
  if (c.vocab < 8 || c.vocab % 8) return fail("vocab must be a positive multiple of 8");
  if (c.seq < 1 || c.batch < 1) return fail("seq and batch must be >= 1");
  if (static_cast<int64_t>(c.seq) * c.batch > (int64_t(1) << 30)) return fail("batch*seq too large");
  if (!(c.rms_eps > 0.f) || !(c.rope_theta > 0.f)) return fail("rms_eps and rope_theta must be > 0");
  return true;
}

std::vector<TensorShape> block_shapes(const mt_model_cfg& c, int block) {
  const int64_t h = c.hidden, f = c.ffn, V = c.vocab, hd = c.hidden / c.n_heads;
  const int64_t qd = c.n_heads * hd, kvd = c.n_kv_heads * hd;
  if (block == 0) return {{V, h}};
  if (block == c.n_layers + 1) return {{h, 1}, {V, h}};
  return {{h, 1}, {qd, h}, {kvd, h}, {kvd, h}, {h, qd}, {h, 1}, {f, h}, {f, h}, {h, f}};
}

Layout compute_layout(const mt_model_cfg& c) {
  Layout L;
  L.sections = (c.flags & MT_FLAG_FP32_MASTER) ? 5 : 4;
  uint64_t off = 0;
  const uint64_t esz[kMaxSections] = {2, 2, 4, 4, 4};
  for (int b = 0; b < c.n_layers + 2; ++b) {
    Layout::Block blk;
    blk.offset = off;
    blk.shapes = block_shapes(c, b);
    for (int s = 0; s < L.sections; ++s) {
      blk.sec_offset[s] = off;
      for (const auto& t : blk.shapes) {
        blk.tensor_offset[s].push_back(off);
        off = round_up(off + static_cast<uint64_t>(t.numel()) * esz[s]);
      }
      blk.sec_bytes[s] = off - blk.sec_offset[s];
    }
    blk.bytes = off - blk.offset;
    if (blk.sec_bytes[0] > L.max_wsec) L.max_wsec = blk.sec_bytes[0];
    L.blocks.push_back(std::move(blk));
  }
  L.total = off;
  return L;
}

}  // namespace mt

// ------------------------------------------------------------------ C ABI
namespace {
thread_local std::string g_err;
int fail(int code, const std::string& m) {
  g_err = m;
  return code;
}
}  // namespace

const char* mt_global_error() { return g_err.c_str(); }
void mt_set_global_error(const std::string& m) { g_err = m; }

extern "C" {

int mt_arena_layout(const mt_model_cfg* cfg, mt_layout* out) {
  std::string why;
  if (!cfg || !out) return fail(MT_EINVAL, "null argument");
  if (!mt::validate_cfg(*cfg, &why)) return fail(MT_EINVAL, why);
  if (out->capacity < 0 || (out->capacity > 0 && !out->blocks)) return fail(MT_EINVAL, "bad block array");
  static_assert(mt::kMaxSections == MT_MAX_SECTIONS, "section count");
  const auto L = mt::compute_layout(*cfg);
  out->total_bytes = L.total;
  out->max_w_section = L.max_wsec;
  out->n_blocks = static_cast<int32_t>(L.blocks.size());
  out->n_sections = L.sections;
  const int n = std::min<int>(out->capacity, out->n_blocks);
  for (int b = 0; b < n; ++b) {
    const auto& blk = L.blocks[b];
    mt_block_layout& o = out->blocks[b];
    std::memset(&o, 0, sizeof(o));
    o.offset = blk.offset;
    o.bytes = blk.bytes;
    o.n_tensors = static_cast<int32_t>(blk.shapes.size());
    o.n_sections = L.sections;
    for (int s = 0; s < L.sections; ++s) {
      o.section_offset[s] = blk.sec_offset[s];
      o.section_bytes[s] = blk.sec_bytes[s];
      for (int t = 0; t < o.n_tensors; ++t) o.tensor_offset[s][t] = blk.tensor_offset[s][t];
    }
    for (int t = 0; t < o.n_tensors; ++t) {
      o.rows[t] = blk.shapes[t].rows;
      o.cols[t] = blk.shapes[t].cols;
    }
  }
  return MT_OK;
}

int mt_arena_bytes(const mt_model_cfg* cfg, uint64_t* bytes) {
  std::string why;
  if (!cfg || !bytes) return fail(MT_EINVAL, "null argument");
  if (!mt::validate_cfg(*cfg, &why)) return fail(MT_EINVAL, why);
  *bytes = mt::compute_layout(*cfg).total;
  return MT_OK;
}

int mt_block_count(const mt_model_cfg* cfg, int32_t* n_blocks) {
  std::string why;
  if (!cfg || !n_blocks) return fail(MT_EINVAL, "null argument");
  if (!mt::validate_cfg(*cfg, &why)) return fail(MT_EINVAL, why);
  *n_blocks = cfg->n_layers + 2;
  return MT_OK;
}

int mt_tensor_count(const mt_model_cfg* cfg, int32_t block, int32_t* n_tensors) {
  std::string why;
  if (!cfg || !n_tensors) return fail(MT_EINVAL, "null argument");
  if (!mt::validate_cfg(*cfg, &why)) return fail(MT_EINVAL, why);
  if (block < 0 || block > cfg->n_layers + 1) return fail(MT_EINVAL, "block out of range");
  *n_tensors = static_cast<int32_t>(mt::block_shapes(*cfg, block).size());
  return MT_OK;
}

int mt_block_offset(const mt_model_cfg* cfg, int32_t block, uint64_t* offset, uint64_t* bytes) {
  std::string why;
  if (!cfg || !offset || !bytes) return fail(MT_EINVAL, "null argument");
  if (!mt::validate_cfg(*cfg, &why)) return fail(MT_EINVAL, why);
  if (block < 0 || block > cfg->n_layers + 1) return fail(MT_EINVAL, "block out of range");
  const auto L = mt::compute_layout(*cfg);
  *offset = L.blocks[block].offset;
  *bytes = L.blocks[block].bytes;
  return MT_OK;
}

int mt_tensor_offset(const mt_model_cfg* cfg, int32_t block, int32_t section, int32_t tensor, uint64_t* offset,
                     int64_t* rows, int64_t* cols, int32_t* elem_bytes) {
  std::string why;
  if (!cfg || !offset) return fail(MT_EINVAL, "null argument");
  if (!mt::validate_cfg(*cfg, &why)) return fail(MT_EINVAL, why);
  if (block < 0 || block > cfg->n_layers + 1) return fail(MT_EINVAL, "block out of range");
  const auto L = mt::compute_layout(*cfg);
  if (section < 0 || section >= L.sections) return fail(MT_EINVAL, "section out of range");
  const auto& blk = L.blocks[block];
  if (tensor < 0 || tensor >= static_cast<int32_t>(blk.shapes.size())) return fail(MT_EINVAL, "tensor out of range");
  *offset = blk.tensor_offset[section][tensor];
  if (rows) *rows = blk.shapes[tensor].rows;
  if (cols) *cols = blk.shapes[tensor].cols;
  if (elem_bytes) *elem_bytes = section < 2 ? 2 : 4;
  return MT_OK;
}

}  // extern "C"
