// The streaming engine: context, device buffers, the three-stream double-buffered
// schedule, and the training-step C ABI (mt_create / mt_bind_host_arena /
// mt_train_step / mt_adam_step / mt_get_stats / mt_destroy).
//
// Design ("MegaTrain", chatpaper abstract and chestersoft digest, Methodik):
//  * all parameters, gradients and Adam moments stay in the caller's host arena;
//  * the device holds two layer buffers (ping-pong) for W sections and two for G
//    sections; stream h2d prefetches block i+1's W section into the free buffer
//    (one DMA burst per block) while stream compute runs block i, and stream d2h
//    offloads each block's G section as soon as its backward finishes;
//  * the layer templates are stateless: each pass binds the weights by pointer into
//    whichever buffer currently holds them; no autograd graph or per-layer device
//    state outlives the pass except the layer-boundary activation checkpoints, from
//    which the backward pass recomputes the layer.
// Block uses in order: E (embedding gather), L0 .. L{n-1} (forward), H (head forward,
// loss, head backward), L{n-1} .. L0 (recompute + backward), then the embedding
// gradient (no weights needed). Resident mode uploads every W section first and keeps
// G on the device until the end; it runs the very same kernel sequence.
#include <algorithm>
#include <chrono>
#include <cstdio>
#include <cstdlib>
#include <cmath>
#include <cstring>
#include <string>
#include <thread>
#include <vector>

#include "kernels.h"
#include "layout.h"
#include "mt.h"

const char* mt_global_error();
void mt_set_global_error(const std::string& m);

namespace mt {
void adam_arena(const Layout& L, uint8_t* arena, const mt_adam_cfg& hp);
void master_init(const Layout& L, uint8_t* arena);
void adam_block(const Layout& L, int block, uint8_t* arena, const mt_adam_cfg& hp);
bool adam_cfg_ok(const mt_adam_cfg& hp);
double host_triad_gbs(uint64_t bytes, int reps);
int host_threads();
}  // namespace mt

using mt::bf16;

namespace {

constexpr double kStepWaitSeconds = 3600.0;  // bound on the host wait for one step
constexpr int kStreamH2D = 0, kStreamCompute = 1, kStreamD2H = 2;
constexpr double kMappedEmbedFloorGbs = 25.0;  // below this the embedding block is copied whole

uint64_t align256(uint64_t n) { return (n + 255) / 256 * 256; }

// The LM head and cross-entropy run over token chunks so that the fp32 logits of a long
// sequence are never held whole: a chunk's logits are at most kHeadLogitsBudget bytes
// (every configuration with T * V * 4 within the budget runs as one chunk).
constexpr uint64_t kHeadLogitsBudget = 4ull << 30;

// Rows per head chunk: T split into the fewest equal chunks within the budget, rounded up to a
// multiple of 128 (the GEMM's row tile).
int head_chunk_rows(int T, int V) {
  const uint64_t full = static_cast<uint64_t>(T) * V * 4;
  if (full <= kHeadLogitsBudget) return T;
  const uint64_t chunks = (full + kHeadLogitsBudget - 1) / kHeadLogitsBudget;
  const uint64_t rows = (static_cast<uint64_t>(T) + chunks - 1) / chunks;
  return static_cast<int>((rows + 127) / 128 * 128);
}

// Device workspace plan: byte offsets of every buffer inside one allocation.
struct Plan {
  uint64_t total = 0;
  uint64_t wbuf[2], gbuf[2], res_w, res_g, res_bytes;
  uint64_t ckpt, n_ckpt_slots;
  uint64_t h1, a, bb, y, qkv, o, lse, delta, gu, act, rstd1, rstd2, rstdf;
  uint64_t logits, dlogits, dw_head, row_loss, loss, err;
  int head_rows;  // token rows per LM-head chunk
  uint64_t dgu, dqkv, d_o, db, dh, dh_bf16, dx[2], dx_bf16[2], partial;
  uint64_t rope_cs, tok, lab, order, offsets, erows;
  uint64_t gemm_ws;  // GEMM last-wave split: per-CTA partial slots and flags
};

Plan make_plan(const mt_model_cfg& c, const mt::Layout& L) {
  Plan p{};
  const uint64_t T = static_cast<uint64_t>(c.batch) * c.seq, h = c.hidden, f = c.ffn, V = c.vocab;
  const uint64_t hd = c.hidden / c.n_heads, nqkv = (c.n_heads + 2 * c.n_kv_heads) * hd, qd = c.n_heads * hd;
  uint64_t off = 0;
  auto take = [&](uint64_t bytes) {
    const uint64_t o = off;
    off = align256(off + bytes);
    return o;
  };
  const bool resident = c.flags & MT_FLAG_RESIDENT;
  if (resident) {
    uint64_t sum = 0;
    for (const auto& b : L.blocks) sum += b.sec_bytes[MT_SEC_W];
    p.res_bytes = sum;
    p.res_w = take(sum);
    p.res_g = take(sum);
    p.wbuf[0] = p.wbuf[1] = p.gbuf[0] = p.gbuf[1] = 0;
  } else {
    p.wbuf[0] = take(L.max_wsec);
    p.wbuf[1] = take(L.max_wsec);
    p.gbuf[0] = take(L.max_wsec);
    p.gbuf[1] = take(L.max_wsec);
  }
  p.n_ckpt_slots = (c.flags & MT_FLAG_OFFLOAD_CKPT) ? 2 : static_cast<uint64_t>(c.n_layers) + 1;
  p.ckpt = take(p.n_ckpt_slots * T * h * 4);
  p.h1 = take(T * h * 4);
  p.a = take(T * h * 2);
  p.bb = take(T * h * 2);
  p.y = take(T * h * 2);
  p.qkv = take(T * nqkv * 2);
  p.o = take(T * qd * 2);
  p.lse = take(T * c.n_heads * 4);
  p.delta = take(static_cast<uint64_t>(c.batch) * c.n_heads * ((c.seq + 127) / 128 * 128) * 8);  // (lse2, delta) pairs
  p.gu = take(T * 2 * f * 2);
  p.act = take(T * f * 2);
  p.rstd1 = take(T * 4);
  p.rstd2 = take(T * 4);
  p.rstdf = take(T * 4);
  p.head_rows = head_chunk_rows(static_cast<int>(T), c.vocab);
  p.logits = take(static_cast<uint64_t>(p.head_rows) * V * 4);
  p.dlogits = take(static_cast<uint64_t>(p.head_rows) * V * 2);
  // fp32 accumulator of the LM-head weight gradient over the chunks (used when there are several)
  p.dw_head = take(V * h * 4);
  p.row_loss = take(T * 4);
  p.loss = take(16);
  p.err = take(16);
  p.dgu = take(T * 2 * f * 2);
  p.dqkv = take(T * nqkv * 2);
  p.d_o = take(T * qd * 2);
  p.db = take(T * h * 4);
  p.dh = take(T * h * 4);
  p.dh_bf16 = take(T * h * 2);
  for (int i = 0; i < 2; ++i) {
    p.dx[i] = take(T * h * 4);
    p.dx_bf16[i] = take(T * h * 2);
  }
  p.partial = take(static_cast<uint64_t>(mt::rmsnorm_bwd_parts(static_cast<int>(T))) * h * 4);
  p.rope_cs = take(static_cast<uint64_t>(c.seq) * (hd / 2) * 2 * 4);
  p.tok = take(T * 4);
  p.lab = take(T * 4);
  p.order = take(T * 4);
  p.offsets = take((V + 1) * 4);
  p.erows = take(2 * T * 4);  // embedding rows whose gradient a step writes (this and the last batch's ids)
  p.gemm_ws = take(mt::gemm_workspace_bytes());
  p.total = off;
  return p;
}

struct LayerW {  // device pointers of one decoder layer's W (or G) section
  bf16 *attn_norm, *wqkv, *wo, *ffn_norm, *wgu, *wd;
};

struct TimedLaunch {
  int kind;
  double flops, bytes;
  cudaEvent_t a, b;
};

}  // namespace

struct mt_ctx {
  mt_model_cfg cfg{};
  mt::Layout lay;
  Plan plan;
  int T = 0, h = 0, nh = 0, nkv = 0, hd = 0, f = 0, V = 0, L = 0, qd = 0, nqkv = 0;
  int head_rows = 0;  // token rows per LM-head chunk (plan.head_rows unless set smaller)
  bool resident = false, offload = false, single = false, timing = false;

  uint8_t* ws = nullptr;
  bool own_ws = false;
  cudaStream_t st[3] = {nullptr, nullptr, nullptr};
  bool own_st[3] = {false, false, false};

  // host side
  uint8_t* arena = nullptr;
  uint64_t arena_bytes = 0;
  bool registered = false;
  float* host_ckpt = nullptr;  // pinned, n_layers slots (offload mode)
  int32_t* pin_io = nullptr;   // pinned staging: tokens | labels | order | offsets | embedding rows
  // pinned: [0] loss, [1] error flag (int) at the end of the step; [2] the loss as soon as the
  // head has run; then one int per block: the device error flag when that block's gradients
  // left for the arena (the overlapped Adam stops at the first nonzero one)
  float* pin_out = nullptr;
  int* pin_flags = nullptr;
  bool grads_valid = false;
  bool broken = false;  // a step's wait limit expired: work may still be in flight on the device
  // Sparse embedding block: when the arena is mapped into the device's address space (unified
  // addressing) and the schedule streams, the embedding gather reads the batch's rows of E
  // straight from the arena, and its backward writes only the gradient rows it changes (the
  // batch's token ids, and zeros over the last batch's) into the arena's G section, instead of
  // copying the whole vocabulary-sized W and G sections.
  uint8_t* arena_dev = nullptr;
  bool sparse_e = false;
  bool e_clean = false;                 // E's G section is zero outside e_prev
  std::vector<int32_t> e_prev, e_next;  // token ids of the last completed step / this step
  int n_erows = 0;

  // events
  cudaEvent_t wready[2], wfree[2], gready[2], gfree[2], ck_ready[2], ck_saved[2];
  // decoder-layer sections move in kParts pieces (see kPartFirst): wpart[buf][k] = piece k of the
  // weights in W buffer buf has arrived; gpart[buf][k] = piece k of the gradients in G buffer buf
  // is final
  cudaEvent_t wpart[2][4], gpart[2][4];
  cudaEvent_t ev_start, ev_fwd_end, ev_end, ev_d2h_done, ev_inputs;
  cudaEvent_t ev_emb[2] = {nullptr, nullptr};  // around the embedding gather from the mapped arena
  bool emb_timed = false;                      // the last step recorded them
  std::vector<cudaEvent_t> g_landed;  // per block: its G section has reached the host arena
  std::vector<cudaEvent_t> span_pool;  // per-step spans on each stream
  size_t span_used = 0;
  struct Span {
    int stream;
    cudaEvent_t a, b;
    uint64_t bytes;  // bytes the span's copies move (0 for compute)
  };
  std::vector<Span> spans;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> waits;  // compute-stream waits on copies
  std::vector<cudaEvent_t> kpool;
  size_t kused = 0;
  std::vector<TimedLaunch> klaunch;

  // armed captures of dL/dx_l (layer l, host destination), copied out during each step
  std::vector<std::pair<int, float*>> grad_capture;

  mt_stats stats{};
  mt_kernel_stats kstats[MT_KIND_COUNT]{};
  int64_t launches = 0;
  uint64_t h2d_bytes = 0, d2h_bytes = 0;
  std::string err;

  template <class T>
  T* dev(uint64_t off) const {
    return reinterpret_cast<T*>(ws + off);
  }
};

namespace {

int set_err(mt_ctx* c, int code, const std::string& m) {
  if (c) c->err = m;
  return code;
}

#define CK(call)                                                                                     \
  do {                                                                                               \
    cudaError_t e_ = (call);                                                                         \
    if (e_ != cudaSuccess)                                                                           \
      return set_err(c, e_ == cudaErrorMemoryAllocation ? MT_ENOMEM : MT_ECUDA,                      \
                     std::string(#call) + ": " + cudaGetErrorString(e_));                            \
  } while (0)

cudaEvent_t next_event(std::vector<cudaEvent_t>& pool, size_t& used) {
  if (used == pool.size()) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    pool.push_back(e);
  }
  return pool[used++];
}

// Record a span [a, b) on stream s around `body`.
template <class F>
int span(mt_ctx* c, int s, F&& body) {
  cudaEvent_t a = next_event(c->span_pool, c->span_used), b = next_event(c->span_pool, c->span_used);
  if (!a || !b) return set_err(c, MT_ECUDA, "event pool");
  CK(cudaEventRecord(a, c->st[s]));
  const uint64_t moved0 = c->h2d_bytes + c->d2h_bytes;
  int r = body();
  if (r != MT_OK) return r;
  CK(cudaEventRecord(b, c->st[s]));
  c->spans.push_back({s, a, b, s == kStreamCompute ? 0 : c->h2d_bytes + c->d2h_bytes - moved0});
  return MT_OK;
}

// The compute stream waits for a copy event. Two timing events around the wait measure how long
// the compute stream stood still for a transfer: their sum over a step is its exposed copy time.
int wait_copy(mt_ctx* c, cudaEvent_t ev) {
  cudaEvent_t a = next_event(c->span_pool, c->span_used), b = next_event(c->span_pool, c->span_used);
  if (!a || !b) return set_err(c, MT_ECUDA, "event pool");
  CK(cudaEventRecord(a, c->st[kStreamCompute]));
  CK(cudaStreamWaitEvent(c->st[kStreamCompute], ev, 0));
  CK(cudaEventRecord(b, c->st[kStreamCompute]));
  c->waits.push_back({a, b});
  return MT_OK;
}

// Launch wrapper on the compute stream: counts launches, optionally times them.
template <class F>
int launch(mt_ctx* c, int kind, double flops, double bytes, F&& fn) {
  cudaEvent_t a = nullptr, b = nullptr;
  if (c->timing) {
    a = next_event(c->kpool, c->kused);
    b = next_event(c->kpool, c->kused);
    if (!a || !b) return set_err(c, MT_ECUDA, "event pool");
    CK(cudaEventRecord(a, c->st[kStreamCompute]));
  }
  cudaError_t e = fn();
  if (e != cudaSuccess) return set_err(c, MT_ECUDA, std::string("kernel launch: ") + cudaGetErrorString(e));
  if (c->timing) {
    CK(cudaEventRecord(b, c->st[kStreamCompute]));
    c->klaunch.push_back({kind, flops, bytes, a, b});
  }
  return MT_OK;
}

int gemm_args(mt_ctx* c, const mt::GemmArgs& g) {
  // the SwiGLU forward's paired tile computes gate and up columns: 2 N columns of work
  const double n_eff = g.epi == mt::kEpiSwigluBf16 ? 2.0 * g.N : g.N;
  const double M = g.M, N = g.N, K = g.K;
  // algorithmic bytes: each operand read once, each output written once
  double bytes = 2.0 * M * K + 2.0 * n_eff * K;
  switch (g.epi) {
    case mt::kEpiStoreF32: bytes += 4.0 * M * N; break;
    case mt::kEpiAddF32: bytes += 8.0 * M * N; break;  // R in, C out (fp32)
    case mt::kEpiSwigluBf16: bytes += 2.0 * M * N + (g.C2 ? 4.0 * M * N : 0.0); break;
    case mt::kEpiSwigluBwdBf16: bytes += 8.0 * M * N; break;  // [g|u] in, [dg|du] out (bf16, 2N wide)
    default: bytes += 2.0 * M * N; break;
  }
  c->launches += 1;
  mt::GemmArgs gw = g;
  gw.ws = c->ws + c->plan.gemm_ws;  // every GEMM runs on the compute stream: they never overlap
  return launch(c, MT_KIND_GEMM, 2.0 * g.M * n_eff * static_cast<double>(g.K), bytes,
                [&] { return mt::gemm(gw, c->dev<int>(c->plan.err), c->st[kStreamCompute]); });
}

int gemm(mt_ctx* c, const bf16* A, int64_t lda, bool a_mn, const bf16* B, int64_t ldb, bool b_mn, void* C,
         int64_t ldc, int M, int N, int K, int epi, const float* R = nullptr, int64_t ldr = 0) {
  return gemm_args(c, mt::GemmArgs{A, lda, a_mn, B, ldb, b_mn, C, ldc, R, ldr, M, N, K, epi});
}

LayerW bind_layer(const mt_ctx* c, int block, uint8_t* sec_base, int sec) {
  const auto& blk = c->lay.blocks[block];
  auto p = [&](int t) { return reinterpret_cast<bf16*>(sec_base + (blk.tensor_offset[sec][t] - blk.sec_offset[sec])); };
  return LayerW{p(MT_T_ATTN_NORM), p(MT_T_WQ), p(MT_T_WO), p(MT_T_FFN_NORM), p(MT_T_WG), p(MT_T_WD)};
}

// ------------------------------------------------------------------ layer pieces
// A decoder layer's W and G sections move host<->device in four pieces, in tensor order, so the
// layer can start on the first weights while the rest still stream in, and its first finished
// gradients leave while it still computes the others:
//   piece 0: attn_norm, wq, wk, wv   piece 1: wo   piece 2: ffn_norm, wg, wu   piece 3: wd
constexpr int kParts = 4;
constexpr int kPartFirst[kParts + 1] = {MT_T_ATTN_NORM, MT_T_WO, MT_T_FFN_NORM, MT_T_WD, MT_T_WD + 1};

// Byte range [begin, end) of piece k within a block's section (offsets relative to the section).
void part_range(const mt::Layout::Block& blk, int sec, int k, uint64_t& begin, uint64_t& end) {
  const int t0 = kPartFirst[k], t1 = kPartFirst[k + 1] - 1;
  begin = blk.tensor_offset[sec][t0] - blk.sec_offset[sec];
  end = blk.tensor_offset[sec][t1] - blk.sec_offset[sec] + static_cast<uint64_t>(blk.shapes[t1].numel()) * 2;
}

// Piecewise movement of one decoder layer's sections (null: the whole-section path).
struct Pieces {
  int wbuf = -1;  // W buffer whose pieces the compute waits for (-1: none)
  int gbuf = -1;  // G buffer whose pieces leave as they are finished (-1: none)
  int block = 0;
};

// The compute stream waits until weight piece k has arrived.
int need_w(mt_ctx* c, const Pieces* pc, int k) {
  if (!pc || pc->wbuf < 0) return MT_OK;
  return wait_copy(c, c->wpart[pc->wbuf][k]);
}

// Mark block `block`'s gradients as landed in the arena, on stream s: first copy the device error
// flag as it stands (every kernel that produced these gradients has finished) into the block's
// pinned slot, so the overlapped host Adam can tell good gradients from those of a failed step.
int mark_landed(mt_ctx* c, int block, cudaStream_t s) {
  CK(cudaMemcpyAsync(c->pin_flags + block, c->dev<int>(c->plan.err), sizeof(int), cudaMemcpyDeviceToHost, s));
  CK(cudaEventRecord(c->g_landed[block], s));
  return MT_OK;
}

// Gradient piece k is final in the G buffer: copy it to the arena. The last piece (0) frees the
// buffer and marks the block's gradients as landed.
int grad_done(mt_ctx* c, const Pieces* pc, int k) {
  if (!pc || pc->gbuf < 0) return MT_OK;
  const int gb = pc->gbuf;
  const auto& blk = c->lay.blocks[pc->block];
  CK(cudaEventRecord(c->gpart[gb][k], c->st[kStreamCompute]));
  CK(cudaStreamWaitEvent(c->st[kStreamD2H], c->gpart[gb][k], 0));
  int r = span(c, kStreamD2H, [&]() -> int {
    uint64_t b0, b1;
    part_range(blk, MT_SEC_G, k, b0, b1);
    CK(cudaMemcpyAsync(c->arena + blk.sec_offset[MT_SEC_G] + b0, c->ws + c->plan.gbuf[gb] + b0, b1 - b0,
                       cudaMemcpyDeviceToHost, c->st[kStreamD2H]));
    c->d2h_bytes += b1 - b0;
    return MT_OK;
  });
  if (r) return r;
  if (k == 0) {
    CK(cudaEventRecord(c->gfree[gb], c->st[kStreamD2H]));
    return mark_landed(c, pc->block, c->st[kStreamD2H]);
  }
  return MT_OK;
}

// ------------------------------------------------------------------ layer template
// Forward of one decoder layer bound to weights w: x_out = layer(x_in). With
// recompute = true it stops before the down projection (backward needs act, not x_out).
int layer_forward(mt_ctx* c, const LayerW& w, const float* x_in, float* x_out, bool recompute,
                  const Pieces* pc = nullptr) {
  const Plan& p = c->plan;
  cudaStream_t s = c->st[kStreamCompute];
  const int T = c->T, h = c->h, f = c->f;
  const double Td = T;
  bf16* a = c->dev<bf16>(p.a);
  bf16* qkv = c->dev<bf16>(p.qkv);
  bf16* o = c->dev<bf16>(p.o);
  float* h1 = c->dev<float>(p.h1);
  bf16* bb = c->dev<bf16>(p.bb);
  bf16* gu = c->dev<bf16>(p.gu);
  bf16* act = c->dev<bf16>(p.act);
  int r;
  if ((r = need_w(c, pc, 0))) return r;  // attn_norm, wq, wk, wv
  c->launches += 1;
  r = launch(c, MT_KIND_POINTWISE, 0, Td * h * 6, [&] {
    return mt::rmsnorm_fwd(x_in, w.attn_norm, a, c->dev<float>(p.rstd1), T, h, c->cfg.rms_eps, s);
  });
  if (r) return r;
  {  // QKV projection, RoPE applied to q and k in the epilogue
    mt::GemmArgs g{a, h, false, w.wqkv, h, false, qkv, c->nqkv, nullptr, 0, T, c->nqkv, h, mt::kEpiRopeBf16};
    g.cs = c->dev<float>(p.rope_cs);
    g.rope_cols = (c->nh + c->nkv) * c->hd;
    g.hd = c->hd;
    g.seq = c->cfg.seq;
    if ((r = gemm_args(c, g))) return r;
  }
  c->launches += 1;
  const double attn_flops = 2.0 * c->cfg.batch * static_cast<double>(c->cfg.seq) * c->cfg.seq * c->nh * c->hd;
  r = launch(c, MT_KIND_ATTN_FWD, attn_flops, 0, [&] {
    return mt::attn_fwd(qkv, o, c->dev<float>(p.lse), c->cfg.batch, c->cfg.seq, c->nh, c->nkv, c->hd,
                        c->dev<int>(p.err), s);
  });
  if (r) return r;
  if ((r = need_w(c, pc, 1))) return r;  // wo
  if ((r = gemm(c, o, c->qd, false, w.wo, c->qd, false, h1, h, T, h, c->qd, mt::kEpiAddF32, x_in, h))) return r;
  if ((r = need_w(c, pc, 2))) return r;  // ffn_norm, wg, wu
  c->launches += 1;
  r = launch(c, MT_KIND_POINTWISE, 0, Td * h * 6, [&] {
    return mt::rmsnorm_fwd(h1, w.ffn_norm, bb, c->dev<float>(p.rstd2), T, h, c->cfg.rms_eps, s);
  });
  if (r) return r;
  {  // gate-up projection with SwiGLU in the epilogue; the recompute also keeps [g | u]
    mt::GemmArgs g{bb, h, false, w.wgu, h, false, act, f, nullptr, 0, T, f, h, mt::kEpiSwigluBf16};
    if (recompute) {
      g.C2 = gu;
      g.ldc2 = 2 * f;
    }
    if ((r = gemm_args(c, g))) return r;
  }
  if (!recompute) {
    if ((r = need_w(c, pc, 3))) return r;  // wd
    if ((r = gemm(c, act, f, false, w.wd, f, false, x_out, h, T, h, f, mt::kEpiAddF32, h1, h))) return r;
  }
  return MT_OK;
}

// Backward of one decoder layer: recompute from the checkpoint x_in, then gradients.
// dy = dL/dx_out (fp32 and its bf16 copy); writes dL/dx_in to dx (fp32, bf16) and the
// parameter gradients into g (bf16, same layout as the W section).
int layer_backward(mt_ctx* c, const LayerW& w, const LayerW& g, const float* x_in, const float* dy,
                   const bf16* dy_bf16, float* dx, bf16* dx_bf16, const Pieces* pc = nullptr) {
  const Plan& p = c->plan;
  cudaStream_t s = c->st[kStreamCompute];
  const int T = c->T, h = c->h, f = c->f, qd = c->qd, nqkv = c->nqkv;
  const double Td = T;
  int r;
  if ((r = layer_forward(c, w, x_in, nullptr, true, pc))) return r;
  if ((r = need_w(c, pc, 3))) return r;  // wd
  bf16* a = c->dev<bf16>(p.a);
  bf16* qkv = c->dev<bf16>(p.qkv);
  bf16* o = c->dev<bf16>(p.o);
  float* h1 = c->dev<float>(p.h1);
  bf16* bb = c->dev<bf16>(p.bb);
  bf16* gu = c->dev<bf16>(p.gu);
  bf16* act = c->dev<bf16>(p.act);
  bf16* dgu = c->dev<bf16>(p.dgu);
  float* db = c->dev<float>(p.db);
  float* dh = c->dev<float>(p.dh);
  bf16* dh_bf16 = c->dev<bf16>(p.dh_bf16);
  bf16* d_o = c->dev<bf16>(p.d_o);
  bf16* dqkv = c->dev<bf16>(p.dqkv);
  float* partial = c->dev<float>(p.partial);
  // down projection: dWd = dy^T act ; dact = dy Wd
  if ((r = gemm(c, dy_bf16, h, true, act, f, true, g.wd, f, h, f, T, mt::kEpiStoreBf16))) return r;
  if ((r = grad_done(c, pc, 3))) return r;  // dWd leaves while the layer computes on
  {  // dact = dy Wd, with the SwiGLU backward in the epilogue: dgu = [dg | du]
    mt::GemmArgs g{dy_bf16, h, false, w.wd, f, true, dgu, 2 * f, nullptr, 0, T, f, h, mt::kEpiSwigluBwdBf16};
    g.G = gu;
    g.ldg = 2 * f;
    if ((r = gemm_args(c, g))) return r;
  }
  // gate-up projection: dWgu = dgu^T b ; db = dgu Wgu
  if ((r = gemm(c, dgu, 2 * f, true, bb, h, true, g.wgu, h, 2 * f, h, T, mt::kEpiStoreBf16))) return r;
  if ((r = gemm(c, dgu, 2 * f, false, w.wgu, h, true, db, h, T, h, 2 * f, mt::kEpiStoreF32))) return r;
  c->launches += 2;
  r = launch(c, MT_KIND_POINTWISE, 0, Td * h * 18, [&] {
    return mt::rmsnorm_bwd(db, h1, w.ffn_norm, c->dev<float>(p.rstd2), dy, dh, dh_bf16, partial, g.ffn_norm, T, h, s);
  });
  if (r) return r;
  if ((r = grad_done(c, pc, 2))) return r;  // d ffn_norm, dWg, dWu
  // output projection: dWo = dh^T o ; do = dh Wo
  if ((r = gemm(c, dh_bf16, h, true, o, qd, true, g.wo, qd, h, qd, T, mt::kEpiStoreBf16))) return r;
  if ((r = grad_done(c, pc, 1))) return r;  // dWo
  if ((r = gemm(c, dh_bf16, h, false, w.wo, qd, true, d_o, qd, T, qd, h, mt::kEpiStoreBf16))) return r;
  c->launches += 3;
  const double attn_flops = 5.0 * c->cfg.batch * static_cast<double>(c->cfg.seq) * c->cfg.seq * c->nh * c->hd;
  r = launch(c, MT_KIND_ATTN_BWD, attn_flops, 0, [&] {
    // dq and dk leave the attention backward with the transpose RoPE rotation applied
    return mt::attn_bwd(qkv, o, c->dev<float>(p.lse), d_o, dqkv, c->dev<float>(p.delta), c->dev<float>(p.rope_cs),
                        c->cfg.batch, c->cfg.seq, c->nh, c->nkv, c->hd, c->dev<int>(p.err), s);
  });
  if (r) return r;
  // QKV projection: dWqkv = dqkv^T a ; da = dqkv Wqkv
  if ((r = gemm(c, dqkv, nqkv, true, a, h, true, g.wqkv, h, nqkv, h, T, mt::kEpiStoreBf16))) return r;
  if ((r = gemm(c, dqkv, nqkv, false, w.wqkv, h, true, db, h, T, h, nqkv, mt::kEpiStoreF32))) return r;
  c->launches += 2;
  r = launch(c, MT_KIND_POINTWISE, 0, Td * h * 18, [&] {
    return mt::rmsnorm_bwd(db, x_in, w.attn_norm, c->dev<float>(p.rstd1), dh, dx, dx_bf16, partial, g.attn_norm, T, h,
                           s);
  });
  if (r) return r;
  return grad_done(c, pc, 0);  // d attn_norm, dWq, dWk, dWv: the last piece
}

// Final norm, LM head, cross-entropy, and their backward. w_norm/w_head in the H block.
// The head runs over chunks of p.head_rows tokens: per chunk, logits = y_c W_H^T (fp32), the
// cross-entropy rows and dlogits = (softmax - onehot) / T, dW_H (+)= dlogits^T y_c and
// dy_c = dlogits W_H. With several chunks dW_H is summed in fp32, chunk after chunk (a fixed
// order), then rounded once to bf16.
int head_forward_backward(mt_ctx* c, const bf16* w_norm, const bf16* w_head, bf16* g_norm, bf16* g_head,
                          const float* x, float* dx, bf16* dx_bf16) {
  const Plan& p = c->plan;
  cudaStream_t s = c->st[kStreamCompute];
  const int T = c->T, h = c->h, V = c->V;
  const double Td = T;
  bf16* y = c->dev<bf16>(p.y);
  float* logits = c->dev<float>(p.logits);
  bf16* dlogits = c->dev<bf16>(p.dlogits);
  float* dyf = c->dev<float>(p.db);
  const int rows = c->head_rows;
  const bool chunked = rows < T;
  float* dwf = c->dev<float>(p.dw_head);
  int r;
  c->launches += 1;
  r = launch(c, MT_KIND_POINTWISE, 0, Td * h * 6,
             [&] { return mt::rmsnorm_fwd(x, w_norm, y, c->dev<float>(p.rstdf), T, h, c->cfg.rms_eps, s); });
  if (r) return r;
  for (int r0 = 0; r0 < T; r0 += rows) {
    const int tc = std::min(rows, T - r0);
    const bf16* yc = y + static_cast<int64_t>(r0) * h;
    if ((r = gemm(c, yc, h, false, w_head, h, false, logits, V, tc, V, h, mt::kEpiStoreF32))) return r;
    c->launches += 1;
    r = launch(c, MT_KIND_CROSS_ENTROPY, 0, static_cast<double>(tc) * V * 6, [&] {
      return mt::cross_entropy(logits, c->dev<int32_t>(p.lab) + r0, dlogits, c->dev<float>(p.row_loss) + r0, tc, V,
                               s, T);
    });
    if (r) return r;
    if (!chunked) {
      if ((r = gemm(c, dlogits, V, true, yc, h, true, g_head, h, V, h, tc, mt::kEpiStoreBf16))) return r;
    } else if (r0 == 0) {
      if ((r = gemm(c, dlogits, V, true, yc, h, true, dwf, h, V, h, tc, mt::kEpiStoreF32))) return r;
    } else {
      if ((r = gemm(c, dlogits, V, true, yc, h, true, dwf, h, V, h, tc, mt::kEpiAddF32, dwf, h))) return r;
    }
    if ((r = gemm(c, dlogits, V, false, w_head, h, true, dyf + static_cast<int64_t>(r0) * h, h, tc, h, V,
                  mt::kEpiStoreF32)))
      return r;
  }
  c->launches += 1;
  r = launch(c, MT_KIND_CROSS_ENTROPY, 0, Td * 4,
             [&] { return mt::mean_reduce(c->dev<float>(p.row_loss), T, c->dev<float>(p.loss), s); });
  if (r) return r;
  if (chunked) {
    c->launches += 1;
    r = launch(c, MT_KIND_POINTWISE, 0, static_cast<double>(V) * h * 6,
               [&] { return mt::cast_f32_bf16(dwf, g_head, static_cast<int64_t>(V) * h, s); });
    if (r) return r;
  }
  c->launches += 2;
  return launch(c, MT_KIND_POINTWISE, 0, Td * h * 14, [&] {
    return mt::rmsnorm_bwd(dyf, x, w_norm, c->dev<float>(p.rstdf), nullptr, dx, dx_bf16, c->dev<float>(p.partial),
                           g_norm, T, h, s);
  });
}

// ------------------------------------------------------------------ step schedule
struct Use {
  int block;  // arena block index
  int kind;   // 0 embedding fwd, 1 layer fwd, 2 head, 3 layer bwd
};

float* ckpt_slot(mt_ctx* c, int l) {
  const uint64_t stride = static_cast<uint64_t>(c->T) * c->h;
  const uint64_t slot = c->offload ? static_cast<uint64_t>(l % 2) : static_cast<uint64_t>(l);
  return c->dev<float>(c->plan.ckpt) + slot * stride;
}

int issue_h2d(mt_ctx* c, const std::vector<Use>& uses, int u) {
  const int buf = c->single ? 0 : (u & 1);
  const Use& us = uses[u];
  CK(cudaStreamWaitEvent(c->st[kStreamH2D], c->wfree[buf], 0));
  if (c->sparse_e && us.block == 0) {  // the gather reads its rows from the arena itself
    CK(cudaEventRecord(c->wready[buf], c->st[kStreamH2D]));
    return MT_OK;
  }
  const auto& blk = c->lay.blocks[us.block];
  const bool pieces = !c->single && (us.kind == 1 || us.kind == 3);
  int r = span(c, kStreamH2D, [&]() -> int {
    if (c->offload && us.kind == 3) {
      // bring the layer's input checkpoint back ahead of its weights: the first weight piece's
      // event then covers it too
      const int l = us.block - 1;
      CK(cudaStreamWaitEvent(c->st[kStreamH2D], c->ck_saved[0], 0));  // host copies written in forward
      CK(cudaStreamWaitEvent(c->st[kStreamH2D], c->ck_saved[1], 0));
      const uint64_t bytes = static_cast<uint64_t>(c->T) * c->h * 4;
      CK(cudaMemcpyAsync(ckpt_slot(c, l), c->host_ckpt + static_cast<uint64_t>(l) * c->T * c->h, bytes,
                         cudaMemcpyHostToDevice, c->st[kStreamH2D]));
      c->h2d_bytes += bytes;
    }
    if (pieces) {  // a decoder layer's weights in pieces, each announced as it lands
      for (int k = 0; k < kParts; ++k) {
        uint64_t b0, b1;
        part_range(blk, MT_SEC_W, k, b0, b1);
        CK(cudaMemcpyAsync(c->ws + c->plan.wbuf[buf] + b0, c->arena + blk.sec_offset[MT_SEC_W] + b0, b1 - b0,
                           cudaMemcpyHostToDevice, c->st[kStreamH2D]));
        CK(cudaEventRecord(c->wpart[buf][k], c->st[kStreamH2D]));
        c->h2d_bytes += b1 - b0;
      }
    } else {
      CK(cudaMemcpyAsync(c->ws + c->plan.wbuf[buf], c->arena + blk.sec_offset[MT_SEC_W], blk.sec_bytes[MT_SEC_W],
                         cudaMemcpyHostToDevice, c->st[kStreamH2D]));
      c->h2d_bytes += blk.sec_bytes[MT_SEC_W];
    }
    return MT_OK;
  });
  if (r) return r;
  CK(cudaEventRecord(c->wready[buf], c->st[kStreamH2D]));
  return MT_OK;
}

int issue_d2h_grad(mt_ctx* c, int block, int gb) {
  const auto& blk = c->lay.blocks[block];
  CK(cudaStreamWaitEvent(c->st[kStreamD2H], c->gready[gb], 0));
  int r = span(c, kStreamD2H, [&]() -> int {
    CK(cudaMemcpyAsync(c->arena + blk.sec_offset[MT_SEC_G], c->ws + c->plan.gbuf[gb], blk.sec_bytes[MT_SEC_G],
                       cudaMemcpyDeviceToHost, c->st[kStreamD2H]));
    c->d2h_bytes += blk.sec_bytes[MT_SEC_G];
    return MT_OK;
  });
  if (r) return r;
  CK(cudaEventRecord(c->gfree[gb], c->st[kStreamD2H]));
  if (block == c->L + 1)  // the head lands first: the loss is known from here on
    CK(cudaMemcpyAsync(c->pin_out + 2, c->dev<float>(c->plan.loss), sizeof(float), cudaMemcpyDeviceToHost,
                       c->st[kStreamD2H]));
  return mark_landed(c, block, c->st[kStreamD2H]);
}

// dL/dx_l has just been written to dx (fp32 [T][h]) on the compute stream: copy it to every
// destination armed for layer l.
int capture_grad(mt_ctx* c, int l, const float* dx) {
  for (const auto& cap : c->grad_capture)
    if (cap.first == l)
      CK(cudaMemcpyAsync(cap.second, dx, static_cast<uint64_t>(c->T) * c->h * 4, cudaMemcpyDeviceToHost,
                         c->st[kStreamCompute]));
  return MT_OK;
}

// Compute of use u. wbase/gbase: device bases of this block's W and G sections.
int compute_use(mt_ctx* c, const Use& us, uint8_t* wbase, uint8_t* gbase, int& dx_cur, const Pieces* pc = nullptr) {
  const Plan& p = c->plan;
  cudaStream_t s = c->st[kStreamCompute];
  const auto& blk = c->lay.blocks[us.block];
  const int L = c->L;
  int r = MT_OK;
  if (us.kind == 0) {
    const bf16* E = c->sparse_e ? reinterpret_cast<const bf16*>(c->arena_dev + blk.tensor_offset[MT_SEC_W][0])
                                : reinterpret_cast<const bf16*>(wbase);
    if (c->sparse_e) c->h2d_bytes += static_cast<uint64_t>(c->e_next.size()) * c->h * 2;
    c->launches += 1;
    if (c->sparse_e) CK(cudaEventRecord(c->ev_emb[0], s));
    r = launch(c, MT_KIND_EMBED, 0, static_cast<double>(c->T) * c->h * 6, [&] {
      return mt::embed_fwd(c->dev<int32_t>(p.tok), E, ckpt_slot(c, 0), c->T, c->h, s);
    });
    if (c->sparse_e && r == MT_OK) {
      CK(cudaEventRecord(c->ev_emb[1], s));
      c->emb_timed = true;
    }
  } else if (us.kind == 1) {
    const int l = us.block - 1;
    const LayerW w = bind_layer(c, us.block, wbase, MT_SEC_W);
    r = layer_forward(c, w, ckpt_slot(c, l), ckpt_slot(c, l + 1), false, pc);
  } else if (us.kind == 2) {
    auto wp = [&](int t) {
      return reinterpret_cast<bf16*>(wbase + (blk.tensor_offset[MT_SEC_W][t] - blk.sec_offset[MT_SEC_W]));
    };
    auto gp = [&](int t) {
      return reinterpret_cast<bf16*>(gbase + (blk.tensor_offset[MT_SEC_G][t] - blk.sec_offset[MT_SEC_G]));
    };
    dx_cur = 0;
    r = head_forward_backward(c, wp(MT_T_FINAL_NORM), wp(MT_T_W_HEAD), gp(MT_T_FINAL_NORM), gp(MT_T_W_HEAD),
                              ckpt_slot(c, L), c->dev<float>(p.dx[0]), c->dev<bf16>(p.dx_bf16[0]));
    if (r == MT_OK) r = capture_grad(c, L, c->dev<float>(p.dx[0]));
  } else {
    const int l = us.block - 1;
    const LayerW w = bind_layer(c, us.block, wbase, MT_SEC_W);
    const LayerW g = bind_layer(c, us.block, gbase, MT_SEC_G);
    const int nx = dx_cur ^ 1;
    r = layer_backward(c, w, g, ckpt_slot(c, l), c->dev<float>(p.dx[dx_cur]), c->dev<bf16>(p.dx_bf16[dx_cur]),
                       c->dev<float>(p.dx[nx]), c->dev<bf16>(p.dx_bf16[nx]), pc);
    if (r == MT_OK) r = capture_grad(c, l, c->dev<float>(p.dx[nx]));
    dx_cur = nx;
  }
  return r;
}

int stage_inputs(mt_ctx* c, const int32_t* tokens, const int32_t* labels) {
  const int T = c->T, V = c->V;
  int32_t* tok = c->pin_io;
  int32_t* lab = tok + T;
  int32_t* order = lab + T;
  int32_t* offs = order + T;
  std::memcpy(tok, tokens, sizeof(int32_t) * T);
  std::memcpy(lab, labels, sizeof(int32_t) * T);
  // positions grouped by token id, ascending within each id (stable counting sort)
  std::memset(offs, 0, sizeof(int32_t) * (V + 1));
  for (int t = 0; t < T; ++t) offs[tok[t] + 1] += 1;
  for (int v = 0; v < V; ++v) offs[v + 1] += offs[v];
  std::vector<int32_t> cur(offs, offs + V);
  for (int t = 0; t < T; ++t) order[cur[tok[t]]++] = t;
  const Plan& p = c->plan;
  // on the h2d stream ahead of the first weight copy: the copy engine runs a stream's copies in
  // order, so the ids arrive before the layer weights instead of behind them
  cudaStream_t s = c->st[kStreamH2D];
  if (c->sparse_e) {
    // rows the embedding backward writes: this batch's ids and the last batch's (ascending)
    c->e_next.clear();
    for (int v = 0; v < V; ++v)
      if (offs[v + 1] > offs[v]) c->e_next.push_back(v);
    int32_t* rows = offs + V + 1;
    c->n_erows = static_cast<int>(std::set_union(c->e_next.begin(), c->e_next.end(), c->e_prev.begin(),
                                                 c->e_prev.end(), rows) -
                                  rows);
    CK(cudaMemcpyAsync(c->dev<int32_t>(p.erows), rows, sizeof(int32_t) * c->n_erows, cudaMemcpyHostToDevice, s));
    c->h2d_bytes += sizeof(int32_t) * static_cast<uint64_t>(c->n_erows);
  }
  CK(cudaMemcpyAsync(c->dev<int32_t>(p.tok), tok, sizeof(int32_t) * T, cudaMemcpyHostToDevice, s));
  CK(cudaMemcpyAsync(c->dev<int32_t>(p.lab), lab, sizeof(int32_t) * T, cudaMemcpyHostToDevice, s));
  CK(cudaMemcpyAsync(c->dev<int32_t>(p.order), order, sizeof(int32_t) * T, cudaMemcpyHostToDevice, s));
  CK(cudaMemcpyAsync(c->dev<int32_t>(p.offsets), offs, sizeof(int32_t) * (V + 1), cudaMemcpyHostToDevice, s));
  c->h2d_bytes += sizeof(int32_t) * (3 * static_cast<uint64_t>(T) + V + 1);
  CK(cudaEventRecord(c->ev_inputs, s));
  return wait_copy(c, c->ev_inputs);
}

int enqueue_step(mt_ctx* c, const int32_t* tokens, const int32_t* labels) {
  const Plan& p = c->plan;
  cudaStream_t cs = c->st[kStreamCompute];
  const int L = c->L;
  CK(cudaEventRecord(c->ev_start, cs));
  CK(cudaStreamWaitEvent(c->st[kStreamH2D], c->ev_start, 0));
  CK(cudaStreamWaitEvent(c->st[kStreamD2H], c->ev_start, 0));
  CK(cudaMemsetAsync(c->dev<int>(p.err), 0, sizeof(int), cs));
  int r = stage_inputs(c, tokens, labels);
  if (r) return r;

  std::vector<Use> uses;
  uses.push_back({0, 0});
  for (int l = 0; l < L; ++l) uses.push_back({l + 1, 1});
  uses.push_back({L + 1, 2});
  for (int l = L - 1; l >= 0; --l) uses.push_back({l + 1, 3});
  const int U = static_cast<int>(uses.size());
  int dx_cur = 0;
  int gcount = 0;  // G-buffer uses so far
  // Layout kind (0 E, 1 decoder layer, 2 H) each G buffer last held: the D2H copies a whole
  // section, padding included, so a buffer is zeroed when the layout written into it changes.
  int gkind[2] = {-1, -1};
  auto block_kind = [&](int block) { return block == 0 ? 0 : (block == L + 1 ? 2 : 1); };
  auto prepare_gbuf = [&](int gb, int block) -> int {
    const int k = block_kind(block);
    if (gkind[gb] != k) {
      CK(cudaMemsetAsync(c->ws + p.gbuf[gb], 0, c->lay.max_wsec, cs));
      gkind[gb] = k;
    }
    return MT_OK;
  };

  if (c->resident) {
    // upload every W section, compute everything with G on the device, download every G section
    r = span(c, kStreamH2D, [&]() -> int {
      uint64_t off = 0;
      for (const auto& blk : c->lay.blocks) {
        CK(cudaMemcpyAsync(c->ws + p.res_w + off, c->arena + blk.sec_offset[MT_SEC_W], blk.sec_bytes[MT_SEC_W],
                           cudaMemcpyHostToDevice, c->st[kStreamH2D]));
        c->h2d_bytes += blk.sec_bytes[MT_SEC_W];
        off += blk.sec_bytes[MT_SEC_W];
      }
      return MT_OK;
    });
    if (r) return r;
    CK(cudaEventRecord(c->wready[0], c->st[kStreamH2D]));
    if ((r = wait_copy(c, c->wready[0]))) return r;
    std::vector<uint64_t> base(c->lay.blocks.size());
    uint64_t off = 0;
    for (size_t b = 0; b < base.size(); ++b) {
      base[b] = off;
      off += c->lay.blocks[b].sec_bytes[MT_SEC_W];
    }
    for (int u = 0; u < U; ++u) {
      const Use& us = uses[u];
      if (us.kind == 2) CK(cudaEventRecord(c->ev_fwd_end, cs));
      r = span(c, kStreamCompute, [&] {
        return compute_use(c, us, c->ws + p.res_w + base[us.block], c->ws + p.res_g + base[us.block], dx_cur);
      });
      if (r) return r;
    }
    r = span(c, kStreamCompute, [&]() -> int {
      c->launches += 1;
      return launch(c, MT_KIND_EMBED, 0, static_cast<double>(c->T) * c->h * 4 + static_cast<double>(c->V) * c->h * 2,
                    [&] {
                      return mt::embed_bwd(c->dev<int32_t>(p.order), c->dev<int32_t>(p.offsets),
                                           c->dev<float>(p.dx[dx_cur]),
                                           reinterpret_cast<bf16*>(c->ws + p.res_g + base[0]), c->V, c->h, cs);
                    });
    });
    if (r) return r;
    CK(cudaEventRecord(c->gready[0], cs));
    CK(cudaStreamWaitEvent(c->st[kStreamD2H], c->gready[0], 0));
    CK(cudaMemcpyAsync(c->pin_out + 2, c->dev<float>(p.loss), sizeof(float), cudaMemcpyDeviceToHost,
                       c->st[kStreamD2H]));
    r = span(c, kStreamD2H, [&]() -> int {
      for (size_t b = 0; b < base.size(); ++b) {
        const auto& blk = c->lay.blocks[b];
        CK(cudaMemcpyAsync(c->arena + blk.sec_offset[MT_SEC_G], c->ws + p.res_g + base[b], blk.sec_bytes[MT_SEC_G],
                           cudaMemcpyDeviceToHost, c->st[kStreamD2H]));
        int rr = mark_landed(c, static_cast<int>(b), c->st[kStreamD2H]);
        if (rr) return rr;
        c->d2h_bytes += blk.sec_bytes[MT_SEC_G];
      }
      return MT_OK;
    });
    if (r) return r;
  } else {
    auto compute = [&](int u) -> int {
      const Use& us = uses[u];
      const int buf = c->single ? 0 : (u & 1);
      // decoder layers wait for their weights piece by piece (inside the layer template)
      const bool pieces = !c->single && (us.kind == 1 || us.kind == 3);
      if (!pieces) {
        int rw = wait_copy(c, c->wready[buf]);
        if (rw) return rw;
      }
      int gb = 0;
      const bool writes_g = (us.kind >= 2);
      if (writes_g) {
        gb = c->single ? 0 : (gcount & 1);
        int rr = wait_copy(c, c->gfree[gb]);
        if (rr) return rr;
        rr = prepare_gbuf(gb, us.block);
        if (rr) return rr;
      }
      if (c->offload && us.kind == 1) {
        // x_{l+1} overwrites the slot of x_{l-1}: its host copy must have finished
        const int l = us.block - 1;
        int rw = wait_copy(c, c->ck_saved[(l + 1) & 1]);
        if (rw) return rw;
      }
      if (us.kind == 2) CK(cudaEventRecord(c->ev_fwd_end, cs));
      Pieces pc;
      if (pieces) {
        pc.wbuf = buf;
        pc.gbuf = us.kind == 3 ? gb : -1;  // a layer's gradients leave piece by piece too
        pc.block = us.block;
      }
      int rr = span(c, kStreamCompute, [&] {
        return compute_use(c, us, c->ws + p.wbuf[buf], c->ws + p.gbuf[gb], dx_cur, pieces ? &pc : nullptr);
      });
      if (rr) return rr;
      CK(cudaEventRecord(c->wfree[buf], cs));
      if (c->offload && (us.kind == 0 || (us.kind == 1 && us.block < L))) {
        // checkpoint x_l (l = 0 after the embedding, l = block after layer block-1) to the host
        const int l = (us.kind == 0) ? 0 : us.block;
        CK(cudaEventRecord(c->ck_ready[l & 1], cs));
        CK(cudaStreamWaitEvent(c->st[kStreamD2H], c->ck_ready[l & 1], 0));
        const uint64_t bytes = static_cast<uint64_t>(c->T) * c->h * 4;
        rr = span(c, kStreamD2H, [&]() -> int {
          CK(cudaMemcpyAsync(c->host_ckpt + static_cast<uint64_t>(l) * c->T * c->h, ckpt_slot(c, l), bytes,
                             cudaMemcpyDeviceToHost, c->st[kStreamD2H]));
          c->d2h_bytes += bytes;
          return MT_OK;
        });
        if (rr) return rr;
        CK(cudaEventRecord(c->ck_saved[l & 1], c->st[kStreamD2H]));
      }
      if (writes_g) {
        if (!(pieces && us.kind == 3)) {  // whole-section offload (the head; the single-buffer ablation)
          CK(cudaEventRecord(c->gready[gb], cs));
          rr = issue_d2h_grad(c, us.block, gb);
          if (rr) return rr;
        }
        gcount += 1;
      }
      return MT_OK;
    };
    if (c->single) {
      for (int u = 0; u < U; ++u) {
        if ((r = issue_h2d(c, uses, u))) return r;
        if ((r = compute(u))) return r;
      }
    } else {
      if ((r = issue_h2d(c, uses, 0))) return r;
      for (int u = 0; u < U; ++u) {
        if (u + 1 < U && (r = issue_h2d(c, uses, u + 1))) return r;
        if ((r = compute(u))) return r;
      }
    }
    if (c->sparse_e) {
      // embedding gradient rows straight into the arena's G section
      const auto& eb = c->lay.blocks[0];
      bf16* gE = reinterpret_cast<bf16*>(c->arena_dev + eb.tensor_offset[MT_SEC_G][0]);
      r = span(c, kStreamCompute, [&]() -> int {
        c->launches += 1;
        return launch(c, MT_KIND_EMBED, 0, static_cast<double>(c->T) * c->h * 4 + 2.0 * c->n_erows * c->h, [&] {
          return mt::embed_bwd_rows(c->dev<int32_t>(p.order), c->dev<int32_t>(p.offsets), c->dev<int32_t>(p.erows),
                                    c->n_erows, c->dev<float>(p.dx[dx_cur]), gE, c->h, cs);
        });
      });
      if (r) return r;
      if ((r = mark_landed(c, 0, cs))) return r;
      c->d2h_bytes += static_cast<uint64_t>(c->n_erows) * c->h * 2;
    } else {
    // embedding gradient into a G buffer, then offload
    const int gb = c->single ? 0 : (gcount & 1);
    if ((r = wait_copy(c, c->gfree[gb]))) return r;
    if ((r = prepare_gbuf(gb, 0))) return r;
    const auto& eb = c->lay.blocks[0];
    r = span(c, kStreamCompute, [&]() -> int {
      c->launches += 1;
      return launch(c, MT_KIND_EMBED, 0, static_cast<double>(c->T) * c->h * 4 + static_cast<double>(c->V) * c->h * 2,
                    [&] {
                      return mt::embed_bwd(
                          c->dev<int32_t>(p.order), c->dev<int32_t>(p.offsets), c->dev<float>(p.dx[dx_cur]),
                          reinterpret_cast<bf16*>(c->ws + p.gbuf[gb] +
                                                  (eb.tensor_offset[MT_SEC_G][0] - eb.sec_offset[MT_SEC_G])),
                          c->V, c->h, cs);
                    });
    });
    if (r) return r;
    CK(cudaEventRecord(c->gready[gb], cs));
    if ((r = issue_d2h_grad(c, 0, gb))) return r;
    }
  }
  // join: the compute stream waits for the last copies, then reads back loss and error flag
  CK(cudaEventRecord(c->ev_d2h_done, c->st[kStreamD2H]));
  if ((r = wait_copy(c, c->ev_d2h_done))) return r;
  CK(cudaStreamWaitEvent(cs, c->wready[0], 0));
  CK(cudaStreamWaitEvent(cs, c->wready[1], 0));
  CK(cudaMemcpyAsync(c->pin_out, c->dev<float>(p.loss), sizeof(float), cudaMemcpyDeviceToHost, cs));
  CK(cudaMemcpyAsync(c->pin_out + 1, c->dev<int>(p.err), sizeof(int), cudaMemcpyDeviceToHost, cs));
  CK(cudaEventRecord(c->ev_end, cs));
  return MT_OK;
}

// Poll `ev` until it completes or the deadline passes.
int wait_event(mt_ctx* c, cudaEvent_t ev, double seconds) {
  const auto t0 = std::chrono::steady_clock::now();
  for (;;) {
    cudaError_t e = cudaEventQuery(ev);
    if (e == cudaSuccess) return MT_OK;
    if (e != cudaErrorNotReady) return set_err(c, MT_ECUDA, std::string("step failed: ") + cudaGetErrorString(e));
    const double el = std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
    if (el > seconds) return set_err(c, MT_ETIMEOUT, "step did not complete within the wait limit");
    std::this_thread::sleep_for(std::chrono::microseconds(el < 0.01 ? 20 : 200));
  }
}

float elapsed(cudaEvent_t a, cudaEvent_t b) {
  float ms = 0.f;
  if (cudaEventElapsedTime(&ms, a, b) != cudaSuccess) return 0.f;
  return ms;
}

void release(mt_ctx* c) {
  if (!c) return;
  if (c->broken) {
    // work of a timed-out step may still run on the device: free only what no device work
    // uses (host memory the step does not touch is left registered/allocated: it may still
    // be the target of a copy), and do not wait
    delete c;
    return;
  }
  cudaDeviceSynchronize();
  for (auto e : c->span_pool) cudaEventDestroy(e);
  for (auto e : c->kpool) cudaEventDestroy(e);
  cudaEvent_t* evs[] = {c->wready, c->wfree, c->gready, c->gfree, c->ck_ready, c->ck_saved};
  for (auto arr : evs)
    for (int i = 0; i < 2; ++i)
      if (arr[i]) cudaEventDestroy(arr[i]);
  for (int i = 0; i < 2; ++i)
    for (int k = 0; k < kParts; ++k) {
      if (c->wpart[i][k]) cudaEventDestroy(c->wpart[i][k]);
      if (c->gpart[i][k]) cudaEventDestroy(c->gpart[i][k]);
    }
  for (auto e : {c->ev_start, c->ev_fwd_end, c->ev_end, c->ev_d2h_done, c->ev_inputs, c->ev_emb[0], c->ev_emb[1]})
    if (e) cudaEventDestroy(e);
  for (auto e : c->g_landed)
    if (e) cudaEventDestroy(e);
  for (int i = 0; i < 3; ++i)
    if (c->own_st[i] && c->st[i]) cudaStreamDestroy(c->st[i]);
  if (c->own_ws && c->ws) cudaFree(c->ws);
  if (c->registered && c->arena) cudaHostUnregister(c->arena);
  if (c->host_ckpt) mt::host_free(c->host_ckpt);
  if (c->pin_io) cudaFreeHost(c->pin_io);
  if (c->pin_out) cudaFreeHost(c->pin_out);
  delete c;
}

void build_rope_table(const mt_model_cfg& cfg, std::vector<float>& cs) {
  const int hd = cfg.hidden / cfg.n_heads, half = hd / 2;
  cs.resize(static_cast<size_t>(cfg.seq) * half * 2);
  for (int pos = 0; pos < cfg.seq; ++pos)
    for (int i = 0; i < half; ++i) {
      const double inv = std::pow(static_cast<double>(cfg.rope_theta), -2.0 * i / hd);
      const double ang = static_cast<double>(pos) * inv;
      cs[(static_cast<size_t>(pos) * half + i) * 2 + 0] = static_cast<float>(std::cos(ang));
      cs[(static_cast<size_t>(pos) * half + i) * 2 + 1] = static_cast<float>(std::sin(ang));
    }
}

}  // namespace

// ------------------------------------------------------------------ C ABI
namespace {
int train_step_impl(mt_ctx* c, const int32_t* tokens, const int32_t* labels, float* loss, const mt_adam_cfg* hp);
}  // namespace

extern "C" {

int mt_host_alloc(uint64_t bytes, void** out) {
  mt_ctx* c = nullptr;
  if (!out || bytes == 0) return MT_EINVAL;
  *out = nullptr;
  CK(mt::host_alloc(bytes, out));
  return MT_OK;
}

int mt_host_alloc_query(const void* p, mt_host_alloc_info* out) {
  mt::HostAllocInfo i{};
  if (!p || !out || !mt::host_alloc_info(p, &i) || i.chunk_bytes == 0) return MT_EINVAL;
  out->chunk_bytes = i.chunk_bytes;
  out->chunks = i.chunks;
  out->spare = i.spare;
  out->slow_found = i.slow_found;
  out->replaced = i.replaced;
  out->median_gbs = i.median_gbs;
  out->min_gbs = i.min_gbs;
  return MT_OK;
}

int mt_host_free(void* p) {
  mt_ctx* c = nullptr;
  if (!p) return MT_OK;
  CK(mt::host_free(p));
  return MT_OK;
}

int mt_workspace_bytes(const mt_model_cfg* cfg, uint64_t* bytes) {
  std::string why;
  if (!cfg || !bytes) return MT_EINVAL;
  if (!mt::validate_cfg(*cfg, &why)) return MT_EINVAL;
  *bytes = make_plan(*cfg, mt::compute_layout(*cfg)).total;
  return MT_OK;
}

int mt_create(const mt_model_cfg* cfg, const mt_device_resources* res, mt_ctx** out) {
  if (!out) return MT_EINVAL;
  *out = nullptr;
  std::string why;
  if (!cfg || !mt::validate_cfg(*cfg, &why)) return MT_EINVAL;
  mt_ctx* c = new mt_ctx();
  c->cfg = *cfg;
  c->lay = mt::compute_layout(*cfg);
  c->plan = make_plan(*cfg, c->lay);
  c->T = cfg->batch * cfg->seq;
  c->h = cfg->hidden;
  c->nh = cfg->n_heads;
  c->nkv = cfg->n_kv_heads;
  c->hd = cfg->hidden / cfg->n_heads;
  c->f = cfg->ffn;
  c->V = cfg->vocab;
  c->L = cfg->n_layers;
  c->qd = c->nh * c->hd;
  c->nqkv = (c->nh + 2 * c->nkv) * c->hd;
  c->head_rows = c->plan.head_rows;
  c->resident = cfg->flags & MT_FLAG_RESIDENT;
  c->offload = cfg->flags & MT_FLAG_OFFLOAD_CKPT;
  c->single = cfg->flags & MT_FLAG_SINGLE_BUFFER;
  c->timing = cfg->flags & MT_FLAG_KERNEL_TIMING;
  auto bail = [&](int code) {
    release(c);
    return code;
  };
  if (c->resident && (c->offload || c->single)) return bail(MT_EINVAL);
  // fused projections need wq|wk|wv and wg|wu back to back in the section
  {
    const auto& b1 = c->lay.blocks[1];
    const auto& to = b1.tensor_offset[MT_SEC_W];
    const uint64_t qb = static_cast<uint64_t>(c->qd) * c->h * 2, kb = static_cast<uint64_t>(c->nkv) * c->hd * c->h * 2;
    const uint64_t fb = static_cast<uint64_t>(c->f) * c->h * 2;
    if (to[MT_T_WK] != to[MT_T_WQ] + qb || to[MT_T_WV] != to[MT_T_WK] + kb || to[MT_T_WU] != to[MT_T_WG] + fb)
      return bail(MT_EINVAL);
  }
  if (res && res->workspace) {
    if (res->workspace_bytes < c->plan.total || (reinterpret_cast<uintptr_t>(res->workspace) & 255))
      return bail(MT_EINVAL);
    c->ws = static_cast<uint8_t*>(res->workspace);
  } else {
    if (cudaMalloc(&c->ws, c->plan.total) != cudaSuccess) {
      c->ws = nullptr;
      return bail(MT_ENOMEM);
    }
    c->own_ws = true;
  }
  for (int i = 0; i < 3; ++i) {
    if (res && res->streams[i]) {
      c->st[i] = static_cast<cudaStream_t>(res->streams[i]);
    } else {
      if (cudaStreamCreateWithFlags(&c->st[i], cudaStreamNonBlocking) != cudaSuccess) return bail(MT_ECUDA);
      c->own_st[i] = true;
    }
  }
  cudaEvent_t* evs[] = {c->wready, c->wfree, c->gready, c->gfree, c->ck_ready, c->ck_saved};
  for (auto arr : evs)
    for (int i = 0; i < 2; ++i)
      if (cudaEventCreateWithFlags(&arr[i], cudaEventDisableTiming) != cudaSuccess) return bail(MT_ECUDA);
  for (int i = 0; i < 2; ++i)
    for (int k = 0; k < kParts; ++k)
      if (cudaEventCreateWithFlags(&c->wpart[i][k], cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&c->gpart[i][k], cudaEventDisableTiming) != cudaSuccess)
        return bail(MT_ECUDA);
  for (auto e : {&c->ev_start, &c->ev_fwd_end, &c->ev_end, &c->ev_d2h_done, &c->ev_emb[0], &c->ev_emb[1]})
    if (cudaEventCreate(e) != cudaSuccess) return bail(MT_ECUDA);
  if (cudaEventCreateWithFlags(&c->ev_inputs, cudaEventDisableTiming) != cudaSuccess) return bail(MT_ECUDA);
  c->g_landed.assign(c->lay.blocks.size(), nullptr);
  for (auto& e : c->g_landed)
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return bail(MT_ECUDA);
  // pinned staging
  const uint64_t io = (5 * static_cast<uint64_t>(c->T) + c->V + 1) * sizeof(int32_t);
  if (cudaHostAlloc(reinterpret_cast<void**>(&c->pin_io), io, cudaHostAllocDefault) != cudaSuccess) {
    c->pin_io = nullptr;
    return bail(MT_ENOMEM);
  }
  const uint64_t n_out = 4 + c->lay.blocks.size();
  if (cudaHostAlloc(reinterpret_cast<void**>(&c->pin_out), n_out * 4, cudaHostAllocDefault) != cudaSuccess) {
    c->pin_out = nullptr;
    return bail(MT_ENOMEM);
  }
  std::memset(c->pin_out, 0, n_out * 4);
  c->pin_flags = reinterpret_cast<int*>(c->pin_out + 4);
  if (c->offload) {
    const uint64_t bytes = static_cast<uint64_t>(c->L) * c->T * c->h * 4;
    if (mt::host_alloc(bytes, reinterpret_cast<void**>(&c->host_ckpt)) != cudaSuccess) {
      c->host_ckpt = nullptr;
      return bail(MT_ENOMEM);
    }
  }
  // constant RoPE table; zeroed G buffers (their padding bytes reach the host arena as zeros)
  std::vector<float> cs;
  build_rope_table(*cfg, cs);
  cudaStream_t s = c->st[kStreamCompute];
  if (cudaMemcpyAsync(c->dev<float>(c->plan.rope_cs), cs.data(), cs.size() * sizeof(float), cudaMemcpyHostToDevice,
                      s) != cudaSuccess)
    return bail(MT_ECUDA);
  if (cudaMemsetAsync(c->ws + c->plan.gemm_ws, 0, mt::kGemmFlagBytes, s) != cudaSuccess) return bail(MT_ECUDA);
  if (c->resident) {
    if (cudaMemsetAsync(c->ws + c->plan.res_g, 0, c->plan.res_bytes, s) != cudaSuccess) return bail(MT_ECUDA);
  } else {
    for (int i = 0; i < 2; ++i)
      if (cudaMemsetAsync(c->ws + c->plan.gbuf[i], 0, c->lay.max_wsec, s) != cudaSuccess) return bail(MT_ECUDA);
  }
  if (cudaStreamSynchronize(s) != cudaSuccess) return bail(MT_ECUDA);
  if (mt::gemm_num_sms() <= 0) return bail(MT_ECUDA);
  *out = c;
  return MT_OK;
}

int mt_bind_host_arena(mt_ctx* c, void* base, uint64_t bytes) {
  if (!c || !base) return set_err(c, MT_EINVAL, "null argument");
  if (reinterpret_cast<uintptr_t>(base) % mt::kAlign) return set_err(c, MT_EALIGN, "arena base not 4096-aligned");
  if (bytes < c->lay.total) return set_err(c, MT_EINVAL, "arena smaller than mt_arena_bytes()");
  if (c->registered && c->arena) {
    cudaHostUnregister(c->arena);
    c->registered = false;
  }
  cudaPointerAttributes attr{};
  cudaError_t e = cudaPointerGetAttributes(&attr, base);
  const bool pinned = (e == cudaSuccess && attr.type == cudaMemoryTypeHost);
  if (e != cudaSuccess) cudaGetLastError();
  if (!pinned) {
    e = cudaHostRegister(base, bytes, cudaHostRegisterDefault);
    if (e != cudaSuccess) return set_err(c, MT_ENOMEM, std::string("cudaHostRegister: ") + cudaGetErrorString(e));
    c->registered = true;
  }
  c->arena = static_cast<uint8_t*>(base);
  c->arena_bytes = bytes;
  c->grads_valid = false;
  // the arena's address on the device, when page-locked memory is mapped there (unified addressing)
  cudaPointerAttributes da{};
  if (cudaPointerGetAttributes(&da, base) == cudaSuccess && da.devicePointer) {
    c->arena_dev = static_cast<uint8_t*>(da.devicePointer);
  } else {
    cudaGetLastError();
    c->arena_dev = nullptr;
  }
  c->sparse_e = !c->resident && c->arena_dev != nullptr && !(c->cfg.flags & MT_FLAG_DENSE_EMBED);
  c->e_clean = false;  // E's G section is cleared before the first sparse step
  c->e_prev.clear();
  return MT_OK;
}

int mt_train_step(mt_ctx* c, const int32_t* tokens, const int32_t* labels, float* loss) {
  return train_step_impl(c, tokens, labels, loss, nullptr);
}

int mt_train_step_adam(mt_ctx* c, const int32_t* tokens, const int32_t* labels, const mt_adam_cfg* hp,
                       float* loss) {
  if (!hp) return set_err(c, MT_EINVAL, "null argument");
  if (!mt::adam_cfg_ok(*hp)) return set_err(c, MT_EINVAL, "bad Adam hyperparameters");
  return train_step_impl(c, tokens, labels, loss, hp);
}

}  // extern "C"

namespace {
int train_step_impl(mt_ctx* c, const int32_t* tokens, const int32_t* labels, float* loss, const mt_adam_cfg* hp) {
  if (!c || !tokens || !labels || !loss) return set_err(c, MT_EINVAL, "null argument");
  if (c->broken) return set_err(c, MT_ESTATE, "context unusable: an earlier step's wait limit expired");
  if (!c->arena) return set_err(c, MT_ESTATE, "no host arena bound");
  for (int t = 0; t < c->T; ++t) {  // ids are checked before any work is enqueued
    if (tokens[t] < 0 || tokens[t] >= c->V || labels[t] < 0 || labels[t] >= c->V)
      return set_err(c, MT_EINVAL, "token or label id out of [0, vocab)");
  }
  const auto t0 = std::chrono::steady_clock::now();
  if (c->sparse_e && !c->e_clean) {
    // the sparse embedding backward writes only changed rows: start from a zero G section
    const auto& eb = c->lay.blocks[0];
    std::memset(c->arena + eb.sec_offset[MT_SEC_G], 0, eb.sec_bytes[MT_SEC_G]);
    c->e_prev.clear();
    c->e_clean = true;
  }
  c->span_used = 0;
  c->spans.clear();
  c->waits.clear();
  c->kused = 0;
  c->klaunch.clear();
  c->launches = 0;
  c->h2d_bytes = c->d2h_bytes = 0;
  c->grads_valid = false;
  std::memset(c->pin_flags, 0, sizeof(int) * c->lay.blocks.size());
  c->pin_out[2] = 0.f;
  int r = enqueue_step(c, tokens, labels);
  double adam_ms = 0.0;
  int adam_blocks = 0;    // blocks the overlapped Adam has updated
  int stop_code = MT_OK;  // why the overlapped Adam stopped early (MT_EKERNEL, MT_ECUDA)
  std::string stop_msg;
  if (r == MT_OK && hp) {
    // Adam on each block as soon as its gradients are in the arena, in landing order (head,
    // decoder layers from the last, embedding), while the GPU works on earlier layers
    std::vector<int> order;
    order.push_back(c->L + 1);
    for (int b = c->L; b >= 0; --b) order.push_back(b);
    if (c->resident) {  // resident mode copies the sections in block order at the end
      order.clear();
      for (int b = 0; b <= c->L + 1; ++b) order.push_back(b);
    }
    for (int b : order) {
      if ((r = wait_event(c, c->g_landed[b], kStepWaitSeconds)) != MT_OK) break;
      // the loss is on the host before the first block lands (the head in streamed mode,
      // every block at once in resident mode); a kernel's error flag travels with each block
      if (adam_blocks == 0 && !std::isfinite(c->pin_out[2])) {
        stop_code = MT_ECUDA;
        stop_msg = "non-finite loss; the overlapped Adam updated no block";
        break;
      }
      if (c->pin_flags[b] != 0) {
        stop_code = MT_EKERNEL;
        stop_msg = "a kernel's bounded wait gave up (code " + std::to_string(c->pin_flags[b]) +
                   "); the overlapped Adam stopped after " + std::to_string(adam_blocks) + " block(s)";
        break;
      }
      const auto a0 = std::chrono::steady_clock::now();
      mt::adam_block(c->lay, b, c->arena, *hp);
      adam_ms += std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - a0).count();
      adam_blocks += 1;
    }
  }
  if (r == MT_OK) r = wait_event(c, c->ev_end, kStepWaitSeconds);
  if (r == MT_ETIMEOUT) {
    // the device has not finished within the limit: waiting on it again without a limit would
    // defeat the limit, so the context is given up (mt_destroy releases what it can)
    c->broken = true;
    c->e_clean = false;
    return r;
  }
  if (r != MT_OK) {
    c->e_clean = false;  // the embedding rows written are unknown: clear E's G section next time
    cudaStreamSynchronize(c->st[kStreamCompute]);  // leave no work in flight behind a failed step
    cudaStreamSynchronize(c->st[kStreamH2D]);
    cudaStreamSynchronize(c->st[kStreamD2H]);
    return r;
  }
  int kerr = 0;
  std::memcpy(&kerr, c->pin_out + 1, sizeof(int));
  if (stop_code != MT_OK) {
    c->e_clean = false;
    return set_err(c, stop_code, stop_msg);
  }
  if (kerr != 0) {
    c->e_clean = false;
    return set_err(c, MT_EKERNEL, "a kernel's bounded wait gave up (code " + std::to_string(kerr) + ")");
  }
  if (c->sparse_e) c->e_prev.swap(c->e_next);  // the rows this step's gradient wrote
  *loss = c->pin_out[0];
  if (!std::isfinite(*loss)) return set_err(c, MT_ECUDA, "non-finite loss");
  // statistics
  mt_stats& S = c->stats;
  S.host_step_ms = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
  S.step_ms = elapsed(c->ev_start, c->ev_end);
  S.fwd_ms = elapsed(c->ev_start, c->ev_fwd_end);
  S.bwd_ms = S.step_ms - S.fwd_ms;
  double busy[3] = {0, 0, 0};
  for (auto& v : S.copy_bytes) v[0] = v[1] = 0;
  for (auto& v : S.copy_ms) v[0] = v[1] = 0;
  S.first_copy_ms = 0;
  for (const auto& sp : c->spans) {
    const double d = elapsed(sp.a, sp.b);
    busy[sp.stream] += d;
    if (sp.stream == kStreamCompute) continue;
    const int dir = sp.stream == kStreamH2D ? 0 : 1;
    const int phase = elapsed(c->ev_start, sp.a) < S.fwd_ms ? 0 : 1;
    S.copy_bytes[dir][phase] += sp.bytes;
    S.copy_ms[dir][phase] += d;
    if (dir == 0 && S.first_copy_ms == 0 && sp.bytes >= (1u << 20)) S.first_copy_ms = d;
  }
  // The mapped-arena embedding gather normally reads its rows at close to the link's rate; on
  // this platform it has been seen to fall to 4-8 GB/s for a whole process. When a gather of at
  // least 16 MB runs below kMappedEmbedFloorGbs, later steps copy the embedding block whole
  // instead (the same results, bit for bit); the stats say which path the step took.
  S.sparse_embed = c->sparse_e ? 1 : 0;
  S.embed_gather_gbs = 0;
  if (c->sparse_e && c->emb_timed) {
    const double bytes = static_cast<double>(c->T) * c->h * 2, ms = elapsed(c->ev_emb[0], c->ev_emb[1]);
    S.embed_gather_gbs = ms > 0 ? bytes / (ms * 1e-3) / 1e9 : 0.0;
    if (bytes >= 16e6 && S.embed_gather_gbs < kMappedEmbedFloorGbs) c->sparse_e = false;
  }
  c->emb_timed = false;
  S.h2d_busy_ms = busy[kStreamH2D];
  S.compute_busy_ms = busy[kStreamCompute];
  S.d2h_busy_ms = busy[kStreamD2H];
  S.exposed_ms = 0;
  for (const auto& w : c->waits) S.exposed_ms += elapsed(w.first, w.second);
  S.h2d_bytes = c->h2d_bytes;
  S.d2h_bytes = c->d2h_bytes;
  S.kernel_launches = c->launches;
  S.steps += 1;
  if (const char* tr = std::getenv("MT_TRACE"); tr && tr[0] == '1') {  // per-span timeline on stderr
    static const char* names[3] = {"h2d", "compute", "d2h"};
    for (const auto& sp : c->spans)
      std::fprintf(stderr, "span %s start %.3f ms dur %.3f ms bytes %llu\n", names[sp.stream],
                   elapsed(c->ev_start, sp.a), elapsed(sp.a, sp.b), static_cast<unsigned long long>(sp.bytes));
    for (const auto& w : c->waits)
      std::fprintf(stderr, "wait start %.3f ms dur %.3f ms\n", elapsed(c->ev_start, w.first), elapsed(w.first, w.second));
  }
  for (auto& k : c->kstats) k = mt_kernel_stats{};
  for (const auto& kl : c->klaunch) {
    auto& k = c->kstats[kl.kind];
    k.launches += 1;
    k.ms += elapsed(kl.a, kl.b);
    k.flops += kl.flops;
    k.bytes += kl.bytes;
  }
  if (hp) S.adam_ms = adam_ms;
  c->grads_valid = true;
  return MT_OK;
}
}  // namespace

extern "C" {

int mt_adam_step(mt_ctx* c, const mt_adam_cfg* hp) {
  if (!c || !hp) return set_err(c, MT_EINVAL, "null argument");
  if (!c->arena) return set_err(c, MT_ESTATE, "no host arena bound");
  if (!c->grads_valid) return set_err(c, MT_ESTATE, "gradients invalid: no successful mt_train_step since bind");
  if (!mt::adam_cfg_ok(*hp)) return set_err(c, MT_EINVAL, "bad Adam hyperparameters");
  const auto t0 = std::chrono::steady_clock::now();
  mt::adam_arena(c->lay, c->arena, *hp);
  c->stats.adam_ms = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
  return MT_OK;
}

int mt_adam_apply(const mt_model_cfg* cfg, void* arena, uint64_t bytes, const mt_adam_cfg* hp) {
  std::string why;
  if (!cfg || !arena || !hp || !mt::validate_cfg(*cfg, &why)) return MT_EINVAL;
  if (!mt::adam_cfg_ok(*hp)) return MT_EINVAL;
  const mt::Layout L = mt::compute_layout(*cfg);
  if (bytes < L.total) return MT_EINVAL;
  if (reinterpret_cast<uintptr_t>(arena) % mt::kAlign) return MT_EALIGN;
  mt::adam_arena(L, static_cast<uint8_t*>(arena), *hp);
  return MT_OK;
}

int mt_master_init(const mt_model_cfg* cfg, void* arena, uint64_t bytes) {
  std::string why;
  if (!cfg || !arena) return MT_EINVAL;
  if (!mt::validate_cfg(*cfg, &why)) {
    mt_set_global_error(why);
    return MT_EINVAL;
  }
  if (!(cfg->flags & MT_FLAG_FP32_MASTER)) {
    mt_set_global_error("mt_master_init needs MT_FLAG_FP32_MASTER");
    return MT_EINVAL;
  }
  const mt::Layout L = mt::compute_layout(*cfg);
  if (bytes < L.total) {
    mt_set_global_error("arena shorter than mt_arena_bytes");
    return MT_EINVAL;
  }
  mt::master_init(L, static_cast<uint8_t*>(arena));
  return MT_OK;
}

int mt_host_bandwidth(uint64_t bytes, int32_t reps, double* gbs, int32_t* threads) {
  if (!gbs || bytes < 12 || reps <= 0) return MT_EINVAL;
  *gbs = mt::host_triad_gbs(bytes, reps);
  if (threads) *threads = mt::host_threads();
  return *gbs > 0.0 ? MT_OK : MT_ENOMEM;
}

int mt_get_stats(mt_ctx* c, mt_stats* out) {
  if (!c || !out) return MT_EINVAL;
  *out = c->stats;
  return MT_OK;
}

int mt_get_kernel_stats(mt_ctx* c, int32_t kind, mt_kernel_stats* out) {
  if (!c || !out || kind < 0 || kind >= MT_KIND_COUNT) return MT_EINVAL;
  *out = c->kstats[kind];
  return MT_OK;
}

int mt_read_checkpoint(mt_ctx* c, int32_t layer, float* dst) {
  if (!c || !dst) return set_err(c, MT_EINVAL, "null argument");
  if (layer < 0 || layer > c->L) return set_err(c, MT_EINVAL, "layer out of range");
  if (c->broken) return set_err(c, MT_ESTATE, "context unusable: an earlier step's wait limit expired");
  if (!c->grads_valid) return set_err(c, MT_ESTATE, "no successful mt_train_step");
  const uint64_t bytes = static_cast<uint64_t>(c->T) * c->h * 4;
  if (c->offload) {
    if (layer == c->L) return set_err(c, MT_ESTATE, "the final hidden state is not kept with checkpoint offload");
    std::memcpy(dst, c->host_ckpt + static_cast<uint64_t>(layer) * c->T * c->h, bytes);
    return MT_OK;
  }
  CK(cudaMemcpyAsync(dst, ckpt_slot(c, layer), bytes, cudaMemcpyDeviceToHost, c->st[kStreamCompute]));
  CK(cudaStreamSynchronize(c->st[kStreamCompute]));
  return MT_OK;
}

int mt_capture_input_grad(mt_ctx* c, int32_t layer, float* dst) {
  if (!c) return MT_EINVAL;
  if (layer < 0) {
    c->grad_capture.clear();
    return MT_OK;
  }
  if (layer > c->L || !dst) return set_err(c, MT_EINVAL, "layer out of range or null destination");
  for (auto& cap : c->grad_capture)
    if (cap.first == layer) {
      cap.second = dst;
      return MT_OK;
    }
  if (c->grad_capture.size() >= 8) return set_err(c, MT_EINVAL, "at most 8 captures");
  c->grad_capture.push_back({layer, dst});
  return MT_OK;
}

int mt_set_head_chunk_rows(mt_ctx* c, int32_t rows) {
  if (!c) return MT_EINVAL;
  if (rows < 0 || rows > c->plan.head_rows) return set_err(c, MT_EINVAL, "head chunk rows out of range");
  c->head_rows = rows == 0 ? c->plan.head_rows : rows;
  return MT_OK;
}

int mt_set_kernel_timing(mt_ctx* c, int32_t on) {
  if (!c) return MT_EINVAL;
  c->timing = on != 0;
  return MT_OK;
}

const char* mt_last_error(mt_ctx* c) { return c ? c->err.c_str() : mt_global_error(); }

void mt_destroy(mt_ctx* c) { release(c); }

}  // extern "C"
