// C ABI of the individual layer-template kernels (declared in include/mt_kernels.h).
// Argument checking happens here; the launchers in kernels.h enqueue the work.
#include <atomic>
#include <string>

#include "kernels.h"
#include "mt.h"
#include "mt_kernels.h"
#include "ptx.cuh"
#include "tile_order.cuh"

using mt::bf16;

namespace {
// One thread waits, through the same bounded wait every pipeline kernel uses, for a phase of an
// mbarrier that nothing ever arrives on. No copy or MMA is in flight, so giving up is all it does.
__global__ void bounded_wait_check_kernel(int* err, unsigned long long limit_ns, int* gave_up) {
  __shared__ uint64_t bar;
  mt::mbar_init(&bar, 1);
  mt::fence_mbar_init();
  const bool ok = mt::mbar_wait_limit(&bar, 0, err, mt::kErrTimeoutProbe, limit_ns);
  *gave_up = ok ? 0 : 1;
}
}  // namespace

namespace {
inline cudaStream_t S(void* s) { return reinterpret_cast<cudaStream_t>(s); }
inline int rc(cudaError_t e) {
  if (e == cudaSuccess) return MT_OK;
  if (e == cudaErrorInvalidValue || e == cudaErrorMisalignedAddress) return MT_EINVAL;
  return MT_ECUDA;
}
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
std::atomic<void*> g_gemm_ws{nullptr};  // workspace of the mtk_gemm_* calls (mtk_gemm_use_workspace)
}  // namespace

void mt_set_global_error(const std::string& m);  // message for mt_last_error(NULL)
extern const char* const kRmsBwdAlignMsg;
const char* const kRmsBwdAlignMsg =
    "rmsnorm backward: dy, x, dres, dx and the scratch must be 16-byte aligned, gamma and dx_bf16 8-byte aligned";

extern "C" {

uint64_t mtk_gemm_workspace_bytes(void) { return mt::gemm_workspace_bytes(); }
uint64_t mtk_gemm_workspace_clear_bytes(void) { return mt::kGemmFlagBytes; }

int mtk_gemm_use_workspace(void* ws) {
  if (ws && !aligned16(ws)) return MT_EINVAL;
  g_gemm_ws.store(ws);
  return MT_OK;
}

int mtk_gemm_bf16(const void* A, int64_t lda, int a_mn, const void* B, int64_t ldb, int b_mn, void* C, int64_t ldc,
                  const void* R, int64_t ldr, int M, int N, int K, int epi, int* err_flag, void* stream) {
  if (!A || !B || !C || !err_flag || M <= 0 || N <= 0 || K <= 0) return MT_EINVAL;
  if (epi < MTK_EPI_STORE_BF16 || epi > MTK_EPI_ADD_F32 || (epi == MTK_EPI_ADD_F32 && !R)) return MT_EINVAL;
  if ((a_mn ? lda < M : lda < K) || (b_mn ? ldb < N : ldb < K) || ldc < N) return MT_EINVAL;
  mt::GemmArgs g;
  g.A = static_cast<const bf16*>(A);
  g.lda = lda;
  g.a_mn = a_mn != 0;
  g.B = static_cast<const bf16*>(B);
  g.ldb = ldb;
  g.b_mn = b_mn != 0;
  g.C = C;
  g.ldc = ldc;
  g.R = static_cast<const float*>(R);
  g.ldr = ldr;
  g.M = M;
  g.N = N;
  g.K = K;
  g.epi = epi;
  g.ws = g_gemm_ws.load();
  return rc(mt::gemm(g, err_flag, S(stream)));
}

int mtk_gemm_qkv_rope(const void* a, const void* w, void* qkv, const void* cos_sin, int T, int h, int n_heads,
                      int n_kv_heads, int head_dim, int seq, int* err_flag, void* stream) {
  if (!a || !w || !qkv || !cos_sin || !err_flag || T <= 0 || h <= 0 || n_heads <= 0 || n_kv_heads <= 0 || seq <= 0 ||
      (head_dim != 64 && head_dim != 128))
    return MT_EINVAL;
  const int n = (n_heads + 2 * n_kv_heads) * head_dim;
  mt::GemmArgs g{static_cast<const bf16*>(a), h, false, static_cast<const bf16*>(w), h, false, qkv, n, nullptr, 0,
                 T, n, h, mt::kEpiRopeBf16};
  g.cs = static_cast<const float*>(cos_sin);
  g.rope_cols = (n_heads + n_kv_heads) * head_dim;
  g.hd = head_dim;
  g.seq = seq;
  g.ws = g_gemm_ws.load();
  return rc(mt::gemm(g, err_flag, S(stream)));
}

int mtk_gemm_swiglu(const void* b, const void* wgu, void* act, void* gu, int T, int h, int f, int* err_flag,
                    void* stream) {
  if (!b || !wgu || !act || !err_flag || T <= 0 || h <= 0 || f <= 0 || f % 8) return MT_EINVAL;
  mt::GemmArgs g{static_cast<const bf16*>(b), h, false, static_cast<const bf16*>(wgu), h, false, act, f, nullptr, 0,
                 T, f, h, mt::kEpiSwigluBf16};
  g.C2 = gu;
  g.ldc2 = 2 * static_cast<int64_t>(f);
  g.ws = g_gemm_ws.load();
  return rc(mt::gemm(g, err_flag, S(stream)));
}

int mtk_gemm_swiglu_bwd(const void* dy, const void* wd, const void* gu, void* dgu, int T, int h, int f, int* err_flag,
                        void* stream) {
  if (!dy || !wd || !gu || !dgu || !err_flag || T <= 0 || h <= 0 || f <= 0 || f % 8) return MT_EINVAL;
  mt::GemmArgs g{static_cast<const bf16*>(dy), h, false, static_cast<const bf16*>(wd), f, true, dgu, 2 * f, nullptr,
                 0, T, f, h, mt::kEpiSwigluBwdBf16};
  g.G = static_cast<const bf16*>(gu);
  g.ldg = 2 * static_cast<int64_t>(f);
  g.ws = g_gemm_ws.load();
  return rc(mt::gemm(g, err_flag, S(stream)));
}

int mtk_rmsnorm_fwd(const void* x, const void* gamma, void* y, void* rstd, int T, int h, float eps, void* stream) {
  if (!x || !gamma || !y || !rstd || T <= 0 || h <= 0 || !aligned16(x) || !aligned16(y)) return MT_EINVAL;
  return rc(mt::rmsnorm_fwd(static_cast<const float*>(x), static_cast<const bf16*>(gamma), static_cast<bf16*>(y),
                            static_cast<float*>(rstd), T, h, eps, S(stream)));
}

int mtk_rmsnorm_bwd_parts(int T) { return T > 0 ? mt::rmsnorm_bwd_parts(T) : 0; }

int mtk_rmsnorm_bwd(const void* dy, const void* x, const void* gamma, const void* rstd, const void* dres, void* dx,
                    void* dx_bf16, void* partial, void* dgamma, int T, int h, void* stream) {
  if (!dy || !x || !gamma || !rstd || !dx || !partial || !dgamma || T <= 0 || h <= 0) return MT_EINVAL;
  if (!mt::rmsnorm_bwd_aligned(static_cast<const float*>(dy), static_cast<const float*>(x),
                               static_cast<const bf16*>(gamma), static_cast<const float*>(dres),
                               static_cast<const float*>(dx), static_cast<const bf16*>(dx_bf16),
                               static_cast<const float*>(partial))) {
    mt_set_global_error(kRmsBwdAlignMsg);
    return MT_EINVAL;
  }
  return rc(mt::rmsnorm_bwd(static_cast<const float*>(dy), static_cast<const float*>(x),
                            static_cast<const bf16*>(gamma), static_cast<const float*>(rstd),
                            static_cast<const float*>(dres), static_cast<float*>(dx), static_cast<bf16*>(dx_bf16),
                            static_cast<float*>(partial), static_cast<bf16*>(dgamma), T, h, S(stream)));
}

int mtk_rope(void* qkv, int64_t ld, int T, int seq, int n_heads, int n_kv_heads, int head_dim, const void* cos_sin,
             int inverse, void* stream) {
  if (!qkv || !cos_sin || T <= 0 || seq <= 0 || n_heads <= 0 || n_kv_heads <= 0) return MT_EINVAL;
  if (ld < static_cast<int64_t>(n_heads + n_kv_heads) * head_dim) return MT_EINVAL;
  return rc(mt::rope(static_cast<bf16*>(qkv), ld, T, seq, n_heads, n_kv_heads, head_dim,
                     static_cast<const float*>(cos_sin), inverse != 0, S(stream)));
}

int mtk_swiglu_fwd(const void* gu, void* act, int T, int f, void* stream) {
  if (!gu || !act || T <= 0 || f <= 0) return MT_EINVAL;
  return rc(mt::swiglu_fwd(static_cast<const bf16*>(gu), static_cast<bf16*>(act), T, f, S(stream)));
}

int mtk_swiglu_bwd(const void* gu, const void* dact, void* dgu, int T, int f, void* stream) {
  if (!gu || !dact || !dgu || T <= 0 || f <= 0) return MT_EINVAL;
  return rc(mt::swiglu_bwd(static_cast<const bf16*>(gu), static_cast<const bf16*>(dact), static_cast<bf16*>(dgu), T,
                           f, S(stream)));
}

int mtk_embed_fwd(const void* tok, const void* E, void* x, int T, int h, void* stream) {
  if (!tok || !E || !x || T <= 0 || h <= 0) return MT_EINVAL;
  return rc(mt::embed_fwd(static_cast<const int32_t*>(tok), static_cast<const bf16*>(E), static_cast<float*>(x), T, h,
                          S(stream)));
}

int mtk_embed_bwd(const void* order, const void* offsets, const void* dx, void* dE, int V, int h, void* stream) {
  if (!order || !offsets || !dx || !dE || V <= 0 || h <= 0) return MT_EINVAL;
  return rc(mt::embed_bwd(static_cast<const int32_t*>(order), static_cast<const int32_t*>(offsets),
                          static_cast<const float*>(dx), static_cast<bf16*>(dE), V, h, S(stream)));
}

int mtk_cross_entropy(const void* logits, const void* labels, void* dlogits, void* row_loss, void* loss, int T, int V,
                      void* stream) {
  if (!logits || !labels || !dlogits || !row_loss || !loss || T <= 0 || V <= 0) return MT_EINVAL;
  cudaError_t e = mt::cross_entropy(static_cast<const float*>(logits), static_cast<const int32_t*>(labels),
                                    static_cast<bf16*>(dlogits), static_cast<float*>(row_loss), T, V, S(stream));
  if (e != cudaSuccess) return rc(e);
  return rc(mt::mean_reduce(static_cast<const float*>(row_loss), T, static_cast<float*>(loss), S(stream)));
}

int mtk_attn_fwd(const void* qkv, void* o, void* lse, int B, int s, int nh, int nkv, int head_dim, int* err_flag,
                 void* stream) {
  if (!qkv || !o || !lse || !err_flag || B <= 0 || s <= 0) return MT_EINVAL;
  return rc(mt::attn_fwd(static_cast<const bf16*>(qkv), static_cast<bf16*>(o), static_cast<float*>(lse), B, s, nh, nkv,
                         head_dim, err_flag, S(stream)));
}

int mtk_attn_bwd(const void* qkv, const void* o, const void* lse, const void* dout, void* dqkv, void* delta, int B,
                 int s, int nh, int nkv, int head_dim, int* err_flag, void* stream) {
  if (!qkv || !o || !lse || !dout || !dqkv || !delta || !err_flag || B <= 0 || s <= 0) return MT_EINVAL;
  return rc(mt::attn_bwd(static_cast<const bf16*>(qkv), static_cast<const bf16*>(o), static_cast<const float*>(lse),
                         static_cast<const bf16*>(dout), static_cast<bf16*>(dqkv), static_cast<float*>(delta), nullptr,
                         B, s, nh, nkv, head_dim, err_flag, S(stream)));
}

int mtk_attn_bwd_rope(const void* qkv, const void* o, const void* lse, const void* dout, void* dqkv, void* delta,
                      const void* cos_sin, int B, int s, int nh, int nkv, int head_dim, int* err_flag, void* stream) {
  if (!qkv || !o || !lse || !dout || !dqkv || !delta || !cos_sin || !err_flag || B <= 0 || s <= 0) return MT_EINVAL;
  return rc(mt::attn_bwd(static_cast<const bf16*>(qkv), static_cast<const bf16*>(o), static_cast<const float*>(lse),
                         static_cast<const bf16*>(dout), static_cast<bf16*>(dqkv), static_cast<float*>(delta),
                         static_cast<const float*>(cos_sin), B, s, nh, nkv, head_dim, err_flag, S(stream)));
}

int mtk_bounded_wait_check(int* err_flag, int* gave_up, int64_t limit_ns, void* stream) {
  if (!err_flag || !gave_up || limit_ns < 0 || limit_ns > static_cast<int64_t>(mt::kWaitLimitNs)) return MT_EINVAL;
  bounded_wait_check_kernel<<<1, 1, 0, S(stream)>>>(err_flag, static_cast<unsigned long long>(limit_ns), gave_up);
  return rc(cudaGetLastError());
}

int mtk_attn_block_slot(int lin, int n_tiles, int n_hb, int* rank, int* hb) {
  if (!rank || !hb || n_tiles <= 0 || n_hb <= 0 || lin < 0 ||
      static_cast<int64_t>(lin) >= static_cast<int64_t>(n_tiles) * n_hb)
    return MT_EINVAL;
  const mt::TileSlot s = mt::heavy_first_slot(lin, n_tiles, n_hb);
  *rank = s.rank;
  *hb = s.hb;
  return MT_OK;
}

}  // extern "C"
