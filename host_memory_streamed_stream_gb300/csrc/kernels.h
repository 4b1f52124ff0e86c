// Internal launchers of the layer-template kernels. All pointers are device pointers;
// every launcher enqueues on `stream` and returns a cudaError_t (cudaSuccess or the
// launch error). Matrices are row-major with explicit row strides in elements.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace mt {

using bf16 = __nv_bfloat16;

// ------------------------------------------------------------------ GEMM
// C[M,N] = A[M,K] * B[K,N] with bf16 operands and fp32 accumulation on tcgen05.
//   a_mn = false: A stored as [M rows][K] (K contiguous, row stride lda)
//   a_mn = true : A stored as [K rows][M] (M contiguous, row stride lda)
//   b_mn = false: B stored as [N rows][K] (K contiguous), i.e. C = A * B_stored^T
//   b_mn = true : B stored as [K rows][N] (N contiguous)
// Strides are multiples of 8 elements and base pointers 16-byte aligned.
enum GemmEpilogue : int {
  kEpiStoreBf16 = 0,  // C (bf16)  = acc
  kEpiStoreF32 = 1,   // C (fp32)  = acc
  kEpiAddF32 = 2,     // C (fp32)  = R (fp32) + acc   (R may alias C)
  // QKV projection with RoPE: C (bf16) = acc, the q and k heads (columns < rope_cols, heads of
  // hd columns) rotated by the rotate-half rule at position (row % seq) with table cs
  // (fp32 [seq][hd/2][2] = cos, sin). N is a multiple of hd; hd is 64 or 128.
  kEpiRopeBf16 = 3,
  // Gate-up projection with SwiGLU (forward layout only): N = f, B = [gate rows; up rows]
  // stored [2f][K]; C (bf16 [M][f]) = silu(g) * u with g, u the bf16-rounded gate and up
  // projections; if C2 is set it receives [g | u] (bf16 [M][2f], row stride ldc2).
  kEpiSwigluBf16 = 4,
  // Down-projection data gradient with the SwiGLU backward: acc = dact [M][N = f]; G = [g | u]
  // (bf16 [M][2f], stride ldg); C (bf16 [M][2f]) = [dact*u*silu'(g) | dact*silu(g)].
  kEpiSwigluBwdBf16 = 5,
};
struct GemmArgs {
  const bf16* A;
  int64_t lda;
  bool a_mn;
  const bf16* B;
  int64_t ldb;
  bool b_mn;
  void* C;
  int64_t ldc;
  const float* R;
  int64_t ldr;
  int M, N, K;
  int epi;
  void* C2 = nullptr;        // kEpiSwigluBf16: optional [g | u] output
  int64_t ldc2 = 0;
  const bf16* G = nullptr;   // kEpiSwigluBwdBf16: [g | u]
  int64_t ldg = 0;
  const float* cs = nullptr; // kEpiRopeBf16: rotation table
  int rope_cols = 0, hd = 0, seq = 0;
  // optional workspace of gemm_workspace_bytes(): the last wave's tiles are split over K
  // (per-CTA fp32 partial slots and flags). Its first kSplitFlagBytes must be zero before its
  // first use; launches that share it must not overlap on the GPU.
  void* ws = nullptr;
};
cudaError_t gemm(const GemmArgs& g, int* err_flag, cudaStream_t stream);
// Page-locked host memory (host_alloc.cpp): huge-page backed and registered where possible,
// else cudaHostAlloc; zero-filled when huge-page backed. host_free releases either kind.
cudaError_t host_alloc(uint64_t bytes, void** out);
cudaError_t host_free(void* p);
struct HostAllocInfo {  // what host_alloc found and did (huge-page backed allocations only)
  uint64_t chunk_bytes;
  int32_t chunks, spare, slow_found, replaced;
  double median_gbs, min_gbs;
};
bool host_alloc_info(const void* p, HostAllocInfo* out);
int gemm_num_sms();
uint64_t gemm_workspace_bytes();
constexpr uint64_t kGemmFlagBytes = 256 * 8 * 4;  // leading bytes of the workspace to clear once

// ------------------------------------------------------------------ pointwise
// RMSNorm forward: y = x * rstd * gamma, rstd = 1/sqrt(mean(x^2) + eps); x fp32 [T,h].
cudaError_t rmsnorm_fwd(const float* x, const bf16* gamma, bf16* y, float* rstd, int T, int h, float eps,
                        cudaStream_t s);
// RMSNorm backward: dx = dres + rstd*(dy*gamma - xhat*mean(dy*gamma*xhat)), xhat = x*rstd.
// dy fp32 [T,h]; dres fp32 or null; writes dx fp32 and (if non-null) its bf16 copy;
// dgamma (bf16 [h]) via a fixed-order two-stage reduction through `partial` (fp32 [parts][h]).
int rmsnorm_bwd_parts(int T);
// The pointer alignment rmsnorm_bwd needs (null pointers pass): dy, x, dres, dx, partial on 16
// bytes, gamma and dx_bf16 on 8. rmsnorm_bwd returns cudaErrorInvalidValue without launching
// otherwise.
bool rmsnorm_bwd_aligned(const float* dy, const float* x, const bf16* gamma, const float* dres, const float* dx,
                         const bf16* dx_bf16, const float* partial);
cudaError_t rmsnorm_bwd(const float* dy, const float* x, const bf16* gamma, const float* rstd, const float* dres,
                        float* dx, bf16* dx_bf16, float* partial, bf16* dgamma, int T, int h, cudaStream_t s);
// Rotate-half RoPE in place on the q and k column ranges of qkv [T, ld] (bf16);
// inverse = true applies the transpose (backward). cs: fp32 [seq][hd/2][2] (cos, sin).
cudaError_t rope(bf16* qkv, int64_t ld, int T, int seq, int n_heads, int n_kv_heads, int hd, const float* cs,
                 bool inverse, cudaStream_t s);
// SwiGLU: act = silu(g) * u with gu [T, 2f] = [g | u]; backward writes dgu [T, 2f].
cudaError_t swiglu_fwd(const bf16* gu, bf16* act, int T, int f, cudaStream_t s);
cudaError_t swiglu_bwd(const bf16* gu, const bf16* dact, bf16* dgu, int T, int f, cudaStream_t s);
// Embedding gather x[t] = E[tok[t]] (fp32 out) and ordered scatter-add of dx into dE (bf16):
// dE[v] = sum over positions order[offsets[v] .. offsets[v+1]) of dx[pos], positions ascending.
cudaError_t embed_fwd(const int32_t* tok, const bf16* E, float* x, int T, int h, cudaStream_t s);
cudaError_t embed_bwd(const int32_t* order, const int32_t* offsets, const float* dx, bf16* dE, int V, int h,
                      cudaStream_t s);
// The same for the listed rows only (rows[0 .. n_rows)); dE may be a host-mapped pointer.
cudaError_t embed_bwd_rows(const int32_t* order, const int32_t* offsets, const int32_t* rows, int n_rows,
                           const float* dx, bf16* dE, int h, cudaStream_t s);
// Cross-entropy on fp32 logits [T, V]: per-row loss lse - z[label] into row_loss, and
// dlogits = (softmax - onehot) / n (bf16), n = mean_over if positive (the whole batch's token
// count when these T rows are one chunk of it), else T. Then loss = mean(row_loss) in fixed order.
cudaError_t cross_entropy(const float* logits, const int32_t* labels, bf16* dlogits, float* row_loss, int T, int V,
                          cudaStream_t s, int mean_over = 0);
cudaError_t mean_reduce(const float* v, int n, float* out, cudaStream_t s);
cudaError_t cast_f32_bf16(const float* x, bf16* y, int64_t n, cudaStream_t s);

// ------------------------------------------------------------------ attention
// Causal grouped-query flash attention over qkv [B*s, (nh + 2 nkv) hd] (q | k | v columns,
// RoPE already applied). o bf16 [B*s, nh*hd]; lse fp32 [B, nh, s] in base-2 units of the
// scaled scores (log2 of the softmax denominator plus the row max).
// tcgen05 kernel; err receives a nonzero code if a bounded internal wait gives up.
cudaError_t attn_fwd(const bf16* qkv, bf16* o, float* lse, int B, int s, int nh, int nkv, int hd, int* err,
                     cudaStream_t st);
// Backward: dqkv (same layout as qkv) from do [B*s, nh*hd]; delta fp32 scratch of
// B*nh*s128*2 floats (s128 = s rounded up to 128). With rope_cs (the forward's table, fp32
// [s][hd/2][2]) dq and dk leave with the transpose RoPE rotation applied.
cudaError_t attn_bwd(const bf16* qkv, const bf16* o, const float* lse, const bf16* dout, bf16* dqkv, float* delta,
                     const float* rope_cs, int B, int s, int nh, int nkv, int hd, int* err, cudaStream_t st);

}  // namespace mt
