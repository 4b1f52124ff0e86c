/*
 * mt_kernels.h — kernel-level C ABI of the layer templates.
 *
 * These entry points launch one kernel (or one fixed kernel sequence) of the
 * stateless layer templates on caller-provided device buffers. They exist so
 * that each kernel can be checked alone against the oracle; mt_train_step()
 * (mt.h) runs the same launchers. The stateless-template idea itself —
 * kernels that bind a layer's weights by pointer as they stream in, with no
 * persistent autograd graph — is from "MegaTrain: Full Precision Training of
 * 100B+ Parameter Large Language Models on a Single GPU" (chatpaper
 * abstract, optimisation 2) and the chestersoft digest (Methodik, "Stateless
 * Layer Templates").
 *
 * Conventions for every function here:
 *  - all pointer arguments are DEVICE pointers, owned by the caller, 16-byte
 *    aligned; matrices are row-major with a row stride in elements that is a
 *    multiple of 8;
 *  - bf16 means IEEE bfloat16 (uint16 storage), f32 IEEE binary32;
 *  - `stream` is a cudaStream_t (NULL = legacy default stream);
 *  - the call only enqueues work; it returns MT_OK (0), MT_EINVAL for bad
 *    sizes or alignment (nothing enqueued), or MT_ECUDA for a launch error;
 *  - `err_flag` (device int, may be NULL where unused) receives a nonzero
 *    code if a kernel's bounded internal wait gave up; it is never cleared
 *    by the library.
 */
#ifndef MT_KERNELS_H
#define MT_KERNELS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Epilogues of mtk_gemm_bf16. */
#define MTK_EPI_STORE_BF16 0 /* C (bf16) = A*B                          */
#define MTK_EPI_STORE_F32 1  /* C (f32)  = A*B                          */
#define MTK_EPI_ADD_F32 2    /* C (f32)  = R (f32) + A*B, R may equal C */

/*
 * C[M,N] = A * B on the tcgen05 tensor cores, bf16 operands, f32 accumulation.
 *  a_mn = 0: A is stored [M][K] (row stride lda);  a_mn = 1: A is stored [K][M].
 *  b_mn = 0: B is stored [N][K] (C = A * B^T);     b_mn = 1: B is stored [K][N].
 * With a_mn = b_mn = 0 this is the forward projection y = x W^T; (0, 1) is the
 * data gradient dx = dy W; (1, 1) is the weight gradient dW = dy^T x.
 * M, N, K > 0. Deterministic: fixed K order, no atomics. When a workspace is
 * set (mtk_gemm_use_workspace), the tiles of the last, partial wave are split
 * over K between CTAs and their fp32 partial sums added in a fixed order: the
 * result then differs from the unsplit one in the order of the K sum only, and
 * is the same from run to run.
 */
int mtk_gemm_bf16(const void* A, int64_t lda, int a_mn, const void* B, int64_t ldb, int b_mn, void* C,
                  int64_t ldc, const void* R, int64_t ldr, int M, int N, int K, int epi, int* err_flag,
                  void* stream);

/*
 * Workspace of the mtk_gemm_* calls (this stream-ordered split is a scheduling
 * device of this library; the pages have no counterpart). ws: device memory of
 * mtk_gemm_workspace_bytes() bytes, 16-byte aligned, owned by the caller, whose
 * first mtk_gemm_workspace_clear_bytes() bytes are zero before its first use
 * (the calls leave them in a state later calls accept); NULL (the default)
 * turns the split off. The setting is process-wide and kept until changed.
 * Calls that use the same workspace must not overlap on the GPU (use one
 * stream). Returns MT_EINVAL for a misaligned pointer.
 */
uint64_t mtk_gemm_workspace_bytes(void);
uint64_t mtk_gemm_workspace_clear_bytes(void);
int mtk_gemm_use_workspace(void* ws);

/* RMSNorm forward on x f32 [T,h]: y bf16 = x*rstd*gamma, rstd f32 [T] = 1/sqrt(mean(x^2)+eps).
 * h a multiple of 8; x 16-byte aligned, gamma and y 8-byte aligned (else MT_EINVAL). */
int mtk_rmsnorm_fwd(const void* x, const void* gamma, void* y, void* rstd, int T, int h, float eps, void* stream);

/* Number of rows of the f32 [parts][h] scratch `partial` that mtk_rmsnorm_bwd needs for T rows. */
int mtk_rmsnorm_bwd_parts(int T);

/*
 * RMSNorm backward: dx f32 = dres + rstd*(dy*gamma - xhat*mean(dy*gamma*xhat)), xhat = x*rstd,
 * dy f32 [T,h], dres f32 [T,h] or NULL; dx_bf16 (optional) receives dx rounded to bf16;
 * dgamma bf16 [h] = sum_t dy*xhat, reduced in a fixed order through `partial`.
 * h a multiple of 8. dy, x, dres, dx and partial must be 16-byte aligned, gamma and dx_bf16
 * 8-byte aligned: a row slice at an odd offset is rejected with MT_EINVAL before anything is
 * launched (message in mt_last_error(NULL)).
 */
int mtk_rmsnorm_bwd(const void* dy, const void* x, const void* gamma, const void* rstd, const void* dres, void* dx,
                    void* dx_bf16, void* partial, void* dgamma, int T, int h, void* stream);

/*
 * The same RMSNorm backward with no scratch argument: for callers that cannot allocate
 * device memory where they need this kernel (code under a memory manager that owns the
 * whole device, or paths where the implicit device synchronisation of cudaMalloc/cudaFree
 * is not allowed). The paper has no counterpart of this entry point. It allocates nothing:
 * its scratch is a fixed 9.5 MiB array (304 * 8192 floats) inside the library, held by
 * every GPU that loads it until the process exits. Sizes with min(T, 304) * h above that
 * are rejected with MT_EINVAL (message in mt_last_error(NULL)), and so are pointers that break
 * mtk_rmsnorm_bwd's alignment rule. The first call on a device
 * looks up the array's device address (cudaGetSymbolAddress) with that device current;
 * make that first call before any stream capture. All calls share the array: calls that
 * overlap on the GPU race on it and must be serialised by the caller. Nothing in it needs
 * to start at zero (every element read is written earlier by the same call).
 */
int mtk_rmsnorm_bwd_noalloc(const void* dy, const void* x, const void* gamma, const void* rstd, const void* dres,
                            void* dx, void* dx_bf16, void* dgamma, int T, int h, void* stream);

/*
 * Rotate-half RoPE, in place, on the q and k column ranges of qkv bf16 [T, ld]
 * (columns [0, nh*hd) are q, the next nkv*hd are k). Token t has position t % seq.
 * cos_sin: f32 [seq][hd/2][2]. inverse = 1 applies the transpose (the backward pass).
 */
int mtk_rope(void* qkv, int64_t ld, int T, int seq, int n_heads, int n_kv_heads, int head_dim, const void* cos_sin,
             int inverse, void* stream);

/* SwiGLU on gu bf16 [T, 2f] = [g | u]: act bf16 [T,f] = silu(g)*u; backward dgu bf16 [T,2f]. */
int mtk_swiglu_fwd(const void* gu, void* act, int T, int f, void* stream);
int mtk_swiglu_bwd(const void* gu, const void* dact, void* dgu, int T, int f, void* stream);

/*
 * The projections with their pointwise step fused into the GEMM epilogue (what the layer
 * template runs; the unfused kernels above remain for checking each step alone). The fused
 * step works on the f32 accumulator, so results can differ from GEMM-then-kernel by the one
 * bf16 rounding of the intermediate. Deterministic like mtk_gemm_bf16.
 *
 * mtk_gemm_qkv_rope: qkv bf16 [T, (nh+2*nkv)*hd] = a W^T with the q and k heads rotated as
 *   mtk_rope(inverse = 0) does (token t at position t % seq, cos_sin f32 [seq][hd/2][2]);
 *   a bf16 [T,h], w bf16 [(nh+2*nkv)*hd, h]. head_dim 64 or 128.
 * mtk_gemm_swiglu: act bf16 [T,f] = silu(g)*u with g = bf16(b Wg^T), u = bf16(b Wu^T);
 *   b bf16 [T,h], wgu bf16 [2f, h] = [Wg; Wu]; gu (NULL or bf16 [T,2f]) receives [g | u].
 *   f a multiple of 8.
 * mtk_gemm_swiglu_bwd: dact = dy Wd (dy bf16 [T,h], wd bf16 [h,f]) and, from gu bf16 [T,2f] =
 *   [g | u], dgu bf16 [T,2f] = [dact*u*s*(1+g*(1-s)) | dact*g*s], s = sigmoid(g).
 *   f a multiple of 8.
 */
int mtk_gemm_qkv_rope(const void* a, const void* w, void* qkv, const void* cos_sin, int T, int h, int n_heads,
                      int n_kv_heads, int head_dim, int seq, int* err_flag, void* stream);
int mtk_gemm_swiglu(const void* b, const void* wgu, void* act, void* gu, int T, int h, int f, int* err_flag,
                    void* stream);
int mtk_gemm_swiglu_bwd(const void* dy, const void* wd, const void* gu, void* dgu, int T, int h, int f, int* err_flag,
                        void* stream);

/* Embedding gather x f32 [T,h] = E bf16 [V,h] rows tok[t]. */
int mtk_embed_fwd(const void* tok, const void* E, void* x, int T, int h, void* stream);
/* dE bf16 [V,h]: row v = sum of dx f32 rows order[offsets[v]..offsets[v+1]) in that order. */
int mtk_embed_bwd(const void* order, const void* offsets, const void* dx, void* dE, int V, int h, void* stream);

/*
 * Cross-entropy over logits f32 [T,V] with labels int32 [T]:
 * row_loss f32 [T] = logsumexp(z_t) - z_t[label_t]; dlogits bf16 [T,V] = (softmax(z_t) - onehot)/T;
 * loss f32 [1] = mean of row_loss (fixed-order reduction).
 */
int mtk_cross_entropy(const void* logits, const void* labels, void* dlogits, void* row_loss, void* loss, int T, int V,
                      void* stream);

/*
 * Causal grouped-query flash attention on qkv bf16 [B*s, (nh+2*nkv)*hd] (q | k | v), on the
 * tcgen05 tensor cores. o bf16 [B*s, nh*hd]; lse f32 [B, nh, s] = log2 of the softmax
 * denominator of the scores scaled by log2(e)/sqrt(hd), plus the max it was taken against.
 * head_dim is 64 or 128. err_flag: device int, required (bounded internal waits).
 */
int mtk_attn_fwd(const void* qkv, void* o, void* lse, int B, int s, int nh, int nkv, int head_dim, int* err_flag,
                 void* stream);
/* Backward on the tcgen05 tensor cores, deterministic (KV-outer dK/dV, Q-outer dQ, no atomics):
 * dqkv bf16 (layout of qkv) from dout bf16 [B*s, nh*hd]. delta: f32 scratch of
 * B * nh * s128 * 2 floats, s128 = s rounded up to a multiple of 128, 16-byte aligned; it receives
 * (lse2, rowsum(dO * O)) per query row. err_flag: device int, required. */
int mtk_attn_bwd(const void* qkv, const void* o, const void* lse, const void* dout, void* dqkv, void* delta, int B,
                 int s, int nh, int nkv, int head_dim, int* err_flag, void* stream);
/* The same backward with the RoPE backward fused into its output: dq and dk are written with the
 * transpose rotation of mtk_rope(inverse = 1) applied (cos_sin f32 [s][hd/2][2], position = row
 * index within the sequence), which is what the layer template needs when RoPE was applied to q
 * and k after the QKV projection. dv is unchanged. */
int mtk_attn_bwd_rope(const void* qkv, const void* o, const void* lse, const void* dout, void* dqkv, void* delta,
                      const void* cos_sin, int B, int s, int nh, int nkv, int head_dim, int* err_flag, void* stream);

/* Block order of the causal attention grids (host-only, pure; no GPU needed). The forward, dQ
 * and dK/dV grids are one-dimensional with n_tiles * n_hb blocks (n_tiles 128-row tiles per
 * sequence; n_hb = heads * batch, KV heads for dK/dV). Block `lin` works on tile rank *rank
 * (0 = the heaviest tile of its head: the last query tile, or the first key tile) of head pair
 * *hb = head + heads * batch. Blocks take ranks heaviest first over groups of 16 head pairs.
 * Returns MT_EINVAL unless 0 <= lin < n_tiles * n_hb and both pointers are set. */
int mtk_attn_block_slot(int lin, int n_tiles, int n_hb, int* rank, int* hb);

/*
 * Self-check of the kernels' bounded waits: one thread waits, through the same wait routine the
 * GEMM and attention pipelines use, on an mbarrier phase that never completes. After limit_ns
 * (0 .. 4e9, the pipelines' own limit) it gives up, stores code 6 in *err_flag (unless a code is
 * already there), writes *gave_up = 1 and returns; no copy or MMA is in flight. This is how a
 * stalled pipeline ends instead of hanging the GPU: the host reads the flag after the step
 * (mt_train_step returns MT_EKERNEL) and the context stays usable. err_flag and gave_up are
 * device ints; the call only enqueues.
 */
int mtk_bounded_wait_check(int* err_flag, int* gave_up, int64_t limit_ns, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MT_KERNELS_H */
