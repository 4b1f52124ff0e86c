/*
 * mt.h — C ABI of the layer-streamed training step.
 *
 * The method: "MegaTrain: Full Precision Training of 100B+ Parameter Large
 * Language Models on a Single GPU" (Yuan, Sun, Sun, Ye). Parameters,
 * gradients and Adam states live in host memory; the GPU is a transient
 * per-layer compute engine that receives one layer's weights, runs its
 * forward and backward passes, and sends its gradients back
 * (chatpaper abstract; ecosistemastartup article, "Innovaciones técnicas
 * clave", 1). A double-buffered pipeline on three CUDA streams overlaps the
 * parameter prefetch of layer i+1, the computation of layer i, and the
 * gradient offload (chestersoft digest, Methodik, "Pipelined Double-Buffered
 * Execution Engine"). Each layer's state is one contiguous 4 KB-aligned block
 * of bf16 weights, bf16 gradients and fp32 Adam moments (Methodik,
 * "Layer-Contiguous Tiling"), and the Adam step runs on the host (same
 * passage).
 *
 * Model: decoder-only transformer, RMSNorm, rotate-half RoPE, causal
 * grouped-query attention, SwiGLU FFN, untied embedding and LM head, no
 * biases, mean token cross-entropy.
 *
 * Host arena layout (one block after another, blocks 4096-aligned):
 *   block 0             E: emb [vocab][hidden]
 *   blocks 1..n_layers  decoder layers: attn_norm [h], wq [nh*hd][h],
 *                       wk [nkv*hd][h], wv [nkv*hd][h], wo [h][nh*hd],
 *                       ffn_norm [h], wg [ffn][h], wu [ffn][h], wd [h][ffn]
 *   block n_layers+1    H: final_norm [h], w_head [vocab][h]
 * Inside a block: sections W (bf16), G (bf16), M (fp32), V (fp32), in that
 * order; each section holds the block's tensors in the order above; every
 * section and every tensor starts on a 4096-byte boundary. Matrices are
 * row-major [out][in]. Padding bytes are zero and stay zero.
 *
 * Threading: a context is used by one host thread at a time.
 * Errors: every int-returning call returns MT_OK (0) or a negative MT_E*
 * code; mt_last_error() gives a message for the most recent failure.
 */
#ifndef MT_H
#define MT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MT_OK 0
#define MT_EINVAL (-1)   /* bad argument (sizes, ranges, null pointers); nothing changed */
#define MT_ENOMEM (-2)   /* device or pinned host allocation failed */
#define MT_EALIGN (-3)   /* arena base not 4096-aligned */
#define MT_ESTATE (-4)   /* call out of order (no arena bound, gradients invalid, ...) */
#define MT_ECUDA (-5)    /* a CUDA runtime call or kernel launch failed */
#define MT_ETIMEOUT (-6) /* a bounded wait on the GPU expired; the step did not complete */
#define MT_EKERNEL (-7)  /* a kernel's internal bounded wait gave up (device error flag set) */

/* Configuration flags. */
#define MT_FLAG_RESIDENT 1u      /* all blocks resident in HBM for the step, no streaming (same kernels) */
#define MT_FLAG_OFFLOAD_CKPT 2u  /* layer-boundary activation checkpoints kept in pinned host memory */
#define MT_FLAG_SINGLE_BUFFER 4u /* one device layer buffer: copy, then compute (double-buffering ablation) */
#define MT_FLAG_KERNEL_TIMING 8u /* time every kernel launch with CUDA events (mt_get_kernel_stats) */
#define MT_FLAG_FP32_MASTER 16u  /* each block also holds an fp32 master copy P of its weights (section
                                    MT_SEC_P, 16 B/param in all); Adam updates P in fp32 and writes W as
                                    bf16(P), so updates below half a bf16 step accumulate instead of
                                    being rounded away. The streamed sections and the kernels are the same. */
#define MT_FLAG_DENSE_EMBED 32u  /* copy the embedding block's W and G sections whole, as for every other
                                    block, instead of reading and writing the batch's rows through the
                                    mapped arena */

typedef struct {
  int32_t n_layers;   /* decoder layers, >= 1 */
  int32_t hidden;     /* h, multiple of 64 */
  int32_t n_heads;    /* query heads; head_dim = hidden / n_heads must be 64 or 128 */
  int32_t n_kv_heads; /* key/value heads, divides n_heads */
  int32_t ffn;        /* SwiGLU inner width, multiple of 8 */
  int32_t vocab;      /* multiple of 8 */
  int32_t seq;        /* sequence length, >= 1 */
  int32_t batch;      /* sequences per step, >= 1 */
  float rms_eps;      /* RMSNorm epsilon (1e-5) */
  float rope_theta;   /* RoPE base (10000) */
  uint32_t flags;     /* MT_FLAG_* */
} mt_model_cfg;

/* Indices of sections and tensors for mt_tensor_offset(). */
#define MT_SEC_W 0
#define MT_SEC_G 1
#define MT_SEC_M 2
#define MT_SEC_V 3
#define MT_SEC_P 4 /* fp32 master weights; present only with MT_FLAG_FP32_MASTER */
#define MT_T_ATTN_NORM 0
#define MT_T_WQ 1
#define MT_T_WK 2
#define MT_T_WV 3
#define MT_T_WO 4
#define MT_T_FFN_NORM 5
#define MT_T_WG 6
#define MT_T_WU 7
#define MT_T_WD 8
#define MT_T_EMB 0        /* in block 0 */
#define MT_T_FINAL_NORM 0 /* in block n_layers + 1 */
#define MT_T_W_HEAD 1     /* in block n_layers + 1 */

/* ---------------------------------------------------------------- layout (host only, pure) */
/* The packed-block layout in one call (chestersoft digest, Methodik, "Layer-Contiguous Tiling":
 * one contiguous, 4 KB-aligned block per layer holding its bf16 weights, bf16 gradients and fp32
 * Adam moments; chatpaper abstract: parameters and optimizer states stored in host memory).
 * Per block: its byte range, the byte range of each section and the absolute byte offset and
 * shape of each tensor in each section (offsets from the arena base; all multiples of 4096). */
#define MT_MAX_SECTIONS 5
#define MT_MAX_TENSORS 9
typedef struct {
  uint64_t offset;                                          /* block start */
  uint64_t bytes;                                           /* block size (sections back to back) */
  int32_t n_tensors;                                        /* 1 (E), 9 (decoder layer) or 2 (H) */
  int32_t n_sections;                                       /* 4, or 5 with MT_FLAG_FP32_MASTER */
  uint64_t section_offset[MT_MAX_SECTIONS];                 /* W, G, M, V[, P]; unused entries 0 */
  uint64_t section_bytes[MT_MAX_SECTIONS];
  uint64_t tensor_offset[MT_MAX_SECTIONS][MT_MAX_TENSORS];  /* [section][tensor]; unused entries 0 */
  int64_t rows[MT_MAX_TENSORS];                             /* tensor shape [rows][cols], cols = 1 */
  int64_t cols[MT_MAX_TENSORS];                             /*   for a gain vector */
} mt_block_layout;
typedef struct {
  uint64_t total_bytes;     /* out: arena bytes (a multiple of 4096) */
  uint64_t max_w_section;   /* out: largest W section = size of one device layer buffer */
  int32_t n_blocks;         /* out: n_layers + 2 (E, the decoder layers, H) */
  int32_t n_sections;       /* out: 4, or 5 with MT_FLAG_FP32_MASTER */
  int32_t capacity;         /* in: entries the caller's `blocks` array holds (0: counts only) */
  mt_block_layout* blocks;  /* in: caller-owned array of `capacity` entries, or NULL; on success
                               entries [0, min(capacity, n_blocks)) are filled */
} mt_layout;
/* Fill *out for cfg. Pure host arithmetic (no GPU, no allocation). MT_EINVAL on a NULL
 * argument, an invalid cfg or capacity < 0 (nothing written then). A capacity smaller than
 * n_blocks is not an error: the counts are set and only the first `capacity` blocks filled,
 * so a caller may query n_blocks first and call again with an array of that size. */
int mt_arena_layout(const mt_model_cfg* cfg, mt_layout* out);

/* Total arena bytes for cfg (a multiple of 4096). */
int mt_arena_bytes(const mt_model_cfg* cfg, uint64_t* bytes);
/* Number of blocks (n_layers + 2) and tensors in block `block` (1, 9 or 2). */
int mt_block_count(const mt_model_cfg* cfg, int32_t* n_blocks);
int mt_tensor_count(const mt_model_cfg* cfg, int32_t block, int32_t* n_tensors);
/* Byte offset of block `block` from the arena base, and its size. */
int mt_block_offset(const mt_model_cfg* cfg, int32_t block, uint64_t* offset, uint64_t* bytes);
/* Byte offset of tensor `tensor` of section `section` of block `block` from the arena base,
 * its shape (rows, cols; cols = 1 for a gain vector) and element size (2 or 4 bytes). */
int mt_tensor_offset(const mt_model_cfg* cfg, int32_t block, int32_t section, int32_t tensor, uint64_t* offset,
                     int64_t* rows, int64_t* cols, int32_t* elem_bytes);

/* ---------------------------------------------------------------- pinned host memory */
/* Page-locked host allocation usable as an arena (4096-aligned). Caller frees with mt_host_free.
 * (chestersoft digest, Methodik, "Layer-Contiguous Tiling": blocks leave host memory as single
 * DMA bursts, which page-locked memory allows.) Where the kernel offers transparent huge
 * pages, the memory is an anonymous mapping of huge pages (aligned to their size, zero-filled)
 * registered with CUDA: the call faults the pages in together with spare ones (6 % more, at
 * least 8, released before it returns), times a host-to-device copy of each huge page on the
 * current device (using one huge page of device memory for the duration of the call) and, in
 * up to three rounds, moves spare pages that copy at full rate over pages that copy below
 * 0.6 x the median; memory from cudaHostAlloc otherwise. Needs a CUDA device; MT_ECUDA if
 * neither way works. */
int mt_host_alloc(uint64_t bytes, void** out);
int mt_host_free(void* p);

/* What mt_host_alloc found for a huge-page backed allocation (a diagnostic; the pages' design
 * has no counterpart). */
typedef struct {
  uint64_t chunk_bytes; /* huge-page size */
  int32_t chunks;       /* huge pages in the allocation */
  int32_t spare;        /* spare huge pages faulted in to stand in for slow ones */
  int32_t slow_found;   /* pages whose first host-to-device copy ran below 0.6 x the median */
  int32_t replaced;     /* pages swapped for spare pages that copied at full rate (all rounds) */
  double median_gbs;    /* host-to-device GB/s over the pages, after the last round */
  double min_gbs;       /* the slowest page's */
} mt_host_alloc_info;
/* MT_EINVAL if p is not the start of a huge-page backed allocation from mt_host_alloc (for
 * example memory from cudaHostAlloc, or no probe could run). */
int mt_host_alloc_query(const void* p, mt_host_alloc_info* out);

/* ---------------------------------------------------------------- context */
typedef struct mt_ctx mt_ctx;

/* Optional device resources supplied by the caller (for example PyTorch allocations).
 * workspace: device memory of at least mt_workspace_bytes() bytes, 256-aligned, owned by the
 * caller and kept alive until mt_destroy; NULL makes the library allocate its own.
 * streams: cudaStream_t handles for host-to-device copies, compute and device-to-host copies;
 * a NULL entry makes the library create that stream. */
typedef struct {
  void* workspace;
  uint64_t workspace_bytes;
  void* streams[3];
} mt_device_resources;

/* Device bytes a context for cfg needs (layer buffers, activations, checkpoints). Two W and two
 * G layer buffers, per the double-buffered engine (chestersoft digest, Methodik, "Pipelined
 * Double-Buffered Execution Engine"). */
int mt_workspace_bytes(const mt_model_cfg* cfg, uint64_t* bytes);

/* Validate cfg, set up device buffers, streams, events and the RoPE table on the current device.
 * res may be NULL. On failure *out is NULL and nothing is leaked. The three streams are the
 * digest's prefetch / compute / offload streams (chestersoft digest, Methodik, "Pipelined
 * Double-Buffered Execution Engine"). */
int mt_create(const mt_model_cfg* cfg, const mt_device_resources* res, mt_ctx** out);

/* Bind the caller-owned host arena (mt_arena_bytes() bytes, 4096-aligned). Memory not already
 * page-locked is registered with cudaHostRegister for the context's lifetime. The arena is
 * never freed by the library. Returns MT_EALIGN / MT_EINVAL on a bad base or size.
 * (chatpaper abstract: parameters and optimizer states stay in host memory.) */
int mt_bind_host_arena(mt_ctx* ctx, void* base, uint64_t bytes);

/* One training step: tokens and labels are host int32 arrays of batch*seq ids in [0, vocab)
 * (token t = b*seq + position). Streams every block's W section in, runs forward and
 * backward, and writes every gradient (overwriting) into the G sections of the arena.
 * Returns after the step has finished on the GPU, with the mean cross-entropy in *loss.
 * Ids out of range: MT_EINVAL before any work. A failure after work started leaves the G
 * sections invalid (mt_adam_step then returns MT_ESTATE until a step succeeds). MT_ETIMEOUT
 * (the step did not finish within the host's one-hour wait limit) leaves the context unusable:
 * work may still be in flight, so every later call on it returns MT_ESTATE without waiting,
 * and mt_destroy then frees only host-side bookkeeping (it does not wait for the device).
 * (chatpaper abstract: "for each layer, stream parameters in and compute gradients out";
 * chestersoft digest, Methodik, "Pipelined Double-Buffered Execution Engine".) */
int mt_train_step(mt_ctx* ctx, const int32_t* tokens, const int32_t* labels, float* loss);

/* Copy the layer-boundary activation x_l of the last successful step to host memory
 * (the checkpoints of the stateless templates: chestersoft digest, Methodik, "Stateless Layer
 * Templates"):
 * fp32 [batch*seq][hidden], l = 0 the embedding output (input of layer 0), l = n_layers the
 * final hidden state (input of the final norm). These are the checkpoints the backward pass
 * recomputes from. With MT_FLAG_OFFLOAD_CKPT, l = n_layers is not kept (MT_ESTATE).
 * Valid until the next mt_train_step. Blocks until the copy has finished. */
int mt_read_checkpoint(mt_ctx* ctx, int32_t layer, float* dst);

/* Arm a copy of dL/dx_layer, the loss gradient with respect to the layer-boundary activation
 * x_layer (fp32 [batch*seq][hidden]; layer 0 .. n_layers, the same indexing as
 * mt_read_checkpoint), into dst during every later step, as soon as the backward pass has
 * produced it. dst is a host buffer of batch*seq*hidden floats (page-locked memory, e.g. from
 * mt_host_alloc, keeps the copy asynchronous), owned by the caller and valid while armed; it
 * holds the value once the step returns. Up to 8 layers; arming a layer again replaces its
 * destination; layer < 0 disarms all. Together with the checkpoints this lets a checker run one
 * layer's forward and backward on its own (teacher forcing): the input x_layer and the upstream
 * gradient dL/dx_{layer+1} both come from the step. MT_EINVAL for a layer above n_layers or a
 * NULL dst. */
int mt_capture_input_grad(mt_ctx* ctx, int32_t layer, float* dst);

/* The LM head and the cross-entropy run over chunks of token rows, so that the fp32 logits of a
 * long sequence are never held whole: by default the fewest equal chunks (rounded up to 128
 * rows) whose logits take at most 4 GiB, i.e. one chunk whenever batch*seq*vocab*4 <= 4 GiB.
 * Per chunk: logits (fp32), the cross-entropy rows and dlogits = (softmax - onehot)/(batch*seq),
 * the LM-head weight gradient's share and the chunk's gradient rows. With several chunks the
 * weight gradient is summed in fp32 chunk after chunk and rounded once to bf16. This call sets a
 * smaller chunk for later steps (1 .. the default; 0 restores the default), e.g. to exercise the
 * chunked path on a small model. MT_EINVAL outside that range. */
int mt_set_head_chunk_rows(mt_ctx* ctx, int32_t rows);

typedef struct {
  double lr;    /* 1e-3 */
  double beta1; /* 0.9 */
  double beta2; /* 0.999 */
  double eps;   /* 1e-8 */
  int64_t step; /* 1 for the first update (bias correction 1 - beta^step) */
} mt_adam_cfg;

/* Host-side Adam on every tensor of the bound arena, from the G sections of the last
 * successful step: m = b1 m + (1-b1) g; v = b2 v + (1-b2) g^2; w -= lr mhat/(sqrt(vhat)+eps),
 * fp32 arithmetic per element (the constants 1-b1, 1-b2 and the bias corrections are formed
 * in double, then rounded once), w stored back as bf16 (round to nearest even), m and v as fp32.
 * Multithreaded (OpenMP) over the arena. (chestersoft digest, Methodik, "Layer-Contiguous
 * Tiling": the optimizer step runs on the CPU over the packed blocks.) */
int mt_adam_step(mt_ctx* ctx, const mt_adam_cfg* hp);

/* mt_train_step followed by mt_adam_step, overlapped: a host thread applies Adam to each block
 * as soon as that block's G section has reached the arena (head first, then the decoder layers
 * from the last, then the embedding), while the GPU is still working on earlier layers. The
 * per-element arithmetic is that of mt_adam_step, so the arena ends bit-identical to the two
 * calls in sequence. Each block's gradients arrive with the device error flag as it stood when
 * they left, and the loss is on the host before the first block lands: a non-finite loss
 * updates no block (MT_ECUDA), and a kernel whose bounded wait gave up stops the update before
 * the first block whose gradients came after it (MT_EKERNEL; blocks that landed earlier are
 * updated, and mt_last_error says how many). Other failures after work started (MT_ECUDA,
 * MT_ETIMEOUT) may leave some blocks updated. mt_get_stats reports the Adam time in adam_ms.
 * (Overlapping the CPU optimizer with the backward pass is this library's extension of the
 * chestersoft digest's CPU Adam, Methodik, "Layer-Contiguous Tiling".) */
int mt_train_step_adam(mt_ctx* ctx, const int32_t* tokens, const int32_t* labels, const mt_adam_cfg* hp,
                       float* loss);

/* Host memory bandwidth the host Adam is bounded by: a STREAM-style triad (a = b + s c, fp32,
 * 12 bytes moved per element) over three arrays of bytes/12 elements each, on the threads the
 * Adam update uses (OpenMP), best of `reps` passes, in GB/s. Allocates and frees about `bytes`
 * of host memory in all. *threads (may be NULL) receives the thread count. The Adam update moves 22 bytes
 * per parameter (bf16 W and G read, W written; fp32 m and v read and written), so 22 P / gbs is
 * its floor. MT_EINVAL for bytes < 12 or reps <= 0, MT_ENOMEM if the arrays cannot be had. */
int mt_host_bandwidth(uint64_t bytes, int32_t reps, double* gbs, int32_t* threads);

/* The same update on an arena without a context (no GPU needed), as mt_adam_step. */
int mt_adam_apply(const mt_model_cfg* cfg, void* arena, uint64_t bytes, const mt_adam_cfg* hp);

/* With MT_FLAG_FP32_MASTER: set every master tensor P to its bf16 weights W (exactly; P = W is
 * representable), as a freshly initialised arena needs before the first mt_adam_step. Host only;
 * MT_EINVAL if the flag is not set or the arena is shorter than mt_arena_bytes. The optional
 * fp32 master copy is the chestersoft digest's "full precision" reading taken the other way
 * (Kernaussagen / Methodik): 16 bytes per parameter instead of 12. */
int mt_master_init(const mt_model_cfg* cfg, void* arena, uint64_t bytes);

typedef struct {
  double step_ms;            /* device time of the last mt_train_step (first copy to last kernel/copy) */
  double compute_busy_ms;    /* summed spans of compute-stream work of that step */
  double h2d_busy_ms;        /* summed spans of host-to-device copies */
  double d2h_busy_ms;        /* summed spans of device-to-host copies */
  double exposed_ms;         /* time the compute stream stood still waiting for transfers: the summed
                                durations of its waits on copy events (weights arriving, gradient
                                buffers draining, checkpoints, the final gradient copies), each
                                measured by timing events recorded around the wait */
  double fwd_ms, bwd_ms;     /* device time of the forward phase (embedding .. head) and the rest */
  double adam_ms;            /* host wall time of the last mt_adam_step */
  double host_step_ms;       /* host wall time of the last mt_train_step call */
  uint64_t h2d_bytes;        /* bytes copied host-to-device in the last step */
  uint64_t d2h_bytes;        /* bytes copied device-to-host in the last step */
  int64_t kernel_launches;   /* kernels launched by the last step */
  int64_t steps;             /* successful steps so far */
  /* the copies split by direction [0 host-to-device, 1 device-to-host] and by the phase they
   * start in [0 forward (up to the head), 1 backward]: bytes moved and summed copy time, so
   * bytes / ms is the link speed the step's own copies reached in that phase */
  uint64_t copy_bytes[2][2];
  double copy_ms[2][2];
  double first_copy_ms;      /* duration of the step's first host-to-device copy of >= 1 MiB */
  double embed_gather_gbs;   /* rate of the embedding gather through the mapped arena (0: not used) */
  int32_t sparse_embed;      /* 1 if the step read and wrote the embedding block's rows through the
                                mapped arena; a gather of >= 16 MB below 25 GB/s switches later steps of
                                the context to whole-block copies (identical results) */
} mt_stats;
int mt_get_stats(mt_ctx* ctx, mt_stats* out);

/* Per-kind kernel timing of the last step (needs MT_FLAG_KERNEL_TIMING). Kinds: 0 GEMM,
 * 1 attention forward, 2 attention backward, 3 pointwise/norm, 4 cross-entropy, 5 embedding.
 * launches, summed device ms, and the algorithmic work: flops (GEMM, attention) or bytes. */
typedef struct {
  int64_t launches;
  double ms;
  double flops;
  double bytes;
} mt_kernel_stats;
#define MT_KIND_GEMM 0
#define MT_KIND_ATTN_FWD 1
#define MT_KIND_ATTN_BWD 2
#define MT_KIND_POINTWISE 3
#define MT_KIND_CROSS_ENTROPY 4
#define MT_KIND_EMBED 5
#define MT_KIND_COUNT 6
int mt_get_kernel_stats(mt_ctx* ctx, int32_t kind, mt_kernel_stats* out);
/* Turn per-launch kernel timing on (nonzero) or off for later steps (the same switch as
 * MT_FLAG_KERNEL_TIMING at creation). Timing records two CUDA events around every launch,
 * which costs the step a few percent. */
int mt_set_kernel_timing(mt_ctx* ctx, int32_t on);

/* Message of the last failure on ctx (or of the last failed context-free call if ctx is NULL). */
const char* mt_last_error(mt_ctx* ctx);

/* Release the context's device buffers, streams it created, pinned checkpoint memory and the
 * host registration of the arena, after waiting for the device. Never frees the arena or
 * caller-supplied resources. After an MT_ETIMEOUT step it does not wait and frees only the
 * host-side bookkeeping (device buffers, events and pinned staging are left to process exit). */
void mt_destroy(mt_ctx* ctx);

#ifdef __cplusplus
}
#endif
#endif /* MT_H */
