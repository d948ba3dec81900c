/*
 * stt.h -- C ABI of the EAGLE-3 training-time-test (TTT) draft-step core on
 * NVIDIA GB300 (sm_103a).
 *
 * Two operations, as defined by the xllm-io review of "SpecForge: A Flexible
 * and Efficient Open-Source Training Framework for Speculative Decoding"
 * (cited as "SpecForge review"):
 *
 *  1. Sparse-tree TTT attention (SpecForge review, §三 "稀疏树注意力" and §四
 *     "BlockMask 构造").  At TTT step k the queries q attend to the
 *     concatenation of k+1 KV blocks (each Q_LEN rows) under the mask
 *         M = (q >= kv AND kv < T) OR
 *             (kv >= Q_LEN AND kv mod Q_LEN < T AND (kv - q) mod Q_LEN == 0)
 *     i.e. block 0 is causal with the padded columns kv >= T cut, and a query
 *     q < T additionally sees exactly key q of every later block j = 1..k.
 *     Queries q >= T ("padded rows") see the T keys kv < T and nothing else.
 *
 *  2. Masked soft-target softmax cross-entropy with the gradient written in
 *     place over the logits (SpecForge review, §三 "内存高效梯度计算", §四
 *     "掩码 Softmax 损失" / "原地反向传播"):
 *         pi = softmax(z_r), l_r = -sum_v p_rv log pi_rv,
 *         s_r = sum_v p_rv g_r,  z_rv <- -(p_rv g_r - pi_rv s_r),
 *         L = sum_r g_r l_r.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor arguments are DEVICE pointers into memory the caller owns
 *    (cudaMalloc'd, or a framework's allocator); arrays of pointers and T are
 *    HOST arrays.  The library allocates no device memory, never synchronises
 *    the device, and enqueues all work on `stream` (a cudaStream_t passed as
 *    void*; NULL means the legacy default stream).
 *  - Argument errors are detected on the host before any launch and returned
 *    as a negative stt_status; nothing is enqueued in that case.  A CUDA
 *    launch error is returned as STT_ERR_CUDA.  No C++ exception crosses the
 *    ABI.  Functions are thread-safe; calls that share output buffers must be
 *    ordered by the caller.
 *  - Asynchronous device-side failures (a bounded wait that ran out inside a
 *    kernel) are recorded in a library-wide error word that
 *    stt_device_error() reads and clears.
 *  - Layouts are dense row-major (C order), innermost dimension last.
 */
#ifndef STT_H_
#define STT_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define STT_API __attribute__((visibility("default")))
#else
#define STT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  STT_OK = 0,
  STT_ERR_INVALID_ARG = -1, /* null pointer, bad size, bad T, H % H_kv != 0 ... */
  STT_ERR_UNSUPPORTED = -2, /* valid but not implemented (e.g. D not 64/128)  */
  STT_ERR_MISALIGNED = -3,  /* a pointer is not 16-byte aligned               */
  STT_ERR_CUDA = -4,        /* a CUDA call failed (launch or driver)          */
  STT_ERR_TIMEOUT = -5,     /* a kernel's bounded wait ran out (device word)  */
  STT_ERR_WORKSPACE = -6    /* workspace missing or smaller than required     */
} stt_status;

/* Limits of this build. */
#define STT_MAX_BATCH 1024   /* B: T[] travels in the kernel parameters */
#define STT_MAX_STEP 31      /* k: at most 32 KV blocks                 */

/* Static, NUL-terminated description of a status code.  Thread-safe. */
STT_API const char* stt_status_string(int status);

/* Library version as 10000*major + 100*minor + patch. */
STT_API int stt_version(void);

/*
 * The cudaError_t code of the last CUDA failure (a status of STT_ERR_CUDA or
 * STT_ERR_UNSUPPORTED from a CUDA call) of a library call made by the calling
 * thread, 0 if none since the last read; reading clears it.  If `name` is not
 * NULL it receives the code's static name (cudaGetErrorName).  Every
 * launching entry point first clears an error that an earlier runtime call of
 * the same thread left pending, so a failure reported by the library is its
 * own.
 */
STT_API int stt_last_cuda_error(const char** name);

/*
 * Reads and clears the device-side error word (bitwise OR of the STT_DEVERR_*
 * sites whose bounded wait ran out since the last call).  Synchronises
 * `stream` first, then stores the word in *word and returns STT_ERR_TIMEOUT
 * if any STT_DEVERR_*_WAIT bit is set, STT_OK otherwise (the word is stored
 * in both cases), or STT_ERR_CUDA if the synchronisation or a read failed.
 */
STT_API int stt_device_error(void* stream, uint32_t* word);

/*
 * Failure-detection test hooks (no counterpart on the pages).  Every wait of
 * the kernels on an mbarrier is bounded by a wall-clock budget (2 s by
 * default); when it runs out, the waiting thread records its site in the
 * device error word and gives up, the other roles of the CTA give up in turn,
 * and the kernel returns (its outputs are then undefined).
 *
 * stt_debug_set_wait_budget(ns) sets that budget, in nanoseconds, on the
 * current device for every kernel of the library launched afterwards; 0
 * restores the default.  Returns STT_OK or STT_ERR_CUDA.
 *
 * stt_debug_inject(what) makes every later launch of the named kernels skip
 * one step on purpose, so that a bounded wait runs out without any fault:
 *   STT_INJECT_FWD_WITHHOLD_Q  the attention forward's producer never loads
 *                              the query tile, so the wait for it runs out;
 *                              every copy already issued is waited for before
 *                              the CTA exits, and no tensor-core product is
 *                              issued.
 * 0 switches injection off.  Unknown bits return STT_ERR_INVALID_ARG.  The
 * setting is process-wide; it is meant for tests, never for production runs.
 */
STT_API int stt_debug_set_wait_budget(uint64_t ns);
STT_API int stt_debug_inject(uint32_t what);
#define STT_INJECT_FWD_WITHHOLD_Q 0x1u

/* --------------------------------------------------------------------------
 * Sparse-tree attention, forward.
 *
 *  q        bf16 [B, H, Q_LEN, D], the step-k queries.
 *  k_blocks host array of k+1 device pointers; k_blocks[j] is bf16
 *           [B, H_kv, Q_LEN, D], the keys of TTT block j (block 0 = causal).
 *  v_blocks host array of k+1 device pointers, same shape as k_blocks[j].
 *  T_host   host int32 [B], valid length of each sequence, 0 <= T[b] <= Q_LEN.
 *  B        1 <= B <= STT_MAX_BATCH.
 *  H, H_kv  query / KV heads; H % H_kv == 0; query head h reads KV head
 *           h / (H / H_kv).
 *  D        head dimension, 64 or 128.
 *  Q_LEN    block length, >= 1.
 *  k        TTT step, 0 <= k <= STT_MAX_STEP.
 *  scale    softmax scale applied to q.K (1/sqrt(D) in the usual case); finite
 *           and > 0 (STT_ERR_INVALID_ARG otherwise).
 *  out      bf16 [B, H, Q_LEN, D]: O = softmax(scale q Kc^T + mask) Vc,
 *           rounded to nearest even.  A row with no visible key (T[b] = 0)
 *           is written as zeros.
 *  lse      fp32 [B, H, Q_LEN]: natural-log logsumexp of the visible scaled
 *           scores (-inf for a row with no visible key).
 *  All device pointers must be 16-byte aligned (TMA requirement).
 * ------------------------------------------------------------------------ */
STT_API int stt_attn_fwd(const void* q, const void* const* k_blocks, const void* const* v_blocks,
                 const int32_t* T_host, int B, int H, int H_kv, int D, int Q_LEN, int k,
                 float scale, void* out, float* lse, void* stream);

/* Bytes of device workspace stt_attn_bwd needs for these sizes (>= 16). */
STT_API size_t stt_attn_bwd_workspace_size(int B, int H, int H_kv, int D, int Q_LEN, int k);

/* --------------------------------------------------------------------------
 * Sparse-tree attention, backward: the gradient of sum(O * dout) with respect
 * to q and every K/V block (the page trains through this attention; the
 * backward is the derivative of the definition, recomputing P from lse).
 *
 *  q, k_blocks, v_blocks, T_host, B, H, H_kv, D, Q_LEN, k, scale: as forward.
 *  out      bf16 [B, H, Q_LEN, D], the forward output.
 *  dout     bf16 [B, H, Q_LEN, D], upstream gradient of out.
 *  lse      fp32 [B, H, Q_LEN], the forward logsumexp.
 *  dq       fp32 [B, H, Q_LEN, D], OVERWRITTEN with dL/dq.
 *  dk_blocks host array of k+1 device pointers, fp32 [B, H_kv, Q_LEN, D],
 *           each OVERWRITTEN with dL/dK_j (summed over the query heads of the
 *           group; zero for rows no query sees).
 *  dv_blocks same for dL/dV_j.
 *  workspace device scratch of at least stt_attn_bwd_workspace_size() bytes,
 *           256-byte aligned; contents on entry are ignored.
 * ------------------------------------------------------------------------ */
STT_API int stt_attn_bwd(const void* q, const void* const* k_blocks, const void* const* v_blocks,
                 const int32_t* T_host, int B, int H, int H_kv, int D, int Q_LEN, int k,
                 float scale, const void* out, const void* dout, const float* lse, float* dq,
                 float* const* dk_blocks, float* const* dv_blocks, void* workspace,
                 size_t workspace_bytes, void* stream);

/* --------------------------------------------------------------------------
 * Sparse-tree attention, backward with options.  Same operation and
 * arguments as stt_attn_bwd, plus `flags`:
 *
 *  STT_BWD_ACCUMULATE_KV  dL/dK_j and dL/dV_j are ADDED to what dk_blocks[j]
 *           and dv_blocks[j] hold instead of overwriting them (dq is still
 *           overwritten).  This is the training use of the TTT step loop
 *           (SpecForge review, §三 "稀疏树注意力", TTT length 7, and §六
 *           "训练时测试（TTT）长度的影响"): block j is read by every step k >= j,
 *           so its gradient is the sum over those steps; each step's call adds
 *           its part in place, with no separate pass over the block gradients.
 *           Rows that no query of the step sees are left unchanged.
 *  STT_BWD_BF16_GRADS  dq, dk_blocks[j] and dv_blocks[j] are bf16 (round to
 *           nearest even) instead of fp32.  Sums across key tiles and heads
 *           are taken in fp32 in the workspace and rounded once at the end;
 *           with STT_BWD_ACCUMULATE_KV the existing bf16 value is added in fp32
 *           and the sum rounded once per call.
 *
 *  dq, dk_blocks, dv_blocks  device pointers of the element type the flags
 *           select, layouts as in stt_attn_bwd.
 *  workspace at least stt_attn_bwd_ex_workspace_size(..., flags) bytes,
 *           256-byte aligned (STT_ERR_MISALIGNED otherwise); contents on entry
 *           are ignored.
 * Unknown flag bits return STT_ERR_INVALID_ARG.  stt_attn_bwd is this call
 * with flags = 0.
 * ------------------------------------------------------------------------ */
#define STT_BWD_ACCUMULATE_KV 0x1u
#define STT_BWD_BF16_GRADS 0x2u
STT_API size_t stt_attn_bwd_ex_workspace_size(int B, int H, int H_kv, int D, int Q_LEN, int k,
                                              uint32_t flags);
STT_API int stt_attn_bwd_ex(const void* q, const void* const* k_blocks,
                            const void* const* v_blocks, const int32_t* T_host, int B, int H,
                            int H_kv, int D, int Q_LEN, int k, float scale, const void* out,
                            const void* dout, const float* lse, void* dq, void* const* dk_blocks,
                            void* const* dv_blocks, uint32_t flags, void* workspace,
                            size_t workspace_bytes, void* stream);

/* Bytes of device workspace soft_ce_fwd_bwd_inplace needs (>= 16). */
STT_API size_t soft_ce_workspace_size(int64_t N, int64_t V);

/* --------------------------------------------------------------------------
 * Masked soft-target cross-entropy, loss and in-place gradient, one pass.
 *
 *  z        fp32 [N, V] logits; OVERWRITTEN with dL/dz = pi*s - p*g.
 *  p        fp32 [N, V] target distribution (rows need not sum to 1).
 *  g        fp32 [N] per-row upstream gradient / loss weight (mask / N).
 *  N        rows, >= 0.   V  vocabulary, >= 1.
 *  row_loss fp32 [N] or NULL: l_r = -sum_v p log softmax(z_r) for rows with
 *           g_r != 0, and 0 for rows with g_r == 0 (masked rows are not read).
 *  loss     fp32 scalar (device): L = sum_r g_r l_r, summed in a fixed order
 *           (deterministic).  0 when N == 0.
 *  workspace device scratch of at least soft_ce_workspace_size(N, V) bytes.
 *  Rows with g_r == 0 get an exact-zero gradient.  z and p should be 16-byte
 *  aligned with V % 4 == 0 for the bulk-copy path; other layouts take a
 *  slower element-wise path with identical results.
 * ------------------------------------------------------------------------ */
STT_API int soft_ce_fwd_bwd_inplace(float* z, const float* p, const float* g, int64_t N, int64_t V,
                            float* row_loss, float* loss, void* workspace,
                            size_t workspace_bytes, void* stream);

/* --------------------------------------------------------------------------
 * Soft-CE variants the formula admits (SpecForge review, §三 "内存高效梯度计算":
 * s = sum(p * g), z <- -(p * g - pi * s)).  `flags`:
 *
 *  STT_CE_BF16           z and p are bf16 [N, V]; every sum is taken in fp32
 *                        and the gradient is written over z rounded to bf16
 *                        (nearest even).
 *  STT_CE_G_PER_ELEMENT  g is fp32 [N, V], one upstream gradient per logit:
 *                            s_r = sum_v p_rv g_rv,  z_rv <- pi_rv s_r - p_rv g_rv,
 *                            row_loss_r = -sum_v g_rv p_rv log pi_rv,
 *                            L = sum_r row_loss_r
 *                        (row_loss is then already weighted, and every row is
 *                        read).
 * flags = 0 is soft_ce_fwd_bwd_inplace (fp32 z and p, per-row g).  Other
 * arguments, the workspace and the status codes as there; V may be at most
 * 16 slices of the shared memory a CTA can hold (above ~270000 for fp32 with
 * a per-element g) and STT_ERR_UNSUPPORTED is returned beyond that.  Unknown
 * flag bits return STT_ERR_INVALID_ARG.  Rows whose addresses are 16-byte
 * aligned with V % 8 == 0 take bulk copies; others an element-wise path with
 * identical results.
 * ------------------------------------------------------------------------ */
#define STT_CE_BF16 0x1u
#define STT_CE_G_PER_ELEMENT 0x2u
STT_API int soft_ce_fwd_bwd_inplace_ex(void* z, const void* p, const float* g, int64_t N,
                                       int64_t V, uint32_t flags, float* row_loss, float* loss,
                                       void* workspace, size_t workspace_bytes, void* stream);

/* --------------------------------------------------------------------------
 * Allocation-free soft-CE (the paper has no counterpart; this is a library
 * convenience).  Identical results to soft_ce_fwd_bwd_inplace, but it takes no
 * workspace: its per-row scratch is a fixed 256 KB array inside the library
 * (allocated when the library is loaded, held on every GPU that loads it until
 * the process exits).  It is for callers that cannot call cudaMalloc: for
 * example an operator plugged into a host framework that hands it only its
 * input and output buffers and owns all device memory itself, or code in a
 * phase where device allocation is not permitted.  The call itself allocates
 * nothing and calls no allocating routine.
 *
 *  z, p, g, N, V, row_loss, loss: as soft_ce_fwd_bwd_inplace.
 *  N must be <= 65536 rows (the scratch size); larger N returns
 *  STT_ERR_WORKSPACE without launching anything.
 *  Every call looks up the scratch array's device address on the current
 *  device (cudaGetSymbolAddress), so the address stays right after a
 *  cudaDeviceReset or a new primary context; the first call on a device also
 *  loads the library's kernels there, so make that first call before any
 *  stream capture.  All calls share the one array, so calls whose kernels
 *  overlap on the GPU (different streams, or threads without ordering) race
 *  on it and must be serialised by the caller.  Every scratch entry a call
 *  reads is written earlier in the same call, so the previous call's
 *  leftovers never affect the result.  Status codes are those of
 *  soft_ce_fwd_bwd_inplace (a CUDA failure the device does not support is
 *  STT_ERR_UNSUPPORTED, any other STT_ERR_CUDA).
 * ------------------------------------------------------------------------ */
STT_API int soft_ce_fwd_bwd_inplace_noalloc(float* z, const float* p, const float* g, int64_t N,
                                            int64_t V, float* row_loss, float* loss,
                                            void* stream);

/* --------------------------------------------------------------------------
 * The draft's LM head fused with the soft-CE, chunked over the vocabulary
 * (SpecForge review, §三 "内存高效梯度计算": the logits are the activation the
 * in-place gradient saves memory on; §四 "原地反向传播").  With hidden states
 * h, head weights W, targets p and per-row upstream gradients g:
 *     z = h W^T,  L = sum_r g_r l_r (l_r and dL/dz as soft_ce_fwd_bwd_inplace),
 *     dh = (dL/dz) W,  dW = (dL/dz)^T h.
 * The logits are never stored: a tensor-core pass computes per-row softmax
 * statistics from z tile by tile, and a second pass recomputes z one
 * vocabulary chunk at a time and turns it into dL/dz (bf16, in the
 * workspace), which feeds dh and dW at once.
 *
 *  h        bf16 [N, Hd] row-major.      W  bf16 [V, Hd] row-major.
 *  p        fp32 [N, V].                 g  fp32 [N].
 *  N >= 0; Hd and V multiples of 8 (STT_ERR_UNSUPPORTED otherwise), >= 8.
 *  dh       fp32 [N, Hd], OVERWRITTEN with dL/dh.
 *  dW       fp32 [V, Hd], OVERWRITTEN with dL/dW.
 *  row_loss fp32 [N] or NULL: l_r (0 for rows with g_r = 0).
 *  loss     fp32 scalar (device): L, summed in a fixed order.
 *  workspace at least stt_lm_head_ce_workspace_size(N, Hd, V) bytes,
 *           256-byte aligned; h, W, p, dh, dW 16-byte aligned.
 * dL/dz enters the two gradient products rounded to bf16 (as the operands of
 * any bf16 training step); sums are fp32.
 * ------------------------------------------------------------------------ */
STT_API size_t stt_lm_head_ce_workspace_size(int64_t N, int64_t Hd, int64_t V);
STT_API int stt_lm_head_ce(const void* h, const void* W, const float* p, const float* g,
                           int64_t N, int64_t Hd, int64_t V, float* dh, float* dW,
                           float* row_loss, float* loss, void* workspace,
                           size_t workspace_bytes, void* stream);

/* --------------------------------------------------------------------------
 * Speculative-decoding verification by rejection sampling (the "FlashSpec"
 * practice page, §3.4 "验证器的具体实现").  For each sequence b the draft's
 * tokens x_0..x_{gamma-1} are tested in order: x_i is accepted with
 * probability min(1, p_t[x_i] / p_d[x_i]), evaluated as
 * u_accept[b, i] * p_d < p_t in fp64 (a token with p_d = 0 is accepted iff
 * p_t > 0; a token outside [0, V) never).  At the first rejection one token
 * is drawn from norm(max(0, p_t - p_d)) at that position -- the smallest y
 * whose running residual sum (fp64) exceeds u_sample[b] times the total, or
 * from p_t itself if the residual is all zero -- and the sequence stops.
 * Nothing is drawn when every token is accepted.
 *
 *  p_target   fp32 [B, gamma, V]: the target model's distribution at each
 *             draft position.
 *  p_draft    fp32 [B, gamma, V]: the draft's distribution there.
 *  draft_tokens int32 [B, gamma].
 *  u_accept   fp32 [B, gamma], uniform in [0, 1): the acceptance draws.
 *  u_sample   fp32 [B], uniform in [0, 1): the resampling draw.
 *  B >= 0 (0 does nothing), 1 <= gamma <= STT_VERIFY_MAX_GAMMA, V >= 1.
 *  n_accepted int32 [B]: accepted draft tokens per sequence.
 *  out_tokens int32 [B, gamma]: the accepted tokens, then the drawn token if
 *             n_accepted < gamma, then -1.
 * All pointers device, 4-byte aligned (rows that are 16-byte aligned with
 * V % 4 == 0 are read with 16-byte loads).  V above 16 x 51200 returns
 * STT_ERR_UNSUPPORTED (a rejected row is split over at most 16 CTAs, each
 * holding its slice in shared memory).  The random numbers are inputs, so a
 * call is deterministic.
 * ------------------------------------------------------------------------ */
#define STT_VERIFY_MAX_GAMMA 32
STT_API int stt_verify(const float* p_target, const float* p_draft, const int32_t* draft_tokens,
                       const float* u_accept, const float* u_sample, int B, int gamma, int64_t V,
                       int32_t* n_accepted, int32_t* out_tokens, void* stream);

/* --------------------------------------------------------------------------
 * Per-launch timing (measurement support; no counterpart on the pages).
 * stt_profile_start(capacity) makes every subsequent kernel launch of the
 * library (from any thread) record a CUDA event pair around itself on its
 * launch stream, for up to `capacity` launches.  stt_profile_stop() waits for
 * the recorded events, writes up to `capacity` (kernel id, milliseconds)
 * pairs into the caller's host arrays (either may be NULL), stores the count
 * in *n and disables recording.  Events are host-side objects: no device
 * memory is allocated.  Returns STT_ERR_INVALID_ARG when not in the right
 * state, STT_ERR_CUDA if an event call failed.
 * ------------------------------------------------------------------------ */
STT_API int stt_profile_start(int capacity);
STT_API int stt_profile_stop(int* n, int* kernel_ids, float* ms, int capacity);
/* Static name of a kernel id ("attn_fwd", ...). */
STT_API const char* stt_kernel_name(int kernel_id);

#define STT_KERNEL_SOFT_CE 1
/* The soft-CE row kernel and its loss sum are recorded together as
 * STT_KERNEL_SOFT_CE; STT_KERNEL_SOFT_CE_LOSS_SUM only names the second. */
#define STT_KERNEL_SOFT_CE_LOSS_SUM 2
#define STT_KERNEL_ATTN_FWD 3
#define STT_KERNEL_ATTN_BWD_PREP 4
#define STT_KERNEL_ATTN_BWD_CAUSAL 5
#define STT_KERNEL_ATTN_BWD_CAST 6
#define STT_KERNEL_SOFT_CE_VARIANT 7
#define STT_KERNEL_VERIFY 8
#define STT_KERNEL_LM_HEAD_CE 9

/* Device error-word bits: sites of bounded waits that gave up, and blocks
 * whose dynamic shared memory did not have the 1024-byte alignment the
 * swizzled tiles need (such a block skips its work). */
#define STT_DEVERR_FWD_WAIT 0x1u
#define STT_DEVERR_BWD_WAIT 0x2u
#define STT_DEVERR_CE_WAIT 0x4u
#define STT_DEVERR_SMEM_ALIGN 0x8u
#define STT_DEVERR_LM_WAIT 0x10u
#define STT_DEVERR_WAIT_MASK \
  (STT_DEVERR_FWD_WAIT | STT_DEVERR_BWD_WAIT | STT_DEVERR_CE_WAIT | STT_DEVERR_LM_WAIT)

#ifdef __cplusplus
}
#endif

#endif /* STT_H_ */
