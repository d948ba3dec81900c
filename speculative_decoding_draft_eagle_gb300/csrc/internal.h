// internal.h -- declarations shared by the host-side ABI (stt_api.cu) and the
// kernel translation units.  Not part of the public interface.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace stt {

// ------------------------------------------------------------- soft-CE ----
struct CePlan {
  bool bulk;     // bulk-copy (TMA) path: 16-byte aligned rows
  int C;         // CTAs per row (thread-block cluster size)
  int slice;     // elements of a row per CTA
  int smem;      // dynamic shared memory bytes per CTA
  bool persistent;  // persistent clusters walking the rows, nb row buffers per CTA
  bool split;       // persistent with z and p in separate buffers (large slices)
  int nb;
};
CePlan soft_ce_plan(const float* z, const float* p, int64_t N, int64_t V);
constexpr int64_t kCeMaxV = 409600;  // 16 CTAs x 25600 elements
cudaError_t soft_ce_launch(const CePlan& plan, float* z, const float* p, const float* g, int64_t N,
                           int64_t V, float* row_loss, float* loss, float* wl, cudaStream_t s);

// Fixed-order sum of the per-row weighted losses wl[0..N) into *loss, launched
// as a programmatic dependent of the kernel before it on the stream.
cudaError_t soft_ce_loss_sum_launch(const float* wl, int64_t N, float* loss, cudaStream_t s);

// Variants (the STT_CE_* bits of the public header).
constexpr uint32_t kCeBf16 = 0x1u;         // z and p are bf16
constexpr uint32_t kCeGPerElement = 0x2u;  // g is fp32 [N, V]
struct CeVariantPlan {
  bool ok;     // the slice fits in shared memory
  bool bulk;   // 16-byte aligned rows (bulk copies)
  int C;       // CTAs per row (cluster size)
  int slice;   // elements per CTA
  int chunk;   // elements per bulk-copy chunk
  int smem;    // dynamic shared bytes per CTA
};
CeVariantPlan soft_ce_variant_plan(const void* z, const void* p, const float* g, int64_t V,
                                   uint32_t flags);
cudaError_t soft_ce_variant_launch(const CeVariantPlan& plan, uint32_t flags, void* z,
                                   const void* p, const float* g, int64_t N, int64_t V,
                                   float* row_loss, float* loss, float* wl, cudaStream_t s);
// The variants on the persistent cluster kernel (rows 16-byte aligned, V a
// multiple of 8, slices within its registers' reach); cudaErrorNotSupported
// when a call does not fit it, before anything is launched.
cudaError_t soft_ce_variant_persistent_launch(uint32_t flags, void* z, const void* p,
                                              const float* g, int64_t N, int64_t V,
                                              float* row_loss, float* loss, float* wl,
                                              cudaStream_t s);

// ------------------------------------------------------- LM head + soft-CE --
size_t lm_head_ce_workspace(int64_t N, int64_t V);
cudaError_t lm_head_ce_launch(const void* h, const void* W, const float* p, const float* g,
                              int64_t N, int64_t Hd, int64_t V, float* dh, float* dW,
                              float* row_loss, float* loss, void* workspace, cudaStream_t s);
cudaError_t lm_head_error_word(uint32_t* w);
cudaError_t lm_head_set_wait_budget(uint64_t ns);

// ---------------------------------------------------------- verification --
cudaError_t verify_launch(const float* p_t, const float* p_d, const int32_t* tokens,
                          const float* u_accept, const float* u_sample, int B, int gamma,
                          int64_t V, int32_t* n_acc, int32_t* out, cudaStream_t s);

// ----------------------------------------------------------- attention ----
constexpr int kMaxBatch = 1024;
constexpr int kMaxBlocks = 32;

struct AttnArgs {
  const void* q;
  const void* k_blocks[kMaxBlocks];
  const void* v_blocks[kMaxBlocks];
  int B, H, H_kv, D, Q_LEN, k;
  float scale;
  int T[kMaxBatch];
};

cudaError_t attn_fwd_launch(const AttnArgs& a, void* out, float* lse, cudaStream_t s);

// Flags of the backward (the STT_BWD_* bits of the public header).
constexpr uint32_t kBwdAccumulate = 0x1u;  // add into dK_j / dV_j instead of overwriting
constexpr uint32_t kBwdBf16 = 0x2u;        // dq, dK_j, dV_j are bf16

struct AttnBwdArgs {
  const void* out;
  const void* dout;
  const float* lse;
  void* dq;                     // fp32, or bf16 with kBwdBf16
  void* dk_blocks[kMaxBlocks];  // same element type as dq
  void* dv_blocks[kMaxBlocks];
  uint32_t flags;
  void* workspace;  // attn_bwd_workspace(...) bytes, 256-byte aligned
};
// Workspace: Delta [B, H, Q_LEN] fp32; with kBwdBf16 also fp32 accumulators
// for dq [B, H, Q_LEN, D] and dK_0, dV_0 [B, H_kv, Q_LEN, D].
size_t attn_bwd_workspace(int B, int H, int H_kv, int D, int Q_LEN, uint32_t flags);
cudaError_t attn_bwd_launch(const AttnArgs& a, const AttnBwdArgs& g, cudaStream_t s);

// Per-file device error words (read and cleared).
cudaError_t soft_ce_error_word(uint32_t* w);
cudaError_t attn_fwd_error_word(uint32_t* w);
cudaError_t attn_bwd_error_word(uint32_t* w);
// Per-file bounded-wait budgets (nanoseconds; 0 restores the default).
cudaError_t soft_ce_set_wait_budget(uint64_t ns);
cudaError_t attn_fwd_set_wait_budget(uint64_t ns);
cudaError_t attn_bwd_set_wait_budget(uint64_t ns);

// Streaming multiprocessors of the current device (cached per device; 1 if
// the query fails, which only shrinks persistent grids).
int sm_count();

// Test hooks set by stt_debug_inject (STT_INJECT_* bits), read at launch.
uint32_t debug_inject();

// Status code of a CUDA error: cudaErrorNotSupported (an unsupported device
// or driver feature) is STT_ERR_UNSUPPORTED (-2), every other failure
// STT_ERR_CUDA (-4).
inline int status_from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return 0;
  if (e == cudaErrorNotSupported) return -2;
  return -4;
}

// Per-launch timing hooks (profile.cu); no-ops unless stt_profile_start ran.
void prof_before(cudaStream_t s, int kernel_id);
void prof_after(cudaStream_t s);

// Resolves cuTensorMapEncodeTiled through the runtime (no link against libcuda).
void* tensor_map_encoder();

// Makes the current device's primary context current on the calling thread.
// The tensor-map encoder is a driver call: on a thread that has not yet made
// a runtime call that binds the context (a fresh thread, e.g. the autograd
// engine's), it fails.  Called before any encoding.
cudaError_t bind_device_context();

}  // namespace stt
