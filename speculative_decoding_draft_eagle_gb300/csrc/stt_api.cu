// stt_api.cu -- the C ABI declared in include/stt.h: argument validation,
// status codes, and dispatch to the kernel launchers.  No entry point
// allocates device memory or synchronises (except stt_device_error, which is
// documented to synchronise its stream).
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "../../include/stt.h"
#include "internal.h"

namespace stt {

void* tensor_map_encoder() {
  static void* fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = f;
  });
  return fn;
}

cudaError_t bind_device_context() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  return cudaSetDevice(dev);
}

namespace {
std::atomic<uint32_t> g_inject{0};
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
}  // namespace

int sm_count() {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
  if (dev < kMaxDevices) {
    const int c = g_sm_count[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
    return 1;
  if (dev < kMaxDevices) g_sm_count[dev].store(v, std::memory_order_relaxed);
  return v;
}

uint32_t debug_inject() { return g_inject.load(std::memory_order_relaxed); }

}  // namespace stt

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The CUDA error the last failing call of this thread returned (read and
// cleared by stt_last_cuda_error).
thread_local int t_last_cuda_error = 0;

int from_cuda(cudaError_t e) {
  if (e != cudaSuccess) t_last_cuda_error = (int)e;
  return stt::status_from_cuda(e);
}

// Every launching entry point starts here: an error that an earlier runtime
// call of this thread left behind (someone else's) is cleared, so that the
// check after our own launches reports only them.  A sticky error (a faulted
// context) cannot be cleared and still fails the launches.
inline void begin_call() { (void)cudaGetLastError(); }

static_assert(STT_ERR_UNSUPPORTED == -2 && STT_ERR_CUDA == -4, "status_from_cuda codes");
static_assert(STT_CE_BF16 == stt::kCeBf16 && STT_CE_G_PER_ELEMENT == stt::kCeGPerElement,
              "soft-CE flags");
static_assert(STT_BWD_ACCUMULATE_KV == stt::kBwdAccumulate && STT_BWD_BF16_GRADS == stt::kBwdBf16,
              "backward flags");

// Shared validation of the attention arguments; fills `a` on success.
int check_attn(const void* q, const void* const* k_blocks, const void* const* v_blocks,
               const int32_t* T_host, int B, int H, int H_kv, int D, int Q_LEN, int k, float scale,
               stt::AttnArgs* a) {
  if (!q || !k_blocks || !v_blocks || !T_host) return STT_ERR_INVALID_ARG;
  if (B < 1 || B > STT_MAX_BATCH || H < 1 || H_kv < 1 || Q_LEN < 1) return STT_ERR_INVALID_ARG;
  if (H % H_kv != 0) return STT_ERR_INVALID_ARG;
  if (k < 0 || k > STT_MAX_STEP) return STT_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return STT_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return STT_ERR_UNSUPPORTED;
  if (H / H_kv > 8) return STT_ERR_UNSUPPORTED;
  if ((long long)B * H * Q_LEN > (1ll << 31) - 1) return STT_ERR_UNSUPPORTED;
  if (!aligned16(q)) return STT_ERR_MISALIGNED;
  for (int j = 0; j <= k; ++j) {
    if (!k_blocks[j] || !v_blocks[j]) return STT_ERR_INVALID_ARG;
    if (!aligned16(k_blocks[j]) || !aligned16(v_blocks[j])) return STT_ERR_MISALIGNED;
  }
  for (int b = 0; b < B; ++b)
    if (T_host[b] < 0 || T_host[b] > Q_LEN) return STT_ERR_INVALID_ARG;
  std::memset(a, 0, sizeof(*a));
  a->q = q;
  for (int j = 0; j <= k; ++j) {
    a->k_blocks[j] = k_blocks[j];
    a->v_blocks[j] = v_blocks[j];
  }
  a->B = B;
  a->H = H;
  a->H_kv = H_kv;
  a->D = D;
  a->Q_LEN = Q_LEN;
  a->k = k;
  a->scale = scale;
  for (int b = 0; b < B; ++b) a->T[b] = T_host[b];
  return STT_OK;
}

}  // namespace

extern "C" {

const char* stt_status_string(int status) {
  switch (status) {
    case STT_OK: return "ok";
    case STT_ERR_INVALID_ARG: return "invalid argument";
    case STT_ERR_UNSUPPORTED: return "unsupported configuration";
    case STT_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case STT_ERR_CUDA: return "CUDA error";
    case STT_ERR_TIMEOUT: return "device-side bounded wait ran out";
    case STT_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

int stt_version(void) { return 100; }

int stt_device_error(void* stream, uint32_t* word) {
  if (!word) return STT_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return STT_ERR_CUDA;
  uint32_t w = 0, part = 0;
  if (stt::soft_ce_error_word(&part) != cudaSuccess) return STT_ERR_CUDA;
  w |= part;
  if (stt::attn_fwd_error_word(&part) != cudaSuccess) return STT_ERR_CUDA;
  w |= part;
  if (stt::attn_bwd_error_word(&part) != cudaSuccess) return STT_ERR_CUDA;
  w |= part;
  if (stt::lm_head_error_word(&part) != cudaSuccess) return STT_ERR_CUDA;
  w |= part;
  *word = w;
  return (w & STT_DEVERR_WAIT_MASK) ? STT_ERR_TIMEOUT : STT_OK;
}

int stt_last_cuda_error(const char** name) {
  const int e = t_last_cuda_error;
  t_last_cuda_error = 0;
  if (name) *name = cudaGetErrorName(static_cast<cudaError_t>(e));
  return e;
}

int stt_debug_set_wait_budget(uint64_t ns) {
  cudaError_t e = stt::soft_ce_set_wait_budget(ns);
  if (e == cudaSuccess) e = stt::attn_fwd_set_wait_budget(ns);
  if (e == cudaSuccess) e = stt::attn_bwd_set_wait_budget(ns);
  if (e == cudaSuccess) e = stt::lm_head_set_wait_budget(ns);
  return from_cuda(e);
}

int stt_debug_inject(uint32_t what) {
  if (what & ~(uint32_t)STT_INJECT_FWD_WITHHOLD_Q) return STT_ERR_INVALID_ARG;
  stt::g_inject.store(what, std::memory_order_relaxed);
  return STT_OK;
}

int stt_attn_fwd(const void* q, const void* const* k_blocks, const void* const* v_blocks,
                 const int32_t* T_host, int B, int H, int H_kv, int D, int Q_LEN, int k,
                 float scale, void* out, float* lse, void* stream) {
  try {
    begin_call();
    static thread_local stt::AttnArgs a;
    int st = check_attn(q, k_blocks, v_blocks, T_host, B, H, H_kv, D, Q_LEN, k, scale, &a);
    if (st != STT_OK) return st;
    if (!out || !lse) return STT_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(lse)) return STT_ERR_MISALIGNED;
    return from_cuda(stt::attn_fwd_launch(a, out, lse, static_cast<cudaStream_t>(stream)));
  } catch (...) {
    return STT_ERR_CUDA;
  }
}

size_t stt_attn_bwd_workspace_size(int B, int H, int H_kv, int D, int Q_LEN, int k) {
  return stt_attn_bwd_ex_workspace_size(B, H, H_kv, D, Q_LEN, k, 0u);
}

size_t stt_attn_bwd_ex_workspace_size(int B, int H, int H_kv, int D, int Q_LEN, int k,
                                      uint32_t flags) {
  (void)k;
  if (B < 1 || H < 1 || H_kv < 1 || Q_LEN < 1 || D < 1) return 16;
  return stt::attn_bwd_workspace(B, H, H_kv, D, Q_LEN, flags);
}

int stt_attn_bwd_ex(const void* q, const void* const* k_blocks, const void* const* v_blocks,
                    const int32_t* T_host, int B, int H, int H_kv, int D, int Q_LEN, int k,
                    float scale, const void* out, const void* dout, const float* lse, void* dq,
                    void* const* dk_blocks, void* const* dv_blocks, uint32_t flags,
                    void* workspace, size_t workspace_bytes, void* stream) {
  try {
    begin_call();
    static thread_local stt::AttnArgs a;
    int st = check_attn(q, k_blocks, v_blocks, T_host, B, H, H_kv, D, Q_LEN, k, scale, &a);
    if (st != STT_OK) return st;
    if (flags & ~(uint32_t)(STT_BWD_ACCUMULATE_KV | STT_BWD_BF16_GRADS)) return STT_ERR_INVALID_ARG;
    if (!out || !dout || !lse || !dq || !dk_blocks || !dv_blocks) return STT_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(dout) || !aligned16(lse) || !aligned16(dq))
      return STT_ERR_MISALIGNED;
    stt::AttnBwdArgs g;
    std::memset(&g, 0, sizeof(g));
    for (int j = 0; j <= k; ++j) {
      if (!dk_blocks[j] || !dv_blocks[j]) return STT_ERR_INVALID_ARG;
      if (!aligned16(dk_blocks[j]) || !aligned16(dv_blocks[j])) return STT_ERR_MISALIGNED;
      g.dk_blocks[j] = dk_blocks[j];
      g.dv_blocks[j] = dv_blocks[j];
    }
    const size_t need = stt::attn_bwd_workspace(B, H, H_kv, D, Q_LEN, flags);
    if (!workspace || workspace_bytes < need) return STT_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return STT_ERR_MISALIGNED;
    g.out = out;
    g.dout = dout;
    g.lse = lse;
    g.dq = dq;
    g.flags = flags;
    g.workspace = workspace;
    return from_cuda(stt::attn_bwd_launch(a, g, static_cast<cudaStream_t>(stream)));
  } catch (...) {
    return STT_ERR_CUDA;
  }
}

int stt_attn_bwd(const void* q, const void* const* k_blocks, const void* const* v_blocks,
                 const int32_t* T_host, int B, int H, int H_kv, int D, int Q_LEN, int k,
                 float scale, const void* out, const void* dout, const float* lse, float* dq,
                 float* const* dk_blocks, float* const* dv_blocks, void* workspace,
                 size_t workspace_bytes, void* stream) {
  return stt_attn_bwd_ex(q, k_blocks, v_blocks, T_host, B, H, H_kv, D, Q_LEN, k, scale, out, dout,
                         lse, dq, reinterpret_cast<void* const*>(dk_blocks),
                         reinterpret_cast<void* const*>(dv_blocks), 0u, workspace,
                         workspace_bytes, stream);
}

size_t soft_ce_workspace_size(int64_t N, int64_t V) {
  (void)V;
  if (N < 0) return 16;
  size_t b = (size_t)N * sizeof(float);
  b = (b + 15) / 16 * 16;
  return b < 16 ? 16 : b;
}

int soft_ce_fwd_bwd_inplace(float* z, const float* p, const float* g, int64_t N, int64_t V,
                            float* row_loss, float* loss, void* workspace,
                            size_t workspace_bytes, void* stream) {
  try {
    begin_call();
    if (N < 0 || V < 1 || !loss) return STT_ERR_INVALID_ARG;
    if (N > 0 && (!z || !p || !g)) return STT_ERR_INVALID_ARG;
    if (N > 0 && V > INT64_MAX / N) return STT_ERR_INVALID_ARG;
    if (V > stt::kCeMaxV) return STT_ERR_UNSUPPORTED;
    if (N * (V > 16 ? 16 : V) > 0x7fffffffLL) return STT_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < soft_ce_workspace_size(N, V)) return STT_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 3u) != 0) return STT_ERR_MISALIGNED;
    const stt::CePlan plan = stt::soft_ce_plan(z, p, N, V);
    if (N * (int64_t)plan.C > 0x7fffffffLL) return STT_ERR_UNSUPPORTED;
    return from_cuda(stt::soft_ce_launch(plan, z, p, g, N, V, row_loss, loss,
                                         static_cast<float*>(workspace),
                                         static_cast<cudaStream_t>(stream)));
  } catch (...) {
    return STT_ERR_CUDA;
  }
}

int soft_ce_fwd_bwd_inplace_ex(void* z, const void* p, const float* g, int64_t N, int64_t V,
                               uint32_t flags, float* row_loss, float* loss, void* workspace,
                               size_t workspace_bytes, void* stream) {
  try {
    begin_call();
    if (flags & ~(uint32_t)(STT_CE_BF16 | STT_CE_G_PER_ELEMENT)) return STT_ERR_INVALID_ARG;
    if (flags == 0)
      return soft_ce_fwd_bwd_inplace(static_cast<float*>(z), static_cast<const float*>(p), g, N,
                                     V, row_loss, loss, workspace, workspace_bytes, stream);
    if (N < 0 || V < 1 || !loss) return STT_ERR_INVALID_ARG;
    if (N > 0 && (!z || !p || !g)) return STT_ERR_INVALID_ARG;
    if (N > 0 && V > INT64_MAX / N) return STT_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < soft_ce_workspace_size(N, V)) return STT_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 3u) != 0) return STT_ERR_MISALIGNED;
    const stt::CeVariantPlan plan = stt::soft_ce_variant_plan(z, p, g, V, flags);
    if (!plan.ok) return STT_ERR_UNSUPPORTED;
    if (N * (int64_t)plan.C > 0x7fffffffLL) return STT_ERR_UNSUPPORTED;
    return from_cuda(stt::soft_ce_variant_launch(plan, flags, z, p, g, N, V, row_loss, loss,
                                                 static_cast<float*>(workspace),
                                                 static_cast<cudaStream_t>(stream)));
  } catch (...) {
    return STT_ERR_CUDA;
  }
}

size_t stt_lm_head_ce_workspace_size(int64_t N, int64_t Hd, int64_t V) {
  (void)Hd;
  if (N < 0 || V < 1) return 16;
  return stt::lm_head_ce_workspace(N, V);
}

int stt_lm_head_ce(const void* h, const void* W, const float* p, const float* g, int64_t N,
                   int64_t Hd, int64_t V, float* dh, float* dW, float* row_loss, float* loss,
                   void* workspace, size_t workspace_bytes, void* stream) {
  try {
    begin_call();
    if (N < 0 || Hd < 8 || V < 8 || !loss) return STT_ERR_INVALID_ARG;
    if (Hd % 8 != 0 || V % 8 != 0) return STT_ERR_UNSUPPORTED;
    if (N > 0x7fffffffLL || Hd > 0x7fffffffLL || V > 0x7fffffffLL) return STT_ERR_UNSUPPORTED;
    if (N > 0 && (!h || !W || !p || !g || !dh || !dW)) return STT_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < stt::lm_head_ce_workspace(N, V)) return STT_ERR_WORKSPACE;
    const uintptr_t a = reinterpret_cast<uintptr_t>(h) | reinterpret_cast<uintptr_t>(W) |
                        reinterpret_cast<uintptr_t>(p) | reinterpret_cast<uintptr_t>(dh) |
                        reinterpret_cast<uintptr_t>(dW);
    if ((a & 15u) != 0 || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
      return STT_ERR_MISALIGNED;
    return from_cuda(stt::lm_head_ce_launch(h, W, p, g, N, Hd, V, dh, dW, row_loss, loss,
                                            workspace, static_cast<cudaStream_t>(stream)));
  } catch (...) {
    return STT_ERR_CUDA;
  }
}

int stt_verify(const float* p_target, const float* p_draft, const int32_t* draft_tokens,
               const float* u_accept, const float* u_sample, int B, int gamma, int64_t V,
               int32_t* n_accepted, int32_t* out_tokens, void* stream) {
  try {
    begin_call();
    if (B < 0 || gamma < 1 || gamma > STT_VERIFY_MAX_GAMMA || V < 1) return STT_ERR_INVALID_ARG;
    if (B == 0) return STT_OK;
    if (!p_target || !p_draft || !draft_tokens || !u_accept || !u_sample || !n_accepted ||
        !out_tokens)
      return STT_ERR_INVALID_ARG;
    if ((long long)B * gamma > INT64_MAX / V) return STT_ERR_INVALID_ARG;
    if (V > 0x7fffffffLL) return STT_ERR_UNSUPPORTED;
    const uintptr_t a = reinterpret_cast<uintptr_t>(p_target) |
                        reinterpret_cast<uintptr_t>(p_draft) |
                        reinterpret_cast<uintptr_t>(draft_tokens) |
                        reinterpret_cast<uintptr_t>(u_accept) |
                        reinterpret_cast<uintptr_t>(u_sample) |
                        reinterpret_cast<uintptr_t>(n_accepted) |
                        reinterpret_cast<uintptr_t>(out_tokens);
    if (a & 3u) return STT_ERR_MISALIGNED;
    return from_cuda(stt::verify_launch(p_target, p_draft, draft_tokens, u_accept, u_sample, B,
                                        gamma, V, n_accepted, out_tokens,
                                        static_cast<cudaStream_t>(stream)));
  } catch (...) {
    return STT_ERR_CUDA;
  }
}

}  // extern "C"
