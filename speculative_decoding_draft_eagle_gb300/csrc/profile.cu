// profile.cu -- optional per-launch timing.  While enabled, every kernel the
// library launches is bracketed by two CUDA events recorded on the launch
// stream; stt_profile_stop() returns each launch's kernel id and duration.
// Disabled (the default) it costs one relaxed atomic load per launch.
#include <atomic>
#include <mutex>
#include <vector>

#include "../../include/stt.h"
#include "internal.h"

namespace stt {
namespace {

struct Profiler {
  std::mutex m;
  std::atomic<bool> on{false};
  std::vector<cudaEvent_t> ev;  // 2 per launch
  std::vector<int> ids;
  int n = 0;
  int cap = 0;
  int dropped = 0;
};

Profiler& prof() {
  static Profiler p;
  return p;
}

}  // namespace

void prof_before(cudaStream_t s, int kernel_id) {
  Profiler& p = prof();
  if (!p.on.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> g(p.m);
  if (p.n >= p.cap) {
    ++p.dropped;
    return;
  }
  p.ids[p.n] = kernel_id;
  cudaEventRecord(p.ev[2 * p.n], s);
}

void prof_after(cudaStream_t s) {
  Profiler& p = prof();
  if (!p.on.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> g(p.m);
  if (p.n >= p.cap) return;
  cudaEventRecord(p.ev[2 * p.n + 1], s);
  ++p.n;
}

}  // namespace stt

extern "C" {

int stt_profile_start(int capacity) {
  if (capacity < 1 || capacity > (1 << 20)) return STT_ERR_INVALID_ARG;
  stt::Profiler& p = stt::prof();
  std::lock_guard<std::mutex> g(p.m);
  if (p.on.load()) return STT_ERR_INVALID_ARG;
  p.ev.assign(2 * (size_t)capacity, nullptr);
  for (auto& e : p.ev)
    if (cudaEventCreate(&e) != cudaSuccess) return STT_ERR_CUDA;
  p.ids.assign((size_t)capacity, 0);
  p.n = 0;
  p.cap = capacity;
  p.dropped = 0;
  p.on.store(true);
  return STT_OK;
}

int stt_profile_stop(int* n, int* kernel_ids, float* ms, int capacity) {
  if (!n) return STT_ERR_INVALID_ARG;
  stt::Profiler& p = stt::prof();
  std::lock_guard<std::mutex> g(p.m);
  if (!p.on.load()) return STT_ERR_INVALID_ARG;
  p.on.store(false);
  int st = STT_OK;
  const int count = p.n < capacity ? p.n : capacity;
  for (int i = 0; i < count; ++i) {
    if (cudaEventSynchronize(p.ev[2 * i + 1]) != cudaSuccess) st = STT_ERR_CUDA;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, p.ev[2 * i], p.ev[2 * i + 1]) != cudaSuccess) st = STT_ERR_CUDA;
    if (kernel_ids) kernel_ids[i] = p.ids[i];
    if (ms) ms[i] = t;
  }
  for (auto e : p.ev) cudaEventDestroy(e);
  p.ev.clear();
  *n = count;
  return st;
}

const char* stt_kernel_name(int kernel_id) {
  switch (kernel_id) {
    case STT_KERNEL_SOFT_CE: return "soft_ce";
    case STT_KERNEL_SOFT_CE_LOSS_SUM: return "soft_ce_loss_sum";
    case STT_KERNEL_ATTN_FWD: return "attn_fwd";
    case STT_KERNEL_ATTN_BWD_PREP: return "attn_bwd_prep";
    case STT_KERNEL_ATTN_BWD_CAUSAL: return "attn_bwd_causal";
    case STT_KERNEL_ATTN_BWD_CAST: return "attn_bwd_cast";
    case STT_KERNEL_SOFT_CE_VARIANT: return "soft_ce_variant";
    case STT_KERNEL_VERIFY: return "verify";
    case STT_KERNEL_LM_HEAD_CE: return "lm_head_ce";
    default: return "unknown";
  }
}

}  // extern "C"
