// verify.cu -- speculative-decoding verification by rejection sampling (the
// "FlashSpec" practice page, §3.4 "验证器的具体实现"): for each sequence the draft
// tokens x_0..x_{gamma-1} are tested in order, x_i kept with probability
// min(1, p_t[x_i] / p_d[x_i]); at the first rejection one token is drawn from
// norm(max(0, p_t - p_d)) at that position and the sequence stops.
//
// One CTA per sequence.  Warp 0 makes all gamma tests at once (lane i loads
// p_t[i, x_i] and p_d[i, x_i] and tests u_i p_d < p_t in fp64, exact for fp32
// inputs); a ballot gives the first rejection.  Only then is a row read: the
// CTA sums the residual r_v = max(0, p_t[v] - p_d[v]) in fp64 (one coalesced
// pass over both rows), and walks the row again in tiles of 4 elements per
// thread with a block-wide fp64 scan until the running sum passes
// u_sample * sum(r): the inverse-CDF draw.  The second pass reads the rows
// from L2 and stops at the drawn token.
#include <cstdint>

#include "../../include/stt.h"
#include "internal.h"

namespace stt {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;

struct VerifyParams {
  const float* p_t;        // [B, gamma, V]
  const float* p_d;        // [B, gamma, V]
  const int32_t* tokens;   // [B, gamma]
  const float* u_accept;   // [B, gamma]
  const float* u_sample;   // [B]
  int32_t* n_acc;          // [B]
  int32_t* out;            // [B, gamma]
  long long V;
  int gamma;
};

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Residual weight of element v (fp64, exact for fp32 inputs); with `target`
// the weights are p_t itself (the draw when the residual sums to zero).
__device__ __forceinline__ double weight(float pt, float pd, bool target) {
  const double d = target ? (double)pt : (double)pt - (double)pd;
  return d > 0.0 ? d : 0.0;
}

// Inclusive block-wide scan of one fp64 value per thread; returns the
// exclusive prefix and stores the block total in *total (all threads).
__device__ __forceinline__ double block_scan_excl(double v, double* s_warp, double* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  double incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  double before = 0.0, all = 0.0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const double x = s_warp[w];
    if (w < warp) before += x;
    all += x;
  }
  __syncthreads();  // s_warp is reused by the next call
  *total = all;
  return before + incl - v;
}

template <bool VEC>
__global__ void __launch_bounds__(kThreads) verify_kernel(const VerifyParams P) {
  __shared__ int s_rej;
  __shared__ double s_warp[kWarps];
  __shared__ double s_red[kWarps];
  __shared__ int s_last;
  __shared__ int s_found;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long b = blockIdx.x;
  const int gamma = P.gamma;
  const long long V = P.V;

  // ---- the gamma acceptance tests, one lane each
  if (warp == 0) {
    bool reject = false;
    if (lane < gamma) {
      const long long i = b * gamma + lane;
      const int x = P.tokens[i];
      float pt = 0.f, pd = 0.f;
      if (x >= 0 && x < V) {  // a token outside the vocabulary is never accepted
        pt = __ldg(P.p_t + i * V + x);
        pd = __ldg(P.p_d + i * V + x);
      }
      const double u = (double)P.u_accept[i];
      const bool accept = pd > 0.f ? (u * (double)pd < (double)pt) : (pt > 0.f);
      reject = !accept;
    }
    const unsigned m = __ballot_sync(0xffffffffu, reject);
    if (lane == 0) {
      s_rej = m ? __ffs((int)m) - 1 : gamma;
      s_last = -1;
      s_found = 0;
    }
  }
  __syncthreads();
  const int r = s_rej;
  if (tid < gamma) P.out[b * gamma + tid] = tid < r ? P.tokens[b * gamma + tid] : -1;
  if (tid == 0) P.n_acc[b] = r;
  if (r == gamma) return;

  // ---- the draw at position r
  const float* pt_row = P.p_t + (b * gamma + r) * V;
  const float* pd_row = P.p_d + (b * gamma + r) * V;
  bool target = false;
  double R = 0.0;
  for (int pass = 0; pass < 2; ++pass) {
    // sum of the weights, and the last index with a positive weight
    double s = 0.0;
    int last = -1;
    if constexpr (VEC) {
      const float4* t4 = reinterpret_cast<const float4*>(pt_row);
      const float4* d4 = reinterpret_cast<const float4*>(pd_row);
      for (long long i = tid; i < V / 4; i += kThreads) {
        const float4 a = __ldg(t4 + i), c = __ldg(d4 + i);
        const double w0 = weight(a.x, c.x, target), w1 = weight(a.y, c.y, target);
        const double w2 = weight(a.z, c.z, target), w3 = weight(a.w, c.w, target);
        s += (w0 + w1) + (w2 + w3);
        if (w3 > 0.0) last = (int)(4 * i + 3);
        else if (w2 > 0.0) last = (int)(4 * i + 2);
        else if (w1 > 0.0) last = (int)(4 * i + 1);
        else if (w0 > 0.0) last = (int)(4 * i);
      }
    } else {
      for (long long i = tid; i < V; i += kThreads) {
        const double w = weight(__ldg(pt_row + i), __ldg(pd_row + i), target);
        s += w;
        if (w > 0.0) last = (int)i;
      }
    }
    s = warp_sum_d(s);
    if (lane == 0) s_red[warp] = s;
    if (last >= 0) atomicMax(&s_last, last);
    __syncthreads();
    R = 0.0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) R += s_red[w];
    __syncthreads();
    if (R > 0.0 || target) break;
    target = true;  // the residual is empty: draw from p_t itself
    if (tid == 0) s_last = -1;
    __syncthreads();
  }
  const double thresh = (double)P.u_sample[b] * R;

  // Second walk: tiles of kThreads * E elements, block-wide scan per tile.
  constexpr int E = VEC ? 4 : 1;
  double running = 0.0;
  for (long long base = 0; base < V; base += (long long)kThreads * E) {
    const long long i0 = base + (long long)tid * E;
    double w[E];
#pragma unroll
    for (int e = 0; e < E; ++e) w[e] = 0.0;
    if (i0 < V) {
      if constexpr (VEC) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(pt_row + i0));
        const float4 c = __ldg(reinterpret_cast<const float4*>(pd_row + i0));
        w[0] = weight(a.x, c.x, target);
        w[1] = weight(a.y, c.y, target);
        w[2] = weight(a.z, c.z, target);
        w[3] = weight(a.w, c.w, target);
      } else {
        w[0] = weight(__ldg(pt_row + i0), __ldg(pd_row + i0), target);
      }
    }
    double mine = 0.0;
#pragma unroll
    for (int e = 0; e < E; ++e) mine += w[e];
    double tile_total;
    const double before = running + block_scan_excl(mine, s_warp, &tile_total);
    // the crossing lies in this thread's elements: before <= thresh < before + mine
    if (mine > 0.0 && before <= thresh && thresh < before + mine) {
      double acc = before;
      int y = -1;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        acc += w[e];
        if (y < 0 && acc > thresh) y = (int)(i0 + e);
      }
      if (y < 0) {  // rounding inside the thread's partial sum: its last positive element
#pragma unroll
        for (int e = 0; e < E; ++e)
          if (w[e] > 0.0) y = (int)(i0 + e);
      }
      P.out[b * gamma + r] = y;
      s_found = 1;
    }
    running += tile_total;
    __syncthreads();
    if (s_found) return;
  }
  // The threshold fell past the (block-order) total by rounding: the last
  // positive weight.
  if (tid == 0) P.out[b * gamma + r] = s_last;
}

}  // namespace

cudaError_t verify_launch(const float* p_t, const float* p_d, const int32_t* tokens,
                          const float* u_accept, const float* u_sample, int B, int gamma,
                          int64_t V, int32_t* n_acc, int32_t* out, cudaStream_t s) {
  VerifyParams P{p_t, p_d, tokens, u_accept, u_sample, n_acc, out, (long long)V, gamma};
  const bool vec = (V % 4 == 0) && ((reinterpret_cast<uintptr_t>(p_t) & 15u) == 0) &&
                   ((reinterpret_cast<uintptr_t>(p_d) & 15u) == 0);
  prof_before(s, STT_KERNEL_VERIFY);
  if (vec)
    verify_kernel<true><<<(unsigned)B, kThreads, 0, s>>>(P);
  else
    verify_kernel<false><<<(unsigned)B, kThreads, 0, s>>>(P);
  prof_after(s);
  return cudaGetLastError();
}

}  // namespace stt
