// verify.cu -- speculative-decoding verification by rejection sampling (the
// "FlashSpec" practice page, §3.4 "验证器的具体实现"): for each sequence the draft
// tokens x_0..x_{gamma-1} are tested in order, x_i kept with probability
// min(1, p_t[x_i] / p_d[x_i]); at the first rejection one token is drawn from
// norm(max(0, p_t - p_d)) at that position and the sequence stops.
//
// One CTA per sequence.  Warp 0 makes all gamma tests at once (lane i loads
// p_t[i, x_i] and p_d[i, x_i] and tests u_i p_d < p_t in fp64, exact for fp32
// inputs); a ballot gives the first rejection.  Only then is a row read.  The
// draw is an inverse CDF over exact integer weights, so the token it decides
// does not depend on the order of any floating-point sum: the residual
// r_v = min(1, max(0, p_t[v] - p_d[v])) (difference rounded to fp32) becomes
// q_v = floor(r_v 2^s), s = 62 - bitlen(V), so every running sum is an exact
// int64 below 2^63.  The CTA sums q in one coalesced pass over both rows, forms
// the threshold t = floor(u24 Q / 2^24) (u24 = floor(u 2^24), a 128-bit
// product), and walks the row again in tiles of 4 elements per thread with a
// block-wide int64 scan until the running sum passes t.  The second pass
// reads the rows from L2 and stops at the drawn token.  (fp64 is avoided on
// the row: its rate on this GPU is a small fraction of fp32's.)
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
  int shift;  // s = 62 - bitlen(V): weights are floor(w 2^s)
};

__device__ __forceinline__ long long warp_sum_ll(long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Quantised weight of element v: floor(min(1, max(0, w)) 2^s) with w the
// fp32 residual p_t - p_d (or p_t itself when `target`).
__device__ __forceinline__ long long qweight(float pt, float pd, bool target, float scale) {
  float w = target ? pt : __fsub_rn(pt, pd);
  w = fminf(1.0f, fmaxf(0.0f, w));
  return __float2ll_rz(__fmul_rn(w, scale));  // exact: scale is a power of two
}

// Exclusive block-wide scan of one int64 per thread; *total receives the sum.
__device__ __forceinline__ long long block_scan_excl(long long v, long long* s_warp,
                                                     long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  long long before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const long long x = s_warp[w];
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
  __shared__ long long s_warp[kWarps];
  __shared__ long long s_red[kWarps];
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
  const float scale = __uint_as_float((uint32_t)(127 + P.shift) << 23);  // 2^s
  bool target = false;
  long long Q = 0;
  for (int pass = 0; pass < 2; ++pass) {
    long long s = 0;
    if constexpr (VEC) {
      const float4* t4 = reinterpret_cast<const float4*>(pt_row);
      const float4* d4 = reinterpret_cast<const float4*>(pd_row);
      for (long long i = tid; i < V / 4; i += kThreads) {
        const float4 a = __ldg(t4 + i), c = __ldg(d4 + i);
        s += qweight(a.x, c.x, target, scale) + qweight(a.y, c.y, target, scale) +
             qweight(a.z, c.z, target, scale) + qweight(a.w, c.w, target, scale);
      }
    } else {
      for (long long i = tid; i < V; i += kThreads)
        s += qweight(__ldg(pt_row + i), __ldg(pd_row + i), target, scale);
    }
    s = warp_sum_ll(s);
    if (lane == 0) s_red[warp] = s;
    __syncthreads();
    Q = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) Q += s_red[w];
    __syncthreads();
    if (Q > 0 || target) break;
    target = true;  // the residual is empty: draw from p_t itself
  }
  if (Q == 0) {  // nothing to draw from (an all-zero target row)
    if (tid == 0) P.out[b * gamma + r] = -1;
    return;
  }
  // t = floor(u24 Q / 2^24) with u24 = floor(u 2^24), from the 128-bit product
  const unsigned long long u24 =
      (unsigned long long)__float2ll_rz(__fmul_rn(P.u_sample[b], 16777216.0f));
  const unsigned long long lo = u24 * (unsigned long long)Q;
  const unsigned long long hi = __umul64hi(u24, (unsigned long long)Q);
  const long long thresh = (long long)((hi << 40) | (lo >> 24));

  // Second walk: tiles of kThreads * E elements, block-wide scan per tile.
  constexpr int E = VEC ? 4 : 1;
  long long running = 0;
  for (long long base = 0; base < V; base += (long long)kThreads * E) {
    const long long i0 = base + (long long)tid * E;
    long long w[E];
#pragma unroll
    for (int e = 0; e < E; ++e) w[e] = 0;
    if (i0 < V) {
      if constexpr (VEC) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(pt_row + i0));
        const float4 c = __ldg(reinterpret_cast<const float4*>(pd_row + i0));
        w[0] = qweight(a.x, c.x, target, scale);
        w[1] = qweight(a.y, c.y, target, scale);
        w[2] = qweight(a.z, c.z, target, scale);
        w[3] = qweight(a.w, c.w, target, scale);
      } else {
        w[0] = qweight(__ldg(pt_row + i0), __ldg(pd_row + i0), target, scale);
      }
    }
    long long mine = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) mine += w[e];
    long long tile_total;
    const long long before = running + block_scan_excl(mine, s_warp, &tile_total);
    // the crossing lies in this thread's elements: before <= t < before + mine
    if (before <= thresh && thresh < before + mine) {
      long long acc = before;
      int y = -1;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        acc += w[e];
        if (y < 0 && acc > thresh) y = (int)(i0 + e);
      }
      P.out[b * gamma + r] = y;
      s_found = 1;
    }
    running += tile_total;
    __syncthreads();
    if (s_found) return;
  }
}

}  // namespace

cudaError_t verify_launch(const float* p_t, const float* p_d, const int32_t* tokens,
                          const float* u_accept, const float* u_sample, int B, int gamma,
                          int64_t V, int32_t* n_acc, int32_t* out, cudaStream_t s) {
  int bits = 0;
  for (long long v = V; v > 0; v >>= 1) ++bits;
  VerifyParams P{p_t, p_d, tokens, u_accept, u_sample, n_acc, out, (long long)V, gamma, 62 - bits};
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
