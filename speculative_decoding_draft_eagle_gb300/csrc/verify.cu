// verify.cu -- speculative-decoding verification by rejection sampling (the
// "FlashSpec" practice page, §3.4 "验证器的具体实现"): for each sequence the draft
// tokens x_0..x_{gamma-1} are tested in order, x_i kept with probability
// min(1, p_t[x_i] / p_d[x_i]); at the first rejection one token is drawn from
// norm(max(0, p_t - p_d)) at that position and the sequence stops.
//
// One thread-block cluster of C CTAs per sequence; CTA c owns a slice of the
// vocabulary.  Warp 0 of every CTA makes all gamma tests at once (lane i loads
// p_t[i, x_i] and p_d[i, x_i] and tests u_i p_d < p_t in fp64, exact for fp32
// inputs); a ballot gives the first rejection, the same in every CTA, so a
// sequence whose tokens are all accepted reads nothing more.  At a rejection
// the draw is an inverse CDF over exact integer weights, so the token it
// decides does not depend on the order of any sum: the residual
// r_v = min(1, max(0, p_t[v] - p_d[v])) (difference rounded to fp32) becomes
// q_v = floor(r_v 2^s), s = 62 - bitlen(V), and every running sum is an exact
// int64 below 2^63.  Each CTA streams its slice of both rows once (coalesced
// 16-byte loads), keeps the fp32 residuals in shared memory and sums its q;
// the C slice sums are exchanged through distributed shared memory, giving the
// total Q and each slice's prefix; the threshold is t = floor(u24 Q / 2^24)
// (u24 = floor(u 2^24), a 128-bit product); only the CTA whose prefix range
// holds t scans its slice (from shared memory: one block-wide scan of the
// threads' contiguous runs, then the thread whose run holds t walks it) for
// the smallest y whose running sum exceeds t.  fp64 is kept off the rows:
// its rate on this GPU is a small fraction of fp32's.
#include <cstdint>

#include "../../include/stt.h"
#include "internal.h"
#include "ptx.cuh"

namespace stt {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 16;
constexpr int kSliceTarget = 16384;   // preferred elements per CTA (64 KB of residuals)
constexpr int kSliceMax = 50 * 1024;  // elements per CTA at most (200 KB)

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
  int shift;               // s = 62 - bitlen(V): weights are floor(w 2^s)
  int C;                   // CTAs per sequence (cluster size)
  int slice;               // elements per CTA (a multiple of 4)
};

__device__ __forceinline__ long long warp_sum_ll(long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// The fp32 weight of an element: the residual p_t - p_d rounded to fp32, or
// p_t itself when `target`, clamped to [0, 1].
__device__ __forceinline__ float fweight(float pt, float pd, bool target) {
  const float w = target ? pt : __fsub_rn(pt, pd);
  return fminf(1.0f, fmaxf(0.0f, w));
}
__device__ __forceinline__ long long quant(float w, float scale) {
  return __float2ll_rz(__fmul_rn(w, scale));  // exact: scale is a power of two
}

// Block-wide sum of one int64 per thread (every thread gets it).
__device__ __forceinline__ long long block_sum(long long v, long long* s_warp) {
  v = warp_sum_ll(v);
  if ((threadIdx.x & 31) == 0) s_warp[threadIdx.x >> 5] = v;
  __syncthreads();
  long long all = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) all += s_warp[w];
  __syncthreads();
  return all;
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
  __syncthreads();
  *total = all;
  return before + incl - v;
}

// Sum of the quantised weights of this CTA's slice [0, len), read from global
// memory; the fp32 weights are kept in shared memory for the scan.
template <bool VEC>
__device__ __forceinline__ long long slice_weights(const float* pt, const float* pd, int len,
                                                   bool target, float scale, float* sw,
                                                   long long* s_warp) {
  long long s = 0;
  if constexpr (VEC) {
    const float4* t4 = reinterpret_cast<const float4*>(pt);
    const float4* d4 = reinterpret_cast<const float4*>(pd);
    float4* w4 = reinterpret_cast<float4*>(sw);
    const int n4 = len / 4;
    // kBatch float4 of each row in flight per thread (half a slice of
    // kSliceTarget elements per batch; registers for two CTAs per SM)
    constexpr int kBatch = kSliceTarget / 8 / kThreads;
    for (int base = 0; base < n4; base += kBatch * kThreads) {
      float4 a[kBatch], c[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int i = base + u * kThreads + threadIdx.x;
        if (i < n4) {
          a[u] = __ldg(t4 + i);
          c[u] = __ldg(d4 + i);
        }
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int i = base + u * kThreads + threadIdx.x;
        if (i < n4) {
          const float4 w = make_float4(fweight(a[u].x, c[u].x, target), fweight(a[u].y, c[u].y, target),
                                       fweight(a[u].z, c[u].z, target), fweight(a[u].w, c[u].w, target));
          w4[i] = w;
          s += quant(w.x, scale) + quant(w.y, scale) + quant(w.z, scale) + quant(w.w, scale);
        }
      }
    }
  } else {
    for (int i = threadIdx.x; i < len; i += kThreads) {
      const float w = fweight(__ldg(pt + i), __ldg(pd + i), target);
      sw[i] = w;
      s += quant(w, scale);
    }
  }
  return block_sum(s, s_warp);
}

template <bool VEC>
__global__ void __launch_bounds__(kThreads, 2) verify_kernel(const VerifyParams P) {
  extern __shared__ __align__(16) float sw[];  // this CTA's fp32 weights
  __shared__ int s_rej;
  __shared__ long long s_warp[kWarps];
  __shared__ __align__(16) long long s_sum;   // read by the other CTAs of the cluster

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int C = P.C;
  const int rank = C > 1 ? (int)cluster_ctarank() : 0;
  const long long b = blockIdx.x / C;
  const int gamma = P.gamma;
  const long long V = P.V;

  // ---- the gamma acceptance tests, one lane each (the same in every CTA)
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
    if (lane == 0) s_rej = m ? __ffs((int)m) - 1 : gamma;
  }
  __syncthreads();
  const int r = s_rej;
  if (rank == 0) {
    if (tid < gamma) P.out[b * gamma + tid] = tid < r ? P.tokens[b * gamma + tid] : -1;
    if (tid == 0) P.n_acc[b] = r;
  }
  if (r == gamma) return;  // the same in every CTA of the cluster: no exchange follows

  // ---- the draw at position r
  const long long begin = (long long)rank * P.slice;
  const long long rem = V - begin;
  const int len = rem <= 0 ? 0 : (rem < P.slice ? (int)rem : P.slice);
  const float* pt_row = P.p_t + (b * gamma + r) * V + begin;
  const float* pd_row = P.p_d + (b * gamma + r) * V + begin;
  const float scale = __uint_as_float((uint32_t)(127 + P.shift) << 23);  // 2^s
  bool target = false;
  long long Q = 0, prefix = 0, mine = 0;
  for (int pass = 0; pass < 2; ++pass) {
    mine = slice_weights<VEC>(pt_row, pd_row, len, target, scale, sw, s_warp);
    Q = mine;
    prefix = 0;
    if (C > 1) {
      if (tid == 0) s_sum = mine;
      cluster_arrive_release();
      cluster_wait_acquire();
      Q = 0;
      for (int c = 0; c < C; ++c) {
        const uint32_t a = mapa_shared(smem_u32(&s_sum), (uint32_t)c);
        long long v;
        asm volatile("ld.shared::cluster.b64 %0, [%1];" : "=l"(v) : "r"(a) : "memory");
        if (c < rank) prefix += v;
        Q += v;
      }
      // every CTA has read every slice sum before s_sum is written again or a
      // CTA exits
      cluster_arrive_release();
      cluster_wait_acquire();
    }
    if (Q > 0 || target) break;
    target = true;  // the residual is empty: draw from p_t itself
  }
  if (Q == 0) {  // nothing to draw from (an all-zero target row)
    if (rank == 0 && tid == 0) P.out[b * gamma + r] = -1;
    return;
  }
  // t = floor(u24 Q / 2^24) with u24 = floor(u 2^24), from the 128-bit product
  const unsigned long long u24 =
      (unsigned long long)__float2ll_rz(__fmul_rn(P.u_sample[b], 16777216.0f));
  const unsigned long long lo = u24 * (unsigned long long)Q;
  const unsigned long long hi = __umul64hi(u24, (unsigned long long)Q);
  const long long thresh = (long long)((hi << 40) | (lo >> 24));
  if (!(prefix <= thresh && thresh < prefix + mine)) return;  // not in this slice

  // This CTA holds the crossing: every thread sums a contiguous run of the
  // slice, one block-wide scan places the runs, and the thread whose run holds
  // the threshold walks it.
  __syncthreads();  // the weights in shared memory are complete
  const int per = (len + kThreads - 1) / kThreads;
  const int i0 = tid * per, i1 = min(len, i0 + per);
  long long run = 0;
  for (int i = i0; i < i1; ++i) run += quant(sw[i], scale);
  long long total;
  const long long before = prefix + block_scan_excl(run, s_warp, &total);
  if (before <= thresh && thresh < before + run) {
    long long acc = before;
    for (int i = i0; i < i1; ++i) {
      acc += quant(sw[i], scale);
      if (acc > thresh) {
        P.out[b * gamma + r] = (int)(begin + i);
        break;
      }
    }
  }
}

}  // namespace

cudaError_t verify_launch(const float* p_t, const float* p_d, const int32_t* tokens,
                          const float* u_accept, const float* u_sample, int B, int gamma,
                          int64_t V, int32_t* n_acc, int32_t* out, cudaStream_t s) {
  int bits = 0;
  for (long long v = V; v > 0; v >>= 1) ++bits;
  long long C = (V + kSliceTarget - 1) / kSliceTarget;
  if (C < 1) C = 1;
  if (C > kMaxCluster) C = kMaxCluster;
  long long slice = ((V + C - 1) / C + 3) / 4 * 4;
  while (C > 1 && (C - 1) * slice >= V) {
    --C;
    slice = ((V + C - 1) / C + 3) / 4 * 4;
  }
  if (slice > kSliceMax) return cudaErrorNotSupported;
  if ((long long)B * C > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const bool vec = (V % 4 == 0) && ((reinterpret_cast<uintptr_t>(p_t) & 15u) == 0) &&
                   ((reinterpret_cast<uintptr_t>(p_d) & 15u) == 0);
  VerifyParams P{p_t, p_d, tokens, u_accept, u_sample, n_acc, out, (long long)V, gamma, 62 - bits,
                 (int)C, (int)slice};
  void (*kern)(const VerifyParams) = vec ? verify_kernel<true> : verify_kernel<false>;
  const int smem = (int)(slice * 4);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if (C > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(B * C), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_before(s, STT_KERNEL_VERIFY);
  e = cudaLaunchKernelEx(&cfg, kern, P);
  prof_after(s);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace stt
