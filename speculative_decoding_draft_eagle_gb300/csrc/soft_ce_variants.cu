// soft_ce_variants.cu -- the in-place soft-CE in the forms the formula admits
// beyond fp32 logits with a per-row g (SpecForge review, §三 "内存高效梯度计算":
// s = sum(p * g), z <- -(p * g - pi * s); §四 "掩码 Softmax 损失" /
// "原地反向传播"):
//   * bf16 logits z and targets p (the gradient is written back over z in
//     bf16, rounded once to nearest even; every sum is taken in fp32);
//   * a per-element upstream gradient G of the logits' shape (fp32 [N, V]):
//         s_r = sum_v p G,  z <- pi s - p G,
//         row_loss_r = sum_v G p (lse_r - z_rv),  L = sum_r row_loss_r.
//
// HBM-bound like the fp32 kernel: z and p (and G) are read once and z is
// written once.  One row per thread-block cluster of C CTAs: each CTA pulls its
// slice of the row into shared memory with bulk copies (chunked, so the first
// pass starts when the first chunk lands), reduces it to (max, sum exp, S1,
// S2) -- S1 = sum p (per-row g) or sum p G, S2 = sum p z or sum p G z --
// exchanges the partials through distributed shared memory, and streams the
// gradient out of the on-chip copy.  Rows with a per-row g of 0 are never
// read: their gradient is exactly 0.  Rows or slices that are not 16-byte
// aligned take element-wise loads with the same arithmetic.
#include <cmath>
#include <cstdint>

#include "../../include/stt.h"
#include "internal.h"
#include "ptx.cuh"

namespace stt {
namespace {

constexpr int kVThreads = 256;
constexpr int kVWarps = kVThreads / 32;
constexpr int kVMaxCluster = 16;
constexpr int kVMaxChunks = 8;
constexpr int kVSmemMax = 200 * 1024;     // shared bytes per CTA for the slice
constexpr int kVSmemTarget = 96 * 1024;   // preferred, so two CTAs fit on an SM
constexpr float kLog2eV = 1.4426950408889634f;

struct CeVParams {
  void* z;
  const void* p;
  const float* g;  // [N] per-row, or [N, V] per-element
  float* row_loss;
  float* wl;
  long long N, V;
  int C;
  int slice;   // elements of a row per CTA (a multiple of 8)
  int chunk;   // elements per bulk-copy chunk (a multiple of 8)
};

__device__ __forceinline__ float warp_max_v(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum_v(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Four consecutive elements as floats, from shared memory.
template <bool BF16>
__device__ __forceinline__ float4 ld4(const unsigned char* base, int i) {
  if constexpr (BF16) {
    const uint2 u = *reinterpret_cast<const uint2*>(base + (size_t)i * 2);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
  } else {
    return *reinterpret_cast<const float4*>(base + (size_t)i * 4);
  }
}
template <bool BF16>
__device__ __forceinline__ float ld1(const unsigned char* base, int i) {
  if constexpr (BF16) {
    const uint16_t u = *reinterpret_cast<const uint16_t*>(base + (size_t)i * 2);
    return __uint_as_float((uint32_t)u << 16);
  } else {
    return *reinterpret_cast<const float*>(base + (size_t)i * 4);
  }
}
__device__ __forceinline__ uint32_t bf16_bits_rn(float x) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  return (uint32_t)*reinterpret_cast<const uint16_t*>(&h);
}

// Four gradient values to global memory (streaming stores).
template <bool BF16>
__device__ __forceinline__ void st4(void* zrow, long long i, float4 v) {
  if constexpr (BF16) {
    const uint2 u = make_uint2(bf16_bits_rn(v.x) | (bf16_bits_rn(v.y) << 16),
                               bf16_bits_rn(v.z) | (bf16_bits_rn(v.w) << 16));
    __stcs(reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(zrow) + i), u);
  } else {
    st_global_cs_f4(static_cast<float*>(zrow) + i, v);
  }
}
template <bool BF16>
__device__ __forceinline__ void st1(void* zrow, long long i, float v) {
  if constexpr (BF16) {
    static_cast<__nv_bfloat16*>(zrow)[i] = __float2bfloat16_rn(v);
  } else {
    static_cast<float*>(zrow)[i] = v;
  }
}

// BF16: z and p are bf16.  GEL: g is per element.  BULK: 16-byte aligned
// rows and slices (bulk copies, 4-wide vector access).
template <bool BF16, bool GEL, bool BULK>
__global__ void __launch_bounds__(kVThreads) soft_ce_variant_kernel(const CeVParams P) {
  constexpr int ESZ = BF16 ? 2 : 4;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ uint64_t bars[kVMaxChunks];
  __shared__ float red[3][kVWarps];
  __shared__ float redm[kVWarps];
  __shared__ __align__(16) float stats[4];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = P.C;
  const uint32_t rank = (C > 1) ? cluster_ctarank() : 0u;
  const long long row = blockIdx.x / C;
  const long long begin = (long long)rank * P.slice;
  const long long rem = P.V - begin;
  const int len = rem <= 0 ? 0 : (rem < P.slice ? (int)rem : P.slice);
  unsigned char* zrow_b = static_cast<unsigned char*>(P.z) + (row * P.V + begin) * ESZ;
  const unsigned char* prow_b = static_cast<const unsigned char*>(P.p) + (row * P.V + begin) * ESZ;
  const float* grow = GEL ? P.g + row * P.V + begin : nullptr;
  const float g_row = GEL ? 1.0f : __ldg(P.g + row);

  if (!GEL && g_row == 0.0f) {
    // Masked row: gradient exactly 0, nothing read.
    if (BULK) {
      for (int i = tid * 4; i < len; i += kVThreads * 4)
        st4<BF16>(zrow_b, i, make_float4(0.f, 0.f, 0.f, 0.f));
    } else {
      for (int i = tid; i < len; i += kVThreads) st1<BF16>(zrow_b, i, 0.f);
    }
    if (rank == 0 && tid == 0) {
      if (P.row_loss) P.row_loss[row] = 0.0f;
      P.wl[row] = 0.0f;
    }
    return;
  }

  unsigned char* zs = smem_raw;
  unsigned char* ps = zs + (size_t)P.slice * ESZ;
  float* gs = reinterpret_cast<float*>(ps + (size_t)P.slice * ESZ);
  const int nchunks = len > 0 ? (len + P.chunk - 1) / P.chunk : 0;

  if (BULK) {
    if (tid == 0) {
      for (int c = 0; c < nchunks; ++c) mbar_init(&bars[c], 1);
      fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
      for (int c = 0; c < nchunks; ++c) {
        const int c0 = c * P.chunk;
        const int n = min(P.chunk, len - c0);
        const uint32_t bytes = (uint32_t)n * ESZ;
        mbar_arrive_expect_tx(&bars[c], 2u * bytes + (GEL ? (uint32_t)n * 4u : 0u));
        bulk_load(zs + (size_t)c0 * ESZ, zrow_b + (size_t)c0 * ESZ, bytes, &bars[c]);
        bulk_load(ps + (size_t)c0 * ESZ, prow_b + (size_t)c0 * ESZ, bytes, &bars[c]);
        if (GEL) bulk_load(gs + c0, grow + c0, (uint32_t)n * 4u, &bars[c]);
      }
    }
  } else {
    for (int i = tid; i < len; i += kVThreads) {
      if constexpr (BF16) {
        reinterpret_cast<uint16_t*>(zs)[i] = reinterpret_cast<const uint16_t*>(zrow_b)[i];
        reinterpret_cast<uint16_t*>(ps)[i] = reinterpret_cast<const uint16_t*>(prow_b)[i];
      } else {
        reinterpret_cast<float*>(zs)[i] = reinterpret_cast<const float*>(zrow_b)[i];
        reinterpret_cast<float*>(ps)[i] = reinterpret_cast<const float*>(prow_b)[i];
      }
      if (GEL) gs[i] = grow[i];
    }
    __syncthreads();
  }

  // Pass 1: max z, S1 = sum p (G), S2 = sum p (G) z.
  float m = -INFINITY, s1 = 0.f, s2 = 0.f;
  bool ok = true;
  for (int c = 0; c < nchunks; ++c) {
    const int c0 = c * P.chunk;
    const int c1 = min(len, c0 + P.chunk);
    if (BULK) {
      ok = mbar_wait(&bars[c], 0, STT_DEVERR_CE_WAIT) && ok;
      for (int i = c0 + tid * 4; i < c1; i += kVThreads * 4) {
        const float4 zv = ld4<BF16>(zs, i);
        float4 pv = ld4<BF16>(ps, i);
        if (GEL) {
          const float4 gv = *reinterpret_cast<const float4*>(gs + i);
          pv = make_float4(pv.x * gv.x, pv.y * gv.y, pv.z * gv.z, pv.w * gv.w);
        }
        m = fmaxf(m, fmaxf(fmaxf(zv.x, zv.y), fmaxf(zv.z, zv.w)));
        s1 += (pv.x + pv.y) + (pv.z + pv.w);
        s2 = fmaf(pv.x, zv.x, s2);
        s2 = fmaf(pv.y, zv.y, s2);
        s2 = fmaf(pv.z, zv.z, s2);
        s2 = fmaf(pv.w, zv.w, s2);
      }
    } else {
      for (int i = c0 + tid; i < c1; i += kVThreads) {
        const float zv = ld1<BF16>(zs, i);
        const float pv = ld1<BF16>(ps, i) * (GEL ? gs[i] : 1.0f);
        m = fmaxf(m, zv);
        s1 += pv;
        s2 = fmaf(pv, zv, s2);
      }
    }
  }
  m = warp_max_v(m);
  if (lane == 0) redm[warp] = m;
  __syncthreads();
  m = redm[0];
#pragma unroll
  for (int w = 1; w < kVWarps; ++w) m = fmaxf(m, redm[w]);

  // Pass 2: sum exp(z - m).
  float l = 0.f;
  if (len > 0 && ok) {
    const float mb = m * kLog2eV;
    if (BULK) {
      for (int i = tid * 4; i < len; i += kVThreads * 4) {
        const float4 zv = ld4<BF16>(zs, i);
        l += ex2(fmaf(zv.x, kLog2eV, -mb)) + ex2(fmaf(zv.y, kLog2eV, -mb)) +
             ex2(fmaf(zv.z, kLog2eV, -mb)) + ex2(fmaf(zv.w, kLog2eV, -mb));
      }
    } else {
      for (int i = tid; i < len; i += kVThreads) l += ex2(fmaf(ld1<BF16>(zs, i), kLog2eV, -mb));
    }
  }
  l = warp_sum_v(l);
  s1 = warp_sum_v(s1);
  s2 = warp_sum_v(s2);
  if (lane == 0) {
    red[0][warp] = l;
    red[1][warp] = s1;
    red[2][warp] = s2;
  }
  __syncthreads();
  l = s1 = s2 = 0.f;
#pragma unroll
  for (int w = 0; w < kVWarps; ++w) {
    l += red[0][w];
    s1 += red[1][w];
    s2 += red[2][w];
  }

  // Combine the C slices of the row through distributed shared memory.
  float M = m, Ls = l, S1 = s1, S2 = s2;
  if (C > 1) {
    if (tid == 0) {
      stats[0] = m;
      stats[1] = l;
      stats[2] = s1;
      stats[3] = s2;
    }
    cluster_arrive_release();
    cluster_wait_acquire();
    float4 part[kVMaxCluster];
    M = -INFINITY;
    for (int r = 0; r < C; ++r) {
      part[r] = ld_shared_cluster_f4(mapa_shared(smem_u32(stats), (uint32_t)r));
      M = fmaxf(M, part[r].x);
    }
    Ls = S1 = S2 = 0.f;
    for (int r = 0; r < C; ++r) {
      if (part[r].y > 0.f) Ls += part[r].y * ex2((part[r].x - M) * kLog2eV);
      S1 += part[r].z;
      S2 += part[r].w;
    }
    cluster_arrive_release();  // done reading the others' statistics
  }
  const float lse = M + logf(Ls);
  const float lse2 = lse * kLog2eV;
  // s = sum p G (per element) or g sum p (per row); the gradient is pi s - p G.
  const float s = GEL ? S1 : g_row * S1;

  // Pass 3: the gradient from the on-chip copy.
  if (ok) {
    if (BULK) {
      for (int i = tid * 4; i < len; i += kVThreads * 4) {
        const float4 zv = ld4<BF16>(zs, i);
        float4 pg = ld4<BF16>(ps, i);
        if (GEL) {
          const float4 gv = *reinterpret_cast<const float4*>(gs + i);
          pg = make_float4(pg.x * gv.x, pg.y * gv.y, pg.z * gv.z, pg.w * gv.w);
        } else {
          pg = make_float4(pg.x * g_row, pg.y * g_row, pg.z * g_row, pg.w * g_row);
        }
        float4 o;
        o.x = fmaf(ex2(fmaf(zv.x, kLog2eV, -lse2)), s, -pg.x);
        o.y = fmaf(ex2(fmaf(zv.y, kLog2eV, -lse2)), s, -pg.y);
        o.z = fmaf(ex2(fmaf(zv.z, kLog2eV, -lse2)), s, -pg.z);
        o.w = fmaf(ex2(fmaf(zv.w, kLog2eV, -lse2)), s, -pg.w);
        st4<BF16>(zrow_b, i, o);
      }
    } else {
      for (int i = tid; i < len; i += kVThreads) {
        const float pg = ld1<BF16>(ps, i) * (GEL ? gs[i] : g_row);
        st1<BF16>(zrow_b, i, fmaf(ex2(fmaf(ld1<BF16>(zs, i), kLog2eV, -lse2)), s, -pg));
      }
    }
  }
  if (rank == 0 && tid == 0) {
    // per row: l_r = lse Sp - Spz, weighted by g; per element: already weighted
    const float ell = fmaf(lse, S1, -S2);
    if (P.row_loss) P.row_loss[row] = ell;
    P.wl[row] = GEL ? ell : g_row * ell;
  }
  if (C > 1) cluster_wait_acquire();
}

}  // namespace

CeVariantPlan soft_ce_variant_plan(const void* z, const void* p, const float* g, int64_t V,
                                   uint32_t flags) {
  const bool bf16 = (flags & kCeBf16) != 0, gel = (flags & kCeGPerElement) != 0;
  const int esz = bf16 ? 2 : 4;
  const int per_elem = 2 * esz + (gel ? 4 : 0);  // shared bytes per element
  CeVariantPlan plan{};
  const uintptr_t a = reinterpret_cast<uintptr_t>(z) | reinterpret_cast<uintptr_t>(p) |
                      (gel ? reinterpret_cast<uintptr_t>(g) : 0);
  plan.bulk = ((a & 15u) == 0) && (V % 8 == 0);
  long long C = ((long long)per_elem * V + kVSmemTarget - 1) / kVSmemTarget;
  if (C < 1) C = 1;
  if (C > kVMaxCluster) C = kVMaxCluster;
  long long slice = ((V + C - 1) / C + 7) / 8 * 8;
  while (C > 1 && (C - 1) * slice >= V) {
    --C;
    slice = ((V + C - 1) / C + 7) / 8 * 8;
  }
  plan.C = (int)C;
  plan.slice = (int)slice;
  plan.smem = (int)(slice * per_elem);
  long long chunk = (slice + kVMaxChunks - 1) / kVMaxChunks;
  chunk = (chunk + 7) / 8 * 8;
  if (chunk < 1024) chunk = 1024;
  plan.chunk = (int)chunk;
  plan.ok = plan.smem <= kVSmemMax;
  return plan;
}

cudaError_t soft_ce_variant_launch(const CeVariantPlan& plan, uint32_t flags, void* z,
                                   const void* p, const float* g, int64_t N, int64_t V,
                                   float* row_loss, float* loss, float* wl, cudaStream_t s) {
  const bool bf16 = (flags & kCeBf16) != 0, gel = (flags & kCeGPerElement) != 0;
  // Aligned rows that fit the persistent cluster kernel take it; the rest the
  // one-row-per-cluster kernel below.
  const cudaError_t ep = soft_ce_variant_persistent_launch(flags, z, p, g, N, V, row_loss, loss, wl, s);
  if (ep != cudaErrorNotSupported) return ep;
  if (N > 0) {
    if (N * (long long)plan.C > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    CeVParams P{z, p, g, row_loss, wl, (long long)N, (long long)V, plan.C, plan.slice, plan.chunk};
    void (*kern)(const CeVParams);
    if (bf16)
      kern = gel ? (plan.bulk ? soft_ce_variant_kernel<true, true, true>
                              : soft_ce_variant_kernel<true, true, false>)
                 : (plan.bulk ? soft_ce_variant_kernel<true, false, true>
                              : soft_ce_variant_kernel<true, false, false>);
    else
      kern = gel ? (plan.bulk ? soft_ce_variant_kernel<false, true, true>
                              : soft_ce_variant_kernel<false, true, false>)
                 : (plan.bulk ? soft_ce_variant_kernel<false, false, true>
                              : soft_ce_variant_kernel<false, false, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, plan.smem);
    if (e != cudaSuccess) return e;
    if (plan.C > 8) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(N * plan.C), 1, 1);
    cfg.blockDim = dim3(kVThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)plan.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)plan.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    prof_before(s, STT_KERNEL_SOFT_CE_VARIANT);
    e = cudaLaunchKernelEx(&cfg, kern, P);
    if (e != cudaSuccess) {
      prof_after(s);
      return e;
    }
  } else {
    prof_before(s, STT_KERNEL_SOFT_CE_VARIANT);
  }
  const cudaError_t e2 = soft_ce_loss_sum_launch(wl, N, loss, s);
  prof_after(s);
  if (e2 != cudaSuccess) return e2;
  return cudaGetLastError();
}

static_assert(kVMaxChunks * 1024 >= 8, "chunks");

}  // namespace stt
