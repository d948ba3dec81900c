// soft_ce.cu -- masked soft-target softmax cross-entropy with the gradient
// written in place over the logits (SpecForge review, §三 "内存高效梯度计算",
// §四 "掩码 Softmax 损失" / "原地反向传播").
//
// Per row r:  m = max z, l = sum exp(z - m), lse = m + log l,
//             Sp = sum p, Spz = sum p z, loss_r = lse Sp - Spz,
//             s = g_r Sp, z <- exp(z - lse) s - p g_r.
//
// Design (HBM-bound: 12 bytes per element, read z, read p, write z):
//   * One row is split across a thread-block cluster of C CTAs; each CTA pulls
//     its slice of z and p into shared memory with bulk (TMA) copies, so every
//     byte of z and p is read from HBM exactly once.
//   * Each CTA reduces its slice to (max, sum exp, Sp, Spz); the C partials are
//     exchanged through distributed shared memory and combined with the usual
//     max-rescaling, so every CTA knows the row's lse.
//   * The gradient is streamed out with coalesced 16-byte stores.  Rows with
//     g = 0 are never read: their gradient is exactly zero and is written
//     directly.
//   * Per-row weighted losses g_r * loss_r go to the workspace; a one-CTA kernel
//     sums them in a fixed order, so the scalar loss is deterministic.
// Two kernels implement this.  soft_ce_persistent_kernel (16-byte aligned rows,
// slices of at most kPSliceMaxSplit elements) keeps one cluster per group of SMs
// resident and pipelines rows through it; soft_ce_kernel (any row, one cluster
// per row) covers the rest.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/stt.h"
#include "internal.h"
#include "ptx.cuh"

namespace stt {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 4096;     // elements per bulk-copy chunk (16 KB per array)
constexpr int kMaxChunks = 8;
constexpr int kSliceBudget = 81920;  // preferred shared bytes per CTA (two arrays)
constexpr int kSliceMax = 25600;     // elements per CTA at most (200 KB)
constexpr int kMaxCluster = 16;
constexpr float kLog2e = 1.4426950408889634f;

struct CeParams {
  float* z;
  const float* p;
  const float* g;
  float* row_loss;
  float* wl;
  long long N, V;
  int C;
  int slice;
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <bool kBulk>
__global__ void __launch_bounds__(kThreads) soft_ce_kernel(const CeParams P) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ uint64_t bars[kMaxChunks];
  __shared__ float red[3][kWarps];
  __shared__ float redm[kWarps];
  __shared__ __align__(16) float stats[4];

  const int tid = threadIdx.x;
  const int C = P.C;
  const uint32_t rank = (C > 1) ? cluster_ctarank() : 0u;
  const long long row = blockIdx.x / C;
  const long long begin = (long long)rank * P.slice;
  const long long rem = P.V - begin;
  const int len = rem <= 0 ? 0 : (rem < P.slice ? (int)rem : P.slice);
  float* zrow = P.z + row * P.V + begin;
  const float* prow = P.p + row * P.V + begin;
  const float g = __ldg(P.g + row);

  if (g == 0.0f) {
    // Masked row: gradient is exactly 0 and nothing needs to be read.
    if (kBulk) {
      const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int i = tid * 4; i < len; i += kThreads * 4) st_global_cs_f4(zrow + i, zero);
    } else {
      for (int i = tid; i < len; i += kThreads) zrow[i] = 0.0f;
    }
    if (rank == 0 && tid == 0) {
      if (P.row_loss) P.row_loss[row] = 0.0f;
      P.wl[row] = 0.0f;
    }
    return;
  }

  float* zs = reinterpret_cast<float*>(smem_raw);
  float* ps = zs + P.slice;
  const int nchunks = (len + kChunk - 1) / kChunk;

  if (kBulk) {
    if (tid == 0) {
      for (int c = 0; c < nchunks; ++c) mbar_init(&bars[c], 1);
      fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
      for (int c = 0; c < nchunks; ++c) {
        const int n = min(kChunk, len - c * kChunk);
        const uint32_t bytes = (uint32_t)n * 4u;
        mbar_arrive_expect_tx(&bars[c], 2u * bytes);
        bulk_load(zs + c * kChunk, zrow + c * kChunk, bytes, &bars[c]);
        bulk_load(ps + c * kChunk, prow + c * kChunk, bytes, &bars[c]);
      }
    }
  } else {
    for (int i = tid; i < len; i += kThreads) {
      zs[i] = zrow[i];
      ps[i] = prow[i];
    }
    __syncthreads();
  }

  // Pass 1: max, sum p, sum p*z over the slice.
  float m = -INFINITY, sp = 0.f, spz = 0.f;
  for (int c = 0; c < nchunks; ++c) {
    const int c0 = c * kChunk;
    const int c1 = min(len, c0 + kChunk);
    if (kBulk) {
      mbar_wait(&bars[c], 0, STT_DEVERR_CE_WAIT);
      for (int i = c0 + tid * 4; i < c1; i += kThreads * 4) {
        const float4 zv = *reinterpret_cast<const float4*>(zs + i);
        const float4 pv = *reinterpret_cast<const float4*>(ps + i);
        m = fmaxf(m, fmaxf(fmaxf(zv.x, zv.y), fmaxf(zv.z, zv.w)));
        sp += (pv.x + pv.y) + (pv.z + pv.w);
        spz = fmaf(pv.x, zv.x, spz);
        spz = fmaf(pv.y, zv.y, spz);
        spz = fmaf(pv.z, zv.z, spz);
        spz = fmaf(pv.w, zv.w, spz);
      }
    } else {
      for (int i = c0 + tid; i < c1; i += kThreads) {
        const float zv = zs[i], pv = ps[i];
        m = fmaxf(m, zv);
        sp += pv;
        spz = fmaf(pv, zv, spz);
      }
    }
  }
  const int warp = tid >> 5, lane = tid & 31;
  m = warp_max(m);
  if (lane == 0) redm[warp] = m;
  __syncthreads();
  m = redm[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) m = fmaxf(m, redm[w]);

  // Pass 2: sum exp(z - m) over the slice (exp as 2^(z log2e - m log2e)).
  float l = 0.f;
  if (len > 0) {
    const float mb = m * kLog2e;
    if (kBulk) {
      for (int i = tid * 4; i < len; i += kThreads * 4) {
        const float4 zv = *reinterpret_cast<const float4*>(zs + i);
        l += ex2(fmaf(zv.x, kLog2e, -mb)) + ex2(fmaf(zv.y, kLog2e, -mb)) +
             ex2(fmaf(zv.z, kLog2e, -mb)) + ex2(fmaf(zv.w, kLog2e, -mb));
      }
    } else {
      for (int i = tid; i < len; i += kThreads) l += ex2(fmaf(zs[i], kLog2e, -mb));
    }
  }
  l = warp_sum(l);
  sp = warp_sum(sp);
  spz = warp_sum(spz);
  if (lane == 0) {
    red[0][warp] = l;
    red[1][warp] = sp;
    red[2][warp] = spz;
  }
  __syncthreads();
  l = 0.f;
  sp = 0.f;
  spz = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    l += red[0][w];
    sp += red[1][w];
    spz += red[2][w];
  }

  // Combine the C slices of the row through distributed shared memory.
  float M = m, Ls = l, Sp = sp, Spz = spz;
  if (C > 1) {
    if (tid == 0) {
      stats[0] = m;
      stats[1] = l;
      stats[2] = sp;
      stats[3] = spz;
    }
    cluster_arrive_release();
    cluster_wait_acquire();
    float4 part[kMaxCluster];
    M = -INFINITY;
    for (int r = 0; r < C; ++r) {
      part[r] = ld_shared_cluster_f4(mapa_shared(smem_u32(stats), (uint32_t)r));
      M = fmaxf(M, part[r].x);
    }
    Ls = 0.f;
    Sp = 0.f;
    Spz = 0.f;
    for (int r = 0; r < C; ++r) {
      if (part[r].y > 0.f) Ls += part[r].y * ex2((part[r].x - M) * kLog2e);
      Sp += part[r].z;
      Spz += part[r].w;
    }
    // Done reading the other CTAs' statistics; the matching wait sits at the end.
    cluster_arrive_release();
  }
  const float lse = M + logf(Ls);
  const float lse2 = lse * kLog2e;
  const float s = g * Sp;

  // Pass 3: gradient from the on-chip copy, streamed to HBM.
  if (kBulk) {
    for (int i = tid * 4; i < len; i += kThreads * 4) {
      const float4 zv = *reinterpret_cast<const float4*>(zs + i);
      const float4 pv = *reinterpret_cast<const float4*>(ps + i);
      float4 o;
      o.x = fmaf(ex2(fmaf(zv.x, kLog2e, -lse2)), s, -pv.x * g);
      o.y = fmaf(ex2(fmaf(zv.y, kLog2e, -lse2)), s, -pv.y * g);
      o.z = fmaf(ex2(fmaf(zv.z, kLog2e, -lse2)), s, -pv.z * g);
      o.w = fmaf(ex2(fmaf(zv.w, kLog2e, -lse2)), s, -pv.w * g);
      st_global_cs_f4(zrow + i, o);
    }
  } else {
    for (int i = tid; i < len; i += kThreads)
      zrow[i] = fmaf(ex2(fmaf(zs[i], kLog2e, -lse2)), s, -ps[i] * g);
  }
  if (rank == 0 && tid == 0) {
    const float ell = fmaf(lse, Sp, -Spz);
    if (P.row_loss) P.row_loss[row] = ell;
    P.wl[row] = g * ell;
  }
  if (C > 1) cluster_wait_acquire();
}

// ---------------------------------------------------------------------------
// Persistent variant (bulk path, V up to kPSliceMaxSplit * kMaxCluster).
//
// A cluster of C CTAs (one per SM) walks the rows cid, cid + ncl, ... where
// ncl is the number of co-resident clusters.  Each CTA owns one slice of every
// row.  A producer warp streams the CTA's slices of the cluster's rows with
// g != 0 into nb shared-memory buffers (z slice, p slice) with bulk copies, as
// far ahead as the buffers allow; kPWarps consumer warps process them.
//
// The consumers are software-pipelined over the exchange of partial
// statistics.  In iteration v (the v-th row with g != 0) each consumer warp
// runs
//   reduce(v)   copy its part of the slice (at most kPVec float4 of z and of p
//               per thread) into registers and release the buffer; reduce it
//               to (max m_w, sum e, Sp, Spz) with e = exp(z - m_w) kept in
//               registers; lane r pushes this warp partial into slot
//               [v & 3][rank * kPWarps + warp] of CTA r with st.async, which
//               counts 16 bytes on CTA r's mbarrier xbar[v & 3];
//   finish(v-1) wait until xbar[(v-1) & 3] has seen the C * kPWarps partials
//               of row v-1, fold them into lse, and write the gradient
//               e exp(m_w - lse) g Sp - p g of row v-1 from the registers kept
//               for it.
// The exchange of row v-1 has all of reduce(v) to land in, and no block-wide
// or cluster-wide barrier sits in the loop (the release of a cluster barrier
// would also wait for the CTA's global stores to drain).
// Slot and mbarrier reuse: a warp pushes row v + 4 after its finish(v + 2),
// which needed the push of row v + 2 by every warp of every CTA; each warp
// makes that push after its own finish(v).  So all readers of a slot (and all
// waiters on its phase) are done before the slot is written again.
// Masked rows take no buffer and no exchange: all CTAs of a cluster see the
// same g and write zeros.
constexpr int kPWarps = 8;                     // consumer warps
constexpr int kPThreads = (kPWarps + 1) * 32;  // + the producer warp
constexpr int kPConsumers = kPWarps * 32;
constexpr int kPVec = 7;                  // float4 of z (and of p) per consumer thread at most
constexpr int kPSliceTarget = 7168;       // preferred elements per CTA
// Two row buffers: more let the producer run further ahead but measured
// slower (5.1 vs 5.8 TB/s with three), so the smaller shared footprint wins.
constexpr int kPMinBufs = 2;
constexpr int kPMaxBufs = 2;
constexpr int kPSmemBudget = 200 * 1024;  // shared bytes for the row buffers
constexpr int kPSliceMax = kPConsumers * kPVec * 4;
// Larger slices (vocabularies past 16 x 7168) keep only exp(z - m_w) in
// registers (kPVecSplit float4 per thread) and read p from shared memory again
// for the gradient: z has two buffers (free once reduced), p three (free once
// the gradient is written).
constexpr int kPVecSplit = 10;
constexpr int kPSliceMaxSplit = kPConsumers * kPVecSplit * 4;  // 10240
static_assert(20 * kPSliceMaxSplit <= kPSmemBudget, "split buffers for the largest slice");
constexpr int kPParts = kMaxCluster * kPWarps;  // warp partials of one row, at most
static_assert(kPSliceMax * 8 * kPMinBufs <= kPSmemBudget, "buffers for the largest slice");

struct CePParams {
  float* z;
  const float* p;
  const float* g;
  float* row_loss;
  float* wl;
  long long N, V;
  int C;
  int slice;
  int nb;
};

// One row's slice as a consumer thread keeps it between reduce and finish
// (p only when it is not kept in shared memory).
template <int VEC, bool HAS_P>
struct CeRowRegs {
  float4 e[VEC];  // exp(z - m_w)
  float4 p[HAS_P ? VEC : 1];
  long long row;
  float g;
  float m;        // the warp's max m_w
};

// Four consecutive elements (group i) of a row slice in shared memory as
// fp32: float4, or four bf16 (8 bytes) widened.
template <bool BF16>
__device__ __forceinline__ float4 lds_group(const unsigned char* base, int i) {
  if constexpr (BF16) {
    const uint2 u = reinterpret_cast<const uint2*>(base)[i];
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
  } else {
    return reinterpret_cast<const float4*>(base)[i];
  }
}
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
// Four gradient values (group i of a row slice starting at `row`) to global
// memory with streaming stores: fp32, or bf16 rounded to nearest even.
template <bool BF16>
__device__ __forceinline__ void stg_group(void* row, int i, float4 v) {
  if constexpr (BF16) {
    asm volatile("st.global.cs.v2.b32 [%0], {%1, %2};" ::"l"(static_cast<uint2*>(row) + i),
                 "r"(bf16x2_rn(v.x, v.y)), "r"(bf16x2_rn(v.z, v.w))
                 : "memory");
  } else {
    st_global_cs_f4(static_cast<float*>(row) + 4 * i, v);
  }
}

// SPLIT: the split layout of large fp32 slices.  BF16: z and p are bf16 (the
// gradient is written back in bf16).  GEL: g is per element ([N, V] fp32): the
// row's sums take p g in place of p, and no row is masked.
template <bool SPLIT, bool BF16 = false, bool GEL = false>
__global__ void __launch_bounds__(kPThreads, 1) soft_ce_persistent_kernel(const CePParams P) {
  static_assert(!SPLIT || (!BF16 && !GEL), "the split layout is fp32 with a per-row g");
  constexpr int VEC = SPLIT ? kPVecSplit : kPVec;
  constexpr int ESZ = BF16 ? 2 : 4;                      // bytes per z / p element
  constexpr int PER = 2 * ESZ + (GEL ? 4 : 0);           // buffer bytes per element (unsplit)
  using Row = CeRowRegs<VEC, !SPLIT>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ uint64_t full[kPMaxBufs];
  __shared__ uint64_t empty[kPMaxBufs];
  __shared__ uint64_t pfull[3], pempty[3];  // p buffers of the split layout
  __shared__ uint64_t xbar[4];
  __shared__ __align__(16) float4 stats[4][kPParts];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = P.C;
  const uint32_t rank = cluster_ctarank();
  const long long ncl = gridDim.x / C;
  const long long cid = blockIdx.x / C;
  const long long begin = (long long)rank * P.slice;
  const long long rem = P.V - begin;
  const int len = rem <= 0 ? 0 : (rem < P.slice ? (int)rem : P.slice);
  const int n4 = len >> 2;
  const int nb = SPLIT ? 2 : P.nb;  // z (and, unsplit, p and g) buffers
  // Buffer b of z (and, unsplit, of p and of a per-element g); p buffer c of
  // the split layout.
  auto zbuf = [&](int b) {
    return smem_raw + (size_t)b * (SPLIT ? 4 : PER) * P.slice;
  };
  auto pbuf = [&](int b, int c) {
    return SPLIT ? smem_raw + (size_t)(2 + c) * 4 * P.slice
                 : smem_raw + (size_t)b * PER * P.slice + (size_t)ESZ * P.slice;
  };
  auto gbuf = [&](int b) { return smem_raw + (size_t)b * PER * P.slice + (size_t)2 * ESZ * P.slice; };
  // The rows' per-row weight (1 with a per-element g: such rows are never masked).
  auto row_g = [&](long long r) -> float { return GEL ? 1.0f : __ldg(P.g + r); };

  if (tid == 0) {
    for (int b = 0; b < nb; ++b) {
      mbar_init(&full[b], 1);
      mbar_init(&empty[b], kPWarps);
    }
    if (SPLIT)
      for (int c = 0; c < 3; ++c) {
        mbar_init(&pfull[c], 1);
        mbar_init(&pempty[c], kPWarps);
      }
    for (int k = 0; k < 4; ++k) mbar_init(&xbar[k], 1);
    fence_mbar_init();
  }
  // Every CTA's mbarriers are initialised before any CTA pushes to them.
  cluster_arrive_release();
  cluster_wait_acquire();
  // The loss sum may be scheduled now; it waits for this grid to finish.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == kPWarps) {
    // Producer: the slices of the cluster's rows with g != 0, in order.
    if (lane == 0 && len > 0) {
      int j = 0;
      float gr = cid < P.N ? row_g(cid) : 0.0f;
      for (long long r = cid; r < P.N; r += ncl) {
        const float gcur = gr;
        if (r + ncl < P.N) gr = row_g(r + ncl);
        if (gcur == 0.0f) continue;
        const int b = j % nb;
        if (j >= nb) mbar_wait(&empty[b], (uint32_t)(j / nb - 1) & 1u, STT_DEVERR_CE_WAIT);
        unsigned char* zs = zbuf(b);
        const unsigned char* zsrc = reinterpret_cast<const unsigned char*>(P.z) + (r * P.V + begin) * ESZ;
        const unsigned char* psrc = reinterpret_cast<const unsigned char*>(P.p) + (r * P.V + begin) * ESZ;
        if (SPLIT) {
          mbar_arrive_expect_tx(&full[b], 4u * (uint32_t)len);
          for (int c = 0; c < len; c += kChunk)
            bulk_load(zs + 4 * c, zsrc + 4 * c, (uint32_t)min(kChunk, len - c) * 4u, &full[b]);
          const int pc = j % 3;
          if (j >= 3) mbar_wait(&pempty[pc], (uint32_t)(j / 3 - 1) & 1u, STT_DEVERR_CE_WAIT);
          unsigned char* ps = pbuf(b, pc);
          mbar_arrive_expect_tx(&pfull[pc], 4u * (uint32_t)len);
          for (int c = 0; c < len; c += kChunk)
            bulk_load(ps + 4 * c, psrc + 4 * c, (uint32_t)min(kChunk, len - c) * 4u, &pfull[pc]);
        } else {
          unsigned char* ps = pbuf(b, 0);
          unsigned char* gs = gbuf(b);
          const float* gsrc = P.g + r * P.V + begin;
          mbar_arrive_expect_tx(&full[b], (uint32_t)PER * (uint32_t)len);
          for (int c = 0; c < len; c += kChunk) {
            const uint32_t n = (uint32_t)min(kChunk, len - c);
            bulk_load(zs + (size_t)ESZ * c, zsrc + (size_t)ESZ * c, n * ESZ, &full[b]);
            bulk_load(ps + (size_t)ESZ * c, psrc + (size_t)ESZ * c, n * ESZ, &full[b]);
            if (GEL) bulk_load(gs + (size_t)4 * c, gsrc + c, n * 4u, &full[b]);
          }
        }
        ++j;
      }
    }
    __syncwarp();
  } else {
    // Consumers.
    Row ra, rb;
    long long row = cid;
    float g_row = cid < P.N ? row_g(cid) : 0.0f;
    int v = 0;  // valid rows reduced so far

    // Moves `row` to the cluster's next row with g != 0, writing zeros (and
    // zero losses) for the masked rows passed on the way.  False at the end.
    auto next_valid = [&]() -> bool {
      while (row < P.N && g_row == 0.0f) {
        void* zrow = reinterpret_cast<unsigned char*>(P.z) + (row * P.V + begin) * ESZ;
        const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < VEC; ++k) {
          const int i = tid + k * kPConsumers;
          if (i < n4) stg_group<BF16>(zrow, i, zero);
        }
        if (rank == 0 && tid == 0) {
          if (P.row_loss) P.row_loss[row] = 0.0f;
          P.wl[row] = 0.0f;
        }
        row += ncl;
        g_row = row < P.N ? row_g(row) : 0.0f;
      }
      return row < P.N;
    };

    // reduce(v) of the current row into `cur`, then push the warp partial.
    auto reduce = [&](Row& cur) {
      const int b = v % nb;
      const unsigned char* zs = zbuf(b);
      const unsigned char* ps = pbuf(b, v % 3);
      const float4* gs4 = reinterpret_cast<const float4*>(gbuf(b));
      cur.row = row;
      cur.g = g_row;
      row += ncl;
      g_row = row < P.N ? row_g(row) : 0.0f;
      float m = -INFINITY;
      if (len > 0) {
        mbar_wait(&full[b], (uint32_t)(v / nb) & 1u, STT_DEVERR_CE_WAIT);
        if (SPLIT) mbar_wait(&pfull[v % 3], (uint32_t)(v / 3) & 1u, STT_DEVERR_CE_WAIT);
#pragma unroll
        for (int k = 0; k < VEC; ++k) {
          const int i = tid + k * kPConsumers;
          if (i < n4) {
            cur.e[k] = lds_group<BF16>(zs, i);
            if constexpr (!SPLIT) {
              cur.p[k] = lds_group<BF16>(ps, i);
              if constexpr (GEL) {
                // p g per element stands in for p from here on
                const float4 gv = gs4[i];
                cur.p[k] = make_float4(cur.p[k].x * gv.x, cur.p[k].y * gv.y, cur.p[k].z * gv.z,
                                       cur.p[k].w * gv.w);
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[b]);  // this warp is done with buffer b
#pragma unroll
        for (int k = 0; k < VEC; ++k) {
          const int i = tid + k * kPConsumers;
          if (i < n4)
            m = fmaxf(m, fmaxf(fmaxf(cur.e[k].x, cur.e[k].y), fmaxf(cur.e[k].z, cur.e[k].w)));
        }
      }
      m = warp_max(m);
      cur.m = m;
      float l = 0.f, sp = 0.f, spz = 0.f;
      if (m != -INFINITY) {
        const float mb = m * kLog2e;
#pragma unroll
        for (int k = 0; k < VEC; ++k) {
          const int i = tid + k * kPConsumers;
          if (i < n4) {
            const float4 zv = cur.e[k];
            float4 pv;
            if constexpr (SPLIT)
              pv = lds_group<false>(ps, i);
            else
              pv = cur.p[k];
            float4 e;
            e.x = ex2(fmaf(zv.x, kLog2e, -mb));
            e.y = ex2(fmaf(zv.y, kLog2e, -mb));
            e.z = ex2(fmaf(zv.z, kLog2e, -mb));
            e.w = ex2(fmaf(zv.w, kLog2e, -mb));
            l += (e.x + e.y) + (e.z + e.w);
            sp += (pv.x + pv.y) + (pv.z + pv.w);
            spz = fmaf(pv.x, zv.x, spz);
            spz = fmaf(pv.y, zv.y, spz);
            spz = fmaf(pv.z, zv.z, spz);
            spz = fmaf(pv.w, zv.w, spz);
            cur.e[k] = e;
          }
        }
      }
      l = warp_sum(l);
      sp = warp_sum(sp);
      spz = warp_sum(spz);
      if (tid == 0) mbar_arrive_expect_tx(&xbar[v & 3], 16u * (uint32_t)(C * kPWarps));
      if (lane < C)
        st_async_f4(mapa_shared(smem_u32(&stats[v & 3][rank * kPWarps + warp]), (uint32_t)lane),
                    make_float4(m, l, sp, spz), mapa_shared(smem_u32(&xbar[v & 3]), (uint32_t)lane));
    };

    // finish(u) of the row kept in `prv`.
    auto finish = [&](const Row& prv, int u) {
      mbar_wait_cluster(&xbar[u & 3], (uint32_t)(u >> 2) & 1u, STT_DEVERR_CE_WAIT);
      const int np = C * kPWarps;
      float4 q[kPParts / 32];
      float M = -INFINITY;
#pragma unroll
      for (int t = 0; t < kPParts / 32; ++t) {
        const int j = lane + 32 * t;
        q[t] = j < np ? stats[u & 3][j] : make_float4(-INFINITY, 0.f, 0.f, 0.f);
        M = fmaxf(M, q[t].x);
      }
      M = warp_max(M);
      float Ls = 0.f, Sp = 0.f, Spz = 0.f;
#pragma unroll
      for (int t = 0; t < kPParts / 32; ++t) {
        if (q[t].y > 0.f) Ls += q[t].y * ex2((q[t].x - M) * kLog2e);
        Sp += q[t].z;
        Spz += q[t].w;
      }
      Ls = warp_sum(Ls);
      Sp = warp_sum(Sp);
      Spz = warp_sum(Spz);
      const float lse = M + logf(Ls);
      const float g = prv.g;
      // exp(z - lse) g Sp = e exp(m_w - lse) g Sp; m_w <= lse, so this cannot overflow.
      const float scale = (prv.m == -INFINITY) ? 0.f : ex2((prv.m - lse) * kLog2e) * (g * Sp);
      void* zrow = reinterpret_cast<unsigned char*>(P.z) + (prv.row * P.V + begin) * ESZ;
      const unsigned char* ps = pbuf(0, u % 3);
#pragma unroll
      for (int k = 0; k < VEC; ++k) {
        const int i = tid + k * kPConsumers;
        if (i < n4) {
          float4 pv;
          if constexpr (SPLIT)
            pv = lds_group<false>(ps, i);
          else
            pv = prv.p[k];
          float4 o;
          o.x = fmaf(prv.e[k].x, scale, -pv.x * g);
          o.y = fmaf(prv.e[k].y, scale, -pv.y * g);
          o.z = fmaf(prv.e[k].z, scale, -pv.z * g);
          o.w = fmaf(prv.e[k].w, scale, -pv.w * g);
          stg_group<BF16>(zrow, i, o);
        }
      }
      if (SPLIT && len > 0) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&pempty[u % 3]);  // this warp is done with p of row u
      }
      if (rank == 0 && tid == 0) {
        const float ell = fmaf(lse, Sp, -Spz);
        if (P.row_loss) P.row_loss[prv.row] = ell;
        P.wl[prv.row] = g * ell;
      }
    };

    // Two register sets, alternating, so that each stays in registers.
    while (true) {
      if (!next_valid()) break;
      reduce(ra);
      if (v > 0) finish(rb, v - 1);
      ++v;
      if (!next_valid()) break;
      reduce(rb);
      finish(ra, v - 1);
      ++v;
    }
    if (v > 0) {
      if ((v - 1) & 1)
        finish(rb, v - 1);
      else
        finish(ra, v - 1);
    }
  }
  // Every CTA stays until the whole cluster is done, so no push can target a
  // CTA that has left, even after a timed-out wait.
  __syncwarp();
  cluster_arrive_release();
  cluster_wait_acquire();
}

// Fixed-order sum of the per-row weighted losses (one CTA, deterministic).
// Launched as a programmatic dependent of the row kernel, so its launch
// overlaps the row kernel's tail; it reads wl only after that grid has
// completed and its writes are visible (griddepcontrol.wait).
__global__ void __launch_bounds__(1024) soft_ce_loss_sum(const float* wl, long long N,
                                                         float* loss) {
  __shared__ double part[1024];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  double acc = 0.0;
  for (long long i = threadIdx.x; i < N; i += 1024) acc += (double)wl[i];
  part[threadIdx.x] = acc;
  __syncthreads();
  for (int w = 512; w > 0; w >>= 1) {
    if ((int)threadIdx.x < w) part[threadIdx.x] += part[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) *loss = (float)part[0];
}

}  // namespace

namespace {

// One cluster per row (the non-persistent kernel).
CePlan soft_ce_plan_cta(const float* z, const float* p, int64_t V) {
  CePlan plan;
  plan.bulk = (V % 4 == 0) && ((reinterpret_cast<uintptr_t>(z) & 15u) == 0) &&
              ((reinterpret_cast<uintptr_t>(p) & 15u) == 0);
  long long C = (8 * V + kSliceBudget - 1) / kSliceBudget;
  if (C < 1) C = 1;
  if (C > kMaxCluster) C = kMaxCluster;
  long long slice = (V + C - 1) / C;
  slice = (slice + 3) / 4 * 4;
  // Never leave a CTA of the cluster without elements when V is small.
  while (C > 1 && (C - 1) * slice >= V) {
    --C;
    slice = ((V + C - 1) / C + 3) / 4 * 4;
  }
  plan.C = (int)C;
  plan.slice = (int)slice;
  plan.smem = (int)(8 * slice);
  plan.persistent = false;
  plan.split = false;
  plan.nb = 1;
  return plan;
}

}  // namespace

CePlan soft_ce_plan(const float* z, const float* p, int64_t N, int64_t V) {
  (void)N;
  CePlan plan = soft_ce_plan_cta(z, p, V);
  if (plan.bulk) {
    // Persistent clusters: slices of about kPSliceTarget elements, at least
    // kPMinBufs row buffers per CTA; slices past kPSliceMax take the split
    // layout (z and p in separate buffers, p read again from shared memory).
    auto split = [&](long long slice_max, long long* C_out, long long* sl_out) {
      long long Cp = (V + kPSliceTarget - 1) / kPSliceTarget;
      const long long Cmin = (V + slice_max - 1) / slice_max;
      if (Cp < Cmin) Cp = Cmin;
      if (Cp < 1) Cp = 1;
      if (Cp > kMaxCluster) Cp = kMaxCluster;
      long long sl = ((V + Cp - 1) / Cp + 3) / 4 * 4;
      while (Cp > 1 && (Cp - 1) * sl >= V) {
        --Cp;
        sl = ((V + Cp - 1) / Cp + 3) / 4 * 4;
      }
      *C_out = Cp;
      *sl_out = sl;
    };
    long long Cp, sl;
    split(kPSliceMax, &Cp, &sl);
    long long nb = kPSmemBudget / (8 * sl);
    if (nb > kPMaxBufs) nb = kPMaxBufs;
    if (sl <= kPSliceMax && nb >= kPMinBufs) {
      plan.persistent = true;
      plan.C = (int)Cp;
      plan.slice = (int)sl;
      plan.nb = (int)nb;
      plan.smem = (int)(nb * 8 * sl);
    } else {
      split(kPSliceMaxSplit, &Cp, &sl);
      if (sl <= kPSliceMaxSplit) {
        plan.persistent = true;
        plan.split = true;
        plan.C = (int)Cp;
        plan.slice = (int)sl;
        plan.nb = 2;
        plan.smem = (int)(20 * sl);  // two z buffers, three p buffers
      }
    }
  }
  return plan;
}

namespace {

// Co-resident clusters of soft_ce_persistent_kernel<SPLIT, BF16, GEL> for
// (C, smem) on the current device; 0 if the query fails.  Cached per device
// (and instantiation) for the last configuration.
template <bool SPLIT, bool BF16 = false, bool GEL = false>
int persistent_clusters(int C, int smem) {
  static std::mutex mu;
  static int cache_dev[64], cache_C[64], cache_smem[64], cache_n[64];
  static bool init = false;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!init) {
    for (int i = 0; i < 64; ++i) cache_dev[i] = -1;
    init = true;
  }
  if (cache_dev[dev] == dev && cache_C[dev] == C && cache_smem[dev] == smem) return cache_n[dev];
  auto kern = soft_ce_persistent_kernel<SPLIT, BF16, GEL>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return 0;
  if (C > 8 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                   cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)C, 1, 1);
  cfg.blockDim = dim3(kPThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  cache_dev[dev] = dev;
  cache_C[dev] = C;
  cache_smem[dev] = smem;
  cache_n[dev] = n;
  return n;
}

}  // namespace

cudaError_t soft_ce_launch(const CePlan& plan, float* z, const float* p, const float* g,
                           int64_t N, int64_t V, float* row_loss, float* loss, float* wl,
                           cudaStream_t s) {
  int ncl = 0;
  if (N > 0 && plan.persistent)
    ncl = plan.split ? persistent_clusters<true>(plan.C, plan.smem)
                     : persistent_clusters<false>(plan.C, plan.smem);
  if (ncl > 0) {
    const long long n_clusters = ncl < N ? ncl : N;
    CePParams P{z, p, g, row_loss, wl, (long long)N, (long long)V, plan.C, plan.slice, plan.nb};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(n_clusters * plan.C), 1, 1);
    cfg.blockDim = dim3(kPThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)plan.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)plan.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    prof_before(s, STT_KERNEL_SOFT_CE);
    cudaError_t e = plan.split ? cudaLaunchKernelEx(&cfg, soft_ce_persistent_kernel<true>, P)
                               : cudaLaunchKernelEx(&cfg, soft_ce_persistent_kernel<false>, P);
    if (e != cudaSuccess) {
      prof_after(s);
      return e;
    }
  } else if (N > 0) {
    // One cluster per row (also taken if the persistent kernel cannot be resident).
    const CePlan fb = plan.persistent ? soft_ce_plan_cta(z, p, V) : plan;
    if (N * (long long)fb.C > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    CeParams P{z, p, g, row_loss, wl, (long long)N, (long long)V, fb.C, fb.slice};
    void (*kern)(const CeParams) = fb.bulk ? soft_ce_kernel<true> : soft_ce_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         fb.smem);
    if (e != cudaSuccess) return e;
    if (fb.C > 8) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(N * fb.C), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)fb.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)fb.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    prof_before(s, STT_KERNEL_SOFT_CE);
    e = cudaLaunchKernelEx(&cfg, kern, P);
    if (e != cudaSuccess) {
      prof_after(s);
      return e;
    }
  } else {
    prof_before(s, STT_KERNEL_SOFT_CE);
  }
  // The loss sum follows the row kernel directly (no profiling event between
  // them, which would serialise the pair), as a programmatic dependent launch;
  // the profiled unit STT_KERNEL_SOFT_CE covers both kernels.
  const cudaError_t e2 = soft_ce_loss_sum_launch(wl, N, loss, s);
  prof_after(s);
  if (e2 != cudaSuccess) return e2;
  return cudaGetLastError();
}

cudaError_t soft_ce_loss_sum_launch(const float* wl, int64_t N, float* loss, cudaStream_t s) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(1, 1, 1);
  lc.blockDim = dim3(1024, 1, 1);
  lc.dynamicSmemBytes = 0;
  lc.stream = s;
  cudaLaunchAttribute la[1];
  la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  la[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = la;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, soft_ce_loss_sum, wl, (long long)N, loss);
}

namespace {

template <bool BF16, bool GEL>
cudaError_t variant_persistent(void* z, const void* p, const float* g, int64_t N, int64_t V,
                               float* row_loss, float* loss, float* wl, cudaStream_t s) {
  constexpr int per = 2 * (BF16 ? 2 : 4) + (GEL ? 4 : 0);  // shared bytes per element
  // Slices of about kPSliceTarget elements (at most kPSliceMax, the registers'
  // reach), multiples of 8 so that every bf16 slice starts 16-byte aligned.
  long long C = (V + kPSliceTarget - 1) / kPSliceTarget;
  const long long Cmin = (V + kPSliceMax - 1) / kPSliceMax;
  if (C < Cmin) C = Cmin;
  if (C < 1) C = 1;
  if (C > kMaxCluster) return cudaErrorNotSupported;
  long long sl = ((V + C - 1) / C + 7) / 8 * 8;
  while (C > 1 && (C - 1) * sl >= V) {
    --C;
    sl = ((V + C - 1) / C + 7) / 8 * 8;
  }
  if (sl > kPSliceMax) return cudaErrorNotSupported;
  long long nb = kPSmemBudget / (per * sl);
  if (nb > kPMaxBufs) nb = kPMaxBufs;
  if (nb < kPMinBufs) return cudaErrorNotSupported;
  const int smem = (int)(nb * per * sl);
  const int ncl = persistent_clusters<false, BF16, GEL>((int)C, smem);
  if (ncl <= 0) return cudaErrorNotSupported;
  const long long n_clusters = ncl < N ? ncl : N;
  CePParams P{static_cast<float*>(z), static_cast<const float*>(p), g, row_loss, wl,
              (long long)N, (long long)V, (int)C, (int)sl, (int)nb};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(n_clusters * C), 1, 1);
  cfg.blockDim = dim3(kPThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_before(s, STT_KERNEL_SOFT_CE_VARIANT);
  cudaError_t e = cudaLaunchKernelEx(&cfg, soft_ce_persistent_kernel<false, BF16, GEL>, P);
  if (e == cudaSuccess) e = soft_ce_loss_sum_launch(wl, N, loss, s);
  prof_after(s);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t soft_ce_variant_persistent_launch(uint32_t flags, void* z, const void* p,
                                              const float* g, int64_t N, int64_t V,
                                              float* row_loss, float* loss, float* wl,
                                              cudaStream_t s) {
  const bool bf16 = (flags & kCeBf16) != 0, gel = (flags & kCeGPerElement) != 0;
  const uintptr_t a = reinterpret_cast<uintptr_t>(z) | reinterpret_cast<uintptr_t>(p) |
                      (gel ? reinterpret_cast<uintptr_t>(g) : 0);
  // bf16 rows with a per-row g stay on the one-row-per-cluster kernel: at
  // 6 bytes an element the persistent kernel's per-row exchange and arithmetic,
  // not its bytes, set its pace (2.8 against 4.2 TB/s at V = 32000).
  if (N <= 0 || V % 8 != 0 || (a & 15u) != 0 || (bf16 && !gel)) return cudaErrorNotSupported;
  if (bf16) return variant_persistent<true, true>(z, p, g, N, V, row_loss, loss, wl, s);
  return gel ? variant_persistent<false, true>(z, p, g, N, V, row_loss, loss, wl, s)
             : variant_persistent<false, false>(z, p, g, N, V, row_loss, loss, wl, s);
}

STT_DEFINE_ERROR_ACCESSOR(soft_ce_error_word)
STT_DEFINE_BUDGET_SETTER(soft_ce_set_wait_budget)

// ---------------------------------------------------------------------------
// Allocation-free variant of the in-place soft-CE.
//
// The per-row weighted losses, which the regular entry point keeps in a
// caller-provided workspace, live here in a fixed file-scope device array.
// Every GPU that loads the library holds this array (256 KB) until the
// process exits.  In host code `g_noalloc_scratch` is only a host-side stand-in
// for the symbol, not a device address, so the device address is looked up
// with cudaGetSymbolAddress on the current device at every call (a cached
// address would go stale after cudaDeviceReset or a new primary context);
// kernels are always handed that looked-up pointer.
namespace {

constexpr int64_t kNoAllocMaxRows = 65536;
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocMaxRows];

// Device address of the scratch array on the current device.
int noalloc_scratch(float** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return status_from_cuda(e);
  if (p == nullptr) return STT_ERR_CUDA;
  *out = static_cast<float*>(p);
  return STT_OK;
}

}  // namespace

}  // namespace stt

extern "C" int soft_ce_fwd_bwd_inplace_noalloc(float* z, const float* p, const float* g,
                                               int64_t N, int64_t V, float* row_loss,
                                               float* loss, void* stream) {
  try {
    (void)cudaGetLastError();  // clear an error an earlier call of this thread left behind
    if (N < 0 || V < 1 || !loss) return STT_ERR_INVALID_ARG;
    if (N > 0 && (!z || !p || !g)) return STT_ERR_INVALID_ARG;
    if (N > 0 && V > INT64_MAX / N) return STT_ERR_INVALID_ARG;
    if (N > stt::kNoAllocMaxRows) return STT_ERR_WORKSPACE;
    if (V > stt::kCeMaxV) return STT_ERR_UNSUPPORTED;
    float* scratch = nullptr;
    const int st = stt::noalloc_scratch(&scratch);
    if (st != STT_OK) return st;
    // Every row of the scratch that the loss sum reads is written first by the
    // row kernel (masked rows included), so nothing has to be cleared.
    const stt::CePlan plan = stt::soft_ce_plan(z, p, N, V);
    if (N * (int64_t)plan.C > 0x7fffffffLL) return STT_ERR_UNSUPPORTED;
    const cudaError_t e = stt::soft_ce_launch(plan, z, p, g, N, V, row_loss, loss, scratch,
                                              static_cast<cudaStream_t>(stream));
    return stt::status_from_cuda(e);
  } catch (...) {
    return STT_ERR_CUDA;
  }
}

namespace stt {

static_assert(kSliceMax * 8 <= 227 * 1024, "slice must fit in shared memory");
static_assert((long long)kSliceMax * kMaxCluster == kCeMaxV, "max V");
static_assert(kSliceMax <= kChunk * kMaxChunks, "chunks");
static_assert(kPSmemBudget + 2048 <= 227 * 1024, "persistent shared memory");

}  // namespace stt
