// attn_bwd.cu -- sparse-tree TTT attention, backward.
//
// The page trains through the masked attention (SpecForge review, §三
// "稀疏树注意力": FlexAttention streams the computation and keeps no
// intermediate activations), so the backward is the derivative of the masked
// softmax attention, with P recomputed from the saved logsumexp:
//     Delta_q = sum_d dO * O,  P = exp(S - lse),  dS = P (dP - Delta),
//     dq = scale dS Kc,  dKc = scale dS^T q,  dVc = P^T dO.
//
// Three kernels, in stream order:
//   1. prep (CUDA cores, one warp per (b, KV head, row q)): Delta for every
//      query head of the group; the whole backward of the diagonal suffix keys
//      (q < T, blocks j = 1..k: one key per query, so dK_j / dV_j row q is owned
//      by this warp and written directly); dq initialised with the suffix part;
//      dK_0 / dV_0 zeroed for the causal kernel's accumulation.
//   2. dq (tcgen05, one CTA per 128-row query tile of a head, like the
//      forward): S = Q K^T and dP = dO V^T in TMEM, dS written back into TMEM
//      as bf16, dQ += dS K (A operand read from TMEM); dq += scale dQ.
//   3. dkdv (tcgen05, one CTA per 128-row key tile of a query head): S^T =
//      K Q^T and dP^T = V dO^T in TMEM, P^T and dS^T written back into TMEM as
//      bf16, dV += P^T dO and dK += dS^T Q accumulate in TMEM over the query
//      tiles; the group's query heads are summed with fp32 atomics.
// In both tcgen05 kernels 8 compute warps share the element-wise phase: warps
// w and w+4 read the same TMEM lane quarter and split its columns in halves.
// dq is written once per row by exactly one CTA (deterministic); dK_0 / dV_0
// sum G partials per element in arrival order.
#include "../../include/stt.h"
#include "attn_common.cuh"

namespace stt {
namespace {

constexpr int kThreads = 320;   // warps 0-7 compute, 8 TMA, 9 MMA
constexpr int kCompute = 256;
constexpr int kWarpTma = 8, kWarpMma = 9;

struct BwdParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* kb[kMaxBlocks];
  const __nv_bfloat16* vb[kMaxBlocks];
  const __nv_bfloat16* out;
  const __nv_bfloat16* dout;
  const float* lse;
  float* dq;
  float* dkb[kMaxBlocks];
  float* dvb[kMaxBlocks];
  float* delta;
  int B, H, H_kv, Q_LEN, k, n_t, G;
  float scale, scale_log2;
  int T[kMaxBatch];
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int E>
__device__ __forceinline__ void load_bf16(const __nv_bfloat16* p, float (&v)[E]) {
  if constexpr (E == 4) {
    const uint2 x = __ldg(reinterpret_cast<const uint2*>(p));
    v[0] = bf16lo(x.x);
    v[1] = bf16hi(x.x);
    v[2] = bf16lo(x.y);
    v[3] = bf16hi(x.y);
  } else {
    const uint32_t x = __ldg(reinterpret_cast<const uint32_t*>(p));
    v[0] = bf16lo(x);
    v[1] = bf16hi(x);
  }
}

template <int E>
__device__ __forceinline__ void store_f32(float* p, const float (&v)[E]) {
  if constexpr (E == 4)
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  else
    *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
}

// ------------------------------------------------------------------ prep --
// GM: compile-time upper bound of the group size (the loops over heads are
// unrolled so per-head values stay in registers); G <= GM at run time.
template <int D, int GM>
__global__ void __launch_bounds__(256) attn_bwd_prep_kernel(const __grid_constant__ BwdParams P) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * 8;
  const long long rows = (long long)P.B * P.H_kv * P.Q_LEN;
  const int G = P.G;
  for (long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5); row < rows; row += warps) {
    const int q = (int)(row % P.Q_LEN);
    const int bhk = (int)(row / P.Q_LEN);
    const int b = bhk / P.H_kv, hk = bhk % P.H_kv;
    const bool valid = q < P.T[b];
    const size_t kvoff = ((size_t)bhk * P.Q_LEN + q) * D + lane * E;
    float qv[GM][E], dov[GM][E], dq[GM][E], lse2[GM], dl[GM];
#pragma unroll
    for (int i = 0; i < GM; ++i) {
      if (i < G) {
        const size_t rq = (size_t)(b * P.H + hk * G + i) * P.Q_LEN + q;
        const size_t off = rq * D + lane * E;
        float ov[E];
        load_bf16<E>(P.dout + off, dov[i]);
        load_bf16<E>(P.out + off, ov);
        load_bf16<E>(P.q + off, qv[i]);
        float d = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) d = fmaf(dov[i][e], ov[e], d);
        dl[i] = warp_sum(d);
        lse2[i] = P.lse[rq] * kLog2e;
        if (lane == 0) P.delta[rq] = dl[i];
#pragma unroll
        for (int e = 0; e < E; ++e) dq[i][e] = 0.f;
      }
    }
    // Blocks are taken kJ at a time with all their row loads issued up front, so
    // each warp keeps 2*kJ loads in flight.
    constexpr int kJ = 4;
    for (int j0 = 1; j0 <= P.k; j0 += kJ) {
      float kv[kJ][E], vv[kJ][E];
      if (valid) {
#pragma unroll
        for (int u = 0; u < kJ; ++u) {
          if (j0 + u <= P.k) {
            load_bf16<E>(P.kb[j0 + u] + kvoff, kv[u]);
            load_bf16<E>(P.vb[j0 + u] + kvoff, vv[u]);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kJ; ++u) {
        const int j = j0 + u;
        if (j > P.k) break;
        float dk[E], dv[E];
#pragma unroll
        for (int e = 0; e < E; ++e) dk[e] = dv[e] = 0.f;
        if (valid) {
#pragma unroll
          for (int i = 0; i < GM; ++i) {
            if (i < G) {
              float s = 0.f, dp = 0.f;
#pragma unroll
              for (int e = 0; e < E; ++e) {
                s = fmaf(qv[i][e], kv[u][e], s);
                dp = fmaf(dov[i][e], vv[u][e], dp);
              }
              s = warp_sum(s);
              dp = warp_sum(dp);
              const float p = ex2(s * P.scale_log2 - lse2[i]);
              const float ds = p * (dp - dl[i]);
              const float dss = ds * P.scale;
#pragma unroll
              for (int e = 0; e < E; ++e) {
                dq[i][e] = fmaf(dss, kv[u][e], dq[i][e]);
                dk[e] = fmaf(dss, qv[i][e], dk[e]);
                dv[e] = fmaf(p, dov[i][e], dv[e]);
              }
            }
          }
        }
        store_f32<E>(P.dkb[j] + kvoff, dk);
        store_f32<E>(P.dvb[j] + kvoff, dv);
      }
    }
#pragma unroll
    for (int i = 0; i < GM; ++i)
      if (i < G)
        store_f32<E>(P.dq + ((size_t)(b * P.H + hk * G + i) * P.Q_LEN + q) * D + lane * E, dq[i]);
    float z[E];
#pragma unroll
    for (int e = 0; e < E; ++e) z[e] = 0.f;
    store_f32<E>(P.dkb[0] + kvoff, z);
    store_f32<E>(P.dvb[0] + kvoff, z);
  }
}

// TMEM columns shared by both tcgen05 kernels.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColDP = 128, kColAcc0 = 256, kColAcc1 = 384;

// -------------------------------------------------------------------- dq --
template <int D>
struct DqSmem {
  static constexpr int kTileB = kTile * D * 2;
  static constexpr int kStages = 2;
  static constexpr int q = 0;
  static constexpr int dO = kTileB;
  static constexpr int k0 = 2 * kTileB;
  static constexpr int v0 = 2 * kTileB + kStages * kTileB;
  static constexpr int total = 2 * kTileB + 2 * kStages * kTileB;
  static constexpr int alloc = total + 1024;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ BwdParams P, const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmDO,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV) {
  using L = DqSmem<D>;
  constexpr int NS = L::kStages;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_qdo, bar_kv_full[NS], bar_kv_empty[NS], bar_sdp_full, bar_ds_ready,
      bar_dq_done, bar_drain, bar_grp;
  __shared__ uint32_t tmem_base;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nb = P.H * P.B;
  const int t = P.n_t - 1 - (int)(blockIdx.x / nb);
  const int bh = (int)(blockIdx.x % nb);
  const int b = bh / P.H, h = bh % P.H, hk = h / P.G;
  const int q0 = t * kTile;
  const int T = P.T[b];
  const int n_kv = causal_kv_tiles(q0, T);

  if (tid == 0) {
    mbar_init(&bar_qdo, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bar_kv_full[s], 1);
      mbar_init(&bar_kv_empty[s], 1);
    }
    mbar_init(&bar_sdp_full, 1);
    mbar_init(&bar_ds_ready, kCompute);
    mbar_init(&bar_dq_done, 1);
    mbar_init(&bar_drain, 1);
    mbar_init(&bar_grp, kCompute);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;

  if (warp == kWarpTma) {
    if (lane == 0 && n_kv > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmDO);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const int bhk = b * P.H_kv + hk;
      mbar_arrive_expect_tx(&bar_qdo, 2 * L::kTileB);
      for (int cb = 0; cb < D / kColBlock; ++cb) {
        tma_load_3d(smem + L::q + cb * kTile * 128, &tmQ, &bar_qdo, cb * kColBlock, q0, bh);
        tma_load_3d(smem + L::dO + cb * kTile * 128, &tmDO, &bar_qdo, cb * kColBlock, q0, bh);
      }
      int issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % NS;
        if (j >= NS && !mbar_wait(&bar_kv_empty[st], ((uint32_t)(j / NS) & 1u) ^ 1u, STT_DEVERR_BWD_WAIT))
          break;
        mbar_arrive_expect_tx(&bar_kv_full[st], 2 * L::kTileB);
        for (int cb = 0; cb < D / kColBlock; ++cb) {
          tma_load_3d(smem + L::k0 + st * L::kTileB + cb * kTile * 128, &tmK, &bar_kv_full[st],
                      cb * kColBlock, j * kTile, bhk);
          tma_load_3d(smem + L::v0 + st * L::kTileB + cb * kTile * 128, &tmV, &bar_kv_full[st],
                      cb * kColBlock, j * kTile, bhk);
        }
        ++issued;
      }
      if (issued < n_kv) {
        mbar_wait(&bar_qdo, 0, STT_DEVERR_BWD_WAIT);
        for (int j = (issued > NS ? issued - NS : 0); j < issued; ++j)
          mbar_wait(&bar_kv_full[j % NS], (uint32_t)(j / NS) & 1u, STT_DEVERR_BWD_WAIT);
      }
    }
  } else if (warp == kWarpMma) {
    if (lane == 0 && n_kv > 0) {
      const uint32_t idSS = idesc_bf16(128, kTile, false, false);
      const uint32_t idDQ = idesc_bf16(128, D, false, true);
      const uint32_t aQ = smem_u32(smem + L::q), aDO = smem_u32(smem + L::dO);
      bool ok = mbar_wait(&bar_qdo, 0, STT_DEVERR_BWD_WAIT);
      for (int j = 0; ok && j < n_kv; ++j) {
        const int st = j % NS;
        ok = mbar_wait(&bar_kv_full[st], (uint32_t)(j / NS) & 1u, STT_DEVERR_BWD_WAIT);
        if (ok && j > 0) ok = mbar_wait(&bar_dq_done, (uint32_t)(j - 1) & 1u, STT_DEVERR_BWD_WAIT);
        if (!ok) break;
        tc_fence_after();
        const uint32_t aK = smem_u32(smem + L::k0 + st * L::kTileB);
        const uint32_t aV = smem_u32(smem + L::v0 + st * L::kTileB);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kTile * 128 + (kk & 3) * 32;
          umma_bf16_ss(tmem + kColS, sdesc_sw128(aQ + off, 16, 1024), sdesc_sw128(aK + off, 16, 1024),
                       idSS, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kTile * 128 + (kk & 3) * 32;
          umma_bf16_ss(tmem + kColDP, sdesc_sw128(aDO + off, 16, 1024),
                       sdesc_sw128(aV + off, 16, 1024), idSS, kk > 0 ? 1u : 0u);
        }
        umma_commit(&bar_sdp_full);
        ok = mbar_wait(&bar_ds_ready, (uint32_t)j & 1u, STT_DEVERR_BWD_WAIT);
        if (!ok) break;
        tc_fence_after();
        // dQ += dS K: A = dS (bf16 in TMEM, 8 columns per 16 keys), B = K [kv][d] MN-major.
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          umma_bf16_ts(tmem + kColAcc0, tmem + kColS + kk * 8,
                       sdesc_sw128(aK + kk * 2048, kTile * 128, 1024), idDQ,
                       (j > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&bar_dq_done);
        umma_commit(&bar_kv_empty[st]);
      }
      umma_commit(&bar_drain);
      mbar_wait(&bar_drain, 0, STT_DEVERR_BWD_WAIT);
    }
  } else {
    // Compute warps: row r = TMEM lane; `half` selects the 64-column half.
    const int quarter = warp & 3, half = warp >> 2;
    const int r = quarter * 32 + lane;
    const int qrow = q0 + r;
    const int lim = causal_row_limit(qrow, T);
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const bool in_range = qrow < P.Q_LEN;
    const size_t rq = (size_t)bh * P.Q_LEN + qrow;
    const float lse2 = in_range ? P.lse[rq] * kLog2e : 0.f;
    const float dlt = in_range ? P.delta[rq] : 0.f;
    const float sl2 = P.scale_log2;
    uint32_t grp_uses = 0;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      ok = warp_wait(&bar_sdp_full, (uint32_t)j & 1u, STT_DEVERR_BWD_WAIT);
      if (!ok) break;
      tc_fence_after();
      const int c0 = j * kTile;
      uint32_t s[2][32], dp[2][32];
      tmem_ld64x2(tmem + lane_off + kColS + half * 64, tmem + lane_off + kColDP + half * 64, s[0],
                  s[1], dp[0], dp[1]);
      // Every compute thread holds its S / dP columns before dS overwrites S.
      ok = group_sync(&bar_grp, grp_uses, STT_DEVERR_BWD_WAIT);
      if (!ok) break;
      const bool full = (c0 + kTile - 1 <= lim) && in_range;
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        const int cc = half * 2 + c2;
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          float p0 = ex2(fmaf(__uint_as_float(s[c2][i]), sl2, -lse2));
          float p1 = ex2(fmaf(__uint_as_float(s[c2][i + 1]), sl2, -lse2));
          if (!full) {
            if (!(in_range && c0 + cc * 32 + i <= lim)) p0 = 0.f;
            if (!(in_range && c0 + cc * 32 + i + 1 <= lim)) p1 = 0.f;
          }
          const float d0 = p0 * (__uint_as_float(dp[c2][i]) - dlt);
          const float d1 = p1 * (__uint_as_float(dp[c2][i + 1]) - dlt);
          pk[i >> 1] = pack_bf16(d0, d1);
        }
        tmem_st16(tmem + lane_off + kColS + cc * 16, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar_ds_ready);
    }
    if (ok && n_kv > 0) {
      ok = warp_wait(&bar_dq_done, (uint32_t)(n_kv - 1) & 1u, STT_DEVERR_BWD_WAIT);
      tc_fence_after();
      if (ok) {
        float* dqrow = P.dq + rq * D;
#pragma unroll
        for (int c2 = 0; c2 < D / 64; ++c2) {
          const int c = half * (D / 64) + c2;
          uint32_t u[32];
          tmem_ld32(tmem + lane_off + kColAcc0 + c * 32, u);
          if (in_range) {
            float4* d4 = reinterpret_cast<float4*>(dqrow + c * 32);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
              float4 v = d4[q4];
              v.x = fmaf(P.scale, __uint_as_float(u[4 * q4 + 0]), v.x);
              v.y = fmaf(P.scale, __uint_as_float(u[4 * q4 + 1]), v.y);
              v.z = fmaf(P.scale, __uint_as_float(u[4 * q4 + 2]), v.z);
              v.w = fmaf(P.scale, __uint_as_float(u[4 * q4 + 3]), v.w);
              d4[q4] = v;
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ dkdv --
template <int D>
struct DkvSmem {
  static constexpr int kTileB = kTile * D * 2;
  static constexpr int kStages = 2;
  static constexpr int k = 0;
  static constexpr int v = kTileB;
  static constexpr int q0 = 2 * kTileB;
  static constexpr int do0 = 2 * kTileB + kStages * kTileB;
  static constexpr int total = 2 * kTileB + 2 * kStages * kTileB;
  static constexpr int alloc = total + 1024;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ BwdParams P, const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmDO,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV) {
  using L = DkvSmem<D>;
  constexpr int NS = L::kStages;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_kv, bar_qdo_full[NS], bar_qdo_empty[NS], bar_sdp_full, bar_pds_ready,
      bar_acc_done, bar_drain, bar_grp;
  __shared__ uint32_t tmem_base;
  __shared__ float s_stat[2][2][kTile];  // [slot][lse2 | delta][query]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nb = P.H * P.B;
  const int c = (int)(blockIdx.x / nb);  // key tile; low tiles see the most query tiles
  const int bh = (int)(blockIdx.x % nb);
  const int b = bh / P.H, h = bh % P.H, hk = h / P.G;
  const int c0 = c * kTile;
  const int T = P.T[b];
  const int t_first = c;                      // query tiles t >= c see this key tile
  const int n_q = (c0 < T) ? (P.n_t - t_first) : 0;

  if (tid == 0) {
    mbar_init(&bar_kv, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bar_qdo_full[s], 1);
      mbar_init(&bar_qdo_empty[s], 1);
    }
    mbar_init(&bar_sdp_full, 1);
    mbar_init(&bar_pds_ready, kCompute);
    mbar_init(&bar_acc_done, 1);
    mbar_init(&bar_drain, 1);
    mbar_init(&bar_grp, kCompute);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;

  if (warp == kWarpTma) {
    if (lane == 0 && n_q > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmDO);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const int bhk = b * P.H_kv + hk;
      mbar_arrive_expect_tx(&bar_kv, 2 * L::kTileB);
      for (int cb = 0; cb < D / kColBlock; ++cb) {
        tma_load_3d(smem + L::k + cb * kTile * 128, &tmK, &bar_kv, cb * kColBlock, c0, bhk);
        tma_load_3d(smem + L::v + cb * kTile * 128, &tmV, &bar_kv, cb * kColBlock, c0, bhk);
      }
      int issued = 0;
      for (int i = 0; i < n_q; ++i) {
        const int st = i % NS;
        const int tq = (t_first + i) * kTile;
        if (i >= NS && !mbar_wait(&bar_qdo_empty[st], ((uint32_t)(i / NS) & 1u) ^ 1u, STT_DEVERR_BWD_WAIT))
          break;
        mbar_arrive_expect_tx(&bar_qdo_full[st], 2 * L::kTileB);
        for (int cb = 0; cb < D / kColBlock; ++cb) {
          tma_load_3d(smem + L::q0 + st * L::kTileB + cb * kTile * 128, &tmQ, &bar_qdo_full[st],
                      cb * kColBlock, tq, bh);
          tma_load_3d(smem + L::do0 + st * L::kTileB + cb * kTile * 128, &tmDO, &bar_qdo_full[st],
                      cb * kColBlock, tq, bh);
        }
        ++issued;
      }
      if (issued < n_q) {
        mbar_wait(&bar_kv, 0, STT_DEVERR_BWD_WAIT);
        for (int i = (issued > NS ? issued - NS : 0); i < issued; ++i)
          mbar_wait(&bar_qdo_full[i % NS], (uint32_t)(i / NS) & 1u, STT_DEVERR_BWD_WAIT);
      }
    }
  } else if (warp == kWarpMma) {
    if (lane == 0 && n_q > 0) {
      const uint32_t idSS = idesc_bf16(128, kTile, false, false);
      const uint32_t idACC = idesc_bf16(128, D, false, true);
      const uint32_t aK = smem_u32(smem + L::k), aV = smem_u32(smem + L::v);
      bool ok = mbar_wait(&bar_kv, 0, STT_DEVERR_BWD_WAIT);
      for (int i = 0; ok && i < n_q; ++i) {
        const int st = i % NS;
        ok = mbar_wait(&bar_qdo_full[st], (uint32_t)(i / NS) & 1u, STT_DEVERR_BWD_WAIT);
        if (ok && i > 0) ok = mbar_wait(&bar_acc_done, (uint32_t)(i - 1) & 1u, STT_DEVERR_BWD_WAIT);
        if (!ok) break;
        tc_fence_after();
        const uint32_t aQ = smem_u32(smem + L::q0 + st * L::kTileB);
        const uint32_t aDO = smem_u32(smem + L::do0 + st * L::kTileB);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kTile * 128 + (kk & 3) * 32;
          umma_bf16_ss(tmem + kColS, sdesc_sw128(aK + off, 16, 1024), sdesc_sw128(aQ + off, 16, 1024),
                       idSS, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kTile * 128 + (kk & 3) * 32;
          umma_bf16_ss(tmem + kColDP, sdesc_sw128(aV + off, 16, 1024),
                       sdesc_sw128(aDO + off, 16, 1024), idSS, kk > 0 ? 1u : 0u);
        }
        umma_commit(&bar_sdp_full);
        ok = mbar_wait(&bar_pds_ready, (uint32_t)i & 1u, STT_DEVERR_BWD_WAIT);
        if (!ok) break;
        tc_fence_after();
        // dV += P^T dO, dK += dS^T Q: A from TMEM (query index = K dim), B MN-major.
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          umma_bf16_ts(tmem + kColAcc0, tmem + kColS + kk * 8,
                       sdesc_sw128(aDO + kk * 2048, kTile * 128, 1024), idACC,
                       (i > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          umma_bf16_ts(tmem + kColAcc1, tmem + kColDP + kk * 8,
                       sdesc_sw128(aQ + kk * 2048, kTile * 128, 1024), idACC,
                       (i > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&bar_acc_done);
        umma_commit(&bar_qdo_empty[st]);
      }
      umma_commit(&bar_drain);
      mbar_wait(&bar_drain, 0, STT_DEVERR_BWD_WAIT);
    }
  } else {
    // Compute warps: key row = TMEM lane; `half` selects the 64-query half.
    const int quarter = warp & 3, half = warp >> 2;
    const int kv = c0 + quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const float sl2 = P.scale_log2;
    const bool kv_live = kv < T;  // T <= Q_LEN, so also kv < Q_LEN
    // Thread tid stages one statistic of one query of the tile: lse2 (tid < 128)
    // or Delta (tid >= 128) of query tq0 + (tid & 127); prefetched a tile ahead.
    const int st_which = tid >> 7, st_idx = tid & 127;
    auto fetch_stat = [&](int i) -> float {
      const int qq = (t_first + i) * kTile + st_idx;
      if (qq >= P.Q_LEN) return 0.f;
      const size_t rq = (size_t)bh * P.Q_LEN + qq;
      return st_which == 0 ? P.lse[rq] * kLog2e : P.delta[rq];
    };
    float stat_next = n_q > 0 ? fetch_stat(0) : 0.f;
    uint32_t grp_uses = 0;
    bool ok = true;
    for (int i = 0; i < n_q; ++i) {
      const int tq0 = (t_first + i) * kTile;
      const int slot = i & 1;
      s_stat[slot][st_which][st_idx] = stat_next;
      if (i + 1 < n_q) stat_next = fetch_stat(i + 1);
      ok = group_sync(&bar_grp, grp_uses, STT_DEVERR_BWD_WAIT);
      if (!ok) break;
      ok = warp_wait(&bar_sdp_full, (uint32_t)i & 1u, STT_DEVERR_BWD_WAIT);
      if (!ok) break;
      tc_fence_after();
      uint32_t s[2][32], dp[2][32];
      tmem_ld64x2(tmem + lane_off + kColS + half * 64, tmem + lane_off + kColDP + half * 64, s[0],
                  s[1], dp[0], dp[1]);
      // Every compute thread holds its S^T / dP^T columns before they are overwritten.
      ok = group_sync(&bar_grp, grp_uses, STT_DEVERR_BWD_WAIT);
      if (!ok) break;
      // entry (kv, q) is visible iff kv < T, kv <= q and q < Q_LEN
      const bool full = kv_live && kv <= tq0 && tq0 + kTile <= P.Q_LEN;
      const float* lse_s = s_stat[slot][0];
      const float* dl_s = s_stat[slot][1];
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        const int cc = half * 2 + c2;
        uint32_t pp[16], dd[16];
#pragma unroll
        for (int x = 0; x < 32; x += 2) {
          const int ql = cc * 32 + x;
          const int qa = tq0 + ql;
          float p0 = ex2(fmaf(__uint_as_float(s[c2][x]), sl2, -lse_s[ql]));
          float p1 = ex2(fmaf(__uint_as_float(s[c2][x + 1]), sl2, -lse_s[ql + 1]));
          if (!full) {
            if (!(kv_live && kv <= qa && qa < P.Q_LEN)) p0 = 0.f;
            if (!(kv_live && kv <= qa + 1 && qa + 1 < P.Q_LEN)) p1 = 0.f;
          }
          const float d0 = p0 * (__uint_as_float(dp[c2][x]) - dl_s[ql]);
          const float d1 = p1 * (__uint_as_float(dp[c2][x + 1]) - dl_s[ql + 1]);
          pp[x >> 1] = pack_bf16(p0, p1);
          dd[x >> 1] = pack_bf16(d0, d1);
        }
        tmem_st16(tmem + lane_off + kColS + cc * 16, pp);
        tmem_st16(tmem + lane_off + kColDP + cc * 16, dd);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar_pds_ready);
    }
    if (ok && n_q > 0) {
      ok = warp_wait(&bar_acc_done, (uint32_t)(n_q - 1) & 1u, STT_DEVERR_BWD_WAIT);
      tc_fence_after();
      if (ok) {
        const size_t off = ((size_t)(b * P.H_kv + hk) * P.Q_LEN + kv) * D;
        float* dkr = P.dkb[0] + off;
        float* dvr = P.dvb[0] + off;
#pragma unroll
        for (int c2 = 0; c2 < D / 64; ++c2) {
          const int cc = half * (D / 64) + c2;
          uint32_t uv[32], uk[32];
          tmem_ld32x2(tmem + lane_off + kColAcc0 + cc * 32, tmem + lane_off + kColAcc1 + cc * 32,
                      uv, uk);
          if (kv_live) {
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
              atomicAdd(reinterpret_cast<float4*>(dvr + cc * 32) + q4,
                        make_float4(__uint_as_float(uv[4 * q4]), __uint_as_float(uv[4 * q4 + 1]),
                                    __uint_as_float(uv[4 * q4 + 2]), __uint_as_float(uv[4 * q4 + 3])));
              atomicAdd(reinterpret_cast<float4*>(dkr + cc * 32) + q4,
                        make_float4(P.scale * __uint_as_float(uk[4 * q4]),
                                    P.scale * __uint_as_float(uk[4 * q4 + 1]),
                                    P.scale * __uint_as_float(uk[4 * q4 + 2]),
                                    P.scale * __uint_as_float(uk[4 * q4 + 3])));
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, int GM>
void launch_prep(const BwdParams& P, long long blocks, cudaStream_t s) {
  attn_bwd_prep_kernel<D, GM><<<(unsigned)blocks, 256, 0, s>>>(P);
}

template <int D>
cudaError_t launch(const AttnArgs& a, const AttnBwdArgs& g, cudaStream_t s) {
  static thread_local BwdParams P;
  P.q = static_cast<const __nv_bfloat16*>(a.q);
  for (int j = 0; j < kMaxBlocks; ++j) {
    P.kb[j] = static_cast<const __nv_bfloat16*>(a.k_blocks[j]);
    P.vb[j] = static_cast<const __nv_bfloat16*>(a.v_blocks[j]);
    P.dkb[j] = g.dk_blocks[j];
    P.dvb[j] = g.dv_blocks[j];
  }
  P.out = static_cast<const __nv_bfloat16*>(g.out);
  P.dout = static_cast<const __nv_bfloat16*>(g.dout);
  P.lse = g.lse;
  P.dq = g.dq;
  P.delta = g.delta;
  P.B = a.B;
  P.H = a.H;
  P.H_kv = a.H_kv;
  P.Q_LEN = a.Q_LEN;
  P.k = a.k;
  P.n_t = (a.Q_LEN + kTile - 1) / kTile;
  P.G = a.H / a.H_kv;
  P.scale = a.scale;
  P.scale_log2 = a.scale * kLog2e;
  for (int b = 0; b < a.B; ++b) P.T[b] = a.T[b];

  CUtensorMap tmQ, tmDO, tmK, tmV;
  cudaError_t e;
  if ((e = encode_tile_map(&tmQ, a.q, D, a.Q_LEN, a.B * a.H, kTile)) != cudaSuccess) return e;
  if ((e = encode_tile_map(&tmDO, g.dout, D, a.Q_LEN, a.B * a.H, kTile)) != cudaSuccess) return e;
  if ((e = encode_tile_map(&tmK, a.k_blocks[0], D, a.Q_LEN, a.B * a.H_kv, kTile)) != cudaSuccess)
    return e;
  if ((e = encode_tile_map(&tmV, a.v_blocks[0], D, a.Q_LEN, a.B * a.H_kv, kTile)) != cudaSuccess)
    return e;

  const long long rows = (long long)a.B * a.H_kv * a.Q_LEN;
  long long blocks = (rows + 7) / 8;
  if (blocks > 152 * 32) blocks = 152 * 32;
  prof_before(s, STT_KERNEL_ATTN_BWD_PREP);
  if (P.G == 1)
    launch_prep<D, 1>(P, blocks, s);
  else if (P.G == 2)
    launch_prep<D, 2>(P, blocks, s);
  else if (P.G <= 4)
    launch_prep<D, 4>(P, blocks, s);
  else
    launch_prep<D, 8>(P, blocks, s);
  prof_after(s);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  const unsigned grid = (unsigned)(P.n_t * a.H * a.B);
  e = cudaFuncSetAttribute(attn_bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           DqSmem<D>::alloc);
  if (e != cudaSuccess) return e;
  prof_before(s, STT_KERNEL_ATTN_BWD_DQ);
  attn_bwd_dq_kernel<D><<<grid, kThreads, DqSmem<D>::alloc, s>>>(P, tmQ, tmDO, tmK, tmV);
  prof_after(s);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  e = cudaFuncSetAttribute(attn_bwd_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           DkvSmem<D>::alloc);
  if (e != cudaSuccess) return e;
  prof_before(s, STT_KERNEL_ATTN_BWD_DKDV);
  attn_bwd_dkdv_kernel<D><<<grid, kThreads, DkvSmem<D>::alloc, s>>>(P, tmQ, tmDO, tmK, tmV);
  prof_after(s);
  return cudaGetLastError();
}

}  // namespace

size_t attn_bwd_workspace(int B, int H, int Q_LEN) {
  return ((size_t)B * H * Q_LEN * sizeof(float) + 15) / 16 * 16;
}

cudaError_t attn_bwd_launch(const AttnArgs& a, const AttnBwdArgs& g, cudaStream_t s) {
  if (a.D == 128) return launch<128>(a, g, s);
  if (a.D == 64) return launch<64>(a, g, s);
  return cudaErrorNotSupported;
}

STT_DEFINE_ERROR_ACCESSOR(attn_bwd_error_word)

}  // namespace stt
