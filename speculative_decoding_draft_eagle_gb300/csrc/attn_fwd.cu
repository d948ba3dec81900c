// attn_fwd.cu -- sparse-tree TTT attention, forward (SpecForge review, §三
// "稀疏树注意力", §四 "BlockMask 构造").
//
// At TTT step k a query q sees (i) keys 0..min(q, T-1) of the causal block 0
// and (ii) for q < T, key q of each later block j = 1..k.  The kernel:
//   * runs the causal block as a flash-style bf16 tcgen05 contraction: TMA
//     brings 128x128 Q/K/V tiles into swizzled shared memory, S = Q K^T and
//     O += P V accumulate in tensor memory (TMEM), fully masked key tiles are
//     never visited and the padded columns kv >= T are cut (tile count and
//     per-element limit);
//   * folds the k diagonal suffix keys into the same online softmax as per-row
//     dot products (CUDA cores): their scores seed the running max / sum
//     before the first tile, and their V rows are added in the epilogue.
//
// Warp roles (192 threads, one CTA per 128-row query tile of one head):
//   warps 0-3  softmax: thread r owns query row q0+r (= TMEM lane r); loads S
//              from TMEM, masks, exponentiates, writes P (bf16) to shared
//              memory, rescales O in TMEM when the running max grows by more
//              than 2^8, and writes O / lse in the epilogue.
//   warp 4     TMA producer (one lane): Q once, then K/V tiles, 2 stages.
//   warp 5     MMA issuer (one lane): S(j) into one of two TMEM buffers, then
//              O += P(j-1) V(j-1), so S(j+1) overlaps the softmax of tile j.
#include "../../include/stt.h"
#include "attn_common.cuh"

namespace stt {
namespace {

constexpr int kStages = 2;
constexpr int kThreads = 192;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P <= 2^8 between rescales

struct FwdParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* kb[kMaxBlocks];
  const __nv_bfloat16* vb[kMaxBlocks];
  __nv_bfloat16* out;
  float* lse;
  int B, H, H_kv, Q_LEN, k, n_qt, G;
  float scale_log2;
  int T[kMaxBatch];
};

template <int D>
struct FwdSmem {
  static constexpr int kQ = kTile * D * 2;
  static constexpr int kKV = kTile * D * 2;
  static constexpr int kP = kTile * kTile * 2;
  static constexpr int q = 0;
  static constexpr int k0 = kQ;
  static constexpr int v0 = kQ + kStages * kKV;
  static constexpr int p = kQ + 2 * kStages * kKV;
  static constexpr int total = p + kP;
  static constexpr int alloc = total + 1024;  // slack for 1024-byte alignment
};

// TMEM columns: S buffers at 0 and 128, O at 256.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColO = 256;

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ FwdParams P, const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
  using L = FwdSmem<D>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_q, bar_k_full[kStages], bar_v_full[kStages], bar_k_empty[kStages],
      bar_v_empty[kStages], bar_s_full[2], bar_s_free[2], bar_p_full, bar_o_done, bar_drain;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nb = P.H * P.B;
  const int t = P.n_qt - 1 - (int)(blockIdx.x / nb);  // heaviest query tiles first
  const int bh = (int)(blockIdx.x % nb);
  const int b = bh / P.H, h = bh % P.H;
  const int hk = h / P.G;
  const int q0 = t * kTile;
  const int T = P.T[b];
  const int n_kv = causal_kv_tiles(q0, T);

  if (tid == 0) {
    mbar_init(&bar_q, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_k_full[s], 1);
      mbar_init(&bar_v_full[s], 1);
      mbar_init(&bar_k_empty[s], 1);
      mbar_init(&bar_v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bar_s_full[s], 1);
      mbar_init(&bar_s_free[s], 128);
    }
    mbar_init(&bar_p_full, 128);
    mbar_init(&bar_o_done, 1);
    mbar_init(&bar_drain, 1);
    abort_flag = 0;
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
  unsigned char* sQ = smem + L::q;
  unsigned char* sP = smem + L::p;

  if (warp == 4) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0 && n_kv > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const int bhk = b * P.H_kv + hk;
      mbar_arrive_expect_tx(&bar_q, L::kQ);
      for (int cb = 0; cb < D / kColBlock; ++cb)
        tma_load_3d(sQ + cb * kTile * 128, &tmQ, &bar_q, cb * kColBlock, q0, bh);
      int issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % kStages;
        const uint32_t ph = (uint32_t)(j / kStages) & 1u;
        if (j >= kStages && !mbar_wait(&bar_k_empty[st], ph ^ 1u, STT_DEVERR_FWD_WAIT)) break;
        mbar_arrive_expect_tx(&bar_k_full[st], L::kKV);
        for (int cb = 0; cb < D / kColBlock; ++cb)
          tma_load_3d(smem + L::k0 + st * L::kKV + cb * kTile * 128, &tmK, &bar_k_full[st],
                      cb * kColBlock, j * kTile, bhk);
        if (j >= kStages && !mbar_wait(&bar_v_empty[st], ph ^ 1u, STT_DEVERR_FWD_WAIT)) {
          ++issued;
          break;
        }
        mbar_arrive_expect_tx(&bar_v_full[st], L::kKV);
        for (int cb = 0; cb < D / kColBlock; ++cb)
          tma_load_3d(smem + L::v0 + st * L::kKV + cb * kTile * 128, &tmV, &bar_v_full[st],
                      cb * kColBlock, j * kTile, bhk);
        ++issued;
      }
      if (issued < n_kv) {
        // Gave up: let every copy already issued land before the CTA exits.
        abort_flag = 1;
        mbar_wait(&bar_q, 0, STT_DEVERR_FWD_WAIT);
        for (int j = (issued > kStages ? issued - kStages : 0); j < issued; ++j) {
          const int st = j % kStages;
          const uint32_t ph = (uint32_t)(j / kStages) & 1u;
          mbar_wait(&bar_k_full[st], ph, STT_DEVERR_FWD_WAIT);
          mbar_wait(&bar_v_full[st], ph, STT_DEVERR_FWD_WAIT);
        }
      }
    }
  } else if (warp == 5) {
    // -------------------------------------------------------- MMA issuer --
    if (lane == 0 && n_kv > 0) {
      const uint32_t idS = idesc_bf16(128, kTile, false, false);
      const uint32_t idO = idesc_bf16(128, D, false, true);
      const uint32_t aQ = smem_u32(sQ), aP = smem_u32(sP);
      bool ok = mbar_wait(&bar_q, 0, STT_DEVERR_FWD_WAIT);
      auto issue_pv = [&](int i) -> bool {
        const int st = i % kStages;
        if (!mbar_wait(&bar_p_full, (uint32_t)i & 1u, STT_DEVERR_FWD_WAIT)) return false;
        if (!mbar_wait(&bar_v_full[st], (uint32_t)(i / kStages) & 1u, STT_DEVERR_FWD_WAIT))
          return false;
        tc_fence_after();
        const uint32_t aV = smem_u32(smem + L::v0 + st * L::kKV);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(aP + (kk >> 2) * kTile * 128 + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(aV + kk * 2048, kTile * 128, 1024);
          umma_bf16_ss(tmem + kColO, ad, bd, idO, (i > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&bar_o_done);
        umma_commit(&bar_v_empty[st]);
        return true;
      };
      for (int j = 0; ok && j < n_kv; ++j) {
        const int st = j % kStages, sb = j & 1;
        ok = mbar_wait(&bar_k_full[st], (uint32_t)(j / kStages) & 1u, STT_DEVERR_FWD_WAIT);
        if (ok && j >= 2)
          ok = mbar_wait(&bar_s_free[sb], (uint32_t)((j - 2) >> 1) & 1u, STT_DEVERR_FWD_WAIT);
        if (!ok) break;
        tc_fence_after();
        const uint32_t aK = smem_u32(smem + L::k0 + st * L::kKV);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(aQ + (kk >> 2) * kTile * 128 + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(aK + (kk >> 2) * kTile * 128 + (kk & 3) * 32, 16, 1024);
          umma_bf16_ss(tmem + kColS0 + sb * kTile, ad, bd, idS, kk > 0 ? 1u : 0u);
        }
        umma_commit(&bar_s_full[sb]);
        umma_commit(&bar_k_empty[st]);
        if (j >= 1) ok = issue_pv(j - 1);
      }
      if (ok) ok = issue_pv(n_kv - 1);
      if (!ok) abort_flag = 1;
      // Every MMA issued by this thread is complete before TMEM is released.
      umma_commit(&bar_drain);
      mbar_wait(&bar_drain, 0, STT_DEVERR_FWD_WAIT);
    }
  } else {
    // ------------------------------------------------------------ softmax --
    const int r = tid;  // 0..127 = TMEM lane = query row in the tile
    const int qrow = q0 + r;
    const int lim = causal_row_limit(qrow, T);
    const bool sfx_row = qrow < T;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const float sl2 = P.scale_log2;
    const size_t row_kv = ((size_t)(b * P.H_kv + hk) * P.Q_LEN + qrow) * D;

    // Suffix keys (one per later block) seed the running max and sum.
    float m_run = -INFINITY, l_run = 0.f;
    float sfx[kMaxBlocks - 1];
    if (sfx_row) {
      const __nv_bfloat16* qp = P.q + ((size_t)bh * P.Q_LEN + qrow) * D;
      for (int j = 1; j <= P.k; ++j) {
        const float s = dot_bf16_rows<D>(qp, P.kb[j] + row_kv) * sl2;
        sfx[j - 1] = s;
        m_run = fmaxf(m_run, s);
      }
      for (int j = 1; j <= P.k; ++j) l_run += ex2(sfx[j - 1] - m_run);
    }

    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int sb = j & 1;
      ok = warp_wait(&bar_s_full[sb], (uint32_t)(j >> 1) & 1u, STT_DEVERR_FWD_WAIT);
      if (!ok) break;
      tc_fence_after();
      uint32_t s[kTile / 32][32];
#pragma unroll
      for (int c = 0; c < kTile / 32; ++c) tmem_ld32(tmem + lane_off + kColS0 + sb * kTile + c * 32, s[c]);
      tc_fence_before();
      mbar_arrive(&bar_s_free[sb]);

      const int c0 = j * kTile;
      float mt = -INFINITY;
      if (c0 + kTile - 1 <= lim) {
#pragma unroll
        for (int c = 0; c < kTile / 32; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float x = __uint_as_float(s[c][i]) * sl2;
            s[c][i] = __float_as_uint(x);
            mt = fmaxf(mt, x);
          }
      } else {
#pragma unroll
        for (int c = 0; c < kTile / 32; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float x = (c0 + c * 32 + i <= lim) ? __uint_as_float(s[c][i]) * sl2 : -INFINITY;
            s[c][i] = __float_as_uint(x);
            mt = fmaxf(mt, x);
          }
      }
      float alpha = 1.f;
      bool rescale_o = false;
      const float m_new = fmaxf(m_run, mt);
      if (m_new > m_run + kRescaleThreshold) {
        alpha = ex2(m_run - m_new);
        l_run *= alpha;
        m_run = m_new;
        rescale_o = j > 0;
      }
      const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
      uint32_t pk[kTile / 2];
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < kTile / 32; ++c)
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float p0 = ex2(__uint_as_float(s[c][i]) - m_use);
          const float p1 = ex2(__uint_as_float(s[c][i + 1]) - m_use);
          rs += p0 + p1;
          pk[(c * 32 + i) >> 1] = pack_bf16(p0, p1);
        }
      l_run += rs;

      if (j > 0) {
        ok = warp_wait(&bar_o_done, (uint32_t)(j - 1) & 1u, STT_DEVERR_FWD_WAIT);
        if (!ok) break;
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, rescale_o)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          const uint32_t addr = tmem + lane_off + kColO + c * 32;
          tmem_ld32(addr, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(addr, o);
        }
        tmem_st_wait();
      }
      // P row -> swizzled K-major tile (A operand of O += P V).
#pragma unroll
      for (int c = 0; c < kTile / 8; ++c) {
        const uint4 v = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        *reinterpret_cast<uint4*>(sP + swz_chunk_offset(r, c, kTile)) = v;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bar_p_full);
    }
    if (ok && n_kv > 0) {
      ok = warp_wait(&bar_o_done, (uint32_t)(n_kv - 1) & 1u, STT_DEVERR_FWD_WAIT);
      tc_fence_after();
    }
    if (!ok) abort_flag = 1;

    // ----------------------------------------------------------- epilogue --
    const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
    const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
    if (sfx_row)
      for (int j = 1; j <= P.k; ++j) sfx[j - 1] = ex2(sfx[j - 1] - m_use);
    __nv_bfloat16* orow = P.out + ((size_t)bh * P.Q_LEN + qrow) * D;
    const bool in_range = qrow < P.Q_LEN;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      float o[32];
      if (ok && n_kv > 0) {
        uint32_t u[32];
        tmem_ld32(tmem + lane_off + kColO + c * 32, u);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(u[i]);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = 0.f;
      }
      if (sfx_row) {
        for (int j = 1; j <= P.k; ++j) {
          const uint4* vp = reinterpret_cast<const uint4*>(P.vb[j] + row_kv + c * 32);
          const float w = sfx[j - 1];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const uint4 x = __ldg(vp + q4);
            const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              o[q4 * 8 + 2 * e] = fmaf(w, bf16lo(xs[e]), o[q4 * 8 + 2 * e]);
              o[q4 * 8 + 2 * e + 1] = fmaf(w, bf16hi(xs[e]), o[q4 * 8 + 2 * e + 1]);
            }
          }
        }
      }
      if (in_range) {
        uint4* op = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          op[q4] = make_uint4(pack_bf16(o[q4 * 8 + 0] * inv_l, o[q4 * 8 + 1] * inv_l),
                              pack_bf16(o[q4 * 8 + 2] * inv_l, o[q4 * 8 + 3] * inv_l),
                              pack_bf16(o[q4 * 8 + 4] * inv_l, o[q4 * 8 + 5] * inv_l),
                              pack_bf16(o[q4 * 8 + 6] * inv_l, o[q4 * 8 + 7] * inv_l));
      }
    }
    if (in_range)
      P.lse[(size_t)bh * P.Q_LEN + qrow] = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
cudaError_t launch(const AttnArgs& a, void* out, float* lse, cudaStream_t s) {
  CUtensorMap tmQ, tmK, tmV;
  cudaError_t e;
  if ((e = encode_tile_map(&tmQ, a.q, D, a.Q_LEN, a.B * a.H, kTile)) != cudaSuccess) return e;
  if ((e = encode_tile_map(&tmK, a.k_blocks[0], D, a.Q_LEN, a.B * a.H_kv, kTile)) != cudaSuccess)
    return e;
  if ((e = encode_tile_map(&tmV, a.v_blocks[0], D, a.Q_LEN, a.B * a.H_kv, kTile)) != cudaSuccess)
    return e;
  static thread_local FwdParams P;
  P.q = static_cast<const __nv_bfloat16*>(a.q);
  for (int j = 0; j < kMaxBlocks; ++j) {
    P.kb[j] = static_cast<const __nv_bfloat16*>(a.k_blocks[j]);
    P.vb[j] = static_cast<const __nv_bfloat16*>(a.v_blocks[j]);
  }
  P.out = static_cast<__nv_bfloat16*>(out);
  P.lse = lse;
  P.B = a.B;
  P.H = a.H;
  P.H_kv = a.H_kv;
  P.Q_LEN = a.Q_LEN;
  P.k = a.k;
  P.n_qt = (a.Q_LEN + kTile - 1) / kTile;
  P.G = a.H / a.H_kv;
  P.scale_log2 = a.scale * kLog2e;
  for (int b = 0; b < a.B; ++b) P.T[b] = a.T[b];
  const int smem = FwdSmem<D>::alloc;
  e = cudaFuncSetAttribute(attn_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)(P.n_qt * a.H * a.B);
  prof_before(s, STT_KERNEL_ATTN_FWD);
  attn_fwd_kernel<D><<<grid, kThreads, smem, s>>>(P, tmQ, tmK, tmV);
  prof_after(s);
  return cudaGetLastError();
}

}  // namespace

cudaError_t attn_fwd_launch(const AttnArgs& a, void* out, float* lse, cudaStream_t s) {
  if (a.D == 128) return launch<128>(a, out, lse, s);
  if (a.D == 64) return launch<64>(a, out, lse, s);
  return cudaErrorNotSupported;
}

STT_DEFINE_ERROR_ACCESSOR(attn_fwd_error_word)

}  // namespace stt
