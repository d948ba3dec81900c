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
//   * then folds the k diagonal suffix keys into the same online softmax as
//     per-row dot products on CUDA cores: TMA brings rows q0..q0+127 of K_j and
//     V_j (the only rows this query tile needs) into shared memory, and each
//     thread updates its O row (held in registers) with one key per block.
//     The online softmax is order independent, so taking the suffix keys last
//     gives the same result as any other order.
//
// Warp roles (352 threads, one CTA per 128-row query tile of one head):
//   warps 0-7  softmax: warps w and w+4 own the 32 query rows of TMEM lane
//              quarter w%4 and split the 128 key columns (and O's D columns)
//              in halves ("parts"); the row max is exchanged through shared
//              memory between the two warps of a quarter.
//              They load S from TMEM, mask, exponentiate, write P (bf16) back
//              over their own S columns in TMEM, rescale O in TMEM when the
//              running max grows by more than 2^8, and finish with the suffix
//              keys and O / lse.
//   warp 8     TMA producer (two lanes: Q and K, V): Q once, then K/V tiles
//              (2 stages), then the suffix K_j / V_j tiles through the same
//              buffers.
//   warp 9     S issuer (one lane): S(j) into TMEM buffer j % 3 as soon as
//              K(j) is in and O += P(j-3) V has read the buffer.
//   warp 10    P V issuer (one lane): O += P(j) V(j), P read from TMEM.  Two
//              issuing threads, because one thread's issue, commit and wait
//              latencies per key tile exceed the tensor cores' time for it.
#include "../../include/stt.h"
#include "attn_common.cuh"

namespace stt {
namespace {

constexpr int kStages = 2;
// Two softmax warps per TMEM lane quarter (each a 64-key half of the tile).
// Four per quarter (the code takes any of the two) measured slower, 882 vs
// 927 TFLOP/s: the four-way max exchange and the extra arrivals cost more than
// the added overlap gains.
constexpr int kSoftmax = 256;
constexpr int kSoftmaxWarps = kSoftmax / 32;  // barriers count one arrival per warp
constexpr int kParts = kSoftmaxWarps / 4;     // softmax warps per TMEM lane quarter
constexpr int kPartCols = kTile / kParts;     // key columns per softmax thread and tile
constexpr int kThreads = kSoftmax + 96;
constexpr int kWarpTma = kSoftmaxWarps, kWarpMma = kSoftmaxWarps + 1, kWarpPv = kSoftmaxWarps + 2;
static_assert(kPartCols == 32 || kPartCols == 64, "one or two 32-column TMEM loads per tile");
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P <= 2^8 between rescales

struct FwdParams {
  __nv_bfloat16* out;
  float* lse;
  int B, H, H_kv, Q_LEN, k, n_qt, G;
  float scale_log2;
  uint32_t inject;  // STT_INJECT_* test hooks (0 in normal use)
  int T[kMaxBatch];
};

// Tensor maps of the later blocks' keys and values (j = 1..k).
struct SfxMaps {
  CUtensorMap k[kMaxBlocks - 1];
  CUtensorMap v[kMaxBlocks - 1];
};

template <int D>
struct FwdSmem {
  static constexpr int kQ = kTile * D * 2;
  static constexpr int kKV = kTile * D * 2;
  static constexpr int q = 0;
  static constexpr int k0 = kQ;
  static constexpr int v0 = kQ + kStages * kKV;
  static constexpr int total = kQ + 2 * kStages * kKV;
  static constexpr int alloc = total + 1024;  // slack for 1024-byte alignment
};

// TMEM columns: S buffers at 0, 128 and 256 (P of softmax part p is written
// back into columns [p kPartCols, + kPartCols / 2) of its S buffer, inside the
// S columns that part itself reads), O at 384.
constexpr uint32_t kTmemCols = 512;
constexpr int kSBufs = 3;
constexpr uint32_t kColS0 = 0, kColO = kSBufs * kTile;
static_assert(kColO + 128 <= kTmemCols, "three S buffers and O fit in TMEM");

// Dot product of part p (of NP equal parts) of row r of two swizzled
// [128 x D] bf16 tiles in shared memory.
template <int D, int NP>
__device__ __forceinline__ float smem_part_row_dot(const unsigned char* a, const unsigned char* b,
                                                   int r, int p) {
  float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
  for (int c = p * (D / 8 / NP); c < (p + 1) * (D / 8 / NP); ++c) {
    const uint32_t off = swz_chunk_offset(r, c, kTile);
    const uint4 x = *reinterpret_cast<const uint4*>(a + off);
    const uint4 y = *reinterpret_cast<const uint4*>(b + off);
    acc0 = fmaf(bf16lo(x.x), bf16lo(y.x), acc0);
    acc1 = fmaf(bf16hi(x.x), bf16hi(y.x), acc1);
    acc0 = fmaf(bf16lo(x.y), bf16lo(y.y), acc0);
    acc1 = fmaf(bf16hi(x.y), bf16hi(y.y), acc1);
    acc0 = fmaf(bf16lo(x.z), bf16lo(y.z), acc0);
    acc1 = fmaf(bf16hi(x.z), bf16hi(y.z), acc1);
    acc0 = fmaf(bf16lo(x.w), bf16lo(y.w), acc0);
    acc1 = fmaf(bf16hi(x.w), bf16hi(y.w), acc1);
  }
  return acc0 + acc1;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ FwdParams P, const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmO, const __grid_constant__ SfxMaps sfx) {
  using L = FwdSmem<D>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // s_full / s_free per S buffer (S(j) uses buffer j % 3); p_full and o_done
  // alternate by tile parity so that a waiter can never miss a phase: when the
  // softmax warps hold S(j), O += P(j-3) V is complete (S(j) reused its
  // buffer), so O += P(j-2) V and O += P(j-1) V may both still be pending, and
  // one barrier counting every product could then not tell them apart.
  __shared__ uint64_t bar_q, bar_k_full[kStages], bar_v_full[kStages], bar_k_empty[kStages],
      bar_v_empty[kStages], bar_s_full[kSBufs], bar_s_free[kSBufs], bar_p_full[2], bar_o_done[2],
      bar_drain, bar_grp, bar_quad[4], bar_sfx_full[kStages], bar_sfx_empty[kStages];
  __shared__ uint32_t tmem_base;
  __shared__ float s_max[2][kParts][kTile];  // [tile parity][part][row] partial row max
  __shared__ float s_sum[kParts][kTile];     // [part][row] partial row sum
  __shared__ float s_dot[2][kParts][kTile];  // [block parity][part][row] partial suffix score

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nb = P.H * P.B;
  const int t = P.n_qt - 1 - (int)(blockIdx.x / nb);  // heaviest query tiles first
  const int bh = (int)(blockIdx.x % nb);
  const int b = bh / P.H, h = bh % P.H;
  const int hk = h / P.G;
  const int q0 = t * kTile;
  const int T = P.T[b];
  const int n_kv = causal_kv_tiles(q0, T);
  const int n_sfx = (q0 < T) ? P.k : 0;  // suffix blocks this tile needs (q0 < T => n_kv >= 1)

  if (tid == 0) {
    mbar_init(&bar_q, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_k_full[s], 1);
      mbar_init(&bar_v_full[s], 1);
      mbar_init(&bar_k_empty[s], 1);
      mbar_init(&bar_v_empty[s], 1);
      mbar_init(&bar_sfx_full[s], 2);  // one arrival per producer lane
      mbar_init(&bar_sfx_empty[s], kSoftmaxWarps);
    }
    for (int s = 0; s < kSBufs; ++s) {
      mbar_init(&bar_s_full[s], 1);
      mbar_init(&bar_s_free[s], 1);
    }
    for (int s = 0; s < 2; ++s) mbar_init(&bar_p_full[s], kSoftmaxWarps);
    for (int s = 0; s < 2; ++s) mbar_init(&bar_o_done[s], 1);
    mbar_init(&bar_drain, 2);  // one commit from each issuing thread
    mbar_init(&bar_grp, kSoftmaxWarps);
    for (int q = 0; q < 4; ++q) mbar_init(&bar_quad[q], kParts);  // warps q, q + 4, ...
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

  if (warp == kWarpTma) {
    // ------------------------------------------------------ TMA producer --
    // Lane 0 loads Q and the K tiles, lane 1 the V tiles, so that a K load
    // never queues behind a V stage that O += P V still holds.
    if (lane < 2 && n_kv > 0) {
      const bool is_k = lane == 0;
      const int bhk = b * P.H_kv + hk;
      // Test hook: the query tile is never loaded, so the S issuer's wait for
      // it runs out and every role of the CTA gives up in turn.
      const bool withhold_q = (P.inject & STT_INJECT_FWD_WITHHOLD_Q) != 0;
      if (is_k && !withhold_q) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        mbar_arrive_expect_tx(&bar_q, L::kQ);
        for (int cb = 0; cb < D / kColBlock; ++cb)
          tma_load_3d(sQ + cb * kTile * 128, &tmQ, &bar_q, cb * kColBlock, q0, bh);
      } else {
        tma_prefetch_desc(&tmV);
      }
      unsigned char* const base = smem + (is_k ? L::k0 : L::v0);
      const CUtensorMap* const tm = is_k ? &tmK : &tmV;
      uint64_t* const full = is_k ? bar_k_full : bar_v_full;
      uint64_t* const empty = is_k ? bar_k_empty : bar_v_empty;
      bool ok = true;
      int issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % kStages;
        const uint32_t ph = (uint32_t)(j / kStages) & 1u;
        if (j >= kStages && !mbar_wait(&empty[st], ph ^ 1u, STT_DEVERR_FWD_WAIT)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[st], L::kKV);
        for (int cb = 0; cb < D / kColBlock; ++cb)
          tma_load_3d(base + st * L::kKV + cb * kTile * 128, tm, &full[st], cb * kColBlock,
                      j * kTile, bhk);
        ++issued;
      }
      // Suffix tiles continue the K/V stage sequence: suffix block w + 1 takes
      // stage (n_kv + w) % kStages.  Its K half is loaded as soon as the S
      // product of the stage's last causal tile has read the K buffer, its V
      // half once the P V product has read the V buffer; a stage's later
      // suffix uses wait for the softmax warps to release it.  The suffix
      // barrier counts one arrival from each lane.
      int issued_s = 0;
      for (int w = 0; ok && w < n_sfx; ++w) {
        const int u = n_kv + w;
        const int st = u % kStages;
        const int m = w / kStages;  // earlier suffix uses of this stage
        if (m == 0) {
          if (u >= kStages &&
              !mbar_wait(&empty[st], (uint32_t)(u / kStages - 1) & 1u, STT_DEVERR_FWD_WAIT)) {
            ok = false;
            break;
          }
        } else if (!mbar_wait(&bar_sfx_empty[st], (uint32_t)(m - 1) & 1u, STT_DEVERR_FWD_WAIT)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&bar_sfx_full[st], L::kKV);
        for (int cb = 0; cb < D / kColBlock; ++cb)
          tma_load_3d(base + st * L::kKV + cb * kTile * 128, is_k ? &sfx.k[w] : &sfx.v[w],
                      &bar_sfx_full[st], cb * kColBlock, q0, bhk);
        ++issued_s;
      }
      if (!ok || withhold_q) {
        // Gave up (or nothing will consume the copies): let every copy this
        // lane issued land before the CTA exits.
        if (is_k && !withhold_q) mbar_wait(&bar_q, 0, STT_DEVERR_FWD_WAIT);
        for (int j = (issued > kStages ? issued - kStages : 0); j < issued; ++j)
          mbar_wait(&full[j % kStages], (uint32_t)(j / kStages) & 1u, STT_DEVERR_FWD_WAIT);
        for (int i = (issued_s > kStages ? issued_s - kStages : 0); i < issued_s; ++i)
          mbar_wait(&bar_sfx_full[(n_kv + i) % kStages], (uint32_t)(i / kStages) & 1u,
                    STT_DEVERR_FWD_WAIT);
      }
    }
  } else if (warp == kWarpMma || warp == kWarpPv) {
    // ------------------------------------------------------- MMA issuers --
    if (lane == 0 && n_kv > 0) {
      const uint32_t idS = idesc_bf16(128, kTile, false, false);
      const uint32_t idO = idesc_bf16(128, D, false, true);
      // Base descriptors; each MMA only advances the start address.
      const uint64_t dQ = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dK0 = sdesc_sw128(smem_u32(smem + L::k0), 16, 1024);
      const uint64_t dV0 = sdesc_sw128(smem_u32(smem + L::v0), kTile * 128, 1024);
      bool ok = true;
      if (warp == kWarpMma) {
        // S(j) = Q K_j^T into buffer j % 3 once O += P(j-3) V has read it.
        ok = mbar_wait(&bar_q, 0, STT_DEVERR_FWD_WAIT);
        for (int j = 0; ok && j < n_kv; ++j) {
          const int st = j % kStages, sb = j % kSBufs;
          ok = mbar_wait(&bar_k_full[st], (uint32_t)(j / kStages) & 1u, STT_DEVERR_FWD_WAIT);
          if (ok && j >= kSBufs)
            ok = mbar_wait(&bar_s_free[sb], (uint32_t)(j / kSBufs - 1) & 1u, STT_DEVERR_FWD_WAIT);
          if (!ok) break;
          tc_fence_after();
          const uint64_t dK = sdesc_add(dK0, st * L::kKV);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kTile * 128 + (kk & 3) * 32;
            umma_bf16_ss(tmem + kColS0 + sb * kTile, sdesc_add(dQ, off), sdesc_add(dK, off), idS,
                         kk > 0 ? 1u : 0u);
          }
          umma_commit(&bar_s_full[sb]);
          umma_commit(&bar_k_empty[st]);
        }
      } else {
        // O += P(i) V(i): A = P in TMEM (the keys of softmax part p live at
        // column p kPartCols of its S buffer, 8 columns per 16 keys), B = V
        // MN-major.
        for (int i = 0; ok && i < n_kv; ++i) {
          const int st = i % kStages, sb = i % kSBufs;
          ok = mbar_wait(&bar_p_full[i & 1], (uint32_t)(i >> 1) & 1u, STT_DEVERR_FWD_WAIT) &&
               mbar_wait(&bar_v_full[st], (uint32_t)(i / kStages) & 1u, STT_DEVERR_FWD_WAIT);
          if (!ok) break;
          tc_fence_after();
          const uint64_t dV = sdesc_add(dV0, st * L::kKV);
          const uint32_t aP = tmem + kColS0 + sb * kTile;
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            umma_bf16_ts(tmem + kColO,
                         aP + (kk / (kPartCols / 16)) * kPartCols + (kk % (kPartCols / 16)) * 8,
                         sdesc_add(dV, kk * 2048),
                         idO, (i > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&bar_o_done[i & 1]);
          umma_commit(&bar_s_free[sb]);
          umma_commit(&bar_v_empty[st]);
        }
      }
      // Every MMA issued by either thread is complete before TMEM or the stage
      // buffers are reused.
      umma_commit(&bar_drain);
      mbar_wait(&bar_drain, 0, STT_DEVERR_FWD_WAIT);
    }
  } else {
    // ------------------------------------------------------------ softmax --
    constexpr int DH = D / kParts;  // O columns per thread
    const int quarter = warp & 3, part = warp >> 2;
    const int r = quarter * 32 + lane;  // query row in the tile = TMEM lane
    const int qrow = q0 + r;
    const int lim = causal_row_limit(qrow, T);
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const float sl2 = P.scale_log2;
    uint32_t grp_uses = 0, quad_uses = 0;
    constexpr int NC = kPartCols / 32;  // 32-column TMEM loads per tile

    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; ok && j < n_kv; ++j) {
      const int sb = j % kSBufs;
      ok = warp_wait(&bar_s_full[sb], (uint32_t)(j / kSBufs) & 1u, STT_DEVERR_FWD_WAIT);
      if (!ok) break;
      tc_fence_after();
      const uint32_t scol = tmem + lane_off + kColS0 + sb * kTile + part * kPartCols;
      uint32_t s[NC][32];
      if constexpr (NC == 2)
        tmem_ld32x2(scol, scol + 32, s[0], s[1]);
      else
        tmem_ld32(scol, s[0]);

      const int cbase = j * kTile + part * kPartCols;
      // Maximum of the raw scores (the scale is > 0 and is applied to the
      // maximum alone), as eight independent three-input partial maxima.
      float mp[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mp[k] = -INFINITY;
      if (cbase + kPartCols - 1 <= lim) {
#pragma unroll
        for (int c2 = 0; c2 < NC; ++c2)
#pragma unroll
          for (int i = 0; i < 32; i += 2)
            mp[(i >> 1) & 7] = fmax3(mp[(i >> 1) & 7], __uint_as_float(s[c2][i]),
                                     __uint_as_float(s[c2][i + 1]));
      } else {
#pragma unroll
        for (int c2 = 0; c2 < NC; ++c2)
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float x = (cbase + c2 * 32 + i <= lim) ? __uint_as_float(s[c2][i]) : -INFINITY;
            s[c2][i] = __float_as_uint(x);
            mp[i & 7] = fmaxf(mp[i & 7], x);
          }
      }
      float mt = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                       fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7]))) * sl2;
      // Combine the parts' maxima (buffer double-buffered by tile parity);
      // only the warps of one lane quarter meet here.
      s_max[j & 1][part][r] = mt;
      ok = group_sync(&bar_quad[quarter], quad_uses, STT_DEVERR_FWD_WAIT);
      if (!ok) break;
#pragma unroll
      for (int p2 = 0; p2 < kParts; ++p2) mt = fmaxf(mt, s_max[j & 1][p2][r]);

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
      // p = 2^(s sl2 - m): two elements per packed fp32x2 FMA, and the row sum
      // in four packed partial accumulators.
      uint32_t pk[NC * 16];
      const uint64_t sl2x2 = f32x2(sl2, sl2), negm2 = f32x2(-m_use, -m_use);
      uint64_t rp[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) rp[k] = f32x2(0.f, 0.f);
#pragma unroll
      for (int c2 = 0; c2 < NC; ++c2)
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          float x0, x1;
          unpack_f32x2(fma_f32x2(f32x2(__uint_as_float(s[c2][i]), __uint_as_float(s[c2][i + 1])),
                                 sl2x2, negm2),
                       x0, x1);
          const float p0 = ex2(x0), p1 = ex2(x1);
          rp[(i >> 1) & 3] = add_f32x2(rp[(i >> 1) & 3], f32x2(p0, p1));
          pk[(c2 * 32 + i) >> 1] = pack_bf16(p0, p1);
        }
      float ra, rb;
      unpack_f32x2(add_f32x2(add_f32x2(rp[0], rp[1]), add_f32x2(rp[2], rp[3])), ra, rb);
      l_run += ra + rb;

      // P(j) goes to its own S buffer, and O += P(j) V(j) is ordered after
      // O += P(j-1) V(j-1) on the tensor pipe, so only a rescale of O has to
      // wait for the previous product (its commit also covers every earlier
      // one of the issuing thread).
      if (__any_sync(0xffffffffu, rescale_o)) {
        ok = warp_wait(&bar_o_done[(j - 1) & 1], (uint32_t)((j - 1) >> 1) & 1u, STT_DEVERR_FWD_WAIT);
        if (!ok) break;
        tc_fence_after();
        const uint32_t ocol = tmem + lane_off + kColO + part * DH;
        if constexpr (DH >= 32) {
#pragma unroll
          for (int c2 = 0; c2 < DH / 32; ++c2) {
            uint32_t o[32];
            tmem_ld32(ocol + c2 * 32, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(ocol + c2 * 32, o);
          }
        } else {
          uint32_t o[16];
          tmem_ld16(ocol, o);
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st16(ocol, o);
        }
        tmem_st_wait();
      }
      // P of this thread's keys (bf16 pairs) into the first columns of its own
      // S columns: the A operand of O += P V.
#pragma unroll
      for (int c2 = 0; c2 < NC; ++c2) {
        uint32_t pp[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) pp[c] = pk[c2 * 16 + c];
        tmem_st16(scol + c2 * 16, pp);
      }
      tmem_st_wait();
      tc_fence_before();
      warp_arrive(&bar_p_full[j & 1]);
    }
    if (ok && n_kv > 0) {
      // Every product is complete (the issuers' drain barrier fires once).
      ok = warp_wait(&bar_drain, 0, STT_DEVERR_FWD_WAIT);
      tc_fence_after();
    }

    // This thread's DH columns of the O row, in registers.
    float o[DH];
    if (ok && n_kv > 0) {
      const uint32_t ocol = tmem + lane_off + kColO + part * DH;
      if constexpr (DH >= 32) {
#pragma unroll
        for (int c2 = 0; c2 < DH / 32; ++c2) {
          uint32_t u[32];
          tmem_ld32(ocol + c2 * 32, u);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[c2 * 32 + i] = __uint_as_float(u[i]);
        }
      } else {
        uint32_t u[16];
        tmem_ld16(ocol, u);
#pragma unroll
        for (int i = 0; i < 16; ++i) o[i] = __uint_as_float(u[i]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < DH; ++i) o[i] = 0.f;
    }

    // ------------------------------------------- suffix keys (blocks 1..k) --
    // Query q < T sees key q of every later block: one score per block, a
    // register-level online-softmax update of this thread's O columns.
    // The threads of a row each take their part of the score's dot product
    // and exchange the parts through shared memory.
    const bool sfx_row = qrow < T;
    for (int w = 0; ok && w < n_sfx; ++w) {
      const int st = (n_kv + w) % kStages;
      ok = warp_wait(&bar_sfx_full[st], (uint32_t)(w / kStages) & 1u, STT_DEVERR_FWD_WAIT);
      if (!ok) break;
      const unsigned char* sK = smem + L::k0 + st * L::kKV;
      const unsigned char* sV = smem + L::v0 + st * L::kKV;
      s_dot[w & 1][part][r] = sfx_row ? smem_part_row_dot<D, kParts>(sQ, sK, r, part) : 0.f;
      ok = group_sync(&bar_grp, grp_uses, STT_DEVERR_FWD_WAIT);
      if (!ok) break;
      if (sfx_row) {
        float dsum = 0.f;
#pragma unroll
        for (int p2 = 0; p2 < kParts; ++p2) dsum += s_dot[w & 1][p2][r];
        const float sj = dsum * sl2;
        if (sj > m_run) {
          const float alpha = ex2(m_run - sj);  // 0 when m_run is -inf
          l_run *= alpha;
#pragma unroll
          for (int i = 0; i < DH; ++i) o[i] *= alpha;
          m_run = sj;
        }
        const float pj = ex2(sj - m_run);
        if (part == 0) l_run += pj;
#pragma unroll
        for (int c = 0; c < DH / 8; ++c) {
          const uint4 x = *reinterpret_cast<const uint4*>(sV + swz_chunk_offset(r, part * (DH / 8) + c, kTile));
          o[c * 8 + 0] = fmaf(pj, bf16lo(x.x), o[c * 8 + 0]);
          o[c * 8 + 1] = fmaf(pj, bf16hi(x.x), o[c * 8 + 1]);
          o[c * 8 + 2] = fmaf(pj, bf16lo(x.y), o[c * 8 + 2]);
          o[c * 8 + 3] = fmaf(pj, bf16hi(x.y), o[c * 8 + 3]);
          o[c * 8 + 4] = fmaf(pj, bf16lo(x.z), o[c * 8 + 4]);
          o[c * 8 + 5] = fmaf(pj, bf16hi(x.z), o[c * 8 + 5]);
          o[c * 8 + 6] = fmaf(pj, bf16lo(x.w), o[c * 8 + 6]);
          o[c * 8 + 7] = fmaf(pj, bf16hi(x.w), o[c * 8 + 7]);
        }
      }
      warp_arrive(&bar_sfx_empty[st]);
    }

    // ----------------------------------------------------------- epilogue --
    if (ok) {
      s_sum[part][r] = l_run;
      ok = group_sync(&bar_grp, grp_uses, STT_DEVERR_FWD_WAIT);
      l_run = 0.f;
#pragma unroll
      for (int p2 = 0; p2 < kParts; ++p2) l_run += s_sum[p2][r];
    }
    if (ok) {
      // O (bf16) is staged in the Q buffer, which every reader is done with
      // (the last S product and, behind the group barrier above, the suffix
      // dot products), in the swizzled layout of the tile loads, and leaves
      // through one TMA store; rows past Q_LEN are clipped by TMA.
      const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
      for (int c = 0; c < DH / 8; ++c)
        *reinterpret_cast<uint4*>(sQ + swz_chunk_offset(r, part * (DH / 8) + c, kTile)) =
            make_uint4(pack_bf16(o[c * 8 + 0] * inv_l, o[c * 8 + 1] * inv_l),
                       pack_bf16(o[c * 8 + 2] * inv_l, o[c * 8 + 3] * inv_l),
                       pack_bf16(o[c * 8 + 4] * inv_l, o[c * 8 + 5] * inv_l),
                       pack_bf16(o[c * 8 + 6] * inv_l, o[c * 8 + 7] * inv_l));
      if (part == 0 && qrow < P.Q_LEN)
        P.lse[(size_t)bh * P.Q_LEN + qrow] =
            l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
      fence_proxy_async_smem();
      ok = group_sync(&bar_grp, grp_uses, STT_DEVERR_FWD_WAIT);
      if (ok && tid == 0) {
        for (int cb = 0; cb < D / kColBlock; ++cb)
          tma_store_3d(&tmO, sQ + cb * kTile * 128, cb * kColBlock, q0, bh);
        bulk_commit_group();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  // The O store completes with the grid; its source must be read first.
  if (tid == 0) bulk_wait_group_read0();
}

template <int D>
cudaError_t launch(const AttnArgs& a, void* out, float* lse, cudaStream_t s) {
  CUtensorMap tmQ, tmK, tmV, tmO;
  static thread_local SfxMaps sfx;
  cudaError_t e;
  if ((e = bind_device_context()) != cudaSuccess) return e;
  if ((e = encode_tile_map(&tmQ, a.q, D, a.Q_LEN, a.B * a.H, kTile)) != cudaSuccess) return e;
  if ((e = encode_tile_map(&tmO, out, D, a.Q_LEN, a.B * a.H, kTile)) != cudaSuccess) return e;
  if ((e = encode_tile_map(&tmK, a.k_blocks[0], D, a.Q_LEN, a.B * a.H_kv, kTile)) != cudaSuccess)
    return e;
  if ((e = encode_tile_map(&tmV, a.v_blocks[0], D, a.Q_LEN, a.B * a.H_kv, kTile)) != cudaSuccess)
    return e;
  for (int j = 1; j <= a.k; ++j) {
    if ((e = encode_tile_map(&sfx.k[j - 1], a.k_blocks[j], D, a.Q_LEN, a.B * a.H_kv, kTile)) !=
        cudaSuccess)
      return e;
    if ((e = encode_tile_map(&sfx.v[j - 1], a.v_blocks[j], D, a.Q_LEN, a.B * a.H_kv, kTile)) !=
        cudaSuccess)
      return e;
  }
  static thread_local FwdParams P;
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
  P.inject = debug_inject();
  for (int b = 0; b < a.B; ++b) P.T[b] = a.T[b];
  const int smem = FwdSmem<D>::alloc;
  e = cudaFuncSetAttribute(attn_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)(P.n_qt * a.H * a.B);
  prof_before(s, STT_KERNEL_ATTN_FWD);
  attn_fwd_kernel<D><<<grid, kThreads, smem, s>>>(P, tmQ, tmK, tmV, tmO, sfx);
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
STT_DEFINE_BUDGET_SETTER(attn_fwd_set_wait_budget)

}  // namespace stt
