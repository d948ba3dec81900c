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
// Persistent: one CTA per SM walks a static list of work items, one 128-row
// query tile of one head each.  The list runs heaviest first -- query tiles
// from the last one down, within a tile the sequences by decreasing T, the
// heads innermost, so that the query heads of a KV group run side by side and
// share their K/V tiles in L2 -- and is dealt to the CTAs in snake order
// (round r left to right when r is even, right to left when odd), which keeps
// the CTAs' sums of key tiles within a few per cent of each other.  Every
// pipeline runs on across item boundaries: the next item's query tile goes to
// the second of two Q buffers and its first S products are issued while the
// softmax warps finish the current item's suffix keys and epilogue, so a
// tile's fixed costs (first loads, first S product, last P V product, O
// store) overlap other work instead of being paid one after another.
//
// Warp roles (384 threads):
//   warps 0-7  softmax: warps w and w+4 own the 32 query rows of TMEM lane
//              quarter w%4 and split the 128 key columns (and O's D columns)
//              in halves ("parts"); the row max is exchanged through shared
//              memory between the two warps of a quarter.
//              They load S from TMEM, mask, exponentiate, write P (bf16) back
//              over their own S columns in TMEM, rescale O in TMEM when the
//              running max grows by more than 2^8, and finish each item with
//              its suffix keys and O / lse (O staged in the item's Q buffer).
//   warp 8     TMA producer (two lanes: Q and K, V): per item the Q tile, then
//              its K/V tiles and its suffix K_j / V_j tiles through two shared
//              stages.
//   warp 9     S issuer (one lane): S(j) into TMEM buffer j % 3 as soon as
//              K(j) is in and O += P(j-3) V has read the buffer.
//   warp 10    P V issuer (one lane): O += P(j) V(j), P read from TMEM.  Two
//              issuing threads, because one thread's issue, commit and wait
//              latencies per key tile exceed the tensor cores' time for it.
//   warp 11    O store (one lane): sends an item's staged O tile out by TMA and
//              frees its Q buffer once the store has read it.
// Barrier phases and TMEM / stage buffer indices count S products, P V
// products and stage uses over the CTA's whole item sequence, not per item.
#include <algorithm>

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
constexpr int kWarpTma = kSoftmaxWarps, kWarpMma = kSoftmaxWarps + 1, kWarpPv = kSoftmaxWarps + 2,
              kWarpStore = kSoftmaxWarps + 3;
constexpr int kThreads = kSoftmax + 128;
static_assert(kPartCols == 32 || kPartCols == 64, "one or two 32-column TMEM loads per tile");
static_assert(kStages == 2, "the stage of unit u is u & 1");
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P <= 2^8 between rescales

struct FwdParams {
  float* lse;
  int B, H, H_kv, Q_LEN, k, n_qt, G;
  int n_items;      // n_qt * B * H work items
  float scale_log2;
  uint32_t inject;  // STT_INJECT_* test hooks (0 in normal use)
  int T[kMaxBatch];
  uint16_t bperm[kMaxBatch];  // sequences by decreasing T (stable)
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
  static constexpr int q = 0;  // two Q buffers (item parity)
  static constexpr int k0 = 2 * kQ;
  static constexpr int v0 = 2 * kQ + kStages * kKV;
  static constexpr int total = 2 * kQ + 2 * kStages * kKV;
  static constexpr int alloc = total + 1024;  // slack for 1024-byte alignment
};

// TMEM columns: S buffers at 0, 128 and 256 (P of softmax part p is written
// back into columns [p kPartCols, + kPartCols / 2) of its S buffer, inside the
// S columns that part itself reads), O at 384.
constexpr uint32_t kTmemCols = 512;
constexpr int kSBufs = 3;
constexpr uint32_t kColS0 = 0, kColO = kSBufs * kTile;
static_assert(kColO + 128 <= kTmemCols, "three S buffers and O fit in TMEM");

// One work item: query tile q0 of head h of sequence b.
struct Item {
  int b, h, bh, q0, T, n_kv, n_sfx;
};

// s_b / s_T: the sequences in work order (decreasing T) and their T, copied
// to shared memory at kernel start.
__device__ __forceinline__ Item item_at(const FwdParams& P, const uint16_t* s_b, const int* s_T,
                                        int w) {
  Item it;
  const int pi = w / P.H;
  it.h = w - pi * P.H;
  const int rank = pi / P.B;  // query tiles from the last one down
  const int idx = pi - rank * P.B;
  it.b = s_b[idx];
  it.T = s_T[idx];
  it.bh = it.b * P.H + it.h;
  it.q0 = (P.n_qt - 1 - rank) * kTile;
  it.n_kv = causal_kv_tiles(it.q0, it.T);
  it.n_sfx = (it.q0 < it.T) ? P.k : 0;  // q0 < T => n_kv >= 1
  return it;
}

// This CTA's item of round r (snake order), or -1 past the end of the list.
__device__ __forceinline__ int item_of_round(int r, int n_items) {
  const long long G = gridDim.x, c = blockIdx.x;
  const long long w = (long long)r * G + ((r & 1) ? G - 1 - c : c);
  return w < n_items ? (int)w : -1;
}

// Position in the sequence of K/V stage uses that the causal tiles and the
// suffix tiles of consecutive items share (use u takes stage u & 1).  A causal
// use signals k_full / v_full and is released by the tensor-core commits; a
// suffix use signals sfx_full and is released by the softmax warps.  Each
// role counts the uses of each kind per stage, so the parity of a use is its
// index among the same-kind uses of its stage.
struct StageSeq {
  uint32_t u = 0, c0 = 0, c1 = 0, s0 = 0, s1 = 0;
  uint32_t last_sfx = 0;  // bit st: the latest use of stage st was a suffix use

  // Next use (of the given kind): its stage, the parity of its full barrier,
  // and whether the stage held an earlier use, of which kind and with which
  // release parity.
  __device__ __forceinline__ int next(bool sfx, uint32_t& ph, bool& has_prev, bool& prev_sfx,
                                      uint32_t& prev_ph) {
    const int st = (int)(u & 1u);
    const uint32_t c = st ? c1 : c0, s = st ? s1 : s0;
    has_prev = u >= (uint32_t)kStages;
    prev_sfx = ((last_sfx >> st) & 1u) != 0;
    prev_ph = ((prev_sfx ? s : c) - 1u) & 1u;
    ph = (sfx ? s : c) & 1u;
    if (sfx) {
      if (st) ++s1; else ++s0;
      last_sfx |= 1u << st;
    } else {
      if (st) ++c1; else ++c0;
      last_sfx &= ~(1u << st);
    }
    ++u;
    return st;
  }
  __device__ __forceinline__ int next(bool sfx, uint32_t& ph) {
    bool hp, ps;
    uint32_t pp;
    return next(sfx, ph, hp, ps, pp);
  }
  // Skips n uses of one kind.
  __device__ __forceinline__ void skip(bool sfx, uint32_t n) {
    if (n == 0) return;
    const uint32_t a = (n + 1) >> 1, b = n >> 1;  // uses of stage u & 1, of the other one
    const uint32_t n0 = (u & 1u) ? b : a, n1 = (u & 1u) ? a : b;
    if (sfx) {
      s0 += n0;
      s1 += n1;
    } else {
      c0 += n0;
      c1 += n1;
    }
    const uint32_t touched = (n0 ? 1u : 0u) | (n1 ? 2u : 0u);
    last_sfx = sfx ? (last_sfx | touched) : (last_sfx & ~touched);
    u += n;
  }
};

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
                    const __grid_constant__ CUtensorMap tmO, const __grid_constant__ SfxMaps sfxm) {
  using L = FwdSmem<D>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // s_full / s_free / p_full per S buffer (S product g uses buffer g % 3).
  // p_full counts one arrival per softmax warp, and the warps of different
  // lane quarters never meet inside the tile loop: a quarter can be up to two
  // tiles ahead of another (S(g+3) waits for every warp's P(g)), so the
  // arrivals for g, g+1 and g+2 must go to three different barriers or a
  // phase could complete with one warp's P missing.  A parity wait is only
  // sound while the waited-for phase is the barrier's current or latest one,
  // so every waiter below either waits for every phase of its barrier in turn
  // or knows the phase before the one it waits for is complete.  o_done
  // alternates by the parity of g: when the softmax warps hold S(g) and
  // rescale O, O += P(g-3) V is complete (S(g) reused its buffer), so the
  // phase of o_done[(g-1) & 1] before the one of g-1 is complete, while
  // O += P(g-2) V may still be pending.  At the end of an item the last two
  // products may both be pending, so O is read after o_final, one phase per
  // item with key tiles.  q_full / q_empty / o_staged per Q buffer (item
  // parity).
  __shared__ uint64_t bar_q_full[2], bar_q_empty[2], bar_o_staged[2], bar_k_full[kStages],
      bar_v_full[kStages], bar_k_empty[kStages], bar_v_empty[kStages], bar_s_full[kSBufs],
      bar_s_free[kSBufs], bar_p_full[kSBufs], bar_o_done[2], bar_o_final, bar_drain, bar_quad[4],
      bar_sfx_full[kStages], bar_sfx_empty[kStages];
  __shared__ uint32_t tmem_base;
  __shared__ float s_max[2][kParts][kTile];  // [S product parity][part][row] partial row max
  __shared__ float s_sum[2][kParts][kTile];  // [item parity][part][row] partial row sum
  __shared__ float s_dot[2][kParts][kTile];  // [block parity][part][row] partial suffix score
  __shared__ uint16_t s_b[kMaxBatch];         // sequences in work order
  __shared__ int s_T[kMaxBatch];              // their valid lengths

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bar_q_full[x], 1);
      mbar_init(&bar_q_empty[x], 1);
      mbar_init(&bar_o_staged[x], kSoftmaxWarps);
      mbar_init(&bar_o_done[x], 1);
    }
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
      mbar_init(&bar_p_full[s], kSoftmaxWarps);
    }
    mbar_init(&bar_o_final, 1);
    mbar_init(&bar_drain, 2);  // one commit from each issuing thread
    for (int q = 0; q < 4; ++q) mbar_init(&bar_quad[q], kParts);  // warps q, q + 4, ...
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base, kTmemCols);
    tmem_relinquish();
  }
  for (int x = tid; x < P.B; x += kThreads) {
    const int b = P.bperm[x];
    s_b[x] = (uint16_t)b;
    s_T[x] = P.T[b];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;

  if (warp == kWarpTma) {
    // ------------------------------------------------------ TMA producer --
    // Lane 0 loads Q and the K tiles, lane 1 the V tiles, so that a K load
    // never queues behind a V stage that O += P V still holds.
    if (lane < 2) {
      const bool is_k = lane == 0;
      // Test hook: no query tile is ever loaded, so the S issuer's wait for
      // it runs out and every role of the CTA gives up in turn.
      const bool withhold_q = (P.inject & STT_INJECT_FWD_WITHHOLD_Q) != 0;
      if (is_k) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
      } else {
        tma_prefetch_desc(&tmV);
      }
      unsigned char* const base = smem + (is_k ? L::k0 : L::v0);
      const CUtensorMap* const tm = is_k ? &tmK : &tmV;
      uint64_t* const full = is_k ? bar_k_full : bar_v_full;
      uint64_t* const empty = is_k ? bar_k_empty : bar_v_empty;
      StageSeq seq;
      bool ok = true;
      // The barrier and parity of the latest copy into each stage and each Q
      // buffer (parity + 1; 0 = none), waited for on the failure path.
      uint64_t* pend_bar0 = nullptr;
      uint64_t* pend_bar1 = nullptr;
      uint32_t pend_ph0 = 0, pend_ph1 = 0, q_pend0 = 0, q_pend1 = 0;
      int i = 0;
      for (int r = 0; ok; ++r) {
        const int w = item_of_round(r, P.n_items);
        if (w < 0) break;
        const Item it = item_at(P, s_b, s_T, w);
        const int bhk = it.b * P.H_kv + it.h / P.G;
        if (is_k) {
          // The Q buffer of this item was last used by item i - 2, whose O
          // tile was staged there; the store frees it.
          const int qs = i & 1;
          if (i >= 2 && !mbar_wait(&bar_q_empty[qs], (uint32_t)((i >> 1) - 1) & 1u,
                                   STT_DEVERR_FWD_WAIT)) {
            ok = false;
            break;
          }
          if (!withhold_q) {
            if (it.n_kv > 0) {
              mbar_arrive_expect_tx(&bar_q_full[qs], L::kQ);
              for (int cb = 0; cb < D / kColBlock; ++cb)
                tma_load_3d(smem + L::q + qs * L::kQ + cb * kTile * 128, &tmQ, &bar_q_full[qs],
                            cb * kColBlock, it.q0, it.bh);
              (qs ? q_pend1 : q_pend0) = ((uint32_t)(i >> 1) & 1u) + 1u;
            } else {
              mbar_arrive(&bar_q_full[qs]);  // only the O staging uses the buffer
            }
          }
        }
        // Causal tiles, then the suffix tiles (rows q0.. of K_j / V_j).
        for (int j = 0; j < it.n_kv + it.n_sfx; ++j) {
          const bool sfx = j >= it.n_kv;
          uint32_t ph, prev_ph;
          bool has_prev, prev_sfx;
          const int st = seq.next(sfx, ph, has_prev, prev_sfx, prev_ph);
          if (has_prev && !mbar_wait(prev_sfx ? &bar_sfx_empty[st] : &empty[st], prev_ph,
                                     STT_DEVERR_FWD_WAIT)) {
            ok = false;
            break;
          }
          uint64_t* const fb = sfx ? &bar_sfx_full[st] : &full[st];
          const CUtensorMap* const m =
              sfx ? (is_k ? &sfxm.k[j - it.n_kv] : &sfxm.v[j - it.n_kv]) : tm;
          const int row = sfx ? it.q0 : j * kTile;
          mbar_arrive_expect_tx(fb, L::kKV);
          for (int cb = 0; cb < D / kColBlock; ++cb)
            tma_load_3d(base + st * L::kKV + cb * kTile * 128, m, fb, cb * kColBlock, row, bhk);
          if (st) {
            pend_bar1 = fb;
            pend_ph1 = ph;
          } else {
            pend_bar0 = fb;
            pend_ph0 = ph;
          }
        }
        ++i;
      }
      if (!ok || withhold_q) {
        // Gave up (or nothing will consume the copies): let every copy this
        // lane issued land before the CTA exits.
        if (q_pend0) mbar_wait(&bar_q_full[0], q_pend0 - 1u, STT_DEVERR_FWD_WAIT);
        if (q_pend1) mbar_wait(&bar_q_full[1], q_pend1 - 1u, STT_DEVERR_FWD_WAIT);
        if (pend_bar0) mbar_wait(pend_bar0, pend_ph0, STT_DEVERR_FWD_WAIT);
        if (pend_bar1) mbar_wait(pend_bar1, pend_ph1, STT_DEVERR_FWD_WAIT);
      }
    }
  } else if (warp == kWarpMma || warp == kWarpPv) {
    // ------------------------------------------------------- MMA issuers --
    if (lane == 0) {
      const uint32_t idS = idesc_bf16(128, kTile, false, false);
      const uint32_t idO = idesc_bf16(128, D, false, true);
      // Base descriptors; each MMA only advances the start address.
      const uint64_t dK0 = sdesc_sw128(smem_u32(smem + L::k0), 16, 1024);
      const uint64_t dV0 = sdesc_sw128(smem_u32(smem + L::v0), kTile * 128, 1024);
      StageSeq seq;
      uint32_t g = 0;  // S (or P V) products so far
      bool ok = true;
      int i = 0;
      for (int r = 0; ok; ++r) {
        const int w = item_of_round(r, P.n_items);
        if (w < 0) break;
        const Item it = item_at(P, s_b, s_T, w);
        if (warp == kWarpMma) {
          // S(g) = Q K_j^T into buffer g % 3 once O += P(g-3) V has read it.
          // Every item's q_full phase is waited for (an item without key tiles
          // completes it with a plain arrival), so the phases stay in turn.
          ok = mbar_wait(&bar_q_full[i & 1], (uint32_t)(i >> 1) & 1u, STT_DEVERR_FWD_WAIT);
          const uint64_t dQ = sdesc_sw128(smem_u32(smem + L::q + (i & 1) * L::kQ), 16, 1024);
          for (int j = 0; ok && j < it.n_kv; ++j, ++g) {
            uint32_t ph;
            const int st = seq.next(false, ph);
            const int sb = (int)(g % kSBufs);
            ok = mbar_wait(&bar_k_full[st], ph, STT_DEVERR_FWD_WAIT);
            if (ok && g >= (uint32_t)kSBufs)
              ok = mbar_wait(&bar_s_free[sb], (g / kSBufs - 1u) & 1u, STT_DEVERR_FWD_WAIT);
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
          // O += P(g) V: A = P in TMEM (the keys of softmax part p live at
          // column p kPartCols of its S buffer, 8 columns per 16 keys), B = V
          // MN-major.  The first product of an item overwrites O.
          for (int j = 0; ok && j < it.n_kv; ++j, ++g) {
            uint32_t ph;
            const int st = seq.next(false, ph);
            const int sb = (int)(g % kSBufs);
            ok = mbar_wait(&bar_p_full[sb], (g / kSBufs) & 1u, STT_DEVERR_FWD_WAIT) &&
                 mbar_wait(&bar_v_full[st], ph, STT_DEVERR_FWD_WAIT);
            if (!ok) break;
            tc_fence_after();
            const uint64_t dV = sdesc_add(dV0, st * L::kKV);
            const uint32_t aP = tmem + kColS0 + sb * kTile;
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              umma_bf16_ts(tmem + kColO,
                           aP + (kk / (kPartCols / 16)) * kPartCols + (kk % (kPartCols / 16)) * 8,
                           sdesc_add(dV, kk * 2048), idO, (j > 0 || kk > 0) ? 1u : 0u);
            umma_commit(&bar_o_done[g & 1]);
            umma_commit(&bar_s_free[sb]);
            umma_commit(&bar_v_empty[st]);
          }
          if (ok && it.n_kv > 0) umma_commit(&bar_o_final);  // the item's O is complete
        }
        seq.skip(true, (uint32_t)it.n_sfx);
        ++i;
      }
      // Every MMA issued by either thread is complete before TMEM or the stage
      // buffers are released.
      umma_commit(&bar_drain);
      mbar_wait(&bar_drain, 0, STT_DEVERR_FWD_WAIT);
    }
  } else if (warp == kWarpStore) {
    // ----------------------------------------------------------- O store --
    if (lane == 0) {
      tma_prefetch_desc(&tmO);
      int i = 0;
      for (int r = 0;; ++r) {
        const int w = item_of_round(r, P.n_items);
        if (w < 0) break;
        const Item it = item_at(P, s_b, s_T, w);
        const int qs = i & 1;
        if (!mbar_wait(&bar_o_staged[qs], (uint32_t)(i >> 1) & 1u, STT_DEVERR_FWD_WAIT)) break;
        // Rows past Q_LEN are clipped by TMA.
        for (int cb = 0; cb < D / kColBlock; ++cb)
          tma_store_3d(&tmO, smem + L::q + qs * L::kQ + cb * kTile * 128, cb * kColBlock, it.q0,
                       it.bh);
        bulk_commit_group();
        bulk_wait_group_read0();
        mbar_arrive(&bar_q_empty[qs]);
        ++i;
      }
    }
  } else {
    // ------------------------------------------------------------ softmax --
    constexpr int DH = D / kParts;  // O columns per thread
    const int quarter = warp & 3, part = warp >> 2;
    const int r = quarter * 32 + lane;  // query row in the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const float sl2 = P.scale_log2;
    // The two warps of a lane quarter hold the two parts of the same rows
    // and exchange partial maxima, suffix dot products and row sums through
    // shared memory behind their own barrier.
    uint32_t quad_uses = 0;
    constexpr int NC = kPartCols / 32;  // 32-column TMEM loads per tile
    StageSeq seq;
    uint32_t g = 0;        // S products so far
    uint32_t n_final = 0;  // items with key tiles so far (o_final phases)
    bool ok = true;
    int i = 0;
    for (int rr = 0; ok; ++rr) {
      const int w = item_of_round(rr, P.n_items);
      if (w < 0) break;
      const Item it = item_at(P, s_b, s_T, w);
      const int qs = i & 1;
      unsigned char* const sQ = smem + L::q + qs * L::kQ;
      const int qrow = it.q0 + r;
      const int lim = causal_row_limit(qrow, it.T);

      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; ok && j < it.n_kv; ++j) {
        const uint32_t gg = g + (uint32_t)j;
        const int sb = (int)(gg % kSBufs);
        ok = warp_wait(&bar_s_full[sb], (gg / kSBufs) & 1u, STT_DEVERR_FWD_WAIT);
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
            for (int x = 0; x < 32; x += 2)
              mp[(x >> 1) & 7] = fmax3(mp[(x >> 1) & 7], __uint_as_float(s[c2][x]),
                                       __uint_as_float(s[c2][x + 1]));
        } else {
#pragma unroll
          for (int c2 = 0; c2 < NC; ++c2)
#pragma unroll
            for (int x = 0; x < 32; ++x) {
              const float v = (cbase + c2 * 32 + x <= lim) ? __uint_as_float(s[c2][x]) : -INFINITY;
              s[c2][x] = __float_as_uint(v);
              mp[x & 7] = fmaxf(mp[x & 7], v);
            }
        }
        float mt = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                         fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7]))) * sl2;
        // Combine the parts' maxima (buffer double-buffered by product
        // parity); only the warps of one lane quarter meet here.
        s_max[gg & 1][part][r] = mt;
        ok = group_sync(&bar_quad[quarter], quad_uses, STT_DEVERR_FWD_WAIT);
        if (!ok) break;
#pragma unroll
        for (int p2 = 0; p2 < kParts; ++p2) mt = fmaxf(mt, s_max[gg & 1][p2][r]);

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
        // p = 2^(s sl2 - m): two elements per packed fp32x2 FMA, and the row
        // sum in four packed partial accumulators.
        uint32_t pk[NC * 16];
        const uint64_t sl2x2 = f32x2(sl2, sl2), negm2 = f32x2(-m_use, -m_use);
        uint64_t rp[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) rp[k] = f32x2(0.f, 0.f);
#pragma unroll
        for (int c2 = 0; c2 < NC; ++c2)
#pragma unroll
          for (int x = 0; x < 32; x += 2) {
            float x0, x1;
            unpack_f32x2(fma_f32x2(f32x2(__uint_as_float(s[c2][x]), __uint_as_float(s[c2][x + 1])),
                                   sl2x2, negm2),
                         x0, x1);
            const float p0 = ex2(x0), p1 = ex2(x1);
            rp[(x >> 1) & 3] = add_f32x2(rp[(x >> 1) & 3], f32x2(p0, p1));
            pk[(c2 * 32 + x) >> 1] = pack_bf16(p0, p1);
          }
        float ra, rb;
        unpack_f32x2(add_f32x2(add_f32x2(rp[0], rp[1]), add_f32x2(rp[2], rp[3])), ra, rb);
        l_run += ra + rb;

        // P(g) goes to its own S buffer, and O += P(g) V is ordered after
        // O += P(g-1) V on the tensor pipe, so only a rescale of O has to wait
        // for the previous product (its commit also covers every earlier one
        // of the issuing thread).
        if (__any_sync(0xffffffffu, rescale_o)) {
          ok = warp_wait(&bar_o_done[(gg - 1u) & 1u], ((gg - 1u) >> 1) & 1u, STT_DEVERR_FWD_WAIT);
          if (!ok) break;
          tc_fence_after();
          const uint32_t ocol = tmem + lane_off + kColO + part * DH;
          if constexpr (DH >= 32) {
#pragma unroll
            for (int c2 = 0; c2 < DH / 32; ++c2) {
              uint32_t o[32];
              tmem_ld32(ocol + c2 * 32, o);
#pragma unroll
              for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * alpha);
              tmem_st32(ocol + c2 * 32, o);
            }
          } else {
            uint32_t o[16];
            tmem_ld16(ocol, o);
#pragma unroll
            for (int x = 0; x < 16; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * alpha);
            tmem_st16(ocol, o);
          }
          tmem_st_wait();
        }
        // P of this thread's keys (bf16 pairs) into the first columns of its
        // own S columns: the A operand of O += P V.
#pragma unroll
        for (int c2 = 0; c2 < NC; ++c2) {
          uint32_t pp[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) pp[c] = pk[c2 * 16 + c];
          tmem_st16(scol + c2 * 16, pp);
        }
        tmem_st_wait();
        tc_fence_before();
        warp_arrive(&bar_p_full[sb]);
      }

      // This thread's DH columns of the O row, in registers, once the item's
      // last P V product is complete (its o_final commit covers the earlier
      // ones).  The next item's first P V product overwrites O only after
      // these warps have produced its P, i.e. after this read.
      float o[DH];
      if (ok && it.n_kv > 0) {
        ok = warp_wait(&bar_o_final, n_final & 1u, STT_DEVERR_FWD_WAIT);
        ++n_final;
        tc_fence_after();
      }
      if (ok && it.n_kv > 0) {
        const uint32_t ocol = tmem + lane_off + kColO + part * DH;
        if constexpr (DH == 64) {
          uint32_t u0[32], u1[32];
          tmem_ld32x2(ocol, ocol + 32, u0, u1);
#pragma unroll
          for (int x = 0; x < 32; ++x) {
            o[x] = __uint_as_float(u0[x]);
            o[32 + x] = __uint_as_float(u1[x]);
          }
        } else if constexpr (DH >= 32) {
#pragma unroll
          for (int c2 = 0; c2 < DH / 32; ++c2) {
            uint32_t u[32];
            tmem_ld32(ocol + c2 * 32, u);
#pragma unroll
            for (int x = 0; x < 32; ++x) o[c2 * 32 + x] = __uint_as_float(u[x]);
          }
        } else {
          uint32_t u[16];
          tmem_ld16(ocol, u);
#pragma unroll
          for (int x = 0; x < 16; ++x) o[x] = __uint_as_float(u[x]);
        }
      } else {
#pragma unroll
        for (int x = 0; x < DH; ++x) o[x] = 0.f;
      }
      g += (uint32_t)it.n_kv;
      seq.skip(false, (uint32_t)it.n_kv);

      // ----------------------------------------- suffix keys (blocks 1..k) --
      // Query q < T sees key q of every later block: one score per block, a
      // register-level online-softmax update of this thread's O columns.
      // The threads of a row (one per part, in the two warps of a lane
      // quarter) each take their part of the score's dot product and exchange
      // the parts through shared memory.
      const bool sfx_row = qrow < it.T;
      for (int w2 = 0; ok && w2 < it.n_sfx; ++w2) {
        uint32_t ph;
        const int st = seq.next(true, ph);
        ok = warp_wait(&bar_sfx_full[st], ph, STT_DEVERR_FWD_WAIT);
        if (!ok) break;
        const unsigned char* sK = smem + L::k0 + st * L::kKV;
        const unsigned char* sV = smem + L::v0 + st * L::kKV;
        s_dot[w2 & 1][part][r] = sfx_row ? smem_part_row_dot<D, kParts>(sQ, sK, r, part) : 0.f;
        ok = group_sync(&bar_quad[quarter], quad_uses, STT_DEVERR_FWD_WAIT);
        if (!ok) break;
        if (sfx_row) {
          float dsum = 0.f;
#pragma unroll
          for (int p2 = 0; p2 < kParts; ++p2) dsum += s_dot[w2 & 1][p2][r];
          const float sj = dsum * sl2;
          if (sj > m_run) {
            const float alpha = ex2(m_run - sj);  // 0 when m_run is -inf
            l_run *= alpha;
#pragma unroll
            for (int x = 0; x < DH; ++x) o[x] *= alpha;
            m_run = sj;
          }
          const float pj = ex2(sj - m_run);
          if (part == 0) l_run += pj;
#pragma unroll
          for (int c = 0; c < DH / 8; ++c) {
            const uint4 x =
                *reinterpret_cast<const uint4*>(sV + swz_chunk_offset(r, part * (DH / 8) + c, kTile));
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

      // --------------------------------------------------------- epilogue --
      if (ok) {
        s_sum[qs][part][r] = l_run;
        ok = group_sync(&bar_quad[quarter], quad_uses, STT_DEVERR_FWD_WAIT);
        l_run = 0.f;
#pragma unroll
        for (int p2 = 0; p2 < kParts; ++p2) l_run += s_sum[qs][p2][r];
      }
      // An item without key tiles never waits for its Q buffer on the way
      // here; the buffer is free once the producer has passed it.
      if (ok && it.n_kv == 0)
        ok = warp_wait(&bar_q_full[qs], (uint32_t)(i >> 1) & 1u, STT_DEVERR_FWD_WAIT);
      if (ok) {
        // O (bf16) is staged in the item's Q buffer, in the swizzled layout of
        // the tile loads: every S product of the item is complete, and each
        // thread overwrites only the chunks its own suffix dot products read.
        const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
        for (int c = 0; c < DH / 8; ++c)
          *reinterpret_cast<uint4*>(sQ + swz_chunk_offset(r, part * (DH / 8) + c, kTile)) =
              make_uint4(pack_bf16(o[c * 8 + 0] * inv_l, o[c * 8 + 1] * inv_l),
                         pack_bf16(o[c * 8 + 2] * inv_l, o[c * 8 + 3] * inv_l),
                         pack_bf16(o[c * 8 + 4] * inv_l, o[c * 8 + 5] * inv_l),
                         pack_bf16(o[c * 8 + 6] * inv_l, o[c * 8 + 7] * inv_l));
        if (part == 0 && qrow < P.Q_LEN)
          P.lse[(size_t)it.bh * P.Q_LEN + qrow] =
              l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
        fence_proxy_async_smem();
        warp_arrive(&bar_o_staged[qs]);
      }
      ++i;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
cudaError_t launch(const AttnArgs& a, float* lse, void* out, cudaStream_t s) {
  CUtensorMap tmQ, tmK, tmV, tmO;
  static thread_local SfxMaps sfxm;
  cudaError_t e;
  if ((e = bind_device_context()) != cudaSuccess) return e;
  if ((e = encode_tile_map(&tmQ, a.q, D, a.Q_LEN, a.B * a.H, kTile)) != cudaSuccess) return e;
  if ((e = encode_tile_map(&tmO, out, D, a.Q_LEN, a.B * a.H, kTile)) != cudaSuccess) return e;
  if ((e = encode_tile_map(&tmK, a.k_blocks[0], D, a.Q_LEN, a.B * a.H_kv, kTile)) != cudaSuccess)
    return e;
  if ((e = encode_tile_map(&tmV, a.v_blocks[0], D, a.Q_LEN, a.B * a.H_kv, kTile)) != cudaSuccess)
    return e;
  for (int j = 1; j <= a.k; ++j) {
    if ((e = encode_tile_map(&sfxm.k[j - 1], a.k_blocks[j], D, a.Q_LEN, a.B * a.H_kv, kTile)) !=
        cudaSuccess)
      return e;
    if ((e = encode_tile_map(&sfxm.v[j - 1], a.v_blocks[j], D, a.Q_LEN, a.B * a.H_kv, kTile)) !=
        cudaSuccess)
      return e;
  }
  static thread_local FwdParams P;
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
  const long long n_items = (long long)P.n_qt * a.H * a.B;
  if (n_items > 0x7fffffffll) return cudaErrorInvalidValue;
  if (n_items == 0) return cudaSuccess;
  P.n_items = (int)n_items;
  for (int b = 0; b < a.B; ++b) {
    P.T[b] = a.T[b];
    P.bperm[b] = (uint16_t)b;
  }
  std::stable_sort(P.bperm, P.bperm + a.B,
                   [&](uint16_t x, uint16_t y) { return a.T[x] > a.T[y]; });
  const int smem = FwdSmem<D>::alloc;
  e = cudaFuncSetAttribute(attn_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int sms = sm_count();
  const unsigned grid = (unsigned)(n_items < sms ? n_items : sms);
  prof_before(s, STT_KERNEL_ATTN_FWD);
  attn_fwd_kernel<D><<<grid, kThreads, smem, s>>>(P, tmQ, tmK, tmV, tmO, sfxm);
  prof_after(s);
  return cudaGetLastError();
}

}  // namespace

cudaError_t attn_fwd_launch(const AttnArgs& a, void* out, float* lse, cudaStream_t s) {
  if (a.D == 128) return launch<128>(a, lse, out, s);
  if (a.D == 64) return launch<64>(a, lse, out, s);
  return cudaErrorNotSupported;
}

STT_DEFINE_ERROR_ACCESSOR(attn_fwd_error_word)
STT_DEFINE_BUDGET_SETTER(attn_fwd_set_wait_budget)

}  // namespace stt
