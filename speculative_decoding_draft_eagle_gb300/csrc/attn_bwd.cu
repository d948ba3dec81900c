// attn_bwd.cu -- sparse-tree TTT attention, backward.
//
// The page trains through the masked attention (SpecForge review, §三
// "稀疏树注意力": FlexAttention streams the computation and keeps no
// intermediate activations), so the backward is the derivative of the masked
// softmax attention, with P recomputed from the saved logsumexp:
//     Delta_q = sum_d dO * O,  P = exp(S - lse),  dS = P (dP - Delta),
//     dq = scale dS Kc,  dKc = scale dS^T q,  dVc = P^T dO.
//
// Two kernels, in stream order:
//   1. prep (CUDA cores fed by bulk copies, one CTA per SM walking units of
//      rows of one (b, KV head); per (b, KV head, row q) a lane group): Delta
//      for every query head of the group; the whole backward of the diagonal
//      suffix keys (q < T, blocks j = 1..k: one key per query, so dK_j / dV_j
//      row q is owned by one lane group and written directly); dq initialised
//      with the suffix part; dK_0 / dV_0 zeroed for the causal kernel's
//      accumulation.
//   2. causal (tcgen05, one CTA per 128-row key tile of a subgroup of the
//      query heads of one KV group, looping over the heads' query tiles that
//      see it, head after head): S^T = K Q^T and dP^T = V dO^T in
//      TMEM; 8 compute warps form P^T (written back into TMEM as bf16), then
//      dS^T (written to shared memory as bf16); dV += P^T dO (A from TMEM),
//      dK += dS^T Q and dQ = dS K (A = the dS^T tile read MN-major, i.e.
//      transposed) run on the tensor cores.  The MMA warp issues S^T(i+1)
//      right after dV(i), so it runs while the compute warps form dS(i).  dV
//      and dK stay in TMEM across the query tiles of all the subgroup's heads.
//      P^T is formed by a warp-uniform choice of a body with or without the
//      visibility test, and carries the attention scale (so dS, dQ and dK do).
//      Each tile's dQ is read out
//      of TMEM, staged in shared memory and added to the fp32 dq by TMA
//      reduce-add (issued by the producer warp, which releases each staging
//      buffer as soon as TMA has read it); the final dK / dV of the key tile
//      are reduce-added the same way into dK_0 / dV_0, once per subgroup.
// Every causal score entry costs 5 tensor-core products (the useful 10*D
// flops); dq, dK_0 and dV_0 receive their partial sums in arrival order.
#include "../../include/stt.h"
#include "attn_common.cuh"

namespace stt {
namespace {

// warps 0-7 compute, 8 TMA, 9 and 14 MMA issue, 10-13 dQ epilogue
constexpr int kThreads = 480;
constexpr int kCompute = 256;
constexpr int kComputeWarps = kCompute / 32;  // barriers count one arrival per warp
constexpr int kWarpTma = 8, kWarpMma = 9, kWarpEpi = 10, kWarpMma2 = 14;
// Heads per group of key-tile CTAs scheduled together: as many as keep their
// Q, dO (bf16) and dq (fp32) -- 8 bytes per element -- within kChunkBytes of L2.
constexpr long long kChunkBytes = 64ll << 20;
constexpr int kHeadChunkMax = 16;
constexpr int kEpiWarps = 4;  // one per TMEM lane quarter (warp % 4)

struct BwdParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* kb[kMaxBlocks];
  const __nv_bfloat16* vb[kMaxBlocks];
  const __nv_bfloat16* out;
  const __nv_bfloat16* dout;
  const float* lse;
  float* dq;                // fp32 dq accumulator (the caller's dq, or workspace)
  void* dkb[kMaxBlocks];    // the caller's dK_j / dV_j (fp32, or bf16 with kBwdBf16)
  void* dvb[kMaxBlocks];
  float* dk0;               // fp32 accumulators of dK_0 / dV_0 (the caller's, or workspace)
  float* dv0;
  float* delta;
  int B, H, H_kv, Q_LEN, k, n_t, G;
  int g_sub;                // query heads per CTA (a divisor of G, all of one KV group)
  int chunk_subs;           // head subgroups per group of CTAs scheduled together
  int accumulate;           // add into dK_j / dV_j, j >= 1 (read-modify-write)
  int zero_acc0;            // the prep kernel zeroes dk0 / dv0 first
  float scale, scale_log2;
  float log2_scale;         // log2(scale): folds scale into P in the causal kernel
  float inv_scale;
  int T[kMaxBatch];
};

// Byte offsets of the workspace parts, each 256-byte aligned.
struct WorkspaceLayout {
  size_t delta, dq, dk0, dv0, total;
};
inline size_t align256(size_t x) { return (x + 255) / 256 * 256; }
inline WorkspaceLayout workspace_layout(int B, int H, int H_kv, int D, int Q_LEN, uint32_t flags) {
  WorkspaceLayout W{};
  W.delta = 0;
  W.total = align256((size_t)B * H * Q_LEN * sizeof(float));
  if (flags & kBwdBf16) {
    W.dq = W.total;
    W.total += align256((size_t)B * H * Q_LEN * D * sizeof(float));
    W.dk0 = W.total;
    W.total += align256((size_t)B * H_kv * Q_LEN * D * sizeof(float));
    W.dv0 = W.total;
    W.total += align256((size_t)B * H_kv * Q_LEN * D * sizeof(float));
  }
  return W;
}

// Sum over the L lanes of an aligned lane group (L a power of two <= 32).
template <int L>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = L / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Four fp32 values of a gradient row into fp32 (OUT = float) or bf16 (OUT =
// __nv_bfloat16, rounded to nearest even) memory at element `off` of `base`;
// with `acc` they are added to what is there (in fp32, then rounded once).
// Overwritten rows go out with streaming stores: this kernel never reads them.
template <typename OUT>
__device__ __forceinline__ void put_grad4(void* base, size_t off, const float* v, bool acc) {
  if constexpr (sizeof(OUT) == 4) {
    float4* p = reinterpret_cast<float4*>(static_cast<float*>(base) + off);
    if (acc) {
      const float4 x = *p;
      *p = make_float4(x.x + v[0], x.y + v[1], x.z + v[2], x.w + v[3]);
    } else {
      __stcs(p, make_float4(v[0], v[1], v[2], v[3]));
    }
  } else {
    uint2* p = reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(base) + off);
    if (acc) {
      const uint2 x = *p;
      *p = make_uint2(pack_bf16(bf16lo(x.x) + v[0], bf16hi(x.x) + v[1]),
                      pack_bf16(bf16lo(x.y) + v[2], bf16hi(x.y) + v[3]));
    } else {
      __stcs(p, make_uint2(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3])));
    }
  }
}

// Row r, 16-byte chunk w of a swizzled [128 rows x 128 bytes] staging block.
__device__ __forceinline__ uint32_t swz128(int r, int w) {
  return (uint32_t)(r * 128 + ((w ^ (r & 7)) << 4));
}

// ------------------------------------------------------------------ prep --
// The prep kernel streams: per (b, KV head, row q) it reads the O, dO (and,
// with suffix keys, q) rows of the group's query heads and the K_j, V_j rows,
// and writes Delta, dq, dK_j, dV_j (and zeroed dK_0 / dV_0 rows); a handful
// of flops per byte.  Units of R consecutive rows q0.. of one (b, KV head) are
// dealt round robin to one CTA per SM.  Warp kComputeWarps (one lane) copies
// each unit into a ring of shared-memory slots, one [rows x D] bf16 block per
// slot and bulk copy, as far ahead as the ring reaches (176 KB per SM in
// flight), in groups that complete on one mbarrier: the O and dO blocks of
// the group's heads; when the unit has rows q < T and k > 0, their q blocks;
// then K_j with V_j for j = 1..k (rows q < T only).  The compute warps take
// each unit together and give a slot back as soon as every warp has read it
// into registers.  L = D/8 lanes serve one (row, head half); lane l holds
// elements [4l, 4l + 4) and [D/2 + 4l, +4) of the row as fp32 pairs (packed
// f32x2 arithmetic), so each 16-byte fp32 store of a lane group writes 2D
// contiguous bytes.  Groups of eight heads are split between two lane groups
// per row (SH = 2), which add their dK_j / dV_j partial sums with one shuffle.
// GM is the compile-time bound of the group size; head slots past G hold zeros.
template <int D, int GM>
struct PrepCfg {
  static constexpr int L = D / 8;                // lanes per (row, head half)
  static constexpr int SH = GM >= 8 ? 2 : 1;     // lane groups sharing a row's heads
  static constexpr int GH = GM / SH;             // head slots per thread
  // Twelve warps in all, three per SM sub-partition, so that a thread may
  // hold up to 168 registers (four warps per sub-partition would cap it at
  // 128 and spill the per-head values).
  static constexpr int kComputeWarps = 11;
  static constexpr int kCompute = kComputeWarps * 32;
  static constexpr int kThreads = kCompute + 32;  // + the copy warp
  static constexpr int R = kCompute / (L * SH);  // query rows per unit
  static constexpr int kSlotB = R * D * 2;       // one [R x D] bf16 block (5.5 KB / SH)
  static constexpr int kLogSlots = SH == 1 ? 5 : 6;
  static constexpr int kSlots = 1 << kLogSlots;  // 176 KB of slots
  static constexpr int kSmem = kSlots * kSlotB;
  static_assert(2 * GM <= kSlots, "a unit's O and dO blocks fit in the ring at once");
  static_assert(kSlotB % 16 == 0 && (D * 2) % 16 == 0, "bulk copies move 16-byte multiples");
};

// Elements [4l, 4l + 4) and [D/2 + 4l, D/2 + 4l + 4) of a bf16 row as four
// fp32 pairs.
template <int D>
__device__ __forceinline__ void lds_row8(const unsigned char* row, int l, uint64_t (&v)[4]) {
  const uint2 a = *reinterpret_cast<const uint2*>(row + 8 * l);
  const uint2 b = *reinterpret_cast<const uint2*>(row + D + 8 * l);
  v[0] = f32x2(bf16lo(a.x), bf16hi(a.x));
  v[1] = f32x2(bf16lo(a.y), bf16hi(a.y));
  v[2] = f32x2(bf16lo(b.x), bf16hi(b.x));
  v[3] = f32x2(bf16lo(b.y), bf16hi(b.y));
}

// Sum of the four pair products a[m] b[m] (both halves).
__device__ __forceinline__ float dot_pairs(const uint64_t (&a)[4], const uint64_t (&b)[4]) {
  uint64_t acc = mul_f32x2(a[0], b[0]);
  acc = fma_f32x2(a[1], b[1], acc);
  acc = fma_f32x2(a[2], b[2], acc);
  acc = fma_f32x2(a[3], b[3], acc);
  float lo, hi;
  unpack_f32x2(acc, lo, hi);
  return lo + hi;
}

// Sums of V values over the L lanes of an aligned lane group (V <= L, both
// powers of two) by a reduce-scatter butterfly: at level t (offset L >> (t+1))
// each lane keeps half of its current values, adding its partner's copy of
// them, and sends the other half; after log2 V levels a lane holds one value
// index, summed over the rest of the group by plain levels.  log2 V + log2 L
// shuffles where one butterfly per value takes V log2 L.  Returns the total
// of value scatter_index<L, V>(lane).
template <int L, int V>
__device__ __forceinline__ float reduce_scatter(float (&x)[V], int lane) {
  constexpr int LV = V == 1 ? 0 : V == 2 ? 1 : V == 4 ? 2 : 3;
  static_assert(V == (1 << LV) && V <= L, "V: a power of two, at most L");
#pragma unroll
  for (int t = 0; t < LV; ++t) {
    const int o = L >> (t + 1);
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int m = 0; m < (V >> (t + 1)); ++m) {
      const float lo = x[m], hi = x[m + (V >> (t + 1))];
      const float keep = up ? hi : lo, send = up ? lo : hi;
      x[m] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  float v = x[0];
#pragma unroll
  for (int o = L >> (LV + 1); o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
// The value index whose total reduce_scatter<L, V> leaves in `lane`, and the
// lane (within the group) that holds the total of value index v.
template <int L, int V>
__device__ __forceinline__ int scatter_index(int lane) {
  int v = 0;
#pragma unroll
  for (int t = 0; (V >> (t + 1)) > 0; ++t)
    if (lane & (L >> (t + 1))) v += V >> (t + 1);
  return v;
}
template <int L, int V>
__host__ __device__ constexpr int scatter_lane(int v) {
  int l = 0;
  for (int t = 0; (V >> (t + 1)) > 0; ++t)
    if (v & (V >> (t + 1))) l += L >> (t + 1);
  return l;
}

template <int D, int GM, typename OUT>
__global__ void __launch_bounds__(PrepCfg<D, GM>::kThreads, 1)
    attn_bwd_prep_kernel(const __grid_constant__ BwdParams P) {
  using C = PrepCfg<D, GM>;
  constexpr int L = C::L, SH = C::SH, GH = C::GH, R = C::R, NS = C::kSlots, LNS = C::kLogSlots;
  extern __shared__ __align__(128) unsigned char prep_smem[];
  __shared__ uint64_t bar_full[NS], bar_empty[NS];
  if ((smem_u32(prep_smem) & 15u) != 0) {
    if (threadIdx.x == 0) record_error(STT_DEVERR_SMEM_ALIGN);
    return;
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = P.G;
  const int n_qb = (P.Q_LEN + R - 1) / R;
  const long long n_units = (long long)P.B * P.H_kv * n_qb;
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], C::kComputeWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  // Unit u: rows [q0, q0 + R) of (b, KV head hk); nrows of them exist
  // (q < Q_LEN) and the first nv have suffix keys (q < T, k > 0).
  struct Unit {
    int b, hk, q0, nrows, nv;
  };
  auto unit_at = [&](long long u) {
    Unit x;
    const long long bhk = u / n_qb;
    x.q0 = (int)(u - bhk * n_qb) * R;
    x.b = (int)(bhk / P.H_kv);
    x.hk = (int)(bhk - (long long)x.b * P.H_kv);
    x.nrows = min(R, P.Q_LEN - x.q0);
    const int T = P.T[x.b];
    x.nv = (P.k > 0 && x.q0 < T) ? min(R, T - x.q0) : 0;
    return x;
  };

  if (warp == C::kComputeWarps) {
    // ------------------------------------------------------------- copies --
    if (lane == 0) {
      uint32_t seq = 0;  // slots filled so far; slot seq % NS, use seq / NS
      bool ok = true;
      // Slots [seq, seq + cnt) take cnt blocks of `rows` rows (src(c) for
      // block c); all their bytes complete on the first slot's barrier, whose
      // phase the compute warps wait for; the others' phases are completed
      // at once so that every slot's barrier keeps one phase per use.
      auto put_group = [&](int cnt, int rows, auto src) {
        for (int c = 0; ok && c < cnt; ++c) {
          const uint32_t n = seq + c;
          if (n >= (uint32_t)NS)
            ok = mbar_wait(&bar_empty[n & (NS - 1)], ((n >> LNS) - 1u) & 1u, STT_DEVERR_BWD_WAIT);
        }
        if (!ok) return;
        const uint32_t bytes = (uint32_t)rows * D * 2;
        uint64_t* bar = &bar_full[seq & (NS - 1)];
        mbar_arrive_expect_tx(bar, bytes * cnt);
        for (int c = 1; c < cnt; ++c) mbar_arrive(&bar_full[(seq + c) & (NS - 1)]);
        for (int c = 0; c < cnt; ++c)
          bulk_load(prep_smem + (size_t)((seq + c) & (NS - 1)) * C::kSlotB, src(c), bytes, bar);
        seq += cnt;
      };
      for (long long u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
        const Unit x = unit_at(u);
        // row q0 of query head hk G of sequence b; head h is Q_LEN rows further
        const size_t hq = ((size_t)x.b * P.H + (size_t)x.hk * G) * P.Q_LEN + x.q0;
        put_group(2 * G, x.nrows, [&](int c) {
          const __nv_bfloat16* t = c < G ? P.out : P.dout;
          return t + (hq + (size_t)(c < G ? c : c - G) * P.Q_LEN) * D;
        });
        if (x.nv > 0) {
          put_group(G, x.nv, [&](int c) { return P.q + (hq + (size_t)c * P.Q_LEN) * D; });
          const size_t kvo = (((size_t)x.b * P.H_kv + x.hk) * P.Q_LEN + x.q0) * D;
          for (int j = 1; ok && j <= P.k; ++j)
            put_group(2, x.nv, [&](int c) { return (c == 0 ? P.kb[j] : P.vb[j]) + kvo; });
        }
      }
      // Every copy issued lands before the CTA exits (on the normal path the
      // compute warps have waited for all of them already): the last use of
      // each slot is complete once its phase is.
      for (uint32_t n = seq > (uint32_t)NS ? seq - NS : 0u; n < seq; ++n)
        mbar_wait(&bar_full[n & (NS - 1)], (n >> LNS) & 1u, STT_DEVERR_BWD_WAIT);
    }
    return;
  }

  // ----------------------------------------------------------- compute --
  const int r = tid / (L * SH), hh = (tid / L) % SH, l = tid % L;
  const int e0 = 4 * l, e1 = D / 2 + 4 * l;  // this lane's two 4-element column groups
  uint32_t seq = 0;
  bool ok = true;
  auto slot_row = [&](uint32_t n) -> const unsigned char* {
    return prep_smem + (size_t)(n & (NS - 1)) * C::kSlotB + (size_t)r * D * 2;
  };
  // Waits for the group starting at slot n0; false (warp-uniform) on a give-up.
  auto wait_group = [&](uint32_t n0) -> bool {
    if (ok) ok = mbar_wait(&bar_full[n0 & (NS - 1)], (n0 >> LNS) & 1u, STT_DEVERR_BWD_WAIT);
    ok = __all_sync(0xffffffffu, ok) != 0;
    return ok;
  };
  // The warp gives slots [n0, n0 + cnt) back once all its lanes have read them.
  auto release = [&](uint32_t n0, int cnt) {
    __syncwarp();
    if (lane == 0)
      for (int c = 0; c < cnt; ++c) mbar_arrive(&bar_empty[(n0 + c) & (NS - 1)]);
  };
  // Four fp32 pairs (elements e0.. and e1..) of a gradient row.
  auto put8 = [&](void* base, size_t row_off, const uint64_t (&v)[4], bool acc) {
    float f[8];
#pragma unroll
    for (int m = 0; m < 4; ++m) unpack_f32x2(v[m], f[2 * m], f[2 * m + 1]);
    put_grad4<OUT>(base, row_off + e0, f, acc);
    put_grad4<OUT>(base, row_off + e1, f + 4, acc);
  };

  for (long long u = blockIdx.x; u < n_units; u += gridDim.x) {
    const Unit x = unit_at(u);
    const int q = x.q0 + r;
    const bool live = r < x.nrows;  // q < Q_LEN
    const bool valid = r < x.nv;    // q < T: the row has suffix keys
    const size_t hq = ((size_t)x.b * P.H + (size_t)x.hk * G) * P.Q_LEN + q;  // head hk G, row q
    const size_t kvr = (((size_t)x.b * P.H_kv + x.hk) * P.Q_LEN + q) * D;
    // Sums over a lane group are taken by reduce-scatter: the group's GH
    // Delta partials leave lane l with the Delta of head slot i_me, and per
    // suffix block its 2 GH partials (score and dP of each slot) leave it with
    // one half of slot i_me's pair; it forms that head's p and dS, which the
    // group then broadcasts.
    constexpr int NV = 2 * GH;
    constexpr int kPairOff = L >> (NV == 2 ? 1 : NV == 4 ? 2 : 3);  // lane holding the pair's other half
    const int i_me = scatter_index<L, GH>(l);
    const int h_me = hh * GH + i_me;
    const bool my_dp = (scatter_index<L, NV>(l) & 1) != 0;  // this lane's half: score or dP
    // Rows without suffix keys never use the lse (it may be -inf there).
    const float my_lse2 = (h_me < G && valid) ? P.lse[hq + (size_t)h_me * P.Q_LEN] * kLog2e : 0.f;

    // ---- Delta = sum_d dO O for every head; dO stays in registers.
    uint64_t do2[GH][4];
    float dpart[GH];
    if (!wait_group(seq)) break;
#pragma unroll
    for (int i = 0; i < GH; ++i) {
      const int h = hh * GH + i;
      uint64_t o2[4];
      if (h < G && live) {
        lds_row8<D>(slot_row(seq + h), l, o2);
        lds_row8<D>(slot_row(seq + G + h), l, do2[i]);
      } else {
#pragma unroll
        for (int m = 0; m < 4; ++m) o2[m] = do2[i][m] = 0ull;
      }
      dpart[i] = dot_pairs(do2[i], o2);
    }
    release(seq, 2 * G);
    seq += 2 * G;
    const float my_dl = reduce_scatter<L, GH>(dpart, l);
    if (h_me < G && live && l == scatter_lane<L, GH>(i_me)) P.delta[hq + (size_t)h_me * P.Q_LEN] = my_dl;

    // ---- suffix keys: blocks j = 1..k, one key per query row.
    uint64_t dq2[GH][4];
#pragma unroll
    for (int i = 0; i < GH; ++i)
#pragma unroll
      for (int m = 0; m < 4; ++m) dq2[i][m] = 0ull;
    // Rows without suffix keys get no contribution: written as zeros when the
    // gradients are overwritten, left alone when they are accumulated.
    const bool put = live && (valid || !P.accumulate);
    if (x.nv > 0) {
      uint64_t q2[GH][4];
      if (!wait_group(seq)) break;
#pragma unroll
      for (int i = 0; i < GH; ++i) {
        const int h = hh * GH + i;
        if (h < G && valid) {
          lds_row8<D>(slot_row(seq + h), l, q2[i]);
        } else {
#pragma unroll
          for (int m = 0; m < 4; ++m) q2[i][m] = 0ull;
        }
      }
      release(seq, G);
      seq += G;
      for (int j = 1; j <= P.k; ++j) {
        if (!wait_group(seq)) break;
        uint64_t k2[4], v2[4];
        if (valid) {
          lds_row8<D>(slot_row(seq), l, k2);
          lds_row8<D>(slot_row(seq + 1), l, v2);
        } else {
#pragma unroll
          for (int m = 0; m < 4; ++m) k2[m] = v2[m] = 0ull;
        }
        release(seq, 2);
        seq += 2;
        uint64_t dk2[4], dv2[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) dk2[m] = dv2[m] = 0ull;
        // Head slots past G: q = dO = 0 and Delta = 0, so dS = 0 and p dO = 0
        // (the sums still run on every lane).
        float part[NV];
#pragma unroll
        for (int i = 0; i < GH; ++i) {
          part[2 * i] = dot_pairs(q2[i], k2);
          part[2 * i + 1] = dot_pairs(do2[i], v2);
        }
        const float tot = reduce_scatter<L, NV>(part, l);
        const float oth = __shfl_xor_sync(0xffffffffu, tot, kPairOff);
        const float s_me = my_dp ? oth : tot, dp_me = my_dp ? tot : oth;
        const float p_me = valid ? ex2(s_me * P.scale_log2 - my_lse2) : 0.f;
        const float dss_me = p_me * (dp_me - my_dl) * P.scale;
#pragma unroll
        for (int i = 0; i < GH; ++i) {
          const float p = __shfl_sync(0xffffffffu, p_me, scatter_lane<L, NV>(2 * i), L);
          const float dss = __shfl_sync(0xffffffffu, dss_me, scatter_lane<L, NV>(2 * i), L);
          const uint64_t dss2 = f32x2(dss, dss), p2 = f32x2(p, p);
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            dq2[i][m] = fma_f32x2(dss2, k2[m], dq2[i][m]);
            dk2[m] = fma_f32x2(dss2, q2[i][m], dk2[m]);
            dv2[m] = fma_f32x2(p2, do2[i][m], dv2[m]);
          }
        }
        if constexpr (SH == 2) {
          // The other lane group of the row holds the other heads: add, then
          // group 0 writes dK_j and group 1 dV_j.
          uint64_t out[4];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const uint64_t ok2 = __shfl_xor_sync(0xffffffffu, dk2[m], L);
            const uint64_t ov2 = __shfl_xor_sync(0xffffffffu, dv2[m], L);
            out[m] = hh == 0 ? add_f32x2(dk2[m], ok2) : add_f32x2(dv2[m], ov2);
          }
          if (put) put8(hh == 0 ? P.dkb[j] : P.dvb[j], kvr, out, P.accumulate != 0);
        } else if (put) {
          put8(P.dkb[j], kvr, dk2, P.accumulate != 0);
          put8(P.dvb[j], kvr, dv2, P.accumulate != 0);
        }
      }
      if (!ok) break;
    } else if (live && !P.accumulate) {
      const uint64_t z[4] = {0ull, 0ull, 0ull, 0ull};
      for (int j = 1; j <= P.k; ++j) {
        if (SH == 1 || hh == 0) put8(P.dkb[j], kvr, z, false);
        if (SH == 1 || hh == 1) put8(P.dvb[j], kvr, z, false);
      }
    }
    if (live) {
      // dq starts as the suffix part; the causal kernel adds into it next, so
      // these rows take ordinary (L2-allocating) stores.
#pragma unroll
      for (int i = 0; i < GH; ++i) {
        const int h = hh * GH + i;
        if (h < G) {
          float f[8];
#pragma unroll
          for (int m = 0; m < 4; ++m) unpack_f32x2(dq2[i][m], f[2 * m], f[2 * m + 1]);
          float* row = P.dq + (hq + (size_t)h * P.Q_LEN) * D;
          *reinterpret_cast<float4*>(row + e0) = make_float4(f[0], f[1], f[2], f[3]);
          *reinterpret_cast<float4*>(row + e1) = make_float4(f[4], f[5], f[6], f[7]);
        }
      }
      if (P.zero_acc0) {
        const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (SH == 1 || hh == 0) {
          *reinterpret_cast<float4*>(P.dk0 + kvr + e0) = z4;
          *reinterpret_cast<float4*>(P.dk0 + kvr + e1) = z4;
        }
        if (SH == 1 || hh == 1) {
          *reinterpret_cast<float4*>(P.dv0 + kvr + e0) = z4;
          *reinterpret_cast<float4*>(P.dv0 + kvr + e1) = z4;
        }
      }
    }
  }
}

// ---------------------------------------------------------------- causal --
// TMEM columns: S^T (P^T is written back into it), dP^T (reused for the
// tile's dQ), dV, dK.  Column half h of P^T lives in S^T columns
// [64h, 64h + 32), inside the S^T columns its own warps read, so the write-back
// needs no barrier between the two halves.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 384;

// Shared memory: K and V of the key tile, two stages of Q and dO, the dS^T
// tile.  A query tile's dQ leaves through fp32 staging blocks of [128 x 32]
// (16 KB; block h holds 32 columns of compute half h) in the tile's own Q and
// dO buffers, free once dK (Q's last reader) and dV (dO's) are done: part A in
// the Q buffer, and for D = 128 part B in the dO buffer (for D = 64 part A's
// second block).  The next tiles' Q and dO are loaded into them once TMA has
// read the staging.
template <int D>
struct CausalSmem {
  static constexpr int kTileB = kTile * D * 2;  // one 128 x D bf16 tile
  static constexpr int kDsB = kTile * kTile * 2;
  static constexpr int kStages = 2;
  static constexpr int kParts = D / 64;
  static constexpr int kStageBlkB = kTile * 32 * 4;
  static constexpr int k = 0;
  static constexpr int v = kTileB;
  static constexpr int q0 = 2 * kTileB;
  static constexpr int do0 = q0 + kStages * kTileB;
  static constexpr int ds = do0 + kStages * kTileB;
  static constexpr int total = ds + kDsB;
  static constexpr int alloc = total;  // the dynamic array is declared 1024-byte aligned
  static_assert(D == 64 ? kStageBlkB == kTileB : 2 * kStageBlkB == kTileB,
                "a dQ staging part fills one Q or dO buffer");
  // The final dK / dV staging (2 x D/32 blocks) overwrites K, V and the Q
  // stages, once TMA has read every dQ staging.
  static_assert(2 * (D / 32) * kStageBlkB <= do0, "dK/dV staging must stay below the dO stages");
};

// Staging block hh of part p of stage st: dQ columns [hh D/2 + 32 p, +32).
template <int D>
__device__ __forceinline__ unsigned char* dq_staging(unsigned char* smem, int p, int hh, int st) {
  using L = CausalSmem<D>;
  const int q = L::q0 + st * L::kTileB, o = L::do0 + st * L::kTileB;
  if constexpr (D == 64) return smem + (hh == 0 ? q : o);
  return smem + (p == 0 ? q : o) + hh * L::kStageBlkB;
}

// P^T = 2^(S^T sl2 - lse2) for the 64 queries of one compute thread's half
// (fp32 kept in pf for dS), written back as bf16 into the thread's own S^T
// columns at tcol.  kMask: the tile holds masked entries (kv > q, kv >= T or
// q >= Q_LEN), which get P = 0; full tiles take the body without the test.
template <bool kMask>
__device__ __forceinline__ void form_p(uint32_t (&pf)[2][32], const float* nlse_s, float sl2,
                                       int qh, int kv, bool kv_live, int q_len, uint32_t tcol) {
  const uint64_t sl2x2 = f32x2(sl2, sl2);
#pragma unroll
  for (int c2 = 0; c2 < 2; ++c2) {
    uint32_t pp[16];
#pragma unroll
    for (int x4 = 0; x4 < 32; x4 += 4) {
      // 2^(S sl2 - lse2), two queries per packed FMA
      const float4 l4 = *reinterpret_cast<const float4*>(nlse_s + c2 * 32 + x4);
      float xv[4];
      unpack_f32x2(fma_f32x2(f32x2(__uint_as_float(pf[c2][x4]), __uint_as_float(pf[c2][x4 + 1])),
                             sl2x2, f32x2(l4.x, l4.y)),
                   xv[0], xv[1]);
      unpack_f32x2(fma_f32x2(f32x2(__uint_as_float(pf[c2][x4 + 2]), __uint_as_float(pf[c2][x4 + 3])),
                             sl2x2, f32x2(l4.z, l4.w)),
                   xv[2], xv[3]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float pv = ex2(xv[e]);
        if constexpr (kMask) {
          const int qa = qh + c2 * 32 + x4 + e;
          if (!(kv_live && kv <= qa && qa < q_len)) pv = 0.f;
        }
        pf[c2][x4 + e] = __float_as_uint(pv);
      }
      pp[x4 >> 1] = pack_bf16(__uint_as_float(pf[c2][x4]), __uint_as_float(pf[c2][x4 + 1]));
      pp[(x4 >> 1) + 1] =
          pack_bf16(__uint_as_float(pf[c2][x4 + 2]), __uint_as_float(pf[c2][x4 + 3]));
    }
    // P^T of queries [qh + 32 c2, +32) into this half's own S^T columns.
    tmem_st16(tcol + c2 * 16, pp);
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_causal_kernel(const __grid_constant__ BwdParams P,
                           const __grid_constant__ CUtensorMap tmQ,
                           const __grid_constant__ CUtensorMap tmDO,
                           const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV,
                           const __grid_constant__ CUtensorMap tmDQ,
                           const __grid_constant__ CUtensorMap tmDK,
                           const __grid_constant__ CUtensorMap tmDV) {
  using L = CausalSmem<D>;
  constexpr int NS = L::kStages;
  constexpr int NP = L::kParts;
  // The swizzled tiles need 1024-byte alignment, which the declaration asks
  // of the launch; a block that does not get it does no work and reports it.
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw;
  if ((smem_u32(smem_raw) & 1023u) != 0) {
    if (threadIdx.x == 0) record_error(STT_DEVERR_SMEM_ALIGN);
    return;
  }
  // Producer -> MMA: kv, q_full, do_full.  MMA -> compute: s_full, dp_full,
  // dk_done, final.  Compute -> MMA: p_ready, ds_ready.  MMA -> epilogue:
  // dq_full, dk_done.  Epilogue -> MMA: dq_free.  Epilogue -> producer:
  // stg_full.  MMA -> MMA: pt_free.  Issuers: drain.  Compute group: grp.
  __shared__ uint64_t bar_kv, bar_q_full[NS], bar_do_full[NS], bar_s_full,
      bar_dp_full, bar_p_ready, bar_pt_free, bar_ds_ready, bar_dq_full, bar_dk_done, bar_dq_free,
      bar_stg_full[2], bar_stg_done, bar_final, bar_drain, bar_grp;
  __shared__ uint32_t tmem_base;
  // [tile parity][-lse2 | -Delta][query]: tile i's statistics sit in buffer i & 1.
  __shared__ __align__(16) float s_stat[2][2][kTile];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // A CTA takes one key tile for g_sub query heads of one KV group (a head
  // subgroup): the heads' query tiles run through one pipeline, head after
  // head, and dK / dV accumulate over all of them in TMEM, so K and V are
  // loaded once and the key tile's gradients leave once per subgroup.
  // Subgroups are taken in chunks of P.chunk_subs: the CTAs of one chunk run
  // together and re-read only their heads' Q and dO, and add into only their
  // heads' dq, which stay in L2; within a chunk the key tiles go longest first.
  const int gs = P.g_sub;
  const int subs_per_b = P.H / gs;
  const int nsub = subs_per_b * P.B;
  const int ch = nsub < P.chunk_subs ? nsub : P.chunk_subs;
  const int chunk = (int)(blockIdx.x / (unsigned)(P.n_t * ch));
  const int chunk_n = min(ch, nsub - chunk * ch);
  const int rem = (int)blockIdx.x - chunk * P.n_t * ch;
  const int c = rem / chunk_n;  // key tile; low tiles see the most query tiles
  const int sg = chunk * ch + rem % chunk_n;
  const int b = sg / subs_per_b;
  const int bh0 = b * P.H + (sg - b * subs_per_b) * gs;  // first (b, h) of the subgroup
  const int hk = (bh0 - b * P.H) / P.G;
  const int c0 = c * kTile;
  const int T = P.T[b];
  const int t_first = c;                          // query tiles t >= c see this key tile
  const int n_qh = (c0 < T) ? (P.n_t - t_first) : 0;  // query tiles per head
  const int n_q = n_qh * gs;                      // tiles of the CTA, head-major
  // Tile i: head bh0 + i / n_qh, query tile t_first + i % n_qh.
  auto tile_bh = [&](int i) { return bh0 + i / n_qh; };
  auto tile_q0 = [&](int i) { return (t_first + i % n_qh) * kTile; };

  if (tid == 0) {
    mbar_init(&bar_kv, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bar_q_full[s], 1);
      mbar_init(&bar_do_full[s], 1);
    }
    mbar_init(&bar_s_full, 1);
    mbar_init(&bar_dp_full, 1);
    mbar_init(&bar_p_ready, kComputeWarps);
    mbar_init(&bar_pt_free, 1);
    mbar_init(&bar_ds_ready, kComputeWarps);
    mbar_init(&bar_dq_full, 1);
    mbar_init(&bar_dk_done, 1);
    mbar_init(&bar_dq_free, kEpiWarps);
    // stg_full alternates by tile parity: the epilogue warps meet no other
    // barrier between one tile's staging and the next, so one of them could
    // arrive for tile i + 1 before another has arrived for tile i.
    mbar_init(&bar_stg_full[0], kEpiWarps);
    mbar_init(&bar_stg_full[1], kEpiWarps);
    mbar_init(&bar_final, 1);
    mbar_init(&bar_stg_done, 1);  // producer: every dQ staging read by TMA
    mbar_init(&bar_drain, 2);  // one commit from each issuing thread
    mbar_init(&bar_grp, kComputeWarps);
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
    // ------------------------------------------- TMA producer and dQ adds --
    if (lane == 0 && n_q > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmDO);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDQ);
      const int bhk = b * P.H_kv + hk;
      mbar_arrive_expect_tx(&bar_kv, 2 * L::kTileB);
      for (int cb = 0; cb < D / kColBlock; ++cb) {
        tma_load_3d(smem + L::k + cb * kTile * 128, &tmK, &bar_kv, cb * kColBlock, c0, bhk);
        tma_load_3d(smem + L::v + cb * kTile * 128, &tmV, &bar_kv, cb * kColBlock, c0, bhk);
      }
      auto load_q = [&](int i) {
        const int st = i % NS;
        mbar_arrive_expect_tx(&bar_q_full[st], L::kTileB);
        for (int cb = 0; cb < D / kColBlock; ++cb)
          tma_load_3d(smem + L::q0 + st * L::kTileB + cb * kTile * 128, &tmQ, &bar_q_full[st],
                      cb * kColBlock, tile_q0(i), tile_bh(i));
      };
      auto load_do = [&](int i) {
        const int st = i % NS;
        mbar_arrive_expect_tx(&bar_do_full[st], L::kTileB);
        for (int cb = 0; cb < D / kColBlock; ++cb)
          tma_load_3d(smem + L::do0 + st * L::kTileB + cb * kTile * 128, &tmDO, &bar_do_full[st],
                      cb * kColBlock, tile_q0(i), tile_bh(i));
      };
      int issued_q = 0, issued_do = 0;
      for (; issued_q < NS && issued_q < n_q; ++issued_q) {
        load_q(issued_q);
        load_do(issued_q);
        ++issued_do;
      }
      bool ok = true;
      for (int i = 0; ok && i < n_q; ++i) {
        const int st = i % NS;
        const int tq0 = tile_q0(i), tbh = tile_bh(i);
        const bool more = i + NS < n_q;
        // dQ of tile i, staged in its Q and dO buffers (dK(i) and dV(i) done).
        ok = mbar_wait(&bar_stg_full[i & 1], (uint32_t)(i >> 1) & 1u, STT_DEVERR_BWD_WAIT);
        if (!ok) break;
        // Part A first; Q(i + NS) follows as soon as TMA has read it, ahead of
        // part B in TMA's queue, since S^T(i + NS) needs it first.
        for (int hh = 0; hh < 2; ++hh)
          tma_reduce_add_3d(&tmDQ, dq_staging<D>(smem, 0, hh, st), hh * (D / 2), tq0, tbh);
        bulk_commit_group();
        bulk_wait_group_read0();
        if (more) {
          load_q(i + NS);
          ++issued_q;
        }
        if constexpr (NP == 2) {
          for (int hh = 0; hh < 2; ++hh)
            tma_reduce_add_3d(&tmDQ, dq_staging<D>(smem, 1, hh, st), hh * (D / 2) + 32, tq0, tbh);
          bulk_commit_group();
          bulk_wait_group_read0();
        }
        if (more) {
          load_do(i + NS);
          ++issued_do;
        }
      }
      // The compute warps' final dK / dV staging reuses the Q buffers.
      if (ok) mbar_arrive(&bar_stg_done);
      if (!ok) {
        // Gave up: let every copy already issued land before the CTA exits.
        mbar_wait(&bar_kv, 0, STT_DEVERR_BWD_WAIT);
        for (int i = (issued_q > NS ? issued_q - NS : 0); i < issued_q; ++i)
          mbar_wait(&bar_q_full[i % NS], (uint32_t)(i / NS) & 1u, STT_DEVERR_BWD_WAIT);
        for (int i = (issued_do > NS ? issued_do - NS : 0); i < issued_do; ++i)
          mbar_wait(&bar_do_full[i % NS], (uint32_t)(i / NS) & 1u, STT_DEVERR_BWD_WAIT);
      }
      // The reduce-adds complete with the grid; the CTA only has to stay
      // until TMA has read their shared-memory sources.
      bulk_wait_group_read0();
    }
  } else if (warp == kWarpMma || warp == kWarpMma2) {
    // ------------------------------------------------------- MMA issuers --
    // Two issuing threads, because one thread's issue, commit and wait
    // latencies for the five products of a tile exceed the tensor cores' time.
    //   warp 9:  S^T(i) once dV(i-1) has consumed P^T(i-1) from the S^T
    //            columns; dP^T(i) once dQ(i-1) is out of the dP^T columns.
    //   warp 14: dV(i) once P^T(i) is in TMEM; dQ(i) then dK(i) once dS^T(i)
    //            is in shared memory (dQ first: its read-out overlaps dK).
    // Each commit's mbarrier fires when every MMA issued before it by the
    // committing thread is complete.
    if (lane == 0 && n_q > 0) {
      const uint32_t idSS = idesc_bf16(128, kTile, false, false);  // S^T, dP^T
      const uint32_t idKV = idesc_bf16(128, D, false, true);       // dV, dK (B MN-major)
      const uint32_t idQ = idesc_bf16(128, D, true, true);         // dQ (A, B MN-major)
      // Base descriptors; each MMA only advances the start address.
      const uint64_t kK = sdesc_sw128(smem_u32(smem + L::k), 16, 1024);     // K, K-major
      const uint64_t kV = sdesc_sw128(smem_u32(smem + L::v), 16, 1024);     // V, K-major
      const uint64_t mK = sdesc_sw128(smem_u32(smem + L::k), kTile * 128, 1024);  // K, MN-major
      const uint64_t kQ0 = sdesc_sw128(smem_u32(smem + L::q0), 16, 1024);
      const uint64_t mQ0 = sdesc_sw128(smem_u32(smem + L::q0), kTile * 128, 1024);
      const uint64_t kDO0 = sdesc_sw128(smem_u32(smem + L::do0), 16, 1024);
      const uint64_t mDO0 = sdesc_sw128(smem_u32(smem + L::do0), kTile * 128, 1024);
      const uint64_t kDS = sdesc_sw128(smem_u32(smem + L::ds), 16, 1024);
      const uint64_t mDS = sdesc_sw128(smem_u32(smem + L::ds), kTile * 128, 1024);
      bool ok = true;
      if (warp == kWarpMma) {
        ok = mbar_wait(&bar_kv, 0, STT_DEVERR_BWD_WAIT);
        for (int i = 0; ok && i < n_q; ++i) {
          const int st = i % NS;
          const uint32_t ph = (uint32_t)(i / NS) & 1u, prev = (uint32_t)(i - 1) & 1u;
          ok = mbar_wait(&bar_q_full[st], ph, STT_DEVERR_BWD_WAIT);
          if (ok && i > 0) ok = mbar_wait(&bar_pt_free, prev, STT_DEVERR_BWD_WAIT);
          if (!ok) break;
          tc_fence_after();
          const uint64_t kQ = sdesc_add(kQ0, st * L::kTileB);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kTile * 128 + (kk & 3) * 32;
            umma_bf16_ss(tmem + kColS, sdesc_add(kK, off), sdesc_add(kQ, off), idSS, kk > 0 ? 1u : 0u);
          }
          umma_commit(&bar_s_full);
          ok = mbar_wait(&bar_do_full[st], ph, STT_DEVERR_BWD_WAIT);
          if (ok && i > 0) ok = mbar_wait(&bar_dq_free, prev, STT_DEVERR_BWD_WAIT);
          if (!ok) break;
          tc_fence_after();
          const uint64_t kDO = sdesc_add(kDO0, st * L::kTileB);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kTile * 128 + (kk & 3) * 32;
            umma_bf16_ss(tmem + kColDP, sdesc_add(kV, off), sdesc_add(kDO, off), idSS, kk > 0 ? 1u : 0u);
          }
          umma_commit(&bar_dp_full);
        }
      } else {
        for (int i = 0; ok && i < n_q; ++i) {
          const int st = i % NS;
          const uint32_t par = (uint32_t)i & 1u;
          // dV(i) reads dO(i): its load is waited for here too, since P^T(i)
          // can be ready before dP^T(i) (the other thread's wait) is issued.
          ok = mbar_wait(&bar_do_full[st], (uint32_t)(i / NS) & 1u, STT_DEVERR_BWD_WAIT) &&
               mbar_wait(&bar_p_ready, par, STT_DEVERR_BWD_WAIT);
          if (!ok) break;
          tc_fence_after();
          const uint64_t mQ = sdesc_add(mQ0, st * L::kTileB), mDO = sdesc_add(mDO0, st * L::kTileB);
          // dV += P^T dO: A = P^T in TMEM (8 columns per 16 queries; queries
          // 64h.. live at column 64h), B = dO MN-major.
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            umma_bf16_ts(tmem + kColDV, tmem + kColS + (kk >> 2) * 64 + (kk & 3) * 8,
                         sdesc_add(mDO, kk * 2048), idKV, (i > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&bar_pt_free);
          ok = mbar_wait(&bar_ds_ready, par, STT_DEVERR_BWD_WAIT);
          if (!ok) break;
          tc_fence_after();
          // dQ = dS K: A = the dS^T tile read MN-major (rows = keys = K dim),
          // B = K MN-major; into the dP^T columns.
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            umma_bf16_ss(tmem + kColDP, sdesc_add(mDS, kk * 2048), sdesc_add(mK, kk * 2048), idQ,
                         kk > 0 ? 1u : 0u);
          umma_commit(&bar_dq_full);
          // dK += dS^T Q: A = dS^T in smem (K-major over queries), B = Q MN-major.
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            umma_bf16_ss(tmem + kColDK, sdesc_add(kDS, (kk >> 2) * kTile * 128 + (kk & 3) * 32),
                         sdesc_add(mQ, kk * 2048), idKV, (i > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&bar_dk_done);
        }
        // The last dK also follows every S^T / dP^T product of the tile loop
        // (the compute warps consumed them before dS^T was ready).
        if (ok) umma_commit(&bar_final);
      }
      // Every MMA issued by either thread is complete before TMEM is released.
      umma_commit(&bar_drain);
      mbar_wait(&bar_drain, 0, STT_DEVERR_BWD_WAIT);
    }
  } else if (warp >= kWarpEpi) {
    // ------------------------------------------------------- dQ epilogue --
    // Thread = query row r of TMEM lane quarter warp % 4.  Per tile: the
    // columns of staging part B (the dO buffer, free since dV) go first, then
    // the part A columns are read into registers, TMEM is released to dP^T of
    // the next tile, and part A (the Q buffer) is written once dK, its last
    // reader, is done.  Staging part p, block hh holds dQ columns
    // [hh D/2 + 32 p, +32) of all 128 rows.
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    // dQ comes out of TMEM already scaled (dS carries the scale).
    auto stage = [&](unsigned char* blk, const uint32_t (&u)[32]) {
#pragma unroll
      for (int w = 0; w < 8; ++w)
        *reinterpret_cast<float4*>(blk + swz128(r, w)) =
            make_float4(__uint_as_float(u[4 * w]), __uint_as_float(u[4 * w + 1]),
                        __uint_as_float(u[4 * w + 2]), __uint_as_float(u[4 * w + 3]));
    };
    bool ok = true;
    for (int i = 0; ok && i < n_q; ++i) {
      const int st = i % NS;
      const uint32_t par = (uint32_t)i & 1u;
      ok = warp_wait(&bar_dq_full, par, STT_DEVERR_BWD_WAIT);
      if (!ok) break;
      tc_fence_after();
      if constexpr (NP == 2) {
        // Part B into the dO buffer (dV, its last reader, is done).
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t u[32];
          tmem_ld32(tmem + lane_off + kColDP + hh * (D / 2) + 32, u);
          stage(dq_staging<D>(smem, 1, hh, st), u);
        }
      }
      uint32_t a0[32], a1[32];
      tmem_ld32x2(tmem + lane_off + kColDP, tmem + lane_off + kColDP + D / 2, a0, a1);
      // dQ is out of TMEM: the MMA warp may overwrite the dP^T columns.
      tc_fence_before();
      warp_arrive(&bar_dq_free);
      ok = warp_wait(&bar_dk_done, par, STT_DEVERR_BWD_WAIT);
      if (!ok) break;
      stage(dq_staging<D>(smem, 0, 0, st), a0);
      stage(dq_staging<D>(smem, 0, 1, st), a1);
      fence_proxy_async_smem();
      warp_arrive(&bar_stg_full[i & 1]);
    }
  } else {
    // ------------------------------------------------------ compute warps --
    // Row r of the TMEM lane quarter is key row c0 + r for S^T / dP^T / dV /
    // dK; `half` selects the 64-query half of the tile.
    const int quarter = warp & 3, half = warp >> 2;
    const int r = quarter * 32 + lane;
    const int kv = c0 + r;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const float sl2 = P.scale_log2;
    const bool kv_live = kv < T;  // T <= Q_LEN, so also kv < Q_LEN
    unsigned char* sDS = smem + L::ds;
    // Thread tid stages one statistic of one query of a tile: -lse2 (tid < 128)
    // or -Delta (tid >= 128) of query tq0 + (tid & 127), negated for the
    // packed FMA / add below.  The raw value is fetched a tile ahead and
    // scaled only when it is stored.
    const int st_which = tid >> 7, st_idx = tid & 127;
    auto fetch_stat = [&](int i) -> float {
      const int qq = tile_q0(i) + st_idx;
      if (qq >= P.Q_LEN) return 0.f;
      const size_t rq = (size_t)tile_bh(i) * P.Q_LEN + qq;
      return st_which == 0 ? P.lse[rq] : P.delta[rq];
    };
    auto put_stat = [&](int buf, float raw) {
      // P is formed as scale * 2^(S sl2 - lse2) = 2^(S sl2 - lse2 + log2 scale):
      // dS, dQ and dK then carry the attention scale with no multiply of their
      // own, and dV (P^T dO) comes out scaled once, undone at the end.
      s_stat[buf][st_which][st_idx] = st_which == 0 ? -raw * kLog2e + P.log2_scale : -raw;
    };
    uint32_t grp_uses = 0;
    bool ok = true;
    float stat_next = 0.f;
    if (n_q > 0) {
      put_stat(0, fetch_stat(0));
      if (n_q > 1) put_stat(1, fetch_stat(1));
      if (n_q > 2) stat_next = fetch_stat(2);
      ok = group_sync(&bar_grp, grp_uses, STT_DEVERR_BWD_WAIT);
    }
    for (int i = 0; ok && i < n_q; ++i) {
      const uint32_t par = (uint32_t)i & 1u;
      const int tq0 = tile_q0(i);
      const int qh = tq0 + half * 64;  // first query of this thread's half
      // entry (kv, q) is visible iff kv < T, kv <= q and q < Q_LEN
      const bool full = kv_live && kv <= qh && qh + 64 <= P.Q_LEN;
      const float* nlse_s = s_stat[par][0] + half * 64;
      const float* ndl_s = s_stat[par][1] + half * 64;

      // ---- P^T = exp(S^T - lse): queries [qh, qh + 64) of key row kv.  The
      // fp32 P overwrites the loaded S^T values (it is needed again for dS).
      ok = warp_wait(&bar_s_full, par, STT_DEVERR_BWD_WAIT);
      if (!ok) break;
      tc_fence_after();
      uint32_t pf[2][32];
      tmem_ld32x2(tmem + lane_off + kColS + half * 64, tmem + lane_off + kColS + half * 64 + 32,
                  pf[0], pf[1]);
      // The choice of body must be warp-uniform: form_p ends in a warp-wide
      // TMEM store (tcgen05.st .sync.aligned), which every lane of the warp
      // has to reach through the same instruction.
      const uint32_t tcol = tmem + lane_off + kColS + half * 64;
      if (__all_sync(0xffffffffu, full))
        form_p<false>(pf, nlse_s, sl2, qh, kv, kv_live, P.Q_LEN, tcol);
      else
        form_p<true>(pf, nlse_s, sl2, qh, kv, kv_live, P.Q_LEN, tcol);
      tmem_st_wait();
      tc_fence_before();
      warp_arrive(&bar_p_ready);

      // ---- dS^T = P^T (dP^T - Delta) -> swizzled [key][query] tile in smem,
      // once dQ(i-1) and dK(i-1), the previous tile's readers, are done (the
      // other issuing thread commits dk_done after both).
      ok = warp_wait(&bar_dp_full, par, STT_DEVERR_BWD_WAIT);
      if (ok && i > 0) ok = warp_wait(&bar_dk_done, (uint32_t)(i - 1) & 1u, STT_DEVERR_BWD_WAIT);
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        uint32_t dp[32], dd[16];
        tmem_ld32(tmem + lane_off + kColDP + half * 64 + c2 * 32, dp);
#pragma unroll
        for (int x4 = 0; x4 < 32; x4 += 4) {
          // P (dP - Delta), two queries per packed add and multiply
          const float4 d4 = *reinterpret_cast<const float4*>(ndl_s + c2 * 32 + x4);
          float sv[4];
          unpack_f32x2(mul_f32x2(f32x2(__uint_as_float(pf[c2][x4]), __uint_as_float(pf[c2][x4 + 1])),
                                 add_f32x2(f32x2(__uint_as_float(dp[x4]), __uint_as_float(dp[x4 + 1])),
                                           f32x2(d4.x, d4.y))),
                       sv[0], sv[1]);
          unpack_f32x2(mul_f32x2(f32x2(__uint_as_float(pf[c2][x4 + 2]), __uint_as_float(pf[c2][x4 + 3])),
                                 add_f32x2(f32x2(__uint_as_float(dp[x4 + 2]), __uint_as_float(dp[x4 + 3])),
                                           f32x2(d4.z, d4.w))),
                       sv[2], sv[3]);
          dd[x4 >> 1] = pack_bf16(sv[0], sv[1]);
          dd[(x4 >> 1) + 1] = pack_bf16(sv[2], sv[3]);
        }
#pragma unroll
        for (int w = 0; w < 4; ++w)
          *reinterpret_cast<uint4*>(sDS + swz_chunk_offset(r, half * 8 + c2 * 4 + w, kTile)) =
              make_uint4(dd[4 * w], dd[4 * w + 1], dd[4 * w + 2], dd[4 * w + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      warp_arrive(&bar_ds_ready);

      // Every warp is done with this tile's statistics: its buffer takes
      // those of tile i + 2, which the next tile's ds_ready barrier publishes.
      ok = warp_wait(&bar_ds_ready, par, STT_DEVERR_BWD_WAIT);
      if (!ok) break;
      if (i + 2 < n_q) {
        put_stat(par, stat_next);
        if (i + 3 < n_q) stat_next = fetch_stat(i + 3);
      }
    }
    if (ok && n_q > 0) {
      // dV and dK of this key tile into the block-0 gradients, summed over the
      // group's query heads: once every MMA is done and TMA has read every dQ
      // staging, K, V and the Q stages are free and all D/32 chunks of both
      // are staged at once and reduce-added by TMA (rows kv >= T hold zeros;
      // rows past Q_LEN are clipped).
      ok = warp_wait(&bar_final, 0, STT_DEVERR_BWD_WAIT) &&
           warp_wait(&bar_stg_done, 0, STT_DEVERR_BWD_WAIT);
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int c2 = 0; c2 < D / 64; ++c2) {
          const int cc = half * (D / 64) + c2;
          uint32_t uv[32], uk[32];
          tmem_ld32x2(tmem + lane_off + kColDV + cc * 32, tmem + lane_off + kColDK + cc * 32, uv, uk);
          unsigned char* bv = smem + cc * L::kStageBlkB;
          unsigned char* bk = smem + (D / 32 + cc) * L::kStageBlkB;
#pragma unroll
          for (int w = 0; w < 8; ++w) {
            const uint32_t o = swz128(r, w);
            *reinterpret_cast<float4*>(bv + o) = make_float4(
                P.inv_scale * __uint_as_float(uv[4 * w]), P.inv_scale * __uint_as_float(uv[4 * w + 1]),
                P.inv_scale * __uint_as_float(uv[4 * w + 2]),
                P.inv_scale * __uint_as_float(uv[4 * w + 3]));
            *reinterpret_cast<float4*>(bk + o) =
                make_float4(__uint_as_float(uk[4 * w]), __uint_as_float(uk[4 * w + 1]),
                            __uint_as_float(uk[4 * w + 2]), __uint_as_float(uk[4 * w + 3]));
          }
        }
        fence_proxy_async_smem();
        ok = group_sync(&bar_grp, grp_uses, STT_DEVERR_BWD_WAIT);
      }
      if (ok && tid == 0) {
        const int bhk = b * P.H_kv + hk;
        for (int cc = 0; cc < D / 32; ++cc) {
          tma_reduce_add_3d(&tmDV, smem + cc * L::kStageBlkB, cc * 32, c0, bhk);
          tma_reduce_add_3d(&tmDK, smem + (D / 32 + cc) * L::kStageBlkB, cc * 32, c0, bhk);
        }
        bulk_commit_group();
        // The issuing thread waits until TMA has read the staging before the
        // CTA's shared memory goes away; the reductions complete with the grid.
        bulk_wait_group_read0();
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

// ------------------------------------------------------------------ cast --
// bf16 gradients: dq, dK_0 and dV_0 were accumulated in fp32 in the workspace;
// round them to the caller's bf16 buffers (dK_0 / dV_0 added to the values
// already there when accumulating).  n4 groups of four elements per tensor.
struct CastParams {
  const float* src[3];
  __nv_bfloat16* dst[3];
  long long n4[3];
  int accumulate_kv;  // tensors 1 and 2 (dK_0, dV_0) add to dst
};

__global__ void __launch_bounds__(256) attn_bwd_cast_kernel(const __grid_constant__ CastParams C) {
  const long long stride = (long long)gridDim.x * blockDim.x;
#pragma unroll 1
  for (int t = 0; t < 3; ++t) {
    const float4* src = reinterpret_cast<const float4*>(C.src[t]);
    uint2* dst = reinterpret_cast<uint2*>(C.dst[t]);
    const bool acc = t > 0 && C.accumulate_kv;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < C.n4[t]; i += stride) {
      float4 v = __ldcs(src + i);
      if (acc) {
        const uint2 o = dst[i];
        v.x += bf16lo(o.x);
        v.y += bf16hi(o.x);
        v.z += bf16lo(o.y);
        v.w += bf16hi(o.y);
      }
      const uint2 y = make_uint2(pack_bf16(v.x, v.y), pack_bf16(v.z, v.w));
      __stcs(dst + i, y);
    }
  }
}

template <int D, int GM>
cudaError_t launch_prep(const BwdParams& P, bool bf16, cudaStream_t s) {
  using C = PrepCfg<D, GM>;
  const long long units = (long long)P.B * P.H_kv * ((P.Q_LEN + C::R - 1) / C::R);
  const long long sms = sm_count();
  const long long grid = units < sms ? units : sms;
  if (grid <= 0) return cudaSuccess;
  auto kern = bf16 ? attn_bwd_prep_kernel<D, GM, __nv_bfloat16> : attn_bwd_prep_kernel<D, GM, float>;
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)grid, C::kThreads, C::kSmem, s>>>(P);
  return cudaSuccess;
}

template <int D>
cudaError_t launch(const AttnArgs& a, const AttnBwdArgs& g, cudaStream_t s) {
  static thread_local BwdParams P;
  const bool bf16 = (g.flags & kBwdBf16) != 0;
  const bool acc = (g.flags & kBwdAccumulate) != 0;
  const WorkspaceLayout W = workspace_layout(a.B, a.H, a.H_kv, D, a.Q_LEN, g.flags);
  unsigned char* ws = static_cast<unsigned char*>(g.workspace);
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
  P.delta = reinterpret_cast<float*>(ws + W.delta);
  if (bf16) {
    P.dq = reinterpret_cast<float*>(ws + W.dq);
    P.dk0 = reinterpret_cast<float*>(ws + W.dk0);
    P.dv0 = reinterpret_cast<float*>(ws + W.dv0);
  } else {
    P.dq = static_cast<float*>(g.dq);
    P.dk0 = static_cast<float*>(g.dk_blocks[0]);
    P.dv0 = static_cast<float*>(g.dv_blocks[0]);
  }
  P.accumulate = acc ? 1 : 0;
  // fp32 accumulation adds straight into the caller's dK_0 / dV_0; otherwise
  // the accumulators start at zero.
  P.zero_acc0 = (acc && !bf16) ? 0 : 1;
  P.B = a.B;
  P.H = a.H;
  P.H_kv = a.H_kv;
  P.Q_LEN = a.Q_LEN;
  P.k = a.k;
  P.n_t = (a.Q_LEN + kTile - 1) / kTile;
  P.G = a.H / a.H_kv;
  {
    // Heads per CTA: the divisor g of G that minimises an estimate of the
    // busiest SM's work, in units of one (key tile, query tile) pair: the
    // mean load (every pair, plus kCtaFixedPairs per CTA that has work) plus
    // kTailShare of the heaviest CTA (g n_t pairs and its fixed cost), which
    // the longest-first order leaves partly unbalanced at the end.  More
    // heads per CTA pay the fixed cost (K/V load, first tile, final dK / dV)
    // less often but make the heaviest CTAs longer.
    constexpr double kCtaFixedPairs = 3.7;  // ~9.2 us of set-up and tail against ~2.5 us per pair
    constexpr double kTailShare = 0.2;      // from a simulation of the longest-first dispatch
    const int sms = sm_count();
    long long pairs = 0, live_tiles = 0;
    for (int b = 0; b < a.B; ++b) {
      const long long live = ((long long)a.T[b] + kTile - 1) / kTile;  // key tiles with c0 < T
      pairs += live * P.n_t - live * (live - 1) / 2;
      live_tiles += live;
    }
    pairs *= a.H;
    P.g_sub = 1;
    double best = 0.0;
    for (int gsub = 1; gsub <= P.G; ++gsub) {
      if (P.G % gsub != 0) continue;
      const double ctas = (double)live_tiles * (a.H / gsub);
      const double est = ((double)pairs + ctas * kCtaFixedPairs) / sms +
                         kTailShare * ((double)gsub * P.n_t + kCtaFixedPairs);
      if (gsub == 1 || est < best) {
        best = est;
        P.g_sub = gsub;
      }
    }
    // Subgroups per chunk: as many as keep their Q, dO (bf16) and dq (fp32) --
    // 8 bytes per element -- within kChunkBytes of L2.  Even when a chunk is
    // smaller than a wave of CTAs this order pays: a head's dq tiles take the
    // reduce-adds of every key tile while they are still in L2 (one chunk
    // spanning all heads made the varlen backward 18 % slower).
    const long long per_head = (long long)a.Q_LEN * D * 8;
    long long heads = kChunkBytes / (per_head > 0 ? per_head : 1);
    heads = heads < 1 ? 1 : (heads > kHeadChunkMax ? kHeadChunkMax : heads);
    const long long nsub = (long long)a.B * a.H / P.g_sub;
    long long cs = heads / P.g_sub;
    if (cs < 1) cs = 1;
    P.chunk_subs = (int)(cs > nsub ? nsub : cs);
  }
  P.scale = a.scale;
  P.scale_log2 = a.scale * kLog2e;
  P.log2_scale = log2f(a.scale);
  P.inv_scale = 1.0f / a.scale;
  for (int b = 0; b < a.B; ++b) P.T[b] = a.T[b];

  CUtensorMap tmQ, tmDO, tmK, tmV;
  cudaError_t e;
  if ((e = bind_device_context()) != cudaSuccess) return e;
  if ((e = encode_tile_map(&tmQ, a.q, D, a.Q_LEN, a.B * a.H, kTile)) != cudaSuccess) return e;
  if ((e = encode_tile_map(&tmDO, g.dout, D, a.Q_LEN, a.B * a.H, kTile)) != cudaSuccess) return e;
  if ((e = encode_tile_map(&tmK, a.k_blocks[0], D, a.Q_LEN, a.B * a.H_kv, kTile)) != cudaSuccess)
    return e;
  if ((e = encode_tile_map(&tmV, a.v_blocks[0], D, a.Q_LEN, a.B * a.H_kv, kTile)) != cudaSuccess)
    return e;
  CUtensorMap tmDQ, tmDK, tmDV;
  if ((e = encode_f32_map(&tmDQ, P.dq, D, a.Q_LEN, a.B * a.H, kTile)) != cudaSuccess) return e;
  if ((e = encode_f32_map(&tmDK, P.dk0, D, a.Q_LEN, a.B * a.H_kv, kTile)) != cudaSuccess) return e;
  if ((e = encode_f32_map(&tmDV, P.dv0, D, a.Q_LEN, a.B * a.H_kv, kTile)) != cudaSuccess) return e;

  prof_before(s, STT_KERNEL_ATTN_BWD_PREP);
  if (P.G == 1)
    e = launch_prep<D, 1>(P, bf16, s);
  else if (P.G == 2)
    e = launch_prep<D, 2>(P, bf16, s);
  else if (P.G <= 4)
    e = launch_prep<D, 4>(P, bf16, s);
  else
    e = launch_prep<D, 8>(P, bf16, s);
  prof_after(s);
  if (e != cudaSuccess) return e;
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  const unsigned grid = (unsigned)(P.n_t * (a.H / P.g_sub) * a.B);
  e = cudaFuncSetAttribute(attn_bwd_causal_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           CausalSmem<D>::alloc);
  if (e != cudaSuccess) return e;
  prof_before(s, STT_KERNEL_ATTN_BWD_CAUSAL);
  attn_bwd_causal_kernel<D><<<grid, kThreads, CausalSmem<D>::alloc, s>>>(P, tmQ, tmDO, tmK, tmV,
                                                                        tmDQ, tmDK, tmDV);
  prof_after(s);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (!bf16) return cudaSuccess;

  CastParams C;
  C.src[0] = P.dq;
  C.src[1] = P.dk0;
  C.src[2] = P.dv0;
  C.dst[0] = static_cast<__nv_bfloat16*>(g.dq);
  C.dst[1] = static_cast<__nv_bfloat16*>(g.dk_blocks[0]);
  C.dst[2] = static_cast<__nv_bfloat16*>(g.dv_blocks[0]);
  C.n4[0] = (long long)a.B * a.H * a.Q_LEN * D / 4;
  C.n4[1] = C.n4[2] = (long long)a.B * a.H_kv * a.Q_LEN * D / 4;
  C.accumulate_kv = acc ? 1 : 0;
  long long blocks = (C.n4[0] + 255) / 256;
  if (blocks > 152 * 8) blocks = 152 * 8;
  prof_before(s, STT_KERNEL_ATTN_BWD_CAST);
  attn_bwd_cast_kernel<<<(unsigned)blocks, 256, 0, s>>>(C);
  prof_after(s);
  return cudaGetLastError();
}

}  // namespace

size_t attn_bwd_workspace(int B, int H, int H_kv, int D, int Q_LEN, uint32_t flags) {
  return workspace_layout(B, H, H_kv, D, Q_LEN, flags).total;
}

cudaError_t attn_bwd_launch(const AttnArgs& a, const AttnBwdArgs& g, cudaStream_t s) {
  if (a.D == 128) return launch<128>(a, g, s);
  if (a.D == 64) return launch<64>(a, g, s);
  return cudaErrorNotSupported;
}

STT_DEFINE_ERROR_ACCESSOR(attn_bwd_error_word)
STT_DEFINE_BUDGET_SETTER(attn_bwd_set_wait_budget)

}  // namespace stt
