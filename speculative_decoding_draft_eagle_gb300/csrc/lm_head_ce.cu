// lm_head_ce.cu -- the draft's LM head z = h W^T fused with the masked
// soft-target cross-entropy and its gradient, chunked over the vocabulary so
// that z is never materialised (SpecForge review, §三 "内存高效梯度计算": the
// logits are the activation the in-place gradient saves; §四 "原地反向传播").
//
//   z = h W^T,  lse_r = log sum_v exp z_rv,  l_r = lse_r Sp_r - sum_v p z,
//   dz = pi s - p g  (s_r = g_r Sp_r),  dh = dz W,  dW = dz^T h.
//
// All four contractions run on one persistent tcgen05 GEMM kernel (bf16
// operands staged by TMA in 128-byte-swizzled shared memory, fp32 accumulators
// in TMEM), C[M, N] = A[M, K] B[N, K]^T with each operand K-major or MN-major,
// tiles of 128 x 256, four pipeline stages, and two accumulators in TMEM so
// that the epilogue of one tile overlaps the products of the next.  Warp 0
// issues the TMA loads, warp 1 the MMAs, warps 2-5 run the epilogue (one TMEM
// lane quarter each; thread = row of C).  The epilogue decides what the GEMM
// is:
//   STATS  z tile -> per-row (max, sum exp, sum p, sum p z) over its columns,
//          written as partial statistics (p read once, here);
//   DZ     z tile recomputed -> dz = exp(z - lse) s - p g, stored in bf16 to
//          a chunk buffer (p read a second time);
//   STORE  fp32 C (dW of a chunk);  ACCUM  fp32 C added to (dh over chunks).
// The host runs STATS over the whole vocabulary, combines the partials per row
// (lse, loss), then for each vocabulary chunk of Vc columns: DZ, dh += dz W_c
// (ACCUM), dW_c = dz^T h (STORE).  Only a [N, Vc] bf16 chunk of dz ever exists.
#include <cudaTypedefs.h>

#include "../../include/stt.h"
#include "internal.h"
#include "ptx.cuh"

namespace stt {
namespace {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int kStages = 4;
constexpr int kGThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kEpiWarps = 4;
constexpr uint32_t kAccCols = BN;
constexpr uint32_t kTmemCols = 2 * kAccCols;
constexpr int kABytes = BM * BK * 2;
constexpr int kBBytes = BN * BK * 2;
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kSmem = kStages * kStageBytes + 1024;  // + slack for 1024-byte alignment
constexpr float kLog2eG = 1.4426950408889634f;
constexpr float kLn2G = 0.6931471805599453f;
constexpr int kChunkV = 8192;  // vocabulary columns per gradient chunk
constexpr uint32_t kSiteG = STT_DEVERR_LM_WAIT;

enum : int { kEpiStats = 0, kEpiDz = 1, kEpiStore = 2, kEpiAccum = 3 };

struct GemmP {
  int M, N, K;
  int tiles_m, tiles_n, k_steps;
  float* out;            // STORE / ACCUM: fp32 C with row pitch ldo
  long long ldo;
  const float* p;        // STATS / DZ: targets, column n of C is p[row * ldp + n]
  long long ldp;
  const float* g;        // [M] per-row upstream gradient
  const float* lse2;     // DZ: [M] lse * log2(e)
  const float* srow;     // DZ: [M] g * sum p
  float4* part;          // STATS: part[row * n_part + part0 + tile_n]
  int n_part, part0;
  __nv_bfloat16* dz;     // DZ: output with row pitch lddz
  long long lddz;
};

// 3-D bf16 tensor map over [1][rows][inner] with the given row pitch, a
// 64 x box_rows box and 128-byte swizzle; rows and columns past the extents
// read as zeros.
cudaError_t encode_bf16_2d(CUtensorMap* map, const void* base, long long inner, long long rows,
                           long long pitch_bytes, int box_rows) {
  auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encoder());
  if (!enc) return cudaErrorNotSupported;
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, 1};
  cuuint64_t strides[2] = {(cuuint64_t)pitch_bytes, (cuuint64_t)pitch_bytes * (cuuint64_t)rows};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// A: K-major = [M rows][K] (box 64 x 128), MN-major = [K rows][M] (boxes 64 x 64).
// B: K-major = [N rows][K] (box 64 x 256), MN-major = [K rows][N] (boxes 64 x 64).
template <bool A_MN, bool B_MN, int EPI>
__global__ void __launch_bounds__(kGThreads, 1)
    lm_gemm_kernel(const __grid_constant__ GemmP P, const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_full[kStages], bar_empty[kStages], bar_acc_full[2], bar_acc_empty[2],
      bar_drain;
  __shared__ uint32_t tmem_base;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles = P.tiles_m * P.tiles_n;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar_acc_full[b], 1);
      mbar_init(&bar_acc_empty[b], kEpiWarps);
    }
    mbar_init(&bar_drain, 1);
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

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      long long it = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x) {
        const int m0 = (t % P.tiles_m) * BM, n0 = (t / P.tiles_m) * BN;
        for (int ks = 0; ks < P.k_steps; ++ks, ++it) {
          const int st = (int)(it % kStages);
          const long long use = it / kStages;
          if (use > 0 && !mbar_wait(&bar_empty[st], (uint32_t)((use - 1) & 1), kSiteG)) {
            ok = false;
            break;
          }
          unsigned char* sA = smem + st * kStageBytes;
          unsigned char* sB = sA + kABytes;
          const int k0 = ks * BK;
          mbar_arrive_expect_tx(&bar_full[st], kStageBytes);
          if (A_MN) {
            for (int cb = 0; cb < BM / 64; ++cb)
              tma_load_3d(sA + cb * 8192, &tmA, &bar_full[st], m0 + cb * 64, k0, 0);
          } else {
            tma_load_3d(sA, &tmA, &bar_full[st], k0, m0, 0);
          }
          if (B_MN) {
            for (int cb = 0; cb < BN / 64; ++cb)
              tma_load_3d(sB + cb * 8192, &tmB, &bar_full[st], n0 + cb * 64, k0, 0);
          } else {
            tma_load_3d(sB, &tmB, &bar_full[st], k0, n0, 0);
          }
        }
      }
      if (!ok) {
        // Gave up: let the copies of the last stages land before the CTA exits.
        for (long long j = (it > kStages ? it - kStages : 0); j < it; ++j)
          mbar_wait(&bar_full[j % kStages], (uint32_t)((j / kStages) & 1), kSiteG);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(BM, BN, A_MN, B_MN);
      const uint64_t dA0 = sdesc_sw128(smem_u32(smem), A_MN ? 8192 : 16, 1024);
      const uint64_t dB0 = sdesc_sw128(smem_u32(smem + kABytes), B_MN ? 8192 : 16, 1024);
      long long it = 0;
      int lt = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < n_tiles; t += gridDim.x, ++lt) {
        const int buf = lt & 1, use_b = lt >> 1;
        if (use_b > 0 && !mbar_wait(&bar_acc_empty[buf], (uint32_t)((use_b - 1) & 1), kSiteG)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t acc = tmem + buf * kAccCols;
        for (int ks = 0; ks < P.k_steps; ++ks, ++it) {
          const int st = (int)(it % kStages);
          if (!mbar_wait(&bar_full[st], (uint32_t)((it / kStages) & 1), kSiteG)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t dA = sdesc_add(dA0, st * kStageBytes);
          const uint64_t dB = sdesc_add(dB0, st * kStageBytes);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint32_t oa = A_MN ? kk * 2048 : kk * 32;
            const uint32_t ob = B_MN ? kk * 2048 : kk * 32;
            umma_bf16_ss(acc, sdesc_add(dA, oa), sdesc_add(dB, ob), idesc,
                         (ks > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&bar_empty[st]);
        }
        if (ok) umma_commit(&bar_acc_full[buf]);
      }
      // Every product is complete before TMEM is released.
      umma_commit(&bar_drain);
      mbar_wait(&bar_drain, 0, kSiteG);
    }
  } else {
    // --------------------------------------------------------- epilogue --
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    int lt = 0;
    for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++lt) {
      const int tm = t % P.tiles_m, tn = t / P.tiles_m;
      const int m0 = tm * BM, n0 = tn * BN;
      const int buf = lt & 1;
      if (!warp_wait(&bar_acc_full[buf], (uint32_t)((lt >> 1) & 1), kSiteG)) break;
      tc_fence_after();
      const int row = m0 + r;
      const bool vrow = row < P.M;
      const uint32_t acc = tmem + buf * kAccCols + lane_off;
      if constexpr (EPI == kEpiStats || EPI == kEpiDz) {
        const float gr = vrow ? __ldg(P.g + row) : 0.f;
        const bool live = vrow && gr != 0.f;
        const float* prow = P.p + (long long)(vrow ? row : 0) * P.ldp;
        float m = -INFINITY, l = 0.f, sp = 0.f, spz = 0.f;
        float lse2 = 0.f, s = 0.f;
        if (EPI == kEpiDz && live) {
          lse2 = __ldg(P.lse2 + row);
          s = __ldg(P.srow + row);
        }
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          const int col0 = n0 + c * 32;
          float4 pv[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            pv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (live && col0 + 4 * i < P.N)
              pv[i] = __ldg(reinterpret_cast<const float4*>(prow + col0 + 4 * i));
          }
          uint32_t v[32];
          tmem_ld32(acc + c * 32, v);
          if constexpr (EPI == kEpiStats) {
            float mc = -INFINITY;
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (col0 + i < P.N) mc = fmaxf(mc, __uint_as_float(v[i]));
            if (mc > m) {
              l *= ex2((m - mc) * kLog2eG);
              m = mc;
            }
            const float mb = m * kLog2eG;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float z = __uint_as_float(v[i]);
              const float pz = (i & 3) == 0 ? pv[i >> 2].x : (i & 3) == 1 ? pv[i >> 2].y
                                : (i & 3) == 2 ? pv[i >> 2].z : pv[i >> 2].w;
              if (col0 + i < P.N) {
                l += ex2(fmaf(z, kLog2eG, -mb));
                sp += pz;
                spz = fmaf(pz, z, spz);
              }
            }
          } else {
            uint32_t o[16];
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              float d0 = 0.f, d1 = 0.f;
              if (live) {
                const float4 q4 = pv[i >> 2];
                const float pa = (i & 3) == 0 ? q4.x : q4.z, pb = (i & 3) == 0 ? q4.y : q4.w;
                d0 = fmaf(ex2(fmaf(__uint_as_float(v[i]), kLog2eG, -lse2)), s, -pa * gr);
                d1 = fmaf(ex2(fmaf(__uint_as_float(v[i + 1]), kLog2eG, -lse2)), s, -pb * gr);
              }
              o[i >> 1] = pack_bf16(d0, d1);
            }
            if (vrow) {
              __nv_bfloat16* drow = P.dz + (long long)row * P.lddz + col0;
#pragma unroll
              for (int w = 0; w < 4; ++w)
                if (col0 + 8 * w < P.N)
                  *reinterpret_cast<uint4*>(drow + 8 * w) =
                      make_uint4(o[4 * w], o[4 * w + 1], o[4 * w + 2], o[4 * w + 3]);
            }
          }
        }
        if constexpr (EPI == kEpiStats) {
          if (live) P.part[(long long)row * P.n_part + P.part0 + tn] = make_float4(m, l, sp, spz);
        }
      } else {
        float* orow = P.out + (long long)(vrow ? row : 0) * P.ldo;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          const int col0 = n0 + c * 32;
          uint32_t v[32];
          tmem_ld32(acc + c * 32, v);
          if (vrow) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              if (col0 + 4 * i >= P.N) break;
              float4 x = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                     __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
              float4* dst = reinterpret_cast<float4*>(orow + col0 + 4 * i);
              if constexpr (EPI == kEpiAccum) {
                const float4 y = *dst;
                x.x += y.x;
                x.y += y.y;
                x.z += y.z;
                x.w += y.w;
              }
              *dst = x;
            }
          }
        }
      }
      // The accumulator is read: the MMA warp may reuse it.
      tc_fence_before();
      warp_arrive(&bar_acc_empty[buf]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Per-row combination of the STATS partials: lse, the loss and the values the
// DZ epilogue needs.  One warp per row.
__global__ void __launch_bounds__(256) lm_combine_kernel(const float4* part, int n_part,
                                                         const float* g, long long N,
                                                         float* row_loss, float* wl, float* lse2,
                                                         float* srow) {
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= N) return;
  const float gr = g[row];
  if (gr == 0.f) {
    if (lane == 0) {
      if (row_loss) row_loss[row] = 0.f;
      wl[row] = 0.f;
      lse2[row] = 0.f;
      srow[row] = 0.f;
    }
    return;
  }
  const float4* pr = part + row * n_part;
  float M = -INFINITY;
  for (int i = lane; i < n_part; i += 32) M = fmaxf(M, pr[i].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float L = 0.f, Sp = 0.f, Spz = 0.f;
  for (int i = lane; i < n_part; i += 32) {
    const float4 q = pr[i];
    if (q.y > 0.f) L += q.y * ex2((q.x - M) * kLog2eG);
    Sp += q.z;
    Spz += q.w;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    L += __shfl_xor_sync(0xffffffffu, L, o);
    Sp += __shfl_xor_sync(0xffffffffu, Sp, o);
    Spz += __shfl_xor_sync(0xffffffffu, Spz, o);
  }
  if (lane == 0) {
    const float lse = M + log2f(L) * kLn2G;
    const float ell = fmaf(lse, Sp, -Spz);
    if (row_loss) row_loss[row] = ell;
    wl[row] = gr * ell;
    lse2[row] = lse * kLog2eG;
    srow[row] = gr * Sp;
  }
}

template <bool A_MN, bool B_MN, int EPI>
cudaError_t run_gemm(GemmP P, const CUtensorMap& tmA, const CUtensorMap& tmB, cudaStream_t s) {
  P.tiles_m = (P.M + BM - 1) / BM;
  P.tiles_n = (P.N + BN - 1) / BN;
  P.k_steps = (P.K + BK - 1) / BK;
  const int tiles = P.tiles_m * P.tiles_n;
  if (tiles == 0) return cudaSuccess;
  auto kern = lm_gemm_kernel<A_MN, B_MN, EPI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  const int grid = tiles < sm_count() ? tiles : sm_count();
  kern<<<grid, kGThreads, kSmem, s>>>(P, tmA, tmB);
  return cudaGetLastError();
}

}  // namespace

size_t lm_head_ce_workspace(int64_t N, int64_t V) {
  const long long n_part = (V + BN - 1) / BN;
  const long long chunk = V < kChunkV ? V : kChunkV;
  auto al = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t b = al((size_t)N * n_part * 16) + 4 * al((size_t)N * 4) +
                  al((size_t)N * ((chunk + 7) / 8 * 8) * 2);
  return b < 256 ? 256 : b;
}

cudaError_t lm_head_ce_launch(const void* h, const void* W, const float* p, const float* g,
                              int64_t N, int64_t Hd, int64_t V, float* dh, float* dW,
                              float* row_loss, float* loss, void* workspace, cudaStream_t s) {
  cudaError_t e = bind_device_context();
  if (e != cudaSuccess) return e;
  const long long n_part = (V + BN - 1) / BN;
  const long long chunk = V < kChunkV ? V : kChunkV;
  const long long pitch = (chunk + 7) / 8 * 8;  // dz chunk row pitch (elements)
  auto al = [](size_t x) { return (x + 255) / 256 * 256; };
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  float4* part = reinterpret_cast<float4*>(ws);
  ws += al((size_t)N * n_part * 16);
  float* wl = reinterpret_cast<float*>(ws);
  ws += al((size_t)N * 4);
  float* lse2 = reinterpret_cast<float*>(ws);
  ws += al((size_t)N * 4);
  float* srow = reinterpret_cast<float*>(ws);
  ws += al((size_t)N * 4);
  ws += al((size_t)N * 4);  // spare (keeps the dz chunk 256-byte aligned for any N)
  __nv_bfloat16* dz = reinterpret_cast<__nv_bfloat16*>(ws);

  if (N == 0) {
    prof_before(s, STT_KERNEL_LM_HEAD_CE);
    e = soft_ce_loss_sum_launch(wl, N, loss, s);
    prof_after(s);
    return e;
  }
  // ---- STATS over the whole vocabulary: A = h (K-major), B = W (K-major)
  CUtensorMap tmH, tmW;
  if ((e = encode_bf16_2d(&tmH, h, Hd, N, Hd * 2, BM)) != cudaSuccess) return e;
  if ((e = encode_bf16_2d(&tmW, W, Hd, V, Hd * 2, BN)) != cudaSuccess) return e;
  GemmP S{};
  S.M = (int)N;
  S.N = (int)V;
  S.K = (int)Hd;
  S.p = p;
  S.ldp = V;
  S.g = g;
  S.part = part;
  S.n_part = (int)n_part;
  S.part0 = 0;
  prof_before(s, STT_KERNEL_LM_HEAD_CE);
  if ((e = run_gemm<false, false, kEpiStats>(S, tmH, tmW, s)) != cudaSuccess) {
    prof_after(s);
    return e;
  }
  lm_combine_kernel<<<(unsigned)((N + 7) / 8), 256, 0, s>>>(part, (int)n_part, g, N, row_loss, wl,
                                                           lse2, srow);
  if ((e = cudaGetLastError()) != cudaSuccess) {
    prof_after(s);
    return e;
  }
  if ((e = soft_ce_loss_sum_launch(wl, N, loss, s)) != cudaSuccess) {
    prof_after(s);
    return e;
  }

  // ---- the gradients, one vocabulary chunk at a time
  CUtensorMap tmHmn;  // h as an MN-major operand ([N rows = K][Hd = N])
  if ((e = encode_bf16_2d(&tmHmn, h, Hd, N, Hd * 2, 64)) != cudaSuccess) return e;
  for (long long v0 = 0; v0 < V; v0 += chunk) {
    const long long w = (V - v0) < chunk ? (V - v0) : chunk;
    const __nv_bfloat16* Wc = static_cast<const __nv_bfloat16*>(W) + v0 * Hd;
    // DZ: z chunk recomputed, dz = pi s - p g into the chunk buffer
    CUtensorMap tmWc, tmWcMN, tmDzK, tmDzMN;
    if ((e = encode_bf16_2d(&tmWc, Wc, Hd, w, Hd * 2, BN)) != cudaSuccess) break;
    if ((e = encode_bf16_2d(&tmWcMN, Wc, Hd, w, Hd * 2, 64)) != cudaSuccess) break;
    if ((e = encode_bf16_2d(&tmDzK, dz, w, N, pitch * 2, BM)) != cudaSuccess) break;
    if ((e = encode_bf16_2d(&tmDzMN, dz, w, N, pitch * 2, 64)) != cudaSuccess) break;
    GemmP D{};
    D.M = (int)N;
    D.N = (int)w;
    D.K = (int)Hd;
    D.p = p + v0;
    D.ldp = V;
    D.g = g;
    D.lse2 = lse2;
    D.srow = srow;
    D.dz = dz;
    D.lddz = pitch;
    if ((e = run_gemm<false, false, kEpiDz>(D, tmH, tmWc, s)) != cudaSuccess) break;
    // dh (+)= dz_c W_c: A = dz (K-major over the chunk), B = W_c (MN-major)
    GemmP Hh{};
    Hh.M = (int)N;
    Hh.N = (int)Hd;
    Hh.K = (int)w;
    Hh.out = dh;
    Hh.ldo = Hd;
    if (v0 == 0)
      e = run_gemm<false, true, kEpiStore>(Hh, tmDzK, tmWcMN, s);
    else
      e = run_gemm<false, true, kEpiAccum>(Hh, tmDzK, tmWcMN, s);
    if (e != cudaSuccess) break;
    // dW_c = dz_c^T h: A = dz^T (MN-major), B = h (MN-major)
    GemmP Ww{};
    Ww.M = (int)w;
    Ww.N = (int)Hd;
    Ww.K = (int)N;
    Ww.out = dW + v0 * Hd;
    Ww.ldo = Hd;
    if ((e = run_gemm<true, true, kEpiStore>(Ww, tmDzMN, tmHmn, s)) != cudaSuccess) break;
  }
  prof_after(s);
  return e;
}

STT_DEFINE_ERROR_ACCESSOR(lm_head_error_word)
STT_DEFINE_BUDGET_SETTER(lm_head_set_wait_budget)

}  // namespace stt
