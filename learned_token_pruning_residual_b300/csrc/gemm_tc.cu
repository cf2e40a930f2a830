// tcgen05 GEMMs of the gated prefill, bf16 in / fp32 accumulate:
//
//  * gate scoring (TokenGate pages, spke.com "TokenGate – Token-Gated
//    Attention macht das Vollfüllen von langen Kontexten bis zu 11,3-mal
//    schneller", section "Wie hat TokenGate das Pruning von Tokens
//    verstanden?", Gate-Modul): Z = X W1^T with the MLP head fused into the
//    epilogue, s = w2 . GELU(Z + b1) + b2, so Z never leaves the SM;
//  * the QKV projection of the kept rows (the pruned layers above the gate,
//    same section): QKV = X Wqkv^T, stored as bf16.
//
// One persistent CTA per SM walks output tiles of 128 x BN.  Warp 0 streams
// 128 x 64 A and BN x 64 B tiles into a STAGES-deep ring with TMA (128-byte
// swizzle); one thread of warp 1 issues tcgen05.mma (M=128, N=BN, K=16)
// into one of two TMEM accumulators; warps 2-5 drain the other accumulator
// (one row per thread via tcgen05.ld) while the next tile accumulates.
//
// CTAs run in clusters of CL along M: the CL CTAs of a cluster take CL
// consecutive M tiles with the same N tile, and each loads 1/CL of the B
// tile and multicasts it to all of them.  A stage is refilled only after the
// MMAs of every CTA in the cluster are done with it (their commits arrive on
// each CTA's `empty` barrier).  Measured on B300 (N = 131072 rows): clusters
// of two take the QKV projection from 113 to 111 us and leave the gate
// kernel unchanged; clusters of four are slower (the cluster's CTAs must
// free each stage together).
#include "tg_device.cuh"
#include "tg_internal.h"

namespace tg {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;  // 64 bf16 = 128 bytes = one swizzle row
enum { EPI_STORE_BF16 = 0, EPI_GATE = 1 };

// Epilogue warps: the gate's GELU.w2 head is arithmetic-heavy, so two warps
// share each TMEM lane quadrant there, each taking half of the columns.
__host__ __device__ constexpr int epi_warps(int epi) { return epi == EPI_GATE ? 8 : 4; }
__host__ __device__ constexpr int gemm_threads(int epi) { return 64 + 32 * epi_warps(epi); }


struct GemmArgs {
  int M, N, K;
  int tiles_m, tiles_n;
  int num_super;  // groups of CL M tiles x N tiles
  __nv_bfloat16* C;  // EPI_STORE_BF16: [M][ldc]
  int64_t ldc;
  const float* b1;  // EPI_GATE: N = Hg <= BN
  const float* w2;
  float b2;
  float* scores;
  uint32_t* status;
};

template <int BN, int STAGES>
struct GemmSmem {
  uint8_t a[STAGES][BM * BK * 2];  // each 16 KB, 1024-aligned
  uint8_t b[STAGES][BN * BK * 2];
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  float b1[256];
  float w2[256];
  float part[2][BM];  // gate: partial row sums of the column half 1, per accumulator
};

// GELU(z) = z Phi(z) = 0.5 z (1 + erf(z / sqrt 2)), with erf from
// Abramowitz & Stegun, Handbook of Mathematical Functions, 7.1.26:
//   erf(x) = 1 - (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) exp(-x^2),
//   t = 1 / (1 + p x),  x >= 0,  |error| <= 1.5e-7.
// 1 + erf(z / sqrt 2) is formed as 2 - q (z >= 0) or q (z < 0), q = poly * exp,
// so the negative tail has no cancellation.
__device__ __forceinline__ float gelu_as(float z) {
  const float x = fabsf(z) * 0.70710678118654752f;
  float t;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(t) : "f"(fmaf(0.3275911f, x, 1.0f)));
  float poly = fmaf(t, 1.061405429f, -1.453152027f);
  poly = fmaf(t, poly, 1.421413741f);
  poly = fmaf(t, poly, -0.284496736f);
  poly = fmaf(t, poly, 0.254829592f);
  poly *= t;
  const float q = poly * exp2_approx(-x * x * 1.4426950408889634f);
  return 0.5f * z * (z >= 0.f ? 2.0f - q : q);
}

template <int BN, int STAGES, int EPI, int CL>
__global__ void __launch_bounds__(gemm_threads(EPI), 1)
    gemm_bf16_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, const GemmArgs args) {
  using Smem = GemmSmem<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                     ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  constexpr uint32_t kStageBytes = (BM + BN) * BK * 2;
  constexpr uint32_t kTmemCols = 2 * BN;
  constexpr uint32_t kIdesc = idesc_bf16_f32(BM, BN, 0, 0);
  constexpr uint16_t kClusterMask = static_cast<uint16_t>((1u << CL) - 1u);
  constexpr int kEpiWarps = epi_warps(EPI);
  volatile int* abort = &S.abort;
  const int crank = CL > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int cid = static_cast<int>(blockIdx.x) / CL, ncl = static_cast<int>(gridDim.x) / CL;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&S.full[s]), 1);
      mbar_init(smem_u32(&S.empty[s]), CL);  // one MMA commit from each CTA of the cluster
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&S.acc_full[b]), 1);
      mbar_init(smem_u32(&S.acc_empty[b]), kEpiWarps);
    }
    mbar_init(smem_u32(&S.drain), 1);
    S.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&S.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  grid_dependency_wait();  // inputs come from the previous kernel in the stream
  allow_dependents_launch();
  tc_fence_before();
  __syncthreads();
  if (CL > 1) cluster_barrier();  // peers' barriers exist before anyone signals them
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  const int k_blocks = (args.K + BK - 1) / BK;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------- TMA producer
      const uint64_t pol_a = EPI == EPI_GATE ? l2_policy_evict_first() : l2_policy_evict_last();
      const uint64_t pol_b = l2_policy_evict_last();
      uint32_t it = 0;
      bool ok = true;
      for (int st = cid; ok && st < args.num_super; st += ncl) {
        const int tmg = st / args.tiles_n, tn = st - tmg * args.tiles_n;
        const int tm = tmg * CL + crank;
        for (int kb = 0; kb < k_blocks; ++kb) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
          if (!mbar_wait(smem_u32(&S.empty[s]), ph ^ 1, abort, args.status)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&S.full[s]);
          mbar_arrive_expect_tx(fb, kStageBytes);
          tma_load_2d_hint(smem_u32(S.a[s]), &tmA, fb, kb * BK, tm * BM, pol_a);
          if (CL == 1) {
            tma_load_2d_hint(smem_u32(S.b[s]), &tmB, fb, kb * BK, tn * BN, pol_b);
          } else {
            constexpr int kSlice = BN / CL;  // B rows this CTA loads for the cluster
            tma_load_2d_multicast(smem_u32(S.b[s]) + crank * kSlice * BK * 2, &tmB, fb, kb * BK,
                                  tn * BN + crank * kSlice, kClusterMask, pol_b);
          }
          ++it;
        }
      }
      // every issued fill lands before the CTA may exit
      for (uint32_t s = 0; s < STAGES && s < it; ++s) {
        const uint32_t last = ((it - 1 - s) / STAGES) * STAGES + s;
        mbar_wait_drain(smem_u32(&S.full[s]), (last / STAGES) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------ MMA issuer
      // The issuing thread waits for the tensor pipe to take each MMA, so the
      // shared-memory descriptors are formed once per stage; a K step of 16
      // inside the 128-byte swizzle row is +32 bytes on the start-address
      // field (address >> 4, no carry below 256 KB).
      uint64_t a_desc[STAGES], b_desc[STAGES];
#pragma unroll
      for (int s = 0; s < STAGES; ++s) {
        a_desc[s] = smem_desc_sw128(smem_u32(S.a[s]), 16, 1024);
        b_desc[s] = smem_desc_sw128(smem_u32(S.b[s]), 16, 1024);
      }
      uint32_t it = 0, local = 0;
      bool ok = true;
      for (int st = cid; ok && st < args.num_super; st += ncl, ++local) {
        const uint32_t buf = local & 1, aph = (local >> 1) & 1;
        if (!mbar_wait(smem_u32(&S.acc_empty[buf]), aph ^ 1, abort, args.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + buf * BN;
        for (int kb = 0; kb < k_blocks; ++kb, ++it) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
          if (!mbar_wait(smem_u32(&S.full[s]), ph, abort, args.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint64_t ad = 0, bd = 0;
#pragma unroll
          for (int q = 0; q < STAGES; ++q)
            if (q == static_cast<int>(s)) {
              ad = a_desc[q];
              bd = b_desc[q];
            }
          mma_ss(d_tmem, ad, bd, kIdesc, kb != 0);
#pragma unroll
          for (int k = 1; k < BK / 16; ++k) mma_ss(d_tmem, ad + 2 * k, bd + 2 * k, kIdesc, 1u);
          if (CL == 1) {
            mma_commit(smem_u32(&S.empty[s]));
          } else {
            mma_commit_multicast(smem_u32(&S.empty[s]), kClusterMask);
          }
        }
        if (ok) mma_commit(smem_u32(&S.acc_full[buf]));
      }
      // all MMAs of this thread complete before TMEM is released
      mma_commit(smem_u32(&S.drain));
      mbar_wait_drain(smem_u32(&S.drain), 0);
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;  // the TMEM lane quadrant this warp may read
    const int r_in_tile = q * 32 + lane;
    const int chalf = (warp - 2) >> 2;  // gate: the half of the columns this warp reduces
    if (EPI == EPI_GATE) {
      for (int i = threadIdx.x - 64; i < BN; i += 32 * kEpiWarps) {
        S.b1[i] = (i < args.N && args.b1 != nullptr) ? args.b1[i] : 0.f;
        S.w2[i] = (i < args.N) ? args.w2[i] : 0.f;
      }
      asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
    }
    uint32_t local = 0;
    for (int st = cid; st < args.num_super; st += ncl, ++local) {
      const uint32_t buf = local & 1, aph = (local >> 1) & 1;
      const bool ok_w = mbar_wait(smem_u32(&S.acc_full[buf]), aph, abort, args.status);
      if (EPI == EPI_GATE) {
        // the gate's epilogue warps meet at a named barrier below, so they
        // leave the loop together or not at all
        uint32_t any_fail;
        asm volatile(
            "{\n .reg .pred p, f;\n setp.eq.u32 f, %1, 0;\n"
            " barrier.cta.red.or.pred p, 1, %2, f;\n selp.u32 %0, 1, 0, p;\n}"
            : "=r"(any_fail)
            : "r"(static_cast<uint32_t>(ok_w)), "n"(32 * kEpiWarps)
            : "memory");
        if (any_fail) break;
      } else if (!ok_w) {
        break;
      }
      tc_fence_after();
      const int tmg = st / args.tiles_n, tn = st - tmg * args.tiles_n;
      const int tm = tmg * CL + crank;  // past the last M tile: every row fails row_ok
      const int64_t row = static_cast<int64_t>(tm) * BM + r_in_tile;
      const bool row_ok = row < args.M;
      const uint32_t t_row = tmem + buf * BN + (static_cast<uint32_t>(q * 32) << 16);
      if constexpr (EPI == EPI_STORE_BF16) {
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(t_row + c0, r);
          tmem_ld_wait();
          const int col0 = tn * BN + c0;
          if (row_ok && col0 < args.N) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
            __nv_bfloat16* dst = args.C + row * args.ldc + col0;
            if (col0 + 32 <= args.N) {
              uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
            } else {
              uint16_t* d16 = reinterpret_cast<uint16_t*>(dst);
              for (int i = 0; i < 32 && col0 + i < args.N; ++i)
                d16[i] = static_cast<uint16_t>((i & 1) ? (pk[i >> 1] >> 16) : (pk[i >> 1] & 0xFFFFu));
            }
          }
        }
      } else {
        // this warp's half of the columns; padded columns have w2 = 0
        float acc = 0.f;
        const int cbeg = chalf * (BN / 2);
#pragma unroll 1
        for (int c0 = cbeg; c0 < cbeg + BN / 2; c0 += 32) {
          if (c0 >= args.N) break;
          uint32_t r[32];
          tmem_ld32(t_row + c0, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float z = __uint_as_float(r[i]) + S.b1[c0 + i];
            acc = fmaf(S.w2[c0 + i], gelu_as(z), acc);
          }
        }
        if (chalf == 1) S.part[buf][r_in_tile] = acc;
        asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
        if (chalf == 0 && row_ok) args.scores[row] = acc + S.part[buf][r_in_tile] + args.b2;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&S.acc_empty[buf]));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  // no CTA leaves while a peer may still multicast into it or commit to its barriers
  if (CL > 1) cluster_barrier();
}

template <int BN, int STAGES, int EPI, int CL>
cudaError_t launch_gemm(const void* A, const void* B, const GemmArgs& a0, cudaStream_t stream) {
  GemmArgs args = a0;
  args.tiles_n = (args.N + BN - 1) / BN;
  args.tiles_m = (args.M + BM - 1) / BM;
  args.num_super = ((args.tiles_m + CL - 1) / CL) * args.tiles_n;
  args.status = device_status_word();
  if (args.tiles_m == 0 || args.tiles_n == 0) return cudaSuccess;
  CUtensorMap tmA, tmB;
  if (!make_tmap_2d(&tmA, A, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, args.K, args.M,
                    static_cast<uint64_t>(args.K) * 2, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tmB, B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, args.K, args.N,
                    static_cast<uint64_t>(args.K) * 2, BK, BN / CL, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  auto kernel = gemm_bf16_tc_kernel<BN, STAGES, EPI, CL>;
  const size_t smem = sizeof(GemmSmem<BN, STAGES>) + 1024;
  cudaError_t err =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int max_clusters = sm_count() / CL;
  const int clusters = args.num_super < max_clusters ? args.num_super : max_clusters;
  err = launch_pdl(kernel, dim3(static_cast<unsigned>(clusters * CL)), dim3(gemm_threads(EPI)),
                   smem, stream, CL, tmA, tmB, args);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gate_bf16(const void* X, int64_t N, int d, const void* W1, const float* b1,
                             int Hg, const float* w2, float b2, float* scores,
                             cudaStream_t stream) {
  GemmArgs a{};
  a.M = static_cast<int>(N);
  a.N = Hg;
  a.K = d;
  a.b1 = b1;
  a.w2 = w2;
  a.b2 = b2;
  a.scores = scores;
  if (Hg <= 128) return launch_gemm<128, 6, EPI_GATE, 2>(X, W1, a, stream);
  return launch_gemm<256, 4, EPI_GATE, 2>(X, W1, a, stream);
}

cudaError_t launch_qkv_bf16(const void* X, int64_t M, int d, const void* W, int ncols, void* Y,
                            cudaStream_t stream) {
  GemmArgs a{};
  a.M = static_cast<int>(M);
  a.N = ncols;
  a.K = d;
  a.C = static_cast<__nv_bfloat16*>(Y);
  a.ldc = ncols;
  return launch_gemm<256, 4, EPI_STORE_BF16, 2>(X, W, a, stream);
}

}  // namespace tg
