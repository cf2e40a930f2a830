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
// Persistent CTA pairs (clusters of two) walk 256 x BN output tiles; see
// the CTA-pair kernel below.  Warp 0 of each CTA streams its A rows and its
// half of B with TMA (128-byte swizzle) into a 6-stage ring; one thread of
// rank 0 issues the M = 256 tcgen05.mma into one of two TMEM accumulators;
// the epilogue warps of both CTAs drain the other accumulator (one row per
// thread via tcgen05.ld) while the next tile accumulates.
//
// Measured on B300 (N = 131072 rows): the pair form took the gate kernel
// from 120 to 114 us (4.7 TB/s) and the QKV projection from 110 to 99.5 us
// (1420 TFLOP/s) against single-CTA tiles with 4 x 48 KB stages, which were
// latency-bound on their operand loads.
#include "tg_device.cuh"
#include "tg_internal.h"

namespace tg {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;  // 64 bf16 = 128 bytes = one swizzle row
enum {
  EPI_STORE_BF16 = 0,  // C = acc, bf16
  EPI_GATE = 1,        // s = w2 . GELU(acc + b1) + b2
  EPI_QKNORM_ROPE = 2, // per-head RMSNorm of q and k, rotary embedding, bf16
  EPI_RESID_ADD = 3,   // residual (fp32) += acc
  EPI_SWIGLU = 4       // C = silu(acc[:, :BN/2]) * acc[:, BN/2:], bf16
};

// Epilogue warps: the gate's GELU.w2 head is arithmetic-heavy, so two warps
// share each TMEM lane quadrant there, each taking half of the columns.
__host__ __device__ constexpr int epi_warps(int epi) { return epi == EPI_GATE ? 8 : 4; }
__host__ __device__ constexpr int gemm_threads(int epi) { return 64 + 32 * epi_warps(epi); }


struct GemmArgs {
  int M, N, K;
  int tiles_m, tiles_n;
  int num_super;  // pairs of M tiles x N tiles
  __nv_bfloat16* C;  // EPI_STORE_BF16: [M][ldc]
  int64_t ldc;
  const float* b1;  // EPI_GATE: N = Hg <= BN
  const float* w2;
  float b2;
  float* scores;
  SelectWorkspace* sel_ws;  // EPI_GATE, nullable: first radix histogram of the span's keys
  int doc_b, doc_e;
  // EPI_QKNORM_ROPE: heads of 128 columns; q heads [0, Hq), k heads
  // [Hq, Hq + Hkv), then v; gamma_q / gamma_k [128]; rope [M][64] (cos, sin)
  int Hq, Hkv;
  const float* gamma_q;
  const float* gamma_k;
  float eps;
  const float2* rope;
  float* residual;  // EPI_RESID_ADD: [M][ldc] fp32
  uint32_t* status;
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

// Drains one 128 x BN accumulator tile from TMEM (this warp's lane quadrant
// q, row r_in_tile): bf16 store, or the gate's GELU.w2 head (two warps per
// quadrant, column halves chalf, partial sums met in `part`).
template <int BN, int EPI, int kEpiWarps>
__device__ __forceinline__ void epilogue_tile(const GemmArgs& args, const float* b1s,
                                              const float* w2s, float* part, uint32_t* hist,
                                              uint32_t tmem_acc, int tm, int tn, int r_in_tile,
                                              int q, int chalf) {
  const int64_t row = static_cast<int64_t>(tm) * BM + r_in_tile;
  const bool row_ok = row < args.M;
  const uint32_t t_row = tmem_acc + (static_cast<uint32_t>(q * 32) << 16);
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
  } else if constexpr (EPI == EPI_QKNORM_ROPE) {
    // the tile holds two heads of 128 columns; for a q or k head the row is
    // normalised over its 128 columns (RMSNorm with gamma_q / gamma_k), then
    // the pairs (c, c + 64) are rotated by the row's rotary angles
#pragma unroll 1
    for (int hh = 0; hh < BN / 128; ++hh) {
      const int col0 = tn * BN + hh * 128;
      const int hd = col0 / 128;
      if (col0 >= args.N) break;
      float x[128];
#pragma unroll
      for (int c = 0; c < 128; c += 32) {
        uint32_t r[32];
        tmem_ld32(t_row + hh * 128 + c, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) x[c + i] = __uint_as_float(r[i]);
      }
      if (hd < args.Hq + args.Hkv) {
        const float* gam = hd < args.Hq ? args.gamma_q : args.gamma_k;
        float ss0 = 0.f, ss1 = 0.f;
#pragma unroll
        for (int c = 0; c < 128; c += 2) {
          ss0 = fmaf(x[c], x[c], ss0);
          ss1 = fmaf(x[c + 1], x[c + 1], ss1);
        }
        const float rstd = rsqrtf((ss0 + ss1) * (1.f / 128.f) + args.eps);
#pragma unroll
        for (int c = 0; c < 128; ++c) x[c] *= rstd * __ldg(gam + c);
        if (row_ok) {
          const float4* cs = reinterpret_cast<const float4*>(args.rope + row * 64);
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            const float4 t = __ldg(cs + c / 2);  // (cos, sin) of pairs c and c + 1
            const float a0 = x[c], b0 = x[c + 64], a1 = x[c + 1], b1 = x[c + 65];
            x[c] = a0 * t.x - b0 * t.y;
            x[c + 64] = b0 * t.x + a0 * t.y;
            x[c + 1] = a1 * t.z - b1 * t.w;
            x[c + 65] = b1 * t.z + a1 * t.w;
          }
        }
      }
      if (row_ok) {
        uint4* d4 = reinterpret_cast<uint4*>(args.C + row * args.ldc + col0);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          d4[i] = make_uint4(pack_bf16x2(x[8 * i + 0], x[8 * i + 1]),
                             pack_bf16x2(x[8 * i + 2], x[8 * i + 3]),
                             pack_bf16x2(x[8 * i + 4], x[8 * i + 5]),
                             pack_bf16x2(x[8 * i + 6], x[8 * i + 7]));
      }
    }
  } else if constexpr (EPI == EPI_RESID_ADD) {
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 32) {
      uint32_t r[32];
      tmem_ld32(t_row + c0, r);
      tmem_ld_wait();
      const int col0 = tn * BN + c0;
      if (row_ok && col0 < args.N) {
        float4* dst = reinterpret_cast<float4*>(args.residual + row * args.ldc + col0);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float4 v = dst[i];
          v.x += __uint_as_float(r[4 * i + 0]);
          v.y += __uint_as_float(r[4 * i + 1]);
          v.z += __uint_as_float(r[4 * i + 2]);
          v.w += __uint_as_float(r[4 * i + 3]);
          dst[i] = v;
        }
      }
    }
  } else if constexpr (EPI == EPI_SWIGLU) {
    // columns [0, BN/2) of the tile are gate outputs, [BN/2, BN) the matching
    // up outputs (the two CTAs of the pair load their halves of B from W_gate
    // and W_up); silu(g) = g / (1 + 2^(-g log2 e))
#pragma unroll 1
    for (int c0 = 0; c0 < BN / 2; c0 += 32) {
      uint32_t gr[32], ur[32];
      tmem_ld32(t_row + c0, gr);
      tmem_ld32(t_row + BN / 2 + c0, ur);
      tmem_ld_wait();
      const int col0 = tn * (BN / 2) + c0;
      if (row_ok && col0 < args.N / 2) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float y[2];
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const float gv = __uint_as_float(gr[2 * i + k]);
            const float e = exp2_approx(-gv * 1.4426950408889634f);
            float inv;
            asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(inv) : "f"(1.f + e));
            y[k] = gv * inv * __uint_as_float(ur[2 * i + k]);
          }
          pk[i] = pack_bf16x2(y[0], y[1]);
        }
        uint4* d4 = reinterpret_cast<uint4*>(args.C + row * args.ldc + col0);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
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
        const float z = __uint_as_float(r[i]) + b1s[c0 + i];
        acc = fmaf(w2s[c0 + i], gelu_as(z), acc);
      }
    }
    if (chalf == 1) part[r_in_tile] = acc;
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
    if (chalf == 0) {
      const float s = acc + part[r_in_tile] + args.b2;
      if (row_ok) args.scores[row] = s;
      if (args.sel_ws != nullptr) {
        // first radix pass of the select: top 11 bits of the score's key,
        // for document rows only; warp-aggregated shared-memory counts
        uint32_t bin = 0xFFFFFFFFu;
        if (row_ok && row >= args.doc_b && row < args.doc_e) {
          const uint32_t u = __float_as_uint(s);
          bin = ((u & 0x80000000u) ? ~u : (u | 0x80000000u)) >> 21;
        }
        const uint32_t peers = __match_any_sync(0xffffffffu, bin);
        if (bin != 0xFFFFFFFFu && (threadIdx.x & 31) == __ffs(peers) - 1)
          atomicAdd(hist + bin, __popc(peers));
      }
    }
  }
}

// ---------------------------------------------------------------------------
// CTA-pair form (tcgen05 cta_group::2): a cluster of two CTAs computes a
// 256 x BN tile with one M = 256 MMA per K step, issued by rank 0.  Each CTA
// stages its own 128 rows of A and half (BN/2 rows) of B, so a stage is
// 32 KB instead of 48 KB and six stages fit: 3072 MMA cycles of loads in
// flight instead of 2048, and each CTA reads half of B.  Both CTAs' TMA
// loads complete on rank 0's `full` barrier; rank 0's commits release the
// stage (`empty`) and publish the accumulator (`acc_full`) in both CTAs;
// both CTAs' epilogue warps release the accumulator on rank 0's `acc_empty`.
template <int BN, int STAGES>
struct PairSmem {
  uint8_t a[STAGES][BM * BK * 2];         // 16 KB: this CTA's 128 rows of A
  uint8_t b[STAGES][(BN / 2) * BK * 2];   // this CTA's half of the B tile
  uint64_t full[STAGES];                  // rank 0: both CTAs' bytes landed
  uint64_t empty[STAGES];                 // each CTA: rank 0's MMAs are done with the stage
  uint64_t acc_full[2];                   // each CTA: the accumulator is complete
  uint64_t acc_empty[2];                  // rank 0: both CTAs drained the accumulator
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  float b1[256];
  float w2[256];
  float part[2][BM];
  uint32_t hist[2048];  // gate: first radix histogram of this CTA's document rows
};

template <int BN, int STAGES, int EPI>
__global__ void __launch_bounds__(gemm_threads(EPI), 1)
    gemm_bf16_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                          const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmB2, const GemmArgs args) {
  using Smem = PairSmem<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                     ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  constexpr uint32_t kStageBytes = (BM + BN / 2) * BK * 2;  // one CTA's share of a stage
  constexpr uint32_t kTmemCols = 2 * BN;
  constexpr uint32_t kIdesc = idesc_bf16_f32(2 * BM, BN, 0, 0);
  constexpr int kEpiWarps = epi_warps(EPI);
  volatile int* abort = &S.abort;
  const uint32_t crank = cluster_ctarank();
  const int cid = static_cast<int>(blockIdx.x) / 2, ncl = static_cast<int>(gridDim.x) / 2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&S.full[s]), 1);   // rank 0's producer arrives; bytes from both
      mbar_init(smem_u32(&S.empty[s]), 1);  // one commit from rank 0
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&S.acc_full[b]), 1);
      mbar_init(smem_u32(&S.acc_empty[b]), 2 * kEpiWarps);  // both CTAs' epilogue warps
    }
    mbar_init(smem_u32(&S.drain), 1);
    S.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (EPI == EPI_SWIGLU) tma_prefetch_desc(&tmB2);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&S.tmem_base), kTmemCols);
    tmem_relinquish_pair();
  }
  grid_dependency_wait();  // inputs come from the previous kernel in the stream
  allow_dependents_launch();
  tc_fence_before();
  __syncthreads();
  cluster_barrier();  // both CTAs' barriers exist before anyone signals them
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
        const int tmp = st / args.tiles_n, tn = st - tmp * args.tiles_n;
        const int tm = 2 * tmp + static_cast<int>(crank);
        for (int kb = 0; kb < k_blocks; ++kb) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
          if (!mbar_wait(smem_u32(&S.empty[s]), ph ^ 1, abort, args.status)) {
            ok = false;
            break;
          }
          const uint32_t fb = map_shared_to_rank(smem_u32(&S.full[s]), 0);
          if (crank == 0) mbar_arrive_expect_tx(smem_u32(&S.full[s]), 2 * kStageBytes);
          tma_load_2d_pair(smem_u32(S.a[s]), &tmA, fb, kb * BK, tm * BM, pol_a);
          if (EPI == EPI_SWIGLU) {  // rank 0: W_gate rows, rank 1: W_up rows
            tma_load_2d_pair(smem_u32(S.b[s]), crank ? &tmB2 : &tmB, fb, kb * BK,
                             tn * (BN / 2), pol_b);
          } else {
            tma_load_2d_pair(smem_u32(S.b[s]), &tmB, fb, kb * BK,
                             tn * BN + static_cast<int>(crank) * (BN / 2), pol_b);
          }
          ++it;
        }
      }
      // rank 0: every fill of both CTAs landed before the pair may exit
      if (crank == 0) {
        for (uint32_t s = 0; s < STAGES && s < it; ++s) {
          const uint32_t last = ((it - 1 - s) / STAGES) * STAGES + s;
          mbar_wait_drain(smem_u32(&S.full[s]), (last / STAGES) & 1);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && crank == 0) {
      // ------------------------------------------------------ MMA issuer
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
          mma_ss_pair(d_tmem, ad, bd, kIdesc, kb != 0);
#pragma unroll
          for (int k = 1; k < BK / 16; ++k) mma_ss_pair(d_tmem, ad + 2 * k, bd + 2 * k, kIdesc, 1u);
          mma_commit_pair_multicast(smem_u32(&S.empty[s]), 3);
        }
        if (ok) mma_commit_pair_multicast(smem_u32(&S.acc_full[buf]), 3);
      }
      // all MMAs complete before either CTA releases TMEM or shared memory
      mma_commit_pair(smem_u32(&S.drain));
      mbar_wait_drain(smem_u32(&S.drain), 0);
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;  // the TMEM lane quadrant this warp may read
    const int r_in_tile = q * 32 + lane;
    const int chalf = (warp - 2) >> 2;
    if (EPI == EPI_GATE) {
      for (int i = threadIdx.x - 64; i < BN; i += 32 * kEpiWarps) {
        S.b1[i] = (i < args.N && args.b1 != nullptr) ? args.b1[i] : 0.f;
        S.w2[i] = (i < args.N) ? args.w2[i] : 0.f;
      }
      if (args.sel_ws != nullptr)
        for (int i = threadIdx.x - 64; i < 2048; i += 32 * kEpiWarps) S.hist[i] = 0u;
      asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
    }
    const uint32_t acc_empty0 = map_shared_to_rank(smem_u32(&S.acc_empty[0]), 0);
    uint32_t local = 0;
    for (int st = cid; st < args.num_super; st += ncl, ++local) {
      const uint32_t buf = local & 1, aph = (local >> 1) & 1;
      const bool ok_w = mbar_wait(smem_u32(&S.acc_full[buf]), aph, abort, args.status);
      if (EPI == EPI_GATE) {
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
      const int tmp = st / args.tiles_n, tn = st - tmp * args.tiles_n;
      const int tm = 2 * tmp + static_cast<int>(crank);  // past the last M tile: rows fail row_ok
      epilogue_tile<BN, EPI, kEpiWarps>(args, S.b1, S.w2, S.part[buf], S.hist, tmem + buf * BN,
                                        tm, tn, r_in_tile, q, chalf);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc_empty0 + buf * 8);  // rank 0's acc_empty[buf]
    }
    if (EPI == EPI_GATE && args.sel_ws != nullptr) {
      // this CTA's counts into the workspace; one thread stamps the header
      // with the span, so that a select call on the same span skips its
      // first pass
      asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
      for (int i = threadIdx.x - 64; i < 2048; i += 32 * kEpiWarps) {
        const uint32_t c = S.hist[i];
        if (c) atomicAdd(&args.sel_ws->gate_hist[i], c);
      }
      if (blockIdx.x == 0 && threadIdx.x == 64) {
        args.sel_ws->hdr[0] = kSelectHistMagic;
        args.sel_ws->hdr[1] = static_cast<uint32_t>(args.M);
        args.sel_ws->hdr[2] = static_cast<uint32_t>(args.doc_b);
        args.sel_ws->hdr[3] = static_cast<uint32_t>(args.doc_e);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_barrier();  // rank 0's MMAs, which read both CTAs' memory, are complete
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

template <int BN, int STAGES, int EPI>
cudaError_t launch_gemm_pair(const void* A, const void* B, const GemmArgs& a0,
                             cudaStream_t stream, const void* B2 = nullptr) {
  GemmArgs args = a0;
  args.tiles_n = (args.N + BN - 1) / BN;
  args.tiles_m = (args.M + BM - 1) / BM;
  args.num_super = ((args.tiles_m + 1) / 2) * args.tiles_n;
  args.status = device_status_word();
  if (args.tiles_m == 0 || args.tiles_n == 0) return cudaSuccess;
  // B rows: N, or for the gate|up pair each of the two weights' N / 2 rows
  const uint64_t b_rows = EPI == EPI_SWIGLU ? static_cast<uint64_t>(args.N / 2) : args.N;
  CUtensorMap tmA, tmB, tmB2;
  if (!make_tmap_2d(&tmA, A, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, args.K, args.M,
                    static_cast<uint64_t>(args.K) * 2, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tmB, B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, args.K, b_rows,
                    static_cast<uint64_t>(args.K) * 2, BK, BN / 2, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (EPI == EPI_SWIGLU) {
    if (!make_tmap_2d(&tmB2, B2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, args.K, b_rows,
                      static_cast<uint64_t>(args.K) * 2, BK, BN / 2, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  } else {
    tmB2 = tmB;  // unused
  }
  auto kernel = gemm_bf16_pair_kernel<BN, STAGES, EPI>;
  const size_t smem = sizeof(PairSmem<BN, STAGES>) + 1024;
  cudaError_t err =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int max_pairs = sm_count() / 2;
  const int pairs = args.num_super < max_pairs ? args.num_super : max_pairs;
  err = launch_pdl(kernel, dim3(static_cast<unsigned>(2 * pairs)), dim3(gemm_threads(EPI)), smem,
                   stream, 2u, tmA, tmB, tmB2, args);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

// Rotary table of the kept rows: table[m][c] = (cos, sin)(pos[m] theta_c),
// theta_c = base^(-2c / dh), c < dh / 2.  The angle is formed and reduced
// modulo 2 pi in fp64 (a position near 131072 times theta_0 = 1 would lose
// ~1e-2 rad in fp32); the reduced angle's cosine and sine are taken in fp32.
__global__ void __launch_bounds__(256)
    rope_table_kernel(const int32_t* __restrict__ pos, int64_t M, int half, double log2_base,
                      float2* __restrict__ table) {
  grid_dependency_wait();
  allow_dependents_launch();
  const int64_t n = M * half;
  constexpr double kTwoPi = 6.283185307179586476925286766559;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t m = i / half;
    const int c = static_cast<int>(i - m * half);
    const double theta = exp2(-log2_base * (2.0 * c) / (2.0 * half));
    const double a = static_cast<double>(__ldg(pos + m)) * theta;
    const double r = a - kTwoPi * rint(a / kTwoPi);
    float sn, cs;
    sincosf(static_cast<float>(r), &sn, &cs);
    table[i] = make_float2(cs, sn);
  }
}

}  // namespace

cudaError_t launch_gate_bf16(const void* X, int64_t N, int d, const void* W1, const float* b1,
                             int Hg, const float* w2, float b2, float* scores,
                             SelectWorkspace* sel_ws, int64_t doc_b, int64_t doc_e,
                             cudaStream_t stream) {
  GemmArgs a{};
  a.sel_ws = sel_ws;
  a.doc_b = static_cast<int>(doc_b);
  a.doc_e = static_cast<int>(doc_e);
  a.M = static_cast<int>(N);
  a.N = Hg;
  a.K = d;
  a.b1 = b1;
  a.w2 = w2;
  a.b2 = b2;
  a.scores = scores;
  if (Hg <= 128) return launch_gemm_pair<128, 8, EPI_GATE>(X, W1, a, stream);
  return launch_gemm_pair<256, 6, EPI_GATE>(X, W1, a, stream);
}

cudaError_t launch_qkv_bf16(const void* X, int64_t M, int d, const void* W, int ncols, void* Y,
                            cudaStream_t stream) {
  GemmArgs a{};
  a.M = static_cast<int>(M);
  a.N = ncols;
  a.K = d;
  a.C = static_cast<__nv_bfloat16*>(Y);
  a.ldc = ncols;
  return launch_gemm_pair<256, 6, EPI_STORE_BF16>(X, W, a, stream);
}

cudaError_t launch_qkv_qknorm_rope_bf16(const void* X, int64_t M, int d, const void* W, int Hq,
                                       int Hkv, const float* gamma_q, const float* gamma_k,
                                       float eps, const float2* rope, void* Y,
                                       cudaStream_t stream) {
  GemmArgs a{};
  a.M = static_cast<int>(M);
  a.N = (Hq + 2 * Hkv) * 128;
  a.K = d;
  a.C = static_cast<__nv_bfloat16*>(Y);
  a.ldc = a.N;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.gamma_q = gamma_q;
  a.gamma_k = gamma_k;
  a.eps = eps;
  a.rope = rope;
  return launch_gemm_pair<256, 6, EPI_QKNORM_ROPE>(X, W, a, stream);
}

cudaError_t launch_linear_resid_bf16(const void* X, int64_t M, int K, const void* W, int N,
                                     float* residual, cudaStream_t stream) {
  GemmArgs a{};
  a.M = static_cast<int>(M);
  a.N = N;
  a.K = K;
  a.residual = residual;
  a.ldc = N;
  return launch_gemm_pair<256, 6, EPI_RESID_ADD>(X, W, a, stream);
}

cudaError_t launch_swiglu_bf16(const void* X, int64_t M, int d, const void* Wg, const void* Wu,
                               int F, void* Y, cudaStream_t stream) {
  GemmArgs a{};
  a.M = static_cast<int>(M);
  a.N = 2 * F;
  a.K = d;
  a.C = static_cast<__nv_bfloat16*>(Y);
  a.ldc = F;
  return launch_gemm_pair<256, 6, EPI_SWIGLU>(X, Wg, a, stream, Wu);
}

cudaError_t launch_rope_table(const int32_t* pos, int64_t M, int dh, double base, float2* table,
                              cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  const int half = dh / 2;
  const int64_t n = M * half;
  const int64_t want = (n + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  const int grid = static_cast<int>(want < cap ? want : cap);
  return launch_pdl(rope_table_kernel, dim3(grid), dim3(256), 0, stream, 1u, pos, M, half,
                    log2(base), table);
}

}  // namespace tg
