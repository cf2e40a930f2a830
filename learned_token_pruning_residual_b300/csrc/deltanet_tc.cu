// The gated delta rule on the tensor cores (bf16 inputs, head size 128).
// Same recurrence and chunked form as deltanet.cu (TokenGate pages:
// ai4bro.com, section "การใช้งานกับโมเดล hybrid-attention"; spke.com, section
// "Wird es auf Hybrid-Attention-Modellen funktionieren?": the DeltaNet layers
// of a hybrid model run over the kept tokens only).  Per head, chunks of
// C = 64 tokens, g_i the cumulative product of alpha inside the chunk, S the
// state (dv x dk) before the chunk:
//     T   = (I + A)^{-1},      A_ij = (g_i / g_j) beta_j (k_i . k_j), j < i
//     U   = T V - T diag(g) K S^T                     (the delta-rule errors)
//     O   = diag(g) Q S^T + P U,  P_ij = (g_i / g_j) beta_j (q_i . k_j), j <= i
//     S  <- g_C S + U^T diag(beta g_C / g) K
// Two kernels:
//   dn_prep_tc_kernel  one CTA per (pair of chunks, head), all in parallel:
//                      K K^T and Q K^T as one M = 128 MMA each (the two chunks
//                      stacked; the cross-chunk blocks are ignored), A and P
//                      formed from them row by row, T by forward substitution
//                      (one column per thread, fp32), and W- = -T diag(g) K as
//                      one MMA with the block-diagonal T as its A operand.
//                      Writes per chunk W-, diag(g) Q, diag(beta g_C / g) K,
//                      T and P (bf16) and g_C.
//   dn_scan_tc_kernel  one CTA per head, walking the chunks in order.  The
//                      state lives in TMEM as the fp32 accumulator of the
//                      update MMA (lane = row of S); a bf16 copy of it, also
//                      in TMEM, is the A operand of the products with S, so a
//                      chunk costs five MMAs (M = 128 = dv):
//                        U^T  = V^T T^T  +  S (W-)^T     (T V does not need S)
//                        O^T  = S (diag(g) Q)^T  +  U^T P^T
//                        S    = g_C S + U^T (diag(beta g_C / g) K)
//                      and two TMEM round trips by the row threads (U to
//                      bf16; S to bf16 and scaled by the next g_C).  O is read
//                      out one chunk behind, double-buffered.
// All products take bf16 operands with fp32 accumulation; the state, A, T and
// every sum are fp32.
#include <algorithm>

#include "tg_device.cuh"
#include "tg_internal.h"

namespace tg {
namespace {

constexpr int kC = 64;   // tokens per chunk
constexpr int kD = 128;  // dk = dv
constexpr int kThreads = 256;
constexpr uint32_t kBox = 64 * 64 * 2;         // one 64 x 64 bf16 TMA box: 8 KB
constexpr uint32_t kHalf128 = 128 * 64 * 2;    // 128 rows x 64 bf16: 16 KB
constexpr uint32_t kTile128 = 2 * kHalf128;    // 128 rows x 128 bf16: 32 KB

// Per-(chunk, head) operands in the workspace, each array indexed by
// rec = chunk * H + head: wn / qg / kp [rec][64][128], tinv / p [rec][64][64]
// (bf16, row-major), gc [rec] (fp32).
struct DnRec {
  __nv_bfloat16* wn;
  __nv_bfloat16* qg;
  __nv_bfloat16* kp;
  __nv_bfloat16* tinv;
  __nv_bfloat16* p;
  float* gc;
};

DnRec carve(void* ws, int64_t recs) {
  uint8_t* b = static_cast<uint8_t*>(ws);
  const int64_t big = recs * kC * kD * 2, small = recs * kC * kC * 2;
  DnRec r;
  r.wn = reinterpret_cast<__nv_bfloat16*>(b);
  r.qg = reinterpret_cast<__nv_bfloat16*>(b + big);
  r.kp = reinterpret_cast<__nv_bfloat16*>(b + 2 * big);
  r.tinv = reinterpret_cast<__nv_bfloat16*>(b + 3 * big);
  r.p = reinterpret_cast<__nv_bfloat16*>(b + 3 * big + small);
  r.gc = reinterpret_cast<float*>(b + 3 * big + 2 * small);
  return r;
}

// One lane waits, the warp follows (keeps the .sync.aligned TMEM ops
// warp-uniform when a wait gives up).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          uint32_t* status) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort, status) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

__device__ __forceinline__ void row_sync() {  // the four row warps (4-7)
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

// byte offset of element (row, col) of a 128-byte-swizzled K-major tile made
// of 64-column halves `half_bytes` apart
__device__ __forceinline__ uint32_t sw128_offset(int row, int col, uint32_t half_bytes) {
  const int c = col & 63;
  return static_cast<uint32_t>(col >> 6) * half_bytes + row * 128 +
         ((((c >> 3) ^ (row & 7)) << 4) | ((c & 7) << 1));
}

__device__ __forceinline__ uint32_t scale_bf16x2(uint32_t v, float f) {
  return pack_bf16x2(bf16lo_to_f32(v) * f, bf16hi_to_f32(v) * f);
}

// ================================================================== prep ==
struct PrepSmem {
  uint8_t q[kTile128];   // Q of the two chunks: 128 token rows, K-major, 128-byte swizzle
  uint8_t k[kTile128];   // K, same layout (also the MN-major B of W- = A_W K)
  uint8_t aw[kTile128];  // A_W = -T diag(g), block diagonal, K-major, 128-byte swizzle
  float a[2][kC][kC + 4];  // A of each chunk (rows 16-byte aligned)
  float lg[128], beta[128];
  float carry[2];
  uint64_t in_full, g_full, a_ready, w_full, drain;
  uint32_t tmem_base;
  int abort;
};

__global__ void __launch_bounds__(kThreads, 1)
    dn_prep_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k, const float* __restrict__ alpha,
                      const float* __restrict__ beta, int T_len, int H, int n_ch, DnRec rec,
                      uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  PrepSmem& S = *reinterpret_cast<PrepSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pair = static_cast<int>(blockIdx.x) / H, h = static_cast<int>(blockIdx.x) % H;
  const int t0 = pair * 2 * kC;
  volatile int* abort = &S.abort;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&S.in_full), 1);
    mbar_init(smem_u32(&S.g_full), 1);
    mbar_init(smem_u32(&S.a_ready), 1);
    mbar_init(smem_u32(&S.w_full), 1);
    mbar_init(smem_u32(&S.drain), 1);
    S.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&S.tmem_base), 256);
    tmem_relinquish();
  }
  if (warp == 2 || warp == 3) {  // the off-diagonal blocks of A_W stay zero
    uint4* z = reinterpret_cast<uint4*>(S.aw);
    for (int e = threadIdx.x - 64; e < static_cast<int>(kTile128 / 16); e += 64)
      z[e] = make_uint4(0, 0, 0, 0);
  }
  grid_dependency_wait();
  allow_dependents_launch();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------- TMA
      mbar_arrive_expect_tx(smem_u32(&S.in_full), 2 * kTile128);
      for (int bx = 0; bx < 2; ++bx) {
        tma_load_2d(smem_u32(S.q) + bx * kHalf128, &tm_q, smem_u32(&S.in_full), h * kD + bx * 64,
                    t0);
        tma_load_2d(smem_u32(S.k) + bx * kHalf128, &tm_k, smem_u32(&S.in_full), h * kD + bx * 64,
                    t0);
      }
      mbar_wait_drain(smem_u32(&S.in_full), 0);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------- MMA
      bool ok = mbar_wait(smem_u32(&S.in_full), 0, abort, status);
      if (ok) {
        tc_fence_after();
        constexpr uint32_t idesc_g = idesc_bf16_f32(128, 128, 0, 0);
        const uint64_t kd = smem_desc_sw128(smem_u32(S.k), 16, 1024);
        const uint64_t qd = smem_desc_sw128(smem_u32(S.q), 16, 1024);
        // G1 = K K^T -> columns [0, 128), G2 = Q K^T -> [128, 256)
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint64_t off = ((kk >> 2) * kHalf128 + (kk & 3) * 32) >> 4;
          mma_ss(tmem, kd + off, kd + off, idesc_g, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint64_t off = ((kk >> 2) * kHalf128 + (kk & 3) * 32) >> 4;
          mma_ss(tmem + 128, qd + off, kd + off, idesc_g, kk > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&S.g_full));
        ok = mbar_wait(smem_u32(&S.a_ready), 0, abort, status);
      }
      if (ok) {
        tc_fence_after();
        // W- = A_W K: A_W K-major over the 128 tokens, K as the MN-major B
        // (K = tokens, N = dk)
        constexpr uint32_t idesc_w = idesc_bf16_f32(128, 128, 0, 1);
        const uint64_t ad = smem_desc_sw128(smem_u32(S.aw), 16, 1024);
        const uint64_t bd = smem_desc_sw128(smem_u32(S.k), kHalf128, 1024);
#pragma unroll
        for (int kk = 0; kk < 128 / 16; ++kk)
          mma_ss(tmem, ad + (((kk >> 2) * kHalf128 + (kk & 3) * 32) >> 4),
                 bd + ((kk * 16 * 128) >> 4), idesc_w, kk > 0 ? 1u : 0u);
        mma_commit(smem_u32(&S.w_full));
      }
      mma_commit(smem_u32(&S.drain));
      mbar_wait_drain(smem_u32(&S.drain), 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------- row threads
    const int i = threadIdx.x - 128;  // token row of the pair = TMEM lane
    const int ci = i >> 6, li = i & 63, cb = ci * kC;
    const int t = t0 + i;
    const int c = 2 * pair + ci;  // chunk
    const bool chunk_ok = c < n_ch;  // warp-uniform
    const int64_t rc = static_cast<int64_t>(c) * H + h;
    const uint32_t lane_base = static_cast<uint32_t>((warp - 4) * 32) << 16;
    // cumulative log decay inside the chunk (tokens past the end: alpha = 1,
    // beta = 0, so they change nothing)
    const bool valid = t < T_len;
    const float la =
        valid ? __logf(fmaxf(alpha[static_cast<int64_t>(t) * H + h], 1e-30f)) : 0.f;
    const float bt = valid ? beta[static_cast<int64_t>(t) * H + h] : 0.f;
    float incl = la;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (li == 31) S.carry[ci] = incl;
    row_sync();
    if (li >= 32) incl += S.carry[ci];
    S.lg[i] = incl;
    S.beta[i] = bt;
    row_sync();
    const float lg_i = incl;
    bool ok = warp_wait(smem_u32(&S.g_full), 0, abort, status);
    if (ok) {
      tc_fence_after();
      // A row: (g_i / g_j) beta_j (k_i . k_j), j < i, this chunk's columns
      {
        uint32_t u[2][32];
        tmem_ld32(tmem + lane_base + cb, u[0]);
        tmem_ld32(tmem + lane_base + cb + 32, u[1]);
        tmem_ld_wait();
#pragma unroll
        for (int j4 = 0; j4 < kC; j4 += 4) {
          float4 a;
          float* av = reinterpret_cast<float*>(&a);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = j4 + e;
            av[e] = j < li ? __expf(lg_i - S.lg[cb + j]) * S.beta[cb + j] *
                                 __uint_as_float(u[j >> 5][j & 31])
                           : 0.f;
          }
          *reinterpret_cast<float4*>(&S.a[ci][li][j4]) = a;
        }
      }
      // P row: (g_i / g_j) beta_j (q_i . k_j), j <= i, as bf16
      {
        uint32_t u[2][32];
        tmem_ld32(tmem + lane_base + 128 + cb, u[0]);
        tmem_ld32(tmem + lane_base + 128 + cb + 32, u[1]);
        tmem_ld_wait();
        uint4* dst = reinterpret_cast<uint4*>(rec.p + (rc * kC + li) * kC);
#pragma unroll
        for (int j8 = 0; j8 < kC; j8 += 8) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float pv[2];
#pragma unroll
            for (int f = 0; f < 2; ++f) {
              const int j = j8 + 2 * e + f;
              pv[f] = j <= li ? __expf(lg_i - S.lg[cb + j]) * S.beta[cb + j] *
                                    __uint_as_float(u[j >> 5][j & 31])
                              : 0.f;
            }
            w[e] = pack_bf16x2(pv[0], pv[1]);
          }
          if (chunk_ok) dst[j8 / 8] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      // diag(g) Q and diag(beta g_C / g) K rows, from the staged tiles
      {
        const float g_i = __expf(lg_i);
        const float dk_i = bt * __expf(S.lg[cb + kC - 1] - lg_i);
        uint4* dq = reinterpret_cast<uint4*>(rec.qg + (rc * kC + li) * kD);
        uint4* dk = reinterpret_cast<uint4*>(rec.kp + (rc * kC + li) * kD);
#pragma unroll 4
        for (int c16 = 0; c16 < kD / 8; ++c16) {
          const uint32_t off = sw128_offset(i, c16 * 8, kHalf128);
          const uint4 qv = *reinterpret_cast<const uint4*>(S.q + off);
          const uint4 kv = *reinterpret_cast<const uint4*>(S.k + off);
          if (chunk_ok) {
            dq[c16] = make_uint4(scale_bf16x2(qv.x, g_i), scale_bf16x2(qv.y, g_i),
                                 scale_bf16x2(qv.z, g_i), scale_bf16x2(qv.w, g_i));
            dk[c16] = make_uint4(scale_bf16x2(kv.x, dk_i), scale_bf16x2(kv.y, dk_i),
                                 scale_bf16x2(kv.z, dk_i), scale_bf16x2(kv.w, dk_i));
          }
        }
        if (chunk_ok && li == kC - 1) rec.gc[rc] = __expf(lg_i);
      }
    }
    row_sync();  // every row of A is in shared memory
    // T = (I + A)^{-1}, column li of chunk ci, by forward substitution:
    // x_m = [m == li] - sum_{j < m} A_mj x_j (x_j = 0 for j < li)
    float x[kC];
#pragma unroll
    for (int m = 0; m < kC; ++m) x[m] = 0.f;
#pragma unroll
    for (int m = 0; m < kC; ++m) {
      float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
      for (int j4 = 0; j4 < m; j4 += 4) {  // A_mj = 0 and x_j = 0 for j >= m
        const float4 a = *reinterpret_cast<const float4*>(&S.a[ci][m][j4]);
        s0 = fmaf(a.x, x[j4], s0);
        s1 = fmaf(a.y, x[j4 + 1], s1);
        s2 = fmaf(a.z, x[j4 + 2], s2);
        s3 = fmaf(a.w, x[j4 + 3], s3);
      }
      x[m] = (m == li ? 1.f : 0.f) - ((s0 + s1) + (s2 + s3));
    }
    // T as bf16 (row m, column li), and -T diag(g) into the A_W tile
    {
      const float g_l = __expf(S.lg[cb + li]);
      __nv_bfloat16* tcol = rec.tinv + rc * kC * kC + li;
#pragma unroll
      for (int m = 0; m < kC; ++m) {
        if (chunk_ok) tcol[m * kC] = __float2bfloat16_rn(x[m]);
        *reinterpret_cast<__nv_bfloat16*>(S.aw + sw128_offset(cb + m, cb + li, kHalf128)) =
            __float2bfloat16_rn(-x[m] * g_l);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();  // the TMEM loads of G1 / G2 precede the W- MMA over them
    row_sync();
    if (threadIdx.x == 128) {
      tc_fence_after();
      mbar_arrive(smem_u32(&S.a_ready));
    }
    // W- rows
    ok = ok && warp_wait(smem_u32(&S.w_full), 0, abort, status);
    if (ok) {
      tc_fence_after();
      uint4* dst = reinterpret_cast<uint4*>(rec.wn + (rc * kC + li) * kD);
#pragma unroll
      for (int c32 = 0; c32 < kD; c32 += 32) {
        uint32_t u[32];
        tmem_ld32(tmem + lane_base + c32, u);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint4 w = make_uint4(
              pack_bf16x2(__uint_as_float(u[8 * e + 0]), __uint_as_float(u[8 * e + 1])),
              pack_bf16x2(__uint_as_float(u[8 * e + 2]), __uint_as_float(u[8 * e + 3])),
              pack_bf16x2(__uint_as_float(u[8 * e + 4]), __uint_as_float(u[8 * e + 5])),
              pack_bf16x2(__uint_as_float(u[8 * e + 6]), __uint_as_float(u[8 * e + 7])));
          if (chunk_ok) dst[c32 / 8 + e] = w;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// ================================================================== scan ==
struct ScanStage {
  uint8_t v[2 * kBox];   // V [64 tokens][128]: MN-major A of U^T (M = dv)
  uint8_t wn[2 * kBox];  // W- [64][128]: K-major B (N = tokens, K = dk)
  uint8_t qg[2 * kBox];  // diag(g) Q, same
  uint8_t kp[2 * kBox];  // diag(beta g_C / g) K: MN-major B (K = tokens, N = dk)
  uint8_t t[kBox];       // T [64][64]: K-major B (N = rows, K = columns)
  uint8_t p[kBox];       // P, same
};
constexpr uint32_t kStageBytes = 10 * kBox;  // 80 KB

struct ScanSmem {
  ScanStage st[2];
  uint8_t sb[kTile128];    // S as bf16 [128 rows r][128 k], K-major, 128-byte swizzle: A of S W-^T, S Qg^T
  uint8_t ub[kHalf128];    // U^T as bf16 [128 rows r][64 tokens], same: A of U^T K', U^T P^T
  uint8_t ost[2 * kBox];   // O of one chunk, [64 tokens][128 dv] as two 64-column boxes, for the TMA store
  uint64_t op_full[2], op_empty[2];
  uint64_t s_ready, u_full, u_ready, s_full, o_full[2], o_free[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// TMEM columns: D_U [0, 64), D_S' = U^T K' of the chunk [64, 192), D_O
// double-buffered at [192, 256) and [256, 320).
constexpr uint32_t kColU = 0, kColSp = 64, kColO = 192;

__global__ void __launch_bounds__(kThreads, 1)
    dn_scan_tc_kernel(const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_wn,
                      const __grid_constant__ CUtensorMap tm_qg,
                      const __grid_constant__ CUtensorMap tm_kp,
                      const __grid_constant__ CUtensorMap tm_t,
                      const __grid_constant__ CUtensorMap tm_p,
                      const __grid_constant__ CUtensorMap tm_o, int T_len, int H, int n_ch,
                      const float* __restrict__ gc, const float* __restrict__ S0,
                      float* __restrict__ S_out, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  ScanSmem& S = *reinterpret_cast<ScanSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = static_cast<int>(blockIdx.x);
  volatile int* abort = &S.abort;
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&S.op_full[s]), 1);
      mbar_init(smem_u32(&S.op_empty[s]), 1);
      mbar_init(smem_u32(&S.o_full[s]), 1);
      mbar_init(smem_u32(&S.o_free[s]), 4);
    }
    mbar_init(smem_u32(&S.s_ready), 4);
    mbar_init(smem_u32(&S.u_full), 1);
    mbar_init(smem_u32(&S.u_ready), 4);
    mbar_init(smem_u32(&S.s_full), 1);
    mbar_init(smem_u32(&S.drain), 1);
    S.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_wn);
    tma_prefetch_desc(&tm_qg);
    tma_prefetch_desc(&tm_kp);
    tma_prefetch_desc(&tm_t);
    tma_prefetch_desc(&tm_p);
    tma_prefetch_desc(&tm_o);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&S.tmem_base), 512);
    tmem_relinquish();
  }
  grid_dependency_wait();  // the prep kernel's records
  allow_dependents_launch();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------- TMA
      bool ok = true;
      int c = 0;
      for (; ok && c < n_ch; ++c) {
        const int s = c & 1;
        if (!(ok = mbar_wait(smem_u32(&S.op_empty[s]), ((c >> 1) & 1) ^ 1, abort, status))) break;
        const uint32_t bar = smem_u32(&S.op_full[s]);
        ScanStage& st = S.st[s];
        const int rrow = (c * H + h) * kC;
        mbar_arrive_expect_tx(bar, kStageBytes);
        for (int bx = 0; bx < 2; ++bx) {
          tma_load_2d(smem_u32(st.v) + bx * kBox, &tm_v, bar, h * kD + bx * 64, c * kC);
          tma_load_2d(smem_u32(st.wn) + bx * kBox, &tm_wn, bar, bx * 64, rrow);
          tma_load_2d(smem_u32(st.qg) + bx * kBox, &tm_qg, bar, bx * 64, rrow);
          tma_load_2d(smem_u32(st.kp) + bx * kBox, &tm_kp, bar, bx * 64, rrow);
        }
        tma_load_2d(smem_u32(st.t), &tm_t, bar, 0, rrow);
        tma_load_2d(smem_u32(st.p), &tm_p, bar, 0, rrow);
      }
      // drain the fills issued (bounded): the last fill of each stage
      for (int s = 0; s < 2 && s < c; ++s) {
        const int last = ((c - 1 - s) >> 1) & 1;
        mbar_wait_drain(smem_u32(&S.op_full[s]), last);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------- MMA
      // Every operand in shared memory.  Per chunk, in issue order:
      //   U^T = V^T T^T ; [S ready] U^T += S W-^T ; O^T = S Qg^T ;
      //   [U ready] S' = U^T K' ; O^T += U^T P^T
      // so O^T = S Qg^T runs while the row threads round U, and U^T P^T and
      // the next chunk's V^T T^T while they update S.
      constexpr uint32_t idesc_ut = idesc_bf16_f32(128, 64, 1, 0);   // V^T T^T
      constexpr uint32_t idesc_n64 = idesc_bf16_f32(128, 64, 0, 0);  // S W-^T, S Qg^T, U^T P^T
      constexpr uint32_t idesc_up = idesc_bf16_f32(128, 128, 0, 1);  // U^T K'
      const uint64_t vd0 = smem_desc_sw128(smem_u32(S.st[0].v), kBox, 1024);
      const uint64_t wd0 = smem_desc_sw128(smem_u32(S.st[0].wn), 16, 1024);
      const uint64_t qd0 = smem_desc_sw128(smem_u32(S.st[0].qg), 16, 1024);
      const uint64_t kd0 = smem_desc_sw128(smem_u32(S.st[0].kp), kBox, 1024);
      const uint64_t td0 = smem_desc_sw128(smem_u32(S.st[0].t), 16, 1024);
      const uint64_t pd0 = smem_desc_sw128(smem_u32(S.st[0].p), 16, 1024);
      const uint64_t sd = smem_desc_sw128(smem_u32(S.sb), 16, 1024);
      const uint64_t ud = smem_desc_sw128(smem_u32(S.ub), 16, 1024);
      const uint32_t d_u = tmem + kColU, d_s = tmem + kColSp;
      bool ok = true;
      for (int c = 0; ok && c < n_ch; ++c) {
        const int s = c & 1;
        const uint64_t so = static_cast<uint64_t>(s) * (kStageBytes >> 4);
        if (!(ok = mbar_wait(smem_u32(&S.op_full[s]), (c >> 1) & 1, abort, status))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_ss(d_u, vd0 + so + ((kk * 2048) >> 4), td0 + so + ((kk * 32) >> 4), idesc_ut,
                 kk > 0 ? 1u : 0u);
        if (!(ok = mbar_wait(smem_u32(&S.s_ready), c & 1, abort, status))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_ss(d_u, sd + (((kk >> 2) * kHalf128 + (kk & 3) * 32) >> 4),
                 wd0 + so + (((kk >> 2) * kBox + (kk & 3) * 32) >> 4), idesc_n64, 1u);
        mma_commit(smem_u32(&S.u_full));
        if (!(ok = mbar_wait(smem_u32(&S.o_free[s]), ((c >> 1) & 1) ^ 1, abort, status))) break;
        tc_fence_after();
        const uint32_t d_o = tmem + kColO + s * 64;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_ss(d_o, sd + (((kk >> 2) * kHalf128 + (kk & 3) * 32) >> 4),
                 qd0 + so + (((kk >> 2) * kBox + (kk & 3) * 32) >> 4), idesc_n64,
                 kk > 0 ? 1u : 0u);
        if (!(ok = mbar_wait(smem_u32(&S.u_ready), c & 1, abort, status))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_ss(d_s, ud + ((kk * 32) >> 4), kd0 + so + ((kk * 2048) >> 4), idesc_up,
                 kk > 0 ? 1u : 0u);
        mma_commit(smem_u32(&S.s_full));
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          mma_ss(d_o, ud + ((kk * 32) >> 4), pd0 + so + ((kk * 32) >> 4), idesc_n64, 1u);
        mma_commit(smem_u32(&S.o_full[s]));
        mma_commit(smem_u32(&S.op_empty[s]));
      }
      mma_commit(smem_u32(&S.drain));
      mbar_wait_drain(smem_u32(&S.drain), 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------- row threads
    // Thread r owns row r of the state (the dv index, and TMEM lane r) in
    // fp32 registers for the whole walk.
    const int r = threadIdx.x - 128;
    const uint32_t lb = static_cast<uint32_t>((warp - 4) * 32) << 16;
    float sv[kD];
    if (S0 != nullptr) {
      const float4* src = reinterpret_cast<const float4*>(S0 + (static_cast<int64_t>(h) * kD + r) * kD);
#pragma unroll
      for (int e = 0; e < kD / 4; ++e) {
        const float4 a = src[e];
        sv[4 * e] = a.x;
        sv[4 * e + 1] = a.y;
        sv[4 * e + 2] = a.z;
        sv[4 * e + 3] = a.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < kD; ++e) sv[e] = 0.f;
    }
    // S as bf16 into the swizzled A tile (row r), then hand it over
    auto put_state = [&]() {
#pragma unroll
      for (int c8 = 0; c8 < kD / 8; ++c8) {
        const uint4 w = make_uint4(pack_bf16x2(sv[8 * c8], sv[8 * c8 + 1]),
                                   pack_bf16x2(sv[8 * c8 + 2], sv[8 * c8 + 3]),
                                   pack_bf16x2(sv[8 * c8 + 4], sv[8 * c8 + 5]),
                                   pack_bf16x2(sv[8 * c8 + 6], sv[8 * c8 + 7]));
        *reinterpret_cast<uint4*>(S.sb + sw128_offset(r, 8 * c8, kHalf128)) = w;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&S.s_ready));
    };
    // O^T of chunk cc from TMEM (lane r: dv column r of each token) through
    // shared memory to global memory with one TMA store per 64 columns.  All
    // four row warps reach both named barriers whatever happened before (a
    // wait that gave up only skips the work), so none can be left waiting.
    auto read_out = [&](int cc, bool& ok) {
      const int b = cc & 1;
      if (r == 0) bulk_wait_read_all();  // the previous chunk's store has read the staging tile
      row_sync();
      if (ok) ok = warp_wait(smem_u32(&S.o_full[b]), (cc >> 1) & 1, abort, status);
      if (ok) {
        tc_fence_after();
        uint32_t u[2][32];
        tmem_ld32(tmem + lb + kColO + 64 * b, u[0]);
        tmem_ld32(tmem + lb + kColO + 64 * b + 32, u[1]);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&S.o_free[b]));
        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(S.ost + (r >> 6) * kBox) + (r & 63);
#pragma unroll
        for (int i = 0; i < kC; ++i)
          dst[i * 64] = __float2bfloat16_rn(__uint_as_float(u[i >> 5][i & 31]));
        fence_proxy_async_smem();
      }
      row_sync();
      if (r == 0 && *abort == 0) {
        tma_store_2d(&tm_o, smem_u32(S.ost), h * kD, cc * kC);
        tma_store_2d(&tm_o, smem_u32(S.ost) + kBox, h * kD + 64, cc * kC);
        bulk_commit();
      }
    };
    put_state();
    bool ok = true;
    for (int c = 0; c < n_ch; ++c) {
      const float g_c = gc[static_cast<int64_t>(c) * H + h];
      // U^T row r as bf16 into its A tile
      if (ok) ok = warp_wait(smem_u32(&S.u_full), c & 1, abort, status);
      if (ok) {
        tc_fence_after();
        uint32_t u[2][32];
        tmem_ld32(tmem + lb + kColU, u[0]);
        tmem_ld32(tmem + lb + kColU + 32, u[1]);
        tmem_ld_wait();
#pragma unroll
        for (int c8 = 0; c8 < kC / 8; ++c8) {
          const uint32_t* x = &u[c8 >> 2][(c8 & 3) * 8];
          const uint4 w = make_uint4(pack_bf16x2(__uint_as_float(x[0]), __uint_as_float(x[1])),
                                     pack_bf16x2(__uint_as_float(x[2]), __uint_as_float(x[3])),
                                     pack_bf16x2(__uint_as_float(x[4]), __uint_as_float(x[5])),
                                     pack_bf16x2(__uint_as_float(x[6]), __uint_as_float(x[7])));
          *reinterpret_cast<uint4*>(S.ub + sw128_offset(r, 8 * c8, kHalf128)) = w;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&S.u_ready));
      }
      // S <- g_C S + U^T K'
      if (ok) ok = warp_wait(smem_u32(&S.s_full), c & 1, abort, status);
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t d[32];
          tmem_ld32(tmem + lb + kColSp + 32 * q, d);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e)
            sv[32 * q + e] = fmaf(g_c, sv[32 * q + e], __uint_as_float(d[e]));
        }
        tc_fence_before();
        if (c + 1 < n_ch) put_state();
      }
      // this chunk's output, while the next chunk's products run
      read_out(c, ok);
    }
    if (r == 0) bulk_wait_all();
    if (ok && S_out != nullptr) {
      float4* dst = reinterpret_cast<float4*>(S_out + (static_cast<int64_t>(h) * kD + r) * kD);
#pragma unroll
      for (int e = 0; e < kD / 4; ++e)
        dst[e] = make_float4(sv[4 * e], sv[4 * e + 1], sv[4 * e + 2], sv[4 * e + 3]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

size_t deltanet_tc_workspace_bytes(int64_t T_len, int H) {
  const int64_t recs = (T_len + kC - 1) / kC * H;
  return static_cast<size_t>(recs) * (3 * kC * kD * 2 + 2 * kC * kC * 2 + 4);
}

cudaError_t launch_deltanet_tc(const void* q, const void* k, const void* v, const float* alpha,
                               const float* beta, int64_t T_len, int H, const float* S0, void* o,
                               float* S_out, void* workspace, cudaStream_t stream) {
  if (T_len == 0) return cudaSuccess;
  const int n_ch = static_cast<int>((T_len + kC - 1) / kC);
  const int64_t recs = static_cast<int64_t>(n_ch) * H;
  const DnRec rec = carve(workspace, recs);
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
  const uint64_t cols = static_cast<uint64_t>(H) * kD, rows = static_cast<uint64_t>(T_len);
  CUtensorMap tm_q, tm_k, tm_v, tm_o, tm_wn, tm_qg, tm_kp, tm_t, tm_p;
  bool good = make_tmap_2d(&tm_q, q, bf, 2, cols, rows, cols * 2, 64, 2 * kC, sw) &&
              make_tmap_2d(&tm_k, k, bf, 2, cols, rows, cols * 2, 64, 2 * kC, sw) &&
              make_tmap_2d(&tm_v, v, bf, 2, cols, rows, cols * 2, 64, kC, sw) &&
              make_tmap_2d(&tm_o, o, bf, 2, cols, rows, cols * 2, 64, kC,
                           CU_TENSOR_MAP_SWIZZLE_NONE);
  const uint64_t rr = static_cast<uint64_t>(recs) * kC;
  good = good && make_tmap_2d(&tm_wn, rec.wn, bf, 2, kD, rr, kD * 2, 64, kC, sw) &&
         make_tmap_2d(&tm_qg, rec.qg, bf, 2, kD, rr, kD * 2, 64, kC, sw) &&
         make_tmap_2d(&tm_kp, rec.kp, bf, 2, kD, rr, kD * 2, 64, kC, sw) &&
         make_tmap_2d(&tm_t, rec.tinv, bf, 2, kC, rr, kC * 2, 64, kC, sw) &&
         make_tmap_2d(&tm_p, rec.p, bf, 2, kC, rr, kC * 2, 64, kC, sw);
  if (!good) return cudaErrorInvalidValue;
  const size_t s1 = sizeof(PrepSmem) + 1024, s2 = sizeof(ScanSmem) + 1024;
  static_assert(sizeof(ScanSmem) + 1024 <= 232448, "scan shared memory over the 227 KB limit");
  cudaError_t err =
      cudaFuncSetAttribute(dn_prep_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(dn_scan_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)s2);
  if (err != cudaSuccess) return err;
  uint32_t* st = device_status_word();
  const int pairs = (n_ch + 1) / 2;
  err = launch_pdl(dn_prep_tc_kernel, dim3(pairs * H), dim3(kThreads), s1, stream, 1u, tm_q, tm_k,
                   alpha, beta, static_cast<int>(T_len), H, n_ch, rec, st);
  if (err != cudaSuccess) return err;
  err = launch_pdl(dn_scan_tc_kernel, dim3(H), dim3(kThreads), s2, stream, 1u, tm_v, tm_wn, tm_qg,
                   tm_kp, tm_t, tm_p, tm_o, static_cast<int>(T_len), H, n_ch,
                   static_cast<const float*>(rec.gc), S0, S_out, st);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace tg
