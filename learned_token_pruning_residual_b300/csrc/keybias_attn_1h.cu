// Token-gated causal attention, one q head per work unit, persistent CTAs
// (TokenGate pages: spke.com "TokenGate – Token-Gated Attention macht das
// Vollfüllen von langen Kontexten bis zu 11,3-mal schneller", section "Was
// ist token-gated Attention?"; ai4bro.com, section "กลไกการทำงานของ Learned
// Token Pruning"):
//
//   l_ij = t (q_i . k_j) / sqrt(128) + g_h ls_j   (j <= i),   o_i = softmax_j(l_ij) v_j
//
// A work unit is (query block rb of 128 rows, q head h); it walks key tiles
// 0..rb.  Units are ordered heaviest first (rb descending, heads of a kv
// head adjacent so that their K/V tiles are shared through L2) and dealt to
// the CTAs in snake order (round k goes 0..G-1 when k is even, G-1..0 when
// odd), so the longest causal rows start first and the per-CTA sums of
// tiles stay within one unit of each other.  Each CTA stays resident and
// walks its units; the next unit's Q (double-buffered) and K/V tiles load
// while the current unit finishes, and its first Q K^T runs during the
// current unit's epilogue.
//
// Per CTA (384 threads):
//   warp 0      TMA: Q of each unit, the K_j ring (2 stages, 128 x 128
//               bf16, 128-byte swizzle) and the bias inputs ls_j;
//   warp 3      TMA: the V_j ring (its own thread, so that a V fill, which
//               waits for the P V two tiles back, never delays a K fill).
//   warp 1      one thread issues tcgen05.mma:
//                 S_g = Q K_j^T (+ the bias block) into S[g % 2] (SS form),
//                 O_A += P_A V_j[0:64), O_B += P_B V_j[64:128) (TS form,
//                 P read from TMEM).  Q K^T of tile g+1 is issued before
//                 P V of tile g, so it overlaps the softmax of tile g.
//   warp 2      writes each key tile's bias into one extra K = 16 block of
//               the Q K^T product (g_h ls_j sqrt(dh) / t as bf16 hi + lo in
//               two columns; Q holds ones there), so S already carries it.
//   warps 4-7   softmax A: key columns 0..63 of every tile, one query row
//   warps 8-11  softmax B: key columns 64..127     per thread.
// Each half keeps its own running max and sum and its own O accumulator
// (O_A, O_B), so the two halves never exchange anything per tile; the
// epilogue merges them once per unit:
//   o = (O_A 2^(m_A - m) + O_B 2^(m_B - m)) / (l_A 2^(m_A - m) + l_B 2^(m_B - m)).
// A half's running max is only raised when its max grows by more than 2^8
// (log2 units); O_A / O_B is then rescaled in TMEM, after the previous
// tile's P V has completed (pv_done).  TMEM (512 columns): S_0 | S_1 | O_A |
// O_B; P_A (bf16 pairs) overwrites S columns 0..31, P_B columns 64..95.
#include <algorithm>

#include "tg_device.cuh"
#include "tg_internal.h"

namespace tg {
namespace {

constexpr int kBQ = 128;
constexpr int kBK = 128;
constexpr int kDH = 128;
constexpr int kThreads = 384;
constexpr uint32_t kTileBytes = kBK * kDH * 2;   // 32 KB
constexpr uint32_t kHalfBytes = kTileBytes / 2;  // one 64-column TMA box
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
// the bias block: 128 rows x 16 bf16, K-major without swizzle (8-row x
// 16-byte core matrices, 128 B apart along K, 256 B apart along rows)
constexpr uint32_t kXBytes = kBK * 16 * 2;  // 4 KB
constexpr uint32_t kXLbo = 128, kXSbo = 256;
__host__ __device__ constexpr uint32_t xblock_offset(int row, int col) {
  return static_cast<uint32_t>((row >> 3) * 256 + (col >> 3) * 128 + (row & 7) * 16 +
                               (col & 7) * 2);
}

struct Attn1hArgs {
  int M, Hq, Hkv, G;
  int n_rb, n_units;
  float scale2;      // t / sqrt(dh) * log2(e), > 0
  float bias_scale;  // sqrt(dh) / t: the bias in units of the q.k product
  const float* gain;
  __nv_bfloat16* O;
  float* residual;
  float* lse;
  int64_t ldo;  // Hq * dh
  uint32_t* status;
};

struct Attn1hSmem {
  uint8_t q[2][kTileBytes];
  uint8_t k[2][kTileBytes];
  uint8_t v[2][kTileBytes];
  uint8_t qx[kXBytes];     // ones in columns 0 and 1
  uint8_t kx[2][kXBytes];  // per stage: the key bias as bf16 hi, lo in columns 0 and 1
  float ls[2][kBK];
  float ml[2][2][2][kBQ];  // [unit parity][half][max, sum][row]
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[2], k_empty[2];
  uint64_t v_full[2], v_empty[2];
  uint64_t ls_full[2], ls_empty[2];
  uint64_t bias_full[2];
  uint64_t s_full[2], pa_full[2], pb_full[2], pv_done[2];
  uint64_t o_done, o_free;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// The j-th unit in heaviest-first order: query block and q head.
__device__ __forceinline__ void unit_of(const Attn1hArgs& a, int j, int& rb, int& h) {
  rb = a.n_rb - 1 - j / a.Hq;
  h = j % a.Hq;
}

// The k-th unit of CTA c under the snake deal, or -1 past the end.
__device__ __forceinline__ int unit_index(const Attn1hArgs& a, int c, int k) {
  const int G = static_cast<int>(gridDim.x);
  const int j = k * G + ((k & 1) ? (G - 1 - c) : c);
  return j < a.n_units ? j : -1;
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          uint32_t* status) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort, status) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

__device__ __forceinline__ uint32_t split_bf16(float v) {
  const float hi = __bfloat162float(__float2bfloat16_rn(v));
  const float lo = isinf(hi) ? 0.f : v - hi;
  return pack_bf16x2(hi, lo);
}

// Softmax of one half (32 x 2 = 64 key columns of every tile) for one unit,
// then that half's share of the epilogue (64 of the 128 output columns).
__device__ __forceinline__ void softmax_unit(Attn1hSmem& S, const Attn1hArgs& args, uint32_t tmem,
                                             int rb, int h, uint32_t& g, int u_local, bool& ok,
                                             int warp, int lane, volatile int* abort) {
  const int half = (warp - 4) >> 2;
  const int quad = warp & 3;
  const int r = quad * 32 + lane;
  const int64_t row = static_cast<int64_t>(rb) * kBQ + r;
  const int col0 = half * 64;  // this half's key columns in a tile
  const float sc = args.scale2;
  const uint64_t scale2 = f2(sc, sc);
  const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
  const uint32_t o_mine = tmem + 256 + half * 128 + lane_off;
  const int nk = rb + 1;
  float m_run = -INFINITY, l_run = 0.f;
  for (int i = 0; i < nk; ++i, ++g) {
    if (!ok) continue;
    const uint32_t st = g & 1, ph = (g >> 1) & 1;
    if (!(ok = warp_wait(smem_u32(&S.s_full[st]), ph, abort, args.status))) continue;
    tc_fence_after();
    const uint32_t s_tmem = tmem + st * 128 + lane_off + col0;
    uint32_t u[2][32];
    tmem_ld32(s_tmem, u[0]);
    tmem_ld32(s_tmem + 32, u[1]);
    tmem_ld_wait();
    if (i == rb) {  // the diagonal tile: key col0 + c is row rb * 128 + col0 + c
#pragma unroll
      for (int c = 0; c < 64; ++c)
        if (col0 + c > r) u[c >> 5][c & 31] = __float_as_uint(-INFINITY);
    }
    float mc[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      mc[k] = fmaxf(__uint_as_float(u[0][2 * k]), __uint_as_float(u[0][2 * k + 1]));
#pragma unroll
    for (int c = 8; c < 64; c += 8) {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        mc[k] = fmax3(mc[k], __uint_as_float(u[c >> 5][(c + 2 * k) & 31]),
                      __uint_as_float(u[c >> 5][(c + 2 * k + 1) & 31]));
    }
    const float mx = fmax3(mc[0], mc[1], fmaxf(mc[2], mc[3])) * sc;
    const float m_new = fmaxf(m_run, mx);
    const bool need = m_new > m_run + kRescaleThreshold;
    const float m_old = m_run;
    if (need) m_run = m_new;
    // a half with no visible key yet (all -inf) subtracts 0, so p = 0
    const float m_sub = m_run == -INFINITY ? 0.f : m_run;
    const uint64_t neg_m = f2(-m_sub, -m_sub);
    uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
    uint32_t pk[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      const int c = 2 * k;
      float d0, d1;
      f2_split(f2_fma(f2(__uint_as_float(u[c >> 5][c & 31]),
                         __uint_as_float(u[c >> 5][(c + 1) & 31])),
                      scale2, neg_m),
               d0, d1);
      const float p0 = exp2_approx(d0), p1 = exp2_approx(d1);
      acc[k & 3] = f2_add(acc[k & 3], f2(p0, p1));
      pk[k] = pack_bf16x2(p0, p1);
    }
    tmem_st32(tmem + st * 128 + lane_off + col0, pk);  // P over this half's first 32 columns
    float sum;
    {
      float a0, a1;
      f2_split(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), a0, a1);
      sum = a0 + a1;
    }
    // raise this half's O to the new max once the previous tile's P V is in
    if (__any_sync(0xffffffffu, need) && i > 0) {
      const uint32_t pg = g - 1;
      if (!(ok = warp_wait(smem_u32(&S.pv_done[pg & 1]), (pg >> 1) & 1, abort, args.status))) {
        tmem_st_wait();
        continue;
      }
      tc_fence_after();
      const float f = need ? exp2_approx(m_old - m_run) : 1.f;
      l_run *= f;
      uint32_t w[32];
#pragma unroll
      for (int c0 = 0; c0 < kDH; c0 += 32) {
        tmem_ld32(o_mine + c0, w);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 32; ++k) w[k] = __float_as_uint(__uint_as_float(w[k]) * f);
        tmem_st32(o_mine + c0, w);
      }
    }
    tmem_st_wait();
    l_run += sum;
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(half == 0 ? &S.pa_full[st] : &S.pb_full[st]));
  }
  // ------------------------------------------------------------ epilogue
  const bool have = ok && warp_wait(smem_u32(&S.o_done), u_local & 1, abort, args.status);
  ok = have;
  if (have) tc_fence_after();
  float* ml = &S.ml[u_local & 1][0][0][0];
  ml[(half * 2 + 0) * kBQ + r] = m_run;
  ml[(half * 2 + 1) * kBQ + r] = l_run;
  asm volatile("bar.sync 2, 256;" ::: "memory");  // both halves' (max, sum) of every row
  if (have) {
    const float mA = ml[0 * kBQ + r], lA = ml[1 * kBQ + r];
    const float mB = ml[2 * kBQ + r], lB = ml[3 * kBQ + r];
    const float m = fmaxf(mA, mB);
    const float fA = mA == -INFINITY ? 0.f : exp2_approx(mA - m);
    const float fB = mB == -INFINITY ? 0.f : exp2_approx(mB - m);
    const float inv = 1.f / (lA * fA + lB * fB);
    const float cA = fA * inv, cB = fB * inv;
    const bool row_ok = row < args.M;
    if (half == 0 && args.lse != nullptr && row_ok)
      args.lse[static_cast<int64_t>(h) * args.M + row] = (m + log2f(lA * fA + lB * fB)) * kLn2;
    const uint32_t oa = tmem + 256 + lane_off, ob = tmem + 384 + lane_off;
#pragma unroll 1
    for (int c0 = half * 64; c0 < half * 64 + 64; c0 += 32) {
      uint32_t a[32], bv[32];
      tmem_ld32(oa + c0, a);
      tmem_ld32(ob + c0, bv);
      tmem_ld_wait();
      if (row_ok) {
        if (args.residual != nullptr) {
          float4* dst =
              reinterpret_cast<float4*>(args.residual + row * args.ldo + h * kDH + c0);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            float4 x = dst[q];
            x.x += __uint_as_float(a[4 * q + 0]) * cA + __uint_as_float(bv[4 * q + 0]) * cB;
            x.y += __uint_as_float(a[4 * q + 1]) * cA + __uint_as_float(bv[4 * q + 1]) * cB;
            x.z += __uint_as_float(a[4 * q + 2]) * cA + __uint_as_float(bv[4 * q + 2]) * cB;
            x.w += __uint_as_float(a[4 * q + 3]) * cA + __uint_as_float(bv[4 * q + 3]) * cB;
            dst[q] = x;
          }
        } else {
          uint4* dst = reinterpret_cast<uint4*>(args.O + row * args.ldo + h * kDH + c0);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float o[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
              o[k] = __uint_as_float(a[8 * q + k]) * cA + __uint_as_float(bv[8 * q + k]) * cB;
            uint4 w;
            w.x = pack_bf16x2(o[0], o[1]);
            w.y = pack_bf16x2(o[2], o[3]);
            w.z = pack_bf16x2(o[4], o[5]);
            w.w = pack_bf16x2(o[6], o[7]);
            dst[q] = w;
          }
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&S.o_free));  // O may be overwritten
  }
}

// Descriptors of buffer b of a double buffer are those of buffer 0 plus b
// times the buffer size in the start-address field (address >> 4; shared
// memory stays below 256 KB, so the 14-bit field never carries).  Forming
// them this way keeps every descriptor in registers (an array indexed by
// the stage would live in local memory and slow each MMA issue).
template <bool BIAS>
__device__ __forceinline__ void issue_qk(uint32_t tmem, uint32_t g, uint32_t qb,
                                         const uint64_t (&qd0)[kDH / 16], uint64_t kd0,
                                         uint64_t qxd, uint64_t kxd0) {
  constexpr uint32_t idesc_s = idesc_bf16_f32(kBQ, kBK, 0, 0);
  const uint32_t s = g & 1;
  const uint32_t s_tmem = tmem + s * 128;
  const uint64_t kd = kd0 + s * (kTileBytes >> 4);
  const uint64_t qoff = qb * (kTileBytes >> 4);
#pragma unroll
  for (int kk = 0; kk < kDH / 16; ++kk)
    mma_ss(s_tmem, qd0[kk] + qoff, kd + (((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4), idesc_s,
           kk > 0 ? 1u : 0u);
  if (BIAS) mma_ss(s_tmem, qxd, kxd0 + s * (kXBytes >> 4), idesc_s, 1u);
}

// P V of tile t (unit-local index it): both halves, into O_A and O_B.
__device__ __forceinline__ bool issue_pv(Attn1hSmem& S, const Attn1hArgs& args, uint32_t tmem,
                                         uint32_t t, int it, int u_local, uint64_t vd0,
                                         volatile int* abort) {
  constexpr uint32_t idesc_o = idesc_bf16_f32(kBQ, kDH, 0, 1);  // V MN-major
  const uint32_t st = t & 1, ph = (t >> 1) & 1;
  if (!mbar_wait(smem_u32(&S.v_full[st]), ph, abort, args.status)) return false;
  if (it == 0 && u_local > 0 &&
      !mbar_wait(smem_u32(&S.o_free), (u_local - 1) & 1, abort, args.status))
    return false;
  const uint64_t vd = vd0 + st * (kTileBytes >> 4);
  const uint32_t p_tmem = tmem + st * 128;
  if (!mbar_wait(smem_u32(&S.pa_full[st]), ph, abort, args.status)) return false;
  tc_fence_after();
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
    mma_ts(tmem + 256, p_tmem + kk * 8, vd + kk * (2048 >> 4), idesc_o,
           (it > 0 || kk > 0) ? 1u : 0u);
  if (!mbar_wait(smem_u32(&S.pb_full[st]), ph, abort, args.status)) return false;
  tc_fence_after();
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
    mma_ts(tmem + 384, p_tmem + 64 + kk * 8, vd + (4 + kk) * (2048 >> 4), idesc_o,
           (it > 0 || kk > 0) ? 1u : 0u);
  mma_commit(smem_u32(&S.pv_done[st]));
  mma_commit(smem_u32(&S.v_empty[st]));
  return true;
}

template <bool BIAS>
__global__ void __launch_bounds__(kThreads, 1)
    keybias_attn_1h_kernel(const __grid_constant__ CUtensorMap tm_qkv,
                           const __grid_constant__ CUtensorMap tm_ls, const Attn1hArgs args) {
  extern __shared__ uint8_t smem_raw[];
  Attn1hSmem& S = *reinterpret_cast<Attn1hSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                 ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = static_cast<int>(blockIdx.x);
  volatile int* abort = &S.abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&S.q_full[s]), 1);
      mbar_init(smem_u32(&S.q_empty[s]), 1);
      mbar_init(smem_u32(&S.k_full[s]), 1);
      mbar_init(smem_u32(&S.k_empty[s]), 1);
      mbar_init(smem_u32(&S.v_full[s]), 1);
      mbar_init(smem_u32(&S.v_empty[s]), 1);
      mbar_init(smem_u32(&S.ls_full[s]), 1);
      mbar_init(smem_u32(&S.ls_empty[s]), 1);
      mbar_init(smem_u32(&S.bias_full[s]), 1);
      mbar_init(smem_u32(&S.s_full[s]), 1);
      mbar_init(smem_u32(&S.pa_full[s]), 4);
      mbar_init(smem_u32(&S.pb_full[s]), 4);
      mbar_init(smem_u32(&S.pv_done[s]), 1);
    }
    mbar_init(smem_u32(&S.o_done), 1);
    mbar_init(smem_u32(&S.o_free), 8);
    mbar_init(smem_u32(&S.drain), 1);
    S.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_qkv);
    if (BIAS) tma_prefetch_desc(&tm_ls);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&S.tmem_base), 512);
    tmem_relinquish();
  }
  if (BIAS && (warp == 2 || warp == 3)) {
    // the extra K block: zeros, then ones in the bias columns of Q
    uint4* z = reinterpret_cast<uint4*>(S.qx);
    for (int i = threadIdx.x - 64; i < static_cast<int>(3 * kXBytes / 16); i += 64)
      z[i] = make_uint4(0, 0, 0, 0);  // qx and kx are contiguous: 12 KB
    asm volatile("bar.sync 1, 64;" ::: "memory");
    for (int rr = threadIdx.x - 64; rr < kBQ; rr += 64)
      *reinterpret_cast<uint32_t*>(S.qx + xblock_offset(rr, 0)) = 0x3F803F80u;
    fence_proxy_async_smem();
  }
  grid_dependency_wait();  // QKV and ls come from the previous kernels in the stream
  allow_dependents_launch();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  // Registers: launched at 168 per thread (384 x 168 = 64512); the control
  // warpgroup gives back down to 152, the softmax warpgroups take 176:
  // 128 x 152 + 256 x 176 = 64512.
  if (warp >= 4) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 176;" ::: "memory");
    uint32_t g = 0;
    bool ok = true;
    for (int k = 0;; ++k) {
      const int j = unit_index(args, cta, k);
      if (j < 0) break;
      int rb, h;
      unit_of(args, j, rb, h);
      softmax_unit(S, args, tmem, rb, h, g, k, ok, warp, lane, abort);
    }
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 152;" ::: "memory");
    if (warp == 0 && lane == 0) {
      // ------------------------------------------------------------- TMA
      const uint64_t pol = l2_policy_evict_last();  // K/V tiles are re-read by later units
      uint32_t g = 0;
      int nq = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int j = unit_index(args, cta, k);
        if (j < 0) break;
        int rb, h;
        unit_of(args, j, rb, h);
        const int hk = h / args.G;
        const uint32_t qb = k & 1;
        if (!(ok = mbar_wait(smem_u32(&S.q_empty[qb]), ((k >> 1) & 1) ^ 1, abort, args.status)))
          break;
        mbar_arrive_expect_tx(smem_u32(&S.q_full[qb]), kTileBytes);
        for (int bx = 0; bx < 2; ++bx)
          tma_load_2d(smem_u32(S.q[qb]) + bx * kHalfBytes, &tm_qkv, smem_u32(&S.q_full[qb]),
                      h * kDH + bx * 64, rb * kBQ);
        ++nq;
        const int kcol = (args.Hq + hk) * kDH;
        for (int i = 0; i <= rb && ok; ++i, ++g) {
          const uint32_t s = g & 1, ph = (g >> 1) & 1;
          if (!(ok = mbar_wait(smem_u32(&S.k_empty[s]), ph ^ 1, abort, args.status))) break;
          mbar_arrive_expect_tx(smem_u32(&S.k_full[s]), kTileBytes);
          for (int bx = 0; bx < 2; ++bx)
            tma_load_2d_hint(smem_u32(S.k[s]) + bx * kHalfBytes, &tm_qkv, smem_u32(&S.k_full[s]),
                             kcol + bx * 64, i * kBK, pol);
          if (BIAS) {
            if (!(ok = mbar_wait(smem_u32(&S.ls_empty[s]), ph ^ 1, abort, args.status))) break;
            mbar_arrive_expect_tx(smem_u32(&S.ls_full[s]), kBK * 4);
            tma_load_1d(smem_u32(S.ls[s]), &tm_ls, smem_u32(&S.ls_full[s]), i * kBK);
          }
        }
      }
      // drain: every issued copy lands before the CTA may exit.  Each ring's
      // last fill per stage; fills already consumed return at once.  The
      // count g includes a fill whose wait gave up, so on that path a drain
      // wait may give up too (bounded).
      for (uint32_t s = 0; s < 2; ++s) {
        if (static_cast<int>(s) < nq)
          mbar_wait_drain(smem_u32(&S.q_full[s]), ((nq - 1 - s) >> 1) & 1);
        if (s < g) {
          const uint32_t last = ((g - 1 - s) >> 1) & 1;
          mbar_wait_drain(smem_u32(&S.k_full[s]), last);
          if (BIAS) mbar_wait_drain(smem_u32(&S.ls_full[s]), last);
        }
      }
    } else if (warp == 3 && lane == 0) {
      // ------------------------------------------------------------ TMA, V
      // V has a producer of its own: a V fill waits for the P V two tiles
      // back, and must not hold up the K fills behind it.
      const uint64_t pol = l2_policy_evict_last();
      uint32_t g = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int j = unit_index(args, cta, k);
        if (j < 0) break;
        int rb, h;
        unit_of(args, j, rb, h);
        const int vcol = (args.Hq + args.Hkv + h / args.G) * kDH;
        for (int i = 0; i <= rb; ++i, ++g) {
          const uint32_t s = g & 1, ph = (g >> 1) & 1;
          if (!(ok = mbar_wait(smem_u32(&S.v_empty[s]), ph ^ 1, abort, args.status))) break;
          mbar_arrive_expect_tx(smem_u32(&S.v_full[s]), kTileBytes);
          for (int bx = 0; bx < 2; ++bx)
            tma_load_2d_hint(smem_u32(S.v[s]) + bx * kHalfBytes, &tm_qkv, smem_u32(&S.v_full[s]),
                             vcol + bx * 64, i * kBK, pol);
        }
      }
      for (uint32_t s = 0; s < 2 && s < g; ++s)
        mbar_wait_drain(smem_u32(&S.v_full[s]), ((g - 1 - s) >> 1) & 1);
    } else if (warp == 1 && lane == 0) {
      // ------------------------------------------------------------- MMA
      uint64_t qd0[kDH / 16];
#pragma unroll
      for (int kk = 0; kk < kDH / 16; ++kk)
        qd0[kk] = smem_desc_sw128(smem_u32(S.q[0]) + (kk >> 2) * kHalfBytes + (kk & 3) * 32, 16,
                                  1024);
      const uint64_t kd0 = smem_desc_sw128(smem_u32(S.k[0]), 16, 1024);
      const uint64_t qxd = smem_desc_noswizzle(smem_u32(S.qx), kXLbo, kXSbo);
      const uint64_t kxd0 = smem_desc_noswizzle(smem_u32(S.kx[0]), kXLbo, kXSbo);
      const uint64_t vd0 = smem_desc_sw128(smem_u32(S.v[0]), kHalfBytes, 1024);
      uint32_t g = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int j = unit_index(args, cta, k);
        if (j < 0) break;
        int rb, h;
        unit_of(args, j, rb, h);
        const uint32_t qb = k & 1;
        if (!(ok = mbar_wait(smem_u32(&S.q_full[qb]), (k >> 1) & 1, abort, args.status))) break;
        tc_fence_after();
        for (int i = 0; i <= rb; ++i, ++g) {
          const uint32_t s = g & 1, ph = (g >> 1) & 1;
          ok = mbar_wait(smem_u32(&S.k_full[s]), ph, abort, args.status);
          if (ok && BIAS) ok = mbar_wait(smem_u32(&S.bias_full[s]), ph, abort, args.status);
          if (!ok) break;
          tc_fence_after();
          issue_qk<BIAS>(tmem, g, qb, qd0, kd0, qxd, kxd0);
          mma_commit(smem_u32(&S.s_full[s]));
          mma_commit(smem_u32(&S.k_empty[s]));
          if (i == rb) mma_commit(smem_u32(&S.q_empty[qb]));
          if (i > 0 && !(ok = issue_pv(S, args, tmem, g - 1, i - 1, k, vd0, abort))) break;
        }
        if (!ok) break;
        if (!(ok = issue_pv(S, args, tmem, g - 1, rb, k, vd0, abort))) break;
        mma_commit(smem_u32(&S.o_done));
      }
      mma_commit(smem_u32(&S.drain));
      mbar_wait_drain(smem_u32(&S.drain), 0);
    } else if (warp == 2 && BIAS) {
      // ------------------------------------------------------------ bias
      uint32_t g = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int j = unit_index(args, cta, k);
        if (j < 0) break;
        int rb, h;
        unit_of(args, j, rb, h);
        const float f = args.gain[h] * args.bias_scale;
        for (int i = 0; i <= rb; ++i, ++g) {
          const uint32_t s = g & 1, ph = (g >> 1) & 1;
          if (!(ok = warp_wait(smem_u32(&S.ls_full[s]), ph, abort, args.status))) break;
          if (!(ok = warp_wait(smem_u32(&S.k_empty[s]), ph ^ 1, abort, args.status))) break;
          const float4 l = reinterpret_cast<const float4*>(S.ls[s])[lane];
          const float lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint32_t*>(S.kx[s] + xblock_offset(4 * lane + q, 0)) =
                split_bf16(f * lv[q]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(smem_u32(&S.ls_empty[s]));
            mbar_arrive(smem_u32(&S.bias_full[s]));
          }
        }
      }
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

cudaError_t launch_attn_bf16_1h(const void* QKV, int64_t M, int Hq, int Hkv, int dh,
                                const float* logsig, const float* gain, float temperature, void* O,
                                float* residual, float* lse, cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  Attn1hArgs a{};
  a.M = static_cast<int>(M);
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.G = Hq / Hkv;
  a.n_rb = static_cast<int>((M + kBQ - 1) / kBQ);
  a.n_units = a.n_rb * Hq;
  a.scale2 = temperature / sqrtf(static_cast<float>(dh)) * kLog2e;
  a.bias_scale = sqrtf(static_cast<float>(dh)) / temperature;
  a.gain = gain;
  a.O = static_cast<__nv_bfloat16*>(O);
  a.residual = residual;
  a.lse = lse;
  a.ldo = static_cast<int64_t>(Hq) * dh;
  a.status = device_status_word();
  const int cols = (Hq + 2 * Hkv) * dh;
  CUtensorMap tm_qkv, tm_ls;
  if (!make_tmap_2d(&tm_qkv, QKV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, cols, M,
                    static_cast<uint64_t>(cols) * 2, 64, kBQ, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (logsig != nullptr) {
    if (!make_tmap_1d_f32(&tm_ls, logsig, M, kBK)) return cudaErrorInvalidValue;
  } else {
    tm_ls = tm_qkv;  // unused
  }
  const size_t smem = sizeof(Attn1hSmem) + 1024;
  const int grid = std::min(a.n_units, sm_count());
  auto kernel = logsig != nullptr ? keybias_attn_1h_kernel<true> : keybias_attn_1h_kernel<false>;
  cudaError_t err =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  err = launch_pdl(kernel, dim3(grid), dim3(kThreads), smem, stream, 1u, tm_qkv, tm_ls, a);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

// Short kept sequences (the two-head units fit in one wave of the SMs) are
// set by their longest causal row: there the one-head units, whose key tiles
// take about half as long, win (B300, M = 1868: 25 against 31.5 us).  Longer
// ones are set by throughput, where a one-head CTA has to stream twice the
// K/V bytes per MMA cycle through a 2-stage ring and waits on its loads
// (M = 3507: 71.5 against 63.5 us; M = 8432: 304 against 256 us): there the
// two-head kernel runs.
cudaError_t launch_attn_bf16(const void* QKV, int64_t M, int Hq, int Hkv, int dh,
                             const float* logsig, const float* gain, float temperature, void* O,
                             float* residual, float* lse, cudaStream_t stream) {
  const int64_t n_rb = (M + kBQ - 1) / kBQ;
  const int64_t two_head_units = n_rb * Hkv * ((Hq / Hkv) / 2);
  if (two_head_units < static_cast<int64_t>(sm_count()))
    return launch_attn_bf16_1h(QKV, M, Hq, Hkv, dh, logsig, gain, temperature, O, residual, lse,
                               stream);
  return launch_attn_bf16_2h(QKV, M, Hq, Hkv, dh, logsig, gain, temperature, O, residual, lse,
                             stream);
}

}  // namespace tg
