// Token-gated causal attention over the kept rows, bf16 in / fp32 softmax,
// on tcgen05 tensor cores (TokenGate pages: spke.com "TokenGate – Token-
// Gated Attention macht das Vollfüllen von langen Kontexten bis zu 11,3-mal
// schneller", section "Was ist token-gated Attention?": each kept token's
// gate score becomes a bias on the attention logits, with a learnable gain
// per head and a learnable temperature; ai4bro.com, section "กลไกการทำงาน
// ของ Learned Token Pruning"):
//
//   l_ij = t (q_i . k_j) / sqrt(128) + g_h ls_j   (j <= i),   o_i = softmax_j(l_ij) v_j
//
// Layout of one CTA (one 128-row query block, two q heads h0, h0+1 of one
// kv head, so every K/V tile is loaded once and used by both heads):
//   warp 0      TMA: Q tiles of both heads once, then K_j, V_j (128 x 128
//               bf16, 128-byte swizzle, 2-deep rings) and the bias inputs
//               ls_j (128 fp32) per key tile j of the CTA's key range.
//   warp 1      one thread issues tcgen05.mma: S_t = Q_t K_j^T into TMEM
//               (SS form), and O_t += P_t V_j with P_t read from TMEM (TS
//               form, V MN-major).
//   warp 2      writes each key tile's bias into one extra K = 16 block of
//               the Q K^T product (see below).
//   warps 4-7   softmax + epilogue of head h0 (t = 0), one query row per
//   warps 8-11  thread, likewise for head h1 (t = 1).
// The bias is added by the tensor core: Q_t gets two extra columns of ones
// and K_j two extra columns holding g_h ls_c sqrt(dh) / t split into bf16
// hi + lo, so S_t already holds q.k + g_h ls_c / scale and the softmax
// reads nothing but TMEM.  Measured on B300, this removes a shared-memory
// bias read and a barrier handshake from every softmax tile, which cost
// about 30% of the kernel's time, for 1/16 more MMA work.
// TMEM (512 columns): S_0 | S_1 | O_0 | O_1, 128 columns each; P_t (bf16
// pairs) overwrites the first 64 columns of S_t once S_t is in registers.
// The two heads ping-pong: while softmax t works, the tensor cores run
// head 1-t.  The running max is only raised when a row's max grows by more
// than 2^8 (log2 units), so O is rescaled in TMEM rarely; the final division
// by the row sum makes the result exact either way.  Causal tile skipping:
// query block b only visits key tiles 0..b; only tile b is masked.
//
// Work units (query block, kv head pair) are launched heaviest first.  When
// the kept sequence is short, the heaviest query blocks (the longest causal
// rows) run as single-head units instead: two CTAs per head pair, each doing
// one head.  Such a CTA has no second head to ping-pong with, so it does less
// work per cycle, but each key tile takes ~0.65 of a two-head tile, which
// shortens the critical path that sets the kernel time at small M.
#include <algorithm>

#include "tg_device.cuh"
#include "tg_internal.h"

namespace tg {
namespace {

constexpr int kBQ = 128;  // query rows per block
constexpr int kBK = 128;  // keys per tile
constexpr int kDH = 128;  // head dim
constexpr int kThreads = 384;
constexpr uint32_t kTileBytes = kBK * kDH * 2;  // 32 KB
constexpr uint32_t kHalfBytes = kTileBytes / 2;  // one 64-column TMA box
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
// The key bias rides in one extra K = 16 block of the Q K^T product: 128 rows
// x 16 bf16, K-major without swizzle (8-row x 16-byte core matrices, 128 B
// apart along K, 256 B apart along rows).
constexpr uint32_t kXBytes = kBK * 16 * 2;  // 4 KB
constexpr uint32_t kXLbo = 128, kXSbo = 256;
__host__ __device__ constexpr uint32_t xblock_offset(int row, int col) {
  return static_cast<uint32_t>((row >> 3) * 256 + (col >> 3) * 128 + (row & 7) * 16 + (col & 7) * 2);
}
struct AttnArgs {
  int M, Hq, Hkv, G;
  int n_rb, pairs_per_kv;
  int rb_single;     // query blocks >= this run as single-head units (two CTAs per head pair)
  int n_single;      // number of single-head units (launched first)
  float scale2;      // t / sqrt(dh) * log2(e), > 0
  float bias_scale;  // sqrt(dh) / t: the bias in units of the q.k product
  const float* gain;
  __nv_bfloat16* O;
  float* residual;
  float* lse;   // [Hq][M] natural-log row normalisers, or null
  int64_t ldo;  // Hq * dh
  uint32_t* status;
};

struct AttnSmem {
  uint8_t q[2][kTileBytes];
  uint8_t k[2][kTileBytes];
  uint8_t v[2][kTileBytes];
  uint8_t qx[2][kXBytes];  // per head t: ones in columns 2t, 2t+1
  uint8_t kx[2][kXBytes];  // per stage: g_h ls_j sqrt(dh) / t as bf16 hi + lo, per head
  float ls[2][kBK];
  uint64_t q_full;
  uint64_t k_full[2], k_empty[2];
  uint64_t v_full[2], v_empty[2];
  uint64_t ls_full[2], ls_empty[2];
  uint64_t bias_full[2];
  uint64_t s_full[2], p_full[2], o_done[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// One lane waits, the warp follows: keeps the .sync.aligned tcgen05 ops
// below warp-uniform even when a wait gives up.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          uint32_t* status) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort, status) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

// v as a pair of bf16 (hi, lo) packed low-first, hi = RN(v), lo = RN(v - hi);
// an infinite hi carries lo = 0.
__device__ __forceinline__ uint32_t split_bf16(float v) {
  const float hi = __bfloat162float(__float2bfloat16_rn(v));
  const float lo = isinf(hi) ? 0.f : v - hi;
  return pack_bf16x2(hi, lo);
}

// Writes 32 output columns [c0, c0 + 32) of one row: o = acc * inv, either
// as bf16 into O or added in fp32 into the residual stream.
__device__ __forceinline__ void store_out32(const AttnArgs& args, int64_t row, int h, int c0,
                                            const float (&o)[32], float inv) {
  if (args.residual != nullptr) {
    float4* dst = reinterpret_cast<float4*>(args.residual + row * args.ldo + h * kDH + c0);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float4 a = dst[i];
      a.x += o[4 * i + 0] * inv;
      a.y += o[4 * i + 1] * inv;
      a.z += o[4 * i + 2] * inv;
      a.w += o[4 * i + 3] * inv;
      dst[i] = a;
    }
  } else {
    uint4* dst = reinterpret_cast<uint4*>(args.O + row * args.ldo + h * kDH + c0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint4 w;
      w.x = pack_bf16x2(o[8 * i + 0] * inv, o[8 * i + 1] * inv);
      w.y = pack_bf16x2(o[8 * i + 2] * inv, o[8 * i + 3] * inv);
      w.z = pack_bf16x2(o[8 * i + 4] * inv, o[8 * i + 5] * inv);
      w.w = pack_bf16x2(o[8 * i + 6] * inv, o[8 * i + 7] * inv);
      dst[i] = w;
    }
  }
}

// Softmax and epilogue of one head (t = 0 for warps 4-7, t = 1 for warps
// 8-11): one query row per thread, over the CTA's key tiles [j0, j0 + nloc).
__device__ __forceinline__ void softmax_epilogue(AttnSmem& S, const AttnArgs& args, uint32_t tmem,
                                                 int rb, int j0, int nloc, int h0, int warp,
                                                 int lane, volatile int* abort) {
  const int t = (warp - 4) >> 2;
  const int quad = warp & 3;
  const int r = quad * 32 + lane;  // row within the block
  const int64_t row = static_cast<int64_t>(rb) * kBQ + r;
  const int h = h0 + t;
  const float sc = args.scale2;
  const uint64_t scale2 = f2(sc, sc);
  const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
  const uint32_t s_tmem = tmem + t * 128 + lane_off;
  const uint32_t o_tmem = tmem + 256 + t * 128 + lane_off;
  // running max m_run of x = S * scale2 (log2 units) and running sum l_run
  float m_run = -INFINITY, l_run = 0.f;
  bool ok = true;
  for (int i = 0; i < nloc; ++i) {
    const int j = j0 + i;
    if (!(ok = warp_wait(smem_u32(&S.s_full[t]), i & 1, abort, args.status))) break;
    tc_fence_after();
    // the whole S row (128 fp32) in registers: four loads, one wait
    uint32_t u[4][32];
#pragma unroll
    for (int c = 0; c < 4; ++c) tmem_ld32(s_tmem + 32 * c, u[c]);
    tmem_ld_wait();
    if (j == rb) {  // the diagonal tile: key c is row rb*128 + c
#pragma unroll
      for (int c = 0; c < kBK; ++c)
        if (c > r) u[c >> 5][c & 31] = __float_as_uint(-INFINITY);
    }
    // row max of S (scale2 > 0, so it is the max of x / scale2): four
    // independent chains of three-input maxima
    float mc[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      mc[k] = fmaxf(__uint_as_float(u[0][2 * k]), __uint_as_float(u[0][2 * k + 1]));
#pragma unroll
    for (int c = 8; c < kBK; c += 8) {
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
    // p = 2^(S scale2 - m_run): one FFMA per two columns, packed to bf16
    // pairs into the first 64 columns of S_t; the row sum in four
    // independent pair accumulators
    const uint64_t neg_m = f2(-m_run, -m_run);
    uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      uint32_t pk[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const int c = 64 * half + 2 * k;
        float d0, d1;
        f2_split(f2_fma(f2(__uint_as_float(u[c >> 5][c & 31]),
                           __uint_as_float(u[c >> 5][(c + 1) & 31])),
                        scale2, neg_m),
                 d0, d1);
        const float p0 = exp2_approx(d0), p1 = exp2_approx(d1);
        acc[k & 3] = f2_add(acc[k & 3], f2(p0, p1));
        pk[k] = pack_bf16x2(p0, p1);
      }
      tmem_st32(s_tmem + 32 * half, pk);
    }
    tmem_st_wait();
    float sum;
    {
      float a0, a1;
      f2_split(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), a0, a1);
      sum = a0 + a1;
    }
    // raise O to the new max; the P V of the previous tile is complete,
    // since s_full of this tile was committed after it
    if (__any_sync(0xffffffffu, need) && i > 0) {
      const float f = need ? exp2_approx(m_old - m_new) : 1.f;
      l_run *= f;
      uint32_t w[32];
#pragma unroll
      for (int c0 = 0; c0 < kDH; c0 += 32) {
        tmem_ld32(o_tmem + c0, w);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 32; ++k) w[k] = __float_as_uint(__uint_as_float(w[k]) * f);
        tmem_st32(o_tmem + c0, w);
      }
      tmem_st_wait();
    }
    l_run += sum;
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&S.p_full[t]));
  }
  // ------------------------------------------------------------ epilogue
  // own O complete (all of this head's MMAs are done)
  const bool have = ok && nloc > 0 &&
                    warp_wait(smem_u32(&S.o_done[t]), (nloc - 1) & 1, abort, args.status);
  if (have) tc_fence_after();
  if (!have) return;
  const bool row_ok = row < args.M;
  const float inv = 1.f / l_run;
  // log sum_j exp(l_ij) = (m_run + log2 l_run) ln 2, for a backward pass
  if (args.lse != nullptr && row_ok)
    args.lse[static_cast<int64_t>(h) * args.M + row] = (m_run + log2f(l_run)) * kLn2;
#pragma unroll 1
  for (int c0 = 0; c0 < kDH; c0 += 32) {
    uint32_t w[32];
    tmem_ld32(o_tmem + c0, w);
    tmem_ld_wait();
    float o[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) o[k] = __uint_as_float(w[k]);
    if (row_ok) store_out32(args, row, h, c0, o, inv);
  }
}

// MMA issue loop of one CTA: NH heads (1 or 2) is a compile-time constant so
// that the per-head descriptors stay in registers (a runtime head count made
// them dynamically indexed and slowed every MMA issue).
template <bool BIAS, int NH>
__device__ __forceinline__ void mma_loop(AttnSmem& S, const AttnArgs& args, uint32_t tmem,
                                         int nloc, const uint64_t (&qd)[2][kDH / 16],
                                         uint64_t kd0, const uint64_t (&qxd)[2], uint64_t kxd0,
                                         uint64_t vd0,
                                         volatile int* abort) {
  constexpr uint32_t idesc_s = idesc_bf16_f32(kBQ, kBK, 0, 0);  // Q K^T, both K-major
  constexpr uint32_t idesc_o = idesc_bf16_f32(kBQ, kDH, 0, 1);  // P V, V MN-major
  bool ok = mbar_wait(smem_u32(&S.q_full), 0, abort, args.status);
  tc_fence_after();
  for (int i = 0; ok && i <= nloc; ++i) {
    const int s = i & 1;
    if (i < nloc) {
      ok = mbar_wait(smem_u32(&S.k_full[s]), (i >> 1) & 1, abort, args.status);
      if (ok && BIAS)
        ok = mbar_wait(smem_u32(&S.bias_full[s]), (i >> 1) & 1, abort, args.status);
      if (!ok) break;
      tc_fence_after();
    }
#pragma unroll
    for (int t = 0; ok && t < NH; ++t) {
      if (i > 0) {
        const int ip = i - 1, sp = ip & 1;
        if (t == 0) {
          ok = mbar_wait(smem_u32(&S.v_full[sp]), (ip >> 1) & 1, abort, args.status);
          if (!ok) break;
        }
        ok = mbar_wait(smem_u32(&S.p_full[t]), ip & 1, abort, args.status);
        if (!ok) break;
        tc_fence_after();
        const uint32_t o_tmem = tmem + 256 + t * 128;
        const uint32_t p_tmem = tmem + t * 128;
        const uint64_t vd = vd0 + static_cast<uint64_t>(sp) * (kTileBytes >> 4);
        mma_ts(o_tmem, p_tmem, vd, idesc_o, ip > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 1; kk < kBK / 16; ++kk)
          mma_ts(o_tmem, p_tmem + kk * 8, vd + kk * (2048 >> 4), idesc_o, 1u);
        mma_commit(smem_u32(&S.o_done[t]));
        if (t == NH - 1) mma_commit(smem_u32(&S.v_empty[sp]));
      }
      if (i < nloc) {
        const uint64_t kd = kd0 + static_cast<uint64_t>(s) * (kTileBytes >> 4);
        const uint32_t s_tmem = tmem + t * 128;
#pragma unroll
        for (int kk = 0; kk < kDH / 16; ++kk)
          mma_ss(s_tmem, qd[t][kk],
                 kd + (((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4), idesc_s,
                 kk > 0 ? 1u : 0u);
        if (BIAS) mma_ss(s_tmem, qxd[t], kxd0 + static_cast<uint64_t>(s) * (kXBytes >> 4), idesc_s, 1u);
        mma_commit(smem_u32(&S.s_full[t]));
      }
    }
    if (ok && i < nloc) mma_commit(smem_u32(&S.k_empty[s]));
  }
}

template <bool BIAS>
__global__ void __launch_bounds__(kThreads, 1)
    keybias_attn_kernel(const __grid_constant__ CUtensorMap tm_qkv,
                        const __grid_constant__ CUtensorMap tm_ls, const AttnArgs args) {
  extern __shared__ uint8_t smem_raw[];
  AttnSmem& S = *reinterpret_cast<AttnSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &S.abort;

  // work unit: heaviest query blocks first
  const int unit = static_cast<int>(blockIdx.x);
  const int units_per_rb = args.Hkv * args.pairs_per_kv;
  int rb, h0, nh;  // query block, first q head, heads handled (1 or 2)
  int hk;
  if (unit < args.n_single) {
    const int per = 2 * units_per_rb;
    rb = args.n_rb - 1 - unit / per;
    const int rem = unit % per;
    hk = rem / (2 * args.pairs_per_kv);
    h0 = hk * args.G + (rem % (2 * args.pairs_per_kv));
    nh = 1;
  } else {
    const int u2 = unit - args.n_single;
    rb = args.rb_single - 1 - u2 / units_per_rb;
    const int rem = u2 % units_per_rb;
    hk = rem / args.pairs_per_kv;
    h0 = hk * args.G + 2 * (rem % args.pairs_per_kv);
    nh = 2;
  }
  const int nkv = rb + 1;
  const int j0 = 0, nloc = nkv;  // this CTA's key tiles [j0, j0 + nloc)

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&S.q_full), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&S.k_full[s]), 1);
      mbar_init(smem_u32(&S.k_empty[s]), 1);
      mbar_init(smem_u32(&S.v_full[s]), 1);
      mbar_init(smem_u32(&S.v_empty[s]), 1);
      mbar_init(smem_u32(&S.ls_full[s]), 1);
      mbar_init(smem_u32(&S.ls_empty[s]), 1);   // the bias warp
      mbar_init(smem_u32(&S.bias_full[s]), 1);  // the bias warp -> the MMA thread
      mbar_init(smem_u32(&S.s_full[s]), 1);
      mbar_init(smem_u32(&S.p_full[s]), 4);
      mbar_init(smem_u32(&S.o_done[s]), 1);
    }
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
  grid_dependency_wait();  // QKV and ls come from the previous kernels in the stream
  allow_dependents_launch();
  if (BIAS && (warp == 2 || warp == 3)) {
    // the extra K block: zeros, and for Q_t ones in the two bias columns of head t
    uint4* z = reinterpret_cast<uint4*>(S.qx[0]);
    for (int i = threadIdx.x - 64; i < static_cast<int>(4 * kXBytes / 16); i += 64)
      z[i] = make_uint4(0, 0, 0, 0);  // qx and kx are contiguous: 16 KB
    asm volatile("bar.sync 1, 64;" ::: "memory");
    for (int rr = threadIdx.x - 64; rr < kBQ; rr += 64) {
      *reinterpret_cast<uint32_t*>(S.qx[0] + xblock_offset(rr, 0)) = 0x3F803F80u;
      *reinterpret_cast<uint32_t*>(S.qx[1] + xblock_offset(rr, 2)) = 0x3F803F80u;
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  // Registers: launched at 168 per thread (384 x 168 = 64512).  The control
  // warpgroup (warps 0-3) gives back down to 152; the two softmax warpgroups,
  // which hold a whole S row, take up to 176: 128 x 152 + 256 x 176 = 64512.
  // (This split compiles with the fewest spills.)
  if (warp >= 4) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 176;" ::: "memory");
    if (warp < 4 + 4 * nh) softmax_epilogue(S, args, tmem, rb, j0, nloc, h0, warp, lane, abort);
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 152;" ::: "memory");
    if (warp == 0) {
      if (lane == 0 && nloc > 0) {
        // ----------------------------------------------------------- TMA
        const int kcol = (args.Hq + hk) * kDH;
        const int vcol = (args.Hq + args.Hkv + hk) * kDH;
        const uint64_t pol = l2_policy_evict_last();  // K/V tiles are re-read by later blocks
        mbar_arrive_expect_tx(smem_u32(&S.q_full), nh * kTileBytes);
        for (int t = 0; t < nh; ++t)
          for (int bx = 0; bx < 2; ++bx)
            tma_load_2d(smem_u32(S.q[t]) + bx * kHalfBytes, &tm_qkv, smem_u32(&S.q_full),
                        (h0 + t) * kDH + bx * 64, rb * kBQ);
        int nk = 0, nls = 0, nv = 0;  // fills issued per ring
        for (int i = 0; i < nloc; ++i) {
          const int j = j0 + i;
          const int s = i & 1;
          const uint32_t ph = (i >> 1) & 1;
          if (!mbar_wait(smem_u32(&S.k_empty[s]), ph ^ 1, abort, args.status)) break;
          mbar_arrive_expect_tx(smem_u32(&S.k_full[s]), kTileBytes);
          for (int bx = 0; bx < 2; ++bx)
            tma_load_2d_hint(smem_u32(S.k[s]) + bx * kHalfBytes, &tm_qkv, smem_u32(&S.k_full[s]),
                             kcol + bx * 64, j * kBK, pol);
          ++nk;
          if (BIAS) {
            if (!mbar_wait(smem_u32(&S.ls_empty[s]), ph ^ 1, abort, args.status)) break;
            mbar_arrive_expect_tx(smem_u32(&S.ls_full[s]), kBK * 4);
            tma_load_1d(smem_u32(S.ls[s]), &tm_ls, smem_u32(&S.ls_full[s]), j * kBK);
            ++nls;
          }
          if (!mbar_wait(smem_u32(&S.v_empty[s]), ph ^ 1, abort, args.status)) break;
          mbar_arrive_expect_tx(smem_u32(&S.v_full[s]), kTileBytes);
          for (int bx = 0; bx < 2; ++bx)
            tma_load_2d_hint(smem_u32(S.v[s]) + bx * kHalfBytes, &tm_qkv, smem_u32(&S.v_full[s]),
                             vcol + bx * 64, j * kBK, pol);
          ++nv;
        }
        // drain: every issued copy lands before the CTA may exit.  A fill that
        // was already consumed has completed its phase, so in the normal case
        // these waits return at once.
        mbar_wait_drain(smem_u32(&S.q_full), 0);
        for (int s = 0; s < 2; ++s) {
          if (s < nk) mbar_wait_drain(smem_u32(&S.k_full[s]), (((nk - 1 - s) >> 1) & 1));
          if (s < nls) mbar_wait_drain(smem_u32(&S.ls_full[s]), (((nls - 1 - s) >> 1) & 1));
          if (s < nv) mbar_wait_drain(smem_u32(&S.v_full[s]), (((nv - 1 - s) >> 1) & 1));
        }
      }
    } else if (warp == 1) {
      if (lane == 0 && nloc > 0) {
        // ----------------------------------------------------------- MMA
        // The issuing thread waits for the tensor pipe to take each MMA, so
        // every instruction between two MMAs idles the pipe: all shared-memory
        // descriptors are formed here, once.  A K step inside a tile is a
        // constant added to the start-address field (address >> 4; the sum
        // stays below 256 KB, so the field never carries).
        uint64_t qd[2][kDH / 16];
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int kk = 0; kk < kDH / 16; ++kk)
            qd[t][kk] = smem_desc_sw128(smem_u32(S.q[t]) + (kk >> 2) * kHalfBytes + (kk & 3) * 32,
                                        16, 1024);
        // stage 1 of each ring is a constant added to the start-address
        // field (address >> 4; the sum stays below 256 KB, so it never
        // carries): no runtime-indexed arrays, which would live in local memory
        const uint64_t kd0 = smem_desc_sw128(smem_u32(S.k[0]), 16, 1024);
        const uint64_t qxd[2] = {smem_desc_noswizzle(smem_u32(S.qx[0]), kXLbo, kXSbo),
                                 smem_desc_noswizzle(smem_u32(S.qx[1]), kXLbo, kXSbo)};
        const uint64_t kxd = smem_desc_noswizzle(smem_u32(S.kx[0]), kXLbo, kXSbo);
        const uint64_t vd0 = smem_desc_sw128(smem_u32(S.v[0]), kHalfBytes, 1024);
        if (nh == 2) {
          mma_loop<BIAS, 2>(S, args, tmem, nloc, qd, kd0, qxd, kxd, vd0, abort);
        } else {
          mma_loop<BIAS, 1>(S, args, tmem, nloc, qd, kd0, qxd, kxd, vd0, abort);
        }
        mma_commit(smem_u32(&S.drain));
        mbar_wait_drain(smem_u32(&S.drain), 0);
      }
    } else if (warp == 2) {
      if (BIAS) {
        // ------------------------------------------------------------ bias
        // Per key c of tile j and head t: v = g_t ls_c sqrt(dh) / t, split
        // into bf16 hi + lo (|v - hi - lo| <= 2^-17 |v|), written into
        // columns 2t, 2t+1 of the extra K block of stage s.  Q_t holds ones
        // there, so the Q K^T product carries g_t ls_c / scale exactly as
        // the softmax needs it.  Stage s is rewritten once the MMAs of the
        // tile two steps back that read it are complete (k_empty).
        const float f0 = args.gain[h0] * args.bias_scale;
        const float f1 = nh == 2 ? args.gain[h0 + 1] * args.bias_scale : 0.f;
        for (int i = 0; i < nloc; ++i) {
          const int s = i & 1;
          const uint32_t ph = (i >> 1) & 1;
          if (!warp_wait(smem_u32(&S.ls_full[s]), ph, abort, args.status)) break;
          if (!warp_wait(smem_u32(&S.k_empty[s]), ph ^ 1, abort, args.status)) break;
          const float4 l = reinterpret_cast<const float4*>(S.ls[s])[lane];
          const float lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int c = 4 * lane + k;
            uint2 w;
            w.x = split_bf16(f0 * lv[k]);
            w.y = split_bf16(f1 * lv[k]);
            *reinterpret_cast<uint2*>(S.kx[s] + xblock_offset(c, 0)) = w;
          }
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

cudaError_t launch_attn_bf16_2h(const void* QKV, int64_t M, int Hq, int Hkv, int dh,
                                const float* logsig, const float* gain, float temperature, void* O,
                                float* residual, float* lse, cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  AttnArgs a{};
  a.M = static_cast<int>(M);
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.G = Hq / Hkv;
  a.n_rb = static_cast<int>((M + kBQ - 1) / kBQ);
  a.pairs_per_kv = a.G / 2;
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
  const size_t smem = sizeof(AttnSmem) + 1024;
  // Single-head units for the heaviest query blocks when that shortens the
  // estimated makespan: a key tile costs 1 (two heads) or kSingle (one head),
  // query block b has b + 1 tiles, and the kernel takes at least its longest
  // unit and at least the total work spread over the SMs.  Only when the
  // two-head units fit in one wave: measured on B300 (M = 3251, 4000), with
  // more units than SMs the single-head units cost more than they save.
  a.rb_single = a.n_rb;
  a.n_single = 0;
  if (a.n_rb * Hkv * a.pairs_per_kv < sm_count()) {
    constexpr double kSingle = 0.75;  // measured flat optimum 0.6-0.85 at M = 1868
    const int upr = Hkv * a.pairs_per_kv;
    const int sms = sm_count();
    double best = 1e30;
    int best_rb = a.n_rb;
    for (int rs = a.n_rb; rs >= 0; --rs) {
      const int n1 = (a.n_rb - rs) * 2 * upr, n2 = rs * upr;
      if (n1 + n2 > 2 * sms) break;  // more than two waves: balance is not the issue
      double total = 0.0;
      for (int b = 0; b < a.n_rb; ++b)
        total += (b >= rs ? 2.0 * kSingle : 1.0) * (b + 1) * upr;
      const double longest = rs < a.n_rb ? kSingle * a.n_rb : static_cast<double>(a.n_rb);
      const double longest2 = rs > 0 ? static_cast<double>(rs) : 0.0;
      const double est = std::max(std::max(longest, longest2), total / sms);
      if (est < best - 1e-9) {
        best = est;
        best_rb = rs;
      }
    }
    a.rb_single = best_rb;
    a.n_single = (a.n_rb - best_rb) * 2 * upr;
  }
  const int grid = a.n_single + a.rb_single * Hkv * a.pairs_per_kv;
  auto kernel = logsig != nullptr ? keybias_attn_kernel<true> : keybias_attn_kernel<false>;
  cudaError_t err =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  err = launch_pdl(kernel, dim3(grid), dim3(kThreads), smem, stream, 1u, tm_qkv, tm_ls, a);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace tg
