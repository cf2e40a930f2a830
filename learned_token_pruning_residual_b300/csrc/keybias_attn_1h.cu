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
// walks its units; the next unit's Q loads once the current unit's last Q
// K^T is done and its K/V tiles stream in behind the current ones, so its
// first Q K^T runs during the current unit's epilogue.
//
// Per CTA (384 threads):
//   warp 0      TMA: Q of each unit, the K_j ring (3 stages) and V_j ring
//               (2 stages; 128 x 128 bf16, 128-byte swizzle; V one tile
//               behind K);
//   warp 1      one thread issues S_g = Q K_j^T (+ the bias block) into
//               S[g % 3] (SS form) as soon as K_j is in and P V of tile
//               g - 3 (which read P from that buffer) is done;
//   warp 3      one thread issues O += P_g V_j (TS form, P read from TMEM)
//               as soon as the softmax has written P_g.
//               The thread issuing tcgen05.mma waits for the tensor pipe to
//               take each one, and a barrier wait between two MMAs idles the
//               pipe for about 100 cycles (B300: the 17 MMAs of a tile take
//               1090 cycles back to back; one thread with five waits per
//               tile took 1750-2150).  With Q K^T and P V on two threads,
//               each thread's waits are covered by the other's MMAs.
//   warp 2      writes each key tile's bias into one extra K = 16 block of
//               the Q K^T product (g_h ls_j sqrt(dh) / t as bf16 hi + lo in
//               two columns; Q holds ones there), so S already carries it.
//   warps 4-7   softmax A: key columns 0..63 of every tile, one query row
//   warps 8-11  softmax B: key columns 64..127     per thread.
// The two halves of a row share one running max (each tile they swap their
// 64-column maxima through shared memory) and accumulate into one O; each
// keeps its own partial row sum, added in the epilogue.  The max is only
// raised when a row's max grows by more than 2^8 (log2 units); O is then
// rescaled in TMEM (each half its 64 columns of it) after the previous
// tile's P V has completed.  TMEM (512 columns): S_0 | S_1 | S_2 | O; each
// half writes its P over the first 32 of its 64 columns of S_g, so P V of
// tile g reads S_{g%3} and Q K^T of tile g + 3 waits for it.  With three S
// buffers Q K^T runs up to two tiles ahead of the softmax, and the softmax's
// only waits are for S (and, rarely, for O): each wait or arrive taken off
// its path shortens every tile (B300, M = 8432: 254 us with two S buffers and
// separate P buffers, 222 us this way).
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
// The K ring is 3 deep: a K fill waits for the Q K^T of the tile three
// back, so one fill's TMA latency (1.5-3k cycles with every SM loading) spans
// two tiles of work.  With 2 stages the fill of K_{g+2} only starts when Q
// K^T of tile g is done, and that latency set the tile rate.  Q is
// single-buffered to make room (the next unit's Q loads once the current
// unit's last Q K^T is done).
constexpr int kKStages = 3;
// TMEM columns: S_0 | S_1 | S_2 (128 fp32 each) | O (128 fp32).  Each
// half writes its P (64 keys as 32 columns of bf16 pairs) over the first 32
// of its own 64 columns of S_g once S_g is in its registers.
constexpr int kSBufs = 3;  // S ring in TMEM
constexpr uint32_t kOCol = kSBufs * 128;
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
  const float* logsig;  // per kept key, 16-byte aligned
  __nv_bfloat16* O;
  float* residual;
  float* lse;
  int64_t ldo;  // Hq * dh
  uint32_t* status;
};

struct Attn1hSmem {
  uint8_t q[kTileBytes];
  uint8_t k[kKStages][kTileBytes];
  uint8_t v[2][kTileBytes];
  // the epilogue's staging box for TMA stores: 128 rows x 128 bytes (64 bf16
  // or 32 fp32 output columns), 128-byte swizzle
  uint8_t ostage[kBQ * 128];
  uint8_t qx[kXBytes];     // ones in columns 0 and 1
  uint8_t kx[2][kXBytes];  // per tile parity: the key bias as bf16 hi, lo in columns 0 and 1
  float xm[2][2][kBQ];  // [half][tile parity][row]: each half's max of its 64 logits
  float ml[2][2][kBQ];  // [unit parity][half][row]: each half's running sum
  uint64_t q_full, q_empty;
  uint64_t k_full[kKStages], k_empty[kKStages];  // k_empty: that stage's Q K^T is done
  uint64_t bias_full[2];
  uint64_t v_full[2];
  // per TMEM buffer S_s (tile g in s = g % 3): s_full: Q K^T done;
  // p_full: both halves have written P over S_s; pv_done: P V done (S_s
  // free, O updated; also frees V stage g % 2)
  uint64_t s_full[kSBufs], p_full[kSBufs], pv_done[kSBufs];
  uint64_t o_done, o_free;
  uint64_t drain[2];
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

__device__ __forceinline__ void st_shared_v4(uint32_t addr, const uint32_t (&w)[4]) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]), "r"(w[1]),
               "r"(w[2]), "r"(w[3])
               : "memory");
}

// ls of keys key0 .. key0 + 3 (key0 a multiple of 4; 0 past the last key).
__device__ __forceinline__ float4 load_ls4(const float* ls, int M, int key0) {
  if (key0 + 3 < M) return __ldg(reinterpret_cast<const float4*>(ls + key0));
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  if (key0 < M) v.x = __ldg(ls + key0);
  if (key0 + 1 < M) v.y = __ldg(ls + key0 + 1);
  if (key0 + 2 < M) v.z = __ldg(ls + key0 + 2);
  return v;
}

__device__ __forceinline__ uint32_t split_bf16(float v) {
  const float hi = __bfloat162float(__float2bfloat16_rn(v));
  const float lo = isinf(hi) ? 0.f : v - hi;
  return pack_bf16x2(hi, lo);
}

// Softmax of one half (32 x 2 = 64 key columns of every tile) for one unit,
// then that half's share of the epilogue (64 of the 128 output columns).
// The two halves of a row share one running max: per tile each half takes
// the max of its 64 logits, the two threads of a row swap them through
// shared memory (one 64-thread named barrier per warp pair), and both take
// the same decision to raise it.  So both halves accumulate into one O.
__device__ __forceinline__ void softmax_unit(Attn1hSmem& S, const Attn1hArgs& args,
                                             const CUtensorMap& tm_out, uint32_t tmem, int rb,
                                             int h, uint32_t& g, int u_local, bool& ok, int warp,
                                             int lane, volatile int* abort) {
  const int half = (warp - 4) >> 2;
  const int quad = warp & 3;
  const int r = quad * 32 + lane;
  const int64_t row = static_cast<int64_t>(rb) * kBQ + r;
  const int col0 = half * 64;  // this half's key columns in a tile
  const float sc = args.scale2;
  const uint64_t scale2 = f2(sc, sc);
  const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
  const uint32_t o_mine = tmem + kOCol + half * 64 + lane_off;  // this half's 64 O columns
  const int nk = rb + 1;
  float m_run = -INFINITY, l_run = 0.f;
  for (int i = 0; i < nk; ++i, ++g) {
    const uint32_t st = g % kSBufs, ph = (g / kSBufs) & 1, xp = g & 1;
    // Every iteration reaches the pair barrier below, also after a wait gave
    // up (then with nothing to exchange), so that the other half never
    // waits on it in vain.
    const bool live = ok && (ok = warp_wait(smem_u32(&S.s_full[st]), ph, abort, args.status));
    uint32_t u[2][32];
    float mx = -INFINITY;
    if (live) {
      tc_fence_after();
      const uint32_t s_tmem = tmem + st * 128 + lane_off + col0;  // this half's S
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
      mx = fmax3(mc[0], mc[1], fmaxf(mc[2], mc[3])) * sc;
    }
    S.xm[half][xp][r] = mx;
    asm volatile("bar.sync %0, 64;" ::"r"(3 + quad) : "memory");  // warps 4 + quad, 8 + quad
    const float mx_other = S.xm[half ^ 1][xp][r];
    if (!live) continue;
    const float m_new = fmax3(m_run, mx, mx_other);
    const bool need = m_new > m_run + kRescaleThreshold;
    const float m_old = m_run;
    if (need) m_run = m_new;
    // a row with no visible key yet (all -inf) subtracts 0, so p = 0
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
    float sum;
    {
      float a0, a1;
      f2_split(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), a0, a1);
      sum = a0 + a1;
    }
    // P over the first 32 of this half's S columns (this tile's own buffer)
    tmem_st32(tmem + st * 128 + col0 + lane_off, pk);
    // raise O to the new max once the previous tile's P V is in
    if (__any_sync(0xffffffffu, need) && i > 0) {
      const uint32_t pg = g - 1;
      if (!(ok = warp_wait(smem_u32(&S.pv_done[pg % kSBufs]), (pg / kSBufs) & 1, abort,
                           args.status))) {
        tmem_st_wait();
        continue;
      }
      tc_fence_after();
      const float f = need ? exp2_approx(m_old - m_run) : 1.f;
      l_run *= f;
      uint32_t w[32];
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
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
    if (lane == 0) mbar_arrive(smem_u32(&S.p_full[st]));
  }
  // ------------------------------------------------------------ epilogue
  // O (this half's 64 columns of it) is read from TMEM into registers, then
  // written out through the shared staging box with TMA: a bf16 output in
  // two boxes of 64 columns (half A, then half B), an fp32 residual added
  // element-wise by TMA in four boxes of 32 columns.  Thread-per-row stores
  // straight from registers hit 32 rows per instruction and took ~2000
  // cycles per unit.  One thread (warp 4, lane 0) issues the copies and
  // waits for each to have read the box before it is refilled.
  const bool have = ok && warp_wait(smem_u32(&S.o_done), u_local & 1, abort, args.status);
  ok = have;
  if (have) tc_fence_after();
  S.ml[u_local & 1][half][r] = l_run;
  const bool issuer = warp == 4 && lane == 0;
  if (issuer) bulk_wait_read_all();  // the previous unit's last box is out of the staging buffer
  asm volatile("bar.sync 2, 256;" ::: "memory");  // both halves' sums of every row
  const bool res = args.residual != nullptr;
  float inv = 0.f;
  if (have) {
    const float l = S.ml[u_local & 1][0][r] + S.ml[u_local & 1][1][r];
    inv = 1.f / l;
    if (half == 0 && args.lse != nullptr && row < args.M)
      args.lse[static_cast<int64_t>(h) * args.M + row] = (m_run + log2f(l)) * kLn2;
  }
  const int npass = res ? 4 : 2;
  const uint32_t stage = smem_u32(S.ostage);
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    if (p == npass) break;
    if (p > 0) {
      if (issuer) bulk_wait_read_all();
      asm volatile("bar.sync 2, 256;" ::: "memory");  // the staging box is free
    }
    const int owner = res ? (p >> 1) : p;  // the half whose columns this box holds
    if (have && half == owner) {
      // row r's 128 bytes: 16-byte chunk c at chunk position c ^ (r & 7)
      const uint32_t row_base = stage + r * 128;
      if (res) {
        uint32_t a[32];
        tmem_ld32(o_mine + (p & 1) * 32, a);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t w[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) w[k] = __float_as_uint(__uint_as_float(a[4 * c + k]) * inv);
          st_shared_v4(row_base + ((c ^ (r & 7)) << 4), w);
        }
      } else {
#pragma unroll
        for (int hc = 0; hc < 2; ++hc) {
          uint32_t a[32];
          tmem_ld32(o_mine + hc * 32, a);
          tmem_ld_wait();
#pragma unroll
          for (int c = 4 * hc; c < 4 * hc + 4; ++c) {
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
              w[k] = pack_bf16x2(__uint_as_float(a[(8 * c + 2 * k) & 31]) * inv,
                                 __uint_as_float(a[(8 * c + 2 * k + 1) & 31]) * inv);
            st_shared_v4(row_base + ((c ^ (r & 7)) << 4), w);
          }
        }
      }
      if (!res || (p & 1)) {  // this half has read all of its O columns
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&S.o_free));  // O may be overwritten
      }
    }
    fence_proxy_async_smem();
    asm volatile("bar.sync 2, 256;" ::: "memory");  // the box is written
    if (issuer && have) {
      const int x = h * kDH + owner * 64 + (res ? (p & 1) * 32 : 0);
      if (res) tma_reduce_add_2d(&tm_out, stage, x, rb * kBQ);
      else tma_store_2d(&tm_out, stage, x, rb * kBQ);
      bulk_commit();
    }
  }
}

// Descriptors of buffer b of a double buffer are those of buffer 0 plus b
// times the buffer size in the start-address field (address >> 4; shared
// memory stays below 256 KB, so the 14-bit field never carries).  Forming
// them this way keeps every descriptor in registers (an array indexed by
// the stage would live in local memory and slow each MMA issue).
template <bool BIAS>
__device__ __forceinline__ void issue_qk(uint32_t tmem, uint32_t s, uint32_t ks, uint32_t xs,
                                         const uint64_t (&qd)[kDH / 16], uint64_t kd0,
                                         uint64_t qxd, uint64_t kxd0) {
  constexpr uint32_t idesc_s = idesc_bf16_f32(kBQ, kBK, 0, 0);
  const uint32_t s_tmem = tmem + s * 128;
  const uint64_t kd = kd0 + ks * (kTileBytes >> 4);
#pragma unroll
  for (int kk = 0; kk < kDH / 16; ++kk)
    mma_ss(s_tmem, qd[kk], kd + (((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4), idesc_s,
           kk > 0 ? 1u : 0u);
  if (BIAS) mma_ss(s_tmem, qxd, kxd0 + xs * (kXBytes >> 4), idesc_s, 1u);
}

// P V of tile t (unit-local index it): both halves' P (64 + 64 keys) into O.
__device__ __forceinline__ bool issue_pv(Attn1hSmem& S, const Attn1hArgs& args, uint32_t tmem,
                                         uint32_t t, int it, int u_local, uint64_t vd0,
                                         volatile int* abort) {
  constexpr uint32_t idesc_o = idesc_bf16_f32(kBQ, kDH, 0, 1);  // V MN-major
  const uint32_t st = t % kSBufs, ph = (t / kSBufs) & 1;
  const uint32_t vs = t & 1;  // V ring stage
  if (!mbar_wait_spin(smem_u32(&S.v_full[vs]), (t >> 1) & 1, abort, args.status)) return false;
  if (it == 0 && u_local > 0 &&
      !mbar_wait(smem_u32(&S.o_free), (u_local - 1) & 1, abort, args.status))
    return false;
  if (!mbar_wait(smem_u32(&S.p_full[st]), ph, abort, args.status)) return false;
  tc_fence_after();
  const uint64_t vd = vd0 + vs * (kTileBytes >> 4);
  const uint32_t p_tmem = tmem + st * 128;  // P_A in columns 0..31, P_B in 64..95
#pragma unroll
  for (int kk = 0; kk < kBK / 16; ++kk)
    mma_ts(tmem + kOCol, p_tmem + (kk >> 2) * 64 + (kk & 3) * 8, vd + kk * (2048 >> 4), idesc_o,
           (it > 0 || kk > 0) ? 1u : 0u);
  mma_commit(smem_u32(&S.pv_done[st]));
  return true;
}

template <bool BIAS>
__global__ void __launch_bounds__(kThreads, 1)
    keybias_attn_1h_kernel(const __grid_constant__ CUtensorMap tm_qkv,
                           const __grid_constant__ CUtensorMap tm_out, const Attn1hArgs args) {
  extern __shared__ uint8_t smem_raw[];
  Attn1hSmem& S = *reinterpret_cast<Attn1hSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                 ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = static_cast<int>(blockIdx.x);
  volatile int* abort = &S.abort;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&S.q_full), 1);
    mbar_init(smem_u32(&S.q_empty), 1);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(smem_u32(&S.k_full[s]), 1);
      mbar_init(smem_u32(&S.k_empty[s]), 1);
    }
    for (int s = 0; s < kSBufs; ++s) {
      mbar_init(smem_u32(&S.s_full[s]), 1);
      mbar_init(smem_u32(&S.p_full[s]), 8);
      mbar_init(smem_u32(&S.pv_done[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&S.bias_full[s]), 1);
      mbar_init(smem_u32(&S.v_full[s]), 1);
    }
    mbar_init(smem_u32(&S.o_done), 1);
    mbar_init(smem_u32(&S.o_free), 8);
    mbar_init(smem_u32(&S.drain[0]), 1);
    mbar_init(smem_u32(&S.drain[1]), 1);
    S.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_qkv);
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
      softmax_unit(S, args, tm_out, tmem, rb, h, g, k, ok, warp, lane, abort);
    }
    if (warp == 4 && lane == 0) bulk_wait_all();  // the last output box is in global memory
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 152;" ::: "memory");
    if (warp == 0 && lane == 0) {
      // ------------------------------------------------------------- TMA
      // Per tile g: K_g and ls_g, then V of the tile before (V_g is needed one
      // tile later than K_g, and its stage frees later, after the P V two
      // tiles back; issuing it one tile behind keeps that wait off the K
      // fills).
      const uint64_t pol = l2_policy_evict_last();  // K/V tiles are re-read by later units
      uint32_t g = 0, nv = 0, ks = 0, kph = 0;  // tiles, V fills, K-ring stage and phase
      int nq = 0, v_col = 0, v_row = 0;
      bool ok = true;
      auto fill_v = [&]() -> bool {  // V of tile nv
        const uint32_t s = nv & 1;
        if (nv >= 2) {  // V stage s is free once P V of tile nv - 2 is done
          const uint32_t pg = nv - 2;
          if (!mbar_wait(smem_u32(&S.pv_done[pg % kSBufs]), (pg / kSBufs) & 1, abort, args.status))
            return false;
        }
        mbar_arrive_expect_tx(smem_u32(&S.v_full[s]), kTileBytes);
        for (int bx = 0; bx < 2; ++bx)
          tma_load_2d_hint(smem_u32(S.v[s]) + bx * kHalfBytes, &tm_qkv, smem_u32(&S.v_full[s]),
                           v_col + bx * 64, v_row, pol);
        ++nv;
        return true;
      };
      for (int k = 0; ok; ++k) {
        const int j = unit_index(args, cta, k);
        if (j < 0) break;
        int rb, h;
        unit_of(args, j, rb, h);
        const int hk = h / args.G;
        // Q is free once the previous unit's last Q K^T is done
        if (!(ok = mbar_wait(smem_u32(&S.q_empty), (k & 1) ^ 1, abort, args.status))) break;
        mbar_arrive_expect_tx(smem_u32(&S.q_full), kTileBytes);
        for (int bx = 0; bx < 2; ++bx)
          tma_load_2d(smem_u32(S.q) + bx * kHalfBytes, &tm_qkv, smem_u32(&S.q_full),
                      h * kDH + bx * 64, rb * kBQ);
        ++nq;
        const int kcol = (args.Hq + hk) * kDH;
        for (int i = 0; i <= rb && ok; ++i, ++g) {
          // K_g's stage is free once Q K^T of tile g - 3 is done
          if (!(ok = mbar_wait(smem_u32(&S.k_empty[ks]), kph ^ 1, abort, args.status))) break;
          mbar_arrive_expect_tx(smem_u32(&S.k_full[ks]), kTileBytes);
          for (int bx = 0; bx < 2; ++bx)
            tma_load_2d_hint(smem_u32(S.k[ks]) + bx * kHalfBytes, &tm_qkv,
                             smem_u32(&S.k_full[ks]), kcol + bx * 64, i * kBK, pol);
          if (++ks == kKStages) ks = 0, kph ^= 1;
          if (g > 0 && !(ok = fill_v())) break;
          v_col = (args.Hq + args.Hkv + hk) * kDH;
          v_row = i * kBK;
        }
      }
      if (ok && nv < g) fill_v();  // the last tile's V
      // drain: every issued copy lands before the CTA may exit.  Each ring's
      // last fill per stage; fills already consumed return at once.  After a
      // wait gave up the counts may miss a fill, and a drain wait may give up
      // too (bounded).
      if (nq > 0) mbar_wait_drain(smem_u32(&S.q_full), (nq - 1) & 1);
      for (uint32_t s = 0; s < static_cast<uint32_t>(kKStages) && s < g; ++s) {
        const uint32_t last = ((g - 1 - s) / kKStages) & 1;
        mbar_wait_drain(smem_u32(&S.k_full[s]), last);
      }
      for (uint32_t s = 0; s < 2 && s < nv; ++s)
        mbar_wait_drain(smem_u32(&S.v_full[s]), ((nv - 1 - s) >> 1) & 1);
    } else if (warp == 1 && lane == 0) {
      // ------------------------------------------------------- MMA: Q K^T
      uint64_t qd[kDH / 16];
#pragma unroll
      for (int kk = 0; kk < kDH / 16; ++kk)
        qd[kk] = smem_desc_sw128(smem_u32(S.q) + (kk >> 2) * kHalfBytes + (kk & 3) * 32, 16,
                                 1024);
      const uint64_t kd0 = smem_desc_sw128(smem_u32(S.k[0]), 16, 1024);
      const uint64_t qxd = smem_desc_noswizzle(smem_u32(S.qx), kXLbo, kXSbo);
      const uint64_t kxd0 = smem_desc_noswizzle(smem_u32(S.kx[0]), kXLbo, kXSbo);
      uint32_t g = 0, ks = 0, kph = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int j = unit_index(args, cta, k);
        if (j < 0) break;
        int rb, h;
        unit_of(args, j, rb, h);
        if (!(ok = mbar_wait_spin(smem_u32(&S.q_full), k & 1, abort, args.status))) break;
        for (int i = 0; i <= rb; ++i, ++g) {
          const uint32_t s = g % kSBufs, ph = (g / kSBufs) & 1;  // S buffer
          const uint32_t xs = g & 1, xph = (g >> 1) & 1;           // bias block
          ok = mbar_wait_spin(smem_u32(&S.k_full[ks]), kph, abort, args.status);
          if (ok && BIAS) ok = mbar_wait(smem_u32(&S.bias_full[xs]), xph, abort, args.status);
          // S_s is free once P V of tile g - 3 (the P in it) is done
          if (ok) ok = mbar_wait(smem_u32(&S.pv_done[s]), ph ^ 1, abort, args.status);
          if (!ok) break;
          tc_fence_after();
          issue_qk<BIAS>(tmem, s, ks, xs, qd, kd0, qxd, kxd0);
          mma_commit(smem_u32(&S.s_full[s]));
          mma_commit(smem_u32(&S.k_empty[ks]));
          if (i == rb) mma_commit(smem_u32(&S.q_empty));
          if (++ks == kKStages) ks = 0, kph ^= 1;
        }
      }
      mma_commit(smem_u32(&S.drain[0]));
      mbar_wait_drain(smem_u32(&S.drain[0]), 0);
    } else if (warp == 3 && lane == 0) {
      // ---------------------------------------------------------- MMA: P V
      const uint64_t vd0 = smem_desc_sw128(smem_u32(S.v[0]), kHalfBytes, 1024);
      uint32_t g = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int j = unit_index(args, cta, k);
        if (j < 0) break;
        int rb, h;
        unit_of(args, j, rb, h);
        for (int i = 0; i <= rb; ++i, ++g)
          if (!(ok = issue_pv(S, args, tmem, g, i, k, vd0, abort))) break;
        if (!ok) break;
        mma_commit(smem_u32(&S.o_done));
      }
      mma_commit(smem_u32(&S.drain[1]));
      mbar_wait_drain(smem_u32(&S.drain[1]), 0);
    } else if (warp == 2 && BIAS) {
      // ------------------------------------------------------------ bias
      // The key tile's ls values are read straight from global memory (16
      // bytes per lane), one tile ahead: a 512-byte TMA fill queued behind
      // the 32 KB K and V fills took 1.5-3k cycles to land.
      uint32_t g = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int j = unit_index(args, cta, k);
        if (j < 0) break;
        int rb, h;
        unit_of(args, j, rb, h);
        const float f = args.gain[h] * args.bias_scale;
        float4 nxt = load_ls4(args.logsig, args.M, 4 * lane);
        for (int i = 0; i <= rb; ++i, ++g) {
          const uint32_t s = g & 1;
          const float4 l = nxt;
          if (i < rb) nxt = load_ls4(args.logsig, args.M, (i + 1) * kBK + 4 * lane);
          // kx[s] is free once Q K^T of tile g - 2 is done
          if (g >= 2) {
            const uint32_t pg = g - 2;
            if (!(ok = warp_wait(smem_u32(&S.s_full[pg % kSBufs]), (pg / kSBufs) & 1, abort,
                                 args.status)))
              break;
          }
          const float lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint32_t*>(S.kx[s] + xblock_offset(4 * lane + q, 0)) =
                split_bf16(f * lv[q]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&S.bias_full[s]));
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
  a.logsig = logsig;
  a.O = static_cast<__nv_bfloat16*>(O);
  a.residual = residual;
  a.lse = lse;
  a.ldo = static_cast<int64_t>(Hq) * dh;
  a.status = device_status_word();
  // the bias warp reads ls 16 bytes at a time
  if (logsig != nullptr && (reinterpret_cast<uintptr_t>(logsig) & 15) != 0)
    return cudaErrorInvalidValue;
  const int cols = (Hq + 2 * Hkv) * dh;
  CUtensorMap tm_qkv, tm_out;
  if (!make_tmap_2d(&tm_qkv, QKV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, cols, M,
                    static_cast<uint64_t>(cols) * 2, 64, kBQ, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  // the output: boxes of 128 rows x 128 bytes (64 bf16 columns of O, or 32
  // fp32 columns of the residual, which TMA adds into)
  const uint64_t ocols = static_cast<uint64_t>(Hq) * dh;
  const bool ok_out =
      residual != nullptr
          ? make_tmap_2d(&tm_out, residual, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ocols, M, ocols * 4,
                         32, kBQ, CU_TENSOR_MAP_SWIZZLE_128B)
          : make_tmap_2d(&tm_out, O, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ocols, M, ocols * 2, 64,
                         kBQ, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok_out) return cudaErrorInvalidValue;
  const size_t smem = sizeof(Attn1hSmem) + 1024;
  const int grid = std::min(a.n_units, sm_count());
  auto kernel = logsig != nullptr ? keybias_attn_1h_kernel<true> : keybias_attn_1h_kernel<false>;
  cudaError_t err =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  err = launch_pdl(kernel, dim3(grid), dim3(kThreads), smem, stream, 1u, tm_qkv, tm_out, a);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

// The one-head kernel reads each K/V tile once per q head, twice the bytes
// of the two-head kernel, so it runs while K and V together stay well inside
// L2 (48 MB).  There it is faster (B300, bias on: M = 1868: 19.8 against
// 31.7 us; 3507: 50.7 against 61.1; 6784: 151 against 181; 8432: 222
// against 255).  Beyond, HBM traffic decides (M = 131072, 512 MB of K and V:
// 65 against 57 ms) and the two-head kernel runs.
cudaError_t launch_attn_bf16(const void* QKV, int64_t M, int Hq, int Hkv, int dh,
                             const float* logsig, const float* gain, float temperature, void* O,
                             float* residual, float* lse, cudaStream_t stream) {
  const int64_t kv_bytes = 2 * M * Hkv * dh * 2;
  if (kv_bytes <= (int64_t{48} << 20))
    return launch_attn_bf16_1h(QKV, M, Hq, Hkv, dh, logsig, gain, temperature, O, residual, lse,
                               stream);
  return launch_attn_bf16_2h(QKV, M, Hq, Hkv, dh, logsig, gain, temperature, O, residual, lse,
                             stream);
}

}  // namespace tg
