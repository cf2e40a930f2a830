// The gradient that token-gated attention carries back to the scorer
// (TokenGate pages: spke.com "TokenGate – Token-Gated Attention macht das
// Vollfüllen von langen Kontexten bis zu 11,3-mal schneller", section "Was
// ist token-gated Attention?": the kept tokens' scores become a bias on the
// attention logits, which gives the gradient a way back to the scorer;
// ai4bro.com, section "กลไกการทำงานของ Learned Token Pruning", the same
// MoE-router device).
//
// With b_hj = g_h ls_j the bias of kept key j in q head h and
// l_ij = t (q_i . k_j) / sqrt(dh) + b_hj (j <= i), an upstream gradient dO
// of the attention output gives, by the chain rule through the softmax,
//   dL/db_hj = sum_{i >= j} P_ij (dO_i . v_j - D_i),   D_i = dO_i . o_i,
// and from it dL/dls_j = sum_h g_h dL/db_hj, dL/dg_h = sum_j ls_j dL/db_hj,
// dL/ds_j = dL/dls_j sigmoid(-s_j).  P_ij = exp(l_ij - lse_i) is recomputed
// from the forward's per-row log-sum-exp.
//
// Kernels:
//   attn_delta_kernel        D[h][i] = dO_i . o_i per head (HBM-bound).
//   keybias_bias_grad_kernel dL/db (bf16, dh = 128) on tcgen05.  One CTA per
//       (q head, block of 128 keys): the keys sit on the 128 TMEM lanes, so
//       the sum over queries is a sum along one thread's registers.  Per
//       query tile i it runs S^T = K Q_i^T and dP^T = V dO_i^T (two SS MMAs
//       of 128 x 128 x 128, both operands K-major), then each thread adds
//       p (dp - D_i) over the tile's 128 queries.  K and V stay in shared
//       memory; Q_i and dO_i stream through a 2-stage TMA ring; the two
//       accumulator pairs in TMEM (512 columns) alternate between tiles, and
//       two epilogue warpgroups take alternate tiles.
//   bias_grad_f32_kernel     the same sum on CUDA cores for fp32 inputs.
//   bias_grad_reduce_kernel  dL/dls, dL/ds and dL/dg from dL/db, in a fixed
//       summation order (deterministic).
#include "tg_device.cuh"
#include "tg_internal.h"

namespace tg {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------------ delta
// One thread per 16-byte chunk of a row; the `cph` chunks of one head are
// consecutive lanes and reduce with shuffles.
template <typename T>
__global__ void __launch_bounds__(256)
    attn_delta_kernel(const T* __restrict__ dO, const T* __restrict__ Oa, int M, int Hq,
                      int cph, float* __restrict__ delta) {
  grid_dependency_wait();
  allow_dependents_launch();
  const int C = Hq * cph;  // chunks per row
  const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t total = static_cast<int64_t>(M) * C;
  float s = 0.f;
  int row = 0, chunk = 0;
  if (g < total) {
    row = static_cast<int>(g / C);
    chunk = static_cast<int>(g - static_cast<int64_t>(row) * C);
    const uint4 a = reinterpret_cast<const uint4*>(dO)[g];
    const uint4 b = reinterpret_cast<const uint4*>(Oa)[g];
    if constexpr (sizeof(T) == 2) {
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        s = fmaf(bf16lo_to_f32(aw[k]), bf16lo_to_f32(bw[k]), s);
        s = fmaf(bf16hi_to_f32(aw[k]), bf16hi_to_f32(bw[k]), s);
      }
    } else {
      s = __uint_as_float(a.x) * __uint_as_float(b.x);
      s = fmaf(__uint_as_float(a.y), __uint_as_float(b.y), s);
      s = fmaf(__uint_as_float(a.z), __uint_as_float(b.z), s);
      s = fmaf(__uint_as_float(a.w), __uint_as_float(b.w), s);
    }
  }
  // cph is a power of two <= 32 and blocks start on multiples of 32 chunks,
  // so every group of cph lanes is one head of one row
  for (int o = cph >> 1; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (g < total && (chunk & (cph - 1)) == 0)
    delta[static_cast<int64_t>(chunk / cph) * M + row] = s;
}

// ------------------------------------------------------------ reduction
// Blocks [0, Hq): dL/dg_h = sum_j ls_j dL/db_hj (one block per head, fixed
// order).  Blocks [Hq, ...): dL/dls_j = sum_h g_h dL/db_hj in head order,
// and dL/ds_j = dL/dls_j * sigmoid(-s_j) with sigmoid(-s) = -expm1(ls).
constexpr int kRedThreads = 256;
__global__ void __launch_bounds__(kRedThreads)
    bias_grad_reduce_kernel(const float* __restrict__ dbias, int M, int Hq,
                            const float* __restrict__ ls, const float* __restrict__ gain,
                            float* __restrict__ dls, float* __restrict__ dgain,
                            float* __restrict__ dscore) {
  grid_dependency_wait();
  allow_dependents_launch();
  if (static_cast<int>(blockIdx.x) < Hq) {
    __shared__ float warp_sum[kRedThreads / 32];
    const int h = blockIdx.x;
    const float* row = dbias + static_cast<int64_t>(h) * M;
    float s = 0.f;
    for (int j = threadIdx.x; j < M; j += kRedThreads) s = fmaf(ls[j], row[j], s);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if ((threadIdx.x & 31) == 0) warp_sum[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
      float t = 0.f;
      for (int w = 0; w < kRedThreads / 32; ++w) t += warp_sum[w];
      dgain[h] = t;
    }
    return;
  }
  const int64_t j = static_cast<int64_t>(blockIdx.x - Hq) * kRedThreads + threadIdx.x;
  if (j >= M) return;
  float s = 0.f;
  for (int h = 0; h < Hq; ++h) s = fmaf(gain[h], dbias[static_cast<int64_t>(h) * M + j], s);
  dls[j] = s;
  if (dscore != nullptr) dscore[j] = s * -expm1f(ls[j]);
}

// ------------------------------------------------------ fp32 CUDA cores
// One thread per key j (64 keys per block, one q head per grid row): k_j and
// v_j in registers, the query rows i >= (first key of the block) staged
// through shared memory.
template <int DH>
__global__ void __launch_bounds__(64)
    bias_grad_f32_kernel(const float* __restrict__ QKV, const float* __restrict__ dO, int M,
                         int Hq, int Hkv, const float* __restrict__ ls,
                         const float* __restrict__ gain, float scale,
                         const float* __restrict__ lse, const float* __restrict__ delta,
                         float* __restrict__ dbias) {
  constexpr int kRows = DH == 128 ? 16 : 32;
  __shared__ float qs[kRows][DH];
  __shared__ float ds[kRows][DH];
  __shared__ float lse_s[kRows], del_s[kRows];
  grid_dependency_wait();
  allow_dependents_launch();
  const int h = blockIdx.y;
  const int hk = h / (Hq / Hkv);
  const int64_t ld = static_cast<int64_t>(Hq + 2 * Hkv) * DH;
  const int64_t ldo = static_cast<int64_t>(Hq) * DH;
  const int j0 = blockIdx.x * 64;
  const int j = j0 + threadIdx.x;
  const bool valid = j < M;
  float k[DH], v[DH];
#pragma unroll
  for (int c = 0; c < DH; ++c) {
    k[c] = valid ? QKV[j * ld + (Hq + hk) * DH + c] : 0.f;
    v[c] = valid ? QKV[j * ld + (Hq + Hkv + hk) * DH + c] : 0.f;
  }
  const float bj = (ls != nullptr && valid) ? gain[h] * ls[j] : 0.f;
  float acc = 0.f;
  for (int i0 = j0; i0 < M; i0 += kRows) {
    __syncthreads();
    for (int e = threadIdx.x; e < kRows * DH; e += 64) {
      const int r = e / DH, c = e % DH;
      const int64_t i = i0 + r;
      qs[r][c] = i < M ? QKV[i * ld + h * DH + c] : 0.f;
      ds[r][c] = i < M ? dO[i * ldo + h * DH + c] : 0.f;
    }
    for (int r = threadIdx.x; r < kRows; r += 64) {
      const int64_t i = i0 + r;
      lse_s[r] = i < M ? lse[static_cast<int64_t>(h) * M + i] : 0.f;
      del_s[r] = i < M ? delta[static_cast<int64_t>(h) * M + i] : 0.f;
    }
    __syncthreads();
    if (!valid) continue;
    for (int r = 0; r < kRows; ++r) {
      const int i = i0 + r;
      if (i < j || i >= M) continue;
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int c = 0; c < DH; ++c) {
        s = fmaf(qs[r][c], k[c], s);
        dp = fmaf(ds[r][c], v[c], dp);
      }
      const float p = expf(s * scale + bj - lse_s[r]);
      acc = fmaf(p, dp - del_s[r], acc);
    }
  }
  if (valid) dbias[static_cast<int64_t>(h) * M + j] = acc;
}

// ---------------------------------------------------- bf16 on tcgen05
constexpr int kBQ = 128;  // queries per tile: the N of both MMAs
constexpr int kBK = 128;  // keys per CTA: the M of both MMAs, one per TMEM lane
constexpr int kDH = 128;
constexpr int kThreads = 384;
constexpr uint32_t kTileBytes = 128 * 128 * 2;    // 32 KB
constexpr uint32_t kHalfBytes = kTileBytes / 2;   // one 64-column TMA box

struct BwdArgs {
  int M, Hq, Hkv, G, n_kb;
  float scale2;         // t / sqrt(dh) * log2(e)
  const float* ls;      // [M], or null for no bias
  const float* gain;    // [Hq]
  const float* lse;     // [Hq][M], natural log
  const float* delta;   // [Hq][M]
  float* dbias;         // [Hq][M]
  uint32_t* status;
};

struct BwdSmem {
  uint8_t k[kTileBytes];         // K of the CTA's key block (128-byte swizzle)
  uint8_t v[kTileBytes];         // V of the same keys
  uint8_t q[2][kTileBytes];      // Q_i of head h, per ring stage
  uint8_t dout[2][kTileBytes];   // dO_i of head h, per ring stage
  float vec[2][2][2][kBQ];       // [warpgroup][slot][-lse log2e | -D][query]
  float part[kBK];               // warpgroup 1's sums, added by warpgroup 0
  uint64_t kv_full;
  uint64_t qd_full[2], qd_empty[2];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// One lane waits, the warp follows (keeps the .sync.aligned tcgen05 loads
// warp-uniform when a wait gives up).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          uint32_t* status) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort, status) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

// Named barrier over the 128 threads of one epilogue warpgroup that also
// returns whether any of them passes `fail` (so all of them leave a loop
// together).
__device__ __forceinline__ bool group_barrier_any(uint32_t id, bool fail) {
  uint32_t any;
  asm volatile(
      "{\n .reg .pred p, f;\n setp.ne.u32 f, %1, 0;\n"
      " barrier.cta.red.or.pred p, %2, 128, f;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(any)
      : "r"(static_cast<uint32_t>(fail)), "r"(id)
      : "memory");
  return any != 0;
}

// p (dp - D) over 32 query columns [c0, c0 + 32) of one key row, two
// columns per packed instruction.  x = S scale2 + bias2 - lse2 is the logit
// minus the row's log-sum-exp in log2 units; masked columns get p = 0.
template <bool MASK>
__device__ __forceinline__ void accumulate32(const uint32_t (&sv)[32], const uint32_t (&pv)[32],
                                             const float* nl, const float* nd, int c0, int lo,
                                             int hi, uint64_t sc2, uint64_t bj2, uint64_t& acc0,
                                             uint64_t& acc1) {
#pragma unroll
  for (int q4 = 0; q4 < 8; ++q4) {
    const float4 l = *reinterpret_cast<const float4*>(nl + c0 + 4 * q4);
    const float4 d = *reinterpret_cast<const float4*>(nd + c0 + 4 * q4);
    const int c = 4 * q4;
    float x0, x1, x2, x3;
    f2_split(f2_fma(f2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sc2,
                    f2_add(bj2, f2(l.x, l.y))),
             x0, x1);
    f2_split(f2_fma(f2(__uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3])), sc2,
                    f2_add(bj2, f2(l.z, l.w))),
             x2, x3);
    if (MASK) {
      const int cc = c0 + c;
      if (cc < lo || cc >= hi) x0 = -INFINITY;
      if (cc + 1 < lo || cc + 1 >= hi) x1 = -INFINITY;
      if (cc + 2 < lo || cc + 2 >= hi) x2 = -INFINITY;
      if (cc + 3 < lo || cc + 3 >= hi) x3 = -INFINITY;
    }
    const uint64_t p01 = f2(exp2_approx(x0), exp2_approx(x1));
    const uint64_t p23 = f2(exp2_approx(x2), exp2_approx(x3));
    const uint64_t t01 = f2_add(f2(__uint_as_float(pv[c]), __uint_as_float(pv[c + 1])),
                                f2(d.x, d.y));
    const uint64_t t23 = f2_add(f2(__uint_as_float(pv[c + 2]), __uint_as_float(pv[c + 3])),
                                f2(d.z, d.w));
    acc0 = f2_fma(p01, t01, acc0);
    acc1 = f2_fma(p23, t23, acc1);
  }
}

// Epilogue warpgroup wg (warps 4-7: wg = 0, warps 8-11: wg = 1) takes the
// query tiles i = wg, wg + 2, ... of the CTA; TMEM accumulator pair wg.
// Thread r owns key row r of the block.
template <bool BIAS>
__device__ __forceinline__ void bias_grad_epilogue(BwdSmem& S, const BwdArgs& a, uint32_t tmem,
                                                   int kb, int h, int n, int wg, int warp,
                                                   int lane, volatile int* abort) {
  const int quad = warp & 3;
  const int r = quad * 32 + lane;
  const int64_t j = static_cast<int64_t>(kb) * kBK + r;
  const float bias2 = (BIAS && j < a.M) ? a.gain[h] * a.ls[j] * kLog2e : 0.f;
  const uint64_t sc2 = f2(a.scale2, a.scale2);
  const uint64_t bj2 = f2(bias2, bias2);
  const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
  const uint32_t s_tmem = tmem + wg * 256 + lane_off;
  const uint32_t p_tmem = s_tmem + 128;
  const float* lse_h = a.lse + static_cast<int64_t>(h) * a.M;
  const float* del_h = a.delta + static_cast<int64_t>(h) * a.M;
  // thread r stages query column r of each of its tiles: -lse log2(e), -D
  auto fetch = [&](int i, float& nl, float& nd) {
    const int64_t col = static_cast<int64_t>(kb + i) * kBQ + r;
    nl = 0.f;
    nd = 0.f;
    if (i < n && col < a.M) {
      nl = -__ldg(lse_h + col) * kLog2e;
      nd = -__ldg(del_h + col);
    }
  };
  float nl, nd;
  fetch(wg, nl, nd);
  uint64_t acc0 = f2(0.f, 0.f), acc1 = f2(0.f, 0.f);
  int u = 0;
  for (int i = wg; i < n; i += 2, ++u) {
    float* vl = S.vec[wg][u & 1][0];
    float* vd = S.vec[wg][u & 1][1];
    vl[r] = nl;  // slot u & 1 was last read two tiles ago, before the last barrier
    vd[r] = nd;
    const bool ok = warp_wait(smem_u32(&S.acc_full[wg]), u & 1, abort, a.status);
    if (group_barrier_any(1 + wg, !ok)) break;  // also publishes the staged columns
    tc_fence_after();
    fetch(i + 2, nl, nd);
    const int ib = kb + i;
    const bool masked = (i == 0) || (static_cast<int64_t>(ib + 1) * kBQ > a.M);
    const int lo = (i == 0) ? r : 0;  // the diagonal tile: queries at or after key r
    const int64_t rem = a.M - static_cast<int64_t>(ib) * kBQ;  // queries left in the sequence
    const int hi = rem < kBQ ? static_cast<int>(rem) : kBQ;
#pragma unroll 1
    for (int c0 = 0; c0 < kBQ; c0 += 32) {
      uint32_t sv[32], pv[32];
      tmem_ld32(s_tmem + c0, sv);
      tmem_ld32(p_tmem + c0, pv);
      tmem_ld_wait();
      if (masked) {
        accumulate32<true>(sv, pv, vl, vd, c0, lo, hi, sc2, bj2, acc0, acc1);
      } else {
        accumulate32<false>(sv, pv, vl, vd, c0, lo, hi, sc2, bj2, acc0, acc1);
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&S.acc_empty[wg]));
  }
  float a0, a1, a2, a3;
  f2_split(acc0, a0, a1);
  f2_split(acc1, a2, a3);
  const float total = (a0 + a1) + (a2 + a3);
  if (wg == 1) S.part[r] = total;
  asm volatile("bar.sync 3, 256;" ::: "memory");
  if (wg == 0 && j < a.M) a.dbias[static_cast<int64_t>(h) * a.M + j] = total + S.part[r];
}

template <bool BIAS>
__global__ void __launch_bounds__(kThreads, 1)
    keybias_bias_grad_kernel(const __grid_constant__ CUtensorMap tm_qkv,
                             const __grid_constant__ CUtensorMap tm_do, const BwdArgs args) {
  extern __shared__ uint8_t smem_raw[];
  BwdSmem& S = *reinterpret_cast<BwdSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &S.abort;

  // work unit: key block kb (heaviest = most query tiles first), q head h
  const int kb = static_cast<int>(blockIdx.x) / args.Hq;
  const int h = static_cast<int>(blockIdx.x) % args.Hq;
  const int hk = h / args.G;
  const int n = args.n_kb - kb;  // query tiles kb .. n_kb - 1

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&S.kv_full), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&S.qd_full[s]), 1);
      mbar_init(smem_u32(&S.qd_empty[s]), 1);
      mbar_init(smem_u32(&S.acc_full[s]), 1);
      mbar_init(smem_u32(&S.acc_empty[s]), 4);  // the four warps of one epilogue warpgroup
    }
    mbar_init(smem_u32(&S.drain), 1);
    S.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_qkv);
    tma_prefetch_desc(&tm_do);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&S.tmem_base), 512);
    tmem_relinquish();
  }
  grid_dependency_wait();  // lse, D (and QKV, dO) come from earlier kernels in the stream
  allow_dependents_launch();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------- TMA
      const int kcol = (args.Hq + hk) * kDH;
      const int vcol = (args.Hq + args.Hkv + hk) * kDH;
      const int qcol = h * kDH;
      const uint64_t pol = l2_policy_evict_last();  // Q and dO tiles are re-read by other key blocks
      mbar_arrive_expect_tx(smem_u32(&S.kv_full), 2 * kTileBytes);
      for (int bx = 0; bx < 2; ++bx) {
        tma_load_2d(smem_u32(S.k) + bx * kHalfBytes, &tm_qkv, smem_u32(&S.kv_full),
                    kcol + bx * 64, kb * kBK);
        tma_load_2d(smem_u32(S.v) + bx * kHalfBytes, &tm_qkv, smem_u32(&S.kv_full),
                    vcol + bx * 64, kb * kBK);
      }
      int nq = 0;  // ring fills issued
      for (int i = 0; i < n; ++i) {
        const int s = i & 1;
        const uint32_t ph = (i >> 1) & 1;
        if (!mbar_wait(smem_u32(&S.qd_empty[s]), ph ^ 1, abort, args.status)) break;
        mbar_arrive_expect_tx(smem_u32(&S.qd_full[s]), 2 * kTileBytes);
        const int row = (kb + i) * kBQ;
        for (int bx = 0; bx < 2; ++bx) {
          tma_load_2d_hint(smem_u32(S.q[s]) + bx * kHalfBytes, &tm_qkv, smem_u32(&S.qd_full[s]),
                           qcol + bx * 64, row, pol);
          tma_load_2d_hint(smem_u32(S.dout[s]) + bx * kHalfBytes, &tm_do,
                           smem_u32(&S.qd_full[s]), qcol + bx * 64, row, pol);
        }
        ++nq;
      }
      // every issued copy lands before the CTA may exit
      mbar_wait_drain(smem_u32(&S.kv_full), 0);
      for (int s = 0; s < 2; ++s)
        if (s < nq) mbar_wait_drain(smem_u32(&S.qd_full[s]), ((nq - 1 - s) >> 1) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------- MMA
      // S^T = K Q_i^T and dP^T = V dO_i^T: M = 128 keys, N = 128 queries,
      // K = dh, all four operands K-major with 128-byte swizzle.  All
      // descriptors are formed once; a K step inside a tile is a constant
      // added to the start-address field.
      constexpr uint32_t idesc = idesc_bf16_f32(kBK, kBQ, 0, 0);
      uint64_t kd[kDH / 16], vd[kDH / 16];
#pragma unroll
      for (int kk = 0; kk < kDH / 16; ++kk) {
        const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
        kd[kk] = smem_desc_sw128(smem_u32(S.k) + off, 16, 1024);
        vd[kk] = smem_desc_sw128(smem_u32(S.v) + off, 16, 1024);
      }
      const uint64_t qd0[2] = {smem_desc_sw128(smem_u32(S.q[0]), 16, 1024),
                               smem_desc_sw128(smem_u32(S.q[1]), 16, 1024)};
      const uint64_t dd0[2] = {smem_desc_sw128(smem_u32(S.dout[0]), 16, 1024),
                               smem_desc_sw128(smem_u32(S.dout[1]), 16, 1024)};
      bool ok = mbar_wait(smem_u32(&S.kv_full), 0, abort, args.status);
      for (int i = 0; ok && i < n; ++i) {
        const int s = i & 1;  // ring stage, and accumulator pair
        ok = mbar_wait(smem_u32(&S.qd_full[s]), (i >> 1) & 1, abort, args.status);
        if (ok && i >= 2)  // pair s was last read by the epilogue of tile i - 2
          ok = mbar_wait(smem_u32(&S.acc_empty[s]), ((i - 2) >> 1) & 1, abort, args.status);
        if (!ok) break;
        tc_fence_after();
        const uint32_t s_tmem = tmem + s * 256;
        const uint32_t p_tmem = s_tmem + 128;
#pragma unroll
        for (int kk = 0; kk < kDH / 16; ++kk)
          mma_ss(s_tmem, kd[kk], qd0[s] + (((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4), idesc,
                 kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < kDH / 16; ++kk)
          mma_ss(p_tmem, vd[kk], dd0[s] + (((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4), idesc,
                 kk > 0 ? 1u : 0u);
        mma_commit(smem_u32(&S.acc_full[s]));
        mma_commit(smem_u32(&S.qd_empty[s]));
      }
      mma_commit(smem_u32(&S.drain));
      mbar_wait_drain(smem_u32(&S.drain), 0);
    }
  } else if (warp >= 4) {
    bias_grad_epilogue<BIAS>(S, args, tmem, kb, h, n, (warp - 4) >> 2, warp, lane, abort);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_attn_delta(const void* dO, const void* Oa, int x_bf16, int64_t M, int Hq,
                              int dh, float* delta, cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  const int cph = dh * (x_bf16 ? 2 : 4) / 16;  // 16-byte chunks per head
  const int64_t chunks = M * Hq * cph;
  const unsigned grid = static_cast<unsigned>((chunks + 255) / 256);
  cudaError_t err;
  if (x_bf16) {
    err = launch_pdl(attn_delta_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, stream, 1u,
                     static_cast<const __nv_bfloat16*>(dO), static_cast<const __nv_bfloat16*>(Oa),
                     static_cast<int>(M), Hq, cph, delta);
  } else {
    err = launch_pdl(attn_delta_kernel<float>, dim3(grid), dim3(256), 0, stream, 1u,
                     static_cast<const float*>(dO), static_cast<const float*>(Oa),
                     static_cast<int>(M), Hq, cph, delta);
  }
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

cudaError_t launch_bias_grad_reduce(const float* dbias, int64_t M, int Hq, const float* ls,
                                    const float* gain, float* dls, float* dgain, float* dscore,
                                    cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>(Hq + (M + kRedThreads - 1) / kRedThreads);
  cudaError_t err = launch_pdl(bias_grad_reduce_kernel, dim3(grid), dim3(kRedThreads), 0, stream,
                               1u, dbias, static_cast<int>(M), Hq, ls, gain, dls, dgain, dscore);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

cudaError_t launch_bias_grad_f32(const float* QKV, const float* dO, int64_t M, int Hq, int Hkv,
                                 int dh, const float* ls, const float* gain, float temperature,
                                 const float* lse, const float* delta, float* dbias,
                                 cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  dim3 grid(static_cast<unsigned>((M + 63) / 64), Hq);
  const float scale = temperature / sqrtf(static_cast<float>(dh));
  const int m = static_cast<int>(M);
  cudaError_t err;
  switch (dh) {
    case 32:
      err = launch_pdl(bias_grad_f32_kernel<32>, grid, dim3(64), 0, stream, 1u, QKV, dO, m, Hq,
                       Hkv, ls, gain, scale, lse, delta, dbias);
      break;
    case 64:
      err = launch_pdl(bias_grad_f32_kernel<64>, grid, dim3(64), 0, stream, 1u, QKV, dO, m, Hq,
                       Hkv, ls, gain, scale, lse, delta, dbias);
      break;
    case 128:
      err = launch_pdl(bias_grad_f32_kernel<128>, grid, dim3(64), 0, stream, 1u, QKV, dO, m, Hq,
                       Hkv, ls, gain, scale, lse, delta, dbias);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

cudaError_t launch_bias_grad_bf16(const void* QKV, const void* dO, int64_t M, int Hq, int Hkv,
                                  int dh, const float* ls, const float* gain, float temperature,
                                  const float* lse, const float* delta, float* dbias,
                                  cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  BwdArgs a{};
  a.M = static_cast<int>(M);
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.G = Hq / Hkv;
  a.n_kb = static_cast<int>((M + kBK - 1) / kBK);
  a.scale2 = temperature / sqrtf(static_cast<float>(dh)) * kLog2e;
  a.ls = ls;
  a.gain = gain;
  a.lse = lse;
  a.delta = delta;
  a.dbias = dbias;
  a.status = device_status_word();
  const int cols = (Hq + 2 * Hkv) * dh;
  CUtensorMap tm_qkv, tm_do;
  if (!make_tmap_2d(&tm_qkv, QKV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, cols, M,
                    static_cast<uint64_t>(cols) * 2, 64, kBQ, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (!make_tmap_2d(&tm_do, dO, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                    static_cast<uint64_t>(Hq) * dh, M, static_cast<uint64_t>(Hq) * dh * 2, 64,
                    kBQ, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const size_t smem = sizeof(BwdSmem) + 1024;
  const int grid = a.n_kb * Hq;
  auto kernel = ls != nullptr ? keybias_bias_grad_kernel<true> : keybias_bias_grad_kernel<false>;
  cudaError_t err =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  err = launch_pdl(kernel, dim3(grid), dim3(kThreads), smem, stream, 1u, tm_qkv, tm_do, a);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace tg
