// Top-K selection over the document span with the question never pruned
// (TokenGate pages: spke.com "TokenGate – Token-Gated Attention macht das
// Vollfüllen von langen Kontexten bis zu 11,3-mal schneller", section "Wie
// hat TokenGate das Pruning von Tokens verstanden?"; ai4bro.com, section
// "กลไกการทำงานของ Learned Token Pruning", phases 2 and 3).
//
// Order: fp32 score bits mapped to uint32 keys (negative patterns inverted,
// the rest with the sign bit set), larger key first, lower index first on
// equal keys.  The K-th key T is found by a 3-pass radix select (11, 11 and
// 10 bits); then every document token with key > T, and the first k_eq
// tokens with key == T in index order, are kept.  Output indices ascend, so
// the result is unique and deterministic.
//
// One launch of G CTAs (G <= the SM count, ~2048 keys each, one CTA per SM
// at most so that all of them are resident together; B300, 130816 keys:
// 19.0 us with 16 CTAs, 17.1 with 32, 16.4 with 64, 17.7 with 128).  Each CTA caches its
// contiguous slice of the span's keys in shared memory.  Per radix pass every
// CTA adds its shared-memory histogram into a global one in the workspace,
// the CTAs meet at a grid barrier, and every CTA then reads the merged
// histogram and finds the threshold bin itself (no second barrier).  The
// ordered compaction exchanges per-CTA (>T, ==T) counts through one more
// barrier.  The grid barrier is an arrival counter plus a generation word;
// its waiters poll with a sleep and give up after the library's wait bound
// (TG_ERR_TIMEOUT), so a CTA that never arrives cannot hang the GPU.
//
// The gate kernel can count the first histogram from the scores it has just
// computed (its epilogue holds every score) into a slot of its own; it then
// stamps the workspace header with (N, doc_begin, doc_end), and a select
// call on the same span uses that histogram and skips its first pass and
// its first barrier (on another span it ignores it).  The select call leaves
// the histograms, the header and the barrier words zero for the next call.
#include "tg_device.cuh"
#include "tg_internal.h"

namespace tg {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kKeysPerCta = 2048;    // target slice
constexpr int kCacheKeys = 24576;    // largest slice kept in shared memory (96 KB)

__device__ __forceinline__ uint32_t key_of(float s) {
  const uint32_t u = __float_as_uint(s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
  return old;
}

__device__ __forceinline__ void red_add_release(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

struct SelShared {
  uint32_t hist[2048];
  uint32_t warp_a[kWarps];
  uint32_t warp_b[kWarps];
  uint32_t seg_n[kSelectMaxCtas];    // candidates of each CTA
  uint32_t seg_off[kSelectMaxCtas];  // their offsets in the gathered list
  uint32_t seg_at[kSelectMaxCtas];   // where they start in the workspace
  uint32_t cand_at;                  // this CTA's reserved run
  uint32_t found_prefix, found_krem;
  uint32_t gt_base, eq_base;
  uint32_t cand_n, cand_total;
  int nan_seen;
  int abort;
  int overflow;
};

// Inclusive sum over the block of one value per thread; returns this
// thread's inclusive prefix and the block total in *total.
__device__ __forceinline__ uint32_t block_inclusive_scan(uint32_t v, uint32_t* warp_buf,
                                                         uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_buf[warp] = v;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < kWarps ? warp_buf[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    if (lane < kWarps) warp_buf[lane] = w;
  }
  __syncthreads();
  const uint32_t add = warp > 0 ? warp_buf[warp - 1] : 0u;
  *total = warp_buf[kWarps - 1];
  __syncthreads();
  return v + add;
}

// All CTAs of the grid meet here.  Thread 0 of each CTA arrives on the
// counter; the last one resets it and bumps the generation, the others poll
// the generation (sleeping between polls) for at most the wait bound.
// Returns false when this CTA gave up (then the status word has
// TG_ERR_TIMEOUT and the CTA must leave).
__device__ __forceinline__ bool grid_barrier(SelectWorkspace* ws, uint32_t nctas, uint32_t* status,
                                             SelShared& S) {
  __syncthreads();
  if (threadIdx.x == 0 && !S.abort) {
    const uint32_t gen = ld_acquire(&ws->bar_gen);
    // the arrival releases this CTA's global writes (made visible to the
    // CTA's thread 0 by the __syncthreads above)
    const uint32_t arrived = atom_add_acq_rel(&ws->bar_count, 1u) + 1u;
    if (arrived == nctas) {
      // everyone has arrived: reset the counter, then publish the new
      // generation (release: the reset and every CTA's writes, which this
      // thread acquired through the counter, come before it)
      ws->bar_count = 0u;
      red_add_release(&ws->bar_gen, 1u);
    } else {
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire(&ws->bar_gen) == gen) {
        __nanosleep(100);
        if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
          atomicOr(status, kStatusTimeout);
          S.abort = 1;
          break;
        }
      }
    }
  }
  __syncthreads();
  return S.abort == 0;
}

// Finds, in the merged histogram h of `bins` bins, the bin where the krem-th
// largest key falls (counting from the top bin down); writes the bin and the
// rank left inside it to S.found_prefix / S.found_krem.
template <bool GLOBAL = true>
__device__ __forceinline__ void find_threshold_bin(const uint32_t* h, int bins, uint32_t krem,
                                                   SelShared& S) {
  const int per = bins / kThreads;  // 4 (2048 bins) or 2 (1024 bins)
  // thread j owns bins top-down: [bins - per (j + 1), bins - per j)
  uint32_t c[4] = {0, 0, 0, 0};
  uint32_t sum = 0;
  for (int k = 0; k < per; ++k) {
    const uint32_t* p = h + bins - 1 - (per * threadIdx.x + k);
    c[k] = GLOBAL ? __ldcg(p) : *p;
    sum += c[k];
  }
  uint32_t total;
  const uint32_t incl = block_inclusive_scan(sum, S.warp_a, &total);
  uint32_t above = incl - sum;  // keys in higher bins
  for (int k = 0; k < per; ++k) {
    if (above < krem && krem <= above + c[k]) {
      S.found_prefix = static_cast<uint32_t>(bins - 1 - (per * threadIdx.x + k));
      S.found_krem = krem - above;
    }
    above += c[k];
  }
  __syncthreads();
}

template <bool CACHED>
__global__ void __launch_bounds__(kThreads, 1)
    select_topk_kernel(const float* __restrict__ scores, int N, int b, int e, int K,
                       int32_t* __restrict__ idx, uint32_t* status, SelectWorkspace* ws,
                       int slice) {
  extern __shared__ uint32_t keys_smem[];
  __shared__ SelShared S;
  const int tid = threadIdx.x, lane = tid & 31;
  const int cta = static_cast<int>(blockIdx.x);
  const uint32_t G = gridDim.x;
  const int D = e - b;
  const int lo = min(D, cta * slice), hi = min(D, lo + slice);
  const int n = hi - lo;  // this CTA's keys: doc positions b + lo + [0, n)
  const float* src = scores + b + lo;
  if (tid == 0) {
    S.nan_seen = 0;
    S.abort = 0;
  }
  grid_dependency_wait();  // scores (and the gate's histogram) come from the previous kernel
  allow_dependents_launch();

  auto load_key = [&](int i) -> uint32_t {
    if constexpr (CACHED) {
      return keys_smem[i];
    } else {
      return key_of(__ldg(src + i));
    }
  };

  // ---- tokens outside the span are always kept, in order
  for (int i = cta * kThreads + tid; i < N - D; i += static_cast<int>(G) * kThreads) {
    if (i < b) {
      idx[i] = i;
    } else {
      idx[b + K + (i - b)] = e + (i - b);
    }
  }
  // is the first histogram already there (filled by the gate on this span)?
  const bool stamped = __ldcg(&ws->hdr[0]) == kSelectHistMagic;
  const bool prefilled = stamped && __ldcg(&ws->hdr[1]) == static_cast<uint32_t>(N) &&
                         __ldcg(&ws->hdr[2]) == static_cast<uint32_t>(b) &&
                         __ldcg(&ws->hdr[3]) == static_cast<uint32_t>(e);
  __syncthreads();
  {
    int nan_local = 0;
    constexpr int kLoadBatch = 16;  // loads in flight per thread before their stores
    for (int i0 = tid; i0 < n; i0 += kLoadBatch * kThreads) {
      float v[kLoadBatch];
#pragma unroll
      for (int u = 0; u < kLoadBatch; ++u) {
        const int i = i0 + u * kThreads;
        v[u] = i < n ? __ldg(src + i) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < kLoadBatch; ++u) {
        const int i = i0 + u * kThreads;
        nan_local |= (v[u] != v[u]);
        if constexpr (CACHED) {
          if (i < n) keys_smem[i] = key_of(v[u]);
        }
      }
    }
    if (__any_sync(0xffffffffu, nan_local) && lane == 0) S.nan_seen = 1;
  }
  __syncthreads();
  if (tid == 0 && S.nan_seen) atomicOr(status, kStatusNanScore);

  uint32_t T = 0, k_eq = 0;
  bool ok = true;
  bool fast = false;  // the candidate path found T and this CTA's offsets
  const bool trivial = K == 0 || K == D;
  if (K == 0) {
    T = 0xFFFFFFFFu;  // nothing is above, and no tie is taken
  } else if (K == D) {
    T = 0u;  // everything is at or above, and every tie is taken
    k_eq = static_cast<uint32_t>(D);
  } else {
    // ---- three radix passes: 11, 11, 10 bits
    uint32_t prefix = 0, krem = static_cast<uint32_t>(K);
    int pass = 0;
    auto global_pass = [&]() {
      const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
      const int bins = pass == 2 ? 1024 : 2048;
      const int pshift = shift + (pass == 2 ? 10 : 11);  // bits above the digit
      uint32_t* gh = (pass == 0 && prefilled) ? ws->gate_hist : ws->hist[pass];
      if (!(pass == 0 && prefilled)) {
        for (int i = tid; i < bins; i += kThreads) S.hist[i] = 0;
        __syncthreads();
        for (int i = tid; i < n; i += kThreads) {
          const uint32_t k = load_key(i);
          if (pass == 0 || (k >> pshift) == prefix)
            atomicAdd(&S.hist[(k >> shift) & static_cast<uint32_t>(bins - 1)], 1u);
        }
        __syncthreads();
        for (int i = tid; i < bins; i += kThreads) {
          const uint32_t c = S.hist[i];
          if (c) atomicAdd(gh + i, c);
        }
        ok = grid_barrier(ws, G, status, S);
        if (!ok) return;
      }
      find_threshold_bin(gh, bins, krem, S);
      prefix = (prefix << (pass == 2 ? 10 : 11)) | S.found_prefix;
      krem = S.found_krem;
    };
    global_pass();
    pass = 1;
    if constexpr (CACHED) {
      // ---- candidates: the keys whose first digit is the threshold bin.
      // Each CTA reserves a run of the workspace's candidate array (one
      // atomic add; the runs are recorded, so the gather below reads them in
      // CTA order whatever order the reservations came in), writes its
      // candidates there and counts the keys above the bin; after one
      // barrier every CTA gathers all candidates and finishes the select on
      // them alone: the last two passes, and the (> T, == T) counts of the
      // lower-ranked CTAs.  Only the total is capped, so a CTA with more
      // than its share of the bin does not force the slow path.
      if (ok) {
        // per-thread counts of candidates and of keys above the bin (packed
        // as cand + above << 16; each at most a slice), one block scan, then
        // each thread writes its candidates at its offset
        uint32_t packed = 0;
        for (int i = tid; i < n; i += kThreads) {
          const uint32_t top = keys_smem[i] >> 21;
          packed += (top == prefix ? 1u : 0u) + (top > prefix ? 0x10000u : 0u);
        }
        uint32_t tot;
        const uint32_t incl = block_inclusive_scan(packed, S.warp_a, &tot);
        const uint32_t nmine = tot & 0xFFFFu;
        if (tid == 0) {
          const uint32_t at = atomicAdd(&ws->cand_next, nmine);
          S.cand_at = at;
          __stcg(&ws->cand_at[cta], at);
          __stcg(&ws->cnt[cta][0], tot >> 16);
          __stcg(&ws->cnt[cta][1], nmine);
        }
        __syncthreads();
        const uint32_t at = S.cand_at;
        uint32_t pos = (incl - packed) & 0xFFFFu;
        for (int i = tid; i < n; i += kThreads) {
          const uint32_t k = keys_smem[i];
          if ((k >> 21) == prefix) {
            if (at + pos < static_cast<uint32_t>(kSelectCandCap)) __stcg(ws->cand + at + pos, k);
            ++pos;
          }
        }
        ok = grid_barrier(ws, G, status, S);
      }
      if (ok) {
        // every CTA's counts and runs; candidate offsets; keys above the bin
        // in the lower-ranked CTAs
        const uint32_t cn = tid < static_cast<int>(G) ? __ldcg(&ws->cnt[tid][1]) : 0u;
        const uint32_t cat = tid < static_cast<int>(G) ? __ldcg(&ws->cand_at[tid]) : 0u;
        const uint32_t an = tid < cta ? __ldcg(&ws->cnt[tid][0]) : 0u;
        if (tid == 0) S.overflow = 0;
        __syncthreads();
        if (cat + cn > static_cast<uint32_t>(kSelectCandCap)) S.overflow = 1;
        uint32_t total, an_tot;
        const uint32_t off = block_inclusive_scan(cn, S.warp_a, &total) - cn;
        block_inclusive_scan(an, S.warp_b, &an_tot);
        if (tid < static_cast<int>(G)) {
          S.seg_n[tid] = cn;
          S.seg_off[tid] = off;
          S.seg_at[tid] = cat;
        }
        if (tid == 0) S.cand_total = total;
        __syncthreads();
        if (!S.overflow) {
          uint32_t* cand_smem = keys_smem + ((slice + 3) & ~3);
          const uint32_t nc = S.cand_total;
          // gather: warp w copies segments w, w + 16, ...; eight loads in
          // flight per lane before their stores
          constexpr int kBatch = 8;
          for (uint32_t sg = tid >> 5; sg < G; sg += kWarps) {
            const uint32_t ns = S.seg_n[sg], off = S.seg_off[sg];
            const uint32_t* src2 = ws->cand + S.seg_at[sg];
            for (uint32_t j0 = lane; j0 < ns; j0 += kBatch * 32) {
              uint32_t v[kBatch];
#pragma unroll
              for (int u = 0; u < kBatch; ++u) {
                const uint32_t j = j0 + u * 32;
                v[u] = j < ns ? __ldcg(src2 + j) : 0u;
              }
#pragma unroll
              for (int u = 0; u < kBatch; ++u) {
                const uint32_t j = j0 + u * 32;
                if (j < ns) cand_smem[off + j] = v[u];
              }
            }
          }
          __syncthreads();
          for (; pass < 3; ++pass) {
            const int shift = pass == 1 ? 10 : 0;
            const int bins = pass == 2 ? 1024 : 2048;
            const int pshift = shift + (pass == 2 ? 10 : 11);
            for (int i = tid; i < bins; i += kThreads) S.hist[i] = 0;
            __syncthreads();
            for (uint32_t i = tid; i < nc; i += kThreads) {
              const uint32_t k = cand_smem[i];
              if ((k >> pshift) == prefix)
                atomicAdd(&S.hist[(k >> shift) & static_cast<uint32_t>(bins - 1)], 1u);
            }
            __syncthreads();
            find_threshold_bin<false>(S.hist, bins, krem, S);
            prefix = (prefix << (pass == 2 ? 10 : 11)) | S.found_prefix;
            krem = S.found_krem;
          }
          // (> T, == T) among the lower-ranked CTAs' candidates, packed as
          // gt + eq << 16 (each at most kSelectCandCap)
          const uint32_t T2 = prefix;
          uint32_t packed = 0;
          const uint32_t lower = S.seg_off[cta];
          for (uint32_t i = tid; i < lower; i += kThreads) {
            const uint32_t k = cand_smem[i];
            packed += (k > T2 ? 1u : 0u) + (k == T2 ? 0x10000u : 0u);
          }
          uint32_t packed_tot;
          block_inclusive_scan(packed, S.warp_a, &packed_tot);
          if (tid == 0) {
            S.gt_base = an_tot + (packed_tot & 0xFFFFu);
            S.eq_base = packed_tot >> 16;
          }
          __syncthreads();
          fast = true;
        }
      }
    }
    for (; ok && pass < 3; ++pass) global_pass();
    T = prefix;
    k_eq = krem;
  }

  // ---- ordered compaction: thread t owns a contiguous run of L keys, L odd
  // so that the strided shared-memory reads hit distinct banks
  if (ok && K > 0) {
    int L = (n + kThreads - 1) / kThreads;
    L |= 1;
    const int r0 = min(n, tid * L), r1 = min(n, r0 + L);
    uint32_t gt = 0, eq = 0;
    if (K == D) {
      eq = static_cast<uint32_t>(r1 - r0);  // every key is kept, in order
    } else {
      for (int i = r0; i < r1; ++i) {
        const uint32_t k = load_key(i);
        gt += k > T;
        eq += k == T;
      }
    }
    uint32_t gt_tot, eq_tot, gt_incl, eq_incl;
    if constexpr (CACHED) {
      // one scan of gt + eq << 16 (each at most a cached slice, <= 24576 keys)
      uint32_t pk_tot;
      const uint32_t pk_incl = block_inclusive_scan(gt | (eq << 16), S.warp_a, &pk_tot);
      gt_tot = pk_tot & 0xFFFFu;
      eq_tot = pk_tot >> 16;
      gt_incl = pk_incl & 0xFFFFu;
      eq_incl = pk_incl >> 16;
    } else {
      gt_incl = block_inclusive_scan(gt, S.warp_a, &gt_tot);
      eq_incl = block_inclusive_scan(eq, S.warp_b, &eq_tot);
    }
    if (trivial) {
      // K == D: the kept document tokens are the whole span, position = offset
      if (tid == 0) {
        S.gt_base = 0;
        S.eq_base = static_cast<uint32_t>(lo);
      }
      __syncthreads();
    } else if (fast) {
      // S.gt_base / S.eq_base were set from the candidates
    } else {
      if (tid == 0) {
        __stcg(&ws->cnt[cta][0], gt_tot);
        __stcg(&ws->cnt[cta][1], eq_tot);
      }
      ok = grid_barrier(ws, G, status, S);
      if (ok && tid < 32) {  // counts of the lower-ranked CTAs
        uint32_t g = 0, q = 0;
        for (int c = tid; c < cta; c += 32) {
          g += __ldcg(&ws->cnt[c][0]);
          q += __ldcg(&ws->cnt[c][1]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          g += __shfl_xor_sync(0xffffffffu, g, o);
          q += __shfl_xor_sync(0xffffffffu, q, o);
        }
        if (tid == 0) {
          S.gt_base = g;
          S.eq_base = q;
        }
      }
      __syncthreads();
    }
    if (ok) {
      uint32_t gt_before = gt_incl - gt + S.gt_base, eq_before = eq_incl - eq + S.eq_base;
      bool bad = false;
      for (int i = r0; i < r1; ++i) {
        const uint32_t k = K == D ? 0u : load_key(i);
        const bool is_gt = K != D && k > T;
        const bool is_eq = K == D || k == T;
        const bool keep = is_gt || (is_eq && eq_before < k_eq);
        const uint32_t pos = gt_before + min(eq_before, k_eq);
        bad |= keep && pos >= static_cast<uint32_t>(K);
        if (keep && pos < static_cast<uint32_t>(K)) idx[b + pos] = b + lo + i;
        gt_before += is_gt;
        eq_before += is_eq;
      }
      if (bad) atomicOr(status, kStatusBadIndex);  // cannot happen for a consistent threshold
    }
  }

  // ---- leave the workspace clean for the next call.  Every CTA has read
  // the histograms before its last barrier arrival, so after that barrier
  // (or when there was none: the trivial K) CTA 0 may clear them.
  if (cta == 0 && ok) {
    if (tid == 0) __stcg(&ws->cand_next, 0u);  // every CTA reserved before the barrier
    if (!trivial) {
      for (int i = tid; i < 2048; i += kThreads) {
        if (!prefilled) __stcg(&ws->hist[0][i], 0u);
        __stcg(&ws->hist[1][i], 0u);
        if (i < 1024) __stcg(&ws->hist[2][i], 0u);
      }
    }
    if (stamped) {  // a gate histogram, of this span or another one
      for (int i = tid; i < 2048; i += kThreads) __stcg(&ws->gate_hist[i], 0u);
      if (tid == 0)
        for (int i = 0; i < 4; ++i) __stcg(&ws->hdr[i], 0u);
    }
  }
}

// ---------------------------------------------------------------------------
// Single-CTA select for short spans (up to kSelectSmallMaxKeys keys; its
// time grows with the span, B300: 16128 keys 15.1 us, 24320 keys 19.4 us,
// against 13.6 and 14.1 us for the multi-CTA select with 2048 keys per CTA,
// which takes every span longer than 4096 keys): no grid barrier, no
// global scratch beyond the gate's histogram.  All keys are loaded once (16-byte loads, every thread's
// loads in flight together) into shared memory; the first pass's bin comes
// from the gate's histogram when it is there; the other passes and the
// ordered compaction (warp ballots over consecutive keys, a block scan of
// per-warp counts) read shared memory only.
constexpr int kSmallThreads = 1024;
constexpr int kSmallWarps = kSmallThreads / 32;

struct SmallShared {
  uint32_t hist[2048];
  uint32_t warp_a[kSmallWarps];
  uint32_t warp_b[kSmallWarps];
  uint32_t found_prefix, found_krem;
  int nan_seen;
};

__device__ __forceinline__ uint32_t small_block_scan(uint32_t v, uint32_t* warp_buf,
                                                     uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_buf[warp] = v;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = warp_buf[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    warp_buf[lane] = w;
  }
  __syncthreads();
  const uint32_t add = warp > 0 ? warp_buf[warp - 1] : 0u;
  *total = warp_buf[kSmallWarps - 1];
  __syncthreads();
  return v + add;
}

// The bin of `h` (nbins 2048 or 1024) that holds the krem-th largest key;
// h is shared memory or (global_mem) the gate's histogram in the workspace.
__device__ __forceinline__ void small_find_bin(const uint32_t* h, bool global_mem, int nbins,
                                               uint32_t krem, SmallShared& S) {
  const int per = nbins / kSmallThreads;  // 2 or 1
  uint32_t c[2] = {0, 0}, sum = 0;
  for (int k = 0; k < per; ++k) {
    const int bin = nbins - 1 - (per * threadIdx.x + k);
    c[k] = global_mem ? __ldcg(h + bin) : h[bin];
    sum += c[k];
  }
  uint32_t total;
  uint32_t above = small_block_scan(sum, S.warp_a, &total) - sum;
  for (int k = 0; k < per; ++k) {
    if (above < krem && krem <= above + c[k]) {
      S.found_prefix = static_cast<uint32_t>(nbins - 1 - (per * threadIdx.x + k));
      S.found_krem = krem - above;
    }
    above += c[k];
  }
  __syncthreads();
}

// Histogram of the digit (key >> shift) & (nbins - 1) over the cached keys
// whose bits above the digit equal `prefix` (all keys when pshift >= 32).
__device__ __forceinline__ void small_hist(const uint32_t* keys, int n, int shift, int nbins,
                                           int pshift, uint32_t prefix, SmallShared& S) {
  for (int i = threadIdx.x; i < nbins; i += kSmallThreads) S.hist[i] = 0u;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += kSmallThreads) {
    const uint32_t k = keys[i];
    if (pshift >= 32 || (k >> pshift) == prefix)
      atomicAdd(&S.hist[(k >> shift) & static_cast<uint32_t>(nbins - 1)], 1u);
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kSmallThreads, 1)
    select_small_kernel(const float* __restrict__ scores, int N, int b, int e, int K,
                        int32_t* __restrict__ idx, uint32_t* status, SelectWorkspace* ws) {
  extern __shared__ uint32_t small_keys[];  // the span's keys, [D]
  __shared__ SmallShared S;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int D = e - b;
  const float* src = scores + b;
  if (tid == 0) S.nan_seen = 0;
  grid_dependency_wait();  // scores (and the gate's histogram) come from the previous kernel
  allow_dependents_launch();

  // tokens outside the span are always kept, in order
  for (int i = tid; i < N - D; i += kSmallThreads) {
    if (i < b) {
      idx[i] = i;
    } else {
      idx[b + K + (i - b)] = e + (i - b);
    }
  }
  const bool stamped = __ldcg(&ws->hdr[0]) == kSelectHistMagic;
  const bool prefilled = stamped && __ldcg(&ws->hdr[1]) == static_cast<uint32_t>(N) &&
                         __ldcg(&ws->hdr[2]) == static_cast<uint32_t>(b) &&
                         __ldcg(&ws->hdr[3]) == static_cast<uint32_t>(e);
  // ---- all keys into shared memory: the span's first (4 - b % 4) % 4 keys
  // one by one, the rest as 16-byte loads (scores + b rounded up to 16 bytes)
  {
    const int head = min(D, (4 - (b & 3)) & 3);
    int nan_local = 0;
    if (tid < head) {
      const float v = __ldg(src + tid);
      nan_local |= (v != v);
      small_keys[tid] = key_of(v);
    }
    const float4* src4 = reinterpret_cast<const float4*>(src + head);
    const int n4 = (D - head) >> 2;
    constexpr int U = 4;  // float4 loads in flight per thread per round
    for (int i0 = tid; i0 < n4; i0 += U * kSmallThreads) {
      float4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * kSmallThreads;
        v[u] = i < n4 ? __ldg(src4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * kSmallThreads;
        if (i < n4) {
          nan_local |= (v[u].x != v[u].x) | (v[u].y != v[u].y) | (v[u].z != v[u].z) |
                       (v[u].w != v[u].w);
          uint4 k;
          k.x = key_of(v[u].x);
          k.y = key_of(v[u].y);
          k.z = key_of(v[u].z);
          k.w = key_of(v[u].w);
          // head + 4 i is not 16-byte aligned in small_keys unless head == 0
          uint32_t* dst = small_keys + head + 4 * i;
          dst[0] = k.x;
          dst[1] = k.y;
          dst[2] = k.z;
          dst[3] = k.w;
        }
      }
    }
    const int tail0 = head + 4 * n4;
    if (tid < D - tail0) {
      const float v = __ldg(src + tail0 + tid);
      nan_local |= (v != v);
      small_keys[tail0 + tid] = key_of(v);
    }
    if (__any_sync(0xffffffffu, nan_local) && lane == 0) S.nan_seen = 1;
  }
  __syncthreads();
  if (tid == 0 && S.nan_seen) atomicOr(status, kStatusNanScore);

  uint32_t T = 0, k_eq = 0;
  if (K == 0) {
    T = 0xFFFFFFFFu;
  } else if (K == D) {
    k_eq = static_cast<uint32_t>(D);
  } else {
    uint32_t prefix = 0, krem = static_cast<uint32_t>(K);
    for (int pass = 0; pass < 3; ++pass) {
      const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
      const int nbins = pass == 2 ? 1024 : 2048;
      const int pshift = pass == 0 ? 32 : (pass == 1 ? 21 : 10);
      if (pass == 0 && prefilled) {
        small_find_bin(ws->gate_hist, true, 2048, krem, S);
      } else {
        small_hist(small_keys, D, shift, nbins, pshift, prefix, S);
        small_find_bin(S.hist, false, nbins, krem, S);
      }
      prefix = pass == 0 ? S.found_prefix : ((prefix << (pass == 2 ? 10 : 11)) | S.found_prefix);
      krem = S.found_krem;
    }
    T = prefix;
    k_eq = krem;
  }

  // ---- ordered compaction; warp w owns keys [w * chunk, (w + 1) * chunk)
  if (K > 0) {
    const int chunk = ((D + kSmallWarps - 1) / kSmallWarps + 31) & ~31;
    const int c0 = min(D, warp * chunk), c1 = min(D, c0 + chunk);
    const uint32_t lt = (1u << lane) - 1u;
    uint32_t gt = 0, eq = 0;
    if (K == D) {
      eq = static_cast<uint32_t>(c1 - c0);
    } else {
      for (int i0 = c0; i0 < c1; i0 += 32) {
        const int i = i0 + lane;
        const uint32_t k = i < c1 ? small_keys[i] : 0u;
        gt += __popc(__ballot_sync(0xffffffffu, i < c1 && k > T));
        eq += __popc(__ballot_sync(0xffffffffu, i < c1 && k == T));
      }
    }
    uint32_t gt_tot, eq_tot;
    const uint32_t gt_incl = small_block_scan(lane == 0 ? gt : 0u, S.warp_a, &gt_tot);
    const uint32_t eq_incl = small_block_scan(lane == 0 ? eq : 0u, S.warp_b, &eq_tot);
    uint32_t gt_before = __shfl_sync(0xffffffffu, gt_incl - (lane == 0 ? gt : 0u), 0);
    uint32_t eq_before = __shfl_sync(0xffffffffu, eq_incl - (lane == 0 ? eq : 0u), 0);
    for (int i0 = c0; i0 < c1; i0 += 32) {
      const int i = i0 + lane;
      const bool in = i < c1;
      const uint32_t k = (in && K != D) ? small_keys[i] : 0u;
      const bool is_gt = in && K != D && k > T;
      const bool is_eq = in && (K == D || k == T);
      const uint32_t mg = __ballot_sync(0xffffffffu, is_gt);
      const uint32_t me = __ballot_sync(0xffffffffu, is_eq);
      const uint32_t eq_rank = eq_before + __popc(me & lt);
      const bool keep = is_gt || (is_eq && eq_rank < k_eq);
      if (keep) {
        const uint32_t pos = gt_before + __popc(mg & lt) + min(eq_rank, k_eq);
        if (pos < static_cast<uint32_t>(K)) {
          idx[b + pos] = b + i;
        } else {
          atomicOr(status, kStatusBadIndex);  // cannot happen for a consistent threshold
        }
      }
      gt_before += __popc(mg);
      eq_before += __popc(me);
    }
  }
  // a gate histogram (of this span or another) is used up: clear it
  if (stamped) {
    __syncthreads();
    for (int i = tid; i < 2048; i += kSmallThreads) __stcg(&ws->gate_hist[i], 0u);
    if (tid == 0)
      for (int i = 0; i < 4; ++i) __stcg(&ws->hdr[i], 0u);
  }
}

}  // namespace

int select_grid_size(int64_t D) {
  const int64_t want = (D + kKeysPerCta - 1) / kKeysPerCta;
  const int cap = sm_count() < kSelectMaxCtas ? sm_count() : kSelectMaxCtas;
  return static_cast<int>(want < 1 ? 1 : (want > cap ? cap : want));
}

cudaError_t launch_select(const float* scores, int64_t N, int64_t b, int64_t e, int64_t K,
                          int32_t* idx, SelectWorkspace* ws, cudaStream_t stream) {
  const int64_t D = e - b;
  if (D <= kSelectSmallMaxKeys) {
    uint32_t* status = device_status_word();
    if (status == nullptr) return cudaErrorInvalidDevice;
    const size_t smem = static_cast<size_t>(D > 0 ? D : 1) * 4;
    cudaError_t err = cudaFuncSetAttribute(select_small_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(kSelectSmallMaxKeys * 4));
    if (err != cudaSuccess) return err;
    err = launch_pdl(select_small_kernel, dim3(1), dim3(kSmallThreads), smem, stream, 1u, scores,
                     (int)N, (int)b, (int)e, (int)K, idx, status, ws);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
  }
  const int G = select_grid_size(D);
  const int slice = static_cast<int>((D + G - 1) / G);
  uint32_t* status = device_status_word();
  if (status == nullptr) return cudaErrorInvalidDevice;
  if (slice <= kCacheKeys) {
    const size_t smem = (static_cast<size_t>((slice + 3) & ~3) + kSelectCandCap) * 4;
    cudaError_t err = cudaFuncSetAttribute(select_topk_kernel<true>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (kCacheKeys + kSelectCandCap) * 4);
    if (err != cudaSuccess) return err;
    err = launch_pdl(select_topk_kernel<true>, dim3(G), dim3(kThreads), smem, stream, 1u, scores,
                     (int)N, (int)b, (int)e, (int)K, idx, status, ws, slice);
    if (err != cudaSuccess) return err;
  } else {
    cudaError_t err =
        launch_pdl(select_topk_kernel<false>, dim3(G), dim3(kThreads), 0, stream, 1u, scores,
                   (int)N, (int)b, (int)e, (int)K, idx, status, ws, slice);
    if (err != cudaSuccess) return err;
  }
  return cudaGetLastError();
}

}  // namespace tg
