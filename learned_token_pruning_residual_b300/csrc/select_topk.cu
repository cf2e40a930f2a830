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
// One cluster of 8 CTAs x 1024 threads does everything in one launch: each
// CTA caches its slice of the span's keys in shared memory, histograms are
// merged through distributed shared memory, and the passes are separated by
// hardware cluster barriers (no spinning, no global scratch).
#include <cooperative_groups.h>

#include "tg_device.cuh"
#include "tg_internal.h"

namespace cg = cooperative_groups;

namespace tg {
namespace {

constexpr int kCtas = 8;
constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kCacheKeys = 24576;  // keys cached per CTA (96 KB)

__device__ __forceinline__ uint32_t key_of(float s) {
  const uint32_t u = __float_as_uint(s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct SelShared {
  uint32_t hist[2048];
  uint32_t warp_a[kWarps];
  uint32_t warp_b[kWarps];
  uint32_t slice_total;
  uint32_t cta_gt, cta_eq;
  uint32_t found_prefix, found_krem;  // written by the owning CTA into every CTA
  uint32_t above;                     // keys in higher-ranked CTAs' bins (this pass)
  uint32_t gt_base, eq_base;          // kept / tied keys in lower-ranked CTAs' slices
  int nan_seen;
};

// Inclusive sum over the block of one value per thread; returns the
// inclusive prefix of this thread, and the block total in *total.
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
  *total = warp_buf[kWarps - 1];
  __syncthreads();
  return v + add;
}

template <bool CACHED>
__global__ void __cluster_dims__(kCtas, 1, 1) __launch_bounds__(kThreads, 1)
    select_topk_kernel(const float* __restrict__ scores, int N, int b, int e, int K,
                       int32_t* __restrict__ idx, uint32_t* status) {
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int tid = threadIdx.x, lane = tid & 31;
  extern __shared__ uint32_t keys_smem[];
  __shared__ SelShared S;

  const int D = e - b;
  const int chunk = (D + kCtas - 1) / kCtas;
  const int lo = min(D, rank * chunk), hi = min(D, lo + chunk);
  const int n = hi - lo;  // keys owned by this CTA: doc positions b + lo + [0, n)
  const float* src = scores + b + lo;
  grid_dependency_wait();  // the scores come from the previous kernel in the stream
  allow_dependents_launch();

  auto load_key = [&](int i) -> uint32_t {
    if constexpr (CACHED) {
      return keys_smem[i];
    } else {
      return key_of(__ldg(src + i));
    }
  };

  // ---- tokens outside the span are always kept, in order
  for (int i = rank * kThreads + tid; i < N - D; i += kCtas * kThreads) {
    if (i < b) {
      idx[i] = i;
    } else {
      idx[b + K + (i - b)] = e + (i - b);
    }
  }

  if (tid == 0) S.nan_seen = 0;
  __syncthreads();
  {
    int nan_local = 0;
    for (int i = tid; i < n; i += kThreads) {
      const float s = __ldg(src + i);
      nan_local |= (s != s);
      if constexpr (CACHED) keys_smem[i] = key_of(s);
    }
    if (__any_sync(0xffffffffu, nan_local) && lane == 0) S.nan_seen = 1;
  }
  __syncthreads();
  if (tid == 0 && S.nan_seen) atomicOr(status, kStatusNanScore);

  uint32_t T = 0, k_eq = 0;
  if (K == 0) {
    T = 0xFFFFFFFFu;  // nothing is above, and no tie is taken
    k_eq = 0;
  } else if (K == D) {
    T = 0u;  // everything is at or above, and every tie is taken
    k_eq = static_cast<uint32_t>(D);
  } else {
    // ---- three radix passes: 11, 11, 10 bits
    uint32_t prefix = 0, krem = static_cast<uint32_t>(K);
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
      const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
      const int bins = pass == 2 ? 1024 : 2048;
      const int pshift = shift + (pass == 2 ? 10 : 11);  // bits above the digit
      for (int i = tid; i < bins; i += kThreads) S.hist[i] = 0;
      __syncthreads();
      const int n_round = (n + 31) & ~31;
      for (int i = tid; i < n_round; i += kThreads) {
        bool valid = false;
        uint32_t bin = 0xFFFFFFFFu;
        if (i < n) {
          const uint32_t k = load_key(i);
          valid = pass == 0 || (k >> pshift) == prefix;
          if (valid) bin = (k >> shift) & static_cast<uint32_t>(bins - 1);
        }
        const uint32_t peers = __match_any_sync(0xffffffffu, bin);
        if (valid && lane == __ffs(peers) - 1) atomicAdd(&S.hist[bin], __popc(peers));
      }
      cluster.sync();
      // this CTA merges bins [rank * slice, (rank + 1) * slice) of all CTAs
      const int slice = bins / kCtas;
      uint32_t merged = 0;
      if (tid < slice) {
#pragma unroll
        for (int c = 0; c < kCtas; ++c)
          merged += cluster.map_shared_rank(S.hist, c)[rank * slice + tid];
      }
      uint32_t slice_total;
      const uint32_t incl = block_inclusive_scan(merged, S.warp_a, &slice_total);
      if (tid == 0) S.slice_total = slice_total;
      cluster.sync();  // slice totals published; all remote histogram reads done
      // one warp reads the eight slice totals; the block reads the sum from
      // shared memory (one remote load per CTA instead of one per thread)
      if (tid < 32) {
        uint32_t v = (tid > rank && tid < kCtas) ? *cluster.map_shared_rank(&S.slice_total, tid) : 0u;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (tid == 0) S.above = v;
      }
      __syncthreads();
      const uint32_t above = S.above;  // keys in the bins of higher-ranked CTAs
      if (tid < slice) {
        const uint32_t strictly_above = above + slice_total - incl;  // bins > this one
        const uint32_t at_or_above = strictly_above + merged;
        if (strictly_above < krem && krem <= at_or_above) {
          const uint32_t bin = static_cast<uint32_t>(rank * slice + tid);
          const uint32_t np = (prefix << (pass == 2 ? 10 : 11)) | bin;
          const uint32_t nk = krem - strictly_above;
          for (int c = 0; c < kCtas; ++c) {
            SelShared* R = cluster.map_shared_rank(&S, c);
            R->found_prefix = np;
            R->found_krem = nk;
          }
        }
      }
      cluster.sync();
      prefix = S.found_prefix;
      krem = S.found_krem;
    }
    T = prefix;
    k_eq = krem;
  }

  // ---- ordered compaction: thread t owns a contiguous run of L keys, L odd
  // so that the strided shared-memory reads hit distinct banks
  int L = (n + kThreads - 1) / kThreads;
  L |= 1;
  const int r0 = min(n, tid * L), r1 = min(n, r0 + L);
  uint32_t gt = 0, eq = 0;
  for (int i = r0; i < r1; ++i) {
    const uint32_t k = load_key(i);
    gt += k > T;
    eq += k == T;
  }
  uint32_t gt_tot, eq_tot;
  const uint32_t gt_incl = block_inclusive_scan(gt, S.warp_a, &gt_tot);
  const uint32_t eq_incl = block_inclusive_scan(eq, S.warp_b, &eq_tot);
  if (tid == 0) {
    S.cta_gt = gt_tot;
    S.cta_eq = eq_tot;
  }
  cluster.sync();
  if (tid < 32) {  // counts of the lower-ranked CTAs, read once
    uint32_t g = 0, q = 0;
    if (tid < rank) {
      const SelShared* R = cluster.map_shared_rank(&S, tid);
      g = R->cta_gt;
      q = R->cta_eq;
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
  uint32_t gt_before = gt_incl - gt + S.gt_base, eq_before = eq_incl - eq + S.eq_base;
  for (int i = r0; i < r1; ++i) {
    const uint32_t k = load_key(i);
    const bool keep = k > T || (k == T && eq_before < k_eq);
    if (keep) {
      const uint32_t pos = gt_before + min(eq_before, k_eq);
      if (pos < static_cast<uint32_t>(K)) {
        idx[b + pos] = b + lo + i;
      } else {
        atomicOr(status, kStatusBadIndex);  // cannot happen for a consistent threshold
      }
    }
    gt_before += k > T;
    eq_before += k == T;
  }
  cluster.sync();  // no CTA leaves while another may still read its shared memory
}

}  // namespace

cudaError_t launch_select(const float* scores, int64_t N, int64_t b, int64_t e, int64_t K,
                          int32_t* idx, cudaStream_t stream) {
  const int64_t D = e - b;
  const int64_t chunk = (D + kCtas - 1) / kCtas;
  uint32_t* status = device_status_word();
  if (chunk <= kCacheKeys) {
    const size_t smem = static_cast<size_t>(kCacheKeys) * 4;
    cudaError_t err = cudaFuncSetAttribute(select_topk_kernel<true>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    err = launch_pdl(select_topk_kernel<true>, dim3(kCtas), dim3(kThreads), smem, stream, 1u,
                     scores, (int)N, (int)b, (int)e, (int)K, idx, status);
    if (err != cudaSuccess) return err;
  } else {
    cudaError_t err = launch_pdl(select_topk_kernel<false>, dim3(kCtas), dim3(kThreads), 0,
                                 stream, 1u, scores, (int)N, (int)b, (int)e, (int)K, idx, status);
    if (err != cudaSuccess) return err;
  }
  return cudaGetLastError();
}

}  // namespace tg
