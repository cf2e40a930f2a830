// Bandwidth-bound row kernels of the gated prefill.
//
//  * gather: only the kept tokens' rows go up to the pruned layers (TokenGate
//    pages: ai.info "TokenGate riporta un prefill fino a 11,3 volte più
//    veloce sui contesti lunghi", section "TokenGate impara quali token
//    mantenere"), together with log(sigmoid(score)) of each kept token, the
//    input of the attention bias (spke.com "TokenGate – Token-Gated Attention
//    macht das Vollfüllen von langen Kontexten bis zu 11,3-mal schneller",
//    section "Was ist token-gated Attention?").
//  * RMSNorm of a pruned layer's input.
//
// One warp per row, 16-byte vector loads and stores, grid-stride over rows.
#include "tg_device.cuh"
#include "tg_internal.h"

namespace tg {
namespace {

constexpr int kRowThreads = 256;
constexpr int kRowWarps = kRowThreads / 32;

__device__ __forceinline__ float logsigmoid_f32(float s) {
  // log(sigmoid(s)) = min(s, 0) - log1p(exp(-|s|)), stable at both ends
  return fminf(s, 0.f) - log1pf(expf(-fabsf(s)));
}

// copy 8 bf16 -> 8 bf16, 4 f32 -> 4 f32, or 8 bf16 -> 8 f32 per vector step
template <int MODE>  // 0: bf16->bf16, 1: f32->f32, 2: bf16->f32
__global__ void __launch_bounds__(kRowThreads)
    gather_rows_kernel(const uint8_t* __restrict__ X, int64_t N, int d,
                       const int32_t* __restrict__ idx, int64_t M, uint8_t* __restrict__ Y,
                       const float* __restrict__ scores, float* __restrict__ logsig,
                       uint32_t* status) {
  const int lane = threadIdx.x & 31;
  const int64_t warp_global = static_cast<int64_t>(blockIdx.x) * kRowWarps + (threadIdx.x >> 5);
  const int64_t warps = static_cast<int64_t>(gridDim.x) * kRowWarps;
  const int in_bytes = MODE == 1 ? d * 4 : d * 2;
  const int out_bytes = MODE == 0 ? d * 2 : d * 4;
  const int nvec = in_bytes / 16;  // 16-byte input vectors per row
  grid_dependency_wait();  // idx, scores and X come from the previous kernels
  allow_dependents_launch();
  for (int64_t m = warp_global; m < M; m += warps) {
    const int64_t i = idx ? static_cast<int64_t>(__ldg(idx + m)) : m;
    const bool ok = i >= 0 && i < N;
    if (!ok && lane == 0) atomicOr(status, kStatusBadIndex);
    const uint4* src = reinterpret_cast<const uint4*>(X + (ok ? i : 0) * in_bytes);
    uint8_t* dst_row = Y + m * out_bytes;
    if (logsig != nullptr && lane == 0) logsig[m] = ok ? logsigmoid_f32(__ldg(scores + i)) : 0.f;
    constexpr int U = 8;  // a 2048-wide bf16 row in one round trip per lane
    for (int v0 = lane; v0 < nvec; v0 += 32 * U) {
      uint4 buf[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + 32 * u;
        buf[u] = (ok && v < nvec) ? __ldcs(src + v) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + 32 * u;
        if (v >= nvec) break;
        if constexpr (MODE != 2) {
          reinterpret_cast<uint4*>(dst_row)[v] = buf[u];
        } else {
          const uint32_t w[4] = {buf[u].x, buf[u].y, buf[u].z, buf[u].w};
          float4 lo = make_float4(bf16lo_to_f32(w[0]), bf16hi_to_f32(w[0]), bf16lo_to_f32(w[1]),
                                  bf16hi_to_f32(w[1]));
          float4 hi = make_float4(bf16lo_to_f32(w[2]), bf16hi_to_f32(w[2]), bf16lo_to_f32(w[3]),
                                  bf16hi_to_f32(w[3]));
          reinterpret_cast<float4*>(dst_row)[2 * v] = lo;
          reinterpret_cast<float4*>(dst_row)[2 * v + 1] = hi;
        }
      }
    }
  }
}

template <bool X_BF16, bool Y_BF16>
__global__ void __launch_bounds__(kRowThreads)
    rmsnorm_kernel(const void* __restrict__ X, int64_t M, int d, const float* __restrict__ gamma,
                   float eps, void* __restrict__ Y) {
  const int lane = threadIdx.x & 31;
  const int64_t warp_global = static_cast<int64_t>(blockIdx.x) * kRowWarps + (threadIdx.x >> 5);
  const int64_t warps = static_cast<int64_t>(gridDim.x) * kRowWarps;
  const int n8 = d / 8;
  grid_dependency_wait();
  allow_dependents_launch();
  for (int64_t m = warp_global; m < M; m += warps) {
    float ss = 0.f;
    for (int v = lane; v < n8; v += 32) {
      float x[8];
      if constexpr (X_BF16) {
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(X) + m * d) + v);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          x[2 * k] = bf16lo_to_f32(w[k]);
          x[2 * k + 1] = bf16hi_to_f32(w[k]);
        }
      } else {
        const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(X) + m * d) + 2 * v;
        const float4 a = __ldg(p), b = __ldg(p + 1);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) ss = fmaf(x[k], x[k], ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float rstd = rsqrtf(ss / static_cast<float>(d) + eps);
    for (int v = lane; v < n8; v += 32) {
      float x[8];
      if constexpr (X_BF16) {
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(X) + m * d) + v);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          x[2 * k] = bf16lo_to_f32(w[k]);
          x[2 * k + 1] = bf16hi_to_f32(w[k]);
        }
      } else {
        const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(X) + m * d) + 2 * v;
        const float4 a = __ldg(p), b = __ldg(p + 1);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
      }
      const float4 g0 = __ldg(reinterpret_cast<const float4*>(gamma) + 2 * v);
      const float4 g1 = __ldg(reinterpret_cast<const float4*>(gamma) + 2 * v + 1);
      const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
      float y[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) y[k] = x[k] * rstd * g[k];
      if constexpr (Y_BF16) {
        uint4 o;
        o.x = pack_bf16x2(y[0], y[1]);
        o.y = pack_bf16x2(y[2], y[3]);
        o.z = pack_bf16x2(y[4], y[5]);
        o.w = pack_bf16x2(y[6], y[7]);
        reinterpret_cast<uint4*>(static_cast<uint16_t*>(Y) + m * d)[v] = o;
      } else {
        float4* q = reinterpret_cast<float4*>(static_cast<float*>(Y) + m * d) + 2 * v;
        q[0] = make_float4(y[0], y[1], y[2], y[3]);
        q[1] = make_float4(y[4], y[5], y[6], y[7]);
      }
    }
  }
}

int row_grid(int64_t rows) {
  const int64_t want = (rows + kRowWarps - 1) / kRowWarps;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  return static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

cudaError_t launch_gather(const void* X, int x_bf16, int64_t N, int d, const int32_t* idx,
                          int64_t M, void* Y, int y_bf16, const float* scores, float* logsig,
                          cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  const int grid = row_grid(M);
  uint32_t* st = device_status_word();
  const uint8_t* Xb = static_cast<const uint8_t*>(X);
  uint8_t* Yb = static_cast<uint8_t*>(Y);
  if (x_bf16 && y_bf16)
    return launch_pdl(gather_rows_kernel<0>, dim3(grid), dim3(kRowThreads), 0, stream, 1u, Xb, N, d,
                      idx, M, Yb, scores, logsig, st);
  else if (!x_bf16 && !y_bf16)
    return launch_pdl(gather_rows_kernel<1>, dim3(grid), dim3(kRowThreads), 0, stream, 1u, Xb, N, d,
                      idx, M, Yb, scores, logsig, st);
  else
    return launch_pdl(gather_rows_kernel<2>, dim3(grid), dim3(kRowThreads), 0, stream, 1u, Xb, N, d,
                      idx, M, Yb, scores, logsig, st);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm(const void* X, int x_bf16, int64_t M, int d, const float* gamma,
                           float eps, void* Y, int y_bf16, cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  const int grid = row_grid(M);
  if (x_bf16 && y_bf16)
    return launch_pdl(rmsnorm_kernel<true, true>, dim3(grid), dim3(kRowThreads), 0, stream, 1u, X, M, d,
                      gamma, eps, Y);
  else if (x_bf16)
    return launch_pdl(rmsnorm_kernel<true, false>, dim3(grid), dim3(kRowThreads), 0, stream, 1u, X, M, d,
                      gamma, eps, Y);
  else if (y_bf16)
    return launch_pdl(rmsnorm_kernel<false, true>, dim3(grid), dim3(kRowThreads), 0, stream, 1u, X, M, d,
                      gamma, eps, Y);
  else
    return launch_pdl(rmsnorm_kernel<false, false>, dim3(grid), dim3(kRowThreads), 0, stream, 1u, X, M, d,
                      gamma, eps, Y);
  return cudaGetLastError();
}

}  // namespace tg
