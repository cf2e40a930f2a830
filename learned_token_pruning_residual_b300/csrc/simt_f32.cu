// fp32 CUDA-core versions of the gate MLP, the QKV projection and the
// key-bias attention, for fp32 inputs (small models and checking).  Same
// definitions as the bf16 tensor-core kernels:
//   gate  s_i = w2 . GELU(W1 x_i + b1) + b2          (TokenGate pages,
//         spke.com "TokenGate – Token-Gated Attention macht das Vollfüllen
//         von langen Kontexten bis zu 11,3-mal schneller", Gate-Modul)
//   qkv   QKV = X Wqkv^T
//   attn  l_ij = t (q_i . k_j) / sqrt(dh) + g_h ls_j, causal, GQA
//         (same page, section "Was ist token-gated Attention?")
#include "tg_device.cuh"
#include "tg_internal.h"

namespace tg {
namespace {

__device__ __forceinline__ float gelu_erf_f32(float z) {
  return 0.5f * z * (1.0f + erff(z * 0.70710678118654752f));
}

// one CTA per token; threads split the hidden units
__global__ void __launch_bounds__(256)
    gate_f32_kernel(const float* __restrict__ X, int d, const float* __restrict__ W1,
                    const float* __restrict__ b1, int Hg, const float* __restrict__ w2, float b2,
                    float* __restrict__ scores) {
  extern __shared__ float xs[];
  __shared__ float red[8];
  const int64_t i = blockIdx.x;
  for (int c = threadIdx.x; c < d; c += blockDim.x) xs[c] = X[i * d + c];
  __syncthreads();
  float acc = 0.f;
  for (int k = threadIdx.x; k < Hg; k += blockDim.x) {
    const float* w = W1 + static_cast<int64_t>(k) * d;
    float z = 0.f;
    for (int c = 0; c < d; c += 4) {
      const float4 wv = __ldg(reinterpret_cast<const float4*>(w + c));
      z = fmaf(wv.x, xs[c], z);
      z = fmaf(wv.y, xs[c + 1], z);
      z = fmaf(wv.z, xs[c + 2], z);
      z = fmaf(wv.w, xs[c + 3], z);
    }
    if (b1) z += b1[k];
    acc = fmaf(w2[k], gelu_erf_f32(z), acc);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += red[w];
    scores[i] = s + b2;
  }
}

// 32 x 32 output tile per CTA, 16 x 16 threads, 2 x 2 outputs each
constexpr int kT = 32, kKT = 16;
__global__ void __launch_bounds__(256)
    gemm_f32_kernel(const float* __restrict__ A, int64_t M, int K, const float* __restrict__ B,
                    int N, float* __restrict__ C) {
  __shared__ float As[kKT][kT + 1];
  __shared__ float Bs[kKT][kT + 1];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int64_t row0 = static_cast<int64_t>(blockIdx.y) * kT;
  const int col0 = blockIdx.x * kT;
  float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
  for (int k0 = 0; k0 < K; k0 += kKT) {
    for (int e = threadIdx.x; e < kT * kKT; e += 256) {
      const int r = e / kKT, k = e % kKT;
      const int64_t gr = row0 + r;
      const int gc = col0 + r;
      As[k][r] = (gr < M && k0 + k < K) ? A[gr * K + k0 + k] : 0.f;
      Bs[k][r] = (gc < N && k0 + k < K) ? B[static_cast<int64_t>(gc) * K + k0 + k] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kKT; ++k) {
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 2; ++b) acc[a][b] = fmaf(As[k][ty * 2 + a], Bs[k][tx * 2 + b], acc[a][b]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int a = 0; a < 2; ++a)
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const int64_t r = row0 + ty * 2 + a;
      const int c = col0 + tx * 2 + b;
      if (r < M && c < N) C[r * N + c] = acc[a][b];
    }
}

// one thread per (row, q head); keys streamed through shared memory in
// chunks of 64; online softmax in fp32 with expf
template <int DH>
__global__ void __launch_bounds__(64)
    attn_f32_kernel(const float* __restrict__ QKV, int64_t M, int Hq, int Hkv,
                    const float* __restrict__ ls, const float* __restrict__ gain, float scale,
                    float* __restrict__ O, float* __restrict__ residual, float* __restrict__ lse) {
  constexpr int kKeys = DH == 128 ? 32 : 64;  // 32 KB of keys and values at most
  __shared__ float ks[kKeys][DH];
  __shared__ float vs[kKeys][DH];
  __shared__ float bs[kKeys];
  const int h = blockIdx.y;
  const int hk = h / (Hq / Hkv);
  const int64_t ld = static_cast<int64_t>(Hq + 2 * Hkv) * DH;
  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * 64;
  const int64_t i = row0 + threadIdx.x;
  const bool valid = i < M;
  const float g = ls ? gain[h] : 0.f;
  float q[DH], o[DH];
#pragma unroll
  for (int c = 0; c < DH; ++c) {
    q[c] = valid ? QKV[i * ld + h * DH + c] : 0.f;
    o[c] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  const int64_t jend = (row0 + 64 < M ? row0 + 64 : M);  // keys needed by this CTA
  for (int64_t j0 = 0; j0 < jend; j0 += kKeys) {
    __syncthreads();
    for (int e = threadIdx.x; e < kKeys * DH; e += 64) {
      const int r = e / DH, c = e % DH;
      const int64_t j = j0 + r;
      ks[r][c] = j < M ? QKV[j * ld + (Hq + hk) * DH + c] : 0.f;
      vs[r][c] = j < M ? QKV[j * ld + (Hq + Hkv + hk) * DH + c] : 0.f;
    }
    for (int r = threadIdx.x; r < kKeys; r += 64) {
      const int64_t j = j0 + r;
      bs[r] = (ls && j < M) ? g * ls[j] : 0.f;
    }
    __syncthreads();
    for (int r = 0; r < kKeys; ++r) {
      const int64_t j = j0 + r;
      if (j > i || !valid) break;
      float dot = 0.f;
#pragma unroll
      for (int c = 0; c < DH; ++c) dot = fmaf(q[c], ks[r][c], dot);
      const float logit = dot * scale + bs[r];
      if (logit > m) {
        const float f = expf(m - logit);
        l *= f;
#pragma unroll
        for (int c = 0; c < DH; ++c) o[c] *= f;
        m = logit;
      }
      const float p = expf(logit - m);
      l += p;
#pragma unroll
      for (int c = 0; c < DH; ++c) o[c] = fmaf(p, vs[r][c], o[c]);
    }
  }
  if (!valid) return;
  if (lse != nullptr) lse[static_cast<int64_t>(h) * M + i] = m + logf(l);
  const float inv = 1.f / l;
  const int64_t ldo = static_cast<int64_t>(Hq) * DH;
#pragma unroll
  for (int c = 0; c < DH; ++c) {
    const float v = o[c] * inv;
    if (residual)
      residual[i * ldo + h * DH + c] += v;
    else
      O[i * ldo + h * DH + c] = v;
  }
}

}  // namespace

cudaError_t launch_gate_f32(const float* X, int64_t N, int d, const float* W1, const float* b1,
                            int Hg, const float* w2, float b2, float* scores,
                            cudaStream_t stream) {
  if (N == 0) return cudaSuccess;
  const size_t smem = static_cast<size_t>(d) * 4;
  if (smem > 48 * 1024) {
    cudaError_t err = cudaFuncSetAttribute(gate_f32_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
  }
  gate_f32_kernel<<<static_cast<unsigned>(N), 256, smem, stream>>>(X, d, W1, b1, Hg, w2, b2,
                                                                  scores);
  return cudaGetLastError();
}

cudaError_t launch_qkv_f32(const float* X, int64_t M, int d, const float* W, int ncols, float* Y,
                           cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  dim3 grid((ncols + kT - 1) / kT, static_cast<unsigned>((M + kT - 1) / kT));
  gemm_f32_kernel<<<grid, 256, 0, stream>>>(X, M, d, W, ncols, Y);
  return cudaGetLastError();
}

cudaError_t launch_attn_f32(const float* QKV, int64_t M, int Hq, int Hkv, int dh,
                            const float* logsig, const float* gain, float temperature, float* O,
                            float* residual, float* lse, cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  dim3 grid(static_cast<unsigned>((M + 63) / 64), Hq);
  const float scale = temperature / sqrtf(static_cast<float>(dh));
  switch (dh) {
    case 32:
      attn_f32_kernel<32><<<grid, 64, 0, stream>>>(QKV, M, Hq, Hkv, logsig, gain, scale, O, residual, lse);
      break;
    case 64:
      attn_f32_kernel<64><<<grid, 64, 0, stream>>>(QKV, M, Hq, Hkv, logsig, gain, scale, O, residual, lse);
      break;
    case 128:
      attn_f32_kernel<128><<<grid, 64, 0, stream>>>(QKV, M, Hq, Hkv, logsig, gain, scale, O, residual, lse);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace tg
