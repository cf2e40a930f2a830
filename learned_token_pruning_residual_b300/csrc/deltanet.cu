// The gated delta rule of the Gated-DeltaNet layers of a hybrid model, run
// over the kept tokens (TokenGate pages: ai4bro.com, section "การใช้งานกับ
// โมเดล hybrid-attention"; spke.com, section "Wird es auf Hybrid-Attention-
// Modellen funktionieren?"; ai.info, section "I modelli ibridi ampliano le
// possibilità di selezione dei token": the gate can sit in a DeltaNet layer
// of a hybrid model, and the DeltaNet layers above it are pruned too).  Per
// head, with a state S in R^{dv x dk}:
//     S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   o_t = S_t q_t.
// A pruned layer runs the recurrence over the kept tokens only.
//
// Chunked evaluation (chunks of C = 64 tokens; g_i the cumulative product of
// alpha within the chunk, S the state before the chunk):
//   the delta-rule errors U (u_i = v_i - alpha_i S_{i-1} k_i) solve
//       (I + A) U = V - diag(g) K S^T,   A_ij = (g_i/g_j) beta_j (k_i . k_j), j < i,
//   so U = Ut - W S^T with Ut = (I + A)^{-1} V and W = (I + A)^{-1} diag(g) K,
//   which do not depend on S; then
//       O = diag(g) Q S^T + P U,   P_ij = (g_i/g_j) beta_j (q_i . k_j), j <= i,
//       S <- g_C S + U^T diag(beta g_C / g) K.
// Two kernels:
//   deltanet_chunk_kernel   one CTA per (chunk, head), all in parallel: the
//                           Gram products, the unit-triangular solves for Ut
//                           and W (one column per thread, forward
//                           substitution), and P; written to the workspace.
//   deltanet_scan_kernel    one CTA per (head, block of 16 state rows): the
//                           rows of S are independent chains (row r of the
//                           update reads only row r of S), so each CTA walks
//                           the chunks in order with its 16 x dk block of S
//                           in shared memory and writes its 16 output
//                           columns of every token.
// fp32 inputs and arithmetic on CUDA cores throughout; bf16 inputs take the
// tensor-core kernels of deltanet_tc.cu.
#include <algorithm>

#include "tg_device.cuh"
#include "tg_internal.h"

namespace tg {
namespace {

constexpr int kC = 64;        // tokens per chunk
constexpr int kD = 128;       // dk = dv
constexpr int kR = 16;        // state rows per scan CTA
constexpr int kPrepThreads = 256;
constexpr int kScanThreads = 256;

// workspace record of one (chunk, head)
struct ChunkRec {
  float ut[kC][kD];  // (I + A)^{-1} V
  float w[kC][kD];   // (I + A)^{-1} diag(g) K
  float p[kC][kC];   // (g_i / g_j) beta_j (q_i . k_j), j <= i
  float lg[kC];      // log g_i (cumulative log alpha)
  float dk[kC];      // (g_C / g_j) beta_j: the weights of the state update
};

template <typename T>
__device__ __forceinline__ float ld_val(const T* p, int64_t i) {
  if constexpr (sizeof(T) == 2) {
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
  } else {
    return reinterpret_cast<const float*>(p)[i];
  }
}

template <typename T>
__device__ __forceinline__ void st_val(T* p, int64_t i, float v) {
  if constexpr (sizeof(T) == 2) {
    reinterpret_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
  } else {
    reinterpret_cast<float*>(p)[i] = v;
  }
}

struct PrepSmem {
  float k[kC][kD + 1];  // +1: conflict-free column walks
  float x[kC][kD + 1];  // V, then Q
  float a[kC][kC + 1];  // A, then P
  float lg[kC], beta[kC];
};

template <typename T>
__global__ void __launch_bounds__(kPrepThreads)
    deltanet_chunk_kernel(const T* __restrict__ q, const T* __restrict__ k,
                          const T* __restrict__ v, const float* __restrict__ alpha,
                          const float* __restrict__ beta, int T_len, int H,
                          ChunkRec* __restrict__ ws) {
  extern __shared__ uint8_t smem_raw[];
  PrepSmem& S = *reinterpret_cast<PrepSmem*>(smem_raw);
  const int c = blockIdx.x / H, h = blockIdx.x % H;
  const int t0 = c * kC;
  const int n = min(kC, T_len - t0);  // tokens in this chunk
  const int tid = threadIdx.x;
  grid_dependency_wait();
  allow_dependents_launch();
  // K and V rows (zero past the end); alpha = 1, beta = 0 past the end
  for (int e = tid; e < kC * kD; e += kPrepThreads) {
    const int i = e / kD, col = e % kD;
    const int64_t off = (static_cast<int64_t>(t0 + i) * H + h) * kD + col;
    S.k[i][col] = i < n ? ld_val(k, off) : 0.f;
    S.x[i][col] = i < n ? ld_val(v, off) : 0.f;
  }
  if (tid < 32) {
    // cumulative log alpha over the chunk (two lanes' worth of tokens each)
    float la[2], run = 0.f;
    for (int s = 0; s < 2; ++s) {
      const int i = 2 * tid + s;
      la[s] = i < n ? __logf(fmaxf(alpha[static_cast<int64_t>(t0 + i) * H + h], 1e-30f)) : 0.f;
      S.beta[i] = i < n ? beta[static_cast<int64_t>(t0 + i) * H + h] : 0.f;
    }
    float pair = la[0] + la[1];
    float incl = pair;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, incl, o);
      if (tid >= o) incl += y;
    }
    run = incl - pair;
    S.lg[2 * tid] = run + la[0];
    S.lg[2 * tid + 1] = run + la[0] + la[1];
  }
  __syncthreads();
  // A_ij = (g_i / g_j) beta_j (k_i . k_j) for j < i
  for (int e = tid; e < kC * kC; e += kPrepThreads) {
    const int i = e / kC, j = e % kC;
    float a = 0.f;
    if (j < i) {
      float d = 0.f;
#pragma unroll 8
      for (int col = 0; col < kD; ++col) d = fmaf(S.k[i][col], S.k[j][col], d);
      a = __expf(S.lg[i] - S.lg[j]) * S.beta[j] * d;
    }
    S.a[i][j] = a;
  }
  __syncthreads();
  ChunkRec& R = ws[static_cast<int64_t>(c) * H + h];
  // unit lower-triangular solves, one column per thread: threads 0..127 solve
  // (I + A) Ut = V (column tid), threads 128..255 solve (I + A) W = diag(g) K
  {
    const int col = tid & (kD - 1);
    const bool is_w = tid >= kD;
    float xcol[kC];
#pragma unroll
    for (int i = 0; i < kC; ++i) {
      float b = is_w ? __expf(S.lg[i]) * S.k[i][col] : S.x[i][col];
#pragma unroll
      for (int l = 0; l < i; ++l) b = fmaf(-S.a[i][l], xcol[l], b);
      xcol[i] = b;
    }
    float* dst = is_w ? &R.w[0][0] : &R.ut[0][0];
#pragma unroll
    for (int i = 0; i < kC; ++i) dst[i * kD + col] = xcol[i];
  }
  __syncthreads();
  // Q rows into x; P_ij = (g_i / g_j) beta_j (q_i . k_j), j <= i
  for (int e = tid; e < kC * kD; e += kPrepThreads) {
    const int i = e / kD, col = e % kD;
    S.x[i][col] = i < n ? ld_val(q, (static_cast<int64_t>(t0 + i) * H + h) * kD + col) : 0.f;
  }
  __syncthreads();
  for (int e = tid; e < kC * kC; e += kPrepThreads) {
    const int i = e / kC, j = e % kC;
    float pv = 0.f;
    if (j <= i) {
      float d = 0.f;
#pragma unroll 8
      for (int col = 0; col < kD; ++col) d = fmaf(S.x[i][col], S.k[j][col], d);
      pv = __expf(S.lg[i] - S.lg[j]) * S.beta[j] * d;
    }
    R.p[i][j] = pv;
  }
  if (tid < kC) {
    R.lg[tid] = S.lg[tid];
    R.dk[tid] = __expf(S.lg[kC - 1] - S.lg[tid]) * S.beta[tid];
  }
}

struct ScanSmem {
  float s[kR][kD + 1];   // this CTA's rows of the state
  float w[kC][kD + 1];   // W of the chunk
  float qk[kC][kD + 1];  // Q of the chunk, then K
  float p[kC][kC + 1];
  float u[kC][kR + 1];   // U = Ut - W S^T (this CTA's columns)
  float lg[kC], dk[kC];
};

template <typename T>
__global__ void __launch_bounds__(kScanThreads)
    deltanet_scan_kernel(const T* __restrict__ q, const T* __restrict__ k, int T_len, int H,
                         const ChunkRec* __restrict__ ws, const float* __restrict__ S0,
                         T* __restrict__ o, float* __restrict__ S_out) {
  extern __shared__ uint8_t smem_raw[];
  ScanSmem& S = *reinterpret_cast<ScanSmem*>(smem_raw);
  const int blocks = kD / kR;
  const int h = blockIdx.x / blocks, r0 = (blockIdx.x % blocks) * kR;
  const int tid = threadIdx.x;
  const int n_chunks = (T_len + kC - 1) / kC;
  grid_dependency_wait();
  allow_dependents_launch();
  for (int e = tid; e < kR * kD; e += kScanThreads) {
    const int r = e / kD, col = e % kD;
    S.s[r][col] = S0 ? S0[(static_cast<int64_t>(h) * kD + r0 + r) * kD + col] : 0.f;
  }
  for (int c = 0; c < n_chunks; ++c) {
    const ChunkRec& R = ws[static_cast<int64_t>(c) * H + h];
    const int t0 = c * kC;
    const int n = min(kC, T_len - t0);
    __syncthreads();  // the previous chunk is done with w, qk, p, u
    for (int e = tid; e < kC * kD; e += kScanThreads) {
      const int i = e / kD, col = e % kD;
      S.w[i][col] = R.w[i][col];
      S.qk[i][col] = i < n ? ld_val(q, (static_cast<int64_t>(t0 + i) * H + h) * kD + col) : 0.f;
    }
    for (int e = tid; e < kC * kC; e += kScanThreads) S.p[e / kC][e % kC] = R.p[e / kC][e % kC];
    if (tid < kC) {
      S.lg[tid] = R.lg[tid];
      S.dk[tid] = R.dk[tid];
    }
    __syncthreads();
    // U = Ut - W S^T and Z = Q S^T on this CTA's kR columns (4 entries each)
    float z[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int e = tid + m * kScanThreads;
      const int i = e / kR, r = e % kR;
      float y = 0.f, zz = 0.f;
#pragma unroll 8
      for (int col = 0; col < kD; ++col) {
        y = fmaf(S.w[i][col], S.s[r][col], y);
        zz = fmaf(S.qk[i][col], S.s[r][col], zz);
      }
      S.u[i][r] = R.ut[i][r0 + r] - y;
      z[m] = zz;
    }
    __syncthreads();
    // O = diag(g) Q S^T + P U
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int e = tid + m * kScanThreads;
      const int i = e / kR, r = e % kR;
      float acc = __expf(S.lg[i]) * z[m];
      for (int j = 0; j <= i; ++j) acc = fmaf(S.p[i][j], S.u[j][r], acc);
      if (i < n) st_val(o, (static_cast<int64_t>(t0 + i) * H + h) * kD + r0 + r, acc);
    }
    __syncthreads();  // done with qk as Q
    for (int e = tid; e < kC * kD; e += kScanThreads) {
      const int i = e / kD, col = e % kD;
      S.qk[i][col] = i < n ? ld_val(k, (static_cast<int64_t>(t0 + i) * H + h) * kD + col) : 0.f;
    }
    __syncthreads();
    // S <- g_C S + U^T diag(dk) K   (8 entries of S per thread)
    const float gC = __expf(S.lg[kC - 1]);
#pragma unroll
    for (int m = 0; m < kR * kD / kScanThreads; ++m) {
      const int e = tid + m * kScanThreads;
      const int r = e / kD, col = e % kD;
      float acc = gC * S.s[r][col];
      for (int j = 0; j < kC; ++j) acc = fmaf(S.u[j][r] * S.dk[j], S.qk[j][col], acc);
      S.s[r][col] = acc;  // each entry is read and written by this thread only
    }
  }
  __syncthreads();
  if (S_out != nullptr)
    for (int e = tid; e < kR * kD; e += kScanThreads) {
      const int r = e / kD, col = e % kD;
      S_out[(static_cast<int64_t>(h) * kD + r0 + r) * kD + col] = S.s[r][col];
    }
}

template <typename T>
cudaError_t launch_deltanet_t(const void* q, const void* k, const void* v, const float* alpha,
                              const float* beta, int64_t T_len, int H, const float* S0, void* o,
                              float* S_out, void* workspace, cudaStream_t stream) {
  const int n_chunks = static_cast<int>((T_len + kC - 1) / kC);
  ChunkRec* ws = static_cast<ChunkRec*>(workspace);
  const size_t s1 = sizeof(PrepSmem), s2 = sizeof(ScanSmem);
  cudaError_t err = cudaFuncSetAttribute(deltanet_chunk_kernel<T>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(deltanet_scan_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)s2);
  if (err != cudaSuccess) return err;
  err = launch_pdl(deltanet_chunk_kernel<T>, dim3(n_chunks * H), dim3(kPrepThreads), s1, stream,
                   1u, static_cast<const T*>(q), static_cast<const T*>(k),
                   static_cast<const T*>(v), alpha, beta, static_cast<int>(T_len), H, ws);
  if (err != cudaSuccess) return err;
  err = launch_pdl(deltanet_scan_kernel<T>, dim3(H * (kD / kR)), dim3(kScanThreads), s2, stream,
                   1u, static_cast<const T*>(q), static_cast<const T*>(k), static_cast<int>(T_len),
                   H, static_cast<const ChunkRec*>(ws), S0, static_cast<T*>(o), S_out);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace

size_t deltanet_workspace_bytes(int64_t T_len, int H) {
  const int64_t n_chunks = (T_len + kC - 1) / kC;
  return std::max(static_cast<size_t>(n_chunks) * H * sizeof(ChunkRec),
                  deltanet_tc_workspace_bytes(T_len, H));
}

cudaError_t launch_deltanet(const void* q, const void* k, const void* v, int bf16,
                            const float* alpha, const float* beta, int64_t T_len, int H,
                            const float* S0, void* o, float* S_out, void* workspace,
                            cudaStream_t stream) {
  if (T_len == 0) return cudaSuccess;
  if (bf16)  // the tensor-core kernels (deltanet_tc.cu)
    return launch_deltanet_tc(q, k, v, alpha, beta, T_len, H, S0, o, S_out, workspace, stream);
  return launch_deltanet_t<float>(q, k, v, alpha, beta, T_len, H, S0, o, S_out, workspace, stream);
}

}  // namespace tg
