// The C ABI of libtokengate.so: argument checks, the sticky device status
// word, tensor-map encoding, and dispatch to the kernels.  Every check that
// can fail happens here, before anything is launched.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <nvtx3/nvToolsExt.h>

#include <mutex>

#include "tg_device.cuh"
#include "tg_internal.h"

namespace tg {

// The sticky per-device status word.  Kernels OR error bits into it;
// tg_get_device_status reads and clears it.
__device__ uint32_t g_status_word = 0;
// Where tg_get_device_status takes the word to (read and cleared in one
// atomic exchange, so a bit that a kernel on another stream sets at the same
// time is either taken now or left for the next read, never lost).
__device__ uint32_t g_status_taken = 0;

__global__ void status_take_kernel(uint32_t* status, uint32_t* taken) {
  *taken = atomicExch(status, 0u);
}

namespace {
thread_local char t_last_error[512] = "";
constexpr int kMaxDevices = 64;
uint32_t* g_status_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
std::mutex g_mu;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool load_encode() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return false;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return true;
}

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return dev;
}
}  // namespace

tg_status fail(tg_status code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
  va_end(ap);
  return code;
}

uint32_t* device_status_word() {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<uint32_t*>(p);
  }
  return g_status_ptr[dev];
}

cudaError_t launch_status_take(uint32_t** taken, cudaStream_t stream) {
  uint32_t* status = device_status_word();
  if (status == nullptr) return cudaErrorInvalidDevice;
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_status_taken);
  if (e != cudaSuccess) return e;
  *taken = static_cast<uint32_t*>(p);
  status_take_kernel<<<1, 1, 0, stream>>>(status, *taken);
  return cudaGetLastError();
}

int sm_count() {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return 1;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sms[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    g_sms[dev] = n > 0 ? n : 1;
  }
  return g_sms[dev];
}

bool make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem_bytes,
                  uint64_t cols, uint64_t rows, uint64_t row_bytes, uint32_t box_cols,
                  uint32_t box_rows, CUtensorMapSwizzle swizzle) {
  (void)elem_bytes;
  if (!load_encode()) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_1d_f32(CUtensorMap* map, const float* base, uint64_t n, uint32_t box) {
  if (!load_encode()) return false;
  const cuuint64_t dims[1] = {n};
  const cuuint64_t strides[1] = {n * 4};
  const cuuint32_t boxd[1] = {box};
  const cuuint32_t estr[1] = {1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 1, const_cast<float*>(base), dims,
                  strides, boxd, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tg

using tg::fail;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

tg_status from_cuda(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return TG_OK;
  return fail(TG_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// An NVTX range around one C-ABI call (named after the call), so that
// profilers show which call launched which kernels (e.g. ncu --nvtx
// --nvtx-include "tg_keybias_attn/"); a no-op unless a tool is attached.
struct CallRange {
  explicit CallRange(const char* name) { nvtxRangePushA(name); }
  ~CallRange() { nvtxRangePop(); }
  CallRange(const CallRange&) = delete;
  CallRange& operator=(const CallRange&) = delete;
};
#define TG_TRACE_CALL() CallRange tg_call_range_(__func__)

#define TG_REQUIRE(cond, code, ...) \
  do {                              \
    if (!(cond)) return fail(code, __VA_ARGS__); \
  } while (0)

// Token-gated attention, optionally writing the per-row log-sum-exp.
tg_status keybias_attn_impl(const void* QKV, tg_dtype dtype, int64_t M, int32_t Hq, int32_t Hkv,
                            int32_t dh, const float* logsig_kept, const float* gain,
                            float temperature, void* O, float* residual, float* lse,
                            tg_stream_t stream) {
  TG_REQUIRE(dtype == TG_F32 || dtype == TG_BF16, TG_ERR_INVALID_ARG, "attn: bad dtype");
  TG_REQUIRE(M >= 0 && M < (int64_t(1) << 31) && Hq > 0 && Hkv > 0 && dh > 0,
             TG_ERR_INVALID_ARG, "attn: bad sizes");
  TG_REQUIRE(Hq % Hkv == 0, TG_ERR_INVALID_ARG, "attn: Hq %% Hkv != 0");
  TG_REQUIRE(temperature == temperature, TG_ERR_INVALID_ARG, "attn: temperature is NaN");
  if (M == 0) return TG_OK;
  TG_REQUIRE(QKV && (O || residual), TG_ERR_INVALID_ARG, "attn: NULL pointer");
  TG_REQUIRE(!logsig_kept || gain, TG_ERR_INVALID_ARG, "attn: gain needed with a bias");
  TG_REQUIRE(aligned16(QKV) && (!O || aligned16(O)) && (!residual || aligned16(residual)) &&
                 (!logsig_kept || aligned16(logsig_kept)) && (!lse || aligned16(lse)),
             TG_ERR_INVALID_ARG, "attn: pointers must be 16-byte aligned");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == TG_BF16) {
    TG_REQUIRE(dh == 128, TG_ERR_UNSUPPORTED, "attn bf16: dh must be 128");
    TG_REQUIRE((Hq / Hkv) % 2 == 0, TG_ERR_UNSUPPORTED, "attn bf16: Hq / Hkv must be even");
    TG_REQUIRE(temperature > 0.f && temperature <= 3.0e38f, TG_ERR_UNSUPPORTED,
               "attn bf16: temperature must be finite and > 0");
    return from_cuda(tg::launch_attn_bf16(QKV, M, Hq, Hkv, dh, logsig_kept, gain, temperature, O,
                                          residual, lse, st),
                     "attn bf16");
  }
  TG_REQUIRE(dh == 32 || dh == 64 || dh == 128, TG_ERR_UNSUPPORTED,
             "attn f32: dh must be 32, 64 or 128");
  return from_cuda(tg::launch_attn_f32(static_cast<const float*>(QKV), M, Hq, Hkv, dh,
                                       logsig_kept, gain, temperature, static_cast<float*>(O),
                                       residual, lse, st),
                   "attn f32");
}

}  // namespace

extern "C" {

const char* tg_status_string(int status) {
  switch (status) {
    case TG_OK: return "TG_OK";
    case TG_ERR_INVALID_ARG: return "TG_ERR_INVALID_ARG";
    case TG_ERR_UNSUPPORTED: return "TG_ERR_UNSUPPORTED";
    case TG_ERR_CUDA: return "TG_ERR_CUDA";
    case TG_ERR_NAN_SCORE: return "TG_ERR_NAN_SCORE";
    case TG_ERR_BAD_INDEX: return "TG_ERR_BAD_INDEX";
    case TG_ERR_TIMEOUT: return "TG_ERR_TIMEOUT";
    default: return "TG_ERR_UNKNOWN";
  }
}

int tg_abi_version(void) { return TG_ABI_VERSION; }

const char* tg_last_error_message(void) { return tg::t_last_error; }

tg_status tg_gate_score(const void* X, tg_dtype dtype, int64_t N, int32_t d, const void* W1,
                        const float* b1, int32_t Hg, const float* w2, float b2, float* scores,
                        void* select_ws, int64_t doc_begin, int64_t doc_end, tg_stream_t stream) {
  TG_TRACE_CALL();
  TG_REQUIRE(dtype == TG_F32 || dtype == TG_BF16, TG_ERR_INVALID_ARG, "gate: bad dtype");
  TG_REQUIRE(N >= 0 && N < (int64_t(1) << 31), TG_ERR_INVALID_ARG, "gate: N out of range");
  TG_REQUIRE(d > 0 && Hg > 0, TG_ERR_INVALID_ARG, "gate: d and Hg must be positive");
  TG_REQUIRE(!select_ws || (0 <= doc_begin && doc_begin <= doc_end && doc_end <= N),
             TG_ERR_INVALID_ARG, "gate: need 0 <= doc_begin <= doc_end <= N with a workspace");
  TG_REQUIRE(!select_ws || (reinterpret_cast<uintptr_t>(select_ws) & 255u) == 0,
             TG_ERR_INVALID_ARG, "gate: select workspace must be 256-byte aligned");
  if (N == 0) return TG_OK;
  TG_REQUIRE(X && W1 && w2 && scores, TG_ERR_INVALID_ARG, "gate: NULL pointer");
  TG_REQUIRE(aligned16(X) && aligned16(W1) && aligned16(w2) && aligned16(scores) &&
                 (!b1 || aligned16(b1)),
             TG_ERR_INVALID_ARG, "gate: pointers must be 16-byte aligned");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == TG_BF16) {
    TG_REQUIRE(d % 64 == 0, TG_ERR_UNSUPPORTED, "gate bf16: d %% 64 != 0 (d=%d)", d);
    TG_REQUIRE(Hg >= 16 && Hg <= 256 && Hg % 16 == 0, TG_ERR_UNSUPPORTED,
               "gate bf16: need 16 <= Hg <= 256, Hg %% 16 == 0 (Hg=%d)", Hg);
    return from_cuda(tg::launch_gate_bf16(X, N, d, W1, b1, Hg, w2, b2, scores,
                                          static_cast<tg::SelectWorkspace*>(select_ws), doc_begin,
                                          doc_end, st),
                     "gate bf16");
  }
  TG_REQUIRE(d % 4 == 0, TG_ERR_UNSUPPORTED, "gate f32: d %% 4 != 0");
  TG_REQUIRE(Hg <= 1024, TG_ERR_UNSUPPORTED, "gate f32: Hg > 1024");
  TG_REQUIRE(static_cast<int64_t>(d) * 4 <= 200 * 1024, TG_ERR_UNSUPPORTED, "gate f32: d too big");
  // the fp32 path does not fill the histogram: the select then runs its own
  // first pass (the workspace header stays unstamped)
  return from_cuda(tg::launch_gate_f32(static_cast<const float*>(X), N, d,
                                       static_cast<const float*>(W1), b1, Hg, w2, b2, scores, st),
                   "gate f32");
}

size_t tg_select_workspace_bytes(int64_t N) {
  (void)N;
  return tg::kSelectWorkspaceBytes;
}

tg_status tg_select_topk(const float* scores, int64_t N, int64_t doc_begin, int64_t doc_end,
                         int64_t K, int32_t* kept_idx, int64_t* M_out, void* workspace,
                         size_t workspace_bytes, tg_stream_t stream) {
  TG_TRACE_CALL();
  TG_REQUIRE(N >= 0 && N < (int64_t(1) << 31), TG_ERR_INVALID_ARG, "select: N out of range");
  TG_REQUIRE(0 <= doc_begin && doc_begin <= doc_end && doc_end <= N, TG_ERR_INVALID_ARG,
             "select: need 0 <= doc_begin <= doc_end <= N");
  TG_REQUIRE(0 <= K && K <= doc_end - doc_begin, TG_ERR_INVALID_ARG,
             "select: need 0 <= K <= doc_end - doc_begin");
  const int64_t M = N - (doc_end - doc_begin) + K;
  if (M_out) *M_out = M;
  if (M == 0) return TG_OK;  // nothing to write: nothing is launched
  TG_REQUIRE(scores && kept_idx, TG_ERR_INVALID_ARG, "select: NULL pointer");
  TG_REQUIRE(aligned16(scores) && aligned16(kept_idx), TG_ERR_INVALID_ARG,
             "select: pointers must be 16-byte aligned");
  TG_REQUIRE(workspace != nullptr && workspace_bytes >= tg::kSelectWorkspaceBytes,
             TG_ERR_INVALID_ARG, "select: need a workspace of tg_select_workspace_bytes() bytes");
  TG_REQUIRE((reinterpret_cast<uintptr_t>(workspace) & 255u) == 0, TG_ERR_INVALID_ARG,
             "select: workspace must be 256-byte aligned");
  return from_cuda(tg::launch_select(scores, N, doc_begin, doc_end, K, kept_idx,
                                     static_cast<tg::SelectWorkspace*>(workspace),
                                     reinterpret_cast<cudaStream_t>(stream)),
                   "select");
}

tg_status tg_gather_rows(const void* X, tg_dtype x_dtype, int64_t N, int32_t d,
                         const int32_t* idx, int64_t M, void* Y, tg_dtype y_dtype,
                         const float* scores, float* logsig_kept, tg_stream_t stream) {
  TG_TRACE_CALL();
  TG_REQUIRE((x_dtype == TG_BF16 && (y_dtype == TG_BF16 || y_dtype == TG_F32)) ||
                 (x_dtype == TG_F32 && y_dtype == TG_F32),
             TG_ERR_UNSUPPORTED, "gather: dtype pair not supported");
  TG_REQUIRE(N >= 0 && M >= 0 && d > 0, TG_ERR_INVALID_ARG, "gather: bad sizes");
  if (M == 0) return TG_OK;
  TG_REQUIRE(idx != nullptr || M == N, TG_ERR_INVALID_ARG, "gather: idx NULL needs M == N");
  TG_REQUIRE((scores == nullptr) == (logsig_kept == nullptr), TG_ERR_INVALID_ARG,
             "gather: scores and logsig_kept must both be given or both NULL");
  const int64_t in_row = static_cast<int64_t>(d) * (x_dtype == TG_BF16 ? 2 : 4);
  TG_REQUIRE(in_row % 16 == 0, TG_ERR_INVALID_ARG, "gather: row bytes must be a multiple of 16");
  TG_REQUIRE(X && Y, TG_ERR_INVALID_ARG, "gather: NULL pointer");
  TG_REQUIRE(aligned16(X) && aligned16(Y) && (!idx || aligned16(idx)) &&
                 (!scores || aligned16(scores)) && (!logsig_kept || aligned16(logsig_kept)),
             TG_ERR_INVALID_ARG, "gather: pointers must be 16-byte aligned");
  return from_cuda(tg::launch_gather(X, x_dtype == TG_BF16, N, d, idx, M, Y, y_dtype == TG_BF16,
                                     scores, logsig_kept, reinterpret_cast<cudaStream_t>(stream)),
                   "gather");
}

tg_status tg_rmsnorm(const void* X, tg_dtype x_dtype, int64_t M, int32_t d, const float* gamma,
                     float eps, void* Y, tg_dtype y_dtype, tg_stream_t stream) {
  TG_TRACE_CALL();
  TG_REQUIRE((x_dtype == TG_F32 || x_dtype == TG_BF16) && (y_dtype == TG_F32 || y_dtype == TG_BF16),
             TG_ERR_INVALID_ARG, "rmsnorm: bad dtype");
  TG_REQUIRE(M >= 0 && d > 0 && d % 8 == 0, TG_ERR_INVALID_ARG, "rmsnorm: need d %% 8 == 0");
  TG_REQUIRE(eps >= 0.f, TG_ERR_INVALID_ARG, "rmsnorm: eps < 0");
  if (M == 0) return TG_OK;
  TG_REQUIRE(X && Y && gamma, TG_ERR_INVALID_ARG, "rmsnorm: NULL pointer");
  TG_REQUIRE(aligned16(X) && aligned16(Y) && aligned16(gamma), TG_ERR_INVALID_ARG,
             "rmsnorm: pointers must be 16-byte aligned");
  return from_cuda(tg::launch_rmsnorm(X, x_dtype == TG_BF16, M, d, gamma, eps, Y,
                                      y_dtype == TG_BF16, reinterpret_cast<cudaStream_t>(stream)),
                   "rmsnorm");
}

tg_status tg_qkv_proj(const void* X, tg_dtype dtype, int64_t M, int32_t d, const void* Wqkv,
                      int32_t Hq, int32_t Hkv, int32_t dh, void* QKV, tg_stream_t stream) {
  TG_TRACE_CALL();
  TG_REQUIRE(dtype == TG_F32 || dtype == TG_BF16, TG_ERR_INVALID_ARG, "qkv: bad dtype");
  TG_REQUIRE(M >= 0 && M < (int64_t(1) << 31) && d > 0 && Hq > 0 && Hkv > 0 && dh > 0,
             TG_ERR_INVALID_ARG, "qkv: bad sizes");
  const int64_t cols = static_cast<int64_t>(Hq + 2 * Hkv) * dh;
  TG_REQUIRE(cols < (int64_t(1) << 20), TG_ERR_INVALID_ARG, "qkv: too many columns");
  if (M == 0) return TG_OK;
  TG_REQUIRE(X && Wqkv && QKV, TG_ERR_INVALID_ARG, "qkv: NULL pointer");
  TG_REQUIRE(aligned16(X) && aligned16(Wqkv) && aligned16(QKV), TG_ERR_INVALID_ARG,
             "qkv: pointers must be 16-byte aligned");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == TG_BF16) {
    TG_REQUIRE(d % 64 == 0, TG_ERR_UNSUPPORTED, "qkv bf16: d %% 64 != 0");
    TG_REQUIRE(cols % 16 == 0, TG_ERR_UNSUPPORTED, "qkv bf16: output columns %% 16 != 0");
    return from_cuda(tg::launch_qkv_bf16(X, M, d, Wqkv, static_cast<int>(cols), QKV, st),
                     "qkv bf16");
  }
  TG_REQUIRE(d % 4 == 0, TG_ERR_UNSUPPORTED, "qkv f32: d %% 4 != 0");
  return from_cuda(tg::launch_qkv_f32(static_cast<const float*>(X), M, d,
                                      static_cast<const float*>(Wqkv), static_cast<int>(cols),
                                      static_cast<float*>(QKV), st),
                   "qkv f32");
}

tg_status tg_rope_table(const int32_t* positions, int64_t M, int32_t dh, double base,
                        float* table, tg_stream_t stream) {
  TG_TRACE_CALL();
  TG_REQUIRE(M >= 0 && M < (int64_t(1) << 31), TG_ERR_INVALID_ARG, "rope table: bad M");
  TG_REQUIRE(dh > 0 && dh % 2 == 0 && dh <= 1024, TG_ERR_INVALID_ARG,
             "rope table: dh must be even, 2..1024");
  TG_REQUIRE(base > 1.0 && base < 1e300, TG_ERR_INVALID_ARG, "rope table: need base > 1");
  if (M == 0) return TG_OK;
  TG_REQUIRE(positions && table, TG_ERR_INVALID_ARG, "rope table: NULL pointer");
  TG_REQUIRE(aligned16(positions) && aligned16(table), TG_ERR_INVALID_ARG,
             "rope table: pointers must be 16-byte aligned");
  return from_cuda(tg::launch_rope_table(positions, M, dh, base, reinterpret_cast<float2*>(table),
                                         reinterpret_cast<cudaStream_t>(stream)),
                   "rope table");
}

tg_status tg_qkv_proj_qknorm_rope(const void* X, int64_t M, int32_t d, const void* Wqkv,
                                  int32_t Hq, int32_t Hkv, int32_t dh, const float* gamma_q,
                                  const float* gamma_k, float eps, const float* rope_table,
                                  void* QKV, tg_stream_t stream) {
  TG_TRACE_CALL();
  TG_REQUIRE(M >= 0 && M < (int64_t(1) << 31) && d > 0 && Hq > 0 && Hkv > 0,
             TG_ERR_INVALID_ARG, "qkv rope: bad sizes");
  TG_REQUIRE(eps >= 0.f, TG_ERR_INVALID_ARG, "qkv rope: eps < 0");
  TG_REQUIRE(dh == 128, TG_ERR_UNSUPPORTED, "qkv rope: dh must be 128");
  TG_REQUIRE(d % 64 == 0, TG_ERR_UNSUPPORTED, "qkv rope: d %% 64 != 0");
  TG_REQUIRE(static_cast<int64_t>(Hq + 2 * Hkv) * dh < (int64_t(1) << 20), TG_ERR_INVALID_ARG,
             "qkv rope: too many columns");
  if (M == 0) return TG_OK;
  TG_REQUIRE(X && Wqkv && gamma_q && gamma_k && rope_table && QKV, TG_ERR_INVALID_ARG,
             "qkv rope: NULL pointer");
  TG_REQUIRE(aligned16(X) && aligned16(Wqkv) && aligned16(QKV) && aligned16(rope_table),
             TG_ERR_INVALID_ARG, "qkv rope: pointers must be 16-byte aligned");
  return from_cuda(tg::launch_qkv_qknorm_rope_bf16(
                       X, M, d, Wqkv, Hq, Hkv, gamma_q, gamma_k, eps,
                       reinterpret_cast<const float2*>(rope_table), QKV,
                       reinterpret_cast<cudaStream_t>(stream)),
                   "qkv rope");
}

tg_status tg_linear_residual(const void* X, int64_t M, int32_t K, const void* W, int32_t N,
                             float* residual, tg_stream_t stream) {
  TG_TRACE_CALL();
  TG_REQUIRE(M >= 0 && M < (int64_t(1) << 31) && K > 0 && N > 0, TG_ERR_INVALID_ARG,
             "linear residual: bad sizes");
  TG_REQUIRE(K % 64 == 0 && N % 32 == 0, TG_ERR_UNSUPPORTED,
             "linear residual: need K %% 64 == 0 and N %% 32 == 0");
  if (M == 0) return TG_OK;
  TG_REQUIRE(X && W && residual, TG_ERR_INVALID_ARG, "linear residual: NULL pointer");
  TG_REQUIRE(aligned16(X) && aligned16(W) && aligned16(residual), TG_ERR_INVALID_ARG,
             "linear residual: pointers must be 16-byte aligned");
  return from_cuda(tg::launch_linear_resid_bf16(X, M, K, W, N, residual,
                                                reinterpret_cast<cudaStream_t>(stream)),
                   "linear residual");
}

tg_status tg_swiglu(const void* X, int64_t M, int32_t d, const void* W_gate, const void* W_up,
                    int32_t F, void* Y, tg_stream_t stream) {
  TG_TRACE_CALL();
  TG_REQUIRE(M >= 0 && M < (int64_t(1) << 31) && d > 0 && F > 0, TG_ERR_INVALID_ARG,
             "swiglu: bad sizes");
  TG_REQUIRE(d % 64 == 0 && F % 32 == 0 && F <= (1 << 24), TG_ERR_UNSUPPORTED,
             "swiglu: need d %% 64 == 0 and F %% 32 == 0");
  if (M == 0) return TG_OK;
  TG_REQUIRE(X && W_gate && W_up && Y, TG_ERR_INVALID_ARG, "swiglu: NULL pointer");
  TG_REQUIRE(aligned16(X) && aligned16(W_gate) && aligned16(W_up) && aligned16(Y),
             TG_ERR_INVALID_ARG, "swiglu: pointers must be 16-byte aligned");
  return from_cuda(tg::launch_swiglu_bf16(X, M, d, W_gate, W_up, F, Y,
                                          reinterpret_cast<cudaStream_t>(stream)),
                   "swiglu");
}

size_t tg_gated_delta_rule_workspace_bytes(int64_t T, int32_t H) {
  if (T < 0 || H <= 0) return 0;
  return tg::deltanet_workspace_bytes(T, H);
}

tg_status tg_gated_delta_rule(const void* q, const void* k, const void* v, tg_dtype dtype,
                              const float* alpha, const float* beta, int64_t T, int32_t H,
                              int32_t dk, int32_t dv, const float* S0, void* o, float* S_out,
                              void* workspace, size_t workspace_bytes, tg_stream_t stream) {
  TG_TRACE_CALL();
  TG_REQUIRE(dtype == TG_F32 || dtype == TG_BF16, TG_ERR_INVALID_ARG, "delta rule: bad dtype");
  TG_REQUIRE(T >= 0 && T < (int64_t(1) << 31) && H > 0 && H <= 4096, TG_ERR_INVALID_ARG,
             "delta rule: bad sizes");
  TG_REQUIRE(dk == 128 && dv == 128, TG_ERR_UNSUPPORTED, "delta rule: need dk == dv == 128");
  TG_REQUIRE(T * H * 128 < (int64_t(1) << 40), TG_ERR_UNSUPPORTED, "delta rule: too large");
  if (T == 0) return TG_OK;
  TG_REQUIRE(q && k && v && alpha && beta && o && workspace, TG_ERR_INVALID_ARG,
             "delta rule: NULL pointer");
  TG_REQUIRE(workspace_bytes >= tg::deltanet_workspace_bytes(T, H), TG_ERR_INVALID_ARG,
             "delta rule: workspace smaller than tg_gated_delta_rule_workspace_bytes(T, H)");
  TG_REQUIRE(aligned16(q) && aligned16(k) && aligned16(v) && aligned16(alpha) &&
                 aligned16(beta) && aligned16(o) && aligned16(workspace) &&
                 (!S0 || aligned16(S0)) && (!S_out || aligned16(S_out)),
             TG_ERR_INVALID_ARG, "delta rule: pointers must be 16-byte aligned");
  return from_cuda(tg::launch_deltanet(q, k, v, dtype == TG_BF16, alpha, beta, T, H, S0, o, S_out,
                                       workspace, reinterpret_cast<cudaStream_t>(stream)),
                   "delta rule");
}

tg_status tg_keybias_attn(const void* QKV, tg_dtype dtype, int64_t M, int32_t Hq, int32_t Hkv,
                          int32_t dh, const float* logsig_kept, const float* gain,
                          float temperature, void* O, float* residual, tg_stream_t stream) {
  TG_TRACE_CALL();
  return keybias_attn_impl(QKV, dtype, M, Hq, Hkv, dh, logsig_kept, gain, temperature, O,
                           residual, nullptr, stream);
}

tg_status tg_keybias_attn_lse(const void* QKV, tg_dtype dtype, int64_t M, int32_t Hq,
                              int32_t Hkv, int32_t dh, const float* logsig_kept,
                              const float* gain, float temperature, void* O, float* residual,
                              float* lse, tg_stream_t stream) {
  TG_TRACE_CALL();
  TG_REQUIRE(lse || M == 0, TG_ERR_INVALID_ARG, "attn lse: NULL lse");
  return keybias_attn_impl(QKV, dtype, M, Hq, Hkv, dh, logsig_kept, gain, temperature, O,
                           residual, lse, stream);
}

tg_status tg_attn_bwd_delta(const void* dO, const void* O, tg_dtype dtype, int64_t M, int32_t Hq,
                            int32_t dh, float* delta, tg_stream_t stream) {
  TG_TRACE_CALL();
  TG_REQUIRE(dtype == TG_F32 || dtype == TG_BF16, TG_ERR_INVALID_ARG, "delta: bad dtype");
  TG_REQUIRE(M >= 0 && M < (int64_t(1) << 31) && Hq > 0 && dh > 0, TG_ERR_INVALID_ARG,
             "delta: bad sizes");
  TG_REQUIRE(dtype == TG_BF16 ? (dh == 64 || dh == 128 || dh == 256)
                              : (dh == 32 || dh == 64 || dh == 128),
             TG_ERR_UNSUPPORTED, "delta: dh must be 64, 128 or 256 (bf16), 32, 64 or 128 (f32)");
  // one thread per 16-byte chunk, 256 a block: the grid must fit in 2^31 - 1.
  // With M < 2^31, Hq <= 2^16 and at most 32 chunks a head the product stays
  // below 2^52, so it cannot overflow.
  TG_REQUIRE(Hq <= 65536, TG_ERR_UNSUPPORTED, "delta: Hq > 65536");
  TG_REQUIRE(M * Hq * (dh * (dtype == TG_BF16 ? 2 : 4) / 16) / 256 < (int64_t(1) << 31) - 1,
             TG_ERR_UNSUPPORTED, "delta: M * Hq too large");
  if (M == 0) return TG_OK;
  TG_REQUIRE(dO && O && delta, TG_ERR_INVALID_ARG, "delta: NULL pointer");
  TG_REQUIRE(aligned16(dO) && aligned16(O) && aligned16(delta), TG_ERR_INVALID_ARG,
             "delta: pointers must be 16-byte aligned");
  return from_cuda(tg::launch_attn_delta(dO, O, dtype == TG_BF16, M, Hq, dh, delta,
                                         reinterpret_cast<cudaStream_t>(stream)),
                   "delta");
}

tg_status tg_keybias_attn_bias_grad(const void* QKV, const void* dO, tg_dtype dtype, int64_t M,
                                    int32_t Hq, int32_t Hkv, int32_t dh,
                                    const float* logsig_kept, const float* gain,
                                    float temperature, const float* lse, const float* delta,
                                    float* dbias, tg_stream_t stream) {
  TG_TRACE_CALL();
  TG_REQUIRE(dtype == TG_F32 || dtype == TG_BF16, TG_ERR_INVALID_ARG, "bias grad: bad dtype");
  TG_REQUIRE(M >= 0 && M < (int64_t(1) << 31) && Hq > 0 && Hkv > 0 && dh > 0,
             TG_ERR_INVALID_ARG, "bias grad: bad sizes");
  TG_REQUIRE(Hq % Hkv == 0, TG_ERR_INVALID_ARG, "bias grad: Hq %% Hkv != 0");
  TG_REQUIRE(temperature == temperature && temperature <= 3.0e38f && temperature >= -3.0e38f,
             TG_ERR_INVALID_ARG, "bias grad: temperature must be finite");
  if (M == 0) return TG_OK;
  TG_REQUIRE(QKV && dO && lse && delta && dbias, TG_ERR_INVALID_ARG, "bias grad: NULL pointer");
  TG_REQUIRE(!logsig_kept || gain, TG_ERR_INVALID_ARG, "bias grad: gain needed with a bias");
  TG_REQUIRE(aligned16(QKV) && aligned16(dO) && aligned16(lse) && aligned16(delta) &&
                 aligned16(dbias) && (!logsig_kept || aligned16(logsig_kept)),
             TG_ERR_INVALID_ARG, "bias grad: pointers must be 16-byte aligned");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == TG_BF16) {
    TG_REQUIRE(dh == 128, TG_ERR_UNSUPPORTED, "bias grad bf16: dh must be 128");
    TG_REQUIRE((M + 127) / 128 * Hq < (int64_t(1) << 31) - 1, TG_ERR_UNSUPPORTED,
               "bias grad bf16: (M / 128) * Hq blocks exceed the grid limit");
    return from_cuda(tg::launch_bias_grad_bf16(QKV, dO, M, Hq, Hkv, dh, logsig_kept, gain,
                                               temperature, lse, delta, dbias, st),
                     "bias grad bf16");
  }
  TG_REQUIRE(dh == 32 || dh == 64 || dh == 128, TG_ERR_UNSUPPORTED,
             "bias grad f32: dh must be 32, 64 or 128");
  return from_cuda(tg::launch_bias_grad_f32(static_cast<const float*>(QKV),
                                            static_cast<const float*>(dO), M, Hq, Hkv, dh,
                                            logsig_kept, gain, temperature, lse, delta, dbias,
                                            st),
                   "bias grad f32");
}

tg_status tg_bias_grad_reduce(const float* dbias, int64_t M, int32_t Hq,
                              const float* logsig_kept, const float* gain, float* dlogsig,
                              float* dgain, float* dscore, tg_stream_t stream) {
  TG_TRACE_CALL();
  TG_REQUIRE(M >= 0 && M < (int64_t(1) << 31) && Hq > 0, TG_ERR_INVALID_ARG,
             "bias grad reduce: bad sizes");
  TG_REQUIRE(dgain && gain, TG_ERR_INVALID_ARG, "bias grad reduce: NULL pointer");
  TG_REQUIRE(M == 0 || (dbias && logsig_kept && dlogsig), TG_ERR_INVALID_ARG,
             "bias grad reduce: NULL pointer");
  TG_REQUIRE(aligned16(dgain) && aligned16(gain) && (M == 0 || (aligned16(dbias) &&
             aligned16(logsig_kept) && aligned16(dlogsig))) && (!dscore || aligned16(dscore)),
             TG_ERR_INVALID_ARG, "bias grad reduce: pointers must be 16-byte aligned");
  return from_cuda(tg::launch_bias_grad_reduce(dbias, M, Hq, logsig_kept, gain, dlogsig, dgain,
                                               dscore, reinterpret_cast<cudaStream_t>(stream)),
                   "bias grad reduce");
}

tg_status tg_get_device_status(tg_stream_t stream) {
  static std::mutex take_mu;  // one taker at a time per process (one g_status_taken per device)
  std::lock_guard<std::mutex> lk(take_mu);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return fail(TG_ERR_CUDA, "status: %s", cudaGetErrorString(e));
  uint32_t* taken = nullptr;
  e = tg::launch_status_take(&taken, st);
  if (e != cudaSuccess) return fail(TG_ERR_CUDA, "status: %s", cudaGetErrorString(e));
  uint32_t v = 0;
  e = cudaMemcpyAsync(&v, taken, sizeof(v), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return fail(TG_ERR_CUDA, "status: %s", cudaGetErrorString(e));
  if (v & tg::kStatusNanScore) return TG_ERR_NAN_SCORE;
  if (v & tg::kStatusBadIndex) return TG_ERR_BAD_INDEX;
  if (v & tg::kStatusTimeout) return TG_ERR_TIMEOUT;
  return TG_OK;
}

tg_status tg_selftest_bounded_wait(uint32_t timeout_us, unsigned long long* report,
                                   tg_stream_t stream) {
  TG_TRACE_CALL();
  TG_REQUIRE(timeout_us >= 1 && timeout_us <= 1000000, TG_ERR_INVALID_ARG,
             "selftest: need 1 <= timeout_us <= 1000000");
  TG_REQUIRE(!report || (reinterpret_cast<uintptr_t>(report) & 7u) == 0, TG_ERR_INVALID_ARG,
             "selftest: report must be 8-byte aligned");
  return from_cuda(tg::launch_bounded_wait_selftest(static_cast<uint64_t>(timeout_us) * 1000ull,
                                                    report,
                                                    reinterpret_cast<cudaStream_t>(stream)),
                   "selftest");
}

}  // extern "C"
