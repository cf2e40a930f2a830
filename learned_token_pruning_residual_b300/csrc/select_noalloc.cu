// tg_select_topk_noalloc: the top-K select for callers that cannot hand the
// library a workspace.  Some hosts own every byte of device memory and let no
// component allocate once they have started (an inference server that plans
// its memory up front, a plug-in inside a framework's allocator, a C caller
// with no allocator to draw a buffer from), and on a latency-critical path an
// allocation is unwelcome anyway: cudaMalloc can synchronise the device and
// cudaFree does.  This entry point allocates nothing.  Its scratch is the
// file-scope array below, which every GPU that loads this library holds (104
// KiB) until the process exits.
//
// The array is per device.  Its device address is looked up once per device,
// on the first call made while that device is current (cudaGetSymbolAddress);
// that first call should therefore not be made inside a stream capture.  In
// host code the array's name is only a host-side stand-in and must never be
// passed to a kernel: the looked-up address is what the kernels get.
//
// Every call shares the one array and finds it as the last call left it: each
// call clears the part that must start at zero (cudaMemsetAsync on the
// caller's stream) before the select kernel runs, so a call that an error interrupted does not poison the next
// one.  Calls that overlap on the GPU (on different streams, or concurrent
// host threads with one device) race on the array and must not be made.
#include <cuda_runtime.h>

#include <mutex>

#include "tg_device.cuh"
#include "tg_internal.h"

namespace tg {
namespace {

constexpr size_t kNoAllocScratchBytes = kSelectWorkspaceBytes;  // 104 KiB
static_assert(sizeof(SelectWorkspace) <= kNoAllocScratchBytes, "scratch holds a select workspace");

// The scratch of tg_select_topk_noalloc (one copy per device).
static __device__ __align__(256) uint8_t g_select_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// The device address of this device's scratch array, looked up on first use.
cudaError_t scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_select_scratch);
    if (e != cudaSuccess) return e;
    if (p == nullptr || (reinterpret_cast<uintptr_t>(p) & 255u) != 0) return cudaErrorInvalidValue;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace tg

extern "C" tg_status tg_select_topk_noalloc(const float* scores, int64_t N, int64_t doc_begin,
                                            int64_t doc_end, int64_t K, int32_t* kept_idx,
                                            int64_t* M_out, tg_stream_t stream) {
  if (!(N >= 0 && N < (int64_t(1) << 31)))
    return tg::fail(TG_ERR_INVALID_ARG, "select noalloc: N out of range");
  if (!(0 <= doc_begin && doc_begin <= doc_end && doc_end <= N))
    return tg::fail(TG_ERR_INVALID_ARG, "select noalloc: need 0 <= doc_begin <= doc_end <= N");
  if (!(0 <= K && K <= doc_end - doc_begin))
    return tg::fail(TG_ERR_INVALID_ARG, "select noalloc: need 0 <= K <= doc_end - doc_begin");
  // the scratch this call needs must fit the fixed array
  if (tg_select_workspace_bytes(N) > tg::kNoAllocScratchBytes)
    return tg::fail(TG_ERR_UNSUPPORTED,
                    "select noalloc: N = %lld needs %zu bytes of scratch, more than the %zu-byte "
                    "array", static_cast<long long>(N), tg_select_workspace_bytes(N),
                    tg::kNoAllocScratchBytes);
  const int64_t M = N - (doc_end - doc_begin) + K;
  if (M_out) *M_out = M;
  if (M == 0) return TG_OK;  // nothing to write: nothing is launched
  if (!scores || !kept_idx) return tg::fail(TG_ERR_INVALID_ARG, "select noalloc: NULL pointer");
  if ((reinterpret_cast<uintptr_t>(scores) & 15u) || (reinterpret_cast<uintptr_t>(kept_idx) & 15u))
    return tg::fail(TG_ERR_INVALID_ARG, "select noalloc: pointers must be 16-byte aligned");
  void* ws = nullptr;
  cudaError_t e = tg::scratch_address(&ws);
  if (e != cudaSuccess)
    return tg::fail(TG_ERR_CUDA, "select noalloc: scratch address: %s", cudaGetErrorString(e));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  e = cudaMemsetAsync(ws, 0, tg::kSelectZeroedBytes, st);  // the candidate area needs no clearing
  if (e == cudaSuccess)
    e = tg::launch_select(scores, N, doc_begin, doc_end, K, kept_idx,
                          static_cast<tg::SelectWorkspace*>(ws), st);
  if (e != cudaSuccess)
    return tg::fail(TG_ERR_CUDA, "select noalloc: %s", cudaGetErrorString(e));
  return TG_OK;
}
