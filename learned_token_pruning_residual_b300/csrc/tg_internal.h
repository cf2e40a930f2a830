// Host-side declarations shared by the library's translation units: kernel
// launchers, tensor-map helpers and error reporting.
#pragma once

#include <cstddef>

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "tokengate.h"

namespace tg {

// Records a message for tg_last_error_message() and returns `code`.
tg_status fail(tg_status code, const char* fmt, ...);

// Device address of the sticky status word on the current device.
uint32_t* device_status_word();

// Streaming multiprocessors of the current device (cached per device).
int sm_count();

// 2-D tiled tensor map over a row-major matrix [rows][cols] of `elem_bytes`
// elements whose rows are `row_bytes` apart; box = box_cols x box_rows.
bool make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem_bytes,
                  uint64_t cols, uint64_t rows, uint64_t row_bytes, uint32_t box_cols,
                  uint32_t box_rows, CUtensorMapSwizzle swizzle);
// 1-D tiled tensor map over a vector of `n` fp32 values, box of `box` values.
bool make_tmap_1d_f32(CUtensorMap* map, const float* base, uint64_t n, uint32_t box);

// Launches `kernel` on `stream` with programmatic stream serialization (the
// kernel may begin its prologue while the previous kernel in the stream
// drains; every kernel of this library waits for its predecessor with
// griddepcontrol.wait before touching global memory), and as clusters of
// `cluster` CTAs when cluster > 1.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, unsigned cluster, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---- the select workspace (caller-owned device memory, zeroed once before
// its first use; every successful select call leaves it zeroed again)
constexpr int kSelectMaxCtas = 256;
constexpr uint32_t kSelectHistMagic = 0x74676831u;  // header stamp of a gate-filled histogram
// Candidate keys (those in the first digit's threshold bin) that the
// multi-CTA select can keep in the workspace: with them its second and third
// passes and the per-CTA counts are local, after one grid barrier.
constexpr int kSelectCandCap = 16384;
struct SelectWorkspace {
  uint32_t hist[3][2048];           // radix histograms of the select's three passes
  uint32_t gate_hist[2048];         // the first pass, counted by the gate epilogue
  uint32_t cnt[kSelectMaxCtas][2];  // per-CTA counts exchanged between the CTAs
  uint32_t hdr[4];                  // {magic, N, doc_begin, doc_end} when the gate filled gate_hist
  uint32_t bar_count, bar_gen;      // grid barrier: arrivals, generation
  uint32_t cand_next;               // candidates reserved so far in this call
  uint32_t cand_at[kSelectMaxCtas]; // where each CTA's candidates start in `cand`
  uint32_t cand[kSelectCandCap];    // candidate keys, one reserved run per CTA; written before read
};
// Everything before `cand` must start at zero; `cand` needs no clearing.
constexpr size_t kSelectZeroedBytes = offsetof(SelectWorkspace, cand);
constexpr size_t kSelectWorkspaceBytes = 40960 + 4 * static_cast<size_t>(kSelectCandCap);
static_assert(kSelectZeroedBytes <= 40960, "select workspace: zeroed part");
static_assert(sizeof(SelectWorkspace) <= kSelectWorkspaceBytes, "select workspace");
// Spans up to this many keys take the single-CTA select (all keys cached in
// shared memory, no grid barrier); longer spans the multi-CTA one, whose
// launch uses select_grid_size(D) CTAs.
constexpr int64_t kSelectSmallMaxKeys = 4096;
int select_grid_size(int64_t D);

// ---- launchers (argument checking happens in the ABI layer)
// sel_ws (nullable): accumulate the first radix histogram of the keys of
// the scores in [doc_b, doc_e) into it for a following select call.
cudaError_t launch_gate_bf16(const void* X, int64_t N, int d, const void* W1, const float* b1,
                             int Hg, const float* w2, float b2, float* scores,
                             SelectWorkspace* sel_ws, int64_t doc_b, int64_t doc_e,
                             cudaStream_t stream);
cudaError_t launch_gate_f32(const float* X, int64_t N, int d, const float* W1, const float* b1,
                            int Hg, const float* w2, float b2, float* scores,
                            cudaStream_t stream);
cudaError_t launch_qkv_bf16(const void* X, int64_t M, int d, const void* W, int ncols, void* Y,
                            cudaStream_t stream);
// The layers of a full Qwen3 decoder layer on the kept rows (bf16, CTA-pair
// tcgen05 GEMMs with fused epilogues):
//  QKV with per-head q/k RMSNorm and the rotary embedding (dh = 128),
cudaError_t launch_qkv_qknorm_rope_bf16(const void* X, int64_t M, int d, const void* W, int Hq,
                                       int Hkv, const float* gamma_q, const float* gamma_k,
                                       float eps, const float2* rope, void* Y,
                                       cudaStream_t stream);
//  residual (fp32 [M][N]) += X W^T,
cudaError_t launch_linear_resid_bf16(const void* X, int64_t M, int K, const void* W, int N,
                                     float* residual, cudaStream_t stream);
//  Y = silu(X Wg^T) * (X Wu^T) ([M][F] bf16),
cudaError_t launch_swiglu_bf16(const void* X, int64_t M, int d, const void* Wg, const void* Wu,
                               int F, void* Y, cudaStream_t stream);
//  and the rotary table of the kept rows ([M][dh / 2] (cos, sin)).
cudaError_t launch_rope_table(const int32_t* pos, int64_t M, int dh, double base, float2* table,
                              cudaStream_t stream);
// Gated delta rule (Gated-DeltaNet layers), dk = dv = 128, chunked; fp32
// inputs on CUDA cores (deltanet.cu), bf16 inputs on the tensor cores
// (deltanet_tc.cu).  The workspace size covers both.
size_t deltanet_workspace_bytes(int64_t T_len, int H);
size_t deltanet_tc_workspace_bytes(int64_t T_len, int H);
cudaError_t launch_deltanet_tc(const void* q, const void* k, const void* v, const float* alpha,
                               const float* beta, int64_t T_len, int H, const float* S0, void* o,
                               float* S_out, void* workspace, cudaStream_t stream);
cudaError_t launch_deltanet(const void* q, const void* k, const void* v, int bf16,
                            const float* alpha, const float* beta, int64_t T_len, int H,
                            const float* S0, void* o, float* S_out, void* workspace,
                            cudaStream_t stream);
cudaError_t launch_qkv_f32(const float* X, int64_t M, int d, const float* W, int ncols, float* Y,
                           cudaStream_t stream);
cudaError_t launch_select(const float* scores, int64_t N, int64_t b, int64_t e, int64_t K,
                          int32_t* idx, SelectWorkspace* ws, cudaStream_t stream);
cudaError_t launch_gather(const void* X, int x_bf16, int64_t N, int d, const int32_t* idx,
                          int64_t M, void* Y, int y_bf16, const float* scores, float* logsig,
                          cudaStream_t stream);
cudaError_t launch_rmsnorm(const void* X, int x_bf16, int64_t M, int d, const float* gamma,
                           float eps, void* Y, int y_bf16, cudaStream_t stream);
// bf16 token-gated attention: dispatches to one of the two kernels below.
cudaError_t launch_attn_bf16(const void* QKV, int64_t M, int Hq, int Hkv, int dh,
                             const float* logsig, const float* gain, float temperature, void* O,
                             float* residual, float* lse, cudaStream_t stream);
// one CTA per (query block, pair of q heads of a kv head), heads ping-pong
cudaError_t launch_attn_bf16_2h(const void* QKV, int64_t M, int Hq, int Hkv, int dh,
                                const float* logsig, const float* gain, float temperature, void* O,
                                float* residual, float* lse, cudaStream_t stream);
// persistent CTAs, one q head per work unit, key columns split over two
// softmax warpgroups
cudaError_t launch_attn_bf16_1h(const void* QKV, int64_t M, int Hq, int Hkv, int dh,
                                const float* logsig, const float* gain, float temperature, void* O,
                                float* residual, float* lse, cudaStream_t stream);
cudaError_t launch_attn_f32(const float* QKV, int64_t M, int Hq, int Hkv, int dh,
                            const float* logsig, const float* gain, float temperature, float* O,
                            float* residual, float* lse, cudaStream_t stream);
cudaError_t launch_attn_delta(const void* dO, const void* O, int x_bf16, int64_t M, int Hq,
                              int dh, float* delta, cudaStream_t stream);
cudaError_t launch_bias_grad_bf16(const void* QKV, const void* dO, int64_t M, int Hq, int Hkv,
                                  int dh, const float* ls, const float* gain, float temperature,
                                  const float* lse, const float* delta, float* dbias,
                                  cudaStream_t stream);
cudaError_t launch_bias_grad_f32(const float* QKV, const float* dO, int64_t M, int Hq, int Hkv,
                                 int dh, const float* ls, const float* gain, float temperature,
                                 const float* lse, const float* delta, float* dbias,
                                 cudaStream_t stream);
cudaError_t launch_bias_grad_reduce(const float* dbias, int64_t M, int Hq, const float* ls,
                                    const float* gain, float* dls, float* dgain, float* dscore,
                                    cudaStream_t stream);

cudaError_t launch_bounded_wait_selftest(uint64_t timeout_ns, unsigned long long* report,
                                         cudaStream_t stream);
// Reads and clears the status word in one atomic step on `stream`, into a
// device word whose address is returned through *taken.
cudaError_t launch_status_take(uint32_t** taken, cudaStream_t stream);

}  // namespace tg
