// The gated layer as one CUDA graph: the five C-ABI calls of one layer are
// captured once on a private stream and replayed with one launch per prompt.
// Every kernel of the path is launched with programmatic stream
// serialization, so inside the graph each kernel's prologue overlaps its
// predecessor's tail; the graph removes the per-call host work (argument
// checks, tensor-map encoding) and the launch gaps between the calls.
#include <cuda_runtime.h>

#include "tg_device.cuh"
#include "tg_internal.h"

struct tg_plan_s {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  int device = -1;
};

namespace {

tg_status capture_gated_layer(const tg_gated_layer_desc& g, cudaStream_t s) {
  tg_status st = tg_gate_score(g.X, TG_BF16, g.N, g.d, g.W1, g.b1, g.Hg, g.w2, g.b2, g.scores,
                               g.select_ws, g.doc_begin, g.doc_end,
                               reinterpret_cast<tg_stream_t>(s));
  if (st != TG_OK) return st;
  int64_t M = 0;
  st = tg_select_topk(g.scores, g.N, g.doc_begin, g.doc_end, g.K, g.kept_idx, &M, g.select_ws,
                      g.select_ws_bytes, reinterpret_cast<tg_stream_t>(s));
  if (st != TG_OK) return st;
  st = tg_gather_rows(g.X, TG_BF16, g.N, g.d, g.kept_idx, M, g.Xk, TG_BF16, g.scores,
                      g.logsig_kept, reinterpret_cast<tg_stream_t>(s));
  if (st != TG_OK) return st;
  st = tg_qkv_proj(g.Xk, TG_BF16, M, g.d, g.Wqkv, g.Hq, g.Hkv, g.dh, g.QKV,
                   reinterpret_cast<tg_stream_t>(s));
  if (st != TG_OK) return st;
  return tg_keybias_attn(g.QKV, TG_BF16, M, g.Hq, g.Hkv, g.dh, g.logsig_kept, g.gain,
                         g.temperature, g.O, nullptr, reinterpret_cast<tg_stream_t>(s));
}

}  // namespace

extern "C" tg_status tg_gated_layer_plan_create(const tg_gated_layer_desc* desc, tg_plan_t* plan) {
  if (desc == nullptr || plan == nullptr)
    return tg::fail(TG_ERR_INVALID_ARG, "plan: NULL desc or plan");
  *plan = nullptr;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return tg::fail(TG_ERR_CUDA, "plan: %s", cudaGetErrorString(e));
  cudaStream_t s = nullptr;
  e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
  if (e != cudaSuccess) return tg::fail(TG_ERR_CUDA, "plan: %s", cudaGetErrorString(e));
  // relaxed: the first call of a kernel may load its module during capture
  e = cudaStreamBeginCapture(s, cudaStreamCaptureModeRelaxed);
  if (e != cudaSuccess) {
    cudaStreamDestroy(s);
    return tg::fail(TG_ERR_CUDA, "plan: begin capture: %s", cudaGetErrorString(e));
  }
  const tg_status st = capture_gated_layer(*desc, s);
  cudaGraph_t graph = nullptr;
  e = cudaStreamEndCapture(s, &graph);
  cudaStreamDestroy(s);
  if (st != TG_OK) {  // the failing call's message stays the last error
    if (graph) cudaGraphDestroy(graph);
    return st;
  }
  if (e != cudaSuccess || graph == nullptr)
    return tg::fail(TG_ERR_CUDA, "plan: end capture: %s", cudaGetErrorString(e));
  cudaGraphExec_t exec = nullptr;
  e = cudaGraphInstantiate(&exec, graph, 0);
  if (e != cudaSuccess) {
    cudaGraphDestroy(graph);
    return tg::fail(TG_ERR_CUDA, "plan: instantiate: %s", cudaGetErrorString(e));
  }
  tg_plan_s* p = new tg_plan_s;
  p->graph = graph;
  p->exec = exec;
  p->device = dev;
  *plan = p;
  return TG_OK;
}

extern "C" tg_status tg_plan_launch(tg_plan_t plan, tg_stream_t stream) {
  if (plan == nullptr || plan->exec == nullptr)
    return tg::fail(TG_ERR_INVALID_ARG, "plan launch: NULL plan");
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != plan->device)
    return tg::fail(TG_ERR_INVALID_ARG, "plan launch: the plan belongs to device %d", plan->device);
  const cudaError_t e = cudaGraphLaunch(plan->exec, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return tg::fail(TG_ERR_CUDA, "plan launch: %s", cudaGetErrorString(e));
  return TG_OK;
}

extern "C" tg_status tg_plan_destroy(tg_plan_t plan) {
  if (plan == nullptr) return TG_OK;
  if (plan->exec) cudaGraphExecDestroy(plan->exec);
  if (plan->graph) cudaGraphDestroy(plan->graph);
  delete plan;
  return TG_OK;
}
