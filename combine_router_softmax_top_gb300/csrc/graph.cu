// CUDA-graph capture of the layer's launch sequences.
//
// The production benchmark of the MoE expert-parallel overlap skill card
// (section "HybridEP production benchmark") runs the router and the dispatch
// preprocessing under CUDA graphs (Transformer Engine scopes moe_router and
// moe_preprocess). Here a scope's calls are captured once from a caller
// stream, with every buffer address, tensor map and launch shape fixed, and
// replayed with one graph launch: the programmatic-launch edges between
// consecutive kernels and the backward's side-stream fork/join are kept as
// graph edges.
#include <new>
#include <vector>

#include "moe_layer_ops.h"

struct moe_graph {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  int32_t kernels = 0;
};

using namespace moe;

namespace {

moe_status_t capture_scope(const moe_layer_desc_t* d, const moe_mb_bufs_t* b, int32_t scope,
                           void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (scope) {
    case MOE_GRAPH_ROUTER_PREPROCESS: return op_dispatch(*d, b, st);
    case MOE_GRAPH_LAYER_FORWARD: return moe_layer_forward(d, b, stream);
    default: {
      const moe_status_t s = moe_layer_forward(d, b, stream);
      return s != MOE_OK ? s : moe_layer_backward(d, b, 1, stream);
    }
  }
}

}  // namespace

extern "C" {

moe_status_t moe_graph_capture(const moe_layer_desc_t* d, const moe_mb_bufs_t* b, int32_t scope,
                               void* stream, moe_graph_t** out) {
  if (!out) {
    set_error("out is NULL");
    return MOE_ERR_INVALID_ARG;
  }
  *out = nullptr;
  moe_status_t st0 = validate(d);
  if (st0 != MOE_OK) return st0;
  if (scope < MOE_GRAPH_ROUTER_PREPROCESS || scope > MOE_GRAPH_LAYER_STEP) {
    set_error("unknown graph scope %d", scope);
    return MOE_ERR_INVALID_ARG;
  }
  st0 = check_mb(*d, b, scope == MOE_GRAPH_LAYER_STEP);
  if (st0 != MOE_OK) return st0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (st == nullptr || st == cudaStreamLegacy || st == cudaStreamPerThread) {
    set_error("graph capture needs a caller-created stream, not a default stream");
    return MOE_ERR_INVALID_ARG;
  }
  if (profiling_active()) {
    set_error("graph capture while per-launch profiling is on");
    return MOE_ERR_INVALID_ARG;
  }
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(st, &cs);
  if (e == cudaSuccess && cs != cudaStreamCaptureStatusNone) {
    set_error("the stream is already capturing");
    return MOE_ERR_INVALID_ARG;
  }
  // helper streams and events exist before the capture starts
  if (e != cudaSuccess || !copy_lane()) {
    if (e != cudaSuccess) set_error("cudaStreamIsCapturing: %s", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  const unsigned long long l0 = moe_kernel_launches();
  e = cudaStreamBeginCapture(st, cudaStreamCaptureModeRelaxed);
  if (e != cudaSuccess) {
    set_error("cudaStreamBeginCapture: %s", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  const moe_status_t s = capture_scope(d, b, scope, stream);
  cudaGraph_t g = nullptr;
  e = cudaStreamEndCapture(st, &g);
  // captured launches have not run; replays count them
  count_launches(-static_cast<long long>(moe_kernel_launches() - l0));
  if (s != MOE_OK || e != cudaSuccess || !g) {
    if (g) cudaGraphDestroy(g);
    if (s != MOE_OK) return s;
    set_error("cudaStreamEndCapture: %s", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  size_t n = 0;
  e = cudaGraphGetNodes(g, nullptr, &n);
  std::vector<cudaGraphNode_t> nodes(n);
  if (e == cudaSuccess && n) e = cudaGraphGetNodes(g, nodes.data(), &n);
  int32_t kernels = 0;
  for (size_t i = 0; e == cudaSuccess && i < n; ++i) {
    cudaGraphNodeType t;
    e = cudaGraphNodeGetType(nodes[i], &t);
    if (e == cudaSuccess && t == cudaGraphNodeTypeKernel) ++kernels;
  }
  cudaGraphExec_t ex = nullptr;
  if (e == cudaSuccess) e = cudaGraphInstantiate(&ex, g, 0);
  if (e != cudaSuccess) {
    set_error("graph set-up: %s", cudaGetErrorString(e));
    cudaGraphDestroy(g);
    return MOE_ERR_CUDA;
  }
  moe_graph* G = new (std::nothrow) moe_graph;
  if (!G) {
    cudaGraphExecDestroy(ex);
    cudaGraphDestroy(g);
    set_error("out of host memory");
    return MOE_ERR_CUDA;
  }
  G->graph = g;
  G->exec = ex;
  G->kernels = kernels;
  *out = G;
  return MOE_OK;
}

moe_status_t moe_graph_launch(moe_graph_t* g, void* stream) {
  if (!g) {
    set_error("graph is NULL");
    return MOE_ERR_INVALID_ARG;
  }
  const cudaError_t e = cudaGraphLaunch(g->exec, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    set_error("cudaGraphLaunch: %s", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  count_launches(g->kernels);
  return MOE_OK;
}

int32_t moe_graph_kernel_count(const moe_graph_t* g) { return g ? g->kernels : 0; }

void moe_graph_destroy(moe_graph_t* g) {
  if (!g) return;
  if (g->exec) cudaGraphExecDestroy(g->exec);
  if (g->graph) cudaGraphDestroy(g->graph);
  delete g;
}

}  // extern "C"
