// moe_dispatch_layout_static: the dispatch layout for callers that cannot
// allocate device memory.
//
// moe_dispatch_layout() needs a caller-provided workspace for its per-block
// expert histograms. Some callers have no way to provide one: code that owns
// no allocator (a plugin inside a host framework that hands it only its input
// and output tensors), code that must not call cudaMalloc at all (cudaMalloc
// synchronises the device and is not allowed while a stream is being captured
// into a CUDA graph), and real-time paths that must not take allocator locks.
// This variant keeps its scratch in a fixed array in the library's own device
// memory instead, so the caller passes only inputs and outputs.
//
// Limits and sharing: the array holds the histograms of up to kMaxTokens tokens
// and kMaxExperts experts plus a row of totals (257 KB plus 256 bytes of status
// words); larger layers are rejected. Every GPU that loads the library keeps
// the array until the process exits. All calls share the one array, so two
// calls whose work can overlap on the GPU (different streams without ordering
// between them) race and corrupt each other's layout; calls on one stream, or
// otherwise ordered, are safe.
//
// Out-of-range expert indices are skipped (slot = -1) and counted in the
// array's status words, which moe_dispatch_layout_static_status() reads; the
// next layout call clears them.
#include <mutex>

#include "moe_internal.cuh"
#include "moe_layer_ops.h"

namespace moe {
namespace {

constexpr int kMaxTokens = 65536;
constexpr int kMaxExperts = 256;
constexpr int kStatusInts = (int)(kStatusBytes / sizeof(int));
constexpr int kMaxBlocks = kMaxTokens / kLayoutTokensPerBlock;

// status words, then [kMaxBlocks + 1][kMaxExperts] histograms and totals
static __device__ __align__(256) int
    g_layout_scratch[kStatusInts + (kMaxBlocks + 1) * kMaxExperts];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of g_layout_scratch on the current device. Outside stream
// capture it is looked up with cudaGetSymbolAddress on every call (the device
// is current), so a module reloaded after a device reset, or a different
// context of the same device, is followed. While `st` is capturing, the
// address last looked up on this device is used: the first call on a device
// must therefore come before any capture.
moe_status_t scratch_for_current_device(cudaStream_t st, int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_error("cudaGetDevice: %s", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    set_error("device ordinal %d is beyond the %d devices this call supports", dev, kMaxDevices);
    return MOE_ERR_UNSUPPORTED;
  }
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(st, &cap);
  if (e != cudaSuccess) {
    set_error("cudaStreamIsCapturing: %s", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (cap != cudaStreamCaptureStatusNone) {
    if (!g_scratch_addr[dev]) {
      set_error("moe_dispatch_layout_static: the first call on device %d must come before any "
                "stream capture (it looks up the scratch array's address)", dev);
      return MOE_ERR_INVALID_ARG;
    }
    *out = g_scratch_addr[dev];
    return MOE_OK;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_layout_scratch);
  if (e != cudaSuccess || !p) {
    set_error("cudaGetSymbolAddress of the layout scratch failed on device %d: %s", dev,
              cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  g_scratch_addr[dev] = static_cast<int*>(p);
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_dispatch_layout_static(const moe_layer_desc_t* d, const int32_t* idx,
                                                   int32_t* cnt, int32_t* off, int32_t* slot,
                                                   int32_t* row_src, int32_t* cnt_re,
                                                   int32_t* rank_off, void* stream) {
  moe_status_t s = validate(d);
  if (s != MOE_OK) return s;
  if (d->T > kMaxTokens || d->E > kMaxExperts) {
    set_error("moe_dispatch_layout_static handles at most %d tokens and %d experts "
              "(got T=%d, E=%d); use moe_dispatch_layout with a workspace instead",
              kMaxTokens, kMaxExperts, d->T, d->E);
    return MOE_ERR_UNSUPPORTED;
  }
  const void* ptrs[] = {idx, cnt, off, slot, row_src, cnt_re, rank_off};
  const char* names[] = {"idx", "cnt", "off", "slot", "row_src", "cnt_re", "rank_off"};
  for (int i = 0; i < 7; ++i) {
    if (!ptrs[i] || (reinterpret_cast<uintptr_t>(ptrs[i]) & 15u)) {
      set_error("%s is NULL or not 16-byte aligned", names[i]);
      return MOE_ERR_INVALID_ARG;
    }
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* scratch = nullptr;
  s = scratch_for_current_device(st, &scratch);
  if (s != MOE_OK) return s;
  // The histograms are fully rewritten by every call; only the status words
  // keep counts and must start from zero.
  cudaError_t e = cudaMemsetAsync(scratch, 0, kStatusBytes, st);
  if (e != cudaSuccess) {
    set_error("cudaMemsetAsync: %s", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  return launch_layout(*d, idx, cnt, off, slot, row_src, cnt_re, rank_off, scratch + kStatusInts,
                       scratch, st);
}

extern "C" moe_status_t moe_dispatch_layout_static_status(void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) {
    set_error("moe_dispatch_layout_static_status synchronises its stream: not while capturing");
    return MOE_ERR_INVALID_ARG;
  }
  int* scratch = nullptr;
  moe_status_t s = scratch_for_current_device(st, &scratch);
  if (s != MOE_OK) return s;
  int h[ST_NUM] = {0};
  cudaError_t e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaMemcpy(h, scratch, sizeof(h), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(scratch, 0, sizeof(h));
  if (e != cudaSuccess) {
    set_error("moe_dispatch_layout_static_status: %s", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  if (h[ST_BAD_INDEX]) {
    set_error("%d out-of-range expert indices were skipped (slot = -1)", h[ST_BAD_INDEX]);
    return MOE_ERR_INVALID_ARG;
  }
  return MOE_OK;
}
