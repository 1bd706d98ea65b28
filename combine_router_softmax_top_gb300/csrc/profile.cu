// Launch accounting and optional per-launch timing of the library's kernels.
// Every kernel launch goes through a LaunchScope: it counts the launch and,
// while profiling is on, records a CUDA event before and after the launch on
// the launch's own stream, so durations come from the stream the kernel runs on.
#include <atomic>
#include <mutex>
#include <vector>

#include "moe_internal.cuh"

namespace moe {

namespace {

const char* const kNames[K_NUM] = {
    "route_logits", "route_topk", "layout_count", "layout_assign", "permute",
    "combine", "combine_bwd", "permute_bwd", "route_bwd_dx", "route_bwd_dwr", "gemm_fc1_fwd", "gemm_fc2_fwd", "gemm_fc2_dgrad",
    "gemm_fc1_dgrad", "gemm_wgrad_w1", "gemm_wgrad_w2", "dispatch_bwd", "gemm_ffn_fwd",
    "gemm_ffn_dgrad", "dispatch_fused", "gemm_wgrad_w1_accum", "gemm_wgrad_w2_accum",
    "layout_scan", "ep_resort", "gemm_wgrad"};

std::atomic<unsigned long long> g_launches{0};

struct Rec {
  int kernel;
  cudaEvent_t a, b;
};

std::mutex g_mu;
bool g_on = false;
std::vector<cudaEvent_t> g_pool;
std::vector<Rec> g_recs;
size_t g_next = 0;

}  // namespace

LaunchScope::LaunchScope(int kernel, cudaStream_t st) : kernel_(kernel), st_(st), rec_(-1) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_on || g_next + 2 > g_pool.size()) return;
  Rec r{kernel, g_pool[g_next], g_pool[g_next + 1]};
  g_next += 2;
  if (cudaEventRecord(r.a, st) != cudaSuccess) return;
  rec_ = (int)g_recs.size();
  g_recs.push_back(r);
}

bool profiling_active() {
  std::lock_guard<std::mutex> lk(g_mu);
  return g_on;
}

void count_launches(long long n) {
  g_launches.fetch_add(static_cast<unsigned long long>(n), std::memory_order_relaxed);
}

LaunchScope::~LaunchScope() {
  if (rec_ < 0) return;
  std::lock_guard<std::mutex> lk(g_mu);
  cudaEventRecord(g_recs[rec_].b, st_);
}

}  // namespace moe

using namespace moe;

extern "C" {

uint64_t moe_kernel_launches(void) { return g_launches.load(); }

const char* moe_kernel_name(int32_t kernel) {
  return (kernel >= 0 && kernel < K_NUM) ? kNames[kernel] : "";
}

moe_status_t moe_profile_start(int32_t capacity) {
  if (capacity <= 0) {
    set_error("capacity must be positive");
    return MOE_ERR_INVALID_ARG;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  while ((int)g_pool.size() < 2 * capacity) {
    cudaEvent_t e;
    cudaError_t err = cudaEventCreate(&e);
    if (err != cudaSuccess) {
      set_error("cudaEventCreate: %s", cudaGetErrorString(err));
      return MOE_ERR_CUDA;
    }
    g_pool.push_back(e);
  }
  g_recs.clear();
  g_recs.reserve(capacity);
  g_next = 0;
  g_on = true;
  return MOE_OK;
}

moe_status_t moe_profile_stop(moe_kernel_time_t* out, int32_t cap, int32_t* n) {
  if (!n || (cap > 0 && !out)) {
    set_error("invalid arguments");
    return MOE_ERR_INVALID_ARG;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  g_on = false;
  int k = 0;
  for (size_t i = 0; i < g_recs.size() && k < cap; ++i, ++k) {
    float ms = 0.f;
    cudaError_t e = cudaEventSynchronize(g_recs[i].b);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, g_recs[i].a, g_recs[i].b);
    if (e != cudaSuccess) {
      set_error("profile events: %s", cudaGetErrorString(e));
      return MOE_ERR_CUDA;
    }
    out[k].kernel = g_recs[i].kernel;
    out[k].ms = ms;
  }
  *n = k;
  g_recs.clear();
  g_next = 0;
  return MOE_OK;
}

}  // extern "C"
