// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "moe.h"

namespace moe {

typedef __nv_bfloat16 bf16;

// ---------------------------------------------------------------- workspace map
// The workspace starts with status words; the rest is carved per call kind.
enum StatusWord {
  ST_BAD_INDEX = 0,   // count of out-of-range indices a kernel skipped
  ST_TIMEOUT = 1,     // a bounded pipeline wait gave up (nonzero = where)
  ST_NUM = 8
};
constexpr size_t kStatusBytes = 256;
constexpr int kLayoutTokensPerBlock = 256;
constexpr int kRouteBwdRowsPerChunk = 64;

struct WsLayout {
  // dep: the GEMM chains' per-expert counters [E], then dW_r's per-expert,
  // per-column-block chunk counters [E * ceil(H / 2048)]
  size_t status, logits, hist, dz, dwr_part, dep, fhist, bar, total;
};
WsLayout ws_layout(const moe_layer_desc_t& d);

inline int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

// ---------------------------------------------------------------- launch accounting
enum KernelId {
  K_ROUTE_LOGITS = 0, K_ROUTE_TOPK, K_LAYOUT_COUNT, K_LAYOUT_ASSIGN, K_PERMUTE, K_COMBINE,
  K_COMBINE_BWD, K_PERMUTE_BWD, K_ROUTE_BWD_DX, K_ROUTE_BWD_DWR,
  K_GEMM_FC1_FWD, K_GEMM_FC2_FWD, K_GEMM_FC2_DGRAD, K_GEMM_FC1_DGRAD, K_GEMM_WGRAD_W1,
  K_GEMM_WGRAD_W2, K_DISPATCH_BWD, K_GEMM_FFN_FWD, K_GEMM_FFN_DGRAD, K_DISPATCH_FUSED,
  K_GEMM_WGRAD_W1_ACC, K_GEMM_WGRAD_W2_ACC, K_LAYOUT_SCAN, K_EP_RESORT, K_GEMM_WGRAD, K_NUM
};

// Wraps one kernel launch: counts it and, while profiling is on, brackets it
// with CUDA events on its stream.
class LaunchScope {
 public:
  LaunchScope(int kernel, cudaStream_t st);
  ~LaunchScope();
  LaunchScope(const LaunchScope&) = delete;
  LaunchScope& operator=(const LaunchScope&) = delete;

 private:
  int kernel_;
  cudaStream_t st_;
  int rec_;
};

// True while moe_profile_start() has per-launch timing on.
bool profiling_active();
// Adds n (may be negative) to the count moe_kernel_launches() returns.
void count_launches(long long n);

// ---------------------------------------------------------------- errors
void set_error(const char* fmt, ...);
moe_status_t check_launch(const char* what);

int device_sm_count();

// ---------------------------------------------------------------- programmatic dependent launch
// Every kernel is launched with programmatic stream serialisation: the next
// kernel on the stream is launched as the blocks of this one exit, runs its
// set-up (shared memory, barriers, TMEM, descriptor prefetch), then blocks in
// pdl_wait() until this grid has completed and its writes are visible. Each
// kernel calls pdl_wait() before its first global memory access (read or
// write). Kernels do not signal an earlier launch (griddepcontrol.
// launch_dependents): measured on the layer step, that made the dependent
// grids resident too early and cost 0.10 ms per step, while the launch at
// block exit saves 0.04 ms over plain stream order. Without the launch
// attribute pdl_wait() is a no-op, so the order of work is the same either way.
#ifndef MOE_PDL
#define MOE_PDL 1
#endif
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = MOE_PDL;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------- launchers
moe_status_t launch_route(const moe_layer_desc_t& d, const bf16* x, const bf16* w_r,
                          const float* bias, float* logits, int32_t* idx, float* gates,
                          int* status, cudaStream_t st);
// Route + dispatch layout + permute in one cooperative launch (E <= 128, T > 0;
// MOE_ERR_UNSUPPORTED otherwise). fhist: ws area of (ceil(T/4) + 1) * E ints;
// bar: one int, zeroed by the launcher. zero/nzero: as for launch_combine_bwd
// (the layer path clears there the counters of the forward chain that follows).
// max_ctas > 0 caps the grid (blocks then take several token tiles each), so
// the launch can share the GPU with a kernel on the other SMs.
moe_status_t launch_dispatch_fused(const moe_layer_desc_t& d, const bf16* x, const bf16* w_r,
                                   const float* bias, float* z, int32_t* idx, float* gates,
                                   int32_t* cnt, int32_t* off, int32_t* slot, int32_t* row_src,
                                   int32_t* cnt_re, int32_t* rank_off, bf16* x_perm, int* fhist,
                                   int* bar, int* status, cudaStream_t st, int* zero = nullptr,
                                   int nzero = 0, int max_ctas = 0);
// Dispatch layout in three launches. hist: (ceil(T/256) + 1) * E ints of
// scratch (per-block expert counts, then the totals); fully rewritten.
moe_status_t launch_layout(const moe_layer_desc_t& d, const int32_t* idx, int32_t* cnt,
                           int32_t* off, int32_t* slot, int32_t* row_src, int32_t* cnt_re,
                           int32_t* rank_off, int* hist, int* status, cudaStream_t st);
moe_status_t launch_permute(const moe_layer_desc_t& d, const bf16* x, const int32_t* row_src,
                            bf16* x_perm, cudaStream_t st);
moe_status_t launch_combine(const moe_layer_desc_t& d, const bf16* o, const int32_t* slot,
                            const float* gates, bf16* y, cudaStream_t st);
// zero/nzero: nzero ints that block 0 sets to 0 once the previous launch on
// the stream has completed; the layer path clears there the counters of the
// dgrad chain that follows, in place of a memset between the two launches
// (which would stop the chain's launch from overlapping this one's drain).
moe_status_t launch_combine_bwd(const moe_layer_desc_t& d, const bf16* dy, const bf16* o,
                                const int32_t* slot, const float* gates, bf16* d_o,
                                float* dgates, cudaStream_t st, int* zero = nullptr,
                                int nzero = 0);
moe_status_t launch_permute_bwd(const moe_layer_desc_t& d, const bf16* dx_perm,
                                const int32_t* slot, float* dx32, cudaStream_t st);
// Router backward. With dx_perm (and slot) given, the dispatch backward is
// fused in: dx32 is not read and the row sums of dx_perm are formed in
// registers (the layer path); otherwise dx32 comes from launch_permute_bwd.
moe_status_t launch_route_bwd(const moe_layer_desc_t& d, const float* dgates, const float* gates,
                              const int32_t* idx, const bf16* x, const bf16* w_r,
                              const int32_t* row_src, const int32_t* off, const float* dx32,
                              const bf16* dx_perm, const int32_t* slot, bf16* dx, float* dw_r,
                              float* dz, float* dwr_part, int* dwr_cnt, bool cnt_zeroed,
                              int* status, cudaStream_t st);

// Expert-parallel receive re-sort (receive order <-> expert-major) of n_rows
// rows of H bf16; recv_cnt [R][E/R] on the device; off_local [E/R + 1] or NULL.
moe_status_t launch_ep_resort(const moe_layer_desc_t& d, const int32_t* recv_cnt, const bf16* in,
                              bf16* out, int32_t* off_local, int n_rows, int inverse,
                              cudaStream_t st);

enum GemmMode {
  GEMM_FC1_FWD = 0,   // a, h = SwiGLU(x_perm @ W1^T)
  GEMM_FC2_FWD = 1,   // o = h @ W2^T
  GEMM_FC2_DGRAD = 2, // da = SwiGLU'(d_o @ W2, a)
  GEMM_FC1_DGRAD = 3, // dx_perm = da @ W1
  GEMM_WGRAD_W1 = 4,  // dW1_e = da_e^T @ x_perm_e
  GEMM_WGRAD_W2 = 5   // dW2_e = d_o_e^T @ h_e
};

struct GemmArgs {
  int mode;
  const bf16* A;      // activation operand
  const bf16* B;      // weight (fwd/dgrad) or second activation (wgrad)
  const int32_t* off; // [E+1]
  bf16* out0;
  bf16* out1;
  const bf16* aux;
  int* status;
  int max_ctas;       // 0 = all SMs
  int* dep;           // [E] per-expert counters for a chain (workspace), else NULL
  float* acc;         // wgrad: fp32 gradient to add the result into (out0/out1 unused), else NULL
};
moe_status_t launch_grouped_gemm(const moe_layer_desc_t& d, const GemmArgs& g, cudaStream_t st);
// Two GEMMs in one persistent launch: FC1 fwd then FC2 fwd, or FC2 dgrad then
// FC1 dgrad (dependent), or the weight gradients W1 then W2 (independent; bf16
// outputs only, and N > 0: for an empty layer the single-mode launches write
// the zero gradients). A tile of a dependent second GEMM reads the first's
// output of its expert and waits for it through the per-expert counters
// g1.dep (zeroed here, unless counters_zeroed).
// counters_zeroed: g1.dep is already zero (cleared by the launch just before
// on the stream), so no memset is issued between the two launches.
moe_status_t launch_grouped_gemm_chain(const moe_layer_desc_t& d, const GemmArgs& g1,
                                       const GemmArgs& g2, cudaStream_t st,
                                       bool counters_zeroed = false);

}  // namespace moe
