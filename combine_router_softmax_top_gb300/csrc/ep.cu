// Expert-parallel receive re-sort: the receiver's step between the dispatch
// all-to-all and its grouped GEMM, and the inverse step before the return
// all-to-all (the standard all-to-all dispatcher of the MoE expert-parallel
// overlap skill card, section "what it is", dispatcher table; EP16 in its
// benchmark sections).
//
// A rank owning E_l = E/R experts receives, from each source rank s in turn,
// that source's rows for its local experts l = 0..E_l-1 (recv_cnt[s][l] rows
// each, expert-contiguous because the source's send buffer is rank-major and
// expert-contiguous). The grouped GEMM wants its rows expert-major: expert l
// first, inside it source s ascending, inside that the source's own order.
// The forward re-sort gathers each expert-major row from its receive-order
// position; the inverse gathers each receive-order row from its expert-major
// position. Both are row copies bound by HBM: one warp per output row,
// 16-byte vectors, eight loads in flight per lane before the stores.
#include <algorithm>

#include "moe_internal.cuh"
#include "moe_layer_ops.h"

namespace moe {
namespace {

constexpr int kEpThreads = 256;
constexpr int kEpWarps = kEpThreads / 32;
constexpr int kEpMaxSeg = 256;  // R * E_l = E <= 256 segments
constexpr int kEpUnroll = 8;

// Exclusive prefix sum over the block (256 threads) of one int per thread.
__device__ __forceinline__ int block_excl_scan(int v, int* s_w) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += n;
  }
  if (lane == 31) s_w[warp] = x;
  __syncthreads();
  int base = 0;
  for (int w = 0; w < warp; ++w) base += s_w[w];
  __syncthreads();  // s_w is reused by the next scan
  return base + x - v;
}

__global__ void __launch_bounds__(kEpThreads) ep_resort_kernel(
    const int32_t* __restrict__ recv_cnt, const bf16* __restrict__ in, bf16* __restrict__ out,
    int32_t* __restrict__ off_local, int n_rows, int R, int El, int H, int inverse) {
  pdl_wait();
  __shared__ int s_rs[kEpMaxSeg + 1];   // receive-order start of segment i = s*El + l
  __shared__ int s_es[kEpMaxSeg + 1];   // expert-major start of segment j = l*R + s
  __shared__ int s_out[kEpMaxSeg + 1];  // output-order start of output segment q
  __shared__ int s_in[kEpMaxSeg];       // input start of output segment q
  __shared__ int s_w[kEpWarps];
  const int nseg = R * El;
  const int t = threadIdx.x;
  // count of receive-order segment i = t, and of expert-major segment j = t
  // (j = l*R + s is receive-order segment s*El + l); negative counts move nothing
  const int ci = t < nseg ? max(recv_cnt[t], 0) : 0;
  const int cj = t < nseg ? max(recv_cnt[(t % R) * El + t / R], 0) : 0;
  const int rs = block_excl_scan(ci, s_w);
  const int es = block_excl_scan(cj, s_w);
  if (t < nseg) {
    s_rs[t] = rs;
    s_es[t] = es;
  }
  if (t == nseg - 1) {
    s_rs[nseg] = rs + ci;
    s_es[nseg] = es + cj;
  }
  __syncthreads();
  if (t < nseg) {
    if (!inverse) {  // output expert-major (segment j = t), input receive order
      s_out[t] = s_es[t];
      s_in[t] = s_rs[(t % R) * El + t / R];
    } else {         // output receive order (segment i = t), input expert-major
      s_out[t] = s_rs[t];
      s_in[t] = s_es[(t % El) * R + t / El];
    }
  }
  if (t == 0) s_out[nseg] = s_rs[nseg];
  if (blockIdx.x == 0 && off_local != nullptr) {
    if (t < El) off_local[t] = s_es[t * R];
    if (t == 0) off_local[El] = s_es[nseg];
  }
  __syncthreads();

  const int rows = min(s_out[nseg], n_rows);
  const int cpr = H / 8;  // 16-byte chunks per row
  const int lane = t & 31;
  const int nw = gridDim.x * kEpWarps;
  for (int o = blockIdx.x * kEpWarps + (t >> 5); o < rows; o += nw) {
    // the last segment starting at or before o holds it (empty ones share starts)
    int lo = 0, hi = nseg - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_out[mid] <= o) lo = mid; else hi = mid - 1;
    }
    const int src = s_in[lo] + (o - s_out[lo]);
    if (src >= n_rows) continue;  // counts beyond the buffer: not moved
    const uint4* s4 = reinterpret_cast<const uint4*>(in + (size_t)src * H);
    uint4* d4 = reinterpret_cast<uint4*>(out + (size_t)o * H);
    for (int c0 = 0; c0 < cpr; c0 += 32 * kEpUnroll) {
      uint4 v[kEpUnroll];
#pragma unroll
      for (int u = 0; u < kEpUnroll; ++u) {
        const int c = c0 + 32 * u + lane;
        if (c < cpr) v[u] = __ldcs(s4 + c);
      }
#pragma unroll
      for (int u = 0; u < kEpUnroll; ++u) {
        const int c = c0 + 32 * u + lane;
        if (c < cpr) d4[c] = v[u];
      }
    }
  }
}

}  // namespace

moe_status_t launch_ep_resort(const moe_layer_desc_t& d, const int32_t* recv_cnt, const bf16* in,
                              bf16* out, int32_t* off_local, int n_rows, int inverse,
                              cudaStream_t st) {
  const int El = d.E / d.R;
  const int blocks = std::max(1, std::min(ceil_div(std::max(n_rows, 1), kEpWarps),
                                          16 * device_sm_count()));
  {
    LaunchScope _ls(K_EP_RESORT, st);
    launch_k(ep_resort_kernel, blocks, kEpThreads, 0, st, recv_cnt, in, out, off_local, n_rows,
             d.R, El, d.H, inverse);
  }
  return check_launch("ep_resort_kernel");
}

}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_ep_resort(const moe_layer_desc_t* d, const int32_t* recv_cnt,
                                      const moe_bf16* in, moe_bf16* out, int32_t* off_local,
                                      int64_t n_rows, int32_t inverse, void* stream) {
  moe_status_t s = validate(d);
  if (s != MOE_OK) return s;
  if (n_rows < 0 || n_rows >= (1ll << 31)) {
    set_error("n_rows=%lld must be in [0, 2^31)", (long long)n_rows);
    return MOE_ERR_INVALID_ARG;
  }
  if (inverse != 0 && inverse != 1) {
    set_error("inverse must be 0 or 1 (got %d)", inverse);
    return MOE_ERR_INVALID_ARG;
  }
  const void* ptrs[] = {recv_cnt, in, out};
  const char* names[] = {"recv_cnt", "in", "out"};
  for (int i = 0; i < 3; ++i) {
    if (!ptrs[i] || (reinterpret_cast<uintptr_t>(ptrs[i]) & 15u)) {
      set_error("%s is NULL or not 16-byte aligned", names[i]);
      return MOE_ERR_INVALID_ARG;
    }
  }
  if (off_local && (reinterpret_cast<uintptr_t>(off_local) & 15u)) {
    set_error("off_local is not 16-byte aligned");
    return MOE_ERR_INVALID_ARG;
  }
  if (in == out && n_rows > 0) {
    set_error("moe_ep_resort cannot work in place (in == out)");
    return MOE_ERR_INVALID_ARG;
  }
  return launch_ep_resort(*d, recv_cnt, reinterpret_cast<const bf16*>(in),
                          reinterpret_cast<bf16*>(out), off_local, (int)n_rows, inverse,
                          static_cast<cudaStream_t>(stream));
}
