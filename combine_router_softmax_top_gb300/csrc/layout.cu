// Dispatch layout: per-expert counts, exclusive offsets, stable slots, the
// inverse permutation and the per-(rank, expert) tables an EP all-to-all
// exchanges (the "moe_preprocess" step ahead of dispatch in the EP-overlap
// skill card, "HybridEP production benchmark").
//
// Three kernels, all integer-only and deterministic:
//   1. count:  block b histograms the experts of its 256 tokens into
//      hist[b][e] (nb blocks).
//   2. scan:   block e turns column e of the histograms into exclusive
//      prefixes over blocks, in place, and writes the column total to
//      hist[nb][e], so every count is read a fixed, small number of times
//      whatever the number of blocks.
//   3. assign: each block reads its own prefixes and the totals, scans the
//      totals into the expert offsets, then numbers its own entries in token
//      order. Within a block each warp holds 32 tokens; per expert, the warp's
//      tokens that chose it form a 32-bit mask, so the rank of a token among
//      the block's earlier tokens is (earlier warps' popcounts) +
//      popc(mask & lanes_below).
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kTok = kLayoutTokensPerBlock;  // 256 tokens = 8 warps x 32
constexpr int kWarps = kTok / 32;

__global__ void __launch_bounds__(kTok) layout_count_kernel(const int32_t* __restrict__ idx,
                                                            int* __restrict__ hist, int T, int E,
                                                            int k, int* status) {
  pdl_wait();
  extern __shared__ int s_hist[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_hist[e] = 0;
  __syncthreads();
  const int t = blockIdx.x * kTok + threadIdx.x;
  if (t < T) {
    for (int j = 0; j < k; ++j) {
      const int e = idx[(size_t)t * k + j];
      if ((unsigned)e < (unsigned)E) atomicAdd(&s_hist[e], 1);
      else atomicAdd(status + ST_BAD_INDEX, 1);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(size_t)blockIdx.x * E + e] = s_hist[e];
}

// Exclusive prefix of column e = blockIdx.x over the nb block histograms, in
// place, 256 blocks at a time with a carry; the total goes to hist[nb][e].
__global__ void __launch_bounds__(kTok) layout_scan_kernel(int* __restrict__ hist, int E,
                                                           int nb) {
  pdl_wait();
  __shared__ int s_warp[kWarps];
  const int e = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int carry = 0;
  for (int b0 = 0; b0 < nb; b0 += kTok) {
    const int b = b0 + threadIdx.x;
    const int c = b < nb ? hist[(size_t)b * E + e] : 0;
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    int before = carry;
    for (int w = 0; w < warp; ++w) before += s_warp[w];
    if (b < nb) hist[(size_t)b * E + e] = before + incl - c;
    int sum = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) sum += s_warp[w];
    carry += sum;
    __syncthreads();  // s_warp is rewritten by the next round
  }
  if (threadIdx.x == 0) hist[(size_t)nb * E + e] = carry;
}

__global__ void __launch_bounds__(kTok) layout_assign_kernel(
    const int32_t* __restrict__ idx, const int* __restrict__ hist, int32_t* __restrict__ cnt,
    int32_t* __restrict__ off, int32_t* __restrict__ slot, int32_t* __restrict__ row_src,
    int32_t* __restrict__ cnt_re, int32_t* __restrict__ rank_off, int T, int E, int k, int R,
    int nblocks) {
  pdl_wait();
  extern __shared__ int smem[];
  int* s_base = smem;                              // [E]  first row of this block's entries
  int* s_cnt = s_base + E;                         // [E]
  uint32_t* s_mask = reinterpret_cast<uint32_t*>(s_cnt + E);  // [kWarps][E]
  int* s_pre = reinterpret_cast<int*>(s_mask + kWarps * E);   // [kWarps][E]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // totals over all blocks and the part before this block (from the scan)
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    s_cnt[e] = hist[(size_t)nblocks * E + e];
    s_base[e] = hist[(size_t)blockIdx.x * E + e];
  }
  for (int i = threadIdx.x; i < kWarps * E; i += blockDim.x) s_mask[i] = 0u;
  __syncthreads();
  // exclusive scan of the counts over experts (warp 0, 32 experts per step)
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      const int c = e < E ? s_cnt[e] : 0;
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      if (e < E) {
        const int ex = carry + incl - c;
        if (blockIdx.x == 0) {
          off[e] = ex;
          cnt[e] = c;
          cnt_re[e] = c;  // [R][E/R] row-major is the expert order itself
        }
        s_base[e] += ex;
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (blockIdx.x == 0 && lane == 0) off[E] = carry;
  }
  __syncthreads();
  if (blockIdx.x == 0) {
    const int El = E / R;
    for (int r = threadIdx.x; r <= R; r += blockDim.x) {
      // rank r's chunk starts at the first row of its first expert
      int v = 0;
      for (int e = 0; e < r * El; ++e) v += s_cnt[e];
      rank_off[r] = v;
    }
  }
  // per-warp masks of the tokens that chose each expert
  const int t = blockIdx.x * kTok + threadIdx.x;
  const bool valid = t < T;
  if (valid) {
    for (int j = 0; j < k; ++j) {
      const int e = idx[(size_t)t * k + j];
      if ((unsigned)e < (unsigned)E) atomicOr(&s_mask[warp * E + e], 1u << lane);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (int w = 0; w < kWarps; ++w) {
      s_pre[w * E + e] = run;
      run += __popc(s_mask[w * E + e]);
    }
  }
  __syncthreads();
  if (valid) {
    const uint32_t below = (1u << lane) - 1u;
    for (int j = 0; j < k; ++j) {
      const int e = idx[(size_t)t * k + j];
      int s = -1;
      if ((unsigned)e < (unsigned)E) {
        s = s_base[e] + s_pre[warp * E + e] + __popc(s_mask[warp * E + e] & below);
        row_src[s] = t * k + j;
      }
      slot[(size_t)t * k + j] = s;
    }
  }
}

}  // namespace

moe_status_t launch_layout(const moe_layer_desc_t& d, const int32_t* idx, int32_t* cnt,
                           int32_t* off, int32_t* slot, int32_t* row_src, int32_t* cnt_re,
                           int32_t* rank_off, int* hist, int* status, cudaStream_t st) {
  const int nb = d.T > 0 ? ceil_div(d.T, kTok) : 1;
  {
    LaunchScope _ls(K_LAYOUT_COUNT, st);
    launch_k(layout_count_kernel, nb, kTok, d.E * sizeof(int), st, idx, hist, d.T, d.E, d.k,
             status);
  }
  moe_status_t s = check_launch("layout_count_kernel");
  if (s != MOE_OK) return s;
  {
    LaunchScope _ls(K_LAYOUT_SCAN, st);
    launch_k(layout_scan_kernel, d.E, kTok, 0, st, hist, d.E, nb);
  }
  s = check_launch("layout_scan_kernel");
  if (s != MOE_OK) return s;
  const size_t smem = (size_t)d.E * (2 + 2 * kWarps) * sizeof(int);
  {
    LaunchScope _ls(K_LAYOUT_ASSIGN, st);
    launch_k(layout_assign_kernel, nb, kTok, smem, st, idx, hist, cnt, off, slot, row_src, cnt_re,
             rank_off, d.T, d.E, d.k, d.R, nb);
  }
  return check_launch("layout_assign_kernel");
}

}  // namespace moe
