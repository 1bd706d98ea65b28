// Router: fp32 logits in a fixed summation order, softmax over all experts,
// top-k by logit (ties to the lower expert), renormalised gates; and the
// router's backward (gate softmax Jacobian, dx and dW_r).
//
// The router is the "moe_router" scope that precedes dispatch in the EP-overlap
// pages (skill card, "HybridEP production benchmark": CUDA-graph scopes
// moe_router + moe_preprocess). Its arithmetic is the layer definition in moe.h.
#include <float.h>

#include <algorithm>
#include <atomic>

#include "moe_internal.cuh"

namespace moe {

// Time limit of the fused dispatch's grid-barrier waits, read at each launch.
constexpr unsigned long long kDefaultBarrierWaitNs = 2000000000ull;  // 2 s
std::atomic<unsigned long long> g_barrier_wait_ns{kDefaultBarrierWaitNs};

namespace {


__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

__device__ __forceinline__ void unpack8_f32(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    f[2 * q] = __uint_as_float(w[q] << 16);
    f[2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
  }
}

// An unsigned key in the order of the fp32 values (larger value, larger key),
// -0 mapped to +0 so that the two tie as they compare; every key of a value is
// above 0, which marks "no candidate".
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t b = __float_as_uint(v + 0.0f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Top-k (or the forced set), softmax over all E and renormalised gates of one
// token, by one warp; zt is the token's row of logits (global or shared).
template <int EPL>
__device__ __forceinline__ void topk_row(const float* zt, int t, int32_t* __restrict__ idx,
                                         float* __restrict__ gates, int E, int k, int forced,
                                         int lane, int* s_hist = nullptr) {
  float v[EPL];
  float m = -FLT_MAX;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? zt[e] : -INFINITY;
    m = fmaxf(m, v[i]);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < EPL; ++i)
    if (lane + 32 * i < E) s += expf(v[i] - m);
#pragma unroll
  for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);

  // chosen expert and its softmax probability for slot j, held by lane j
  int my_e = -1;
  float my_p = 0.f;
  if (forced) {
    if (lane < k) {
      my_e = (int)(((long long)k * t + lane) % E);
      my_p = expf(zt[my_e] - m) / s;
    }
  } else {
    // k rounds of a warp argmax: the largest value among the experts not yet
    // taken, ties (equal values; -0 equals +0) to the lower expert index. A
    // round is two warp reductions: the largest key, then the lowest expert
    // among the lanes holding it (each lane offers its own best, the first of
    // its equal keys being its lowest expert).
    uint32_t key[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) key[i] = lane + 32 * i < E ? order_key(v[i]) : 0u;
    uint32_t taken = 0;
    for (int j = 0; j < k; ++j) {
      uint32_t lk = 0u;
      int li = 0;
      float lv = 0.f;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const uint32_t ki = ((taken >> i) & 1u) ? 0u : key[i];
        if (ki > lk) {
          lk = ki;
          li = i;
          lv = v[i];
        }
      }
      const uint32_t mk = __reduce_max_sync(0xffffffffu, lk);
      const uint32_t be =
          __reduce_min_sync(0xffffffffu, lk == mk && mk != 0u ? (uint32_t)(lane + 32 * li) : ~0u);
      const float bv = __shfl_sync(0xffffffffu, lv, (int)(be & 31u));
      if (be != ~0u && (int)(be & 31u) == lane) taken |= 1u << (be >> 5);
      if (lane == j) {
        my_e = be != ~0u ? (int)be : -1;
        my_p = be != ~0u ? expf(bv - m) / s : 0.f;
      }
    }
  }
  float ps = lane < k ? my_p : 0.f;
#pragma unroll
  for (int o = 16; o; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
  if (lane < k) {
    idx[(size_t)t * k + lane] = my_e;
    gates[(size_t)t * k + lane] = my_p / ps;
    if (s_hist && (unsigned)my_e < (unsigned)E) atomicAdd(s_hist + my_e, 1);
  }
}

// z[t, e] for a tile of 4*TPL tokens x 128 experts, one block of kRouteNw
// warps. Every logit runs over h = 0..H-1 in ascending order with one fused
// multiply-add per step; since a bf16*bf16 product is exact in fp32, each step
// is a single fp32 rounding of (acc + x*w), the order both sides of the parity
// check use.
//
// Lane (tg, eg) = (lane / 8, lane % 8) of warp w owns tokens tg + 4u (u < TPL)
// and experts EW*w + eg + 8i (i < EW/8, EW = 128/kRouteNw experts per warp).
// The host sizes TPL so that the grid is about one wave of the SMs. The block
// is limited by shared-memory wavefronts per FMA: a warp-wide 16-byte shared
// load costs about one wavefront per 4 bytes a lane receives, broadcast or
// not, so operands stay bf16 in shared memory (8 steps of h per 16-byte load)
// and each step is one mixed-precision fma.rn.f32.bf16: the bf16 factors
// widen exactly and the sum is rounded once, the same bits as fmaf on the
// widened values, with no unpacking instructions.
// Chunks of 64 h are copied with cp.async into a 4-stage ring (rows padded to
// 144 bytes: the 4 token rows and 8 expert rows a warp reads at once sit on
// distinct banks).
//
// With FUSE (E <= 128: the block holds every expert of its tokens), the block
// then parks its logits in shared memory and each warp routes its tokens
// (topk_row), which saves the logits round trip and a launch.
constexpr int kRouteEb = 128;  // experts per block
constexpr int kRouteNw = 8;    // warps per block
// h per staged chunk, HC: 128 when H is a multiple of 128, else 64 (H is a
// multiple of 64). 128 halves the block barriers and cp.async waits per FMA:
// on the 4096-token layer the fused dispatch went from 93 to 89 us.
template <int HC>
struct RouteChunk {
  static constexpr int kPitchB = HC * 2 + 16;  // bytes per staged row
  static constexpr int kPieces = HC / 8;       // 16-byte pieces per staged row
};
// 4 stages: 1 us faster than 3 on the 4096-token layer
constexpr int kRouteStages = 4;

__device__ __forceinline__ void fma_bf16_lo(float& acc, uint32_t x, uint32_t w) {
  asm("{\n\t.reg .b16 xl, xh, wl, wh;\n\tmov.b32 {xl, xh}, %1;\n\tmov.b32 {wl, wh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, xl, wl, %0;\n\t}"
      : "+f"(acc)
      : "r"(x), "r"(w));
}
__device__ __forceinline__ void fma_bf16_hi(float& acc, uint32_t x, uint32_t w) {
  asm("{\n\t.reg .b16 xl, xh, wl, wh;\n\tmov.b32 {xl, xh}, %1;\n\tmov.b32 {wl, wh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, xh, wh, %0;\n\t}"
      : "+f"(acc)
      : "r"(x), "r"(w));
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Shared memory of one tile: the operand ring (and, with FUSE, the parked logits).
template <int TPL, int HC>
constexpr size_t route_tile_smem() {
  return (size_t)kRouteStages * (4 * TPL + kRouteEb) * RouteChunk<HC>::kPitchB;
}

// One tile: tokens t0.. (4*TPL of them) x experts e0..e0+127, by the whole block.
template <int TPL, bool FUSE, int HC>
__device__ __forceinline__ void route_tile(uint8_t* route_smem, int t0, int e0,
                                           const bf16* __restrict__ x,
                                           const bf16* __restrict__ w_r,
                                           const float* __restrict__ bias, float* __restrict__ z,
                                           int32_t* __restrict__ idx, float* __restrict__ gates,
                                           int T, int H, int E, int k, int forced,
                                           int* s_hist = nullptr) {
  constexpr int NW = kRouteNw, NT = NW * 32;
  constexpr int TB = 4 * TPL;
  constexpr int EW = kRouteEb / NW;  // experts per warp
  constexpr int EPL = EW / 8;        // experts per lane
  constexpr int ROWS = TB + kRouteEb;
  constexpr int PITCH = RouteChunk<HC>::kPitchB, PPR = RouteChunk<HC>::kPieces;
  constexpr int STAGE_B = ROWS * PITCH;
  constexpr int PIECES = ROWS * PPR;  // 16-byte pieces per chunk
  static_assert(EPL >= 1, "route tile");
  static_assert(STAGE_B * kRouteStages == route_tile_smem<TPL, HC>(), "route tile smem");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tg = lane >> 3, eg = lane & 7;
  const int nchunks = H / HC;

  // rows 0..TB-1 of a stage: x (tokens, clamped to T-1); rows TB..: w_r
  // (experts; rows past E are zero-filled)
  auto issue = [&](int ch) {
    if (ch < nchunks) {
      uint8_t* stage = route_smem + (ch % kRouteStages) * STAGE_B;
      for (int pc = threadIdx.x; pc < PIECES; pc += NT) {
        const int row = pc / PPR, piece = pc % PPR;
        const bf16* src;
        bool valid = true;
        if (row < TB) {
          src = x + (size_t)min(t0 + row, T - 1) * H;
        } else {
          const int e = e0 + row - TB;
          valid = e < E;
          src = w_r + (size_t)(valid ? e : 0) * H;
        }
        cp_async16(stage + row * PITCH + piece * 16, src + ch * HC + piece * 8,
                   valid);
      }
    }
    cp_async_commit();
  };

  float acc[TPL][EPL];
#pragma unroll
  for (int u = 0; u < TPL; ++u)
#pragma unroll
    for (int i = 0; i < EPL; ++i) acc[u][i] = 0.f;

#pragma unroll
  for (int s0 = 0; s0 < kRouteStages - 1; ++s0) issue(s0);
  for (int ch = 0; ch < nchunks; ++ch) {
    cp_async_wait<kRouteStages - 2>();
    __syncthreads();  // chunk ch landed for every thread; chunk ch-1 fully consumed
    issue(ch + kRouteStages - 1);
    const uint8_t* stage = route_smem + (ch % kRouteStages) * STAGE_B;
    const uint8_t* xrow = stage + tg * PITCH;
    const uint8_t* wrow = stage + (TB + EW * warp + eg) * PITCH;
#pragma unroll
    for (int s8 = 0; s8 < HC / 8; ++s8) {
      uint4 xv[TPL], wv[EPL];
#pragma unroll
      for (int u = 0; u < TPL; ++u)
        xv[u] = *reinterpret_cast<const uint4*>(xrow + 4 * u * PITCH + 16 * s8);
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        wv[i] = *reinterpret_cast<const uint4*>(wrow + 8 * i * PITCH + 16 * s8);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int u = 0; u < TPL; ++u) {
          const uint32_t xq = q == 0 ? xv[u].x : q == 1 ? xv[u].y : q == 2 ? xv[u].z : xv[u].w;
#pragma unroll
          for (int i = 0; i < EPL; ++i) {
            const uint32_t wq = q == 0 ? wv[i].x : q == 1 ? wv[i].y : q == 2 ? wv[i].z : wv[i].w;
            fma_bf16_lo(acc[u][i], xq, wq);
          }
        }
#pragma unroll
        for (int u = 0; u < TPL; ++u) {
          const uint32_t xq = q == 0 ? xv[u].x : q == 1 ? xv[u].y : q == 2 ? xv[u].z : xv[u].w;
#pragma unroll
          for (int i = 0; i < EPL; ++i) {
            const uint32_t wq = q == 0 ? wv[i].x : q == 1 ? wv[i].y : q == 2 ? wv[i].z : wv[i].w;
            fma_bf16_hi(acc[u][i], xq, wq);
          }
        }
      }
    }
  }
  cp_async_wait<0>();
  float* zs = reinterpret_cast<float*>(route_smem);  // TB x 128 floats
  if (FUSE) __syncthreads();
#pragma unroll
  for (int u = 0; u < TPL; ++u) {
    const int tl = tg + 4 * u, t = t0 + tl;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int el = EW * warp + eg + 8 * i, e = e0 + el;
      if (e < E) {
        float v = acc[u][i];
        if (bias) v = __fadd_rn(v, __ldg(bias + e));
        if (t < T) z[(size_t)t * E + e] = v;
        if (FUSE) zs[tl * kRouteEb + el] = v;
      }
    }
  }
  if (FUSE) {
    __syncthreads();
    for (int tl = warp; tl < TB; tl += NW)
      if (t0 + tl < T)
        topk_row<kRouteEb / 32>(zs + tl * kRouteEb, t0 + tl, idx, gates, E, k, forced, lane,
                                s_hist);
  }
}

template <int TPL, bool FUSE, int HC>
__global__ void __launch_bounds__(kRouteNw * 32, 1) route_logits_kernel(
    const bf16* __restrict__ x, const bf16* __restrict__ w_r, const float* __restrict__ bias,
    float* __restrict__ z, int32_t* __restrict__ idx, float* __restrict__ gates, int T, int H,
    int E, int k, int forced) {
  pdl_wait();
  extern __shared__ __align__(16) uint8_t route_smem[];
  route_tile<TPL, FUSE, HC>(route_smem, blockIdx.x * 4 * TPL, blockIdx.y * kRouteEb, x, w_r, bias, z,
                        idx, gates, T, H, E, k, forced);
}

// One warp per token, logits from global memory (E > 128).
template <int EPL>
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ z,
                                                         int32_t* __restrict__ idx,
                                                         float* __restrict__ gates, int T, int E,
                                                         int k, int forced) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  topk_row<EPL>(z + (size_t)t * E, t, idx, gates, E, k, forced, lane);
}

// ------------------------------------------------------------------ fused dispatch
// Routing, dispatch layout and permute of every token in one cooperative
// persistent launch (E <= 128), the fused dispatch the skill card mentions
// (moe_permute_fusion, "HybridEP production benchmark" and the dispatcher
// table). Tiles of 4*TPL tokens (<= 32, so one warp holds a tile's tokens) go
// to blocks round-robin in token order; fhist[tile][e] counts tile entries
// per expert.
//   1. each block routes its tiles (route_tile) and writes their histograms;
//   -- grid barrier --
//   2. block b turns column e = b, b+G, .. of fhist into exclusive prefixes
//      over tiles, in place, and writes the column total to tot[e];
//   -- grid barrier --
//   3. every block scans tot into the expert offsets (block 0 writes cnt, off,
//      cnt_re, rank_off); slot of entry (t, j) with e = idx[t][j] is
//      off[e] + fhist[tile][e] + (tokens of the tile before t that chose e),
//      which is the layout's stable token order; the block then copies each
//      of its tokens' x rows to their k slots of x_perm.
// The results are those of route + layout + permute run separately. The
// launch is cooperative, so every block is resident and the barrier waits
// end; each is still bounded, and on expiry the block records the site and
// returns.

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// All blocks of the grid arrive; true once every block has, false when the
// wait ran longer than wait_ns (the site is then recorded in the status words).
__device__ __forceinline__ bool grid_barrier(int* bar, int target, int* status, int site,
                                             int* s_flag, uint64_t wait_ns) {
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    __threadfence();
    atomicAdd(bar, 1);
    const uint64_t t0 = global_ns();
    while (ld_acquire_gpu(bar) < target) {
      if (global_ns() - t0 > wait_ns) {
        atomicExch(status + ST_TIMEOUT, site);
        ok = 0;
        break;
      }
      __nanosleep(32);
    }
    __threadfence();
    *s_flag = ok;
  }
  __syncthreads();
  return *s_flag != 0;
}

// Shared memory of the fused dispatch beyond the route tile's.
constexpr size_t kFusedExtraInts = 3 * kRouteEb + 32 * 32 + 4;

template <int TPL, int HC>
__global__ void __launch_bounds__(kRouteNw * 32, 1) dispatch_fused_kernel(
    const bf16* __restrict__ x, const bf16* __restrict__ w_r, const float* __restrict__ bias,
    float* __restrict__ z, int32_t* __restrict__ idx, float* __restrict__ gates,
    int32_t* __restrict__ cnt, int32_t* __restrict__ off, int32_t* __restrict__ slot,
    int32_t* __restrict__ row_src, int32_t* __restrict__ cnt_re, int32_t* __restrict__ rank_off,
    bf16* __restrict__ x_perm, int* __restrict__ fhist, int* __restrict__ bar,
    int* __restrict__ status, int T, int H, int E, int k, int R, int forced, uint64_t wait_ns,
    int* __restrict__ zero, int nzero) {
  pdl_wait();
  // the next launch's counters (see launch_dispatch_fused)
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < nzero; i += blockDim.x) zero[i] = 0;
  constexpr int TB = 4 * TPL;
  static_assert(TB <= 32, "one warp holds a tile's tokens");
  extern __shared__ __align__(16) uint8_t route_smem[];
  int* s_hist = reinterpret_cast<int*>(route_smem + route_tile_smem<TPL, HC>());  // [128]
  uint32_t* s_mask = reinterpret_cast<uint32_t*>(s_hist + kRouteEb);        // [128]
  int* s_base = reinterpret_cast<int*>(s_mask + kRouteEb);                  // [128]
  int* s_ent = s_base + kRouteEb;                                           // [TB * k <= 1024]
  int* s_flag = s_ent + 32 * 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntiles = (T + TB - 1) / TB;
  int* tot = fhist + (size_t)ntiles * E;

  // 1. route, counting each tile's entries per expert as the top-k picks them
  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_hist[e] = 0;
    // (route_tile synchronises the block before its top-k step)
    route_tile<TPL, true, HC>(route_smem, tile * TB, 0, x, w_r, bias, z, idx, gates, T, H, E, k,
                          forced, s_hist);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) fhist[(size_t)tile * E + e] = s_hist[e];
    __syncthreads();
  }
  if (!grid_barrier(bar, gridDim.x, status, 20, s_flag, wait_ns)) return;

  // 2. exclusive prefix over tiles, one expert column per block and round;
  // 8 x 32 tiles are loaded before they are scanned
  if (warp == 0) {
    for (int e = blockIdx.x; e < E; e += gridDim.x) {
      int carry = 0;
      for (int b0 = 0; b0 < ntiles; b0 += 256) {
        int c[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int b = b0 + 32 * u + lane;
          c[u] = b < ntiles ? __ldcg(fhist + (size_t)b * E + e) : 0;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int b = b0 + 32 * u + lane;
          int incl = c[u];
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
          }
          if (b < ntiles) fhist[(size_t)b * E + e] = carry + incl - c[u];
          carry += __shfl_sync(0xffffffffu, incl, 31);
        }
      }
      if (lane == 0) tot[e] = carry;
    }
  }
  if (!grid_barrier(bar, 2 * (int)gridDim.x, status, 21, s_flag, wait_ns)) return;

  // 3. expert offsets, then slots and rows tile by tile
  if (warp == 0) {
    int c[kRouteEb / 32];
#pragma unroll
    for (int u = 0; u < kRouteEb / 32; ++u) {
      const int e = 32 * u + lane;
      c[u] = e < E ? __ldcg(tot + e) : 0;
    }
    int carry = 0;
#pragma unroll
    for (int u = 0; u < kRouteEb / 32; ++u) {
      const int e = 32 * u + lane;
      int incl = c[u];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      if (e < E) {
        const int ex = carry + incl - c[u];
        s_base[e] = ex;
        if (blockIdx.x == 0) {
          off[e] = ex;
          cnt[e] = c[u];
          cnt_re[e] = c[u];  // [R][E/R] row-major is the expert order itself
        }
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (blockIdx.x == 0 && lane == 0) off[E] = carry;
    if (lane == 0) *s_flag = carry;  // N
  }
  __syncthreads();
  if (blockIdx.x == 0) {
    const int El = E / R;
    for (int r = threadIdx.x; r <= R; r += blockDim.x)
      rank_off[r] = r < R ? s_base[r * El] : *s_flag;
  }
  const int cpr = H / 8;  // 16-byte chunks per row
  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int t0 = tile * TB, nt = min(TB, T - t0), nent = nt * k;
    // the tile's routing and its entries' offsets within each expert
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      s_mask[e] = 0u;
      s_hist[e] = __ldcg(fhist + (size_t)tile * E + e);
    }
    for (int i = threadIdx.x; i < nent; i += blockDim.x) s_ent[i] = idx[(size_t)t0 * k + i];
    __syncthreads();
    for (int i = threadIdx.x; i < nent; i += blockDim.x) {
      const int e = s_ent[i];
      if ((unsigned)e < (unsigned)E) atomicOr(&s_mask[e], 1u << (i / k));
    }
    __syncthreads();
    // entry i = (token t0 + i / k, choice i % k): its slot, in place of its expert
    for (int i = threadIdx.x; i < nent; i += blockDim.x) {
      const int e = s_ent[i];
      int sl = -1;
      if ((unsigned)e < (unsigned)E) {
        sl = s_base[e] + s_hist[e] + __popc(s_mask[e] & ((1u << (i / k)) - 1u));
        row_src[sl] = t0 * k + i;
      } else {
        atomicAdd(status + ST_BAD_INDEX, 1);
      }
      slot[(size_t)t0 * k + i] = sl;
      s_ent[i] = sl;
    }
    __syncthreads();
    // warp w copies tokens w, w + 8, ..: 4 KB of the row at a time, loaded
    // once and stored to each of the token's k slots
    for (int tl = warp; tl < nt; tl += kRouteNw) {
      const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)(t0 + tl) * H);
      for (int c0 = 0; c0 < cpr; c0 += 256) {
        uint4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int c = c0 + 32 * u + lane;
          v[u] = c < cpr ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
        }
        for (int j = 0; j < k; ++j) {
          const int sl = s_ent[tl * k + j];
          if (sl < 0) continue;
          uint4* dst = reinterpret_cast<uint4*>(x_perm + (size_t)sl * H);
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int c = c0 + 32 * u + lane;
            if (c < cpr) __stcs(dst + c, v[u]);
          }
        }
      }
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ backward
// dz_j = g_j (dg_j - <g, dg>) on the chosen set;
// dx = bf16(dx32 + sum_j dz_j * w_r[i_j]), j ascending.
// A block owns `tok` tokens x one slice of COLS columns of the row: the
// slice of w_r (E x COLS) is staged in shared memory once, so the k expert
// rows a token adds come from shared memory instead of k gathers through L2.
// The block's routing state (k experts, slots, gates and gate gradients of
// each token: a contiguous range of the [T, k] arrays) is staged with
// coalesced loads in one round trip, and one thread per token works out its
// dz there. Then COLS / 8 threads per token each handle one 16-byte chunk of
// the slice, with the token's k row loads in flight together and no
// routing-state load between one token and the next.
// FUSED: the dispatch backward is done in the same pass and dx32 is never
// stored: the row sum dx32[t] = sum_j dx_perm[slot[t,j]] (fp32, j ascending,
// from 0) is formed in registers exactly as the standalone permute backward
// forms it, then the router term is added in the same order as above, so the
// two paths give the same bits.
// Measured on the 4096-token layer: 128-column slices of 64 tokens take 40 us,
// 64-column slices of 128 tokens 43 us, 256 x 64 56 us, and the earlier form,
// whose threads loaded each token's routing state themselves, 46 us. Two
// tokens' row loads in flight per thread took 61 us: the registers they need
// cut the blocks per SM from four to two. Blocks that kept their slice and
// took token blocks in turn, with the next one's routing state loaded beside
// the current rows (as the combine kernels do), took 45 us. The launcher picks
// the tokens per block that fill whole waves of resident blocks (112 there:
// 592 blocks on 608 slots, 37 us), since a partly filled last wave costs more
// than longer blocks: 64 tokens per block (1.7 waves) took 41 us, 96 and 128
// (1.1 and 0.84 waves) 47 us.
constexpr int kDxTokMax = 128;  // tokens per block, at most
constexpr int kDxCols = 128;  // columns per slice when H allows (else 64)
// bytes per staged w_r slice row, for a slice of COLS columns
__host__ __device__ constexpr int dx_pitch(int cols) { return cols * 2 + 16; }

// dynamic shared memory of the dx kernel: the w_r slice, then per routed
// entry of the block's tokens its expert, slot, gate and dz
__host__ __device__ constexpr size_t dx_smem_bytes(int cols, int E, int k, int tok) {
  return (size_t)E * dx_pitch(cols) + (size_t)tok * k * 16;
}

template <int KMAX, bool FUSED, int COLS>
__global__ void __launch_bounds__(256) route_bwd_dx_kernel(
    const float* __restrict__ dgates, const float* __restrict__ gates,
    const int32_t* __restrict__ idx, const bf16* __restrict__ w_r, const float* __restrict__ dx32,
    const bf16* __restrict__ dx_perm, const int32_t* __restrict__ slot, bf16* __restrict__ dx,
    float* __restrict__ dz, int T, int H, int E, int k, int* status, int tok) {
  pdl_wait();
  constexpr int KB = KMAX < 8 ? KMAX : 8;  // row loads per batch
  constexpr int LANES = COLS / 8;            // threads per token: 16 bytes of the slice each
  constexpr int TPP = 256 / LANES;           // tokens per pass of the block
  constexpr int PITCH = dx_pitch(COLS);
  extern __shared__ __align__(16) uint8_t s_wr[];  // [E][PITCH], then the routing state
  int* s_e = reinterpret_cast<int*>(s_wr + (size_t)E * PITCH);  // [tok * k]
  int* s_slot = s_e + tok * k;
  float* s_g = reinterpret_cast<float*>(s_slot + tok * k);
  float* s_dz = s_g + tok * k;  // dg while staged, then dz
  const int t0 = blockIdx.y * tok;
  const int nt = min(tok, T - t0);
  const int nent = nt * k;
  const size_t tk0 = (size_t)t0 * k;
  const long long N = (long long)T * k;
  // slices vary fastest across the grid: blocks resident together read
  // different column windows of the rows
  const int c = blockIdx.x * LANES + (threadIdx.x % LANES);  // 16-byte chunk of the row
  for (int i = threadIdx.x; i < E * LANES; i += blockDim.x) {
    const int e = i / LANES, q = i % LANES;
    *reinterpret_cast<uint4*>(s_wr + e * PITCH + q * 16) =
        __ldg(reinterpret_cast<const uint4*>(w_r + (size_t)e * H) + blockIdx.x * LANES + q);
  }
  for (int i = threadIdx.x; i < nent; i += blockDim.x) {
    const int e = __ldg(idx + tk0 + i);
    s_e[i] = (unsigned)e < (unsigned)E ? e : -1;
    if (FUSED) {
      const int sv = __ldg(slot + tk0 + i);
      s_slot[i] = sv >= 0 && sv < N ? sv : -1;
    }
    s_g[i] = __ldg(gates + tk0 + i);
    s_dz[i] = __ldg(dgates + tk0 + i);
  }
  __syncthreads();
  if ((int)threadIdx.x < nt) {
    const int b = threadIdx.x * k;
    float inner = 0.f;
    for (int j = 0; j < k; ++j) inner = fmaf(s_g[b + j], s_dz[b + j], inner);
    const bool writer = blockIdx.x == 0;
    for (int j = 0; j < k; ++j) {
      const float v = s_g[b + j] * (s_dz[b + j] - inner);
      s_dz[b + j] = v;
      if (writer) {
        dz[tk0 + b + j] = v;
        if (s_e[b + j] < 0) atomicAdd(status + ST_BAD_INDEX, 1);
      }
    }
  }
  __syncthreads();
  const uint8_t* wchunk = s_wr + (threadIdx.x % LANES) * 16;
  for (int tl = threadIdx.x / LANES; tl < nt; tl += TPP) {
    float acc[8];
    if (FUSED) {
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = 0.f;
#pragma unroll
      for (int j0 = 0; j0 < KMAX; j0 += KB) {
        uint4 v[KB];
#pragma unroll
        for (int u = 0; u < KB; ++u) {
          const int j = j0 + u;
          const int sv = j < k ? s_slot[tl * k + j] : -1;
          v[u] = sv >= 0 ? __ldcs(reinterpret_cast<const uint4*>(dx_perm + (size_t)sv * H) + c)
                         : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < KB; ++u) {
          if (j0 + u < k) {
            float f[8];
            unpack8_f32(v[u], f);
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] += f[q];
          }
        }
      }
    } else {
      const float4* src = reinterpret_cast<const float4*>(dx32 + (size_t)(t0 + tl) * H + c * 8);
      const float4 p0 = src[0], p1 = src[1];
      acc[0] = p0.x; acc[1] = p0.y; acc[2] = p0.z; acc[3] = p0.w;
      acc[4] = p1.x; acc[5] = p1.y; acc[6] = p1.z; acc[7] = p1.w;
    }
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (j < k) {
        const int e = s_e[tl * k + j];
        if (e >= 0) {
          const float dzj = s_dz[tl * k + j];
          const uint4 wv = *reinterpret_cast<const uint4*>(wchunk + e * PITCH);
          const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            acc[2 * q] = fmaf(dzj, bf16_bits_to_f32(w[q] & 0xFFFFu), acc[2 * q]);
            acc[2 * q + 1] = fmaf(dzj, bf16_bits_to_f32(w[q] >> 16), acc[2 * q + 1]);
          }
        }
      }
    }
    uint4 out;
    uint32_t* o = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
      o[q] = *reinterpret_cast<uint32_t*>(&b2);
    }
    *reinterpret_cast<uint4*>(dx + (size_t)(t0 + tl) * H + c * 8) = out;
  }
}

// Expert row chunks: expert e's rows off[e]..off[e+1]-1 are cut into chunks of
// kRouteBwdRowsPerChunk; chunk c of the whole layer maps to (e, first row).
// Each block finds its chunk from the per-expert chunk prefix.
__device__ int find_chunk(const int32_t* __restrict__ off, int E, int chunk, int* e_out,
                          int* r0_out, int* r1_out, int* s_prefix) {
  // s_prefix: shared [E+1]; computed by warp 0
  if (threadIdx.x < 32) {
    int carry = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + threadIdx.x;
      int c = 0;
      if (e < E) c = (off[e + 1] - off[e] + kRouteBwdRowsPerChunk - 1) / kRouteBwdRowsPerChunk;
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if ((int)threadIdx.x >= o) incl += n;
      }
      if (e < E) s_prefix[e] = carry + incl - c;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (threadIdx.x == 0) s_prefix[E] = carry;
  }
  __syncthreads();
  if (chunk >= s_prefix[E]) return 0;
  int lo = 0, hi = E - 1;  // last e with s_prefix[e] <= chunk
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_prefix[mid] <= chunk) lo = mid; else hi = mid - 1;
  }
  // skip experts with zero chunks that share the same prefix value
  const int e = lo;
  const int r0 = off[e] + (chunk - s_prefix[e]) * kRouteBwdRowsPerChunk;
  *e_out = e;
  *r0_out = r0;
  *r1_out = min(r0 + kRouteBwdRowsPerChunk, (int)off[e + 1]);
  return 1;
}

// dW_r, in one launch. A block takes one chunk of an expert's rows and one
// column block of 2048 columns: partial[chunk][h] = sum over the chunk's rows s
// (ascending) of dz[row_src[s]] * x[row_src[s] div k][h]. The chunk's sources
// and weights are staged in shared memory first, so each thread then has 8
// independent x-row loads in flight instead of a chain of dependent loads per
// row. The block that completes an expert (a per-expert, per-column-block
// counter, counted after each block's partial is visible) then adds the
// expert's partials in chunk order: dW_r[e][h] = sum_i partial[first + i][h],
// a fixed order whatever the order in which the chunks finish, and resets the
// counter. Blocks past the last chunk write zeros for the experts without
// rows, one each (there are always enough of them: the grid has
// ceil(N / 64) + E blocks along x).
__global__ void __launch_bounds__(256) route_bwd_dwr_kernel(
    const int32_t* __restrict__ off, const int32_t* __restrict__ row_src,
    const float* __restrict__ dz, const bf16* __restrict__ x, float* __restrict__ part,
    float* __restrict__ dw_r, int* __restrict__ cnt, int T, int H, int E, int k,
    int* status) {
  pdl_wait();
  extern __shared__ int s_prefix[];
  __shared__ int s_tok[kRouteBwdRowsPerChunk];
  __shared__ float s_w[kRouteBwdRowsPerChunk];
  __shared__ int s_sel;
  const int c = blockIdx.y * blockDim.x + threadIdx.x;  // 16-byte chunk of the row
  const bool col_ok = c * 8 < H;
  int e, r0, r1;
  if (!find_chunk(off, E, blockIdx.x, &e, &r0, &r1, s_prefix)) {
    // a spare block: the j-th expert without rows, if there is one, gets zeros
    const int j = blockIdx.x - s_prefix[E];
    if (threadIdx.x < 32) {
      int seen = 0, pick = -1;
      for (int base = 0; base < E && pick < 0; base += 32) {
        const int ee = base + threadIdx.x;
        const bool empty = ee < E && off[ee + 1] == off[ee];
        const unsigned m = __ballot_sync(0xffffffffu, empty);
        const int n = __popc(m);
        if (j >= seen && j < seen + n) {
          unsigned mm = m;
          for (int q = 0; q < j - seen; ++q) mm &= mm - 1;  // drop the lower empties
          pick = base + __ffs(mm) - 1;
        }
        seen += n;
      }
      if (threadIdx.x == 0) s_sel = pick;
    }
    __syncthreads();
    if (s_sel >= 0 && col_ok) {
      float4* dst = reinterpret_cast<float4*>(dw_r + (size_t)s_sel * H + c * 8);
      dst[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      dst[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    return;
  }
  const long long N = (long long)T * k;
  const int n = r1 - r0;
  if ((int)threadIdx.x < n) {
    const int src = row_src[r0 + threadIdx.x];
    const bool ok = src >= 0 && src < N;
    s_tok[threadIdx.x] = ok ? src / k : -1;
    s_w[threadIdx.x] = ok ? dz[src] : 0.f;
  }
  __syncthreads();
  if (col_ok) {
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int s0 = 0; s0 < n; s0 += 8) {
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int tok = s0 + u < n ? s_tok[s0 + u] : -1;
        v[u] = tok >= 0 ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)tok * H) + c)
                        : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (s0 + u < n) {
          const float w = s_w[s0 + u];
          const uint32_t q4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            acc[2 * q] = fmaf(w, bf16_bits_to_f32(q4[q] & 0xFFFFu), acc[2 * q]);
            acc[2 * q + 1] = fmaf(w, bf16_bits_to_f32(q4[q] >> 16), acc[2 * q + 1]);
          }
        }
      }
    }
    float4* dst = reinterpret_cast<float4*>(part + (size_t)blockIdx.x * H + c * 8);
    dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
  // publish this partial; the expert's last chunk to finish sums them all
  __threadfence();
  __syncthreads();
  const int first = s_prefix[e];
  const int nch = (n > 0 ? (off[e + 1] - off[e] + kRouteBwdRowsPerChunk - 1) /
                               kRouteBwdRowsPerChunk
                         : 0);
  int* ctr = cnt + (size_t)e * gridDim.y + blockIdx.y;
  if (threadIdx.x == 0) s_sel = atomicAdd(ctr, 1) == nch - 1;
  __syncthreads();
  if (!s_sel) return;
  __threadfence();
  if (col_ok) {
    float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
    for (int i = 0; i < nch; ++i) {
      const float4* p4 = reinterpret_cast<const float4*>(part + (size_t)(first + i) * H + c * 8);
      const float4 p0 = __ldcg(p4), p1 = __ldcg(p4 + 1);
      a0.x += p0.x; a0.y += p0.y; a0.z += p0.z; a0.w += p0.w;
      a1.x += p1.x; a1.y += p1.y; a1.z += p1.z; a1.w += p1.w;
    }
    float4* dst = reinterpret_cast<float4*>(dw_r + (size_t)e * H + c * 8);
    dst[0] = a0;
    dst[1] = a1;
  }
  if (threadIdx.x == 0) *ctr = 0;  // ready for the next launch
}

}  // namespace

template <int TPL, bool FUSE, int HC>
cudaError_t launch_logits_t(const moe_layer_desc_t& d, dim3 grid, const bf16* x, const bf16* w_r,
                            const float* bias, float* logits, int32_t* idx, float* gates,
                            cudaStream_t st) {
  const int forced = d.mode == MOE_ROUTE_FORCED_BALANCED;
  constexpr size_t smem = route_tile_smem<TPL, HC>();
  static cudaError_t attr = cudaFuncSetAttribute(
      route_logits_kernel<TPL, FUSE, HC>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (attr != cudaSuccess) return attr;
  launch_k(route_logits_kernel<TPL, FUSE, HC>, grid, kRouteNw * 32, smem, st, x, w_r, bias, logits,
           idx, gates, d.T, d.H, d.E, d.k, forced);
  return cudaSuccess;
}

template <int TPL>
cudaError_t launch_logits(const moe_layer_desc_t& d, dim3 grid, bool fuse, const bf16* x,
                          const bf16* w_r, const float* bias, float* logits, int32_t* idx,
                          float* gates, cudaStream_t st) {
  // (the unfused form, for E > 128, keeps 64-h chunks: fewer instantiations)
  if (!fuse) return launch_logits_t<TPL, false, 64>(d, grid, x, w_r, bias, logits, idx, gates, st);
  return d.H % 128 == 0
             ? launch_logits_t<TPL, true, 128>(d, grid, x, w_r, bias, logits, idx, gates, st)
             : launch_logits_t<TPL, true, 64>(d, grid, x, w_r, bias, logits, idx, gates, st);
}

moe_status_t launch_route(const moe_layer_desc_t& d, const bf16* x, const bf16* w_r,
                          const float* bias, float* logits, int32_t* idx, float* gates,
                          int* status, cudaStream_t st) {
  (void)status;
  if (d.T == 0) return MOE_OK;
  // tokens per lane: the smallest TPL (<= 7) that covers the tokens in about
  // one wave of one block per SM
  const int gy = ceil_div(d.E, kRouteEb);
  const int per_sm = ceil_div(d.T * gy, 4 * device_sm_count());
  const int tpl = per_sm < 1 ? 1 : per_sm > 7 ? 7 : per_sm;
  const dim3 grid(ceil_div(d.T, 4 * tpl), gy);
  const bool fuse = gy == 1;
  cudaError_t ae;
  {
    LaunchScope _ls(K_ROUTE_LOGITS, st);
    switch (tpl) {
      case 1: ae = launch_logits<1>(d, grid, fuse, x, w_r, bias, logits, idx, gates, st); break;
      case 2: ae = launch_logits<2>(d, grid, fuse, x, w_r, bias, logits, idx, gates, st); break;
      case 3: ae = launch_logits<3>(d, grid, fuse, x, w_r, bias, logits, idx, gates, st); break;
      case 4: ae = launch_logits<4>(d, grid, fuse, x, w_r, bias, logits, idx, gates, st); break;
      case 5: ae = launch_logits<5>(d, grid, fuse, x, w_r, bias, logits, idx, gates, st); break;
      case 6: ae = launch_logits<6>(d, grid, fuse, x, w_r, bias, logits, idx, gates, st); break;
      default: ae = launch_logits<7>(d, grid, fuse, x, w_r, bias, logits, idx, gates, st); break;
    }
  }
  if (ae != cudaSuccess) {
    set_error("route_logits_kernel attribute setup: %s", cudaGetErrorString(ae));
    return MOE_ERR_CUDA;
  }
  moe_status_t s = check_launch("route_logits_kernel");
  if (s != MOE_OK || fuse) return s;
  const int tpb = 256, warps = tpb / 32;
  const int forced = d.mode == MOE_ROUTE_FORCED_BALANCED;
  {
    LaunchScope _ls(K_ROUTE_TOPK, st);
    launch_k(route_topk_kernel<8>, dim3(ceil_div(d.T, warps)), tpb, 0, st, logits, idx, gates, d.T,
             d.E, d.k, forced);
  }
  return check_launch("route_topk_kernel");
}

template <int TPL, int HC>
cudaError_t launch_fused_t(const moe_layer_desc_t& d, const bf16* x, const bf16* w_r,
                           const float* bias, float* z, int32_t* idx, float* gates, int32_t* cnt,
                           int32_t* off, int32_t* slot, int32_t* row_src, int32_t* cnt_re,
                           int32_t* rank_off, bf16* x_perm, int* fhist, int* bar, int* status,
                           cudaStream_t st, int* zero, int nzero, int max_ctas) {
  const int forced = d.mode == MOE_ROUTE_FORCED_BALANCED;
  const size_t smem = route_tile_smem<TPL, HC>() + kFusedExtraInts * sizeof(int);
  // resident blocks per SM, looked up once (with the shared-memory attribute)
  static int per_sm = 0;
  static cudaError_t attr = [smem] {
    cudaError_t a = cudaFuncSetAttribute(dispatch_fused_kernel<TPL, HC>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (a == cudaSuccess)
      a = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dispatch_fused_kernel<TPL, HC>,
                                                        kRouteNw * 32, smem);
    return a;
  }();
  if (attr != cudaSuccess) return attr;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  cudaError_t e;
  // every block must be resident: at most one wave
  const int ntiles = ceil_div(d.T, 4 * TPL);
  int grid = std::min(ntiles, per_sm * device_sm_count());
  if (max_ctas > 0 && max_ctas < grid) grid = max_ctas;
  e = cudaMemsetAsync(bar, 0, sizeof(int), st);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeCooperative;
  at[0].val.cooperative = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kRouteNw * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, dispatch_fused_kernel<TPL, HC>, x, w_r, bias, z, idx, gates, cnt,
                            off, slot, row_src, cnt_re, rank_off, x_perm, fhist, bar, status,
                            d.T, d.H, d.E, d.k, d.R, forced,
                            (uint64_t)g_barrier_wait_ns.load(std::memory_order_relaxed), zero,
                            nzero);
}

template <int KMAX, bool FUSED, int COLS>
cudaError_t launch_dx_c(const moe_layer_desc_t& d, const float* dgates, const float* gates,
                        const int32_t* idx, const bf16* w_r, const float* dx32,
                        const bf16* dx_perm, const int32_t* slot, bf16* dx, float* dz,
                        int* status, cudaStream_t st) {
  // E <= 256, k <= 32: allow the largest once per instantiation
  static const cudaError_t attr = cudaFuncSetAttribute(
      route_bwd_dx_kernel<KMAX, FUSED, COLS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
      (int)dx_smem_bytes(COLS, 256, 32, kDxTokMax));
  if (attr != cudaSuccess) return attr;
  // tokens per block: the fewest waves of resident blocks that hold the layer
  // with at most kDxTokMax tokens a block, then the fewest whole passes of
  // the block's threads (TPP tokens each) that fill those waves
  constexpr int TPP = 256 / (COLS / 8);  // tokens per pass
  int per_sm = 0;
  const cudaError_t oe = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &per_sm, route_bwd_dx_kernel<KMAX, FUSED, COLS>, 256,
      dx_smem_bytes(COLS, d.E, d.k, kDxTokMax));
  if (oe != cudaSuccess) return oe;
  const int slices = d.H / COLS;
  const int per_slice = std::max(1, std::max(per_sm, 1) * device_sm_count() / slices);
  const int waves = ceil_div(d.T, per_slice * kDxTokMax);
  int tok = ceil_div(ceil_div(d.T, waves * per_slice), TPP) * TPP;
  tok = std::min(std::max(tok, TPP), kDxTokMax);
  const dim3 g(slices, ceil_div(d.T, tok));
  const size_t smem = dx_smem_bytes(COLS, d.E, d.k, tok);
  return launch_k(route_bwd_dx_kernel<KMAX, FUSED, COLS>, g, 256, smem, st, dgates, gates, idx,
                  w_r, dx32, dx_perm, slot, dx, dz, d.T, d.H, d.E, d.k, status, tok);
}

// slices of kDxCols columns when H allows, else of 64 (H is a multiple of 64)
template <int KMAX, bool FUSED>
cudaError_t launch_dx_t(const moe_layer_desc_t& d, const float* dgates, const float* gates,
                        const int32_t* idx, const bf16* w_r, const float* dx32,
                        const bf16* dx_perm, const int32_t* slot, bf16* dx, float* dz,
                        int* status, cudaStream_t st) {
  if (d.H % kDxCols == 0)
    return launch_dx_c<KMAX, FUSED, kDxCols>(d, dgates, gates, idx, w_r, dx32, dx_perm, slot, dx,
                                             dz, status, st);
  return launch_dx_c<KMAX, FUSED, 64>(d, dgates, gates, idx, w_r, dx32, dx_perm, slot, dx, dz,
                                      status, st);
}

template <bool FUSED>
cudaError_t launch_dx(const moe_layer_desc_t& d, const float* dgates, const float* gates,
                      const int32_t* idx, const bf16* w_r, const float* dx32, const bf16* dx_perm,
                      const int32_t* slot, bf16* dx, float* dz, int* status, cudaStream_t st) {
  if (d.k <= 4)
    return launch_dx_t<4, FUSED>(d, dgates, gates, idx, w_r, dx32, dx_perm, slot, dx, dz, status,
                                 st);
  if (d.k <= 8)
    return launch_dx_t<8, FUSED>(d, dgates, gates, idx, w_r, dx32, dx_perm, slot, dx, dz, status,
                                 st);
  if (d.k <= 16)
    return launch_dx_t<16, FUSED>(d, dgates, gates, idx, w_r, dx32, dx_perm, slot, dx, dz, status,
                                  st);
  return launch_dx_t<32, FUSED>(d, dgates, gates, idx, w_r, dx32, dx_perm, slot, dx, dz, status,
                                st);
}

moe_status_t launch_dispatch_fused(const moe_layer_desc_t& d, const bf16* x, const bf16* w_r,
                                   const float* bias, float* z, int32_t* idx, float* gates,
                                   int32_t* cnt, int32_t* off, int32_t* slot, int32_t* row_src,
                                   int32_t* cnt_re, int32_t* rank_off, bf16* x_perm, int* fhist,
                                   int* bar, int* status, cudaStream_t st, int* zero, int nzero,
                                   int max_ctas) {
  if (d.T == 0 || d.E > kRouteEb) return MOE_ERR_UNSUPPORTED;
  // tokens per lane as for the router alone: about one wave of one block per SM
  const int per_sm = ceil_div(d.T, 4 * device_sm_count());
  const int tpl = per_sm < 1 ? 1 : per_sm > 7 ? 7 : per_sm;
  cudaError_t e;
  {
    LaunchScope _ls(K_DISPATCH_FUSED, st);
#define MOE_FUSED_CASE(n)                                                                     \
  case n:                                                                                     \
    e = d.H % 128 == 0                                                                        \
            ? launch_fused_t<n, 128>(d, x, w_r, bias, z, idx, gates, cnt, off, slot, row_src, \
                                     cnt_re, rank_off, x_perm, fhist, bar, status, st, zero,  \
                                     nzero, max_ctas)                                         \
            : launch_fused_t<n, 64>(d, x, w_r, bias, z, idx, gates, cnt, off, slot, row_src,  \
                                    cnt_re, rank_off, x_perm, fhist, bar, status, st, zero,   \
                                    nzero, max_ctas);                                         \
    break;
    switch (tpl) {
      MOE_FUSED_CASE(1)
      MOE_FUSED_CASE(2)
      MOE_FUSED_CASE(3)
      MOE_FUSED_CASE(4)
      MOE_FUSED_CASE(5)
      MOE_FUSED_CASE(6)
      default: MOE_FUSED_CASE(7)
    }
#undef MOE_FUSED_CASE
  }
  if (e != cudaSuccess) {
    set_error("dispatch_fused_kernel launch: %s", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  return check_launch("dispatch_fused_kernel");
}

moe_status_t launch_route_bwd(const moe_layer_desc_t& d, const float* dgates, const float* gates,
                              const int32_t* idx, const bf16* x, const bf16* w_r,
                              const int32_t* row_src, const int32_t* off, const float* dx32,
                              const bf16* dx_perm, const int32_t* slot, bf16* dx, float* dw_r,
                              float* dz, float* dwr_part, int* dwr_cnt, bool cnt_zeroed,
                              int* status, cudaStream_t st) {
  const bool fused = dx_perm != nullptr;
  const int cpr = d.H / 8;
  if (d.T > 0) {
    cudaError_t e;
    {
      LaunchScope _ls(fused ? K_DISPATCH_BWD : K_ROUTE_BWD_DX, st);
      if (fused)
        e = launch_dx<true>(d, dgates, gates, idx, w_r, dx32, dx_perm, slot, dx, dz, status, st);
      else
        e = launch_dx<false>(d, dgates, gates, idx, w_r, dx32, dx_perm, slot, dx, dz, status, st);
    }
    if (e != cudaSuccess) {
      set_error("route_bwd_dx_kernel launch: %s", cudaGetErrorString(e));
      return MOE_ERR_CUDA;
    }
    moe_status_t s = check_launch("route_bwd_dx_kernel");
    if (s != MOE_OK) return s;
  }
  const long long N = (long long)d.T * d.k;
  const int max_chunks = (int)((N + kRouteBwdRowsPerChunk - 1) / kRouteBwdRowsPerChunk) + d.E;
  const int ncb = ceil_div(cpr, 256);  // column blocks of 2048 columns
  if (!cnt_zeroed) {
    cudaError_t e = cudaMemsetAsync(dwr_cnt, 0, (size_t)d.E * ncb * sizeof(int), st);
    if (e != cudaSuccess) {
      set_error("cudaMemsetAsync: %s", cudaGetErrorString(e));
      return MOE_ERR_CUDA;
    }
  }
  dim3 ga(max_chunks, ncb);
  {
    LaunchScope _ls(K_ROUTE_BWD_DWR, st);
    launch_k(route_bwd_dwr_kernel, ga, 256, (d.E + 1) * sizeof(int), st, off, row_src, dz, x,
             dwr_part, dw_r, dwr_cnt, d.T, d.H, d.E, d.k, status);
  }
  return check_launch("route_bwd_dwr_kernel");
}

}  // namespace moe

extern "C" uint64_t moe_set_barrier_wait_limit_ns(uint64_t ns) {
  return moe::g_barrier_wait_ns.exchange(ns ? ns : moe::kDefaultBarrierWaitNs);
}
