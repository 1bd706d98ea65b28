// Router: fp32 logits in a fixed summation order, softmax over all experts,
// top-k by logit (ties to the lower expert), renormalised gates; and the
// router's backward (gate softmax Jacobian, dx and dW_r).
//
// The router is the "moe_router" scope that precedes dispatch in the EP-overlap
// pages (skill card, "HybridEP production benchmark": CUDA-graph scopes
// moe_router + moe_preprocess). Its arithmetic is the layer definition in moe.h.
#include <float.h>

#include "moe_internal.cuh"

#ifndef MOE_ROUTE_TPL
#define MOE_ROUTE_TPL 4
#endif

namespace moe {

namespace {

constexpr int kRouteHc = 32;    // hidden elements per chunk

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

// z[t, e] for a tile of 64 tokens x (NW * EPW) experts: lane owns tokens lane
// and lane+32, warp owns EPW experts, 2 x EPW accumulators per thread. Every accumulator
// runs over h = 0..H-1 in ascending order with one fmaf per step; since a
// bf16*bf16 product is exact in fp32, each step is a single fp32 rounding of
// (acc + x*w), the order both sides of the parity check use.
// Per 32-wide chunk of h, x is staged as bf16 (one 16-byte shared load gives a
// lane 8 values of one token; an 80-byte row pitch keeps the 32 lanes' rows on
// distinct banks) and w_r as fp32 read with warp-uniform broadcasts: 24 shared
// wavefronts per 128 FMAs per warp, so the loop is FMA-bound. The next chunk is
// fetched into registers while the current one is consumed (double buffered,
// one barrier per chunk).
constexpr int kRouteXPitchB = 80;  // bytes per staged x row (64 B of data)

template <int NW, int kRouteEpw, int TPL>
__global__ void __launch_bounds__(NW * 32) route_logits_kernel(const bf16* __restrict__ x,
                                                               const bf16* __restrict__ w_r,
                                                               const float* __restrict__ bias,
                                                               float* __restrict__ z, int T,
                                                               int H, int E) {
  constexpr int kRouteTok = 32 * TPL;  // tokens per CTA: lane owns tokens lane + 32u
  constexpr int kThreads = NW * 32;
  constexpr int eb = NW * kRouteEpw;              // experts in this CTA
  constexpr int nxp = kRouteTok * (kRouteHc / 8);  // 16-byte pieces of an x chunk (256)
  constexpr int kXP = nxp / kThreads;              // per thread
  constexpr int kWP = eb * (kRouteHc / 8);         // 16-byte pieces of a w_r chunk
  static_assert(kWP <= kThreads && nxp % kThreads == 0, "staging split");
  __shared__ __align__(16) uint8_t xs[2][kRouteTok * kRouteXPitchB];
  __shared__ __align__(16) float ws[2][eb][kRouteHc];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kRouteTok;
  const int e0 = blockIdx.y * eb;

  float acc[TPL][kRouteEpw];
#pragma unroll
  for (int u = 0; u < TPL; ++u)
#pragma unroll
    for (int i = 0; i < kRouteEpw; ++i) acc[u][i] = 0.f;

  const int wr_row = threadIdx.x / (kRouteHc / 8), wr_col = (threadIdx.x % (kRouteHc / 8)) * 8;
  const bool w_mine = (int)threadIdx.x < kWP;  // this thread stages a w_r piece
  const bool w_ok = w_mine && e0 + wr_row < E;
  const uint4* wrow = reinterpret_cast<const uint4*>(w_r + (size_t)(w_ok ? e0 + wr_row : 0) * H);
  auto fetch = [&](int ch, uint4 (&rx)[kXP], uint4& rw) {
#pragma unroll
    for (int q = 0; q < kXP; ++q) {
      const int i = threadIdx.x + q * kThreads;
      const int row = i / (kRouteHc / 8), col = i % (kRouteHc / 8);
      const int t = min(t0 + row, T - 1);
      rx[q] = __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * H) + ch * (kRouteHc / 8) + col);
    }
    rw = w_ok ? __ldg(wrow + ch * (kRouteHc / 8) + wr_col / 8) : make_uint4(0, 0, 0, 0);
  };
  uint4 rx[kXP], rw;
  fetch(0, rx, rw);
  const int nchunks = H / kRouteHc;
  for (int ch = 0; ch < nchunks; ++ch) {
    const int b = ch & 1;
#pragma unroll
    for (int q = 0; q < kXP; ++q) {
      const int i = threadIdx.x + q * kThreads;
      const int row = i / (kRouteHc / 8), col = i % (kRouteHc / 8);
      *reinterpret_cast<uint4*>(&xs[b][row * kRouteXPitchB + col * 16]) = rx[q];
    }
    if (w_mine) {
      float f[8];
      unpack8_f32(rw, f);
      float4* dst = reinterpret_cast<float4*>(&ws[b][wr_row][wr_col]);
      dst[0] = make_float4(f[0], f[1], f[2], f[3]);
      dst[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
    __syncthreads();
    if (ch + 1 < nchunks) fetch(ch + 1, rx, rw);
    const float* wb = &ws[b][warp * kRouteEpw][0];
    // w_r values of the next 4-wide h step are loaded before the FMAs of the
    // current one, so shared-memory latency overlaps the arithmetic
    float4 wn[kRouteEpw];
#pragma unroll
    for (int i = 0; i < kRouteEpw; ++i) wn[i] = *reinterpret_cast<const float4*>(wb + i * kRouteHc);
    float xv[TPL][8];
#pragma unroll
    for (int s4 = 0; s4 < kRouteHc / 4; ++s4) {
      if ((s4 & 1) == 0) {
#pragma unroll
        for (int u = 0; u < TPL; ++u)
          unpack8_f32(*reinterpret_cast<const uint4*>(&xs[b][(lane + 32 * u) * kRouteXPitchB] +
                                                      (s4 >> 1) * 16),
                      xv[u]);
      }
      float4 wc[kRouteEpw];
#pragma unroll
      for (int i = 0; i < kRouteEpw; ++i) wc[i] = wn[i];
      if (s4 + 1 < kRouteHc / 4) {
#pragma unroll
        for (int i = 0; i < kRouteEpw; ++i)
          wn[i] = *reinterpret_cast<const float4*>(wb + i * kRouteHc + (s4 + 1) * 4);
      }
      const int hh = (s4 & 1) * 4;
#pragma unroll
      for (int i = 0; i < kRouteEpw; ++i) {
#pragma unroll
        for (int u = 0; u < TPL; ++u) {
          acc[u][i] = fmaf(xv[u][hh + 0], wc[i].x, acc[u][i]);
          acc[u][i] = fmaf(xv[u][hh + 1], wc[i].y, acc[u][i]);
          acc[u][i] = fmaf(xv[u][hh + 2], wc[i].z, acc[u][i]);
          acc[u][i] = fmaf(xv[u][hh + 3], wc[i].w, acc[u][i]);
        }
      }
    }
  }
#pragma unroll
  for (int u = 0; u < TPL; ++u) {
    const int t = t0 + lane + 32 * u;
    if (t >= T) continue;
#pragma unroll
    for (int i = 0; i < kRouteEpw; ++i) {
      const int e = e0 + warp * kRouteEpw + i;
      if (e < E) {
        float v = acc[u][i];
        if (bias) v = __fadd_rn(v, __ldg(bias + e));
        z[(size_t)t * E + e] = v;
      }
    }
  }
}

__device__ __forceinline__ bool better(float v1, int e1, float v2, int e2) {
  return v1 > v2 || (v1 == v2 && e1 < e2);
}

// One warp per token: top-k (or the forced set), softmax over all E, gates.
template <int EPL>
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ z,
                                                         int32_t* __restrict__ idx,
                                                         float* __restrict__ gates, int T, int E,
                                                         int k, int forced) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const float* zt = z + (size_t)t * E;
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
    uint32_t taken = 0;
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !((taken >> i) & 1u) && (be == 0x7fffffff || better(v[i], e, bv, be))) {
          bv = v[i];
          be = e;
        }
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (oe != 0x7fffffff && (be == 0x7fffffff || better(ov, oe, bv, be))) {
          bv = ov;
          be = oe;
        }
      }
      if (be != 0x7fffffff && (be & 31) == lane) taken |= 1u << (be >> 5);
      if (lane == j) {
        my_e = be;
        my_p = expf(bv - m) / s;
      }
    }
  }
  float ps = lane < k ? my_p : 0.f;
#pragma unroll
  for (int o = 16; o; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
  if (lane < k) {
    idx[(size_t)t * k + lane] = my_e;
    gates[(size_t)t * k + lane] = my_p / ps;
  }
}

// ------------------------------------------------------------------ backward
// One 256-thread block per group of tokens; each thread owns 16-byte chunks of
// one token row. dz_j = g_j (dg_j - <g, dg>) on the chosen set;
// dx = bf16(dx32 + sum_j dz_j * w_r[i_j]).
template <int KMAX>
__global__ void __launch_bounds__(256, KMAX <= 8 ? 4 : 2) route_bwd_dx_kernel(
    const float* __restrict__ dgates, const float* __restrict__ gates,
    const int32_t* __restrict__ idx, const bf16* __restrict__ w_r, const float* __restrict__ dx32,
    bf16* __restrict__ dx, float* __restrict__ dz, int T, int H, int E, int k, int tpr,
    int* status) {
  // tokens per block = 256 / tpr with tpr >= H/8 >= 8, so at most 32
  __shared__ float s_dz[32][KMAX];
  __shared__ int s_e[32][KMAX];
  const int rpb = blockDim.x / tpr;
  const int tl = threadIdx.x / tpr;
  const int t = blockIdx.x * rpb + tl;
  const int sub = threadIdx.x % tpr;
  // the token's first min(k, tpr) threads work out dz_j and the expert of slot j
  if (t < T && sub < k) {
    float inner = 0.f;
    for (int j = 0; j < k; ++j) inner = fmaf(gates[(size_t)t * k + j], dgates[(size_t)t * k + j], inner);
    const int e = idx[(size_t)t * k + sub];
    s_dz[tl][sub] = gates[(size_t)t * k + sub] * (dgates[(size_t)t * k + sub] - inner);
    s_e[tl][sub] = (unsigned)e < (unsigned)E ? e : -1;
  }
  __syncthreads();
  if (t >= T) return;
  float dzj[KMAX];
  int ej[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    dzj[j] = j < k ? s_dz[tl][j] : 0.f;
    ej[j] = j < k ? s_e[tl][j] : -1;
  }
  const int cpr = H / 8;
  for (int c = sub; c < cpr; c += tpr) {
    const float4* src = reinterpret_cast<const float4*>(dx32 + (size_t)t * H + c * 8);
    const float4 p0 = src[0], p1 = src[1];
    float acc[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
    for (int j0 = 0; j0 < KMAX; j0 += 8) {  // 8 w_r rows in flight at a time
      uint4 wv[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = j0 + u;
        wv[u] = (j < k && ej[j] >= 0)
                    ? __ldg(reinterpret_cast<const uint4*>(w_r + (size_t)ej[j] * H + c * 8))
                    : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = j0 + u;
        if (j < k) {
          const uint32_t w[4] = {wv[u].x, wv[u].y, wv[u].z, wv[u].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            acc[2 * q] = fmaf(dzj[j], bf16_bits_to_f32(w[q] & 0xFFFFu), acc[2 * q]);
            acc[2 * q + 1] = fmaf(dzj[j], bf16_bits_to_f32(w[q] >> 16), acc[2 * q + 1]);
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
    *reinterpret_cast<uint4*>(dx + (size_t)t * H + c * 8) = out;
  }
  if (sub == 0) {
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (j < k) {
        dz[(size_t)t * k + j] = dzj[j];
        if (ej[j] < 0) atomicAdd(status + ST_BAD_INDEX, 1);
      }
    }
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

// Pass A: partial[chunk][h] = sum over the chunk's rows s (ascending) of
// dz[row_src[s]] * x[row_src[s] div k][h]. The chunk's sources and weights are
// staged in shared memory first, so each thread then has 8 independent x-row
// loads in flight instead of a chain of dependent loads per row.
__global__ void __launch_bounds__(256) route_bwd_dwr_partial_kernel(
    const int32_t* __restrict__ off, const int32_t* __restrict__ row_src,
    const float* __restrict__ dz, const bf16* __restrict__ x, float* __restrict__ part, int T,
    int H, int E, int k, int* status) {
  extern __shared__ int s_prefix[];
  __shared__ int s_tok[kRouteBwdRowsPerChunk];
  __shared__ float s_w[kRouteBwdRowsPerChunk];
  int e, r0, r1;
  if (!find_chunk(off, E, blockIdx.x, &e, &r0, &r1, s_prefix)) return;
  const long long N = (long long)T * k;
  const int n = r1 - r0;
  if ((int)threadIdx.x < n) {
    const int src = row_src[r0 + threadIdx.x];
    const bool ok = src >= 0 && src < N;
    s_tok[threadIdx.x] = ok ? src / k : -1;
    s_w[threadIdx.x] = ok ? dz[src] : 0.f;
  }
  __syncthreads();
  const int c = blockIdx.y * blockDim.x + threadIdx.x;  // 16-byte chunk of the row
  if (c * 8 >= H) return;
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

// Pass B: dW_r[e][h] = sum of expert e's chunk partials in chunk order (0 if none).
__global__ void __launch_bounds__(256) route_bwd_dwr_reduce_kernel(
    const int32_t* __restrict__ off, const float* __restrict__ part, float* __restrict__ dw_r,
    int H, int E) {
  __shared__ int s_first, s_n;
  const int e = blockIdx.x;
  if (threadIdx.x < 32) {
    // chunks of experts 0..e-1, summed by one warp
    int sum = 0;
    for (int i = threadIdx.x; i < e; i += 32)
      sum += (off[i + 1] - off[i] + kRouteBwdRowsPerChunk - 1) / kRouteBwdRowsPerChunk;
#pragma unroll
    for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (threadIdx.x == 0) {
      s_first = sum;
      s_n = (off[e + 1] - off[e] + kRouteBwdRowsPerChunk - 1) / kRouteBwdRowsPerChunk;
    }
  }
  __syncthreads();
  const int c = blockIdx.y * blockDim.x + threadIdx.x;
  if (c * 4 >= H) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i = 0; i < s_n; ++i) {
    const float4 p = *reinterpret_cast<const float4*>(part + (size_t)(s_first + i) * H + c * 4);
    acc.x += p.x;
    acc.y += p.y;
    acc.z += p.z;
    acc.w += p.w;
  }
  *reinterpret_cast<float4*>(dw_r + (size_t)e * H + c * 4) = acc;
}

}  // namespace

moe_status_t launch_route(const moe_layer_desc_t& d, const bf16* x, const bf16* w_r,
                          const float* bias, float* logits, int32_t* idx, float* gates,
                          int* status, cudaStream_t st) {
  (void)status;
  if (d.T == 0) return MOE_OK;
  // 4 warps x 4 experts per CTA, ROUTE_TPL tokens per lane: 2 x 4 or 4 x 4
  // accumulators per thread keep the FMA : shared-wavefront ratio at or above 1
  // while giving the SMs enough warps to hide shared-memory latency.
  constexpr int tpl = MOE_ROUTE_TPL;
  const int nw = d.E > 8 ? 4 : d.E > 4 ? 2 : 1;
  const int eb = nw * 4;
  dim3 grid(ceil_div(d.T, 32 * tpl), ceil_div(d.E, eb));
  {
    LaunchScope _ls(K_ROUTE_LOGITS, st);
    if (nw == 4)
      route_logits_kernel<4, 4, tpl><<<grid, 128, 0, st>>>(x, w_r, bias, logits, d.T, d.H, d.E);
    else if (nw == 2)
      route_logits_kernel<2, 4, tpl><<<grid, 64, 0, st>>>(x, w_r, bias, logits, d.T, d.H, d.E);
    else
      route_logits_kernel<1, 4, tpl><<<grid, 32, 0, st>>>(x, w_r, bias, logits, d.T, d.H, d.E);
  }
  moe_status_t s = check_launch("route_logits_kernel");
  if (s != MOE_OK) return s;
  const int tpb = 256, warps = tpb / 32;
  dim3 g2(ceil_div(d.T, warps));
  const int forced = d.mode == MOE_ROUTE_FORCED_BALANCED;
  if (d.E <= 32)
    {
      LaunchScope _ls(K_ROUTE_TOPK, st);
      route_topk_kernel<1><<<g2, tpb, 0, st>>>(logits, idx, gates, d.T, d.E, d.k, forced);
    }
  else if (d.E <= 64)
    {
      LaunchScope _ls(K_ROUTE_TOPK, st);
      route_topk_kernel<2><<<g2, tpb, 0, st>>>(logits, idx, gates, d.T, d.E, d.k, forced);
    }
  else if (d.E <= 128)
    {
      LaunchScope _ls(K_ROUTE_TOPK, st);
      route_topk_kernel<4><<<g2, tpb, 0, st>>>(logits, idx, gates, d.T, d.E, d.k, forced);
    }
  else
    {
      LaunchScope _ls(K_ROUTE_TOPK, st);
      route_topk_kernel<8><<<g2, tpb, 0, st>>>(logits, idx, gates, d.T, d.E, d.k, forced);
    }
  return check_launch("route_topk_kernel");
}

moe_status_t launch_route_bwd(const moe_layer_desc_t& d, const float* dgates, const float* gates,
                              const int32_t* idx, const bf16* x, const bf16* w_r,
                              const int32_t* row_src, const int32_t* off, const float* dx32,
                              bf16* dx, float* dw_r, float* dz, float* dwr_part, int* status,
                              cudaStream_t st) {
  const int cpr = d.H / 8;
  int tpr = 1;
  while ((tpr < cpr || tpr < d.k) && tpr < 256) tpr <<= 1;  // >= k threads per token
  const int rpb = 256 / tpr;
  if (d.T > 0) {
    {
      LaunchScope _ls(K_ROUTE_BWD_DX, st);
      const dim3 g(ceil_div(d.T, rpb));
      if (d.k <= 4)
        route_bwd_dx_kernel<4><<<g, 256, 0, st>>>(dgates, gates, idx, w_r, dx32, dx, dz, d.T, d.H,
                                                  d.E, d.k, tpr, status);
      else if (d.k <= 8)
        route_bwd_dx_kernel<8><<<g, 256, 0, st>>>(dgates, gates, idx, w_r, dx32, dx, dz, d.T, d.H,
                                                  d.E, d.k, tpr, status);
      else if (d.k <= 16)
        route_bwd_dx_kernel<16><<<g, 256, 0, st>>>(dgates, gates, idx, w_r, dx32, dx, dz, d.T, d.H,
                                                   d.E, d.k, tpr, status);
      else
        route_bwd_dx_kernel<32><<<g, 256, 0, st>>>(dgates, gates, idx, w_r, dx32, dx, dz, d.T, d.H,
                                                   d.E, d.k, tpr, status);
    }
    moe_status_t s = check_launch("route_bwd_dx_kernel");
    if (s != MOE_OK) return s;
  }
  const long long N = (long long)d.T * d.k;
  const int max_chunks = (int)((N + kRouteBwdRowsPerChunk - 1) / kRouteBwdRowsPerChunk) + d.E;
  if (N > 0) {
    dim3 ga(max_chunks, ceil_div(cpr, 256));
    {
      LaunchScope _ls(K_ROUTE_BWD_DWR_PARTIAL, st);
      route_bwd_dwr_partial_kernel<<<ga, 256, (d.E + 1) * sizeof(int), st>>>(
          off, row_src, dz, x, dwr_part, d.T, d.H, d.E, d.k, status);
    }
    moe_status_t s = check_launch("route_bwd_dwr_partial_kernel");
    if (s != MOE_OK) return s;
  }
  dim3 gb(d.E, ceil_div(d.H / 4, 256));
  {
    LaunchScope _ls(K_ROUTE_BWD_DWR_REDUCE, st);
    route_bwd_dwr_reduce_kernel<<<gb, 256, 0, st>>>(off, dwr_part, dw_r, d.H, d.E);
  }
  return check_launch("route_bwd_dwr_reduce_kernel");
}

}  // namespace moe
