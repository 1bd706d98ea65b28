// Permute (dispatch: write the EP send buffer), combine (receive + unpermute
// with the gate-weighted sum) and their backward passes. These are the
// "dispatch" and "combine" phases of the EP-overlap note ("1. MoE EP Overlap",
// section "how the 8 fwd/bwd operations are split out") with the all-to-all
// itself replaced by writing the rank-major, expert-contiguous buffer.
//
// All four are HBM-bound row gathers. A thread moves one 16-byte chunk
// (8 bf16) per row at a time; a token's k source rows are loaded before any is
// used so k independent 16-byte loads are in flight per thread. The token
// input x (T*H*2 bytes, e.g. 16.8 MB) stays resident in the 129 MB L2, so the
// k-fold re-reads of permute come from L2 and DRAM sees roughly one read of x
// plus one write of x_perm.
#include "moe_internal.cuh"

namespace moe {

namespace {

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    f[2 * q] = __uint_as_float(w[q] << 16);
    f[2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint4 out;
  uint32_t* o = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    __nv_bfloat162 b2 = __floats2bfloat162_rn(f[2 * q], f[2 * q + 1]);
    o[q] = *reinterpret_cast<uint32_t*>(&b2);
  }
  return out;
}

// x_perm[s] = x[row_src[s] / k]; one warp per destination row, grid-stride.
__global__ void __launch_bounds__(256) permute_kernel(const bf16* __restrict__ x,
                                                      const int32_t* __restrict__ row_src,
                                                      bf16* __restrict__ x_perm, int T, int H,
                                                      int k, long long N) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  const int cpr = H / 8;
  for (long long s = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); s < N;
       s += warps) {
    const int src = row_src[s];
    const int t = src / k;
    uint4* dst = reinterpret_cast<uint4*>(x_perm + s * H);
    if (src < 0 || t >= T) {
      for (int c = lane; c < cpr; c += 32) dst[c] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const uint4* srcp = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    int c = lane;
    for (; c + 96 < cpr; c += 128) {
      const uint4 v0 = __ldg(srcp + c), v1 = __ldg(srcp + c + 32), v2 = __ldg(srcp + c + 64),
                  v3 = __ldg(srcp + c + 96);
      __stcs(dst + c, v0);
      __stcs(dst + c + 32, v1);
      __stcs(dst + c + 64, v2);
      __stcs(dst + c + 96, v3);
    }
    for (; c < cpr; c += 32) __stcs(dst + c, __ldg(srcp + c));
  }
}

// Threads of one token row: tpr threads (a power of two >= H/8, at most 256),
// 256/tpr tokens per block; thread `sub` handles chunks sub, sub+tpr, ...
struct RowMap {
  int t, sub, tpr;
};
__device__ __forceinline__ RowMap row_map(int tpr) {
  RowMap m;
  m.tpr = tpr;
  m.t = blockIdx.x * (blockDim.x / tpr) + threadIdx.x / tpr;
  m.sub = threadIdx.x % tpr;
  return m;
}

constexpr int kMaxKBatch = 8;

// y[t] = bf16(sum_j g[t,j] * o[slot[t,j]]), fp32 in ascending j.
// A block takes groups of 256/tpr tokens in turn (grid-stride). The routing
// state of a group (slots and gates) is staged in shared memory, and the next
// group's is loaded while the current group's rows are in flight, so a token
// costs one round trip to memory instead of a routing-state load followed by
// the row loads that depend on it.
template <int KMAX>
__global__ void __launch_bounds__(256) combine_kernel(const bf16* __restrict__ o,
                                                      const int32_t* __restrict__ slot,
                                                      const float* __restrict__ gates,
                                                      bf16* __restrict__ y, int T, int H, int k,
                                                      long long N, int tpr) {
  pdl_wait();
  constexpr int KB = KMAX < kMaxKBatch ? KMAX : kMaxKBatch;
  __shared__ int s_slot[2][32 * KMAX];  // tpr >= 8 (H >= 64): at most 32 tokens a group
  __shared__ float s_g[2][32 * KMAX];
  const int tpb = blockDim.x / tpr;  // tokens per group
  const int lt = threadIdx.x / tpr, sub = threadIdx.x % tpr;
  const int cpr = H / 8;
  const int ngroups = (T + tpb - 1) / tpb;
  const int nent = tpb * k;
  auto stage = [&](int buf, int grp) {
    const long long e0 = (long long)grp * tpb * k;
    for (int i = threadIdx.x; i < nent; i += blockDim.x) {
      const long long e = e0 + i;
      int sv = -1;
      float gv = 0.f;
      if (grp < ngroups && e < N) {
        sv = slot[e];
        gv = gates[e];
      }
      s_slot[buf][i] = sv >= 0 && sv < N ? sv : -1;
      s_g[buf][i] = gv;
    }
  };
  int buf = 0;
  stage(0, blockIdx.x);
  __syncthreads();
  for (int grp = blockIdx.x; grp < ngroups; grp += gridDim.x, buf ^= 1) {
    const int t = grp * tpb + lt;
    const int* sl = s_slot[buf] + lt * k;
    const float* gl = s_g[buf] + lt * k;
    bool next_staged = false;
    for (int c = sub; c < cpr; c += tpr) {
      float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
      for (int j0 = 0; j0 < KMAX; j0 += KB) {
        uint4 v[KB];
#pragma unroll
        for (int u = 0; u < KB; ++u) {
          const int j = j0 + u;
          const int sv = (t < T && j < k) ? sl[j] : -1;
          v[u] = sv >= 0 ? __ldcs(reinterpret_cast<const uint4*>(o + (size_t)sv * H) + c)
                         : make_uint4(0, 0, 0, 0);
        }
        if (!next_staged) {  // the next group's routing state, beside the row loads
          stage(buf ^ 1, grp + gridDim.x);
          next_staged = true;
        }
#pragma unroll
        for (int u = 0; u < KB; ++u) {
          const int j = j0 + u;
          if (j < k) {
            float f[8];
            unpack8(v[u], f);
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] = fmaf(gl[j], f[q], acc[q]);
          }
        }
      }
      if (t < T) reinterpret_cast<uint4*>(y + (size_t)t * H)[c] = pack8(acc);
    }
    if (!next_staged) stage(buf ^ 1, grp + gridDim.x);
    __syncthreads();
  }
}

// d_o[slot[t,j]] = bf16(g[t,j] * dy[t]); dgates[t,j] = <dy[t], o[slot[t,j]]>.
// The dot product is reduced over the token's threads in a fixed tree order.
// Token groups are taken in turn with their routing state staged in shared
// memory, the next group's loaded beside the current rows (as in combine).
template <int KMAX>
__global__ void __launch_bounds__(256, KMAX <= 8 ? 3 : 1) combine_bwd_kernel(
    const bf16* __restrict__ dy, const bf16* __restrict__ o, const int32_t* __restrict__ slot,
    const float* __restrict__ gates, bf16* __restrict__ d_o, float* __restrict__ dgates, int T,
    int H, int k, long long N, int tpr, int* __restrict__ zero, int nzero) {
  pdl_wait();
  // the next launch's counters (see launch_combine_bwd)
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < nzero; i += blockDim.x) zero[i] = 0;
  __shared__ float s_part[8][KMAX];
  __shared__ int s_slot[2][32 * KMAX];  // tpr >= 8 (H >= 64): at most 32 tokens a group
  __shared__ float s_g[2][32 * KMAX];
  const int tpb = blockDim.x / tpr;
  const int lt = threadIdx.x / tpr, sub = threadIdx.x % tpr;
  const int cpr = H / 8;
  const int ngroups = (T + tpb - 1) / tpb;
  const int nent = tpb * k;
  auto stage = [&](int buf, int grp) {
    const long long e0 = (long long)grp * tpb * k;
    for (int i = threadIdx.x; i < nent; i += blockDim.x) {
      const long long e = e0 + i;
      int sv = -1;
      float gv = 0.f;
      if (grp < ngroups && e < N) {
        sv = slot[e];
        gv = gates[e];
      }
      s_slot[buf][i] = sv >= 0 && sv < N ? sv : -1;
      s_g[buf][i] = gv;
    }
  };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int buf = 0;
  stage(0, blockIdx.x);
  __syncthreads();
  for (int grp = blockIdx.x; grp < ngroups; grp += gridDim.x, buf ^= 1) {
    const int t = grp * tpb + lt;
    const bool active = t < T;
    const int* sl = s_slot[buf] + lt * k;
    const float* gl = s_g[buf] + lt * k;
    float dot[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) dot[j] = 0.f;
    bool next_staged = false;
    if (active) {
      for (int c = sub; c < cpr; c += tpr) {
        float fy[8];
        unpack8(__ldg(reinterpret_cast<const uint4*>(dy + (size_t)t * H) + c), fy);
#pragma unroll
        for (int j0 = 0; j0 < KMAX; j0 += kMaxKBatch) {  // 8 rows of o in flight
          uint4 ov[kMaxKBatch];
#pragma unroll
          for (int u = 0; u < kMaxKBatch; ++u) {
            const int j = j0 + u;
            const int sv = (j < KMAX && j < k) ? sl[j] : -1;
            ov[u] = sv >= 0 ? __ldcs(reinterpret_cast<const uint4*>(o + (size_t)sv * H) + c)
                            : make_uint4(0, 0, 0, 0);
          }
          if (!next_staged) {  // the next group's routing state, beside the row loads
            stage(buf ^ 1, grp + gridDim.x);
            next_staged = true;
          }
#pragma unroll
          for (int u = 0; u < kMaxKBatch; ++u) {
            const int j = j0 + u;
            if (j < KMAX && j < k) {
              const int sv = sl[j];
              if (sv >= 0) {
                float fo[8], prod[8];
                unpack8(ov[u], fo);
                float d = 0.f;
                const float gj = gl[j];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                  d = fmaf(fy[q], fo[q], d);
                  prod[q] = gj * fy[q];
                }
                dot[j] += d;
                __stcs(reinterpret_cast<uint4*>(d_o + (size_t)sv * H) + c, pack8(prod));
              }
            }
          }
        }
      }
    }
    if (!next_staged) stage(buf ^ 1, grp + gridDim.x);
    // reduce dot[] over the tpr threads of the token
    const int width = tpr < 32 ? tpr : 32;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
#pragma unroll
      for (int o2 = 16; o2; o2 >>= 1)
        if (o2 < width) dot[j] += __shfl_xor_sync(0xffffffffu, dot[j], o2, width);
    }
    if (tpr <= 32) {
      if (active && sub == 0) {
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
          if (j < k) dgates[(size_t)t * k + j] = dot[j];
      }
    } else {
      // tpr > 32: the token's tpr/32 warps combine their sums in warp order
      if (lane == 0) {
#pragma unroll
        for (int j = 0; j < KMAX; ++j) s_part[warp][j] = dot[j];
      }
      __syncthreads();
      const int wbase = lt * (tpr / 32);
      if (active && sub < k) {
        float sum = 0.f;
        for (int w = 0; w < tpr / 32; ++w) sum += s_part[wbase + w][sub];
        dgates[(size_t)t * k + sub] = sum;
      }
    }
    __syncthreads();
  }
}

// dx32[t] = sum_j dx_perm[slot[t,j]] in fp32, ascending j.
__global__ void __launch_bounds__(256) permute_bwd_kernel(const bf16* __restrict__ dx_perm,
                                                          const int32_t* __restrict__ slot,
                                                          float* __restrict__ dx32, int T, int H,
                                                          int k, long long N, int tpr) {
  pdl_wait();
  const RowMap m = row_map(tpr);
  if (m.t >= T) return;
  const int cpr = H / 8;
  for (int c = m.sub; c < cpr; c += tpr) {
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int j0 = 0; j0 < k; j0 += kMaxKBatch) {
      const int nj = min(kMaxKBatch, k - j0);
      uint4 v[kMaxKBatch];
#pragma unroll
      for (int u = 0; u < kMaxKBatch; ++u) {
        v[u] = make_uint4(0, 0, 0, 0);
        if (u < nj) {
          const int s = slot[(size_t)m.t * k + j0 + u];
          if (s >= 0 && s < N) v[u] = __ldcs(reinterpret_cast<const uint4*>(dx_perm + (size_t)s * H) + c);
        }
      }
#pragma unroll
      for (int u = 0; u < kMaxKBatch; ++u) {
        if (u < nj) {
          float f[8];
          unpack8(v[u], f);
#pragma unroll
          for (int q = 0; q < 8; ++q) acc[q] += f[q];
        }
      }
    }
    float4* dst = reinterpret_cast<float4*>(dx32 + (size_t)m.t * H + c * 8);
    dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

int threads_per_row(int H) {
  const int cpr = H / 8;
  int tpr = 1;
  while (tpr < cpr && tpr < 256) tpr <<= 1;
  return tpr;
}

}  // namespace

moe_status_t launch_permute(const moe_layer_desc_t& d, const bf16* x, const int32_t* row_src,
                            bf16* x_perm, cudaStream_t st) {
  const long long N = (long long)d.T * d.k;
  if (N == 0) return MOE_OK;
  const int warps_per_block = 8;
  long long blocks = (N + warps_per_block - 1) / warps_per_block;
  const long long cap = (long long)device_sm_count() * 16;
  if (blocks > cap) blocks = cap;
  {
    LaunchScope _ls(K_PERMUTE, st);
    launch_k(permute_kernel, (int)blocks, 256, 0, st, x, row_src, x_perm, d.T, d.H, d.k, N);
  }
  return check_launch("permute_kernel");
}

// One wave of resident blocks (looked up once per instantiation), each taking
// token groups in turn.
template <int KMAX>
cudaError_t launch_combine_t(const moe_layer_desc_t& d, int groups, const bf16* o,
                             const int32_t* slot, const float* gates, bf16* y, long long N,
                             int tpr, cudaStream_t st) {
  static int per_sm = 0;
  static const cudaError_t occ =
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, combine_kernel<KMAX>, 256, 0);
  if (occ != cudaSuccess) return occ;
  const int grid = std::min(groups, std::max(per_sm, 1) * device_sm_count());
  return launch_k(combine_kernel<KMAX>, grid, 256, 0, st, o, slot, gates, y, d.T, d.H, d.k, N,
                  tpr);
}

moe_status_t launch_combine(const moe_layer_desc_t& d, const bf16* o, const int32_t* slot,
                            const float* gates, bf16* y, cudaStream_t st) {
  if (d.T == 0) return MOE_OK;
  const int tpr = threads_per_row(d.H);
  const long long N = (long long)d.T * d.k;
  const int groups = ceil_div(d.T, 256 / tpr);
  cudaError_t e;
  {
    LaunchScope _ls(K_COMBINE, st);
    if (d.k <= 2) e = launch_combine_t<2>(d, groups, o, slot, gates, y, N, tpr, st);
    else if (d.k <= 4) e = launch_combine_t<4>(d, groups, o, slot, gates, y, N, tpr, st);
    else if (d.k <= 8) e = launch_combine_t<8>(d, groups, o, slot, gates, y, N, tpr, st);
    else if (d.k <= 16) e = launch_combine_t<16>(d, groups, o, slot, gates, y, N, tpr, st);
    else e = launch_combine_t<32>(d, groups, o, slot, gates, y, N, tpr, st);
  }
  if (e != cudaSuccess) {
    set_error("combine_kernel launch: %s", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  return check_launch("combine_kernel");
}

moe_status_t launch_combine_bwd(const moe_layer_desc_t& d, const bf16* dy, const bf16* o,
                                const int32_t* slot, const float* gates, bf16* d_o,
                                float* dgates, cudaStream_t st, int* zero, int nzero) {
  if (d.T == 0) return MOE_OK;
  const int tpr = threads_per_row(d.H);
  const long long N = (long long)d.T * d.k;
  // one wave of resident blocks (3 per SM for k <= 8, else 1), each taking
  // token groups in turn
  const int groups = ceil_div(d.T, 256 / tpr);
  const dim3 grid(std::min(groups, (d.k <= 8 ? 3 : 1) * device_sm_count()));
  if (d.k <= 2)
    {
      LaunchScope _ls(K_COMBINE_BWD, st);
      launch_k(combine_bwd_kernel<2>, grid, 256, 0, st, dy, o, slot, gates, d_o, dgates, d.T, d.H,
               d.k, N, tpr, zero, nzero);
    }
  else if (d.k <= 4)
    {
      LaunchScope _ls(K_COMBINE_BWD, st);
      launch_k(combine_bwd_kernel<4>, grid, 256, 0, st, dy, o, slot, gates, d_o, dgates, d.T, d.H,
               d.k, N, tpr, zero, nzero);
    }
  else if (d.k <= 8)
    {
      LaunchScope _ls(K_COMBINE_BWD, st);
      launch_k(combine_bwd_kernel<8>, grid, 256, 0, st, dy, o, slot, gates, d_o, dgates, d.T, d.H,
               d.k, N, tpr, zero, nzero);
    }
  else if (d.k <= 16)
    {
      LaunchScope _ls(K_COMBINE_BWD, st);
      launch_k(combine_bwd_kernel<16>, grid, 256, 0, st, dy, o, slot, gates, d_o, dgates, d.T, d.H,
               d.k, N, tpr, zero, nzero);
    }
  else
    {
      LaunchScope _ls(K_COMBINE_BWD, st);
      launch_k(combine_bwd_kernel<32>, grid, 256, 0, st, dy, o, slot, gates, d_o, dgates, d.T, d.H,
               d.k, N, tpr, zero, nzero);
    }
  return check_launch("combine_bwd_kernel");
}

moe_status_t launch_permute_bwd(const moe_layer_desc_t& d, const bf16* dx_perm,
                                const int32_t* slot, float* dx32, cudaStream_t st) {
  if (d.T == 0) return MOE_OK;
  const int tpr = threads_per_row(d.H);
  {
    LaunchScope _ls(K_PERMUTE_BWD, st);
    launch_k(permute_bwd_kernel, ceil_div(d.T, 256 / tpr), 256, 0, st, dx_perm, slot, dx32, d.T,
             d.H, d.k, (long long)d.T * d.k, tpr);
  }
  return check_launch("permute_bwd_kernel");
}

}  // namespace moe
