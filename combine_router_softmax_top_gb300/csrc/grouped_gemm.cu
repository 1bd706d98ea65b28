// Grouped expert GEMMs of the "mlp" phase on the sm_100-family tensor cores
// (tcgen05 MMA with TMEM accumulators, operands staged by TMA), for the forward,
// the activation gradient (dgrad) and the deferrable weight gradient (wgrad);
// the dgrad/wgrad split follows the EP-overlap note ("1. MoE EP Overlap",
// section "MoE 1F1B overlap": the mlp backward computes the activation gradient
// first so dispatch-backward can start, and the weight gradient later).
//
// One persistent kernel per call, one CTA per SM, warp-specialised:
//   warp 0      TMA producer (4-stage ring of 48 KB A|B stages)
//   warp 1      TMEM allocator + single-thread MMA issuer
//   warps 2..5  epilogue: TMEM -> registers -> fused math -> global stores
// Tiles are 128 x 256 (one tcgen05.mma M=128, N=256, K=16 per step, 4 steps
// per 64-wide K stage). The 512 TMEM columns hold two accumulators, so the
// epilogue of one tile overlaps the MMAs of the next.
//
// Ragged groups. Expert e owns rows off[e]..off[e+1]-1 of the permuted
// activations. Forward and dgrad tiles are (expert, 128-row block, N block):
// a tile's rows past the expert's end are computed on whatever TMA loaded
// (the next expert's rows, or zero fill past the tensor) and masked at the
// store. Wgrad tiles reduce over the expert's rows (K-ragged): in the last K
// stage of an expert the producer zeroes the A rows past the expert's end in
// shared memory before releasing the stage, so other experts' rows add 0.
// The tile list is derived on the device from off[], so no host sync is needed.
//
// Operand layouts (all 128-byte swizzled, as TMA writes them):
//   K-major  (rows x 64 K): rows at 128 B, 8-row atoms of 1024 B (SBO = 1024).
//            Advancing K by 16 elements adds 32 B to the start address.
//   MN-major (64 K rows x 64 MN per atom, 8 KB): K rows at 128 B, 8-row groups
//            at SBO = 1024, MN atoms at LBO = 8192. Advancing K by 16 adds 2 KB.
#include <mutex>

#include "moe_internal.cuh"
#include "sm100_ptx.cuh"

namespace moe {

namespace {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int kStages = 4;
constexpr int kABytes = BM * BK * 2;   // 16 KB
constexpr int kBBytes = BN * BK * 2;   // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kThreads = 192;
constexpr int kTmemCols = 512;
constexpr int kMaxE = 256;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s without progress -> give up
constexpr size_t kDynSmem = (size_t)kStages * kStageBytes + 1024;

struct KParams {
  int E, H, F;
  long long N;
  const int32_t* off;
  bf16* out0;
  bf16* out1;
  const bf16* aux;
  int* status;
};

template <int MODE>
struct Mode {
  static constexpr bool kRagK = MODE == GEMM_WGRAD_W1 || MODE == GEMM_WGRAD_W2;
  static constexpr int kAMn = kRagK ? 1 : 0;
  static constexpr int kBMn = (MODE == GEMM_FC2_DGRAD || MODE == GEMM_FC1_DGRAD || kRagK) ? 1 : 0;
  // reduction depth for the row-ragged modes
  __device__ static int kdim(const KParams& p) {
    return MODE == GEMM_FC1_FWD ? p.H : MODE == GEMM_FC2_FWD ? p.F
         : MODE == GEMM_FC2_DGRAD ? p.H : 2 * p.F;
  }
  // number of N blocks (FC1 forward: 128 gate + 128 up columns per block)
  __device__ static int ntiles(const KParams& p) {
    switch (MODE) {
      case GEMM_FC1_FWD: return (p.F + 127) / 128;
      case GEMM_FC2_FWD: return (p.H + BN - 1) / BN;
      case GEMM_FC2_DGRAD: return (p.F + BN - 1) / BN;
      case GEMM_FC1_DGRAD: return (p.H + BN - 1) / BN;
      case GEMM_WGRAD_W1: return (p.H + BN - 1) / BN;
      default: return (p.F + BN - 1) / BN;
    }
  }
  // wgrad: rows of the weight gradient (M)
  __device__ static int wg_mdim(const KParams& p) { return MODE == GEMM_WGRAD_W1 ? 2 * p.F : p.H; }
  __device__ static int wg_ndim(const KParams& p) { return MODE == GEMM_WGRAD_W1 ? p.H : p.F; }
};

struct Tile {
  int e, m0, n0;
  int rows;  // row-ragged: valid rows in this tile; K-ragged: rows of the expert
  int nk;    // K stages
  int row0;  // off[e]
};

struct SmemCtl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t tail;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int tstart[kMaxE + 1];
  int off[kMaxE + 1];
};

template <int MODE>
__device__ __forceinline__ Tile tile_at(const KParams& p, const SmemCtl& c, int tile, int& cursor) {
  while (c.tstart[cursor + 1] <= tile) ++cursor;
  Tile t;
  t.e = cursor;
  t.row0 = c.off[t.e];
  const int cnt = c.off[t.e + 1] - t.row0;
  const int local = tile - c.tstart[t.e];
  if (Mode<MODE>::kRagK) {
    const int mt = (Mode<MODE>::wg_mdim(p) + BM - 1) / BM;
    t.m0 = (local % mt) * BM;
    t.n0 = (local / mt) * BN;
    t.rows = cnt;
    t.nk = (cnt + BK - 1) / BK;
  } else {
    const int mt = (cnt + BM - 1) / BM;
    t.m0 = (local % mt) * BM;
    t.n0 = (local / mt) * (MODE == GEMM_FC1_FWD ? 128 : BN);
    t.rows = min(BM, cnt - t.m0);
    t.nk = Mode<MODE>::kdim(p) / BK;
  }
  return t;
}

__device__ __forceinline__ void flag_timeout(SmemCtl& c, int* status, int where) {
  c.abort = 1;
  atomicExch(status + ST_TIMEOUT, where);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&b);
}

__device__ __forceinline__ void store32(bf16* dst, const float* v) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    d[q] = make_uint4(pack_bf16x2(v[8 * q + 0], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                      pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
}

__device__ __forceinline__ void load32(const bf16* src, float* v) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 u = s[q];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[8 * q + 2 * i] = __uint_as_float(w[i] << 16);
      v[8 * q + 2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
}

__device__ __forceinline__ float round_bf16(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, const KParams p) {
  using M = Mode<MODE>;
  extern __shared__ uint8_t dyn_smem[];
  __shared__ SmemCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) &
                                             ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E;

  // ---- per-CTA setup: offsets, tile prefix, barriers, TMEM
  for (int e = threadIdx.x; e <= E; e += blockDim.x) ctl.off[e] = p.off[e];
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&ctl.full[s], 1);
      ptx::mbar_init(&ctl.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&ctl.tmem_full[b], 1);
      ptx::mbar_init(&ctl.tmem_empty[b], 128);
    }
    ptx::mbar_init(&ctl.tail, 1);
    ptx::mbar_init(&ctl.drain, 1);
    ctl.abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&ctl.tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  __syncthreads();
  if (warp == 0) {
    // tiles per expert -> exclusive prefix
    int carry = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      int n = 0;
      if (e < E) {
        const int cnt = ctl.off[e + 1] - ctl.off[e];
        if (M::kRagK) n = ((M::wg_mdim(p) + BM - 1) / BM) * M::ntiles(p);
        else n = ((cnt + BM - 1) / BM) * M::ntiles(p);
        if (cnt < 0) n = 0;
      }
      int incl = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (e < E) ctl.tstart[e] = carry + incl - n;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) ctl.tstart[E] = carry;
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const int total = ctl.tstart[E];
  const uint32_t tmem_base = ctl.tmem_base;

  if (warp == 0) {
    // ================================================================ producer
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tmA);
      ptx::tma_prefetch_desc(&tmB);
    }
    int stage = 0, cursor = 0;
    uint32_t phase = 0, tail_phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      const Tile t = tile_at<MODE>(p, ctl, tile, cursor);
      for (int kt = 0; kt < t.nk; ++kt) {
        if (!ptx::mbar_wait(&ctl.empty[stage], phase ^ 1, &ctl.abort, kWaitLimitNs)) {
          if (lane == 0) flag_timeout(ctl, p.status, 1);
          ok = false;
          break;
        }
        uint8_t* sA = smem + stage * kStageBytes;
        uint8_t* sB = sA + kABytes;
        const int k0 = kt * BK;
        const bool tail = M::kRagK && (t.rows - k0 < BK);
        uint64_t* bar = tail ? &ctl.tail : &ctl.full[stage];
        if (lane == 0) {
          ptx::mbar_arrive_expect_tx(bar, kStageBytes);
          if (M::kRagK) {
            const int r = t.row0 + k0;
            ptx::tma_load_2d(sA, &tmA, bar, t.m0, r);
            ptx::tma_load_2d(sA + 8192, &tmA, bar, t.m0 + 64, r);
#pragma unroll
            for (int i = 0; i < 4; ++i) ptx::tma_load_2d(sB + 8192 * i, &tmB, bar, t.n0 + 64 * i, r);
          } else {
            ptx::tma_load_2d(sA, &tmA, bar, k0, t.row0 + t.m0);
            if (MODE == GEMM_FC1_FWD) {
              const int base = t.e * 2 * p.F;
              ptx::tma_load_2d(sB, &tmB, bar, k0, base + t.n0);
              ptx::tma_load_2d(sB + 16384, &tmB, bar, k0, base + p.F + t.n0);
            } else if (MODE == GEMM_FC2_FWD) {
              ptx::tma_load_2d(sB, &tmB, bar, k0, t.e * p.H + t.n0);
            } else {
              const int base = MODE == GEMM_FC2_DGRAD ? t.e * p.H : t.e * 2 * p.F;
#pragma unroll
              for (int i = 0; i < 4; ++i)
                ptx::tma_load_2d(sB + 8192 * i, &tmB, bar, t.n0 + 64 * i, base + k0);
            }
          }
        }
        if (tail) {
          // last K stage of a wgrad tile: zero the A rows past the expert's end
          if (!ptx::mbar_wait(&ctl.tail, tail_phase, &ctl.abort, kWaitLimitNs)) {
            if (lane == 0) flag_timeout(ctl, p.status, 2);
            ok = false;
            break;
          }
          tail_phase ^= 1;
          const int valid = t.rows - k0;  // 1..63
          const int nzero = (BK - valid) * 8;  // 16-byte chunks per atom
          for (int i = lane; i < 2 * nzero; i += 32) {
            const int atom = i / nzero, j = i % nzero;
            uint4* dst = reinterpret_cast<uint4*>(sA + atom * 8192 + valid * 128) + j;
            *dst = make_uint4(0, 0, 0, 0);
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&ctl.full[stage]);
        }
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(BM, BN, M::kAMn, M::kBMn);
      const uint32_t a_lbo = M::kAMn ? 8192 : 16, b_lbo = M::kBMn ? 8192 : 16;
      const uint32_t a_adv = M::kAMn ? (2048 >> 4) : (32 >> 4);
      const uint32_t b_adv = M::kBMn ? (2048 >> 4) : (32 >> 4);
      int stage = 0, cursor = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const Tile t = tile_at<MODE>(p, ctl, tile, cursor);
        if (t.nk == 0) continue;
        if (!ptx::mbar_wait(&ctl.tmem_empty[acc], acc_phase ^ 1, &ctl.abort, kWaitLimitNs)) {
          flag_timeout(ctl, p.status, 3);
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kt = 0; kt < t.nk; ++kt) {
          if (!ptx::mbar_wait(&ctl.full[stage], phase, &ctl.abort, kWaitLimitNs)) {
            flag_timeout(ctl, p.status, 4);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a_addr = ptx::smem_u32(smem + stage * kStageBytes);
          const uint32_t b_addr = a_addr + kABytes;
          const uint64_t adesc = ptx::sdesc_sw128(a_addr, a_lbo, 1024);
          const uint64_t bdesc = ptx::sdesc_sw128(b_addr, b_lbo, 1024);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            ptx::umma_bf16(d_tmem, adesc + (uint64_t)(kk * a_adv), bdesc + (uint64_t)(kk * b_adv),
                           idesc, (kt | kk) != 0);
          ptx::umma_commit(&ctl.empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        ptx::umma_commit(&ctl.tmem_full[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      // make sure no MMA is still running before TMEM is released
      ptx::umma_commit(&ctl.drain);
      if (!ptx::mbar_wait(&ctl.drain, 0, &ctl.abort, kWaitLimitNs)) {
        // abort already flagged: wait once more with the abort flag ignored
        int dummy = 0;
        ptx::mbar_wait(&ctl.drain, 0, &dummy, kWaitLimitNs);
      }
    }
    __syncwarp();
  } else {
    // ================================================================ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int r = q * 32 + lane;
    int cursor = 0, acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const Tile t = tile_at<MODE>(p, ctl, tile, cursor);
      if (M::kRagK) {
        const int Md = M::wg_mdim(p), Nd = M::wg_ndim(p);
        const int row = t.m0 + r;
        bf16* outp = (MODE == GEMM_WGRAD_W1 ? p.out0 : p.out1) + (size_t)t.e * Md * Nd;
        if (t.nk == 0) {
          if (row < Md) {
            float z[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) z[i] = 0.f;
            for (int cc = 0; cc < BN / 32; ++cc)
              if (t.n0 + 32 * cc < Nd) store32(outp + (size_t)row * Nd + t.n0 + 32 * cc, z);
          }
          continue;
        }
        if (!ptx::mbar_wait(&ctl.tmem_full[acc], acc_phase, &ctl.abort, kWaitLimitNs)) {
          if (lane == 0) flag_timeout(ctl, p.status, 5);
          break;
        }
        ptx::tc_fence_after();
        const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
        for (int cc = 0; cc < BN / 32; ++cc) {
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(tbase + 32 * cc, v);
          ptx::tmem_ld_wait();
          if (row < Md && t.n0 + 32 * cc < Nd)
            store32(outp + (size_t)row * Nd + t.n0 + 32 * cc, reinterpret_cast<float*>(v));
        }
      } else {
        if (!ptx::mbar_wait(&ctl.tmem_full[acc], acc_phase, &ctl.abort, kWaitLimitNs)) {
          if (lane == 0) flag_timeout(ctl, p.status, 5);
          break;
        }
        ptx::tc_fence_after();
        const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
        const bool row_ok = r < t.rows;
        const size_t grow = (size_t)t.row0 + t.m0 + r;
        if (MODE == GEMM_FC1_FWD) {
          // columns 0..127: gate f0.., columns 128..255: up f0..
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t g[32], u[32];
            ptx::tmem_ld_32x32b_x32(tbase + 32 * cc, g);
            ptx::tmem_ld_32x32b_x32(tbase + 128 + 32 * cc, u);
            ptx::tmem_ld_wait();
            const int f = t.n0 + 32 * cc;
            if (row_ok && f < p.F) {
              float ag[32], au[32], hv[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                ag[i] = round_bf16(__uint_as_float(g[i]));
                au[i] = round_bf16(__uint_as_float(u[i]));
                hv[i] = ag[i] / (1.f + __expf(-ag[i])) * au[i];
              }
              bf16* arow = p.out0 + grow * (size_t)(2 * p.F);
              store32(arow + f, ag);
              store32(arow + p.F + f, au);
              store32(p.out1 + grow * (size_t)p.F + f, hv);
            }
          }
        } else if (MODE == GEMM_FC2_DGRAD) {
          for (int cc = 0; cc < BN / 32; ++cc) {
            uint32_t v[32];
            ptx::tmem_ld_32x32b_x32(tbase + 32 * cc, v);
            ptx::tmem_ld_wait();
            const int f = t.n0 + 32 * cc;
            if (row_ok && f < p.F) {
              const bf16* arow = p.aux + grow * (size_t)(2 * p.F);
              float ag[32], au[32], dg[32], du[32];
              load32(arow + f, ag);
              load32(arow + p.F + f, au);
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const float dh = __uint_as_float(v[i]);
                const float s = 1.f / (1.f + __expf(-ag[i]));
                du[i] = dh * ag[i] * s;
                dg[i] = dh * au[i] * s * (1.f + ag[i] * (1.f - s));
              }
              bf16* drow = p.out0 + grow * (size_t)(2 * p.F);
              store32(drow + f, dg);
              store32(drow + p.F + f, du);
            }
          }
        } else {
          const int Nd = MODE == GEMM_FC2_FWD || MODE == GEMM_FC1_DGRAD ? p.H : p.F;
          for (int cc = 0; cc < BN / 32; ++cc) {
            uint32_t v[32];
            ptx::tmem_ld_32x32b_x32(tbase + 32 * cc, v);
            ptx::tmem_ld_wait();
            const int n = t.n0 + 32 * cc;
            if (row_ok && n < Nd)
              store32(p.out0 + grow * (size_t)Nd + n, reinterpret_cast<float*>(v));
          }
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(&ctl.tmem_empty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem_base, kTmemCols);
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// rows x cols bf16 row-major matrix, box = box_rows x 64 columns, 128B swizzle
bool make_map(CUtensorMap* m, const void* base, long long rows, long long cols, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return false;
  }
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (%d) for a %lld x %lld map", (int)r, rows, cols);
    return false;
  }
  return true;
}

template <int MODE>
moe_status_t launch_mode(const CUtensorMap& a, const CUtensorMap& b, const KParams& p, int grid,
                         cudaStream_t st) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(grouped_gemm_kernel<MODE>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDynSmem);
  });
  if (attr_err != cudaSuccess) {
    set_error("cudaFuncSetAttribute failed: %s", cudaGetErrorString(attr_err));
    return MOE_ERR_CUDA;
  }
  {
    LaunchScope _ls(K_GEMM_FC1_FWD + MODE, st);
    grouped_gemm_kernel<MODE><<<grid, kThreads, kDynSmem, st>>>(a, b, p);
  }
  return check_launch("grouped_gemm_kernel");
}

}  // namespace

moe_status_t launch_grouped_gemm(const moe_layer_desc_t& d, const GemmArgs& g, cudaStream_t st) {
  const long long N = (long long)d.T * d.k;
  const int E = d.E, H = d.H, F = d.F;
  if (N == 0) {
    if (g.mode == GEMM_WGRAD_W1) {
      cudaError_t e = cudaMemsetAsync(g.out0, 0, (size_t)E * 2 * F * H * 2, st);
      if (e != cudaSuccess) { set_error("cudaMemsetAsync: %s", cudaGetErrorString(e)); return MOE_ERR_CUDA; }
    }
    if (g.mode == GEMM_WGRAD_W2) {
      cudaError_t e = cudaMemsetAsync(g.out1, 0, (size_t)E * H * F * 2, st);
      if (e != cudaSuccess) { set_error("cudaMemsetAsync: %s", cudaGetErrorString(e)); return MOE_ERR_CUDA; }
    }
    return MOE_OK;
  }
  CUtensorMap ma, mb;
  bool ok = true;
  long long ntile_bound = 0;  // upper bound on tiles, for the grid size
  switch (g.mode) {
    case GEMM_FC1_FWD:
      ok = make_map(&ma, g.A, N, H, 128) && make_map(&mb, g.B, (long long)E * 2 * F, H, 128);
      ntile_bound = (N / BM + E) * ((F + 127) / 128);
      break;
    case GEMM_FC2_FWD:
      ok = make_map(&ma, g.A, N, F, 128) && make_map(&mb, g.B, (long long)E * H, F, 256);
      ntile_bound = (N / BM + E) * ((H + BN - 1) / BN);
      break;
    case GEMM_FC2_DGRAD:
      ok = make_map(&ma, g.A, N, H, 128) && make_map(&mb, g.B, (long long)E * H, F, 64);
      ntile_bound = (N / BM + E) * ((F + BN - 1) / BN);
      break;
    case GEMM_FC1_DGRAD:
      ok = make_map(&ma, g.A, N, 2 * F, 128) && make_map(&mb, g.B, (long long)E * 2 * F, H, 64);
      ntile_bound = (N / BM + E) * ((H + BN - 1) / BN);
      break;
    case GEMM_WGRAD_W1:
      ok = make_map(&ma, g.A, N, 2 * F, 64) && make_map(&mb, g.B, N, H, 64);
      ntile_bound = (long long)E * ((2 * F + BM - 1) / BM) * ((H + BN - 1) / BN);
      break;
    case GEMM_WGRAD_W2:
      ok = make_map(&ma, g.A, N, H, 64) && make_map(&mb, g.B, N, F, 64);
      ntile_bound = (long long)E * ((H + BM - 1) / BM) * ((F + BN - 1) / BN);
      break;
    default:
      set_error("unknown grouped GEMM mode %d", g.mode);
      return MOE_ERR_INVALID_ARG;
  }
  if (!ok) return MOE_ERR_CUDA;
  KParams p;
  p.E = E;
  p.H = H;
  p.F = F;
  p.N = N;
  p.off = g.off;
  p.out0 = g.out0;
  p.out1 = g.out1;
  p.aux = g.aux;
  p.status = g.status;
  int grid = device_sm_count();
  if (g.max_ctas > 0 && g.max_ctas < grid) grid = g.max_ctas;
  if (ntile_bound < grid) grid = (int)(ntile_bound > 0 ? ntile_bound : 1);
  switch (g.mode) {
    case GEMM_FC1_FWD: return launch_mode<GEMM_FC1_FWD>(ma, mb, p, grid, st);
    case GEMM_FC2_FWD: return launch_mode<GEMM_FC2_FWD>(ma, mb, p, grid, st);
    case GEMM_FC2_DGRAD: return launch_mode<GEMM_FC2_DGRAD>(ma, mb, p, grid, st);
    case GEMM_FC1_DGRAD: return launch_mode<GEMM_FC1_DGRAD>(ma, mb, p, grid, st);
    case GEMM_WGRAD_W1: return launch_mode<GEMM_WGRAD_W1>(ma, mb, p, grid, st);
    default: return launch_mode<GEMM_WGRAD_W2>(ma, mb, p, grid, st);
  }
}

}  // namespace moe
