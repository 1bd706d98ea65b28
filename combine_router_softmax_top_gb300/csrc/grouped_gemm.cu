// Grouped expert GEMMs of the "mlp" phase on the sm_100-family tensor cores
// (tcgen05 MMA with TMEM accumulators, operands staged by TMA), for the forward,
// the activation gradient (dgrad) and the deferrable weight gradient (wgrad);
// the dgrad/wgrad split follows the EP-overlap note ("1. MoE EP Overlap",
// section "MoE 1F1B overlap": the mlp backward computes the activation gradient
// first so dispatch-backward can start, and the weight gradient later).
//
// One persistent kernel per call, one CTA per SM, warp-specialised:
//   warp 0      TMA producer (ring of A|B stages: 4 x 48 KB, or 6 x 32 KB per CTA in pairs)
//   warp 1      TMEM allocator + single-thread MMA issuer
//   warps 2..9  epilogue: TMEM -> registers -> fused math -> global, by TMA
//               tensor stores (or fp32 TMA reductions when a weight gradient
//               is accumulated) or coalesced warp stores
//               (two warps per TMEM lane quarter, each owning half the columns)
//   warp 10     FC2 dgrad only: loads the saved pre-activation for the epilogue
// Tiles are 128 x 256 (one tcgen05.mma M=128, N=256, K=16 per step, 4 steps
// per 64-wide K stage); forward and dgrad tiles run on CTA pairs (M = 256).
// The 512 TMEM columns hold two accumulators, so the epilogue of one tile
// overlaps the MMAs of the next. A launch may chain two modes (FC1 -> FC2
// forward, FC2 dgrad -> FC1 dgrad): the second mode's tiles of an expert start
// once the first mode's tiles of that expert are stored.
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

#ifndef MOE_ROW_CS
#define MOE_ROW_CS 1
#endif
#ifndef MOE_PAIR
#define MOE_PAIR 1
#endif
#ifndef MOE_WG1_CS
#define MOE_WG1_CS 2
#endif
#ifndef MOE_WG2_CS
#define MOE_WG2_CS 2
#endif

namespace moe {

namespace {

constexpr int BM = 128, BN = 256, BK = 64;  // BN: widest tile (per-mode width is kBN)
constexpr int kStagesMax = 6;
constexpr int kABytes = BM * BK * 2;   // 16 KB
constexpr int kAccCols = 256;          // TMEM columns per accumulator buffer
constexpr int kTmemCols = 512;
constexpr int kMaxE = 256;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s without progress -> give up
constexpr size_t kEpiStageBytes = 8 * 2048;  // one 32x32 bf16 staging buffer per epilogue warp

struct KParams {
  int E, H, F;
  long long N;
  const int32_t* off;
  bf16* out0;
  bf16* out1;
  const bf16* aux;
  int* status;
  int* dep;  // fused launches: per-expert count of first-mode epilogue warps done
};

template <int MODE>
struct Mode {
  static constexpr bool kRagK = MODE == GEMM_WGRAD_W1 || MODE == GEMM_WGRAD_W2;
  static constexpr int kAMn = kRagK ? 1 : 0;
  static constexpr int kBMn = (MODE == GEMM_FC2_DGRAD || MODE == GEMM_FC1_DGRAD || kRagK) ? 1 : 0;
  // CTAs per cluster: kCS consecutive M blocks of one (expert, N block) share
  // the B tile; each CTA loads a slice and multicasts it to all of them.
  // CTA pairs (tcgen05 cta_group::2): M = 256 rows per MMA, each CTA loading
  // its own 128 rows of A and half of B, so a CTA takes in 32 KB per K stage
  // instead of 48 KB and holds 6 stages. Pairs speed up the forward and dgrad
  // GEMMs. The short-K wgrad tiles (4 K stages per expert at 256 rows) stay
  // unpaired and share B across a cluster by multicast. Measured on the
  // 256-rows-per-expert layer, clusters of 2 are fastest (W1 201 us against
  // 208 us unclustered and 220 to 223 us with 3, 4 or 6 CTAs; W2 115 us with
  // 2 to 4, 129 us with 8). A paired wgrad (each CTA loading its own A and
  // half of B, 128 KB per 128 x 256 output instead of 192 KB received) stays
  // slower even with the pair handshakes trimmed (one arrival per stage, the
  // odd CTA's accumulator release forwarded once per tile): W1 222 us, W2
  // 130 us. A trace shows each short tile's MMA resuming 1.3 to 1.6 us after
  // both epilogues released the accumulator, a latency two accumulators do
  // not hide when a tile's MMAs take 1.2 us.
  static constexpr bool kPair = MOE_PAIR && !kRagK;
  static constexpr int kCS = kPair ? 2
                            : MODE == GEMM_WGRAD_W1 ? MOE_WG1_CS
                            : MODE == GEMM_WGRAD_W2 ? MOE_WG2_CS : MOE_ROW_CS;
  // The FC2 dgrad epilogue needs the tile's saved pre-activation (gate and up)
  // next to the accumulator: a dedicated warp TMA-loads it into shared memory
  // ahead of the epilogue, one 64-column quarter (gate and up, 32 KB) at a time.
  static constexpr bool kAux = MODE == GEMM_FC2_DGRAD;
  static constexpr int kBN = 256;
  static constexpr int kBBytes = kBN * BK * 2;            // whole B tile per stage
  static constexpr int kBBytesCta = kPair ? kBBytes / 2 : kBBytes;  // B bytes this CTA loads
  static constexpr int kStageBytes = kABytes + kBBytesCta;
  // stages of the operand ring (with the aux buffer a launch fits 5 pair stages);
  // the warps are a producer, the MMA issuer, 8 epilogue warps and, for kAux,
  // the aux loader (see Fuse below, which sizes a launch)
  static constexpr int kStages = kPair ? (kAux ? 5 : 6) : 4;
  // Plain bf16 outputs leave through TMA tensor stores of 32 x 32 boxes (the
  // staging buffer is the box): 2D [rows, cols] maps for the forward FC2 and
  // FC1 dgrad outputs, 3D [expert, rows, cols] maps for the weight gradients,
  // whose clipping at the matrix edge makes every wgrad box storable. 0: none.
  static constexpr int kStoreDims =
      (MODE == GEMM_FC2_FWD || MODE == GEMM_FC1_DGRAD) ? 2 : kRagK ? 3 : 0;
  static_assert(kStages <= kStagesMax, "barrier arrays");
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
  uint64_t full[kStagesMax];
  uint64_t empty[kStagesMax];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t epi_done[2];  // pair, odd CTA: its epilogue warps released the accumulator
  uint64_t drain;
  uint64_t aux_full;
  uint64_t aux_empty;
  uint32_t tmem_base;
  int abort;
  int tstart[kMaxE + 1];   // tile prefix of the (first) mode, over expert positions
  int tstart2[kMaxE + 1];  // tile prefix of the second mode of a fused launch
  int off[kMaxE + 1];
  int order[kMaxE];        // K-ragged modes: expert at each position (longest first)
};

template <int MODE>
__device__ __forceinline__ Tile tile_at(const KParams& p, const int* tstart, const int* off,
                                       const int* order, int tile, int& cursor,
                                       uint32_t rank = 0) {
  while (tstart[cursor + 1] <= tile) ++cursor;
  Tile t;
  t.e = Mode<MODE>::kRagK ? order[cursor] : cursor;
  t.row0 = off[t.e];
  const int cnt = off[t.e + 1] - t.row0;
  const int local = tile - tstart[cursor];
  if (Mode<MODE>::kRagK) {
    // one cluster tile = kCS consecutive M blocks of one (expert, N block)
    constexpr int cs = Mode<MODE>::kCS;
    const int mg = ((Mode<MODE>::wg_mdim(p) + BM - 1) / BM + cs - 1) / cs;
    t.m0 = ((local % mg) * cs + (int)rank) * BM;
    t.n0 = (local / mg) * BN;
    t.rows = cnt;
    t.nk = (cnt + BK - 1) / BK;
  } else {
    constexpr int cs = Mode<MODE>::kCS;
    const int mg = ((cnt + BM - 1) / BM + cs - 1) / cs;  // cluster tiles along M
    t.m0 = ((local % mg) * cs + (int)rank) * BM;
    t.n0 = (local / mg) * (MODE == GEMM_FC1_FWD ? 128 : Mode<MODE>::kBN);
    t.rows = min(BM, cnt - t.m0);  // <= 0: this CTA's M block is past the expert
    t.nk = Mode<MODE>::kdim(p) / BK;
  }
  return t;
}

// Profiling builds (-DMOE_TRACE) record, for CTA 0, the global time at which
// each role starts and finishes each of its first 128 tiles, into the bytes
// after the status words (the router-logits scratch, unused when the caller
// passes its own logits buffer). Product builds compile this away.
__device__ __forceinline__ void trace(const KParams& p, int mode, int ev, int i) {
#ifdef MOE_TRACE
  if (blockIdx.x == 0 && i < 128)
    reinterpret_cast<uint64_t*>(reinterpret_cast<char*>(p.status) + 256 + mode * 8192)[i * 8 + ev] =
        ptx::globaltimer_ns();
#endif
}

__device__ __forceinline__ void flag_timeout(SmemCtl& c, int* status, int where) {
  c.abort = 1;
  atomicExch(status + ST_TIMEOUT, where);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&b);
}

// Writes a warp's 32 rows x 32 columns (thread i holds row i) to global memory
// as bf16 with full-sector stores: the rows go through a 2 KB shared buffer,
// then each store instruction covers 8 rows x 64 contiguous bytes. 16-byte
// chunk c of row r sits at chunk c ^ ((r >> 1) & 3) of the row in the buffer,
// which keeps both the row-wise writes and the transposed reads free of bank
// conflicts. Rows >= valid_rows and a chunk with cols_ok == false are skipped.
__device__ __forceinline__ void warp_store32(uint4* stage, const float* v, bf16* base, int ld,
                                             int lane, int valid_rows, bool cols_ok) {
#pragma unroll
  for (int q = 0; q < 4; ++q)
    stage[lane * 4 + (q ^ ((lane >> 1) & 3))] =
        make_uint4(pack_bf16x2(v[8 * q + 0], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                   pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
  __syncwarp();
  if (cols_ok) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = i * 8 + (lane >> 2), c = lane & 3;
      if (row < valid_rows)
        reinterpret_cast<uint4*>(base + (size_t)row * ld)[c] = stage[row * 4 + (c ^ ((row >> 1) & 3))];
    }
  }
  __syncwarp();
}

// Element i (0..31) of 32 bf16 held as 4 x uint4.
__device__ __forceinline__ float bf16_at(const uint4 (&u)[4], int i) {
  const uint4& w = u[i >> 3];
  const uint32_t word = ((i >> 1) & 3) == 0 ? w.x : ((i >> 1) & 3) == 1 ? w.y : ((i >> 1) & 3) == 2 ? w.z : w.w;
  return __uint_as_float((i & 1) ? (word & 0xFFFF0000u) : (word << 16));
}

// Stores this warp's half of a plain fp32 accumulator tile (BN/64 chunks of 32
// columns starting at chunk c0) as bf16; the TMEM load of the next chunk is in
// flight while the current one is written out.
//
// With a store map (dims 2 or 3) each 32 x 32 chunk goes out as one TMA store
// of the staging buffer at box (x0 + 32 * chunk, y0[, z0]); lane 0 issues it
// and, before the buffer is rewritten, waits until the previous store has read
// it. A 2D map spans all rows of the output, so a slab with fewer than 32 valid
// rows (the rows past it belong to the next expert) takes the plain stores.
__device__ __forceinline__ void store_chunks(uint4* stage, uint32_t tbase, int c0, bf16* slab,
                                             int ld, int n0, int lane, int slab_rows,
                                             const CUtensorMap* tm, int dims, int x0, int y0,
                                             int z0) {
  const bool tma = dims == 3 || (dims == 2 && slab_rows == 32);
  uint32_t va[32], vb[32];
  ptx::tmem_ld_32x32b_x32(tbase + 32 * c0, va);
  ptx::tmem_ld_wait(va);
#pragma unroll
  for (int i = 0; i < BN / 64; ++i) {
    const int cc = c0 + i;
    uint32_t(&cur)[32] = (i & 1) ? vb : va;
    uint32_t(&nxt)[32] = (i & 1) ? va : vb;
    if (i + 1 < BN / 64) ptx::tmem_ld_32x32b_x32(tbase + 32 * (cc + 1), nxt);
    const bool cols_ok = n0 + 32 * cc < ld;
    if (tma) {
      if (slab_rows > 0 && cols_ok) {
        if (lane == 0) ptx::bulk_wait_group_read0();
        __syncwarp();
        const float* v = reinterpret_cast<const float*>(cur);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          stage[lane * 4 + (q ^ ((lane >> 1) & 3))] = make_uint4(
              pack_bf16x2(v[8 * q + 0], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
              pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (dims == 3) ptx::tma_store_3d(tm, stage, x0 + 32 * cc, y0, z0);
          else ptx::tma_store_2d(tm, stage, x0 + 32 * cc, y0);
          ptx::bulk_commit_group();
        }
      }
    } else {
      if (dims) {
        if (lane == 0) ptx::bulk_wait_group_read0();
        __syncwarp();
      }
      warp_store32(stage, reinterpret_cast<float*>(cur), slab + 32 * cc, ld, lane, slab_rows,
                   cols_ok);
    }
    if (i + 1 < BN / 64) ptx::tmem_ld_wait(nxt);
  }
}

// Adds this warp's half of an fp32 accumulator tile (BN/64 chunks of 32
// columns from chunk c0, rows y0..y0+31) into an fp32 3D [expert, rows, cols]
// buffer. Each chunk leaves as two 16-row x 32-column boxes (full 128-byte
// lines; lanes 0-15, then lanes 16-31, fill the staging buffer), added
// element-wise in L2 by TMA reductions; the map clips boxes at the matrix
// edge, and a box wholly past the last row is skipped. 128-byte rows beat
// 32 x 16 boxes of 64-byte rows by 3.5% (fc1: 647 against 670 us). Every
// element is added exactly once per launch, so the result is fl(old + tile)
// whatever the order in which tiles finish.
__device__ __forceinline__ void reduce_chunks_f32(uint4* stage, uint32_t tbase, int c0, int lane,
                                                  int ncols, int nrows, const CUtensorMap* tm,
                                                  int x0, int y0, int z0) {
  uint32_t va[32], vb[32];
  ptx::tmem_ld_32x32b_x32(tbase + 32 * c0, va);
  ptx::tmem_ld_wait(va);
#pragma unroll
  for (int i = 0; i < BN / 64; ++i) {
    const int cc = c0 + i;
    uint32_t(&cur)[32] = (i & 1) ? vb : va;
    uint32_t(&nxt)[32] = (i & 1) ? va : vb;
    if (i + 1 < BN / 64) ptx::tmem_ld_32x32b_x32(tbase + 32 * (cc + 1), nxt);
    const int x = x0 + 32 * cc;
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      if (x < ncols && y0 + 16 * hb < nrows) {
        if (lane == 0) ptx::bulk_wait_group_read0();
        __syncwarp();
        if ((lane >> 4) == hb) {
          const int r = lane & 15;
#pragma unroll
          for (int q = 0; q < 8; ++q)
            stage[r * 8 + (q ^ (r & 7))] =
                make_uint4(cur[4 * q], cur[4 * q + 1], cur[4 * q + 2], cur[4 * q + 3]);
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          ptx::tma_reduce_add_3d(tm, stage, x, y0 + 16 * hb, z0);
          ptx::bulk_commit_group();
        }
      }
    }
    if (i + 1 < BN / 64) ptx::tmem_ld_wait(nxt);
  }
}

// Logistic sigmoid s(x) = 1 / (1 + e^-x), from the fast exponential and the
// fast division intrinsics. Its relative error stays near 1e-6 over the whole
// range, including large negative x where s is tiny: there e^-x is large and
// both intrinsics keep their relative accuracy (for x below about -88, e^-x is
// inf and s rounds to 0, the correct value to fp32 precision). A form through
// (1 + tanh(x/2)) / 2 with the hardware tanh loses s for negative x: tanh's
// ~2^-11 relative error near t = -1 is an absolute error of ~2.4e-4 in s,
// which is 1.3% of s at x = -4 and exceeds s itself below x = -9.
__device__ __forceinline__ float sigmoid_f(float x) {
  return __fdividef(1.f, 1.f + __expf(-x));
}

__device__ __forceinline__ float round_bf16(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

// Launch-wide constants of a kernel that runs the tiles of MODE and then, when
// MODE2 >= 0, those of MODE2 in the same persistent launch. MODE2's tiles of
// expert e wait until every tile of expert e of MODE has stored its output
// (per-expert counters), so one grid works through both GEMMs and the second
// fills the last, partial round of tiles of the first.
template <int MODE, int MODE2>
struct Fuse {
  using A = Mode<MODE>;
  using B = Mode<(MODE2 >= 0 ? MODE2 : MODE)>;
  static constexpr bool kHas2 = MODE2 >= 0;
  // the second mode reads the first mode's output (forward and dgrad chains);
  // the two weight gradients of a wgrad launch are independent of each other
  static constexpr bool kDep = kHas2 && !A::kRagK;
  static constexpr bool kAux = A::kAux || (kHas2 && B::kAux);
  static constexpr int kStages = A::kStages < B::kStages ? A::kStages : B::kStages;
  static constexpr int kStageBytes = A::kStageBytes;
  static constexpr int kAuxBytes = kAux ? 2 * 16384 : 0;
  static constexpr int kWarps = kAux ? 11 : 10;
  static constexpr bool kPair = A::kPair;
  static constexpr int kCS = A::kCS;
  static constexpr bool kStores = A::kStoreDims != 0 || (kHas2 && B::kStoreDims != 0);
  static constexpr size_t kDynSmem =
      (size_t)kStages * kStageBytes + kAuxBytes + kEpiStageBytes + 1024;
  static_assert(A::kStageBytes == B::kStageBytes && A::kPair == B::kPair && A::kCS == B::kCS &&
                    A::kAMn == B::kAMn && A::kBMn == B::kBMn && A::kBN == B::kBN &&
                    A::kRagK == B::kRagK,
                "fused modes must share the tile machinery");
};

// What every role needs about its CTA.
struct Role {
  uint8_t* smem;
  SmemCtl* ctl;
  uint32_t crank;
  uint16_t cmask;
  uint32_t tmem_base;
  int lane;
};

// Tiles per expert -> exclusive prefix over expert positions (warp 0). The
// K-ragged (wgrad) modes visit the experts longest first (order[]): a tile's
// cost grows with its expert's rows, and with the tiles handed to the CTAs
// in stride order, longest-first deals each CTA a similar mix of long and
// short tiles (on a skewed layer the most loaded CTA drops from 1.15x to
// 1.07x the mean for dW1, and from 1.27x to 1.12x for dW2, in K stages).
// The other modes keep expert order, which their chaining relies on.
template <int MODE>
__device__ __forceinline__ void tile_prefix(const KParams& p, const int* off, const int* order,
                                            int* tstart, int lane) {
  using M = Mode<MODE>;
  int carry = 0;
  for (int base = 0; base < p.E; base += 32) {
    const int pos = base + lane;
    const int e = M::kRagK && pos < p.E ? order[pos] : pos;
    int n = 0;
    if (pos < p.E) {
      const int cnt = off[e + 1] - off[e];
      if (M::kRagK)
        n = (((M::wg_mdim(p) + BM - 1) / BM + M::kCS - 1) / M::kCS) * M::ntiles(p);
      else n = (((cnt + BM - 1) / BM + M::kCS - 1) / M::kCS) * M::ntiles(p);
      if (cnt < 0) n = 0;
    }
    int incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (pos < p.E) tstart[pos] = carry + incl - n;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) tstart[p.E] = carry;
}

// order[r] = the expert with the r-th most rows, ties to the lower index
// (one thread per expert; the identity when all experts have equal rows).
__device__ __forceinline__ void longest_first(const int* off, int E, int* order) {
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int c = off[e + 1] - off[e];
    int r = 0;
    for (int f = 0; f < E; ++f) {
      const int cf = off[f + 1] - off[f];
      r += (cf > c) || (cf == c && f < e);
    }
    order[r] = e;
  }
}

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Producer of a second-mode tile: wait (bounded) until expert e's first-mode
// tiles have all stored their output, then order those generic-proxy writes
// before this thread's TMA (async-proxy) reads of them.
__device__ __forceinline__ bool wait_expert(const KParams& p, int e, int target,
                                            volatile int* abort) {
  if (ld_acquire(p.dep + e) < target) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (ld_acquire(p.dep + e) < target) {
      __nanosleep(128);
      if (*abort) return false;
      if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return true;
}

// ==================================================================== producer
// Loads one tile's K stages (A and B) into the stage ring.
template <int MODE, int KSTAGES>
__device__ __forceinline__ bool producer_tile(const Role& R, const KParams& p,
                                              const CUtensorMap* tmA, const CUtensorMap* tmB,
                                              const Tile& t, int& stage, uint32_t& phase) {
  using M = Mode<MODE>;
  SmemCtl& ctl = *R.ctl;
  const int lane = R.lane;
  const uint32_t crank = R.crank;
  const uint16_t cmask = R.cmask;
  for (int kt = 0; kt < t.nk; ++kt) {
    if (!ptx::mbar_wait(&ctl.empty[stage], phase ^ 1, &ctl.abort, kWaitLimitNs)) {
      if (lane == 0) flag_timeout(ctl, p.status, 1);
      return false;
    }
    uint8_t* sA = R.smem + stage * M::kStageBytes;
    uint8_t* sB = sA + kABytes;
    const int k0 = kt * BK;
    uint64_t* bar = &ctl.full[stage];
    if (lane == 0) {
      if (M::kRagK) {
        // A: this CTA's own M block. B: slice i of the shared tile is loaded
        // by cluster rank i % kCS and multicast to every CTA of the cluster,
        // so full[stage] collects all 32 KB of B in every CTA. In the last K
        // stage of an expert the rows past its end are the next expert's;
        // the MMA warp zeroes them in A once the stage has landed, so the
        // producer never waits for a load.
        ptx::mbar_arrive_expect_tx(&ctl.full[stage], M::kStageBytes);
        const int r = t.row0 + k0;
        ptx::tma_load_2d(sA, tmA, bar, t.m0, r);
        ptx::tma_load_2d(sA + 8192, tmA, bar, t.m0 + 64, r);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (M::kCS == 1)
            ptx::tma_load_2d(sB + 8192 * i, tmB, &ctl.full[stage], t.n0 + 64 * i, r);
          else if (i % M::kCS == (int)crank)
            ptx::tma_load_2d_multicast(sB + 8192 * i, tmB, &ctl.full[stage], t.n0 + 64 * i, r,
                                       cmask);
        }
      } else if (M::kPair) {
        // both CTAs' loads complete on the even CTA's full[stage]
        const uint32_t fb = ptx::mapa_shared(&ctl.full[stage], 0);
        if (crank == 0) ptx::mbar_arrive_expect_tx(&ctl.full[stage], 2 * M::kStageBytes);
        ptx::tma_load_2d_pair(sA, tmA, fb, k0, t.row0 + t.m0);
        if (MODE == GEMM_FC1_FWD) {  // even CTA: 128 gate rows, odd CTA: 128 up rows
          ptx::tma_load_2d_pair(sB, tmB, fb, k0, t.e * 2 * p.F + (crank ? p.F : 0) + t.n0);
        } else if (MODE == GEMM_FC2_FWD) {
          ptx::tma_load_2d_pair(sB, tmB, fb, k0, t.e * p.H + t.n0 + 128 * crank);
        } else {  // MN-major B: this CTA's half of the N columns
          const int base = MODE == GEMM_FC2_DGRAD ? t.e * p.H : t.e * 2 * p.F;
          constexpr int nb = M::kBN / 128;  // 64-wide boxes per CTA
#pragma unroll
          for (int i = 0; i < nb; ++i)
            ptx::tma_load_2d_pair(sB + 8192 * i, tmB, fb, t.n0 + 64 * (crank * nb + i), base + k0);
        }
      } else {
        ptx::mbar_arrive_expect_tx(bar, M::kStageBytes);
        ptx::tma_load_2d(sA, tmA, bar, k0, t.row0 + t.m0);
        // B boxes: box i is loaded by cluster rank i % kCS and multicast
        auto load_b = [&](int i, void* dst, int c0, int c1) {
          if (M::kCS == 1)
            ptx::tma_load_2d(dst, tmB, bar, c0, c1);
          else if (i % M::kCS == (int)crank)
            ptx::tma_load_2d_multicast(dst, tmB, bar, c0, c1, cmask);
        };
        if (MODE == GEMM_FC1_FWD) {
          const int base = t.e * 2 * p.F;
          load_b(0, sB, k0, base + t.n0);                // 128 gate rows
          load_b(1, sB + 16384, k0, base + p.F + t.n0);  // 128 up rows
        } else if (MODE == GEMM_FC2_FWD) {
          load_b(0, sB, k0, t.e * p.H + t.n0);
          load_b(1, sB + 16384, k0, t.e * p.H + t.n0 + 128);
        } else {
          const int base = MODE == GEMM_FC2_DGRAD ? t.e * p.H : t.e * 2 * p.F;
#pragma unroll
          for (int i = 0; i < M::kBN / 64; ++i) load_b(i, sB + 8192 * i, t.n0 + 64 * i, base + k0);
        }
      }
    }
    if (++stage == KSTAGES) {
      stage = 0;
      phase ^= 1;
    }
  }
  return true;
}

// ==================================================================== MMA issuer
// Issues one tile's MMAs into accumulator acc (pair: for both CTAs).
template <int MODE, int KSTAGES>
__device__ __forceinline__ bool mma_tile(const Role& R, const KParams& p, const Tile& t,
                                         int& stage, uint32_t& phase, int& acc,
                                         uint32_t& acc_phase, int ti) {
  using M = Mode<MODE>;
  SmemCtl& ctl = *R.ctl;
  constexpr uint32_t idesc =
      ptx::idesc_bf16_f32(M::kPair ? 2 * BM : BM, M::kBN, M::kAMn, M::kBMn);
  constexpr uint32_t a_lbo = M::kAMn ? 8192 : 16, b_lbo = M::kBMn ? 8192 : 16;
  constexpr uint32_t a_adv = M::kAMn ? (2048 >> 4) : (32 >> 4);
  constexpr uint32_t b_adv = M::kBMn ? (2048 >> 4) : (32 >> 4);
  // K-ragged (wgrad) launches run this on all 32 lanes of the MMA warp, the
  // others on lane 0 alone; one lane issues the MMAs and commits either way
  const bool issuer = !M::kRagK || R.lane == 0;
  // (every lane waits and the warp agrees on the outcome, so it stays converged)
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    const bool got = ptx::mbar_wait(bar, parity, &ctl.abort, kWaitLimitNs);
    return M::kRagK ? __all_sync(0xffffffffu, got) : got;
  };
  if (t.nk == 0) return true;
  if (!wait(&ctl.tmem_empty[acc], acc_phase ^ 1)) {
    flag_timeout(ctl, p.status, 3);
    return false;
  }
  ptx::tc_fence_after();
  if (issuer) trace(p, MODE, 2, ti);
  const uint32_t d_tmem = R.tmem_base + acc * kAccCols;
  for (int kt = 0; kt < t.nk; ++kt) {
    if (!wait(&ctl.full[stage], phase)) {
      flag_timeout(ctl, p.status, 4);
      return false;
    }
    ptx::tc_fence_after();
    uint8_t* sA = R.smem + stage * M::kStageBytes;
    int nkk = BK / 16;
    if (M::kRagK && t.rows - kt * BK < BK) {
      // last K stage of the expert: only the 16-row MMA steps that hold its
      // rows run, and the rows of the next expert inside the last of them
      // are zeroed in A (rows are 128 B in both 8 KB atoms, whatever the
      // swizzle), by the whole warp, before the MMAs read the stage
      const int valid = t.rows - kt * BK;  // 1..63
      nkk = (valid + 15) / 16;
      const int nzero = (nkk * 16 - valid) * 8;  // 16-byte chunks per atom
      for (int i = R.lane; i < 2 * nzero; i += 32) {
        const int atom = i / nzero, j = i % nzero;
        *(reinterpret_cast<uint4*>(sA + atom * 8192 + valid * 128) + j) = make_uint4(0, 0, 0, 0);
      }
      ptx::fence_proxy_async_smem();
      __syncwarp();
      ptx::tc_fence_after();
    }
    const uint32_t a_addr = ptx::smem_u32(sA);
    const uint32_t b_addr = a_addr + kABytes;
    const uint64_t adesc = ptx::sdesc_sw128(a_addr, a_lbo, 1024);
    const uint64_t bdesc = ptx::sdesc_sw128(b_addr, b_lbo, 1024);
    if (issuer) {
#pragma unroll
      for (int kk = 0; kk < BK / 16; ++kk) {
        if (kk >= nkk) break;
        if (M::kPair)
          ptx::umma_bf16_pair(d_tmem, adesc + (uint64_t)(kk * a_adv),
                              bdesc + (uint64_t)(kk * b_adv), idesc, (kt | kk) != 0);
        else
          ptx::umma_bf16(d_tmem, adesc + (uint64_t)(kk * a_adv), bdesc + (uint64_t)(kk * b_adv),
                         idesc, (kt | kk) != 0);
      }
      // the stage is free once every CTA whose shared memory the MMAs read
      // (pair) or that received the multicast B slices has consumed it
      if (M::kPair) ptx::umma_commit_pair(&ctl.empty[stage], 3);
      else if (M::kCS > 1) ptx::umma_commit_multicast(&ctl.empty[stage], R.cmask);
      else ptx::umma_commit(&ctl.empty[stage]);
    }
    if (++stage == KSTAGES) {
      stage = 0;
      phase ^= 1;
    }
  }
  if (issuer) {
    trace(p, MODE, 3, ti);
    if (M::kPair) ptx::umma_commit_pair(&ctl.tmem_full[acc], 3);
    else ptx::umma_commit(&ctl.tmem_full[acc]);
  }
  if (++acc == 2) {
    acc = 0;
    acc_phase ^= 1;
  }
  return true;
}

// ==================================================================== aux loader
// Loads a tile's saved pre-activation (FC2 dgrad), a 64-column quarter at a
// time, each once the epilogue has released the previous quarter.
template <int MODE, int KSTAGES>
__device__ __forceinline__ bool aux_tile(const Role& R, const KParams& p, const CUtensorMap* tmC,
                                         const Tile& t, uint32_t& ph) {
  using M = Mode<MODE>;
  SmemCtl& ctl = *R.ctl;
  uint8_t* aux = R.smem + KSTAGES * M::kStageBytes;
  const int row = t.row0 + t.m0;
  for (int qt = 0; qt < M::kBN / 64; ++qt) {
    if (!ptx::mbar_wait(&ctl.aux_empty, ph ^ 1, &ctl.abort, kWaitLimitNs)) {
      flag_timeout(ctl, p.status, 7);
      return false;
    }
    ph ^= 1;
    const int c = t.n0 + 64 * qt;
    ptx::mbar_arrive_expect_tx(&ctl.aux_full, 2 * 16384);
    ptx::tma_load_2d(aux, tmC, &ctl.aux_full, c, row);                // gate
    ptx::tma_load_2d(aux + 16384, tmC, &ctl.aux_full, p.F + c, row);  // up
  }
  return true;
}

// ==================================================================== epilogue
// One epilogue warp's share of a tile: TMEM -> registers -> fused math ->
// stores; then the warp releases the accumulator and, with SIGNAL (the first
// mode of a fused launch), counts the tile's expert as one warp further done.
template <int MODE, int KSTAGES, int AUXB, bool SIGNAL, bool ACC>
__device__ __forceinline__ bool epilogue_tile(const Role& R, const KParams& p,
                                              const CUtensorMap* tmD, const Tile& t, int& acc,
                                              uint32_t& acc_phase, uint32_t& aux_phase, int ew,
                                              int ti) {
  using M = Mode<MODE>;
  SmemCtl& ctl = *R.ctl;
  const int lane = R.lane;
  const int q = (ew + 2) & 3;  // TMEM lane quarter (hardware rule: warp id % 4)
  const int hf = ew >> 2;
  const int r = q * 32 + lane;
  uint4* stage = reinterpret_cast<uint4*>(R.smem + KSTAGES * M::kStageBytes + AUXB) + ew * 128;
  const bool tr = lane == 0 && (ew == 0 || ew == 4);
  const int c0 = hf * (M::kBN / 64);  // first 32-column chunk of this warp's half
  if (M::kRagK) {
    const int Md = M::wg_mdim(p), Nd = M::wg_ndim(p);
    bf16* outp = (MODE == GEMM_WGRAD_W1 ? p.out0 : p.out1) + (size_t)t.e * Md * Nd;
    const int slab_rows = min(32, Md - (t.m0 + q * 32));
    bf16* slab = outp + (size_t)(t.m0 + q * 32) * Nd;
    if (t.nk == 0) {
      // an expert with no rows: zero weight gradient (plain stores, after
      // the last TMA store has finished reading the staging buffer); when
      // accumulating, nothing is added
      if (ACC) return true;
      float z[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) z[i] = 0.f;
      if (lane == 0) ptx::bulk_wait_group_read0();
      __syncwarp();
      for (int cc = c0; cc < c0 + BN / 64; ++cc)
        warp_store32(stage, z, slab + t.n0 + 32 * cc, Nd, lane, slab_rows, t.n0 + 32 * cc < Nd);
      return true;
    }
    if (!ptx::mbar_wait(&ctl.tmem_full[acc], acc_phase, &ctl.abort, kWaitLimitNs)) {
      if (lane == 0) flag_timeout(ctl, p.status, 5);
      return false;
    }
    ptx::tc_fence_after();
    if (tr) trace(p, MODE, ew == 0 ? 4 : 6, ti);
    const uint32_t tbase = R.tmem_base + ((uint32_t)(q * 32) << 16) + acc * kAccCols;
    if (ACC) {
      if (slab_rows > 0)
        reduce_chunks_f32(stage, tbase, c0, lane, Nd, Md, tmD, t.n0, t.m0 + q * 32, t.e);
    } else {
      store_chunks(stage, tbase, c0, slab + t.n0, Nd, t.n0, lane, slab_rows, tmD, M::kStoreDims,
                   t.n0, t.m0 + q * 32, t.e);
    }
  } else {
    if (!ptx::mbar_wait(&ctl.tmem_full[acc], acc_phase, &ctl.abort, kWaitLimitNs)) {
      if (lane == 0) flag_timeout(ctl, p.status, 5);
      return false;
    }
    ptx::tc_fence_after();
    if (tr) trace(p, MODE, ew == 0 ? 4 : 6, ti);
    const uint32_t tbase = R.tmem_base + ((uint32_t)(q * 32) << 16) + acc * kAccCols;
    // this warp's 32-row slab of the tile, for the coalesced stores
    const size_t slab_row0 = (size_t)t.row0 + t.m0 + q * 32;
    const int slab_rows = min(32, t.rows - q * 32);
    if (MODE == GEMM_FC1_FWD) {
      // columns 0..127: gate f0.., columns 128..255: up f0..; this half: 2 chunks
      for (int cc = 2 * hf; cc < 2 * hf + 2; ++cc) {
        uint32_t g[32], u[32];
        ptx::tmem_ld_32x32b_x32(tbase + 32 * cc, g);
        ptx::tmem_ld_32x32b_x32(tbase + 128 + 32 * cc, u);
        ptx::tmem_ld_wait(g, u);
        const int f = t.n0 + 32 * cc;
        const bool cols_ok = f < p.F;
        // round gate/up to bf16 in place, then h from the rounded values
        float* ag = reinterpret_cast<float*>(g);
        float* au = reinterpret_cast<float*>(u);
        float hv[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          ag[i] = round_bf16(ag[i]);
          au[i] = round_bf16(au[i]);
          hv[i] = ag[i] * sigmoid_f(ag[i]) * au[i];
        }
        bf16* abase = p.out0 + slab_row0 * (size_t)(2 * p.F);
        warp_store32(stage, ag, abase + f, 2 * p.F, lane, slab_rows, cols_ok);
        warp_store32(stage, au, abase + p.F + f, 2 * p.F, lane, slab_rows, cols_ok);
        warp_store32(stage, hv, p.out1 + slab_row0 * (size_t)p.F + f, p.F, lane, slab_rows,
                     cols_ok);
      }
    } else if (MODE == GEMM_FC2_DGRAD) {
      // the pre-activation slab arrives one 64-column quarter at a time: a
      // gate box and an up box of 128 rows x 64 columns, 128-byte swizzled
      // (16-byte chunk j of row r sits at chunk j ^ (r & 7)). A quarter is
      // 2 chunks of 32 columns; each warp takes one.
      const uint8_t* aux = R.smem + KSTAGES * M::kStageBytes;
      bf16* dbase = p.out0 + slab_row0 * (size_t)(2 * p.F);
      for (int qt = 0; qt < M::kBN / 64; ++qt) {
        if (!ptx::mbar_wait(&ctl.aux_full, aux_phase, &ctl.abort, kWaitLimitNs)) {
          if (lane == 0) flag_timeout(ctl, p.status, 6);
          return false;
        }
        aux_phase ^= 1;
        const int cc = 2 * qt + hf;  // chunk within the tile
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(tbase + 32 * cc, v);
        const int cb = hf * 4;
        uint4 gc[4], uc[4];
#pragma unroll
        for (int k2 = 0; k2 < 4; ++k2) {
          const int off = r * 128 + (((cb + k2) ^ (r & 7)) * 16);
          gc[k2] = *reinterpret_cast<const uint4*>(aux + off);
          uc[k2] = *reinterpret_cast<const uint4*>(aux + 16384 + off);
        }
        ptx::tmem_ld_wait(v);
        const int f = t.n0 + 32 * cc;
        const bool cols_ok = f < p.F;
        float out[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {  // da_up = dh * silu(a_g)
          const float ag = bf16_at(gc, i);
          out[i] = __uint_as_float(v[i]) * ag * sigmoid_f(ag);
        }
        ptx::mbar_arrive(&ctl.aux_empty);  // the quarter is in registers now
        warp_store32(stage, out, dbase + p.F + f, 2 * p.F, lane, slab_rows, cols_ok);
#pragma unroll
        for (int i = 0; i < 32; ++i) {  // da_gate = dh * a_u * silu'(a_g)
          const float ag = bf16_at(gc, i);
          const float sg = sigmoid_f(ag);
          out[i] = __uint_as_float(v[i]) * bf16_at(uc, i) * sg * (1.f + ag * (1.f - sg));
        }
        warp_store32(stage, out, dbase + f, 2 * p.F, lane, slab_rows, cols_ok);
      }
    } else {
      const int Nd = MODE == GEMM_FC2_FWD || MODE == GEMM_FC1_DGRAD ? p.H : p.F;
      store_chunks(stage, tbase, c0, p.out0 + slab_row0 * (size_t)Nd + t.n0, Nd, t.n0, lane,
                   slab_rows, tmD, M::kStoreDims, t.n0, (int)slab_row0, 0);
    }
  }
  if (tr) trace(p, MODE, ew == 0 ? 5 : 7, ti);
  if (SIGNAL) {
    // this warp's stores of the tile are done: make them visible device-wide
    // before the expert's counter moves
    __threadfence();
    __syncwarp();
    if (lane == 0) {
      __threadfence();
      atomicAdd(p.dep + t.e, 1);
    }
  }
  // one arrival per epilogue warp once all its lanes' TMEM reads are done
  // (in the odd CTA of a pair, on the local barrier its MMA warp forwards)
  ptx::tc_fence_before();
  __syncwarp();
  if (lane == 0)
    ptx::mbar_arrive(M::kPair && R.crank != 0 ? &ctl.epi_done[acc] : &ctl.tmem_empty[acc]);
  if (++acc == 2) {
    acc = 0;
    acc_phase ^= 1;
  }
  return true;
}

// ACC (weight-gradient modes only): add the fp32 tiles into the store map's
// fp32 buffer instead of storing bf16. A template parameter, so that the
// storing kernels do not carry the reduction path's registers.
template <int MODE, int MODE2, bool ACC = false>
__global__ void __launch_bounds__(Fuse<MODE, MODE2>::kWarps * 32, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC,
                        const __grid_constant__ CUtensorMap tmD,
                        const __grid_constant__ CUtensorMap tmA2,
                        const __grid_constant__ CUtensorMap tmB2,
                        const __grid_constant__ CUtensorMap tmC2,
                        const __grid_constant__ CUtensorMap tmD2, const KParams p,
                        const KParams p2) {
  using F = Fuse<MODE, MODE2>;
  constexpr int MODE_B = MODE2 >= 0 ? MODE2 : MODE;
  constexpr int KS = F::kStages;
  static_assert(!ACC || (Mode<MODE>::kRagK && MODE2 < 0), "accumulation is for weight gradients");
  extern __shared__ uint8_t dyn_smem[];
  __shared__ SmemCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) &
                                             ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E;

  // ---- per-CTA setup: barriers, TMEM, then (once the previous kernel on the
  // stream has completed) offsets and the tile prefixes
  if (threadIdx.x == 0) {
    for (int s = 0; s < KS; ++s) {
      ptx::mbar_init(&ctl.full[s], 1);
      // multicast B: every CTA of the cluster releases the stage; pair: the
      // even CTA's MMA releases it in both CTAs
      ptx::mbar_init(&ctl.empty[s], F::kPair ? 1 : F::kCS);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&ctl.tmem_full[b], 1);
      // one arrival per epilogue warp; pair: the even CTA's MMA also waits
      // for the odd CTA's epilogue, reported by one forwarded arrival
      ptx::mbar_init(&ctl.tmem_empty[b], F::kPair ? 9 : 8);
      ptx::mbar_init(&ctl.epi_done[b], 8);
    }
    ptx::mbar_init(&ctl.drain, 1);
    ptx::mbar_init(&ctl.aux_full, 1);
    ptx::mbar_init(&ctl.aux_empty, 256);
    ctl.abort = 0;
    ptx::fence_mbar_init();
  }
  if (F::kPair) {
    // the pair's TMEM is allocated collectively; barriers must be live in both
    __syncthreads();
    ptx::cluster_sync();
    if (warp == 1) {
      ptx::tmem_alloc_pair(&ctl.tmem_base, kTmemCols);
      ptx::tmem_relinquish_pair();
    }
  } else if (warp == 1) {
    ptx::tmem_alloc(&ctl.tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmB);
    if (F::kHas2) {
      ptx::tma_prefetch_desc(&tmA2);
      ptx::tma_prefetch_desc(&tmB2);
    }
  }
  pdl_wait();
  for (int e = threadIdx.x; e <= E; e += blockDim.x) ctl.off[e] = p.off[e];
  __syncthreads();
  if (Mode<MODE>::kRagK) {
    longest_first(ctl.off, E, ctl.order);
    __syncthreads();
  }
  if (warp == 0) {
    tile_prefix<MODE>(p, ctl.off, ctl.order, ctl.tstart, lane);
    if (F::kHas2) tile_prefix<MODE_B>(p2, ctl.off, ctl.order, ctl.tstart2, lane);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  // peers multicast into this CTA's shared memory and barriers: all must be
  // initialised first
  if (F::kCS > 1 && !F::kPair) ptx::cluster_sync();
  const int total1 = ctl.tstart[E];
  const int total = total1 + (F::kHas2 ? ctl.tstart2[E] : 0);
  Role R;
  R.smem = smem;
  R.ctl = &ctl;
  R.tmem_base = ctl.tmem_base;
  R.crank = F::kCS > 1 ? ptx::cluster_ctarank() : 0;
  R.cmask = (uint16_t)((1u << F::kCS) - 1u);
  R.lane = lane;
  const int first = F::kCS > 1 ? (int)ptx::cluster_id_x() : (int)blockIdx.x;
  const int stride = F::kCS > 1 ? (int)ptx::cluster_count_x() : (int)gridDim.x;
  // tile index -> (mode, tile); cursors walk the expert prefixes
  int cur1 = 0, cur2 = 0;
  auto tile1 = [&](int tile) {
    return tile_at<MODE>(p, ctl.tstart, ctl.off, ctl.order, tile, cur1, R.crank);
  };
  auto tile2 = [&](int tile) {
    return tile_at<MODE_B>(p2, ctl.tstart2, ctl.off, ctl.order, tile - total1, cur2, R.crank);
  };

  if (warp == 0) {
    // ================================================================ producer
    int stage = 0;
    uint32_t phase = 0;
    int ti = 0;
    for (int tile = first; tile < total; tile += stride, ++ti) {
      bool ok;
      if (!F::kHas2 || tile < total1) {
        const Tile t = tile1(tile);
        if (lane == 0) trace(p, MODE, 0, ti);
        ok = producer_tile<MODE, KS>(R, p, &tmA, &tmB, t, stage, phase);
      } else {
        const Tile t = tile2(tile);
        // the A operand of this tile is the first mode's output for expert t.e
        ok = true;
        if (F::kDep && lane == 0) {
          const int target = 8 * F::kCS * (ctl.tstart[t.e + 1] - ctl.tstart[t.e]);
          ok = wait_expert(p, t.e, target, &ctl.abort);
          if (!ok) flag_timeout(ctl, p.status, 10);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (ok) ok = producer_tile<MODE_B, KS>(R, p2, &tmA2, &tmB2, t, stage, phase);
      }
      if (lane == 0) trace(p, MODE, 1, ti);
      if (!ok) break;
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    // (pair mode: only the even CTA issues, for both CTAs)
    // (K-ragged launches: the whole warp, which zeroes the tail rows of A)
    constexpr bool kWarpMma = Mode<MODE>::kRagK;
    if ((kWarpMma || lane == 0) && !(F::kPair && R.crank != 0)) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      int ti = -1;
      for (int tile = first; tile < total; tile += stride) {
        ++ti;
        bool ok;
        if (!F::kHas2 || tile < total1)
          ok = mma_tile<MODE, KS>(R, p, tile1(tile), stage, phase, acc, acc_phase, ti);
        else
          ok = mma_tile<MODE_B, KS>(R, p2, tile2(tile), stage, phase, acc, acc_phase, ti);
        if (!ok) break;
      }
      // make sure no MMA is still running before TMEM is released
      if (lane == 0) {
        if (F::kPair) ptx::umma_commit_pair(&ctl.drain, 1);
        else ptx::umma_commit(&ctl.drain);
      }
      if (!ptx::mbar_wait(&ctl.drain, 0, &ctl.abort, kWaitLimitNs)) {
        // abort already flagged: wait once more with the abort flag ignored
        int dummy = 0;
        ptx::mbar_wait(&ctl.drain, 0, &dummy, kWaitLimitNs);
      }
    } else if (lane == 0 && F::kPair) {
      // odd CTA of a pair: forward "accumulator free" to the even CTA's MMA
      // issuer, one cluster arrival per tile once all 8 epilogue warps have
      // arrived locally (fewer cluster-scope arrivals than one per warp).
      int acc = 0;
      uint32_t acc_phase = 0;
      for (int tile = first; tile < total; tile += stride) {
        const Tile t = (!F::kHas2 || tile < total1) ? tile1(tile) : tile2(tile);
        if (t.nk == 0) continue;
        if (!ptx::mbar_wait(&ctl.epi_done[acc], acc_phase, &ctl.abort, kWaitLimitNs)) {
          flag_timeout(ctl, p.status, 9);
          break;
        }
        ptx::mbar_arrive_cluster(ptx::mapa_shared(&ctl.tmem_empty[acc], 0));
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
    }
    __syncwarp();
  } else if (F::kAux && warp == 10) {
    // ================================================================ aux loader
    if (lane == 0) {
      ptx::tma_prefetch_desc(Mode<MODE>::kAux ? &tmC : &tmC2);
      uint32_t ph = 0;
      for (int tile = first; tile < total; tile += stride) {
        bool ok = true;
        if (!F::kHas2 || tile < total1) {
          const Tile t = tile1(tile);
          if (Mode<MODE>::kAux) ok = aux_tile<MODE, KS>(R, p, &tmC, t, ph);
        } else {
          const Tile t = tile2(tile);
          if (Mode<MODE_B>::kAux) ok = aux_tile<MODE_B, KS>(R, p2, &tmC2, t, ph);
        }
        if (!ok) break;
      }
    }
    __syncwarp();
  } else {
    // ================================================================ epilogue
    // 8 warps: warp w reads TMEM lane quarter w % 4 (hardware rule) and owns
    // half of the tile's columns.
    const int ew = warp - 2;
    int acc = 0;
    uint32_t acc_phase = 0, aux_phase = 0;
    int ti = -1;
    for (int tile = first; tile < total; tile += stride) {
      ++ti;
      bool ok;
      if (!F::kHas2 || tile < total1)
        ok = epilogue_tile<MODE, KS, F::kAuxBytes, F::kDep, ACC>(R, p, &tmD, tile1(tile), acc,
                                                               acc_phase, aux_phase, ew, ti);
      else
        ok = epilogue_tile<MODE_B, KS, F::kAuxBytes, false, false>(R, p2, &tmD2, tile2(tile), acc,
                                                             acc_phase, aux_phase, ew, ti);
      if (!ok) break;
    }
    // the staging buffers and the outputs must outlive the TMA stores
    if (F::kStores && lane == 0) ptx::bulk_wait_group0();
    __syncwarp();
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  // peers may still arrive on this CTA's barriers until they are done
  if (F::kCS > 1) ptx::cluster_sync();
  if (warp == 1) {
    if (F::kPair) ptx::tmem_dealloc_pair(R.tmem_base, kTmemCols);
    else ptx::tmem_dealloc(R.tmem_base, kTmemCols);
  }
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

// Store map of an output: 2D [rows, cols] or 3D [experts, rows, cols],
// row-major. bf16: boxes of 32 rows x 32 columns (x 1 expert), 64-byte
// swizzle, the staging buffer's layout: 16-byte chunk c of row r at chunk
// c ^ ((r >> 1) & 3). fp32 (f32, the accumulated weight gradients): boxes of
// 16 rows x 32 columns, 128-byte swizzle, chunk c of row r at c ^ (r & 7).
bool make_store_map(CUtensorMap* m, void* base, long long experts, long long rows, long long cols,
                    int dims, bool f32 = false) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return false;
  }
  const int es_bytes = f32 ? 4 : 2;
  cuuint64_t dim[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)experts};
  cuuint64_t strides[2] = {(cuuint64_t)cols * es_bytes, (cuuint64_t)(rows * cols * es_bytes)};
  cuuint32_t box[3] = {32, (cuuint32_t)(f32 ? 16 : 32), 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                   dims, base, dim, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE,
                   f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (%d) for a %lld x %lld x %lld store map", (int)r,
              experts, rows, cols);
    return false;
  }
  return true;
}

template <int MODE, int MODE2, bool ACC = false>
moe_status_t launch_mode(const CUtensorMap (&m1)[4], const CUtensorMap (&m2)[4], const KParams& p,
                         const KParams& p2, int grid, int kernel_id, cudaStream_t st) {
  using F = Fuse<MODE, MODE2>;
  constexpr int cs = F::kCS;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  static int max_clusters = 0;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(grouped_gemm_kernel<MODE, MODE2, ACC>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)F::kDynSmem);
    if (attr_err == cudaSuccess && cs > 1) {
      // how many clusters of cs CTAs (one per SM) can be resident at once
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = cs;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(device_sm_count() / cs * cs);
      cfg.blockDim = dim3(F::kWarps * 32);
      cfg.dynamicSmemBytes = F::kDynSmem;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      attr_err = cudaOccupancyMaxActiveClusters(&max_clusters, grouped_gemm_kernel<MODE, MODE2, ACC>,
                                                &cfg);
    }
  });
  if (attr_err != cudaSuccess) {
    set_error("kernel attribute setup failed: %s", cudaGetErrorString(attr_err));
    return MOE_ERR_CUDA;
  }
  LaunchScope _ls(kernel_id, st);
  if (cs == 1) {
    launch_k(grouped_gemm_kernel<MODE, MODE2, ACC>, grid, F::kWarps * 32, F::kDynSmem, st, m1[0],
             m1[1], m1[2], m1[3], m2[0], m2[1], m2[2], m2[3], p, p2);
    return check_launch("grouped_gemm_kernel");
  }
  // a fused launch relies on every CTA being resident at once (second-mode
  // tiles wait on first-mode tiles of other CTAs): never more clusters than fit
  int clusters = (grid + cs - 1) / cs;
  if (max_clusters > 0 && clusters > max_clusters) clusters = max_clusters;
  if (clusters < 1) clusters = 1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = cs;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = MOE_PDL;
  cfg.gridDim = dim3(clusters * cs);
  cfg.blockDim = dim3(F::kWarps * 32);
  cfg.dynamicSmemBytes = F::kDynSmem;
  cfg.stream = st;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<MODE, MODE2, ACC>, m1[0], m1[1], m1[2],
                                     m1[3], m2[0], m2[1], m2[2], m2[3], p, p2);
  if (e != cudaSuccess) {
    set_error("grouped_gemm_kernel cluster launch: %s", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  return check_launch("grouped_gemm_kernel");
}

// Tensor maps (A, B, aux, store), kernel parameters and an upper bound on the
// tiles of one mode.
bool mode_setup(const moe_layer_desc_t& d, const GemmArgs& g, CUtensorMap (&m)[4], KParams& p,
                long long& ntile_bound) {
  const long long N = (long long)d.T * d.k;
  const int E = d.E, H = d.H, F = d.F;
  bool ok = true;
  switch (g.mode) {
    case GEMM_FC1_FWD:
      ok = make_map(&m[0], g.A, N, H, 128) && make_map(&m[1], g.B, (long long)E * 2 * F, H, 128);
      ntile_bound = (N / BM + 2 * E) * ((F + 127) / 128);
      break;
    case GEMM_FC2_FWD:
      ok = make_map(&m[0], g.A, N, F, 128) && make_map(&m[1], g.B, (long long)E * H, F, 128);
      ntile_bound = (N / BM + 2 * E) * ((H + BN - 1) / BN);
      break;
    case GEMM_FC2_DGRAD:
      ok = make_map(&m[0], g.A, N, H, 128) && make_map(&m[1], g.B, (long long)E * H, F, 64) &&
           make_map(&m[2], g.aux, N, 2 * F, 128);
      ntile_bound = (N / BM + 2 * E) * ((F + 127) / 128);
      break;
    case GEMM_FC1_DGRAD:
      ok = make_map(&m[0], g.A, N, 2 * F, 128) && make_map(&m[1], g.B, (long long)E * 2 * F, H, 64);
      ntile_bound = (N / BM + 2 * E) * ((H + BN - 1) / BN);
      break;
    case GEMM_WGRAD_W1:
      ok = make_map(&m[0], g.A, N, 2 * F, 64) && make_map(&m[1], g.B, N, H, 64);
      ntile_bound = (long long)E * ceil_div(ceil_div(2 * F, BM), Mode<GEMM_WGRAD_W1>::kCS) *
                    Mode<GEMM_WGRAD_W1>::kCS * ((H + BN - 1) / BN);
      break;
    case GEMM_WGRAD_W2:
      ok = make_map(&m[0], g.A, N, H, 64) && make_map(&m[1], g.B, N, F, 64);
      ntile_bound = (long long)E * ceil_div(ceil_div(H, BM), Mode<GEMM_WGRAD_W2>::kCS) *
                    Mode<GEMM_WGRAD_W2>::kCS * ((F + BN - 1) / BN);
      break;
    default:
      set_error("unknown grouped GEMM mode %d", g.mode);
      return false;
  }
  if (!ok) return false;
  if (g.mode != GEMM_FC2_DGRAD) m[2] = m[0];  // only FC2 dgrad reads a third tensor
  switch (g.mode) {  // the outputs written by TMA stores
    case GEMM_FC2_FWD:
    case GEMM_FC1_DGRAD: ok = make_store_map(&m[3], g.out0, 1, N, H, 2); break;
    case GEMM_WGRAD_W1:
      ok = g.acc ? make_store_map(&m[3], g.acc, E, 2 * F, H, 3, true)
                 : make_store_map(&m[3], g.out0, E, 2 * F, H, 3);
      break;
    case GEMM_WGRAD_W2:
      ok = g.acc ? make_store_map(&m[3], g.acc, E, H, F, 3, true)
                 : make_store_map(&m[3], g.out1, E, H, F, 3);
      break;
    default: m[3] = m[0];
  }
  if (!ok) return false;
  p.E = E;
  p.H = H;
  p.F = F;
  p.N = N;
  p.off = g.off;
  p.out0 = g.out0;
  p.out1 = g.out1;
  p.aux = g.aux;
  p.status = g.status;
  p.dep = g.dep;
  return true;
}

int grid_for(const GemmArgs& g, long long ntile_bound) {
  int grid = device_sm_count();
  if (g.max_ctas > 0 && g.max_ctas < grid) grid = g.max_ctas;
  if (ntile_bound < grid) grid = (int)(ntile_bound > 0 ? ntile_bound : 1);
  return grid;
}

}  // namespace

moe_status_t launch_grouped_gemm(const moe_layer_desc_t& d, const GemmArgs& g, cudaStream_t st) {
  const long long N = (long long)d.T * d.k;
  const int E = d.E, H = d.H, F = d.F;
  if (N == 0) {
    if (g.acc) return MOE_OK;  // accumulating nothing
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
  CUtensorMap m[4];
  KParams p;
  long long ntile_bound = 0;  // upper bound on tiles, for the grid size
  if (!mode_setup(d, g, m, p, ntile_bound))
    return g.mode > GEMM_WGRAD_W2 ? MOE_ERR_INVALID_ARG : MOE_ERR_CUDA;
  const int grid = grid_for(g, ntile_bound);
  const int id = K_GEMM_FC1_FWD + g.mode;
  switch (g.mode) {
    case GEMM_FC1_FWD: return launch_mode<GEMM_FC1_FWD, -1>(m, m, p, p, grid, id, st);
    case GEMM_FC2_FWD: return launch_mode<GEMM_FC2_FWD, -1>(m, m, p, p, grid, id, st);
    case GEMM_FC2_DGRAD: return launch_mode<GEMM_FC2_DGRAD, -1>(m, m, p, p, grid, id, st);
    case GEMM_FC1_DGRAD: return launch_mode<GEMM_FC1_DGRAD, -1>(m, m, p, p, grid, id, st);
    case GEMM_WGRAD_W1:
      return g.acc ? launch_mode<GEMM_WGRAD_W1, -1, true>(m, m, p, p, grid, K_GEMM_WGRAD_W1_ACC, st)
                   : launch_mode<GEMM_WGRAD_W1, -1>(m, m, p, p, grid, id, st);
    default:
      return g.acc ? launch_mode<GEMM_WGRAD_W2, -1, true>(m, m, p, p, grid, K_GEMM_WGRAD_W2_ACC, st)
                   : launch_mode<GEMM_WGRAD_W2, -1>(m, m, p, p, grid, id, st);
  }
}

moe_status_t launch_grouped_gemm_chain(const moe_layer_desc_t& d, const GemmArgs& g1,
                                       const GemmArgs& g2, cudaStream_t st,
                                       bool counters_zeroed) {
  const long long N = (long long)d.T * d.k;
  if (N == 0) return MOE_OK;
  const bool fwd = g1.mode == GEMM_FC1_FWD && g2.mode == GEMM_FC2_FWD;
  const bool dgrad = g1.mode == GEMM_FC2_DGRAD && g2.mode == GEMM_FC1_DGRAD;
  const bool wgrad = g1.mode == GEMM_WGRAD_W1 && g2.mode == GEMM_WGRAD_W2 && !g1.acc && !g2.acc;
  if (!fwd && !dgrad && !wgrad) {
    set_error("unsupported grouped GEMM chain %d -> %d", g1.mode, g2.mode);
    return MOE_ERR_INVALID_ARG;
  }
  CUtensorMap m1[4], m2[4];
  KParams p1, p2;
  long long b1 = 0, b2 = 0;
  if (wgrad) {
    // two independent weight gradients: W2's tiles fill W1's last round
    if (!mode_setup(d, g1, m1, p1, b1) || !mode_setup(d, g2, m2, p2, b2)) return MOE_ERR_CUDA;
    return launch_mode<GEMM_WGRAD_W1, GEMM_WGRAD_W2>(m1, m2, p1, p2, grid_for(g1, b1 + b2),
                                                     K_GEMM_WGRAD, st);
  }
  if (!g1.dep) {
    set_error("a grouped GEMM chain needs its per-expert counters");
    return MOE_ERR_INVALID_ARG;
  }
  if (!mode_setup(d, g1, m1, p1, b1) || !mode_setup(d, g2, m2, p2, b2)) return MOE_ERR_CUDA;
  p2.dep = p1.dep;
  // the counters start at zero for every launch: cleared here unless the
  // launch just before on the stream has done it
  if (!counters_zeroed) {
    cudaError_t e = cudaMemsetAsync(g1.dep, 0, (size_t)d.E * sizeof(int), st);
    if (e != cudaSuccess) {
      set_error("cudaMemsetAsync: %s", cudaGetErrorString(e));
      return MOE_ERR_CUDA;
    }
  }
  const int grid = grid_for(g1, b1 + b2);
  if (fwd)
    return launch_mode<GEMM_FC1_FWD, GEMM_FC2_FWD>(m1, m2, p1, p2, grid, K_GEMM_FFN_FWD, st);
  return launch_mode<GEMM_FC2_DGRAD, GEMM_FC1_DGRAD>(m1, m2, p1, p2, grid, K_GEMM_FFN_DGRAD, st);
}

}  // namespace moe
