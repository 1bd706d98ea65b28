/*
 * moe.h -- C ABI of a GB300 (sm_103a) MoE layer hot path: router softmax/top-k,
 * dispatch layout, permute into the expert-parallel send layout, grouped SwiGLU
 * expert FFN on tcgen05 tensor cores, gate-weighted combine, and the backward
 * split into activation-gradient (dgrad) and weight-gradient (wgrad) calls so
 * the wgrad can be deferred.
 *
 * Where the operations come from.
 *   - The phases dispatch -> mlp -> combine and the backward chain
 *     combine -> mlp -> dispatch: the "1. MoE EP Overlap" note (obnotes),
 *     section "how the 8 fwd/bwd operations are split out".
 *   - The dgrad-first / wgrad-later split and the deferral (delay_wgrad_compute):
 *     same note, section "MoE 1F1B overlap"; the MoE expert-parallel overlap
 *     skill card, section "what it is".
 *   - The standard all-to-all dispatcher whose send buffer the permute writes:
 *     skill card, "what it is", dispatcher table.
 *   - Two streams and two micro-batches overlapping dispatch/combine with the
 *     expert GEMMs: the note, section "MoE 1F1B overlap".
 *   The pages give no formulas. The arithmetic is the layer definition stated
 *   per function below (fp32 logits, softmax, top-k, renormalised gates,
 *   SwiGLU experts, gate-weighted combine).
 *
 * Conventions for every call.
 *   - Pointers are device pointers unless a name starts with host_. bf16 data is
 *     passed as moe_bf16 (the raw 16-bit pattern). Matrices are row-major.
 *   - The caller allocates and owns every buffer, including the workspace whose
 *     size moe_workspace_size() returns. No call allocates or frees device memory.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Calls only
 *     enqueue work on it; none synchronises the host, except moe_device_status()
 *     and moe_layer_step_host(), which say so.
 *   - Host-side argument checks return MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED
 *     synchronously, before anything is enqueued; moe_last_error() then holds
 *     a message (thread-local). A failed launch gives MOE_ERR_CUDA.
 *   - Device-side checks (an expert index out of range, a pipeline wait that
 *     ran out of time) never trap: the kernel records a code in the workspace's
 *     status words, skips the access, and returns; moe_device_status() reads it.
 *   - Shapes: T >= 0 tokens, H hidden, E experts, k top-k, F expert inner size,
 *     R emulated expert-parallel ranks. N = T*k routed rows (dropless).
 *     Limits: 1 <= E <= 256, 1 <= k <= min(E, 32), E % R == 0, H % 64 == 0,
 *     F % 64 == 0, H <= 16384, F <= 16384, T*k < 2^31.
 *   - Every device pointer must be 16-byte aligned.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16; /* bfloat16 bit pattern */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,
  MOE_ERR_UNSUPPORTED = 2,
  MOE_ERR_CUDA = 3,
  MOE_ERR_TIMEOUT = 4
} moe_status_t;

typedef enum {
  MOE_ROUTE_SOFTMAX_TOPK = 0,   /* top-k experts by logit, ties to the lower index */
  MOE_ROUTE_FORCED_BALANCED = 1 /* token t -> experts (k*t + j) mod E, j = 0..k-1 */
} moe_route_mode_t;

/* Layer flags (moe_layer_desc_t.flags, 0 or a bitwise or of these).
 *
 * MOE_FLAG_WGRAD_ACCUM_FP32: the layer calls (moe_layer_backward,
 * moe_layer_step_host, moe_sched_step) add the expert weight gradients into the
 * fp32 main gradients b->main_dw1 / b->main_dw2 instead of overwriting the bf16
 * b->dw1 / b->dw2 (which may then be NULL). This is gradient accumulation
 * fusion: the MoE expert-parallel overlap skill card, section "compatibility
 * and constraints" and its troubleshooting table (delay_wgrad_compute with
 * gradient_accumulation_fusion), and the "1. MoE EP Overlap" note's backward
 * call with accumulate_grad=True (gradients add into .grad instead of
 * overwriting it). See moe_expert_ffn_bwd_wgrad_accum for the arithmetic. */
#define MOE_FLAG_WGRAD_ACCUM_FP32 1

/* One MoE layer's shape. flags: 0 or MOE_FLAG_* bits. */
typedef struct moe_layer_desc {
  int32_t T, H, E, k, F, R;
  int32_t mode;  /* moe_route_mode_t */
  int32_t flags;
} moe_layer_desc_t;

/* ------------------------------------------------------------------ setup */

/* Checks a descriptor against the limits above. */
moe_status_t moe_layer_desc_validate(const moe_layer_desc_t* d);

/* Bytes of device workspace every call of this layer shape needs (0 on an
 * invalid descriptor). One workspace may be shared by calls on one stream; calls
 * that can overlap on the GPU need workspaces of their own. */
size_t moe_workspace_size(const moe_layer_desc_t* d);

/* Message of the last error on this host thread ("" if none). */
const char* moe_last_error(void);

/* Library ABI version (increments on incompatible changes). */
int32_t moe_abi_version(void);

/* Synchronises `stream`, reads the workspace's device status words and clears
 * them. MOE_OK, MOE_ERR_INVALID_ARG (a kernel met an out-of-range index and
 * skipped it) or MOE_ERR_TIMEOUT (a pipeline wait ran out of time). */
moe_status_t moe_device_status(const moe_layer_desc_t* d, void* ws, void* stream);

/* ------------------------------------------------------------------ diagnostics */

/* Sets the time limit of the grid-barrier waits in moe_dispatch_fused (and in
 * the layer forward, which uses it) for launches enqueued after this call,
 * process-wide; ns = 0 restores the default of 2 s. Returns the previous
 * limit. A graph capture keeps the limit in force at capture time. This is a
 * diagnostic: with a limit shorter than the blocks take to reach a barrier,
 * waiting blocks give up, record MOE_ERR_TIMEOUT in the workspace status and
 * return, leaving the call's outputs incomplete; the next launch starts
 * clean. It lets a caller check its handling of a device-side timeout without
 * any wait that cannot end. */
uint64_t moe_set_barrier_wait_limit_ns(uint64_t ns);

/* Number of kernels this library has launched in the process so far (a graph
 * replay counts its kernel nodes; a capture counts nothing). */
uint64_t moe_kernel_launches(void);

/* Name of kernel id `kernel` as reported by moe_profile_stop ("" if unknown). */
const char* moe_kernel_name(int32_t kernel);

typedef struct moe_kernel_time {
  int32_t kernel; /* kernel id, see moe_kernel_name() */
  float ms;       /* duration between events recorded just before and after the
                     launch on the launch's own stream */
} moe_kernel_time_t;

/* Starts recording per-launch durations of the next `capacity` launches (on any
 * stream). Creates CUDA events on first use; allocates no device memory.
 * While recording, moe_layer_backward runs the weight gradients in order on
 * its `stream` after the dispatch backward, instead of beside it on the side
 * stream, so that each launch is timed alone. */
moe_status_t moe_profile_start(int32_t capacity);

/* Stops recording, waits for the recorded events and returns up to cap entries
 * in launch order; *n receives the count. */
moe_status_t moe_profile_stop(moe_kernel_time_t* out, int32_t cap, int32_t* n);

/* ------------------------------------------------------------------ forward */

/* Router (the "router" scope ahead of dispatch). For each token t:
 *   z[t,e] = sum_{h=0..H-1} x[t,h] * w_r[e,h] in fp32, h ascending from 0
 *            (bf16*bf16 is exact in fp32, so each step is one fp32 rounding),
 *            plus bias[e] in fp32 when bias != NULL;
 *   p = softmax(z[t,:]) over all E;
 *   SOFTMAX_TOPK: idx[t,0..k-1] = the k largest z, descending, ties to the
 *                 lower expert index;
 *   FORCED_BALANCED: idx[t,j] = (k*t + j) mod E;
 *   gates[t,j] = p[idx[t,j]] / sum_l p[idx[t,l]].
 * x [T,H] bf16, w_r [E,H] bf16, bias [E] fp32 or NULL, logits [T,E] fp32 or NULL
 * (written when given), idx [T,k] int32, gates [T,k] fp32. */
moe_status_t moe_route(const moe_layer_desc_t* d, const moe_bf16* x, const moe_bf16* w_r,
                       const float* bias, float* logits, int32_t* idx, float* gates,
                       void* ws, size_t ws_bytes, void* stream);

/* Dispatch layout (the preprocessing ahead of the all-to-all): dropless, stable.
 *   cnt[e]      = #{(t,j) : idx[t,j] = e}
 *   off[0..E]   = exclusive prefix sum of cnt (off[E] = N)
 *   slot[t,j]   = off[e] + #{t' < t : e in idx[t',:]}   (e = idx[t,j])
 *   row_src[s]  = t*k + j for s = slot[t,j]
 *   cnt_re[r,l] = cnt[r*E/R + l]      rows per (destination rank, local expert)
 *   rank_off[r] = off[r*E/R], r = 0..R (first row of each rank's chunk)
 * With rank(e) = e div (E/R) the expert-ordered buffer is the rank-major,
 * expert-contiguous send buffer an EP all-to-all exchanges, and these tables
 * are the counts it exchanges first. Every token must pick k distinct experts.
 * idx [T,k]; cnt [E]; off [E+1]; slot [T,k]; row_src [N]; cnt_re [R,E/R];
 * rank_off [R+1]; all int32. */
moe_status_t moe_dispatch_layout(const moe_layer_desc_t* d, const int32_t* idx, int32_t* cnt,
                                 int32_t* off, int32_t* slot, int32_t* row_src,
                                 int32_t* cnt_re, int32_t* rank_off, void* ws, size_t ws_bytes,
                                 void* stream);

/* The same dispatch layout for callers that cannot allocate device memory:
 * a plugin that receives only its input and output tensors from a host
 * framework that owns the allocator, code recorded into a CUDA graph (where
 * cudaMalloc is not allowed while the stream is being captured), or a path
 * that must not block on allocator locks. Instead of a caller workspace it
 * uses a fixed scratch array inside the library's device memory, sized for at
 * most T = 65536 tokens and E = 256 experts (257 KB plus 256 bytes, held on
 * every GPU that loads the library until the process exits); larger shapes
 * return MOE_ERR_UNSUPPORTED. The pages describe no such call; it exists for
 * these callers only. Each call made outside stream capture looks up the
 * scratch array's device address on the current device (so a reloaded module
 * or another context of the device is followed); a call made while `stream`
 * is capturing reuses the address the last such lookup found on that device,
 * so make the first call on each device before any stream capture (a captured
 * first call returns MOE_ERR_INVALID_ARG). All calls share the one array:
 * calls whose GPU work can overlap (unordered streams) race and must not be
 * issued; calls on one stream are safe. Out-of-range expert indices are
 * skipped (slot = -1, and the entry has no row in row_src, so off[E] < T*k)
 * and counted in the array's status words, which the call clears at its
 * start: moe_dispatch_layout_static_status() reports them until the next call.
 * Outputs and argument meaning as for moe_dispatch_layout. Allocates nothing. */
moe_status_t moe_dispatch_layout_static(const moe_layer_desc_t* d, const int32_t* idx,
                                        int32_t* cnt, int32_t* off, int32_t* slot,
                                        int32_t* row_src, int32_t* cnt_re, int32_t* rank_off,
                                        void* stream);

/* Status of the last moe_dispatch_layout_static call on the current device:
 * synchronises `stream` (the stream that call used; not while it is
 * capturing), reads the scratch array's status words and clears them.
 * MOE_OK, or MOE_ERR_INVALID_ARG when that call skipped out-of-range expert
 * indices (moe_last_error() gives how many). Allocates nothing. Like the
 * layout call it reads the one shared array, so a layout call enqueued in
 * between on another stream would be what it reports. The pages describe no
 * such call; it completes moe_dispatch_layout_static. */
moe_status_t moe_dispatch_layout_static_status(void* stream);

/* Permute = write the EP send buffer: x_perm[s,:] = x[row_src[s] div k, :].
 * x [T,H] bf16, row_src [N] int32, x_perm [N,H] bf16. */
moe_status_t moe_permute(const moe_layer_desc_t* d, const moe_bf16* x, const int32_t* row_src,
                         moe_bf16* x_perm, void* stream);

/* Route + dispatch layout + permute in one call, with the results of moe_route,
 * moe_dispatch_layout and moe_permute run in that order (the same bits). With
 * E <= 128 it is one cooperative persistent launch (the fused dispatch of the
 * skill card: moe_permute_fusion, "HybridEP production benchmark"):
 *   - blocks route their token tiles and count each tile's entries per expert;
 *   - after a grid-wide barrier, each expert's counts are scanned over tiles;
 *   - after a second barrier, every block derives the expert offsets, numbers
 *     its own entries in token order, and copies its tokens' rows into x_perm.
 * The barrier waits are bounded (2 s by default, see
 * moe_set_barrier_wait_limit_ns). On expiry the waiting block records the
 * site, returns without writing the rest of its outputs, and the device status
 * reads MOE_ERR_TIMEOUT. Every block is resident by the launch's construction,
 * so with the default limit the waits end. With E > 128 or T = 0 the three
 * calls run as separate launches.
 * x [T,H], w_r [E,H] bf16; bias [E] fp32 or NULL; logits [T,E] fp32 or NULL
 * -> idx, gates [T,k]; cnt [E]; off [E+1]; slot [T,k]; row_src [N];
 * cnt_re [R,E/R]; rank_off [R+1]; x_perm [N,H] bf16. */
moe_status_t moe_dispatch_fused(const moe_layer_desc_t* d, const moe_bf16* x, const moe_bf16* w_r,
                                const float* bias, float* logits, int32_t* idx, float* gates,
                                int32_t* cnt, int32_t* off, int32_t* slot, int32_t* row_src,
                                int32_t* cnt_re, int32_t* rank_off, moe_bf16* x_perm, void* ws,
                                size_t ws_bytes, void* stream);

/* Expert FFN forward (the "mlp" phase), per expert e on its rows off[e]..off[e+1]-1:
 *   a = bf16(x_perm_e @ w1[e]^T)               [rows, 2F], fp32 accumulate
 *   h = bf16(silu(a[:, :F]) * a[:, F:])        [rows, F] (from the bf16 a)
 *   o = bf16(h @ w2[e]^T)                      [rows, H]
 * w1 [E,2F,H] bf16 (rows 0..F-1 gate, F..2F-1 up), w2 [E,H,F] bf16, off [E+1]
 * int32 on the device (read by the kernels' tile schedulers; never by the host).
 * a [N,2F], h [N,F], o [N,H] bf16; a and h are kept for the backward. */
moe_status_t moe_expert_ffn_fwd(const moe_layer_desc_t* d, const moe_bf16* x_perm,
                                const int32_t* off, const moe_bf16* w1, const moe_bf16* w2,
                                moe_bf16* a, moe_bf16* h, moe_bf16* o, void* ws, size_t ws_bytes,
                                void* stream);

/* Combine = receive + unpermute (the "combine" phase):
 *   y[t,:] = bf16( sum_{j=0..k-1} gates[t,j] * o[slot[t,j], :] ), fp32, j ascending.
 * o [N,H] bf16, slot [T,k] int32, gates [T,k] fp32, y [T,H] bf16. */
moe_status_t moe_combine(const moe_layer_desc_t* d, const moe_bf16* o, const int32_t* slot,
                         const float* gates, moe_bf16* y, void* stream);

/* ------------------------------------------------------------------ backward */

/* Combine backward (first step of the backward chain):
 *   d_o[slot[t,j], :] = bf16(gates[t,j] * dy[t,:])
 *   dgates[t,j]       = sum_h dy[t,h] * o[slot[t,j], h]   (fp32)
 * dy [T,H] bf16, o [N,H] bf16, slot [T,k], gates [T,k] fp32 -> d_o [N,H] bf16,
 * dgates [T,k] fp32. */
moe_status_t moe_combine_bwd(const moe_layer_desc_t* d, const moe_bf16* dy, const moe_bf16* o,
                             const int32_t* slot, const float* gates, moe_bf16* d_o,
                             float* dgates, void* stream);

/* Expert FFN activation gradient (dgrad; runs before wgrad so dispatch-backward
 * can start early), per expert e on its rows:
 *   dh      = d_o_e @ w2[e]                          (fp32, not stored)
 *   da_up   = bf16(dh * silu(a_g))
 *   da_gate = bf16(dh * a_u * s(a_g) * (1 + a_g * (1 - s(a_g))))   s = sigmoid
 *   dx_perm = bf16(da_e @ w1[e])
 * d_o [N,H], a [N,2F] -> da [N,2F] (kept for wgrad), dx_perm [N,H]; bf16. */
moe_status_t moe_expert_ffn_bwd_dgrad(const moe_layer_desc_t* d, const moe_bf16* d_o,
                                      const moe_bf16* a, const int32_t* off, const moe_bf16* w1,
                                      const moe_bf16* w2, moe_bf16* da, moe_bf16* dx_perm,
                                      void* ws, size_t ws_bytes, void* stream);

/* Expert FFN weight gradient (wgrad; may be deferred, delay_wgrad_compute):
 *   dw1[e] = bf16(da_e^T @ x_perm_e)   [2F,H]
 *   dw2[e] = bf16(d_o_e^T @ h_e)       [H,F]
 * The reduction runs over the expert's own rows only; an expert with no rows
 * gets zeros. Overwrites dw1 [E,2F,H] and dw2 [E,H,F] (bf16). */
moe_status_t moe_expert_ffn_bwd_wgrad(const moe_layer_desc_t* d, const moe_bf16* x_perm,
                                      const moe_bf16* h, const moe_bf16* d_o, const moe_bf16* da,
                                      const int32_t* off, moe_bf16* dw1, moe_bf16* dw2, void* ws,
                                      size_t ws_bytes, void* stream);

/* Expert FFN weight gradient accumulated into fp32 main gradients (gradient
 * accumulation fusion, see MOE_FLAG_WGRAD_ACCUM_FP32):
 *   main_dw1[e] = fl32(main_dw1[e] + (da_e^T @ x_perm_e))   [2F,H]
 *   main_dw2[e] = fl32(main_dw2[e] + (d_o_e^T @ h_e))       [H,F]
 * The product is reduced in fp32 over the expert's rows (one tensor-core
 * accumulator per output tile) and added with one fp32 addition per element,
 * so repeated calls accumulate micro-batch after micro-batch in call order.
 * An expert with no rows adds nothing. main_dw1 [E,2F,H] and main_dw2 [E,H,F]
 * are fp32, read and written in place; the other arguments are as for
 * moe_expert_ffn_bwd_wgrad. The call does not look at d->flags. */
moe_status_t moe_expert_ffn_bwd_wgrad_accum(const moe_layer_desc_t* d, const moe_bf16* x_perm,
                                            const moe_bf16* h, const moe_bf16* d_o,
                                            const moe_bf16* da, const int32_t* off,
                                            float* main_dw1, float* main_dw2, void* ws,
                                            size_t ws_bytes, void* stream);

/* Permute backward (dispatch backward): dx32[t,:] = sum_j dx_perm[slot[t,j], :]
 * in fp32, j ascending. dx_perm [N,H] bf16, slot [T,k] -> dx32 [T,H] fp32. */
moe_status_t moe_permute_bwd(const moe_layer_desc_t* d, const moe_bf16* dx_perm,
                             const int32_t* slot, float* dx32, void* stream);

/* Router backward through the renormalised gates (softmax over the chosen set S):
 *   dz[t,i_j] = g_j * (dgates_j - sum_l g_l dgates_l), dz = 0 off S
 *   dx[t,:]   = bf16(dx32[t,:] + sum_j dz[t,i_j] * w_r[i_j,:])
 *   dw_r[e,:] = sum_{t : e in S_t} dz[t,e] * x[t,:]    (fp32, rows of e in layout order)
 * dgates, gates [T,k] fp32; idx [T,k]; x [T,H] bf16; w_r [E,H] bf16; row_src [N],
 * off [E+1] from the layout; dx32 [T,H] fp32 (from moe_permute_bwd);
 * -> dx [T,H] bf16, dw_r [E,H] fp32 (overwritten). */
moe_status_t moe_route_bwd(const moe_layer_desc_t* d, const float* dgates, const float* gates,
                           const int32_t* idx, const moe_bf16* x, const moe_bf16* w_r,
                           const int32_t* row_src, const int32_t* off, const float* dx32,
                           moe_bf16* dx, float* dw_r, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------ expert parallelism */

/* Receive re-sort of the expert-parallel exchange (the standard all-to-all
 * dispatcher: the MoE expert-parallel overlap skill card, section "what it
 * is", dispatcher table; EP16 in its benchmark sections). With R = d->R ranks,
 * each owning E_l = d->E / R experts (rank d owns experts d*E_l..(d+1)*E_l-1),
 * a rank receives from sources s = 0..R-1, in that order, recv_cnt[s][l]
 * rows for each of its local experts l = 0..E_l-1: the chunk rows
 * rank_off[d]..rank_off[d+1]-1 of source s's send buffer, whose counts are
 * that source's cnt_re[d][:] (see moe_dispatch_layout). That is "receive
 * order". The grouped GEMM wants "expert-major" order: expert l's rows
 * contiguous, sources ascending inside it, each source's own order kept.
 *   inverse = 0: out (expert-major) <- in (receive order); also writes
 *                off_local[l] = first row of local expert l, off_local[E_l] =
 *                total (the off[] the expert calls take for E = E_l);
 *   inverse = 1: out (receive order) <- in (expert-major), the order the
 *                return exchange sends o and dx_perm back in.
 * recv_cnt [R, E_l] int32 on the device (negative counts move nothing);
 * in, out [n_rows, H] bf16 (H = d->H), distinct buffers; off_local [E_l + 1]
 * int32 or NULL. Rows the counts place at or beyond n_rows are not moved;
 * output rows beyond the counts' total are not written. T, k and F of d are
 * not used. A row copy: no arithmetic. */
moe_status_t moe_ep_resort(const moe_layer_desc_t* d, const int32_t* recv_cnt, const moe_bf16* in,
                           moe_bf16* out, int32_t* off_local, int64_t n_rows, int32_t inverse,
                           void* stream);

/* ------------------------------------------------------------------ whole layer */

/* Every buffer of one micro-batch (all device pointers, caller-owned). */
typedef struct moe_mb_bufs {
  const moe_bf16* x;  /* [T,H] */
  const moe_bf16* dy; /* [T,H] */
  const moe_bf16* w_r; const float* bias; const moe_bf16* w1; const moe_bf16* w2;
  float* logits; int32_t* idx; float* gates;                            /* route   */
  int32_t* cnt; int32_t* off; int32_t* slot; int32_t* row_src;          /* layout  */
  int32_t* cnt_re; int32_t* rank_off;
  moe_bf16* x_perm; moe_bf16* a; moe_bf16* h; moe_bf16* o; moe_bf16* y; /* forward */
  moe_bf16* d_o; float* dgates; moe_bf16* da; moe_bf16* dx_perm;        /* backward*/
  float* dx32; moe_bf16* dx; float* dw_r; moe_bf16* dw1; moe_bf16* dw2;
  void* ws; size_t ws_bytes;
  float* main_dw1; float* main_dw2; /* fp32 [E,2F,H], [E,H,F]: used (+=) only
                                       with MOE_FLAG_WGRAD_ACCUM_FP32 */
} moe_mb_bufs_t;

/* Forward: route, dispatch layout, permute (as moe_dispatch_fused: one launch
 * when E <= 128), expert FFN, combine. */
moe_status_t moe_layer_forward(const moe_layer_desc_t* d, const moe_mb_bufs_t* b, void* stream);

/* Backward in the chain order combine -> experts (dgrad) -> dispatch -> router,
 * and the expert wgrad when run_wgrad != 0. The wgrad runs on a library-owned
 * side stream (one per device, created by the first call with that device
 * current) beside the dispatch and router backward, forked after the dgrad and
 * joined into `stream` before the call returns. The dispatch backward is fused
 * into the router's dx pass here: the row sums of dx_perm stay in registers,
 * so b->dx32 is not written (dx has the same bits as the two-call path
 * moe_permute_bwd + moe_route_bwd). */
moe_status_t moe_layer_backward(const moe_layer_desc_t* d, const moe_mb_bufs_t* b,
                                int32_t run_wgrad, void* stream);

/* One training step of the layer from host memory: copies host_x and host_dy
 * into b->x and b->dy (which must then be writable device buffers), runs the
 * forward and the backward (with wgrad), and copies y and dx back into host_y
 * and host_dx. Host buffers should be pinned. The dy upload and the y download
 * run on a library-owned copy stream (one per device, created by the first
 * call with that device current), overlapping the forward and the backward,
 * and dx goes out on that stream as soon as the dispatch backward has written
 * it, beside the weight gradients; everything is ordered after the work
 * already on `stream`. Returns once all four copies and the weight gradients
 * are done (synchronises `stream`). */
moe_status_t moe_layer_step_host(const moe_layer_desc_t* d, const moe_mb_bufs_t* b,
                                 const moe_bf16* host_x, const moe_bf16* host_dy,
                                 moe_bf16* host_y, moe_bf16* host_dx, void* stream);

/* n training steps of the layer from host memory, pipelined. Step i copies
 * host_x[i] and host_dy[i] in, runs the forward and the backward (with
 * wgrad) and copies y and dx out into host_y[i] and host_dx[i], as
 * moe_layer_step_host does, on the buffer set b[i % 2]. Step i+1's inputs go
 * in on a library-owned copy stream while step i computes, and step i's
 * outputs come out on a second one while step i+1 computes, so the copies
 * leave the critical path; the computation of the steps runs one after the
 * other on `stream`. The two buffer sets need their own x, dy, y and dx (all
 * writable device buffers); every other pointer may be shared between them
 * (weights, workspace, intermediates, gradients), since no two steps compute
 * at once. Each step's weight gradients go where its set says (overwritten,
 * or added under MOE_FLAG_WGRAD_ACCUM_FP32 in step order). The host arrays
 * hold n pointers each; host buffers should be pinned. Returns once every
 * step is done and every copy has landed (synchronises `stream`). */
moe_status_t moe_layer_steps_host(const moe_layer_desc_t* d, const moe_mb_bufs_t* b /*[2]*/,
                                  int32_t n, const moe_bf16* const* host_x,
                                  const moe_bf16* const* host_dy, moe_bf16* const* host_y,
                                  moe_bf16* const* host_dx, void* stream);

/* ------------------------------------------------------------------ CUDA graphs */

/* Capture scopes. The skill card's production benchmark (section "HybridEP
 * production benchmark") runs the router and the dispatch preprocessing under
 * CUDA graphs (Transformer Engine scopes moe_router + moe_preprocess);
 * MOE_GRAPH_ROUTER_PREPROCESS is that scope. The wider scopes put a whole
 * forward, or forward + backward, into one graph launch. */
typedef enum {
  MOE_GRAPH_ROUTER_PREPROCESS = 0, /* route + dispatch layout + permute          */
  MOE_GRAPH_LAYER_FORWARD = 1,     /* moe_layer_forward                          */
  MOE_GRAPH_LAYER_STEP = 2         /* moe_layer_forward + moe_layer_backward
                                      (with wgrad, as d->flags selects)          */
} moe_graph_scope_t;

typedef struct moe_graph moe_graph_t;

/* Captures the calls of `scope` on buffers b into a CUDA graph and instantiates
 * it. Nothing runs during the capture. `stream` must be a caller-created stream
 * (not a default stream), not already capturing, and per-launch profiling
 * (moe_profile_start) must be off. The graph keeps every device pointer of b,
 * the layer shape and d->flags as they were at capture: a replay reads and
 * writes the same buffers, so new inputs are copied into them before a replay.
 * The backward's side-stream fork/join becomes graph edges. Allocates the
 * graph (host and driver memory), which moe_graph_destroy frees. *out is NULL
 * on error. */
moe_status_t moe_graph_capture(const moe_layer_desc_t* d, const moe_mb_bufs_t* b, int32_t scope,
                               void* stream, moe_graph_t** out);

/* Enqueues one replay of the graph on `stream` (any stream of the device it
 * was captured on). Replays on one stream run in order. */
moe_status_t moe_graph_launch(moe_graph_t* g, void* stream);

/* Kernel nodes in the graph (moe_kernel_launches() grows by this per replay). */
int32_t moe_graph_kernel_count(const moe_graph_t* g);

/* Frees the graph; the caller makes sure no replay is still running. */
void moe_graph_destroy(moe_graph_t* g);

/* ------------------------------------------------------------------ two-stream scheduler */

typedef enum {
  MOE_PHASE_DISPATCH = 0,     /* route + layout + permute            (comm stream) */
  MOE_PHASE_FFN_FWD = 1,      /* expert FFN forward                  (GEMM stream) */
  MOE_PHASE_COMBINE = 2,      /* combine                             (comm stream) */
  MOE_PHASE_COMBINE_BWD = 3,  /* combine backward                    (comm stream) */
  MOE_PHASE_DGRAD = 4,        /* expert dgrad                        (GEMM stream) */
  MOE_PHASE_DISPATCH_BWD = 5, /* permute backward + router backward  (comm stream) */
  MOE_PHASE_WGRAD = 6         /* expert wgrad                        (GEMM stream) */
} moe_phase_t;

typedef struct moe_phase_time {
  int32_t mb;       /* micro-batch 0 or 1 */
  int32_t phase;    /* moe_phase_t */
  int32_t stream;   /* 0 = comm stream, 1 = GEMM stream */
  float start_ms;   /* from the step's start event */
  float end_ms;
} moe_phase_time_t;

typedef struct moe_sched moe_sched_t;

/* Creates a scheduler for two micro-batches of shape d on two caller-owned
 * streams (stream_comm runs route/dispatch/combine and their backward,
 * stream_gemm the grouped GEMMs). gemm_sms (0 = no cap): under overlap = 1 it
 * caps every persistent GEMM grid; under overlap = 2 it splits the GPU for the
 * one overlapped pair, micro-batch 0's expert forward on gemm_sms SMs and
 * micro-batch 1's fused dispatch on the rest. Allocates CUDA events only. */
moe_status_t moe_sched_create(const moe_layer_desc_t* d, void* stream_comm, void* stream_gemm,
                              int32_t gemm_sms, moe_sched_t** out);

/* One step = forward and backward of both micro-batches mb[0], mb[1] (each with
 * its own buffers and workspace; weights may be shared, weight gradients, and
 * the fp32 main gradients under MOE_FLAG_WGRAD_ACCUM_FP32, must not be, so
 * that the order of the fp32 additions does not depend on the schedule).
 * overlap = 0: every phase on stream_comm in the order F0 F1 B0 B1.
 * overlap = 1 (or any value but 0 and 2): phases spread over the two streams
 * so one micro-batch's dispatch/combine runs beside the other's GEMMs, ordered
 * by events on data dependencies only.
 * overlap = 2: only micro-batch 1's dispatch (its router phase is FMA-bound)
 * runs beside micro-batch 0's work; the rest keeps the layer order
 * F0 B0 F1 B1 on stream_gemm, each weight gradient on stream_comm beside its
 * dispatch backward. defer_wgrad = 1: micro-batch 1's wgrad is not run in this
 * step but at the start of the next one (beside micro-batch 0's dispatch), or by
 * moe_sched_flush(). Outputs are bit-identical to the serial schedule's. */
moe_status_t moe_sched_step(moe_sched_t* s, const moe_mb_bufs_t* mb, int32_t overlap,
                            int32_t defer_wgrad);

/* Per-phase timing on (default) or off. On, every phase of a step is
 * bracketed by CUDA events on its stream for moe_sched_timings; those events
 * sit between the kernels of a stream and stop each kernel's launch from
 * overlapping the previous kernel's drain (programmatic dependent launch).
 * Off, a step records only the events of its cross-stream dependencies, and
 * moe_sched_timings reports no phases. */
moe_status_t moe_sched_set_phase_timing(moe_sched_t* s, int32_t on);

/* Runs a deferred wgrad, if one is pending, on stream_gemm. */
moe_status_t moe_sched_flush(moe_sched_t* s);

/* Per-phase start/end times of the last step (synchronises both streams).
 * Writes up to cap entries and the count to *n. */
moe_status_t moe_sched_timings(moe_sched_t* s, moe_phase_time_t* out, int32_t cap, int32_t* n);

void moe_sched_destroy(moe_sched_t* s);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
