// Per-phase operations on one micro-batch's buffers, shared by the C ABI's
// whole-layer calls and the two-stream scheduler.
#pragma once

#include "moe_internal.cuh"

namespace moe {

moe_status_t validate(const moe_layer_desc_t* d);
// The current device's library-owned helper streams (copy stream, backward
// side stream), created on first use; NULL (with an error message) on failure.
struct CopyLane;
CopyLane* copy_lane();
moe_status_t check_mb(const moe_layer_desc_t& d, const moe_mb_bufs_t* b, bool bwd);

// route + dispatch layout + permute; max_ctas > 0 caps the fused launch's grid
moe_status_t op_dispatch(const moe_layer_desc_t& d, const moe_mb_bufs_t* b, cudaStream_t st,
                         int max_ctas = 0);
moe_status_t op_ffn_fwd_mb(const moe_layer_desc_t& d, const moe_mb_bufs_t* b, int max_ctas,
                           cudaStream_t st);
moe_status_t op_combine_mb(const moe_layer_desc_t& d, const moe_mb_bufs_t* b, cudaStream_t st);
moe_status_t op_combine_bwd_mb(const moe_layer_desc_t& d, const moe_mb_bufs_t* b,
                               cudaStream_t st);
moe_status_t op_dgrad_mb(const moe_layer_desc_t& d, const moe_mb_bufs_t* b, int max_ctas,
                         cudaStream_t st);
// permute backward + router backward
moe_status_t op_dispatch_bwd_mb(const moe_layer_desc_t& d, const moe_mb_bufs_t* b,
                                cudaStream_t st);
moe_status_t op_wgrad_mb(const moe_layer_desc_t& d, const moe_mb_bufs_t* b, int max_ctas,
                         cudaStream_t st);

}  // namespace moe
