// Two-stream, two-micro-batch schedule of the MoE layer's phases.
//
// The EP-overlap note ("1. MoE EP Overlap", section "MoE 1F1B overlap")
// replaces the serial forward + backward + all-to-all of one micro-batch with
// two streams and two micro-batches, so one micro-batch's communication
// (dispatch/combine) runs beside the other's computation; its mlp backward
// computes the activation gradient first and the weight gradient later, and
// delay_wgrad_compute (skill card, "what it is") pushes the weight gradient
// behind the next forward. Phases are the note's ScheduleNodes (section "how
// the 8 fwd/bwd operations are split out"), each with a stream and an event.
//
// On one GPU the all-to-all is the permute/combine kernels themselves, so the
// "communication stream" runs route/layout/permute, combine and their
// backward, and the "GEMM stream" runs the grouped expert GEMMs. Cross-stream
// order comes only from events on real data dependencies, so the results are
// bit-identical to the serial order.
#include <stdlib.h>

#include <algorithm>
#include <string.h>

#include "moe_layer_ops.h"

namespace moe {
namespace {

constexpr int kMaxRecords = 32;

struct Record {
  int mb, phase, stream;
  cudaEvent_t s, e;
};

}  // namespace
}  // namespace moe

struct moe_sched {
  moe_layer_desc_t d;
  cudaStream_t sc, sg;
  int gemm_sms;
  cudaEvent_t ev_start;
  cudaEvent_t dep[16];
  cudaEvent_t tev[2 * moe::kMaxRecords];
  moe::Record rec[moe::kMaxRecords];
  int nrec;
  int timing;   // record per-phase events (moe_sched_set_phase_timing)
  int pending;  // micro-batch whose wgrad was deferred, or -1
  moe_mb_bufs_t pending_bufs;
};

using namespace moe;

namespace {

enum Dep {
  D_DISP0 = 0, D_DISP1, D_FFN0, D_FFN1, D_CBWD0, D_CBWD1, D_DGRAD0, D_DGRAD1, D_WGPREV, D_SG_END
};

moe_status_t cuda_ok(cudaError_t e, const char* what) {
  if (e != cudaSuccess) {
    set_error("%s: %s", what, cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

#define SCHK(x)                   \
  do {                            \
    moe_status_t _s = (x);        \
    if (_s != MOE_OK) return _s;  \
  } while (0)

moe_status_t begin(moe_sched* s, int mb, int phase, int stream, cudaStream_t st, Record** out) {
  if (s->nrec >= kMaxRecords) {
    set_error("scheduler: too many phase records");
    return MOE_ERR_INVALID_ARG;
  }
  Record* r = &s->rec[s->nrec];
  r->mb = mb;
  r->phase = phase;
  r->stream = stream;
  r->s = s->tev[2 * s->nrec];
  r->e = s->tev[2 * s->nrec + 1];
  ++s->nrec;
  *out = r;
  return cuda_ok(cudaEventRecord(r->s, st), "cudaEventRecord");
}

moe_status_t end(Record* r, cudaStream_t st) { return cuda_ok(cudaEventRecord(r->e, st), "cudaEventRecord"); }

moe_status_t wait(cudaStream_t st, cudaEvent_t ev) {
  return cuda_ok(cudaStreamWaitEvent(st, ev, 0), "cudaStreamWaitEvent");
}

moe_status_t run_phase(moe_sched* s, const moe_mb_bufs_t* b, int mb, int phase, cudaStream_t st,
                       int stream_id, int max_ctas) {
  Record* r = nullptr;
  if (s->timing) SCHK(begin(s, mb, phase, stream_id, st, &r));
  const moe_layer_desc_t& d = s->d;
  switch (phase) {
    case MOE_PHASE_DISPATCH: SCHK(op_dispatch(d, b, st, max_ctas)); break;
    case MOE_PHASE_FFN_FWD: SCHK(op_ffn_fwd_mb(d, b, max_ctas, st)); break;
    case MOE_PHASE_COMBINE: SCHK(op_combine_mb(d, b, st)); break;
    case MOE_PHASE_COMBINE_BWD: SCHK(op_combine_bwd_mb(d, b, st)); break;
    case MOE_PHASE_DGRAD: SCHK(op_dgrad_mb(d, b, max_ctas, st)); break;
    case MOE_PHASE_DISPATCH_BWD: SCHK(op_dispatch_bwd_mb(d, b, st)); break;
    default: SCHK(op_wgrad_mb(d, b, max_ctas, st)); break;
  }
  return r ? end(r, st) : MOE_OK;
}

}  // namespace

extern "C" {

moe_status_t moe_sched_create(const moe_layer_desc_t* d, void* stream_comm, void* stream_gemm,
                              int32_t gemm_sms, moe_sched_t** out) {
  SCHK(validate(d));
  if (!out) {
    set_error("out is NULL");
    return MOE_ERR_INVALID_ARG;
  }
  *out = nullptr;
  if (stream_comm == stream_gemm) {
    set_error("the scheduler needs two distinct streams");
    return MOE_ERR_INVALID_ARG;
  }
  moe_sched* s = static_cast<moe_sched*>(calloc(1, sizeof(moe_sched)));
  if (!s) {
    set_error("out of host memory");
    return MOE_ERR_INVALID_ARG;
  }
  s->d = *d;
  s->sc = static_cast<cudaStream_t>(stream_comm);
  s->sg = static_cast<cudaStream_t>(stream_gemm);
  s->gemm_sms = gemm_sms;
  s->timing = 1;
  s->pending = -1;
  cudaError_t e = cudaEventCreate(&s->ev_start);
  for (int i = 0; i < 16 && e == cudaSuccess; ++i)
    e = cudaEventCreateWithFlags(&s->dep[i], cudaEventDisableTiming);
  for (int i = 0; i < 2 * kMaxRecords && e == cudaSuccess; ++i) e = cudaEventCreate(&s->tev[i]);
  if (e != cudaSuccess) {
    set_error("cudaEventCreate: %s", cudaGetErrorString(e));
    moe_sched_destroy(s);
    return MOE_ERR_CUDA;
  }
  *out = s;
  return MOE_OK;
}

void moe_sched_destroy(moe_sched_t* s) {
  if (!s) return;
  if (s->ev_start) cudaEventDestroy(s->ev_start);
  for (int i = 0; i < 16; ++i)
    if (s->dep[i]) cudaEventDestroy(s->dep[i]);
  for (int i = 0; i < 2 * kMaxRecords; ++i)
    if (s->tev[i]) cudaEventDestroy(s->tev[i]);
  free(s);
}

moe_status_t moe_sched_step(moe_sched_t* s, const moe_mb_bufs_t* mb, int32_t overlap,
                            int32_t defer_wgrad) {
  if (!s || !mb) {
    set_error("scheduler or buffers NULL");
    return MOE_ERR_INVALID_ARG;
  }
  const moe_layer_desc_t& d = s->d;
  SCHK(check_mb(d, &mb[0], true));
  SCHK(check_mb(d, &mb[1], true));
  const bool acc = (d.flags & MOE_FLAG_WGRAD_ACCUM_FP32) != 0;
  const void* g1[2] = {acc ? (const void*)mb[0].main_dw1 : mb[0].dw1,
                       acc ? (const void*)mb[1].main_dw1 : mb[1].dw1};
  const void* g2[2] = {acc ? (const void*)mb[0].main_dw2 : mb[0].dw2,
                       acc ? (const void*)mb[1].main_dw2 : mb[1].dw2};
  if (mb[0].ws == mb[1].ws || g1[0] == g1[1] || g2[0] == g2[1] || mb[0].dw_r == mb[1].dw_r) {
    set_error("the two micro-batches need their own workspace and weight-gradient buffers");
    return MOE_ERR_INVALID_ARG;
  }
  s->nrec = 0;
  cudaStream_t sc = s->sc, sg = s->sg;
  SCHK(cuda_ok(cudaEventRecord(s->ev_start, sc), "cudaEventRecord"));
  const int pend = s->pending;
  const moe_mb_bufs_t pend_bufs = s->pending_bufs;
  s->pending = -1;

  if (!overlap) {
    if (pend >= 0) SCHK(run_phase(s, &pend_bufs, pend, MOE_PHASE_WGRAD, sc, 0, 0));
    for (int m = 0; m < 2; ++m) {
      SCHK(run_phase(s, &mb[m], m, MOE_PHASE_DISPATCH, sc, 0, 0));
      SCHK(run_phase(s, &mb[m], m, MOE_PHASE_FFN_FWD, sc, 0, 0));
      SCHK(run_phase(s, &mb[m], m, MOE_PHASE_COMBINE, sc, 0, 0));
    }
    for (int m = 0; m < 2; ++m) {
      SCHK(run_phase(s, &mb[m], m, MOE_PHASE_COMBINE_BWD, sc, 0, 0));
      SCHK(run_phase(s, &mb[m], m, MOE_PHASE_DGRAD, sc, 0, 0));
      SCHK(run_phase(s, &mb[m], m, MOE_PHASE_DISPATCH_BWD, sc, 0, 0));
      if (m == 1 && defer_wgrad) {
        s->pending = 1;
        s->pending_bufs = mb[1];
      } else {
        SCHK(run_phase(s, &mb[m], m, MOE_PHASE_WGRAD, sc, 0, 0));
      }
    }
    return MOE_OK;
  }

  const int gs = s->gemm_sms;
  SCHK(wait(sg, s->ev_start));
  if (overlap == 2) {
    // Only micro-batch 1's dispatch runs beside micro-batch 0's work: its
    // router phase is bound by FMA arithmetic and reads little, so it is the
    // one phase that gains beside an HBM-bound GEMM. Everything else keeps the
    // plain layer order F0 B0 F1 B1 on the GEMM stream, so consecutive
    // kernels there keep their programmatic dependent launch; each weight
    // gradient runs on the comm stream beside its dispatch backward, as
    // moe_layer_backward runs it on its side stream. With gemm_sms > 0 the
    // GPU is split for the one overlapped pair: expert forward 0 on gemm_sms
    // SMs, dispatch 1 on the others; every other phase takes the whole GPU.
    const int fwd0_ctas = gs > 0 ? gs : 0;
    const int disp1_ctas = gs > 0 ? std::max(1, device_sm_count() - gs) : 0;
    if (pend >= 0) {
      SCHK(run_phase(s, &pend_bufs, pend, MOE_PHASE_WGRAD, sg, 1, 0));
      SCHK(cuda_ok(cudaEventRecord(s->dep[D_WGPREV], sg), "cudaEventRecord"));
    }
    SCHK(run_phase(s, &mb[0], 0, MOE_PHASE_DISPATCH, sc, 0, 0));
    SCHK(cuda_ok(cudaEventRecord(s->dep[D_DISP0], sc), "cudaEventRecord"));
    // dispatch(1) rewrites micro-batch 1's saved tensors, which a deferred
    // wgrad still reads
    if (pend >= 0) SCHK(wait(sc, s->dep[D_WGPREV]));
    SCHK(run_phase(s, &mb[1], 1, MOE_PHASE_DISPATCH, sc, 0, disp1_ctas));
    SCHK(cuda_ok(cudaEventRecord(s->dep[D_DISP1], sc), "cudaEventRecord"));
    for (int m = 0; m < 2; ++m) {
      SCHK(wait(sg, s->dep[m == 0 ? D_DISP0 : D_DISP1]));
      SCHK(run_phase(s, &mb[m], m, MOE_PHASE_FFN_FWD, sg, 1, m == 0 ? fwd0_ctas : 0));
      SCHK(run_phase(s, &mb[m], m, MOE_PHASE_COMBINE, sg, 1, 0));
      SCHK(run_phase(s, &mb[m], m, MOE_PHASE_COMBINE_BWD, sg, 1, 0));
      SCHK(run_phase(s, &mb[m], m, MOE_PHASE_DGRAD, sg, 1, 0));
      const Dep dg = m == 0 ? D_DGRAD0 : D_DGRAD1;
      SCHK(cuda_ok(cudaEventRecord(s->dep[dg], sg), "cudaEventRecord"));
      if (m == 1 && defer_wgrad) {
        s->pending = 1;
        s->pending_bufs = mb[1];
      } else {
        SCHK(wait(sc, s->dep[dg]));
        SCHK(run_phase(s, &mb[m], m, MOE_PHASE_WGRAD, sc, 0, 0));
      }
      SCHK(run_phase(s, &mb[m], m, MOE_PHASE_DISPATCH_BWD, sg, 1, 0));
    }
    SCHK(cuda_ok(cudaEventRecord(s->dep[D_SG_END], sg), "cudaEventRecord"));
    return wait(sc, s->dep[D_SG_END]);
  }
  // t0: dispatch(0) on the comm stream; a deferred wgrad beside it
  SCHK(run_phase(s, &mb[0], 0, MOE_PHASE_DISPATCH, sc, 0, 0));
  SCHK(cuda_ok(cudaEventRecord(s->dep[D_DISP0], sc), "cudaEventRecord"));
  if (pend >= 0) {
    SCHK(run_phase(s, &pend_bufs, pend, MOE_PHASE_WGRAD, sg, 1, gs));
    SCHK(cuda_ok(cudaEventRecord(s->dep[D_WGPREV], sg), "cudaEventRecord"));
  }
  // t1: experts(0) beside dispatch(1); dispatch(1) rewrites micro-batch 1's
  // saved tensors, so it waits for a deferred wgrad that still reads them
  SCHK(wait(sg, s->dep[D_DISP0]));
  SCHK(run_phase(s, &mb[0], 0, MOE_PHASE_FFN_FWD, sg, 1, gs));
  SCHK(cuda_ok(cudaEventRecord(s->dep[D_FFN0], sg), "cudaEventRecord"));
  if (pend >= 0) SCHK(wait(sc, s->dep[D_WGPREV]));
  SCHK(run_phase(s, &mb[1], 1, MOE_PHASE_DISPATCH, sc, 0, 0));
  SCHK(cuda_ok(cudaEventRecord(s->dep[D_DISP1], sc), "cudaEventRecord"));
  // t2: combine(0) + combine_bwd(0) beside experts(1)
  SCHK(wait(sc, s->dep[D_FFN0]));
  SCHK(run_phase(s, &mb[0], 0, MOE_PHASE_COMBINE, sc, 0, 0));
  SCHK(run_phase(s, &mb[0], 0, MOE_PHASE_COMBINE_BWD, sc, 0, 0));
  SCHK(cuda_ok(cudaEventRecord(s->dep[D_CBWD0], sc), "cudaEventRecord"));
  SCHK(wait(sg, s->dep[D_DISP1]));
  SCHK(run_phase(s, &mb[1], 1, MOE_PHASE_FFN_FWD, sg, 1, gs));
  SCHK(cuda_ok(cudaEventRecord(s->dep[D_FFN1], sg), "cudaEventRecord"));
  // t3: dgrad(0) beside combine(1) + combine_bwd(1)
  SCHK(wait(sg, s->dep[D_CBWD0]));
  SCHK(run_phase(s, &mb[0], 0, MOE_PHASE_DGRAD, sg, 1, gs));
  SCHK(cuda_ok(cudaEventRecord(s->dep[D_DGRAD0], sg), "cudaEventRecord"));
  SCHK(wait(sc, s->dep[D_FFN1]));
  SCHK(run_phase(s, &mb[1], 1, MOE_PHASE_COMBINE, sc, 0, 0));
  SCHK(run_phase(s, &mb[1], 1, MOE_PHASE_COMBINE_BWD, sc, 0, 0));
  SCHK(cuda_ok(cudaEventRecord(s->dep[D_CBWD1], sc), "cudaEventRecord"));
  // t4: dispatch_bwd(0) beside wgrad(0) and dgrad(1)
  SCHK(wait(sc, s->dep[D_DGRAD0]));
  SCHK(run_phase(s, &mb[0], 0, MOE_PHASE_DISPATCH_BWD, sc, 0, 0));
  SCHK(run_phase(s, &mb[0], 0, MOE_PHASE_WGRAD, sg, 1, gs));
  SCHK(wait(sg, s->dep[D_CBWD1]));
  SCHK(run_phase(s, &mb[1], 1, MOE_PHASE_DGRAD, sg, 1, gs));
  SCHK(cuda_ok(cudaEventRecord(s->dep[D_DGRAD1], sg), "cudaEventRecord"));
  // t5: dispatch_bwd(1) beside wgrad(1), unless it is deferred to the next step
  SCHK(wait(sc, s->dep[D_DGRAD1]));
  SCHK(run_phase(s, &mb[1], 1, MOE_PHASE_DISPATCH_BWD, sc, 0, 0));
  if (defer_wgrad) {
    s->pending = 1;
    s->pending_bufs = mb[1];
  } else {
    SCHK(run_phase(s, &mb[1], 1, MOE_PHASE_WGRAD, sg, 1, gs));
  }
  // join: the comm stream ends the step after all GEMM-stream work
  SCHK(cuda_ok(cudaEventRecord(s->dep[D_SG_END], sg), "cudaEventRecord"));
  return wait(sc, s->dep[D_SG_END]);
}

moe_status_t moe_sched_set_phase_timing(moe_sched_t* s, int32_t on) {
  if (!s) {
    set_error("scheduler is NULL");
    return MOE_ERR_INVALID_ARG;
  }
  s->timing = on != 0;
  return MOE_OK;
}

moe_status_t moe_sched_flush(moe_sched_t* s) {
  if (!s) {
    set_error("scheduler is NULL");
    return MOE_ERR_INVALID_ARG;
  }
  if (s->pending < 0) return MOE_OK;
  const moe_mb_bufs_t b = s->pending_bufs;
  const int m = s->pending;
  s->pending = -1;
  SCHK(op_wgrad_mb(s->d, &b, 0, s->sg));
  (void)m;
  cudaEvent_t ev = s->dep[D_SG_END];
  SCHK(cuda_ok(cudaEventRecord(ev, s->sg), "cudaEventRecord"));
  return wait(s->sc, ev);
}

moe_status_t moe_sched_timings(moe_sched_t* s, moe_phase_time_t* out, int32_t cap, int32_t* n) {
  if (!s || !n || (cap > 0 && !out)) {
    set_error("invalid arguments");
    return MOE_ERR_INVALID_ARG;
  }
  SCHK(cuda_ok(cudaStreamSynchronize(s->sc), "cudaStreamSynchronize"));
  SCHK(cuda_ok(cudaStreamSynchronize(s->sg), "cudaStreamSynchronize"));
  int k = 0;
  for (int i = 0; i < s->nrec && k < cap; ++i, ++k) {
    float a = 0.f, b = 0.f;
    SCHK(cuda_ok(cudaEventElapsedTime(&a, s->ev_start, s->rec[i].s), "cudaEventElapsedTime"));
    SCHK(cuda_ok(cudaEventElapsedTime(&b, s->ev_start, s->rec[i].e), "cudaEventElapsedTime"));
    out[k].mb = s->rec[i].mb;
    out[k].phase = s->rec[i].phase;
    out[k].stream = s->rec[i].stream;
    out[k].start_ms = a;
    out[k].end_ms = b;
  }
  *n = k;
  return MOE_OK;
}

}  // extern "C"
