"""GB300-native MoE layer hot path: route -> dispatch layout -> permute -> grouped
SwiGLU experts (tcgen05) -> combine, with the backward split into dgrad and
(deferrable) wgrad, and a two-stream two-micro-batch scheduler.

Everything runs in the CUDA kernels of libmoe.so behind the C ABI in
include/moe.h. This module only marshals arguments: each function has the C
name, takes torch CUDA tensors, passes their data pointers and raises MoeError
on a nonzero status. There is no CPU path: if libmoe.so is missing or cannot
load, importing the functions raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "moe.h")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_TIMEOUT = range(5)
ROUTE_SOFTMAX_TOPK, ROUTE_FORCED_BALANCED = 0, 1
GRAPH_ROUTER_PREPROCESS, GRAPH_LAYER_FORWARD, GRAPH_LAYER_STEP = 0, 1, 2
FLAG_WGRAD_ACCUM_FP32 = 1  # MOE_FLAG_WGRAD_ACCUM_FP32: add wgrad into fp32 main gradients
PHASES = ("dispatch", "ffn_fwd", "combine", "combine_bwd", "dgrad", "dispatch_bwd", "wgrad")

_STATUS = {1: "invalid argument", 2: "unsupported", 3: "CUDA error", 4: "timeout"}


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str, msg: str):
        super().__init__(f"{what}: {_STATUS.get(status, status)}: {msg}")
        self.status = status


class LayerDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("T", "H", "E", "k", "F", "R", "mode", "flags")]

    @classmethod
    def of(cls, T, H, E, k, F, R=1, mode=ROUTE_SOFTMAX_TOPK, flags=0):
        return cls(T, H, E, k, F, R, mode, flags)

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


_MB_FIELDS = ["x", "dy", "w_r", "bias", "w1", "w2", "logits", "idx", "gates", "cnt", "off",
              "slot", "row_src", "cnt_re", "rank_off", "x_perm", "a", "h", "o", "y", "d_o",
              "dgates", "da", "dx_perm", "dx32", "dx", "dw_r", "dw1", "dw2", "ws"]


_MB_FIELDS_TAIL = ["main_dw1", "main_dw2"]


class MbBufs(ctypes.Structure):
    _fields_ = ([(n, ctypes.c_void_p) for n in _MB_FIELDS] + [("ws_bytes", ctypes.c_size_t)]
                + [(n, ctypes.c_void_p) for n in _MB_FIELDS_TAIL])


class PhaseTime(ctypes.Structure):
    _fields_ = [("mb", ctypes.c_int32), ("phase", ctypes.c_int32), ("stream", ctypes.c_int32),
                ("start_ms", ctypes.c_float), ("end_ms", ctypes.c_float)]


class KernelTime(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("ms", ctypes.c_float)]


_lib = None

_VP, _I32, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
_DP = ctypes.POINTER(LayerDesc)
_SIGS = {
    "moe_abi_version": ([], _I32),
    "moe_last_error": ([], ctypes.c_char_p),
    "moe_layer_desc_validate": ([_DP], _I32),
    "moe_workspace_size": ([_DP], _SZ),
    "moe_device_status": ([_DP, _VP, _VP], _I32),
    "moe_kernel_launches": ([], ctypes.c_uint64),
    "moe_set_barrier_wait_limit_ns": ([ctypes.c_uint64], ctypes.c_uint64),
    "moe_kernel_name": ([_I32], ctypes.c_char_p),
    "moe_profile_start": ([_I32], _I32),
    "moe_profile_stop": ([ctypes.POINTER(KernelTime), _I32, ctypes.POINTER(_I32)], _I32),
    "moe_route": ([_DP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP], _I32),
    "moe_dispatch_layout": ([_DP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP], _I32),
    "moe_dispatch_layout_static": ([_DP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP], _I32),
    "moe_dispatch_layout_static_status": ([_VP], _I32),
    "moe_permute": ([_DP, _VP, _VP, _VP, _VP], _I32),
    "moe_dispatch_fused": ([_DP] + [_VP] * 14 + [_SZ, _VP], _I32),
    "moe_expert_ffn_fwd": ([_DP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP], _I32),
    "moe_combine": ([_DP, _VP, _VP, _VP, _VP, _VP], _I32),
    "moe_combine_bwd": ([_DP, _VP, _VP, _VP, _VP, _VP, _VP, _VP], _I32),
    "moe_expert_ffn_bwd_dgrad": ([_DP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP], _I32),
    "moe_expert_ffn_bwd_wgrad": ([_DP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP], _I32),
    "moe_expert_ffn_bwd_wgrad_accum": ([_DP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP],
                                       _I32),
    "moe_permute_bwd": ([_DP, _VP, _VP, _VP, _VP], _I32),
    "moe_route_bwd": ([_DP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP], _I32),
    "moe_ep_resort": ([_DP, _VP, _VP, _VP, _VP, ctypes.c_int64, _I32, _VP], _I32),
    "moe_layer_forward": ([_DP, ctypes.POINTER(MbBufs), _VP], _I32),
    "moe_layer_backward": ([_DP, ctypes.POINTER(MbBufs), _I32, _VP], _I32),
    "moe_layer_step_host": ([_DP, ctypes.POINTER(MbBufs), _VP, _VP, _VP, _VP, _VP], _I32),
    "moe_layer_steps_host": ([_DP, ctypes.POINTER(MbBufs), _I32, ctypes.POINTER(_VP),
                              ctypes.POINTER(_VP), ctypes.POINTER(_VP), ctypes.POINTER(_VP), _VP],
                             _I32),
    "moe_graph_capture": ([_DP, ctypes.POINTER(MbBufs), _I32, _VP, ctypes.POINTER(_VP)], _I32),
    "moe_graph_launch": ([_VP, _VP], _I32),
    "moe_graph_kernel_count": ([_VP], _I32),
    "moe_graph_destroy": ([_VP], None),
    "moe_sched_create": ([_DP, _VP, _VP, _I32, ctypes.POINTER(_VP)], _I32),
    "moe_sched_step": ([_VP, ctypes.POINTER(MbBufs), _I32, _I32], _I32),
    "moe_sched_flush": ([_VP], _I32),
    "moe_sched_set_phase_timing": ([_VP, _I32], _I32),
    "moe_sched_timings": ([_VP, ctypes.POINTER(PhaseTime), _I32, ctypes.POINTER(_I32)], _I32),
    "moe_sched_destroy": ([_VP], None),
}


def lib() -> ctypes.CDLL:
    """The loaded libmoe.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "combine_router_softmax_top_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def _err() -> str:
    return lib().moe_last_error().decode(errors="replace")


def _check(status: int, what: str):
    if status != MOE_OK:
        raise MoeError(status, what, _err())


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _s(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _d(desc: LayerDesc):
    return ctypes.byref(desc)


# ----------------------------------------------------------------------------- entry points
def moe_layer_desc_validate(desc: LayerDesc) -> int:
    return lib().moe_layer_desc_validate(_d(desc))


def moe_workspace_size(desc: LayerDesc) -> int:
    n = lib().moe_workspace_size(_d(desc))
    if n == 0:
        raise MoeError(MOE_ERR_INVALID_ARG, "moe_workspace_size", _err())
    return n


def moe_device_status(desc, ws, stream=None) -> int:
    return lib().moe_device_status(_d(desc), _p(ws), _s(stream))


def moe_kernel_launches() -> int:
    return int(lib().moe_kernel_launches())


def moe_set_barrier_wait_limit_ns(ns: int) -> int:
    """Grid-barrier wait limit of the fused dispatch (0 = default 2 s); returns the old one."""
    return int(lib().moe_set_barrier_wait_limit_ns(int(ns)))


def moe_kernel_name(kernel: int) -> str:
    return lib().moe_kernel_name(int(kernel)).decode()


def moe_profile_start(capacity: int):
    _check(lib().moe_profile_start(int(capacity)), "moe_profile_start")


def moe_profile_stop(cap: int = 4096):
    """[(kernel name, ms), ...] of the launches recorded since moe_profile_start."""
    buf = (KernelTime * cap)()
    n = ctypes.c_int32()
    _check(lib().moe_profile_stop(buf, cap, ctypes.byref(n)), "moe_profile_stop")
    return [(moe_kernel_name(buf[i].kernel), float(buf[i].ms)) for i in range(n.value)]


def moe_route(desc, x, w_r, bias, logits, idx, gates, ws, stream=None):
    _check(lib().moe_route(_d(desc), _p(x), _p(w_r), _p(bias), _p(logits), _p(idx), _p(gates),
                           _p(ws), ws.numel() * ws.element_size(), _s(stream)), "moe_route")


def moe_dispatch_layout(desc, idx, cnt, off, slot, row_src, cnt_re, rank_off, ws, stream=None):
    _check(lib().moe_dispatch_layout(_d(desc), _p(idx), _p(cnt), _p(off), _p(slot), _p(row_src),
                                     _p(cnt_re), _p(rank_off), _p(ws),
                                     ws.numel() * ws.element_size(), _s(stream)),
           "moe_dispatch_layout")


def moe_dispatch_layout_static(desc, idx, cnt, off, slot, row_src, cnt_re, rank_off, stream=None):
    """Dispatch layout without a workspace (library-owned scratch; see include/moe.h)."""
    _check(lib().moe_dispatch_layout_static(_d(desc), _p(idx), _p(cnt), _p(off), _p(slot),
                                            _p(row_src), _p(cnt_re), _p(rank_off), _s(stream)),
           "moe_dispatch_layout_static")


def moe_dispatch_layout_static_status(stream=None) -> int:
    """Status of the last moe_dispatch_layout_static call (synchronises the stream)."""
    return lib().moe_dispatch_layout_static_status(_s(stream))


def moe_permute(desc, x, row_src, x_perm, stream=None):
    _check(lib().moe_permute(_d(desc), _p(x), _p(row_src), _p(x_perm), _s(stream)), "moe_permute")


def moe_dispatch_fused(desc, x, w_r, bias, logits, idx, gates, cnt, off, slot, row_src, cnt_re,
                       rank_off, x_perm, ws, stream=None):
    _check(lib().moe_dispatch_fused(_d(desc), _p(x), _p(w_r), _p(bias), _p(logits), _p(idx),
                                    _p(gates), _p(cnt), _p(off), _p(slot), _p(row_src),
                                    _p(cnt_re), _p(rank_off), _p(x_perm), _p(ws),
                                    ws.numel() * ws.element_size(), _s(stream)),
           "moe_dispatch_fused")


def moe_expert_ffn_fwd(desc, x_perm, off, w1, w2, a, h, o, ws, stream=None):
    _check(lib().moe_expert_ffn_fwd(_d(desc), _p(x_perm), _p(off), _p(w1), _p(w2), _p(a), _p(h),
                                    _p(o), _p(ws), ws.numel() * ws.element_size(), _s(stream)),
           "moe_expert_ffn_fwd")


def moe_combine(desc, o, slot, gates, y, stream=None):
    _check(lib().moe_combine(_d(desc), _p(o), _p(slot), _p(gates), _p(y), _s(stream)), "moe_combine")


def moe_combine_bwd(desc, dy, o, slot, gates, d_o, dgates, stream=None):
    _check(lib().moe_combine_bwd(_d(desc), _p(dy), _p(o), _p(slot), _p(gates), _p(d_o),
                                 _p(dgates), _s(stream)), "moe_combine_bwd")


def moe_expert_ffn_bwd_dgrad(desc, d_o, a, off, w1, w2, da, dx_perm, ws, stream=None):
    _check(lib().moe_expert_ffn_bwd_dgrad(_d(desc), _p(d_o), _p(a), _p(off), _p(w1), _p(w2),
                                          _p(da), _p(dx_perm), _p(ws),
                                          ws.numel() * ws.element_size(), _s(stream)),
           "moe_expert_ffn_bwd_dgrad")


def moe_expert_ffn_bwd_wgrad(desc, x_perm, h, d_o, da, off, dw1, dw2, ws, stream=None):
    _check(lib().moe_expert_ffn_bwd_wgrad(_d(desc), _p(x_perm), _p(h), _p(d_o), _p(da), _p(off),
                                          _p(dw1), _p(dw2), _p(ws),
                                          ws.numel() * ws.element_size(), _s(stream)),
           "moe_expert_ffn_bwd_wgrad")


def moe_expert_ffn_bwd_wgrad_accum(desc, x_perm, h, d_o, da, off, main_dw1, main_dw2, ws,
                                   stream=None):
    _check(lib().moe_expert_ffn_bwd_wgrad_accum(_d(desc), _p(x_perm), _p(h), _p(d_o), _p(da),
                                                _p(off), _p(main_dw1), _p(main_dw2), _p(ws),
                                                ws.numel() * ws.element_size(), _s(stream)),
           "moe_expert_ffn_bwd_wgrad_accum")


def moe_permute_bwd(desc, dx_perm, slot, dx32, stream=None):
    _check(lib().moe_permute_bwd(_d(desc), _p(dx_perm), _p(slot), _p(dx32), _s(stream)),
           "moe_permute_bwd")


def moe_route_bwd(desc, dgates, gates, idx, x, w_r, row_src, off, dx32, dx, dw_r, ws, stream=None):
    _check(lib().moe_route_bwd(_d(desc), _p(dgates), _p(gates), _p(idx), _p(x), _p(w_r),
                               _p(row_src), _p(off), _p(dx32), _p(dx), _p(dw_r), _p(ws),
                               ws.numel() * ws.element_size(), _s(stream)), "moe_route_bwd")


def moe_ep_resort(desc, recv_cnt, inp, out, off_local=None, inverse=False, stream=None):
    """Receive order <-> expert-major re-sort of the EP exchange (include/moe.h)."""
    _check(lib().moe_ep_resort(_d(desc), _p(recv_cnt), _p(inp), _p(out), _p(off_local),
                               int(min(inp.shape[0], out.shape[0])), int(bool(inverse)),
                               _s(stream)),
           "moe_ep_resort")


def moe_layer_forward(desc, bufs: "LayerBuffers", stream=None):
    _check(lib().moe_layer_forward(_d(desc), ctypes.byref(bufs.struct()), _s(stream)),
           "moe_layer_forward")


def moe_layer_backward(desc, bufs: "LayerBuffers", run_wgrad: bool = True, stream=None):
    _check(lib().moe_layer_backward(_d(desc), ctypes.byref(bufs.struct()), int(run_wgrad),
                                    _s(stream)), "moe_layer_backward")


def moe_layer_step_host(desc, bufs: "LayerBuffers", host_x, host_dy, host_y, host_dx, stream=None):
    _check(lib().moe_layer_step_host(_d(desc), ctypes.byref(bufs.struct()), _p(host_x),
                                     _p(host_dy), _p(host_y), _p(host_dx), _s(stream)),
           "moe_layer_step_host")


def moe_layer_steps_host(desc, bufs0: "LayerBuffers", bufs1: "LayerBuffers", host_x, host_dy,
                         host_y, host_dx, stream=None):
    """n pipelined steps from host memory (lists of n pinned CPU tensors each)."""
    n = len(host_x)
    if not (len(host_dy) == len(host_y) == len(host_dx) == n):
        raise ValueError("host lists must have the same length")
    arr = (MbBufs * 2)(bufs0.struct(), bufs1.struct())
    ptrs = lambda ts: (_VP * max(n, 1))(*[t.data_ptr() for t in ts])  # noqa: E731
    _check(lib().moe_layer_steps_host(_d(desc), arr, n, ptrs(host_x), ptrs(host_dy),
                                      ptrs(host_y), ptrs(host_dx), _s(stream)),
           "moe_layer_steps_host")


# ----------------------------------------------------------------------------- buffers
class LayerBuffers:
    """Every device buffer of one micro-batch (torch tensors used as plain memory)."""

    def __init__(self, desc: LayerDesc, device="cuda", weights: Optional["LayerBuffers"] = None):
        T, H, E, k, F, R = desc.T, desc.H, desc.E, desc.k, desc.F, desc.R
        N = T * k
        T = max(T, 1)  # zero-token layers still get valid (unused) pointers
        bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
        z = lambda *s, dt: torch.zeros(*s, dtype=dt, device=device)  # noqa: E731
        self.desc = desc
        self.x, self.dy = z(T, H, dt=bf), z(T, H, dt=bf)
        if weights is None:
            self.w_r, self.w1, self.w2 = z(E, H, dt=bf), z(E, 2 * F, H, dt=bf), z(E, H, F, dt=bf)
            self.bias = None
        else:
            self.w_r, self.w1, self.w2, self.bias = weights.w_r, weights.w1, weights.w2, weights.bias
        self.logits, self.idx, self.gates = z(T, E, dt=f32), z(T, k, dt=i32), z(T, k, dt=f32)
        self.cnt, self.off = z(E, dt=i32), z(E + 1, dt=i32)
        self.slot, self.row_src = z(T, k, dt=i32), z(max(N, 1), dt=i32)
        self.cnt_re, self.rank_off = z(R, E // R, dt=i32), z(R + 1, dt=i32)
        rows = max(N, 1)
        self.x_perm, self.a, self.h = z(rows, H, dt=bf), z(rows, 2 * F, dt=bf), z(rows, F, dt=bf)
        self.o, self.y = z(rows, H, dt=bf), z(T, H, dt=bf)
        self.d_o, self.dgates = z(rows, H, dt=bf), z(T, k, dt=f32)
        self.da, self.dx_perm = z(rows, 2 * F, dt=bf), z(rows, H, dt=bf)
        self.dx32, self.dx = z(T, H, dt=f32), z(T, H, dt=bf)
        self.dw_r = z(E, H, dt=f32)
        if desc.flags & FLAG_WGRAD_ACCUM_FP32:
            # the weight gradients are added into fp32 main gradients
            self.dw1 = self.dw2 = None
            self.main_dw1, self.main_dw2 = z(E, 2 * F, H, dt=f32), z(E, H, F, dt=f32)
        else:
            self.dw1, self.dw2 = z(E, 2 * F, H, dt=bf), z(E, H, F, dt=bf)
            self.main_dw1 = self.main_dw2 = None
        nbytes = moe_workspace_size(desc)
        self.ws = z((nbytes + 15) // 16 * 16, dt=torch.uint8)
        self._struct = None

    def load_inputs(self, inp, weights: bool = True):
        """Copies a moe_synth.LayerInputs into the device buffers."""
        self.x.copy_(inp.x)
        self.dy.copy_(inp.dy)
        if weights:
            self.w_r.copy_(inp.w_r)
            self.w1.copy_(inp.w1)
            self.w2.copy_(inp.w2)
            self.bias = None if inp.bias is None else inp.bias.to(self.x.device)
        self._struct = None

    def struct(self) -> MbBufs:
        if self._struct is None:
            s = MbBufs()
            for n in _MB_FIELDS + _MB_FIELDS_TAIL:
                t = getattr(self, n)
                setattr(s, n, None if t is None else t.data_ptr())
            s.ws_bytes = self.ws.numel()
            self._struct = s
        return self._struct


# ----------------------------------------------------------------------------- graphs
class Graph:
    """A captured CUDA graph of one scope of the layer on fixed buffers
    (moe_graph_capture); replay() enqueues it. The buffers must outlive it."""

    def __init__(self, desc: LayerDesc, bufs: "LayerBuffers", scope: int, stream):
        self._h = ctypes.c_void_p()
        self.desc, self.bufs = desc, bufs
        self._struct = bufs.struct()
        _check(lib().moe_graph_capture(_d(desc), ctypes.byref(self._struct), scope, _s(stream),
                                       ctypes.byref(self._h)), "moe_graph_capture")
        self.kernels = lib().moe_graph_kernel_count(self._h)

    def replay(self, stream=None):
        _check(lib().moe_graph_launch(self._h, _s(stream)), "moe_graph_launch")

    def close(self):
        if self._h:
            lib().moe_graph_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ----------------------------------------------------------------------------- scheduler
class Scheduler:
    """Two-stream, two-micro-batch schedule (moe_sched_*)."""

    def __init__(self, desc: LayerDesc, stream_comm, stream_gemm, gemm_sms: int = 0):
        self.desc = desc
        h = ctypes.c_void_p()
        _check(lib().moe_sched_create(_d(desc), _s(stream_comm), _s(stream_gemm), int(gemm_sms),
                                      ctypes.byref(h)), "moe_sched_create")
        self._h = h

    def step(self, mb0: LayerBuffers, mb1: LayerBuffers, overlap, defer_wgrad: bool):
        """overlap: 0 (or False) serial, 1 (or True) overlapped, 2 dispatch-only
        overlap (moe_sched_step in include/moe.h)."""
        arr = (MbBufs * 2)(mb0.struct(), mb1.struct())
        _check(lib().moe_sched_step(self._h, arr, int(overlap), int(defer_wgrad)), "moe_sched_step")

    def flush(self):
        _check(lib().moe_sched_flush(self._h), "moe_sched_flush")

    def set_phase_timing(self, on: bool):
        """Per-phase events on/off (off keeps programmatic dependent launch)."""
        _check(lib().moe_sched_set_phase_timing(self._h, int(bool(on))),
               "moe_sched_set_phase_timing")

    def timings(self):
        buf = (PhaseTime * 32)()
        n = ctypes.c_int32()
        _check(lib().moe_sched_timings(self._h, buf, 32, ctypes.byref(n)), "moe_sched_timings")
        return [dict(mb=buf[i].mb, phase=PHASES[buf[i].phase], stream=buf[i].stream,
                     start_ms=buf[i].start_ms, end_ms=buf[i].end_ms) for i in range(n.value)]

    def close(self):
        if self._h:
            lib().moe_sched_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def interval_overlap(timings):
    """Union of the dispatch/combine (communication) phase intervals, union of
    the expert-GEMM phase intervals, and the length of their intersection (the
    hidden communication), in ms, measured
    as the EP-overlap skill card's profiling section prescribes (interval
    unions and their intersection, never a sum of kernel durations)."""
    def union(iv):
        iv = sorted(iv)
        out = []
        for s, e in iv:
            if out and s <= out[-1][1]:
                out[-1][1] = max(out[-1][1], e)
            else:
                out.append([s, e])
        return out

    gemm_phases = ("ffn_fwd", "dgrad", "wgrad")
    comm = union([(t["start_ms"], t["end_ms"]) for t in timings if t["phase"] not in gemm_phases])
    gemm = union([(t["start_ms"], t["end_ms"]) for t in timings if t["phase"] in gemm_phases])
    inter = 0.0
    for a0, a1 in comm:
        for b0, b1 in gemm:
            inter += max(0.0, min(a1, b1) - max(a0, b0))
    return (sum(e - s for s, e in comm), sum(e - s for s, e in gemm), inter)
