"""The C-ABI library: it loads, exports every function include/moe.h declares,
and its host-side checks (no GPU work) behave as documented."""
import ctypes
import os
import re

import pytest

import combine_router_softmax_top_gb300 as moe
from combine_router_softmax_top_gb300 import build


@pytest.fixture(scope="module")
def L():
    build.build()
    return moe.lib()


def declared_functions():
    text = open(moe.HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_whole_path():
    names = declared_functions()
    for want in ("moe_route", "moe_dispatch_layout", "moe_permute", "moe_expert_ffn_fwd",
                 "moe_combine", "moe_combine_bwd", "moe_expert_ffn_bwd_dgrad",
                 "moe_expert_ffn_bwd_wgrad", "moe_permute_bwd", "moe_route_bwd",
                 "moe_sched_create", "moe_sched_step", "moe_sched_timings", "moe_sched_destroy"):
        assert want in names
    for want in ("moe_dispatch_fused", "moe_expert_ffn_bwd_wgrad_accum", "moe_graph_capture",
                 "moe_graph_launch", "moe_graph_kernel_count", "moe_graph_destroy"):
        assert want in names


def test_every_declared_symbol_is_exported(L):
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing
    # and the binding wraps every one of them
    assert set(declared_functions()) <= set(moe._SIGS)


def test_library_is_in_tree_and_sm103a(L):
    assert os.path.dirname(moe.LIB_PATH) == os.path.dirname(os.path.abspath(moe.__file__))
    assert L.moe_abi_version() == 2
    assert "compute_103a,code=sm_103a" in " ".join(build.ARCH)


@pytest.mark.parametrize("kw,status", [
    (dict(T=256, H=128, E=8, k=2, F=256), moe.MOE_OK),
    (dict(T=0, H=128, E=8, k=2, F=256), moe.MOE_OK),
    (dict(T=-1, H=128, E=8, k=2, F=256), moe.MOE_ERR_INVALID_ARG),
    (dict(T=16, H=128, E=8, k=9, F=256), moe.MOE_ERR_INVALID_ARG),      # k > E
    (dict(T=16, H=128, E=8, k=2, F=256, R=3), moe.MOE_ERR_INVALID_ARG),  # E % R
    (dict(T=16, H=100, E=8, k=2, F=256), moe.MOE_ERR_UNSUPPORTED),      # H % 64
    (dict(T=16, H=128, E=8, k=2, F=96), moe.MOE_ERR_UNSUPPORTED),       # F % 64
    (dict(T=16, H=128, E=300, k=2, F=256), moe.MOE_ERR_UNSUPPORTED),    # E > 256
    (dict(T=16, H=128, E=64, k=33, F=256), moe.MOE_ERR_UNSUPPORTED),    # k > 32
    (dict(T=16, H=128, E=8, k=2, F=256, mode=7), moe.MOE_ERR_INVALID_ARG),
    (dict(T=16, H=128, E=8, k=2, F=256, flags=moe.FLAG_WGRAD_ACCUM_FP32), moe.MOE_OK),
    (dict(T=16, H=128, E=8, k=2, F=256, flags=2), moe.MOE_ERR_INVALID_ARG),  # unknown flag
])
def test_descriptor_validation(L, kw, status):
    d = moe.LayerDesc.of(**kw)
    assert moe.moe_layer_desc_validate(d) == status
    if status != moe.MOE_OK:
        assert L.moe_last_error()


def test_workspace_size_covers_every_scratch_area(L):
    d = moe.LayerDesc.of(T=4096, H=2048, E=128, k=8, F=768)
    n = moe.moe_workspace_size(d)
    N = 4096 * 8
    # status words + logits + histograms + dz + router-backward partials
    assert n >= 256 + 4096 * 128 * 4 + 16 * 128 * 4 + N * 4 + (N // 64 + 128) * 2048 * 4
    with pytest.raises(moe.MoeError):
        moe.moe_workspace_size(moe.LayerDesc.of(T=1, H=100, E=8, k=2, F=256))


def test_null_and_misaligned_pointers_are_rejected_before_any_launch(L):
    d = moe.LayerDesc.of(T=16, H=128, E=8, k=2, F=256)
    st = L.moe_permute(ctypes.byref(d), None, ctypes.c_void_p(16), ctypes.c_void_p(16), None)
    assert st == moe.MOE_ERR_INVALID_ARG and b"NULL" in L.moe_last_error()
    st = L.moe_permute(ctypes.byref(d), ctypes.c_void_p(18), ctypes.c_void_p(16),
                       ctypes.c_void_p(16), None)
    assert st == moe.MOE_ERR_INVALID_ARG and b"aligned" in L.moe_last_error()
    st = L.moe_route(ctypes.byref(d), ctypes.c_void_p(16), ctypes.c_void_p(16), None, None,
                     ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16), 8, None)
    assert st == moe.MOE_ERR_INVALID_ARG and b"workspace" in L.moe_last_error()


def test_scheduler_needs_two_streams(L):
    d = moe.LayerDesc.of(T=16, H=128, E=8, k=2, F=256)
    h = ctypes.c_void_p()
    st = L.moe_sched_create(ctypes.byref(d), ctypes.c_void_p(1), ctypes.c_void_p(1), 0,
                            ctypes.byref(h))
    assert st == moe.MOE_ERR_INVALID_ARG


def _fake_bufs(d, accum=False):
    """A buffer struct of aligned, never-dereferenced addresses (host checks only)."""
    b = moe.MbBufs()
    for n in moe._MB_FIELDS + moe._MB_FIELDS_TAIL:
        setattr(b, n, 4096)
    if not accum:
        b.main_dw1 = b.main_dw2 = None
    b.ws_bytes = moe.moe_workspace_size(d)
    return b


def test_new_entry_points_check_arguments_before_any_launch(L):
    d = moe.LayerDesc.of(T=16, H=128, E=8, k=2, F=256)
    p = ctypes.c_void_p(4096)
    ws = moe.moe_workspace_size(d)
    # fused dispatch: a NULL input
    st = L.moe_dispatch_fused(ctypes.byref(d), None, p, None, None, p, p, p, p, p, p, p, p, p, p,
                              ws, None)
    assert st == moe.MOE_ERR_INVALID_ARG and b"NULL" in L.moe_last_error()
    # accumulating wgrad: a NULL main gradient, then a misaligned one
    st = L.moe_expert_ffn_bwd_wgrad_accum(ctypes.byref(d), p, p, p, p, p, None, p, p, ws, None)
    assert st == moe.MOE_ERR_INVALID_ARG and b"NULL" in L.moe_last_error()
    st = L.moe_expert_ffn_bwd_wgrad_accum(ctypes.byref(d), p, p, p, p, p, ctypes.c_void_p(4100),
                                          p, p, ws, None)
    assert st == moe.MOE_ERR_INVALID_ARG and b"aligned" in L.moe_last_error()


def test_accumulating_layer_needs_main_gradients_not_bf16_ones(L):
    d = moe.LayerDesc.of(T=16, H=128, E=8, k=2, F=256, flags=moe.FLAG_WGRAD_ACCUM_FP32)
    b = _fake_bufs(d, accum=True)
    b.dw1 = b.dw2 = None  # unused when accumulating: NULL is allowed
    b.main_dw1 = None     # but the main gradients are required
    st = L.moe_layer_backward(ctypes.byref(d), ctypes.byref(b), 1, None)
    assert st == moe.MOE_ERR_INVALID_ARG and b"NULL" in L.moe_last_error()


def test_graph_capture_checks_arguments_before_any_cuda_call(L):
    d = moe.LayerDesc.of(T=16, H=128, E=8, k=2, F=256)
    b = _fake_bufs(d)
    h = ctypes.c_void_p()
    st = L.moe_graph_capture(ctypes.byref(d), ctypes.byref(b), moe.GRAPH_LAYER_STEP,
                             ctypes.c_void_p(64), None)
    assert st == moe.MOE_ERR_INVALID_ARG  # no place for the result
    st = L.moe_graph_capture(ctypes.byref(d), ctypes.byref(b), 9, ctypes.c_void_p(64),
                             ctypes.byref(h))
    assert st == moe.MOE_ERR_INVALID_ARG and b"scope" in L.moe_last_error() and not h.value
    st = L.moe_graph_capture(ctypes.byref(d), ctypes.byref(b), moe.GRAPH_LAYER_STEP, None,
                             ctypes.byref(h))
    assert st == moe.MOE_ERR_INVALID_ARG and b"default stream" in L.moe_last_error()
    assert L.moe_graph_launch(None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_graph_kernel_count(None) == 0
    L.moe_graph_destroy(None)  # a no-op


def test_expert_parallel_and_pipelined_entry_points_check_arguments(L):
    d = moe.LayerDesc.of(T=16, H=128, E=8, k=2, F=256, R=2)
    p = ctypes.c_void_p(4096)
    # the EP re-sort: NULL counts, a negative row count, in place, a bad direction
    assert L.moe_ep_resort(ctypes.byref(d), None, p, ctypes.c_void_p(8192), None, 4, 0,
                           None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_ep_resort(ctypes.byref(d), p, p, ctypes.c_void_p(8192), None, -1, 0,
                           None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_ep_resort(ctypes.byref(d), p, p, p, None, 4, 0, None) == moe.MOE_ERR_INVALID_ARG
    assert b"in place" in L.moe_last_error()
    assert L.moe_ep_resort(ctypes.byref(d), p, p, ctypes.c_void_p(8192), None, 4, 2,
                           None) == moe.MOE_ERR_INVALID_ARG
    # the pipelined host steps: the two buffer sets must not share x, dy, y or dx
    b = _fake_bufs(d)
    arr = (moe.MbBufs * 2)(b, b)
    ptrs = (ctypes.c_void_p * 1)(4096)
    st = L.moe_layer_steps_host(ctypes.byref(d), arr, 1, ptrs, ptrs, ptrs, ptrs, None)
    assert st == moe.MOE_ERR_INVALID_ARG and b"own x" in L.moe_last_error()
    b2 = _fake_bufs(d)
    b2.x, b2.dy, b2.y, b2.dx = 8192, 8192 + 4096, 8192 + 8192, 8192 + 12288
    arr = (moe.MbBufs * 2)(b, b2)
    assert L.moe_layer_steps_host(ctypes.byref(d), arr, -1, ptrs, ptrs, ptrs,
                                  ptrs, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_layer_steps_host(ctypes.byref(d), arr, 0, None, None, None, None,
                                  None) == moe.MOE_OK  # nothing to do
    nul = (ctypes.c_void_p * 1)(None)
    st = L.moe_layer_steps_host(ctypes.byref(d), arr, 1, ptrs, nul, ptrs, ptrs, None)
    assert st == moe.MOE_ERR_INVALID_ARG and b"step 0" in L.moe_last_error()


def test_barrier_wait_limit_round_trips(L):
    old = moe.moe_set_barrier_wait_limit_ns(12345)
    try:
        assert moe.moe_set_barrier_wait_limit_ns(0) == 12345
        assert moe.moe_set_barrier_wait_limit_ns(0) == 2_000_000_000  # 0 restores the default
    finally:
        moe.moe_set_barrier_wait_limit_ns(old)
