"""The key that ties committed ncu counters to kernel sources ignores comments
and blank lines but changes with any code edit."""
import importlib.util
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    argv = sys.argv
    try:
        sys.argv = ["bench.py"]
        spec.loader.exec_module(mod)
    finally:
        sys.argv = argv
    return mod


def test_digest_ignores_comments_not_code():
    b = _bench()
    csrc = os.path.join(ROOT, "combine_router_softmax_top_gb300", "csrc")
    files = {f: open(os.path.join(csrc, f), encoding="utf-8").read()
             for f in b.KERNEL_SOURCES["gemm"]}
    base = b.source_digest("gemm_ffn_dgrad", files.__getitem__)
    assert base == b.source_digest("gemm_ffn_dgrad")
    commented = dict(files)
    commented["grouped_gemm.cu"] = ("// a new line comment\n/* and a\n block one */\n\n"
                                    + files["grouped_gemm.cu"].replace("\n", "  // note\n", 3))
    assert b.source_digest("gemm_ffn_dgrad", commented.__getitem__) == base
    edited = dict(files)
    edited["grouped_gemm.cu"] = files["grouped_gemm.cu"].replace("BK = 64", "BK = 32", 1)
    assert edited["grouped_gemm.cu"] != files["grouped_gemm.cu"]
    assert b.source_digest("gemm_ffn_dgrad", edited.__getitem__) != base

