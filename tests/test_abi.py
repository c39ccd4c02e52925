"""The C ABI library builds, loads without a GPU, exports every entry point
include/moe.h declares, and rejects bad arguments on the host (no GPU call)."""
import ctypes
import os
import re

import pytest

import mixture_experts_layer_gb300 as M

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moe.h")


def declared():
    src = open(HEADER).read()
    return re.findall(r"^MOE_API\s+[\w\s\*]+?\**\s*(moe_\w+)\s*\(", src, flags=re.M)


def test_every_declared_symbol_is_exported():
    names = declared()
    assert len(names) >= 11
    L = M.lib()
    for n in names:
        assert hasattr(L, n), n
        assert hasattr(M, n), f"binding lacks {n}"
    assert M.moe_version() >= 1
    assert M.moe_kernel_name(1, 1) == "gemm_fwd1_swiglu"
    assert M.moe_kernel_name(1, 2) == "gemm_fwd2"
    assert M.moe_kernel_name(7, 2) == "gemm_fwd2_combine"
    assert M.moe_kernel_name(3, 0) == "fused_forward"
    assert M.moe_kernel_name(2, 5) == "gemm_wgrad2"
    assert M.moe_kernel_name(2, 6) is None
    assert M.moe_kernel_name(4, 1) == "fused_backward"
    assert M.moe_kernel_name(8, 4) == "subbatch_rows"
    assert M.moe_kernel_name(8, 8) == "gemm_wgrad2_sb1"
    assert M.moe_kernel_name(8, 9) is None
    assert M.moe_kernel_name(9, 11) == "gemm_wgrad2_sb1"
    assert M.moe_kernel_name(10, 0) == "gemm_fwd1_gather_swiglu"
    assert M.moe_kernel_name(11, 1) == "gemm_fwd2_combine"
    assert M.moe_kernel_name(11, 2) is None


def test_workspace_sizes():
    for T, H, F, E, k in [(256, 128, 256, 8, 2), (4096, 2048, 1408, 64, 6), (131072, 4096, 1536, 128, 8)]:
        d = M.moe_dims(T, H, F, E, k)
        assert M.moe_workspace_bytes(d) > 0
        assert M.moe_plan_tiles_elems(d) >= (T * k) // 128 * 4
    assert M.moe_workspace_bytes(M.moe_dims(16, 128, 128, 4, 5)) == 0   # k > E
    assert M.moe_workspace_bytes(M.moe_dims(16, 100, 128, 4, 2)) == 0   # H % 128
    assert M.moe_workspace_bytes(M.moe_dims(16, 128, 128, 2048, 2)) == 0  # E too large
    assert M.moe_workspace_bytes(M.moe_dims(16, 128, 128, 64, 33)) == 0   # k > 32
    # grouped rows: T*k, or with padding granule P, T*k + min(E, T*k) * (P - 1)
    assert M.moe_rows(M.moe_dims(4096, 2048, 1408, 64, 6)) == 4096 * 6
    assert M.moe_rows(M.moe_dims(4096, 2048, 1408, 64, 6, 1)) == 4096 * 6
    assert M.moe_rows(M.moe_dims(4096, 2048, 1408, 64, 6, 128)) == 4096 * 6 + 64 * 127
    assert M.moe_rows(M.moe_dims(1, 128, 128, 8, 2, 16)) == 2 + 2 * 15
    assert M.moe_rows(M.moe_dims(16, 128, 128, 4, 2, -1)) == 0
    assert M.moe_rows(M.moe_dims(16, 128, 128, 4, 2, 4097)) == 0
    for pad in (0, 128):
        d = M.moe_dims(4096, 2048, 1408, 64, 6, pad)
        assert M.moe_plan_tiles_elems(d) >= M.moe_rows(d) // 128 * 4 + 2 * 64


def test_host_side_rejections():
    d = M.moe_dims(16, 128, 128, 4, 2)
    plan = M.moe_plan_t()
    ws = ctypes.create_string_buffer(M.moe_workspace_bytes(d) + 64)
    base = ctypes.addressof(ws)
    aligned = (base + 15) & ~15
    n = M.moe_workspace_bytes(d)
    assert M.moe_plan(d, aligned, plan, 0, n) == M.MOE_ERR_ARG            # no workspace
    assert M.moe_plan(d, aligned, plan, aligned + 4, n) == M.MOE_ERR_ALIGN  # misaligned workspace
    assert M.moe_plan(d, aligned, plan, aligned, n - 1) == M.MOE_ERR_WS     # too small
    assert M.moe_plan(d, aligned, plan, aligned, n) == M.MOE_ERR_ARG        # plan fields are null
    bad = M.moe_dims(16, 128, 128, 4, 0)
    assert M.moe_plan(bad, aligned, plan, aligned, n) == M.MOE_ERR_ARG
    assert M.moe_plan(M.moe_dims(16, 96, 128, 4, 2), aligned, plan, aligned, n) == M.MOE_ERR_SHAPE
    assert "aligned" in M.moe_strerror(M.MOE_ERR_ALIGN)
    # option checks of moe_backward come before any device work
    args = (d, aligned, aligned, aligned, aligned, M.moe_plan_t(), M.moe_saved_t(), M.moe_grads_t(), aligned, aligned,
            aligned, aligned, aligned, aligned, n)
    for sched, sb in ((2, 2), (0, 3), (0, -1)):
        o = M.moe_opts()
        o.schedule, o.wgrad_subbatches = sched, sb
        assert M.moe_backward(*args, opts=o) == M.MOE_ERR_ARG, (sched, sb)


def test_timeline_diagnosis_build_exports_its_hook():
    """The pipeline timeline (-DMOE_TIMELINE) builds into a library of its own that exports
    moe_debug_timeline, and the product library does not export it."""
    import subprocess
    import sys
    from mixture_experts_layer_gb300 import build as B
    out = os.path.join(os.path.dirname(B.LIB), "libmoe_timeline.so")
    path = B.build(defines=("MOE_TIMELINE",), out=out)
    # Load it in a child process: this process keeps the product library.
    code = ("import ctypes, sys; L = ctypes.CDLL(sys.argv[1]); "
            "print(hasattr(L, 'moe_debug_timeline'), hasattr(L, 'moe_plan'))")
    r = subprocess.run([sys.executable, "-c", code, path], capture_output=True, text=True, timeout=120)
    assert r.stdout.split() == ["True", "True"], r.stdout + r.stderr
    assert not hasattr(M.lib(), "moe_debug_timeline")
