"""Python binding of libmoe.so, the C ABI of the GB300 MoE expert layer.

Argument marshalling only: every function here forwards to the entry point of
the same name declared in include/moe.h.  Device pointers are passed as
integers (e.g. ``tensor.data_ptr()``), streams as integers (``cuda_stream``).
There is no CPU fallback: if the library cannot be built or loaded, the first
call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from ctypes import POINTER, Structure, byref, c_char_p, c_int, c_int32, c_size_t, c_uint64, c_void_p

__all__ = [
    "moe_dims", "moe_plan_t", "moe_saved_t", "moe_grads_t", "moe_opts", "MoeError",
    "moe_workspace_bytes", "moe_plan_tiles_elems", "moe_rows", "moe_plan", "moe_forward", "moe_backward",
    "moe_get_status", "moe_clear_status", "moe_strerror", "moe_version", "moe_launch_count",
    "moe_kernel_name", "moe_plan_noalloc", "moe_router_t", "moe_router_forward", "check", "lib", "lib_path",
]

MOE_OK = 0
MOE_ERR_ARG = -1
MOE_ERR_ALIGN = -2
MOE_ERR_WS = -3
MOE_ERR_LAUNCH = -4
MOE_ERR_SHAPE = -5
MOE_ERR_DEVICE = -6
MOE_ERR_TOO_LARGE = -7
MOE_NOALLOC_SCRATCH_BYTES = 4 << 20
MOE_ERR_TIMEOUT = 1
MOE_ERR_NONFINITE = 2
MOE_ERR_BOUNDS = 3


class moe_dims(Structure):
    _fields_ = [("T", c_int32), ("H", c_int32), ("F", c_int32), ("E", c_int32), ("k", c_int32), ("pad", c_int32)]


class moe_plan_t(Structure):
    _fields_ = [("topk_ids", c_void_p), ("topk_w", c_void_p), ("counts", c_void_p), ("offsets", c_void_p),
                ("dest", c_void_p), ("row_src", c_void_p), ("row_slot", c_void_p), ("tiles", c_void_p)]


class moe_saved_t(Structure):
    _fields_ = [("Xp", c_void_p), ("GU", c_void_p), ("h", c_void_p), ("Y", c_void_p)]


class moe_grads_t(Structure):
    _fields_ = [("dY", c_void_p), ("dGU", c_void_p), ("dXp", c_void_p)]


class moe_router_t(Structure):
    _fields_ = [("x", c_void_p), ("Wr", c_void_p), ("dlogits", c_void_p), ("dWr", c_void_p)]


class moe_opts(Structure):
    _fields_ = [("grid", c_int32), ("schedule", c_int32), ("events", POINTER(c_void_p)), ("n_events", c_int32),
                ("cta_pair", c_int32), ("combine", c_int32), ("debug_drop_task", c_int32),
                ("dispatch", c_int32), ("wgrad_subbatches", c_int32)]


class MoeError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {moe_strerror(code)} ({code})" if what else f"{moe_strerror(code)} ({code})")


_LIB = None
_LOCK = threading.Lock()


def lib_path() -> str:
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe.so")


def lib(path: str | None = None) -> ctypes.CDLL:
    """The loaded library; builds it first if it is missing or older than its sources.

    path: load this build of the library instead (a diagnosis build such as
    libmoe_timeline.so); only before the first load in the process."""
    global _LIB
    if _LIB is not None:
        return _LIB
    with _LOCK:
        if _LIB is None:
            if path is None:
                from . import build as _build
                if not _build.up_to_date():
                    _build.build()
            L = ctypes.CDLL(path or lib_path())
            vp = c_void_p
            sig = {
                "moe_workspace_bytes": (c_size_t, [moe_dims]),
                "moe_plan_tiles_elems": (c_size_t, [moe_dims]),
                "moe_rows": (c_size_t, [moe_dims]),
                "moe_plan": (c_int, [moe_dims, vp, POINTER(moe_plan_t), vp, c_size_t, vp]),
                "moe_forward": (c_int, [moe_dims, vp, vp, vp, vp, POINTER(moe_plan_t), POINTER(moe_saved_t), vp, vp,
                                        c_size_t, POINTER(moe_opts), vp]),
                "moe_backward": (c_int, [moe_dims, vp, vp, vp, vp, POINTER(moe_plan_t), POINTER(moe_saved_t),
                                         POINTER(moe_grads_t), vp, vp, vp, vp, vp, vp, c_size_t, POINTER(moe_opts),
                                         vp, POINTER(moe_router_t)]),
                "moe_router_forward": (c_int, [moe_dims, vp, vp, vp, vp, c_size_t, POINTER(moe_opts), vp]),
                "moe_get_status": (c_int, [vp, vp, POINTER(c_int32), POINTER(c_int32), POINTER(c_int32)]),
                "moe_clear_status": (c_int, [vp, vp]),
                "moe_strerror": (c_char_p, [c_int]),
                "moe_version": (c_int32, []),
                "moe_launch_count": (c_uint64, []),
                "moe_kernel_name": (c_char_p, [c_int32, c_int32]),
                "moe_plan_noalloc": (c_int, [moe_dims, vp, POINTER(moe_plan_t), vp, vp]),
            }
            for name, (res, args) in sig.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _LIB = L
    return _LIB


def _p(v):
    return None if v is None or v == 0 else c_void_p(int(v))


def check(rc: int, what: str = "") -> None:
    if rc != MOE_OK:
        raise MoeError(rc, what)


def moe_workspace_bytes(d: moe_dims) -> int:
    return lib().moe_workspace_bytes(d)


def moe_plan_tiles_elems(d: moe_dims) -> int:
    return lib().moe_plan_tiles_elems(d)


def moe_rows(d: moe_dims) -> int:
    return lib().moe_rows(d)


def moe_plan(d, logits, plan, ws, ws_bytes, stream=0) -> int:
    return lib().moe_plan(d, _p(logits), byref(plan), _p(ws), ws_bytes, _p(stream))


def moe_forward(d, x, W1, W3, W2, plan, saved, out, ws, ws_bytes, opts=None, stream=0) -> int:
    return lib().moe_forward(d, _p(x), _p(W1), _p(W3), _p(W2), byref(plan), byref(saved), _p(out), _p(ws),
                             ws_bytes, byref(opts) if opts is not None else None, _p(stream))


def moe_backward(d, dout, W1, W3, W2, plan, saved, grads, dx, dW1, dW3, dW2, dgate, ws, ws_bytes, opts=None,
                 stream=0, router=None) -> int:
    return lib().moe_backward(d, _p(dout), _p(W1), _p(W3), _p(W2), byref(plan), byref(saved), byref(grads), _p(dx),
                              _p(dW1), _p(dW3), _p(dW2), _p(dgate), _p(ws), ws_bytes,
                              byref(opts) if opts is not None else None, _p(stream),
                              byref(router) if router is not None else None)


def moe_router_forward(d, x, Wr, logits, ws, ws_bytes, opts=None, stream=0) -> int:
    return lib().moe_router_forward(d, _p(x), _p(Wr), _p(logits), _p(ws), ws_bytes,
                                     byref(opts) if opts is not None else None, _p(stream))


def moe_get_status(ws, stream=0):
    """Returns (rc, device_status, where, detail); synchronises the stream."""
    st, wh, de = c_int32(0), c_int32(0), c_int32(0)
    rc = lib().moe_get_status(_p(ws), _p(stream), byref(st), byref(wh), byref(de))
    return rc, st.value, wh.value, de.value


def moe_clear_status(ws, stream=0) -> int:
    return lib().moe_clear_status(_p(ws), _p(stream))


def moe_strerror(code: int) -> str:
    return lib().moe_strerror(code).decode()


def moe_version() -> int:
    return lib().moe_version()


def moe_launch_count() -> int:
    return lib().moe_launch_count()


def moe_kernel_name(call: int, i: int):
    v = lib().moe_kernel_name(call, i)
    return None if v is None else v.decode()


def moe_plan_noalloc(d, logits, plan, status, stream=0) -> int:
    return lib().moe_plan_noalloc(d, _p(logits), byref(plan), _p(status), _p(stream))
