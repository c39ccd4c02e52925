"""Device buffers of one layer step, allocated with PyTorch, driven through the C ABI.

PyTorch only provides memory and the stream here; every step of the layer runs
in libmoe.so's kernels.
"""
from __future__ import annotations

import torch

from . import (check, moe_backward, moe_dims, moe_forward, moe_get_status, moe_grads_t, moe_opts, moe_plan,
               moe_plan_t, moe_plan_tiles_elems, moe_router_forward, moe_router_t, moe_rows, moe_saved_t,
               moe_workspace_bytes)


def _empty(shape, dtype, device):
    n = 1
    for s in shape:
        n *= s
    # An empty tensor still gets a valid (non-null, aligned) pointer.
    return torch.empty(max(n, 16), dtype=dtype, device=device)[:n].view(*shape)


class MoELayer:
    """Buffers of plan, forward and backward for fixed (T, H, F, E, k).

    pad >= 2 selects the static-shape variant: every expert's rows are padded to
    a multiple of pad, and the grouped buffers hold moe_rows(dims) rows."""

    def __init__(self, T, H, F, E, k, device="cuda", with_backward=True, plan_only=False, with_router=False, pad=0):
        self.dims = moe_dims(T, H, F, E, k, pad)
        self.T, self.H, self.F, self.E, self.k, self.pad = T, H, F, E, k, pad
        R = moe_rows(self.dims)
        if R == 0 and T * k > 0:
            raise ValueError("invalid layer dimensions")
        self.R = R
        dev = torch.device(device)
        self.device = dev
        i32, f32, bf = torch.int32, torch.float32, torch.bfloat16
        ws_bytes = moe_workspace_bytes(self.dims)
        if ws_bytes == 0:
            raise ValueError("invalid layer dimensions")
        self.ws_bytes = ws_bytes
        self.ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
        n_tiles = moe_plan_tiles_elems(self.dims)
        self.ids = _empty((T, k), i32, dev)
        self.w = _empty((T, k), f32, dev)
        self.counts = torch.empty(E, dtype=i32, device=dev)
        self.offsets = torch.empty(E + 1, dtype=i32, device=dev)
        self.dest = _empty((T, k), i32, dev)
        self.row_src = _empty((R,), i32, dev)
        self.row_slot = _empty((R,), torch.uint8, dev)
        self.tiles = torch.zeros(n_tiles, dtype=i32, device=dev)
        self.plan_s = moe_plan_t(self.ids.data_ptr(), self.w.data_ptr(), self.counts.data_ptr(),
                                 self.offsets.data_ptr(), self.dest.data_ptr(), self.row_src.data_ptr(),
                                 self.row_slot.data_ptr(), self.tiles.data_ptr())
        if with_router:  # the router on the path: logits from x Wr, and their gradients
            self.logits = _empty((T, E), f32, dev)
            self.dlogits = _empty((T, E), f32, dev)
            self.dWr = torch.empty((H, E), dtype=f32, device=dev)
        if plan_only:  # routing tables only (profiling the routing kernels)
            return
        self.Xp = _empty((R, H), bf, dev)
        self.GU = _empty((R, 2 * F), bf, dev)
        self.h = _empty((R, F), bf, dev)
        self.Y = _empty((R, H), bf, dev)
        self.out = _empty((T, H), bf, dev)
        self.saved = moe_saved_t(self.Xp.data_ptr(), self.GU.data_ptr(), self.h.data_ptr(), self.Y.data_ptr())
        if with_backward:
            self.dY = _empty((R, H), bf, dev)
            self.dGU = _empty((R, 2 * F), bf, dev)
            self.dXp = _empty((R, H), bf, dev)
            self.grads = moe_grads_t(self.dY.data_ptr(), self.dGU.data_ptr(), self.dXp.data_ptr())
            self.dx = _empty((T, H), bf, dev)
            self.dW1 = torch.empty((E, H, F), dtype=f32, device=dev)
            self.dW3 = torch.empty((E, H, F), dtype=f32, device=dev)
            self.dW2 = torch.empty((E, F, H), dtype=f32, device=dev)
            self.dgate = _empty((T, k), f32, dev)

    @staticmethod
    def _stream(stream):
        if stream is None:
            stream = torch.cuda.current_stream()
        return stream.cuda_stream

    def opts(self, grid=0, events=None, schedule=0, cta_pair=0, combine=0, debug_drop_task=0, wgrad_subbatches=0,
             dispatch=0):
        o = moe_opts()
        o.grid = grid
        o.schedule = schedule
        o.cta_pair = cta_pair
        o.combine = combine
        o.debug_drop_task = debug_drop_task
        o.wgrad_subbatches = wgrad_subbatches
        o.dispatch = dispatch
        if events:
            arr = (ctypes_void_p_array(len(events)))(*[e.cuda_event for e in events])
            self._ev_keep = arr
            o.events = arr
            o.n_events = len(events) // 2
        return o

    def plan(self, logits, stream=None):
        check(moe_plan(self.dims, logits.data_ptr(), self.plan_s, self.ws.data_ptr(), self.ws_bytes,
                       self._stream(stream)), "moe_plan")

    def forward(self, x, W1, W3, W2, opts=None, stream=None, out=None):
        """out: a [T, H] bf16 tensor to write the layer output to (default self.out)."""
        out = self.out if out is None else out
        check(moe_forward(self.dims, x.data_ptr(), W1.data_ptr(), W3.data_ptr(), W2.data_ptr(), self.plan_s,
                          self.saved, out.data_ptr(), self.ws.data_ptr(), self.ws_bytes, opts,
                          self._stream(stream)), "moe_forward")
        return out

    def backward(self, dout, W1, W3, W2, opts=None, stream=None, router=None, dx=None):
        """router: (x, Wr) to carry the gradient on through the gating (dlogits, dWr, dx's router share).
        dx: a [T, H] bf16 tensor to write the input gradient to (default self.dx)."""
        dx = self.dx if dx is None else dx
        r = None
        if router is not None:
            x, Wr = router
            r = moe_router_t(x.data_ptr(), Wr.data_ptr(), self.dlogits.data_ptr(), self.dWr.data_ptr())
        check(moe_backward(self.dims, dout.data_ptr(), W1.data_ptr(), W3.data_ptr(), W2.data_ptr(), self.plan_s,
                           self.saved, self.grads, dx.data_ptr(), self.dW1.data_ptr(), self.dW3.data_ptr(),
                           self.dW2.data_ptr(), self.dgate.data_ptr(), self.ws.data_ptr(), self.ws_bytes, opts,
                           self._stream(stream), r), "moe_backward")
        return dx

    def router_forward(self, x, Wr, opts=None, stream=None):
        """logits = x Wr (fp32) into self.logits."""
        check(moe_router_forward(self.dims, x.data_ptr(), Wr.data_ptr(), self.logits.data_ptr(), self.ws.data_ptr(),
                                 self.ws_bytes, opts, self._stream(stream)), "moe_router_forward")
        return self.logits

    def status(self, stream=None):
        rc, st, where, detail = moe_get_status(self.ws.data_ptr(), self._stream(stream))
        check(rc, "moe_get_status")
        return st, where, detail


def ctypes_void_p_array(n):
    import ctypes
    return ctypes.c_void_p * n
