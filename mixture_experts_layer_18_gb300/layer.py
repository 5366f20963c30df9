"""Caller-side buffers for the C ABI, allocated with PyTorch.

PyTorch supplies device memory and the stream handle; every computation is a
call into libmoe_gb300.so through the binding in ``__init__``.  A ``MoELayer``
owns the routing arrays, the saved activations and the three workspaces of
one problem shape, and raises ``MoEError`` on any non-OK return code.
"""
from __future__ import annotations

import torch

from . import (MOE_BF16, MOE_F32, MOE_FP8_BWD, MOE_MXFP8, MOE_OK, MOE_WS_BACKWARD,
               MOE_WS_FORWARD, MOE_WS_ROUTE, MoEError, moe_backward, moe_dims, moe_forward,
               moe_max_rows, moe_route, moe_route_backward, moe_route_out, moe_saved_layout_of,
               moe_workspace_size)

MODES = {"f32": MOE_F32, "bf16": MOE_BF16, "mxfp8": MOE_MXFP8, "fp8_bwd": MOE_FP8_BWD}


def _ptr(t):
    return t.data_ptr() if t is not None and t.numel() > 0 else None


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


class MoELayer:
    """Buffers of one (T, H, E, I, top_k, mode) problem on one device."""

    def __init__(self, T, H, E, I, top_k, mode="bf16", save_for_backward=True,
                 device="cuda", backward=True):
        self.dims = moe_dims(T, H, E, I, top_k, MODES[mode], 1 if save_for_backward else 0)
        self.mode = mode
        self.T, self.H, self.E, self.I, self.k = T, H, E, I, top_k
        self.dtype = torch.float32 if mode == "f32" else torch.bfloat16
        self.device = torch.device(device)
        rows = moe_max_rows(self.dims)
        if rows < 0:
            raise MoEError(1, "invalid dims")
        self.max_rows = rows
        dev = self.device
        i32 = dict(dtype=torch.int32, device=dev)
        self.topk_idx = torch.empty((T, top_k), **i32)
        self.gate = torch.empty((T, top_k), dtype=torch.float32, device=dev)
        self.counts = torch.empty(E, **i32)
        self.offsets = torch.empty(E + 1, **i32)
        self.padded_offsets = torch.empty(E + 1, **i32)
        self.row_of_assign = torch.empty(T * top_k, **i32)
        self.assign_of_row = torch.empty(rows, **i32)
        self.route_out = moe_route_out(
            _ptr(self.topk_idx), _ptr(self.gate), _ptr(self.counts), _ptr(self.offsets),
            _ptr(self.padded_offsets), _ptr(self.row_of_assign), _ptr(self.assign_of_row))
        u8 = dict(dtype=torch.uint8, device=dev)
        self.ws_route = torch.empty(moe_workspace_size(self.dims, MOE_WS_ROUTE), **u8)
        self.ws_fwd = torch.empty(moe_workspace_size(self.dims, MOE_WS_FORWARD), **u8)
        self.ws_bwd = torch.empty(moe_workspace_size(self.dims, MOE_WS_BACKWARD) if backward else 0,
                                  **u8)
        self.layout = moe_saved_layout_of(self.dims)
        self.saved = torch.empty(self.layout.total, **u8)
        self.status = torch.zeros(4, **i32)

    # ------------------------------------------------------------- views
    def _view(self, offset, rows, cols):
        es = 4 if self.dtype == torch.float32 else 2
        n = rows * cols * es
        return self.saved[offset:offset + n].view(self.dtype).view(rows, cols)

    @property
    def x_perm(self):
        """Gathered tokens [rows, H]; None in mxfp8 mode (not stored)."""
        if self.mode == "mxfp8":
            return None
        return self._view(self.layout.x_perm, self.max_rows, self.H)

    @property
    def act_is_gated(self):
        """bf16 mode stores gate * A in `act` (see moe.h)."""
        return self.mode == "bf16"

    @property
    def h13(self):
        return self._view(self.layout.h13, self.max_rows, 2 * self.I)

    @property
    def act(self):
        """The activation [rows, I] (gate * A in bf16 mode); None in mxfp8
        mode, which keeps A only as its MXFP8 encodings."""
        if self.mode == "mxfp8":
            return None
        return self._view(self.layout.act, self.max_rows, self.I)

    def device_status(self) -> int:
        return int(self.status[0].item())

    def clear_status(self):
        self.status.zero_()

    # ------------------------------------------------------------- calls
    def route(self, logits, stream=None):
        rc = moe_route(self.dims, _ptr(logits), self.route_out, _ptr(self.ws_route),
                       self.ws_route.numel(), _ptr(self.status), _stream(stream))
        if rc != MOE_OK:
            raise MoEError(rc, "moe_route")

    def forward(self, X, W13, W2, Y, stream=None, save=None):
        """save: None = the layer's setting; False = inference / checkpointed
        first pass (h13 not kept); True = keep h13 for moe_backward."""
        dims = self.dims
        if save is not None and bool(save) != bool(self.dims.save_for_backward):
            dims = moe_dims(self.dims.T, self.dims.H, self.dims.E, self.dims.I, self.dims.top_k,
                            self.dims.mode, 1 if save else 0)
        rc = moe_forward(dims, _ptr(X), _ptr(W13), _ptr(W2), self.route_out, _ptr(Y),
                         _ptr(self.saved), self.saved.numel(), _ptr(self.ws_fwd),
                         self.ws_fwd.numel(), _ptr(self.status), _stream(stream))
        if rc != MOE_OK:
            raise MoEError(rc, "moe_forward")

    def backward(self, dY, W13, W2, dX, dW13, dW2, dgate, stream=None):
        rc = moe_backward(self.dims, _ptr(dY), _ptr(W13), _ptr(W2), self.route_out,
                          _ptr(self.saved), self.saved.numel(), _ptr(dX), _ptr(dW13), _ptr(dW2),
                          _ptr(dgate), _ptr(self.ws_bwd), self.ws_bwd.numel(),
                          _ptr(self.status), _stream(stream))
        if rc != MOE_OK:
            raise MoEError(rc, "moe_backward")

    def route_backward(self, dgate, dlogits, stream=None):
        rc = moe_route_backward(self.dims, self.route_out, _ptr(dgate), _ptr(dlogits),
                                _ptr(self.status), _stream(stream))
        if rc != MOE_OK:
            raise MoEError(rc, "moe_route_backward")

    # --------------------------------------------------------- allocation
    def empty_io(self):
        """Output tensors of one forward + backward: Y, dX, dW13, dW2, dgate."""
        dev, dt = self.device, self.dtype
        return dict(
            Y=torch.empty((self.T, self.H), dtype=dt, device=dev),
            dX=torch.empty((self.T, self.H), dtype=dt, device=dev),
            dW13=torch.empty((self.E, self.H, 2 * self.I), dtype=dt, device=dev),
            dW2=torch.empty((self.E, self.I, self.H), dtype=dt, device=dev),
            dgate=torch.empty((self.T, self.k), dtype=torch.float32, device=dev),
        )
