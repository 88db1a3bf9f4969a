"""Convenience wrapper: PyTorch allocates the buffers, the C ABI does the work.

``MoELayer`` owns the workspace, the quantised-weight blob and the output
tensors of one layer shape and calls moe_route -> moe_schedule ->
moe_forward and moe_backward on a CUDA stream. PyTorch is used only for
device memory and streams.
"""
from __future__ import annotations

import torch

from . import (config, moe_backward, moe_dispatch, moe_forward, moe_quantize_weights, moe_route, moe_schedule, moe_status,
               moe_weights_size, moe_workspace_size, moe_ws_view, moe_wq_view, MoeError)


class MoELayer:
    def __init__(self, T, d, E, k, n_groups=1, topk_groups=1, I=128, n_shared=0, capacity=0, device="cuda",
                 flags=0, n_mover_warps=0):
        self.cfg = config(T, d, E, k, n_groups, topk_groups, I, n_shared, capacity, flags, n_mover_warps)
        self.T, self.d, self.E, self.k, self.I, self.S = T, d, E, k, I, n_shared
        dev = torch.device(device)
        self.device = dev
        self.ws = torch.zeros(moe_workspace_size(self.cfg), dtype=torch.uint8, device=dev)
        self.wq = torch.zeros(moe_weights_size(self.cfg), dtype=torch.uint8, device=dev)
        self.topk_idx = torch.empty((T, k), dtype=torch.int32, device=dev)
        self.topk_w = torch.empty((T, k), dtype=torch.float32, device=dev)
        self.y = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
        self.dx = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
        self.dw_router = torch.empty((E, d), dtype=torch.bfloat16, device=dev)
        self.dw_gu = torch.empty((E, 2 * I, d), dtype=torch.bfloat16, device=dev)
        self.dw_d = torch.empty((E, d, I), dtype=torch.bfloat16, device=dev)
        self.dws_gu = torch.empty((max(n_shared, 1), 2 * I, d), dtype=torch.bfloat16, device=dev)
        self.dws_d = torch.empty((max(n_shared, 1), d, I), dtype=torch.bfloat16, device=dev)
        self._x = self._w_router = None

    @classmethod
    def from_shape(cls, shape, device="cuda", flags=0, n_mover_warps=0):
        return cls(shape.T, shape.d, shape.E, shape.k, shape.G, shape.g_top, shape.I, shape.S, shape.C, device,
                   flags, n_mover_warps)

    # ------------------------------------------------------------ views
    def ws_tensor(self, name, dtype=torch.uint8, shape=None) -> torch.Tensor:
        ptr, n = moe_ws_view(self.cfg, self.ws.data_ptr(), name)
        off = ptr - self.ws.data_ptr()
        t = self.ws[off:off + n].view(dtype)
        return t if shape is None else t[: _numel(shape)].view(shape)

    def wq_tensor(self, name, shape=None) -> torch.Tensor:
        ptr, n = moe_wq_view(self.cfg, self.wq.data_ptr(), name)
        off = ptr - self.wq.data_ptr()
        t = self.wq[off:off + n]
        return t if shape is None else t.view(shape)

    # ------------------------------------------------------------ steps
    def quantize_weights(self, w_gu, w_d, ws_gu=None, ws_d=None, stream=0):
        moe_quantize_weights(self.cfg, w_gu.data_ptr(), w_d.data_ptr(),
                             ws_gu.data_ptr() if ws_gu is not None and self.S else 0,
                             ws_d.data_ptr() if ws_d is not None and self.S else 0, self.wq.data_ptr(), stream)

    def route(self, x, w_router, bias, stream=0):
        moe_route(self.cfg, x.data_ptr(), w_router.data_ptr(), bias.data_ptr(), self.topk_idx.data_ptr(),
                  self.topk_w.data_ptr(), self.ws.data_ptr(), stream)

    def schedule(self, stream=0):
        moe_schedule(self.cfg, self.topk_idx.data_ptr(), self.ws.data_ptr(), stream)

    def dispatch(self, x, stream=0):
        """MX(x) and the ring dispatch of every lap alone (moe_forward does this itself)."""
        moe_dispatch(self.cfg, x.data_ptr(), self.ws.data_ptr(), stream)

    def forward_experts(self, x, stream=0, y=None):
        y = self.y if y is None else y
        moe_forward(self.cfg, x.data_ptr(), self.wq.data_ptr(), self.topk_w.data_ptr(), y.data_ptr(),
                    self.ws.data_ptr(), stream)
        return y

    def forward(self, x, w_router, bias, stream=0, y=None):
        """Route, schedule and run the experts; writes y (default: self.y) and returns it."""
        self._x, self._w_router = x, w_router
        self.route(x, w_router, bias, stream)
        self.schedule(stream)
        return self.forward_experts(x, stream, y)

    def backward(self, dy, stream=0, dx=None):
        """Gradients of the last forward; writes dx (default: self.dx) and the weight gradients."""
        dx = self.dx if dx is None else dx
        moe_backward(self.cfg, self._x.data_ptr(), self._w_router.data_ptr(), self.topk_idx.data_ptr(),
                     self.topk_w.data_ptr(), dy.data_ptr(), self.wq.data_ptr(), dx.data_ptr(),
                     self.dw_router.data_ptr(), self.dw_gu.data_ptr(), self.dw_d.data_ptr(),
                     self.dws_gu.data_ptr(), self.dws_d.data_ptr(), self.ws.data_ptr(), stream)
        return dx

    def capture_step(self, x, w_router, bias, dy):
        """Record one whole step (route, schedule, forward, backward) into a CUDA graph.

        The library allocates nothing and never synchronises inside these calls,
        so the step captures as-is: 23 kernel nodes (plus the counter memsets),
        including the cooperative all-laps GEMM launches and the backward's
        side-stream branch (reverse-dispatch beside the weight gradients). Replaying the graph
        re-runs the step on whatever x, dy, w_router and bias hold at that time
        (the same device buffers). Returns the torch.cuda.CUDAGraph; call
        .replay() on it.
        """
        s = torch.cuda.Stream(device=self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(s):                 # one eager step: one-time attribute setup happens outside capture
            self.forward(x, w_router, bias, s.cuda_stream)
            self.backward(dy, s.cuda_stream)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s, capture_error_mode="thread_local"):
            self.forward(x, w_router, bias, s.cuda_stream)
            self.backward(dy, s.cuda_stream)
        torch.cuda.current_stream(self.device).wait_stream(s)
        return g

    def status(self, clear=True, stream=0):
        return moe_status(self.cfg, self.ws.data_ptr(), clear, stream)

    def check_status(self):
        code, site = self.status()
        if code:
            raise MoeError("device status (site %d)" % site, code)


def _numel(shape):
    n = 1
    for s in shape:
        n *= s
    return n
