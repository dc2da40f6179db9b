"""B300-native forward pass of one Mixture-of-Experts layer.

The computation runs in libmoe.so (hand-written CUDA for sm_103a behind a C ABI,
include/moe.h). This package is its thin ctypes binding (``_lib``) plus ``MoELayer``, a
convenience holder of the layer's weights and workspace whose ``forward`` is one call of
``moe_forward``. PyTorch only provides device memory and streams.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import _lib
from ._lib import (MoeError, alloc_workspace, make_shape, moe_aux_loss, moe_capacity,  # noqa: F401
                   moe_check_shape, moe_clear_error, moe_combine, moe_dispatch, moe_forward,
                   moe_forward_balanced, moe_forward_fp8w, moe_get_error, moe_grouped_swiglu,
                   moe_grouped_swiglu_fp8w, moe_route_topk,
                   moe_route_topk_balanced, moe_route_topk_noalloc, moe_status_string,
                   moe_update_select_bias, moe_workspace_size, NUM_STAGES, STAGE_NAMES,
                   alloc_workspace_backward, moe_backward, moe_backward_workspace_size,
                   moe_forward_host, HostPipeline, alloc_workspace_mx, moe_forward_mx,
                   moe_mx_quantize, moe_mx_workspace_size)


class MoELayer:
    """Weights (device tensors) + shape + workspace of one MoE layer.

    w_router [E, d]; w1, w3 [E, d_ff, d]; w2 [E, d, d_ff]; optional router_bias [E] fp32 and
    shared expert w1s, w3s [d_ff_shared, d], w2s [d, d_ff_shared]. ``capacity`` None means
    no drop.
    """

    def __init__(self, w_router, w1, w3, w2, *, k: int, gate: str, capacity: Optional[int] = None,
                 router_bias=None, w1s=None, w3s=None, w2s=None, alpha=0.01, beta=1e-3,
                 max_tokens: int, balance_gamma: Optional[float] = None, fp8: Optional[dict] = None,
                 mx: Optional[dict] = None):
        E, d = w_router.shape
        self.w = dict(w_router=w_router, w1=w1, w3=w3, w2=w2, router_bias=router_bias,
                      w1s=w1s, w3s=w3s, w2s=w2s)
        if w1 is not None:
            d_ff = w1.shape[1]
        elif fp8 is not None:
            d_ff = fp8["w1q"].shape[1]
        else:
            d_ff = mx["w1q"].shape[1]
        self.E, self.d, self.k, self.d_ff = E, d, k, d_ff
        self.d_ff_shared = 0 if w1s is None else w1s.shape[0]
        self.gate, self.capacity, self.alpha, self.beta = gate, capacity, alpha, beta
        self.dtype = w_router.dtype
        self.device = w_router.device
        self.max_tokens = max_tokens
        # block-scaled expert weights: dict(fmt, w1q, w1sf, w3q, w3sf, w2q, w2sf) (codes and
        # scale atoms, see moe_forward_mx)
        self.mx = mx
        self.ws = (alloc_workspace_mx if mx is not None else alloc_workspace)(
            self.shape(max_tokens), device=self.device)
        self.counts = torch.zeros(E, dtype=torch.int32, device=self.device)
        self.dropped = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.losses = torch.zeros(2, dtype=torch.float32, device=self.device)
        # 8-bit expert weights: dict(w1q, w1s, w3q, w3s, w2q, w2s) (E4M3 codes + per-row scales)
        self.fp8 = fp8
        # auxiliary-loss-free balancing: a selection bias nudged by gamma after every forward
        self.balance_gamma = balance_gamma
        self.select_bias = (torch.zeros(E, dtype=torch.float32, device=self.device)
                            if balance_gamma is not None else None)

    def shape(self, T: int):
        return make_shape(T, self.d, self.E, self.k, self.d_ff, gate=self.gate, dtype=self.dtype,
                          capacity=self.capacity, d_ff_shared=self.d_ff_shared, alpha=self.alpha,
                          beta=self.beta)

    def forward(self, x: torch.Tensor, y: Optional[torch.Tensor] = None, stream=None, events=None):
        """y = MoE(x) for device x [T, d]; counts, dropped and losses stay on the device."""
        T = x.shape[0]
        if y is None:
            y = torch.empty_like(x)
        if self.mx is not None:
            m = self.mx
            moe_forward_mx(self.shape(T), self.ws, m["fmt"], x, self.w["w_router"], m["w1q"],
                           m["w1sf"], m["w3q"], m["w3sf"], m["w2q"], m["w2sf"], y,
                           router_bias=self.w["router_bias"], counts=self.counts,
                           dropped=self.dropped, losses=self.losses, stream=stream, events=events)
            return y
        if self.fp8 is not None:
            q = self.fp8
            moe_forward_fp8w(self.shape(T), self.ws, x, self.w["w_router"], q["w1q"], q["w1s"],
                             q["w3q"], q["w3s"], q["w2q"], q["w2s"], y,
                             router_bias=self.w["router_bias"], counts=self.counts,
                             dropped=self.dropped, losses=self.losses, stream=stream, events=events)
            return y
        if self.select_bias is not None:
            moe_forward_balanced(self.shape(T), self.ws, x, self.w["w_router"], self.w["w1"],
                                 self.w["w3"], self.w["w2"], y, self.select_bias,
                                 self.balance_gamma, router_bias=self.w["router_bias"],
                                 w1s=self.w["w1s"], w3s=self.w["w3s"], w2s=self.w["w2s"],
                                 counts=self.counts, dropped=self.dropped, losses=self.losses,
                                 stream=stream, events=events)
            return y
        moe_forward(self.shape(T), self.ws, x, self.w["w_router"], self.w["w1"], self.w["w3"],
                    self.w["w2"], y, router_bias=self.w["router_bias"], w1s=self.w["w1s"],
                    w3s=self.w["w3s"], w2s=self.w["w2s"], counts=self.counts,
                    dropped=self.dropped, losses=self.losses, stream=stream, events=events)
        return y

    def route(self, x: torch.Tensor) -> torch.Tensor:
        """Top-k expert indices [T, k] int32 of device x: moe_route_topk with this layer's
        router (selection on the logits alone, without a balancing bias)."""
        T = x.shape[0]
        idx = torch.empty(T, self.k, dtype=torch.int32, device=self.device)
        gate = torch.empty(T, self.k, dtype=torch.float32, device=self.device)
        moe_route_topk(self.shape(T), self.ws, idx, gate, x=x, w_router=self.w["w_router"],
                       router_bias=self.w["router_bias"])
        return idx

    def forward_host_stream(self, x_hosts, y_hosts, losses_hosts=None):
        """End-to-end layer over a sequence of host batches (pinned memory), pipelined.

        Plain bf16/fp32 layers go through the C ABI's host pipeline (moe_host_pipeline): each
        batch's x is uploaded on the pipeline's upload stream, the layer runs on the current
        stream and y (and, if losses_hosts is given, the batch's two losses) come back on its
        download stream, so the upload of batch i+1 and the download of batch i-1 overlap the
        layer on batch i. The current stream waits for every download. Returns after queuing
        all work. (8-bit-weight, block-scaled and balanced layers copy through torch around
        their own forward calls instead.)"""
        if self.fp8 is not None or self.mx is not None or self.select_bias is not None:
            return self._forward_host_stream_copies(x_hosts, y_hosts)
        comp = torch.cuda.current_stream(self.device)
        if getattr(self, "_host_pipe", None) is None:
            self._host_pipe = HostPipeline(self.shape(self.max_tokens), device=self.device)
        for i, (xh, yh) in enumerate(zip(x_hosts, y_hosts)):
            self._host_pipe.forward(self.shape(xh.shape[0]), self.ws, xh, self.w["w_router"],
                               self.w["w1"], self.w["w3"], self.w["w2"], yh,
                               router_bias=self.w["router_bias"], w1s=self.w["w1s"],
                               w3s=self.w["w3s"], w2s=self.w["w2s"],
                               losses_host=None if losses_hosts is None else losses_hosts[i],
                               stream=comp)
        self._host_pipe.join(comp)
        return y_hosts

    def _forward_host_stream_copies(self, x_hosts, y_hosts):
        """forward_host_stream for the layer variants without a host entry point: batch i's
        x is copied to the device on one stream, the layer runs on the current stream, and y
        is copied back on a third; two device buffer pairs let the upload of batch i+1 and the
        download of batch i-1 overlap the layer on batch i."""
        comp = torch.cuda.current_stream(self.device)
        if getattr(self, "_copy_pipe", None) is None:
            self._copy_pipe = dict(h2d=torch.cuda.Stream(self.device), d2h=torch.cuda.Stream(self.device),
                              xbuf=[None, None], ybuf=[None, None],
                              h2d_done=[torch.cuda.Event(), torch.cuda.Event()],
                              fwd_done=[torch.cuda.Event(), torch.cuda.Event()],
                              d2h_done=[torch.cuda.Event(), torch.cuda.Event()])
        p = self._copy_pipe
        for i, (xh, yh) in enumerate(zip(x_hosts, y_hosts)):
            b = i % 2
            if p["xbuf"][b] is None or p["xbuf"][b].shape[0] < xh.shape[0]:
                p["xbuf"][b] = torch.empty(xh.shape, dtype=xh.dtype, device=self.device)
                p["ybuf"][b] = torch.empty(xh.shape, dtype=xh.dtype, device=self.device)
            xd, yd = p["xbuf"][b][:xh.shape[0]], p["ybuf"][b][:xh.shape[0]]
            if i >= 2:
                p["h2d"].wait_event(p["fwd_done"][b])      # x buffer b free
            with torch.cuda.stream(p["h2d"]):
                xd.copy_(xh, non_blocking=True)
                p["h2d_done"][b].record(p["h2d"])
            comp.wait_event(p["h2d_done"][b])
            if i >= 2:
                comp.wait_event(p["d2h_done"][b])          # y buffer b free
            self.forward(xd, yd, stream=comp)
            p["fwd_done"][b].record(comp)
            p["d2h"].wait_event(p["fwd_done"][b])
            with torch.cuda.stream(p["d2h"]):
                yh.copy_(yd, non_blocking=True)
                p["d2h_done"][b].record(p["d2h"])
        comp.wait_stream(p["d2h"])
        return y_hosts

    def device_error(self) -> int:
        """The device error status recorded in this layer's workspace (0 if none).
        Synchronises with the device."""
        return moe_get_error(self.ws)

    def forward_host(self, x_host: torch.Tensor, x_dev: torch.Tensor, y_dev: torch.Tensor,
                     y_host: torch.Tensor, losses_host: Optional[torch.Tensor] = None):
        """End-to-end call from host memory: copy x (pinned) to the device, run the layer,
        copy y (and the two losses) back, all on the current stream. Plain bf16/fp32 layers
        make this one moe_forward_host call (counts, dropped and losses then stay in the
        workspace; losses_host receives the losses); 8-bit and balanced layers copy through
        torch around their forward call."""
        if self.fp8 is None and self.mx is None and self.select_bias is None:
            moe_forward_host(self.shape(x_host.shape[0]), self.ws, x_host, self.w["w_router"],
                             self.w["w1"], self.w["w3"], self.w["w2"], y_host, x_dev, y_dev,
                             router_bias=self.w["router_bias"], w1s=self.w["w1s"],
                             w3s=self.w["w3s"], w2s=self.w["w2s"], losses_host=losses_host,
                             stream=torch.cuda.current_stream(self.device))
            return y_host
        x_dev.copy_(x_host, non_blocking=True)
        self.forward(x_dev, y_dev)
        y_host.copy_(y_dev, non_blocking=True)
        if losses_host is not None:
            losses_host.copy_(self.losses, non_blocking=True)
        return y_host
