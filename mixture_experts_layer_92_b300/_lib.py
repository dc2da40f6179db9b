"""ctypes binding of libmoe (include/moe.h): argument marshalling only.

Every function here passes torch tensors' device pointers, sizes and the current CUDA
stream to the C ABI of the same name. No step of the layer runs in Python or PyTorch.
If libmoe.so is missing the import of this module fails loudly; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe.so")

MOE_OK = 0
MOE_ERR_NONFINITE = -6
STATUS = {0: "MOE_OK", -1: "MOE_ERR_INVALID", -2: "MOE_ERR_UNSUPPORTED", -3: "MOE_ERR_CUDA",
          -4: "MOE_ERR_WORKSPACE", -5: "MOE_ERR_TIMEOUT", -6: "MOE_ERR_NONFINITE"}
GATE_MODES = {"softmax_all": 0, "softmax_topk": 1, "sigmoid_topk": 2, "expert_choice": 3}
DTYPES = {torch.float32: 0, torch.bfloat16: 1}
NUM_STAGES = 8
STAGE_NAMES = ("router_gemm", "gates_topk", "dispatch", "gather", "gemm_gateup_swiglu",
               "gemm_down_scale", "combine", "aux_loss")

EXPORTED = ("moe_capacity", "moe_check_shape", "moe_workspace_size", "moe_route_topk",
            "moe_dispatch", "moe_grouped_swiglu", "moe_combine", "moe_aux_loss", "moe_forward",
            "moe_forward_events", "moe_get_error", "moe_clear_error", "moe_status_string",
            "moe_last_error_detail", "moe_route_topk_noalloc", "moe_route_topk_balanced",
            "moe_update_select_bias", "moe_forward_balanced", "moe_expert_choice",
            "moe_grouped_swiglu_fp8w", "moe_forward_fp8w", "moe_backward_workspace_size",
            "moe_backward", "moe_selftest_wait_timeout", "moe_forward_host",
            "moe_host_pipeline_buffer_size", "moe_host_pipeline_create",
            "moe_host_pipeline_forward", "moe_host_pipeline_join", "moe_host_pipeline_destroy",
            "moe_mx_workspace_size", "moe_forward_mx", "moe_mx_quantize",
            "moe_workspace_dispatch_offsets")
MX_FORMATS = {"e4m3": 0, "e2m1": 1}
NUM_BWD_STAGES = 8
BWD_STAGE_NAMES = ("route_dispatch", "gather_x_dy", "recompute_gu", "gemm_dh_swiglu_bwd",
                   "gate_logit_grads", "gemm_dx", "dx_combine", "gemm_wgrad")


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({detail})")


class moe_shape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("d_ff", ctypes.c_int32), ("d_ff_shared", ctypes.c_int32),
                ("capacity", ctypes.c_int32), ("gate", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("alpha", ctypes.c_float), ("beta", ctypes.c_float)]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmoe.so is not built ({LIB_PATH}); run "
                          "`python -m mixture_experts_layer_92_b300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, sz, dbl = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_double
    sp = ctypes.POINTER(moe_shape)
    sig = {
        "moe_capacity": (ctypes.c_int, [dbl, i32, i32, i32]),
        "moe_check_shape": (ctypes.c_int, [sp]),
        "moe_workspace_size": (sz, [sp]),
        "moe_route_topk": (ctypes.c_int, [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "moe_dispatch": (ctypes.c_int, [sp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "moe_grouped_swiglu": (ctypes.c_int, [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                              vp, sz, vp]),
        "moe_combine": (ctypes.c_int, [sp, vp, vp, vp, vp, vp]),
        "moe_aux_loss": (ctypes.c_int, [sp, vp, vp, vp, vp]),
        "moe_forward": (ctypes.c_int, [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                       vp, sz, vp]),
        "moe_forward_events": (ctypes.c_int, [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                              vp, vp, sz, vp, ctypes.POINTER(vp), ctypes.c_int]),
        "moe_workspace_dispatch_offsets": (ctypes.c_int, [sp, ctypes.POINTER(sz),
                                                          ctypes.POINTER(sz), ctypes.POINTER(sz)]),
        "moe_get_error": (ctypes.c_int, [vp, vp]),
        "moe_clear_error": (ctypes.c_int, [vp, vp]),
        "moe_selftest_wait_timeout": (ctypes.c_int, [vp, sz, vp]),
        "moe_forward_host": (ctypes.c_int, [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                            vp, sz, vp]),
        "moe_host_pipeline_buffer_size": (sz, [sp]),
        "moe_host_pipeline_create": (ctypes.c_int, [sp, vp, sz, ctypes.POINTER(vp)]),
        "moe_host_pipeline_forward": (ctypes.c_int, [vp, sp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                                     vp, vp, vp, sz, vp]),
        "moe_host_pipeline_join": (ctypes.c_int, [vp, vp]),
        "moe_host_pipeline_destroy": (ctypes.c_int, [vp]),
        "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "moe_last_error_detail": (ctypes.c_char_p, []),
        "moe_route_topk_noalloc": (ctypes.c_int, [sp, vp, vp, vp, vp, vp]),
        "moe_route_topk_balanced": (ctypes.c_int, [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz,
                                                   vp]),
        "moe_update_select_bias": (ctypes.c_int, [sp, vp, vp, ctypes.c_float, vp]),
        "moe_expert_choice": (ctypes.c_int, [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz,
                                             vp]),
        "moe_grouped_swiglu_fp8w": (ctypes.c_int, [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                                   vp, sz, vp]),
        "moe_forward_fp8w": (ctypes.c_int, [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                            vp, sz, vp, ctypes.POINTER(vp), ctypes.c_int]),
        "moe_forward_balanced": (ctypes.c_int, [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                                vp, vp, ctypes.c_float, vp, sz, vp,
                                                ctypes.POINTER(vp), ctypes.c_int]),
        "moe_mx_workspace_size": (sz, [sp]),
        "moe_forward_mx": (ctypes.c_int, [sp, ctypes.c_int, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                          vp, vp, vp, vp, sz, vp, ctypes.POINTER(vp),
                                          ctypes.c_int]),
        "moe_mx_quantize": (ctypes.c_int, [vp, ctypes.c_int64, i32, vp, vp, vp, vp]),
        "moe_backward_workspace_size": (sz, [sp]),
        "moe_backward": (ctypes.c_int, [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float,
                                        ctypes.c_float, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                        vp, sz, vp, ctypes.POINTER(vp), ctypes.c_int]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


LIB = _load()


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        if not torch.cuda.is_available():
            return ctypes.c_void_p(None)
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(rc: int, where: str):
    if rc != MOE_OK:
        raise MoeError(rc, where, LIB.moe_last_error_detail().decode())


def make_shape(T, d, E, k, d_ff, gate="softmax_topk", dtype=torch.bfloat16, capacity=None,
               d_ff_shared=0, alpha=0.01, beta=1e-3) -> moe_shape:
    """capacity None means no drop (C = T)."""
    return moe_shape(T=T, d=d, E=E, k=k, d_ff=d_ff, d_ff_shared=d_ff_shared,
                     capacity=T if capacity is None else capacity,
                     gate=GATE_MODES[gate] if isinstance(gate, str) else int(gate),
                     dtype=DTYPES[dtype] if isinstance(dtype, torch.dtype) else int(dtype),
                     alpha=alpha, beta=beta)


def moe_capacity(cf: float, T: int, k: int, E: int) -> int:
    return LIB.moe_capacity(cf, T, k, E)


def moe_check_shape(s: moe_shape) -> int:
    return LIB.moe_check_shape(ctypes.byref(s))


def moe_workspace_size(s: moe_shape) -> int:
    return LIB.moe_workspace_size(ctypes.byref(s))


def alloc_workspace(s: moe_shape, device="cuda") -> torch.Tensor:
    """Zero-filled uint8 device buffer of moe_workspace_size bytes (zero = no error)."""
    n = moe_workspace_size(s)
    if n == 0:
        _check(moe_check_shape(s), "moe_workspace_size")
    ws = torch.zeros(n + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    return ws[off:off + n]


def moe_workspace_dispatch_offsets(s: moe_shape):
    """Byte offsets of perm, inv and offsets (the forward's dispatch results) in a workspace."""
    po, io, oo = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(LIB.moe_workspace_dispatch_offsets(ctypes.byref(s), ctypes.byref(po), ctypes.byref(io),
                                              ctypes.byref(oo)), "moe_workspace_dispatch_offsets")
    return po.value, io.value, oo.value


def workspace_dispatch(s: moe_shape, ws: torch.Tensor):
    """Views (int32) of the perm [T*k], inv [T*k] and offsets [E+1] a forward left in `ws`."""
    po, io, oo = moe_workspace_dispatch_offsets(s)
    A = s.T * s.k

    def view(off, n):
        return ws[off:off + 4 * n].view(torch.int32)

    return view(po, A), view(io, A), view(oo, s.E + 1)


def moe_backward_workspace_size(s: moe_shape) -> int:
    return LIB.moe_backward_workspace_size(ctypes.byref(s))


def alloc_workspace_backward(s: moe_shape, device="cuda") -> torch.Tensor:
    """Zero-filled uint8 device buffer of moe_backward_workspace_size bytes."""
    n = moe_backward_workspace_size(s)
    if n == 0:
        raise MoeError(-2, "moe_backward_workspace_size", "shape not supported by the backward pass")
    ws = torch.zeros(n + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    return ws[off:off + n]


def moe_backward(s, ws, x, w_router, w1, w3, w2, dy, dx, dw_router, dw1, dw3, dw2,
                 router_bias=None, w1s=None, w3s=None, w2s=None, d_aux=1.0, d_z=1.0,
                 d_router_bias=None, dw1s=None, dw3s=None, dw2s=None, dlogits=None, dgate=None,
                 stream=None, events=None):
    arr = None if events is None else _event_array(events)
    _check(LIB.moe_backward(ctypes.byref(s), _p(x), _p(w_router), _p(router_bias), _p(w1), _p(w3),
                            _p(w2), _p(w1s), _p(w3s), _p(w2s), _p(dy), float(d_aux), float(d_z),
                            _p(dx), _p(dw_router), _p(d_router_bias), _p(dw1), _p(dw3), _p(dw2),
                            _p(dw1s), _p(dw3s), _p(dw2s), _p(dlogits), _p(dgate), _p(ws), ws.numel(),
                            _stream(stream), arr, 0 if events is None else len(events)),
           "moe_backward")


def moe_route_topk(s, ws, topk_idx, topk_gate, x=None, w_router=None, router_bias=None,
                   logits_in=None, logits_out=None, stats=None, stream=None):
    _check(LIB.moe_route_topk(ctypes.byref(s), _p(x), _p(w_router), _p(router_bias), _p(logits_in),
                              _p(logits_out), _p(topk_idx), _p(topk_gate), _p(stats), _p(ws),
                              ws.numel(), _stream(stream)), "moe_route_topk")


def moe_dispatch(s, ws, counts, offsets, perm, inv, dropped, topk_idx=None, logits_in=None,
                 stream=None):
    _check(LIB.moe_dispatch(ctypes.byref(s), _p(topk_idx), _p(logits_in), _p(counts), _p(offsets),
                            _p(perm), _p(inv), _p(dropped), _p(ws), ws.numel(), _stream(stream)),
           "moe_dispatch")


def moe_grouped_swiglu(s, ws, x, perm, offsets, w1, w3, w2, y_perm, topk_gate=None, w1s=None,
                       w3s=None, w2s=None, y_shared=None, stream=None):
    _check(LIB.moe_grouped_swiglu(ctypes.byref(s), _p(x), _p(perm), _p(offsets), _p(topk_gate),
                                  _p(w1), _p(w3), _p(w2), _p(w1s), _p(w3s), _p(w2s), _p(y_perm),
                                  _p(y_shared), _p(ws), ws.numel(), _stream(stream)),
           "moe_grouped_swiglu")


def moe_combine(s, y_perm, inv, y, y_shared=None, stream=None):
    _check(LIB.moe_combine(ctypes.byref(s), _p(y_perm), _p(inv), _p(y_shared), _p(y),
                           _stream(stream)), "moe_combine")


def moe_aux_loss(s, stats, counts, losses, stream=None):
    _check(LIB.moe_aux_loss(ctypes.byref(s), _p(stats), _p(counts), _p(losses), _stream(stream)),
           "moe_aux_loss")


def moe_forward(s, ws, x, w_router, w1, w3, w2, y, router_bias=None, w1s=None, w3s=None, w2s=None,
                counts=None, dropped=None, losses=None, stream=None, events=None):
    if events is None:
        _check(LIB.moe_forward(ctypes.byref(s), _p(x), _p(w_router), _p(router_bias), _p(w1), _p(w3),
                               _p(w2), _p(w1s), _p(w3s), _p(w2s), _p(y), _p(counts), _p(dropped),
                               _p(losses), _p(ws), ws.numel(), _stream(stream)), "moe_forward")
        return
    arr = _event_array(events)
    _check(LIB.moe_forward_events(ctypes.byref(s), _p(x), _p(w_router), _p(router_bias), _p(w1),
                                  _p(w3), _p(w2), _p(w1s), _p(w3s), _p(w2s), _p(y), _p(counts),
                                  _p(dropped), _p(losses), _p(ws), ws.numel(), _stream(stream),
                                  arr, len(events)), "moe_forward_events")


def moe_route_topk_noalloc(s, logits_in, topk_idx, topk_gate, stats=None, stream=None):
    """moe_route_topk on precomputed logits with no workspace (scratch inside the library)."""
    _check(LIB.moe_route_topk_noalloc(ctypes.byref(s), _p(logits_in), _p(topk_idx), _p(topk_gate),
                                      _p(stats), _stream(stream)), "moe_route_topk_noalloc")


def moe_route_topk_balanced(s, ws, topk_idx, topk_gate, select_bias, x=None, w_router=None,
                            router_bias=None, logits_in=None, logits_out=None, stats=None,
                            stream=None):
    _check(LIB.moe_route_topk_balanced(ctypes.byref(s), _p(x), _p(w_router), _p(router_bias),
                                       _p(logits_in), _p(select_bias), _p(logits_out),
                                       _p(topk_idx), _p(topk_gate), _p(stats), _p(ws), ws.numel(),
                                       _stream(stream)), "moe_route_topk_balanced")


def moe_expert_choice(s, ws, perm, offsets, row_gate, inv, counts, unrouted, x=None,
                      w_router=None, router_bias=None, logits_in=None, stats=None, stream=None):
    _check(LIB.moe_expert_choice(ctypes.byref(s), _p(x), _p(w_router), _p(router_bias),
                                 _p(logits_in), _p(perm), _p(offsets), _p(row_gate), _p(inv),
                                 _p(counts), _p(unrouted), _p(stats), _p(ws), ws.numel(),
                                 _stream(stream)), "moe_expert_choice")


def moe_grouped_swiglu_fp8w(s, ws, x, perm, offsets, w1q, w1_scale, w3q, w3_scale, w2q, w2_scale,
                            y_perm, topk_gate=None, stream=None):
    _check(LIB.moe_grouped_swiglu_fp8w(ctypes.byref(s), _p(x), _p(perm), _p(offsets),
                                       _p(topk_gate), _p(w1q), _p(w1_scale), _p(w3q), _p(w3_scale),
                                       _p(w2q), _p(w2_scale), _p(y_perm), _p(ws), ws.numel(),
                                       _stream(stream)), "moe_grouped_swiglu_fp8w")


def moe_forward_fp8w(s, ws, x, w_router, w1q, w1_scale, w3q, w3_scale, w2q, w2_scale, y,
                     router_bias=None, counts=None, dropped=None, losses=None, stream=None,
                     events=None):
    arr = None if events is None else _event_array(events)
    _check(LIB.moe_forward_fp8w(ctypes.byref(s), _p(x), _p(w_router), _p(router_bias), _p(w1q),
                                _p(w1_scale), _p(w3q), _p(w3_scale), _p(w2q), _p(w2_scale), _p(y),
                                _p(counts), _p(dropped), _p(losses), _p(ws), ws.numel(),
                                _stream(stream), arr, 0 if events is None else len(events)),
           "moe_forward_fp8w")


def moe_mx_workspace_size(s: moe_shape) -> int:
    return LIB.moe_mx_workspace_size(ctypes.byref(s))


def alloc_workspace_mx(s: moe_shape, device="cuda") -> torch.Tensor:
    """Zero-filled uint8 device buffer of moe_mx_workspace_size bytes."""
    n = moe_mx_workspace_size(s)
    if n == 0:
        _check(moe_check_shape(s), "moe_mx_workspace_size")
    ws = torch.zeros(n + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    return ws[off:off + n]


def moe_forward_mx(s, ws, fmt, x, w_router, w1q, w1_scales, w3q, w3_scales, w2q, w2_scales, y,
                   router_bias=None, counts=None, dropped=None, losses=None, stream=None,
                   events=None):
    """moe_forward on block-scaled expert weights (fmt "e4m3" or "e2m1")."""
    arr = None if events is None else _event_array(events)
    f = MX_FORMATS[fmt] if isinstance(fmt, str) else int(fmt)
    _check(LIB.moe_forward_mx(ctypes.byref(s), f, _p(x), _p(w_router), _p(router_bias), _p(w1q),
                              _p(w1_scales), _p(w3q), _p(w3_scales), _p(w2q), _p(w2_scales),
                              _p(y), _p(counts), _p(dropped), _p(losses), _p(ws), ws.numel(),
                              _stream(stream), arr, 0 if events is None else len(events)),
           "moe_forward_mx")


def moe_mx_quantize(x, codes, scales, ws=None, stream=None):
    """E4M3 blocks of 32 of the bf16 rows x [rows, K]: codes [rows, K] uint8, scale bytes
    [rows, K / 32] uint8 (s + 127)."""
    rows, K = x.shape
    _check(LIB.moe_mx_quantize(_p(x), rows, K, _p(codes), _p(scales), _p(ws), _stream(stream)),
           "moe_mx_quantize")


def moe_update_select_bias(s, counts, select_bias, gamma, stream=None):
    _check(LIB.moe_update_select_bias(ctypes.byref(s), _p(counts), _p(select_bias), gamma,
                                      _stream(stream)), "moe_update_select_bias")


def _event_array(events):
    """cudaEvent_t handles of torch events; None stays NULL (no event at that boundary)."""
    for e in events:
        if e is not None and e.cuda_event == 0:   # torch creates the CUDA event on first record
            e.record()
    return (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(None if e is None else e.cuda_event)
                                            for e in events])


def moe_forward_balanced(s, ws, x, w_router, w1, w3, w2, y, select_bias, gamma, router_bias=None,
                         w1s=None, w3s=None, w2s=None, counts=None, dropped=None, losses=None,
                         stream=None, events=None):
    arr = None if events is None else _event_array(events)
    _check(LIB.moe_forward_balanced(ctypes.byref(s), _p(x), _p(w_router), _p(router_bias), _p(w1),
                                    _p(w3), _p(w2), _p(w1s), _p(w3s), _p(w2s), _p(y), _p(counts),
                                    _p(dropped), _p(losses), _p(select_bias), gamma, _p(ws),
                                    ws.numel(), _stream(stream), arr,
                                    0 if events is None else len(events)), "moe_forward_balanced")


def moe_get_error(ws, stream=None) -> int:
    return LIB.moe_get_error(_p(ws), _stream(stream))


def moe_clear_error(ws, stream=None):
    _check(LIB.moe_clear_error(_p(ws), _stream(stream)), "moe_clear_error")


def moe_forward_host(s, ws, x_host, w_router, w1, w3, w2, y_host, x_dev, y_dev, router_bias=None,
                     w1s=None, w3s=None, w2s=None, losses_host=None, stream=None):
    """The layer from and to host memory (pinned host tensors x_host, y_host; device scratch
    x_dev, y_dev of the same shape); see include/moe.h."""
    _check(LIB.moe_forward_host(ctypes.byref(s), _p(x_host), _p(w_router), _p(router_bias),
                                _p(w1), _p(w3), _p(w2), _p(w1s), _p(w3s), _p(w2s), _p(y_host),
                                _p(losses_host), _p(x_dev), _p(y_dev), _p(ws), ws.numel(),
                                _stream(stream)), "moe_forward_host")


class HostPipeline:
    """Handle of a moe_host_pipeline (see include/moe.h): a stream of pinned host batches
    through one layer, uploads and downloads on the pipeline's own streams overlapping the
    layers on the caller's stream. `s_max` fixes d, dtype and the largest T; the slot buffers
    are one torch allocation on `device`, held by this object."""

    def __init__(self, s_max, device=None):
        n = LIB.moe_host_pipeline_buffer_size(ctypes.byref(s_max))
        if n == 0:
            _check(LIB.moe_check_shape(ctypes.byref(s_max)), "moe_host_pipeline_buffer_size")
        self.buf = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
        h = ctypes.c_void_p()
        _check(LIB.moe_host_pipeline_create(ctypes.byref(s_max), _p(self.buf), self.buf.numel(),
                                            ctypes.byref(h)), "moe_host_pipeline_create")
        self._h = h

    def forward(self, s, ws, x_host, w_router, w1, w3, w2, y_host, router_bias=None, w1s=None,
                w3s=None, w2s=None, losses_host=None, stream=None):
        _check(LIB.moe_host_pipeline_forward(self._h, ctypes.byref(s), _p(x_host), _p(w_router),
                                             _p(router_bias), _p(w1), _p(w3), _p(w2), _p(w1s),
                                             _p(w3s), _p(w2s), _p(y_host), _p(losses_host),
                                             _p(ws), ws.numel(), _stream(stream)),
               "moe_host_pipeline_forward")

    def join(self, stream=None):
        _check(LIB.moe_host_pipeline_join(self._h, _stream(stream)), "moe_host_pipeline_join")

    def close(self):
        if self._h is not None and self._h.value is not None:
            h, self._h = self._h, None
            _check(LIB.moe_host_pipeline_destroy(h), "moe_host_pipeline_destroy")

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def moe_selftest_wait_timeout(ws, stream=None):
    """Runs the bounded-wait diagnostic on `ws` (see include/moe.h); read the result with
    moe_get_error."""
    _check(LIB.moe_selftest_wait_timeout(_p(ws), ws.numel(), _stream(stream)),
           "moe_selftest_wait_timeout")


def moe_status_string(status: int) -> str:
    return LIB.moe_status_string(status).decode()
