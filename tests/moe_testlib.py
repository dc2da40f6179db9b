"""Helpers shared by the GPU parity tests and bench.py: run the CUDA path through the C ABI
binding, and compute the oracle's answer for the same inputs (all of it, or sampled
tokens of a full-size workload)."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
from mixture_experts_layer_92_b300 import _lib as L


def host64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def capacity_of(w) -> int:
    return w.T if w.cf is None else O.capacity(w.cf, w.T, w.k, w.E)


def shape_of(w, C=None, T=None):
    dtype = torch.float32 if w.dtype == "f32" else torch.bfloat16
    T = w.T if T is None else T
    return L.make_shape(T, w.d, w.E, w.k, w.d_ff, gate=w.gate, dtype=dtype,
                        capacity=capacity_of(w) if C is None else C,
                        d_ff_shared=w.d_ff_shared, alpha=w.alpha, beta=w.beta)


def gpu_forward(w, inp: dict, C=None, route_too: bool = True) -> dict:
    """moe_forward on device inputs; optionally also moe_route_topk (logits_out) for the
    routing comparisons."""
    s = shape_of(w, C)
    dev = inp["x"].device
    ws = L.alloc_workspace(s, device=dev)
    y = torch.empty_like(inp["x"])
    counts = torch.zeros(w.E, dtype=torch.int32, device=dev)
    dropped = torch.zeros(1, dtype=torch.int32, device=dev)
    losses = torch.zeros(2, dtype=torch.float32, device=dev)
    L.moe_forward(s, ws, inp["x"], inp["w_router"], inp["w1"], inp["w3"], inp["w2"], y,
                  router_bias=inp["router_bias"], w1s=inp["w1s"], w3s=inp["w3s"], w2s=inp["w2s"],
                  counts=counts, dropped=dropped, losses=losses)
    out = dict(y=y, counts=counts, dropped=dropped, losses=losses, ws=ws, shape=s)
    if route_too:
        T = w.T
        logits = torch.empty(T, w.E, dtype=torch.float32, device=dev)
        idx = torch.empty(T, w.k, dtype=torch.int32, device=dev)
        gate = torch.empty(T, w.k, dtype=torch.float32, device=dev)
        stats = torch.empty(w.E + 1, dtype=torch.float32, device=dev)
        L.moe_route_topk(s, ws, idx, gate, x=inp["x"], w_router=inp["w_router"],
                         router_bias=inp["router_bias"], logits_out=logits, stats=stats)
        out.update(logits=logits, idx=idx, gate=gate, stats=stats)
    torch.cuda.synchronize()
    out["error"] = L.moe_get_error(ws)
    return out


def routing_check(logits64: np.ndarray, gpu_idx: np.ndarray, k: int, eps: float = 1e-3):
    """Oracle top-k on fp64 logits vs the GPU's; returns (mismatching tokens, near-tie
    tokens). Mismatches are allowed only among near ties."""
    o_idx = O.select_topk(logits64, k)
    bad = np.nonzero(np.any(np.sort(o_idx, 1) != np.sort(gpu_idx, 1), axis=1))[0]
    ties = O.near_tie_tokens(logits64, k, eps)
    return bad, ties


def oracle_y_for_tokens(w, inp: dict, logits64: np.ndarray, gpu_idx: np.ndarray,
                        gpu_inv: np.ndarray, tokens: np.ndarray) -> np.ndarray:
    """Oracle output rows y[tokens] given the routing decisions (idx, and inv = the dispatch
    of those decisions over all tokens). Gates come from the oracle's fp64 logits. Expert
    weights are copied to the host one expert at a time."""
    k = w.k
    idx_s = gpu_idx[tokens]
    inv_s = gpu_inv.reshape(-1, k)[tokens]
    g = O.gates(logits64[tokens], idx_s, w.gate)
    x64 = host64(inp["x"][torch.as_tensor(tokens, device=inp["x"].device)])
    n = len(tokens)
    inv_local = np.full((n, k), -1, dtype=np.int64)
    rows = []
    for e in np.unique(idx_s[inv_s >= 0]):
        mask = (idx_s == e) & (inv_s >= 0)
        tl, sl = np.nonzero(mask)
        out = O.swiglu_ffn(x64[tl], host64(inp["w1"][e]), host64(inp["w3"][e]), host64(inp["w2"][e]))
        base = sum(r.shape[0] for r in rows)
        inv_local[tl, sl] = base + np.arange(len(tl))
        rows.append(out)
    rows = np.concatenate(rows, 0) if rows else np.zeros((0, w.d))
    shared = None
    if inp.get("w1s") is not None:
        shared = O.swiglu_ffn(x64, host64(inp["w1s"]), host64(inp["w3s"]), host64(inp["w2s"]))
    return O.combine(g, inv_local, rows, n, k, shared)


def rel_l2(a: np.ndarray, b: np.ndarray) -> float:
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))
