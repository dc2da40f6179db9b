"""Parity of the backward pass at the full workload sizes, in the launch configuration
`bench.py --backward` times (one moe_backward call), on outputs the oracle computes piece by
piece:

* weight gradients of sampled hidden units of two experts (the most loaded one and a
  seeded other): dW1[e][f], dW3[e][f] and dW2[e][:, f] depend on unit f alone (dH[:, f] =
  dout . W2[:, f]), so the oracle's SwiGLU backward on those units' slices of the weights
  gives exactly those rows / columns;
* dx, the gate gradients and the logit gradients of sampled tokens: each token's kept rows
  through the oracle's full SwiGLU backward, its gates' Jacobian, the balance-loss and
  z-loss gradients (computed over all tokens), the router and the shared expert.

The GPU's own routing decisions are used on the oracle side (top-k parity is tested
elsewhere); the bf16 bound (relative L2 <= 2e-2) applies as in the small cases."""
import numpy as np
import pytest
import torch

import oracle as O
from moe_inputs import WORKLOADS, make_inputs
from moe_testlib import capacity_of, host64, rel_l2

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = "cuda:0"
TOL = 2e-2


@pytest.mark.parametrize("name", ["mixtral_prefill", "deepseek_fine", "switch_top1",
                                  "mixtral_decode"])
def test_full_size_backward(name):
    from mixture_experts_layer_92_b300 import _lib as L
    w = WORKLOADS[name]
    inp = make_inputs(w, device=DEV)
    C = capacity_of(w)
    gen = torch.Generator(device=DEV).manual_seed(11)
    dy = torch.randn(inp["x"].shape, generator=gen, device=DEV).to(torch.bfloat16)
    s = L.make_shape(w.T, w.d, w.E, w.k, w.d_ff, gate=w.gate, dtype=torch.bfloat16, capacity=C,
                     d_ff_shared=w.d_ff_shared, alpha=w.alpha, beta=w.beta)
    ws = L.alloc_workspace_backward(s, DEV)
    f32 = dict(device=DEV, dtype=torch.float32)
    g = dict(dx=torch.empty_like(inp["x"]), dw_router=torch.empty((w.E, w.d), **f32),
             dw1=torch.empty((w.E, w.d_ff, w.d), **f32), dw3=torch.empty((w.E, w.d_ff, w.d), **f32),
             dw2=torch.empty((w.E, w.d, w.d_ff), **f32), dlogits=torch.empty((w.T, w.E), **f32),
             dgate=torch.empty((w.T, w.k), **f32))
    if w.d_ff_shared:
        g.update(dw1s=torch.empty((w.d_ff_shared, w.d), **f32),
                 dw3s=torch.empty((w.d_ff_shared, w.d), **f32),
                 dw2s=torch.empty((w.d, w.d_ff_shared), **f32))
    L.moe_backward(s, ws, inp["x"], inp["w_router"], inp["w1"], inp["w3"], inp["w2"], dy,
                   g["dx"], g["dw_router"], g["dw1"], g["dw3"], g["dw2"],
                   router_bias=inp["router_bias"], w1s=inp["w1s"], w3s=inp["w3s"], w2s=inp["w2s"],
                   dw1s=g.get("dw1s"), dw3s=g.get("dw3s"), dw2s=g.get("dw2s"),
                   dlogits=g["dlogits"], dgate=g["dgate"])
    idx = torch.empty(w.T, w.k, dtype=torch.int32, device=DEV)
    gate = torch.empty(w.T, w.k, device=DEV)
    L.moe_route_topk(s, L.alloc_workspace(s, DEV), idx, gate, x=inp["x"], w_router=inp["w_router"],
                     router_bias=inp["router_bias"])
    torch.cuda.synchronize()
    assert L.moe_get_error(ws) == 0

    x64, dy64 = host64(inp["x"]), host64(dy)
    wr64 = host64(inp["w_router"])
    bias = None if inp["router_bias"] is None else host64(inp["router_bias"])
    logits64 = O.router_logits(x64, wr64, bias)
    gidx = idx.cpu().numpy().astype(np.int64)
    disp = O.dispatch(gidx, w.E, C)
    gates64 = O.gates(logits64, gidx, w.gate)
    gflat = gates64.reshape(-1)
    offs, perm = disp["offsets"], disp["perm"]
    rng = np.random.default_rng(3)

    # weight gradients: sampled hidden units of two experts
    kept = np.diff(offs)
    experts = sorted({int(np.argmax(kept)), int(rng.choice(np.nonzero(kept)[0]))})
    for e in experts:
        a = perm[offs[e]:offs[e + 1]]
        toks = a // w.k
        fs = np.sort(rng.choice(w.d_ff, size=16, replace=False))
        fs_t = torch.as_tensor(fs, device=DEV)
        w1e = host64(inp["w1"][e][fs_t])
        w3e = host64(inp["w3"][e][fs_t])
        w2e = host64(inp["w2"][e][:, fs_t])
        r = O.swiglu_ffn_backward(x64[toks], w1e, w3e, w2e, gflat[a][:, None] * dy64[toks])
        assert rel_l2(g["dw1"][e][fs_t].double().cpu().numpy(), r["dw1"]) < TOL, ("dw1", e)
        assert rel_l2(g["dw3"][e][fs_t].double().cpu().numpy(), r["dw3"]) < TOL, ("dw3", e)
        assert rel_l2(g["dw2"][e][:, fs_t].double().cpu().numpy(), r["dw2"]) < TOL, ("dw2", e)

    # sampled tokens: dgate, dlogits, dx
    tokens = np.sort(rng.choice(w.T, size=min(w.T, 6), replace=False))
    dl_bal = (O.aux_loss_backward(logits64, gidx, w.alpha) + O.z_loss_backward(logits64, w.beta))
    dx_ref, dl_ref, dg_ref = [], [], []
    cache = {}

    def expert64(e):
        if e not in cache:
            cache[e] = (host64(inp["w1"][e]), host64(inp["w3"][e]), host64(inp["w2"][e]))
        return cache[e]

    for t in tokens:
        dxt = np.zeros(w.d)
        dgt = np.zeros(w.k)
        for sl in range(w.k):
            r_ = disp["inv"][t * w.k + sl]
            if r_ < 0:
                continue
            e = int(gidx[t, sl])
            w1e, w3e, w2e = expert64(e)
            rb = O.swiglu_ffn_backward(x64[t:t + 1], w1e, w3e, w2e, gates64[t, sl] * dy64[t:t + 1])
            dxt += rb["dx"][0]
            dgt[sl] = float(dy64[t] @ (rb["H"][0] @ w2e.T))
        dlt = O.gate_backward(logits64[t:t + 1], gidx[t:t + 1], w.gate, dgt[None])[0] + dl_bal[t]
        dxt += dlt @ wr64
        if w.d_ff_shared:
            dxt += O.swiglu_ffn_backward(x64[t:t + 1], host64(inp["w1s"]), host64(inp["w3s"]),
                                         host64(inp["w2s"]), dy64[t:t + 1])["dx"][0]
        dx_ref.append(dxt)
        dl_ref.append(dlt)
        dg_ref.append(dgt)
    tt = torch.as_tensor(tokens, device=DEV)
    assert rel_l2(g["dgate"][tt].double().cpu().numpy(), np.array(dg_ref)) < TOL
    assert rel_l2(g["dlogits"][tt].double().cpu().numpy(), np.array(dl_ref)) < TOL
    err = rel_l2(g["dx"][tt].double().cpu().numpy(), np.array(dx_ref))
    print(f"{name}: sampled dx rel L2 = {err:.3e}")
    assert err < TOL
    del inp, g, ws
    torch.cuda.empty_cache()


def test_full_size_backward_expert_choice():
    """The Mixtral prefill layer with expert-choice routing (C = T k / E = 1024 tokens per
    expert), checked like the top-k layers: sampled hidden units of two experts, and the
    gradients of sampled tokens through every expert that chose them (the oracle runs on the
    GPU's own choices; the balance loss has no gradient under expert choice)."""
    from mixture_experts_layer_92_b300 import _lib as L
    w = WORKLOADS["mixtral_prefill"].scaled(gate="expert_choice", cf=1.0)
    inp = make_inputs(w, device=DEV)
    C = capacity_of(w)
    R = w.E * min(C, w.T)
    gen = torch.Generator(device=DEV).manual_seed(12)
    dy = torch.randn(inp["x"].shape, generator=gen, device=DEV).to(torch.bfloat16)
    s = L.make_shape(w.T, w.d, w.E, w.k, w.d_ff, gate=w.gate, dtype=torch.bfloat16, capacity=C,
                     alpha=w.alpha, beta=w.beta)
    ws = L.alloc_workspace_backward(s, DEV)
    f32 = dict(device=DEV, dtype=torch.float32)
    g = dict(dx=torch.empty_like(inp["x"]), dw_router=torch.empty((w.E, w.d), **f32),
             dw1=torch.empty((w.E, w.d_ff, w.d), **f32), dw3=torch.empty((w.E, w.d_ff, w.d), **f32),
             dw2=torch.empty((w.E, w.d, w.d_ff), **f32), dlogits=torch.empty((w.T, w.E), **f32),
             dgate=torch.empty((R,), **f32))
    L.moe_backward(s, ws, inp["x"], inp["w_router"], inp["w1"], inp["w3"], inp["w2"], dy,
                   g["dx"], g["dw_router"], g["dw1"], g["dw3"], g["dw2"],
                   dlogits=g["dlogits"], dgate=g["dgate"])
    perm = torch.empty(R, dtype=torch.int32, device=DEV)
    offsets = torch.empty(w.E + 1, dtype=torch.int32, device=DEV)
    row_gate = torch.empty(R, device=DEV)
    inv = torch.empty(w.T * w.E, dtype=torch.int32, device=DEV)
    counts = torch.empty(w.E, dtype=torch.int32, device=DEV)
    unrouted = torch.empty(1, dtype=torch.int32, device=DEV)
    L.moe_expert_choice(s, L.alloc_workspace(s, DEV), perm, offsets, row_gate, inv, counts,
                        unrouted, x=inp["x"], w_router=inp["w_router"])
    torch.cuda.synchronize()
    assert L.moe_get_error(ws) == 0
    perm_h, offs = perm.cpu().numpy(), offsets.cpu().numpy()
    inv_h = inv.cpu().numpy().reshape(w.T, w.E)

    x64, dy64, wr64 = host64(inp["x"]), host64(dy), host64(inp["w_router"])
    logits64 = O.router_logits(x64, wr64)
    p64 = O.softmax_all(logits64)
    rng = np.random.default_rng(4)

    for e in sorted(rng.choice(w.E, size=2, replace=False)):
        toks = perm_h[offs[e]:offs[e + 1]]
        fs = np.sort(rng.choice(w.d_ff, size=16, replace=False))
        fs_t = torch.as_tensor(fs, device=DEV)
        r = O.swiglu_ffn_backward(x64[toks], host64(inp["w1"][e][fs_t]), host64(inp["w3"][e][fs_t]),
                                  host64(inp["w2"][e][:, fs_t]), p64[toks, e][:, None] * dy64[toks])
        assert rel_l2(g["dw1"][e][fs_t].double().cpu().numpy(), r["dw1"]) < TOL, ("dw1", e)
        assert rel_l2(g["dw3"][e][fs_t].double().cpu().numpy(), r["dw3"]) < TOL, ("dw3", e)
        assert rel_l2(g["dw2"][e][:, fs_t].double().cpu().numpy(), r["dw2"]) < TOL, ("dw2", e)

    tokens = np.sort(rng.choice(w.T, size=6, replace=False))
    dz = O.z_loss_backward(logits64, w.beta)
    dx_ref, dl_ref, dg_ref, dg_got = [], [], [], []
    dgate_h = g["dgate"].double().cpu().numpy()
    cache = {}
    for t in tokens:
        dxt = np.zeros(w.d)
        a = np.zeros(w.E)
        for e in range(w.E):
            r_ = inv_h[t, e]
            if r_ < 0:
                continue
            if e not in cache:
                cache[e] = (host64(inp["w1"][e]), host64(inp["w3"][e]), host64(inp["w2"][e]))
            w1e, w3e, w2e = cache[e]
            rb = O.swiglu_ffn_backward(x64[t:t + 1], w1e, w3e, w2e, p64[t, e] * dy64[t:t + 1])
            dxt += rb["dx"][0]
            a[e] = float(dy64[t] @ (rb["H"][0] @ w2e.T))
            dg_ref.append(a[e])
            dg_got.append(dgate_h[r_])
        dlt = p64[t] * (a - p64[t] @ a) + dz[t]
        dx_ref.append(dxt + dlt @ wr64)
        dl_ref.append(dlt)
    tt = torch.as_tensor(tokens, device=DEV)
    assert len(dg_ref) > 0
    assert rel_l2(np.array(dg_got), np.array(dg_ref)) < TOL
    assert rel_l2(g["dlogits"][tt].double().cpu().numpy(), np.array(dl_ref)) < TOL
    err = rel_l2(g["dx"][tt].double().cpu().numpy(), np.array(dx_ref))
    print(f"mixtral_prefill + expert choice: sampled dx rel L2 = {err:.3e}")
    assert err < TOL
    del inp, g, ws
    torch.cuda.empty_cache()
