"""GPU parity of the backward pass of expert-choice layers against the fp64 oracle
(oracle.expert_choice_backward).

The GPU recomputes the experts' choices; the oracle runs on the GPU's own choices (the
choice itself is tested bit for bit against the oracle in the expert-choice routing tests),
so a near tie in the fp32 probabilities cannot cascade. Bounds as for top-k layers: bf16
relative L2 <= 2e-2 per gradient tensor and per expert, fp32 max-abs <= 1e-4 * RMS."""
import numpy as np
import pytest
import torch

import oracle as O
from moe_inputs import WORKLOADS, make_inputs
from moe_testlib import host64, rel_l2
from mixture_experts_layer_92_b300 import _lib as L

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL = 2e-2


def gpu_choice(s, w, inp, C):
    """perm / offsets / row gates / inv of moe_expert_choice on the layer's inputs."""
    Cp = min(C, w.T)
    R = max(w.E * Cp, 1)
    out = dict(perm=torch.empty(R, dtype=torch.int32, device=DEV),
               offsets=torch.empty(w.E + 1, dtype=torch.int32, device=DEV),
               gate=torch.empty(R, device=DEV),
               inv=torch.empty(max(w.T * w.E, 1), dtype=torch.int32, device=DEV),
               counts=torch.empty(w.E, dtype=torch.int32, device=DEV),
               unrouted=torch.empty(1, dtype=torch.int32, device=DEV))
    ws = L.alloc_workspace(s, DEV)
    L.moe_expert_choice(s, ws, out["perm"], out["offsets"], out["gate"], out["inv"],
                        out["counts"], out["unrouted"], x=inp["x"], w_router=inp["w_router"],
                        router_bias=inp["router_bias"])
    torch.cuda.synchronize()
    assert L.moe_get_error(ws) == 0
    h = {n: t.cpu().numpy() for n, t in out.items()}
    return dict(perm=h["perm"][:w.E * Cp], offsets=h["offsets"],
                inv=h["inv"][:w.T * w.E].reshape(w.T, w.E), unrouted=int(h["unrouted"][0]))


def run(w, C, seed, d_aux=0.7, d_z=1.3):
    inp = make_inputs(w, device=DEV, seed=seed)
    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    dy = torch.randn((w.T, w.d), generator=torch.Generator(device=DEV).manual_seed(seed + 1),
                     device=DEV).to(dt)
    s = L.make_shape(w.T, w.d, w.E, w.k, w.d_ff, gate="expert_choice", dtype=dt, capacity=C,
                     d_ff_shared=w.d_ff_shared, alpha=w.alpha, beta=w.beta)
    ws = L.alloc_workspace_backward(s, DEV)
    R = w.E * min(C, w.T)
    f32 = dict(device=DEV, dtype=torch.float32)
    nan = float("nan")
    g = dict(dx=torch.full_like(inp["x"], nan), dw_router=torch.full((w.E, w.d), nan, **f32),
             dw1=torch.full((w.E, w.d_ff, w.d), nan, **f32),
             dw3=torch.full((w.E, w.d_ff, w.d), nan, **f32),
             dw2=torch.full((w.E, w.d, w.d_ff), nan, **f32),
             d_router_bias=torch.full((w.E,), nan, **f32),
             dlogits=torch.full((w.T, w.E), nan, **f32), dgate=torch.full((R,), nan, **f32))
    if w.d_ff_shared:
        g.update(dw1s=torch.full((w.d_ff_shared, w.d), nan, **f32),
                 dw3s=torch.full((w.d_ff_shared, w.d), nan, **f32),
                 dw2s=torch.full((w.d, w.d_ff_shared), nan, **f32))
    L.moe_backward(s, ws, inp["x"], inp["w_router"], inp["w1"], inp["w3"], inp["w2"], dy,
                   g["dx"], g["dw_router"], g["dw1"], g["dw3"], g["dw2"],
                   router_bias=inp["router_bias"], w1s=inp["w1s"], w3s=inp["w3s"], w2s=inp["w2s"],
                   d_aux=d_aux, d_z=d_z, d_router_bias=g["d_router_bias"], dw1s=g.get("dw1s"),
                   dw3s=g.get("dw3s"), dw2s=g.get("dw2s"), dlogits=g["dlogits"], dgate=g["dgate"])
    torch.cuda.synchronize()
    assert L.moe_get_error(ws) == 0
    choice = gpu_choice(s, w, inp, C)
    opt = lambda t: None if t is None else host64(t)
    ref = O.expert_choice_backward(host64(inp["x"]), host64(inp["w_router"]), host64(inp["w1"]),
                                   host64(inp["w3"]), host64(inp["w2"]), host64(dy), C=C,
                                   router_bias=opt(inp["router_bias"]), w1s=opt(inp["w1s"]),
                                   w3s=opt(inp["w3s"]), w2s=opt(inp["w2s"]), alpha=w.alpha,
                                   beta=w.beta, k=w.k, d_aux=d_aux, d_z=d_z, choice=choice)
    ref["dgate"] = ref["dgate_rows"]
    got = {n: t.double().cpu().numpy() for n, t in g.items()}
    return got, ref, choice


def names_of(w):
    n = ["dx", "dw_router", "dw1", "dw3", "dw2", "dgate", "dlogits", "d_router_bias"]
    return n + (["dw1s", "dw3s", "dw2s"] if w.d_ff_shared else [])


BF16_CASES = {
    # name: (workload at reduced size, capacity C)
    # 8 * 150 = 1200 rows for 600 tokens, shared expert and a skewed router bias
    "shared_bias": (WORKLOADS["deepseek_fine"].scaled(T=600, d=256, E=8, k=2, d_ff=384,
                                                      d_ff_shared=128, zipf_s=1.2), 150),
    # 512 rows per expert: 256-row weight-gradient tiles
    "wide_tiles": (WORKLOADS["mixtral_prefill"].scaled(T=2048, d=256, E=16, k=2, d_ff=512), 512),
    # 8 * 40 = 320 rows for 512 tokens: many tokens no expert chose
    "unrouted_tokens": (WORKLOADS["mixtral_prefill"].scaled(T=512, d=128, E=8, k=1, d_ff=192), 40),
    # C > T: every expert takes every token (C' = T)
    "capacity_above_T": (WORKLOADS["mixtral_prefill"].scaled(T=100, d=128, E=8, k=2, d_ff=128), 130),
}


@pytest.mark.parametrize("name", list(BF16_CASES))
def test_expert_choice_backward_bf16(name):
    w, C = BF16_CASES[name]
    got, ref, choice = run(w, C, seed=7)
    if name == "unrouted_tokens":
        assert choice["unrouted"] > 0
        # a token no expert chose gets only the router's (z-loss) and no expert gradient
    for n in names_of(w):
        assert np.isfinite(got[n]).all(), n
        assert rel_l2(got[n], ref[n]) < TOL, (n, rel_l2(got[n], ref[n]))
    for e in range(w.E):
        for n in ("dw1", "dw3", "dw2"):
            assert rel_l2(got[n][e], ref[n][e]) < TOL, (n, e)


def test_expert_choice_backward_fp32():
    w = WORKLOADS["tiny_fp32"].scaled(d_ff_shared=48, zipf_s=1.2)
    C = max(1, w.T * 2 // w.E)
    got, ref, _ = run(w, C, seed=3)
    for n in names_of(w):
        rms = np.sqrt(np.mean(ref[n] ** 2))
        assert np.abs(got[n] - ref[n]).max() <= 1e-4 * rms, (n, np.abs(got[n] - ref[n]).max(), rms)


def test_expert_choice_backward_ignores_balance_loss():
    """The balance loss is constant under expert choice: d_aux changes no gradient (bit for bit)."""
    w, C = BF16_CASES["unrouted_tokens"]
    a, _, _ = run(w, C, seed=9, d_aux=0.0)
    b, _, _ = run(w, C, seed=9, d_aux=5.0)
    for n in names_of(w):
        np.testing.assert_array_equal(a[n], b[n], err_msg=n)
