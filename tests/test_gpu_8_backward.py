"""GPU parity of the backward pass (moe_backward) against the fp64 backward oracle.

The GPU recomputes its routing; the oracle is run on the GPU's own routing decisions
(idx_override), so that a near-tie flip cannot cascade (the top-k itself is checked bit for
bit elsewhere). Inputs are bf16 and the backward rounds G, U, H, dG, dU, g*dy and the logit
gradient to bf16 with fp32 accumulation, the same rounding regime as the bf16 forward, so
the forward's bf16 bound applies to every gradient: relative L2 <= 2e-2 over the tensor;
expert weight gradients are also checked expert by expert (no tile/row mapping error can
hide in the mean)."""
import numpy as np
import pytest
import torch

import oracle as O
from moe_inputs import WORKLOADS, make_inputs
from moe_testlib import capacity_of, host64, rel_l2
from mixture_experts_layer_92_b300 import _lib as L

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL = 2e-2


def run_backward(w, inp, dy, d_aux=1.0, d_z=1.0, C=None):
    C = capacity_of(w) if C is None else C
    s = L.make_shape(w.T, w.d, w.E, w.k, w.d_ff, gate=w.gate, dtype=inp["x"].dtype, capacity=C,
                     d_ff_shared=w.d_ff_shared, alpha=w.alpha, beta=w.beta)
    ws = L.alloc_workspace_backward(s, DEV)
    f32 = dict(device=DEV, dtype=torch.float32)
    g = dict(dx=torch.full_like(inp["x"], float("nan")),
             dw_router=torch.full((w.E, w.d), float("nan"), **f32),
             dw1=torch.full((w.E, w.d_ff, w.d), float("nan"), **f32),
             dw3=torch.full((w.E, w.d_ff, w.d), float("nan"), **f32),
             dw2=torch.full((w.E, w.d, w.d_ff), float("nan"), **f32),
             d_router_bias=torch.full((w.E,), float("nan"), **f32),
             dlogits=torch.empty((w.T, w.E), **f32), dgate=torch.empty((w.T, w.k), **f32))
    if w.d_ff_shared:
        g.update(dw1s=torch.empty((w.d_ff_shared, w.d), **f32),
                 dw3s=torch.empty((w.d_ff_shared, w.d), **f32),
                 dw2s=torch.empty((w.d, w.d_ff_shared), **f32))
    L.moe_backward(s, ws, inp["x"], inp["w_router"], inp["w1"], inp["w3"], inp["w2"], dy,
                   g["dx"], g["dw_router"], g["dw1"], g["dw3"], g["dw2"],
                   router_bias=inp["router_bias"], w1s=inp["w1s"], w3s=inp["w3s"], w2s=inp["w2s"],
                   d_aux=d_aux, d_z=d_z, d_router_bias=g["d_router_bias"], dw1s=g.get("dw1s"),
                   dw3s=g.get("dw3s"), dw2s=g.get("dw2s"), dlogits=g["dlogits"], dgate=g["dgate"])
    # the routing the backward used: same kernels, same inputs
    idx = torch.empty(w.T, w.k, dtype=torch.int32, device=DEV)
    gate = torch.empty(w.T, w.k, device=DEV)
    fws = L.alloc_workspace(s, DEV)
    L.moe_route_topk(s, fws, idx, gate, x=inp["x"], w_router=inp["w_router"],
                     router_bias=inp["router_bias"])
    torch.cuda.synchronize()
    assert L.moe_get_error(ws) == 0
    g["idx"] = idx.cpu().numpy().astype(np.int64)
    return g, C


def oracle_backward(w, inp, dy, idx, C, d_aux=1.0, d_z=1.0):
    return O.backward(host64(inp["x"]), host64(inp["w_router"]), host64(inp["w1"]),
                      host64(inp["w3"]), host64(inp["w2"]), host64(dy), k=w.k, mode=w.gate, C=C,
                      router_bias=None if inp["router_bias"] is None else host64(inp["router_bias"]),
                      w1s=None if inp["w1s"] is None else host64(inp["w1s"]),
                      w3s=None if inp["w3s"] is None else host64(inp["w3s"]),
                      w2s=None if inp["w2s"] is None else host64(inp["w2s"]),
                      alpha=w.alpha, beta=w.beta, d_aux=d_aux, d_z=d_z, idx_override=idx)


def compare(w, g, ref):
    got = {k: v.double().cpu().numpy() for k, v in g.items() if isinstance(v, torch.Tensor)}
    for name in ("dx", "dw_router", "dw1", "dw3", "dw2", "dgate", "dlogits", "d_router_bias"):
        assert np.isfinite(got[name]).all(), name
        assert rel_l2(got[name], ref[name]) < TOL, (name, rel_l2(got[name], ref[name]))
    kept = np.diff(ref["dispatch"]["offsets"])          # rows each expert received
    for e in range(w.E):
        for name in ("dw1", "dw3", "dw2"):
            if kept[e] == 0:
                assert np.all(got[name][e] == 0.0), (name, e)   # no rows: zero gradient
            else:
                assert rel_l2(got[name][e], ref[name][e]) < TOL, (name, e)
    if w.d_ff_shared:
        for name in ("dw1s", "dw3s", "dw2s"):
            assert rel_l2(got[name], ref[name]) < TOL, name
    # dropped assignments carry no gate gradient, on both sides
    dropped = ref["dispatch"]["inv"].reshape(w.T, w.k) < 0
    assert np.all(got["dgate"][dropped] == 0.0)


def dy_for(w, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    dt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    return torch.randn((w.T, w.d), generator=g, device=DEV).to(dt)


CASES = {
    # name: (workload recipe at reduced size)
    "mixtral_small": WORKLOADS["mixtral_prefill"].scaled(T=256, d=256, E=8, k=2, d_ff=512),
    "switch_drop_ragged": WORKLOADS["switch_top1"].scaled(T=300, d=192, E=8, k=1, d_ff=320,
                                                          cf=1.0, zipf_s=1.2),
    "deepseek_shared": WORKLOADS["deepseek_fine"].scaled(T=500, d=256, E=16, k=4, d_ff=256,
                                                         d_ff_shared=128, zipf_s=1.2),
    "softmax_all_drop": WORKLOADS["mixtral_prefill"].scaled(T=400, d=128, E=8, k=2, d_ff=192,
                                                            gate="softmax_all", cf=0.75),
    "k_equals_E": WORKLOADS["mixtral_prefill"].scaled(T=64, d=128, E=8, k=8, d_ff=128),
    "empty_experts": WORKLOADS["deepseek_fine"].scaled(T=6, d=128, E=16, k=1, d_ff=128,
                                                       d_ff_shared=0),
    "many_row_tiles": WORKLOADS["mixtral_prefill"].scaled(T=3072, d=512, E=8, k=2, d_ff=768),
    # >= 512 rows per expert: 256-row weight-gradient tiles; M = 2*320 = 640 and d = 192 are
    # not multiples of 256 (a last tile without, and one with a partial, second half)
    "wide_tiles_ragged_m": WORKLOADS["mixtral_prefill"].scaled(T=2048, d=192, E=8, k=2,
                                                               d_ff=320),
}


@pytest.mark.parametrize("name", list(CASES))
def test_backward_matches_oracle(name):
    w = CASES[name]
    inp = make_inputs(w, device=DEV, seed=5)
    dy = dy_for(w, 6)
    g, C = run_backward(w, inp, dy, d_aux=0.7, d_z=1.3)
    ref = oracle_backward(w, inp, dy, g["idx"], C, d_aux=0.7, d_z=1.3)
    compare(w, g, ref)


def test_backward_balance_terms_alone():
    """dy = 0: only the balance losses drive the router; every expert gradient is exactly 0
    and the router gradient matches the oracle's aux + z-loss gradient."""
    w = CASES["mixtral_small"].scaled(alpha=0.5, beta=0.25)
    inp = make_inputs(w, device=DEV, seed=2)
    dy = torch.zeros_like(inp["x"])
    g, C = run_backward(w, inp, dy)
    ref = oracle_backward(w, inp, dy, g["idx"], C)
    for name in ("dw1", "dw3", "dw2", "dgate"):
        assert torch.all(g[name] == 0), name
    assert rel_l2(g["dlogits"].double().cpu().numpy(), ref["dlogits"]) < 1e-4
    assert rel_l2(g["dw_router"].double().cpu().numpy(), ref["dw_router"]) < TOL


def test_backward_empty_batch_zeroes_gradients():
    w = CASES["mixtral_small"].scaled(T=0)
    inp = make_inputs(w, device=DEV)
    dy = torch.empty((0, w.d), dtype=torch.bfloat16, device=DEV)
    g, _ = run_backward(w, inp, dy)
    for name in ("dw_router", "dw1", "dw3", "dw2", "d_router_bias"):
        assert torch.all(g[name] == 0), name


def test_backward_deterministic():
    w = CASES["deepseek_shared"]
    inp = make_inputs(w, device=DEV, seed=1)
    dy = dy_for(w, 1)
    a, _ = run_backward(w, inp, dy)
    b, _ = run_backward(w, inp, dy)
    for name in ("dx", "dw_router", "dw1", "dw3", "dw2", "dw1s", "dw3s", "dw2s", "dlogits"):
        assert torch.equal(a[name], b[name]), name


F32_CASES = {
    "tiny_fp32": WORKLOADS["tiny_fp32"],                       # cf 1.25 with drops
    "fp32_shared_sigmoid": WORKLOADS["deepseek_fine"].scaled(T=200, d=96, E=12, k=3, d_ff=80,
                                                             d_ff_shared=48, dtype="f32",
                                                             zipf_s=1.2),
    "fp32_softmax_all_ragged": WORKLOADS["switch_top1"].scaled(T=150, d=40, E=5, k=1, d_ff=24,
                                                               dtype="f32", cf=1.0),
}


@pytest.mark.parametrize("name", list(F32_CASES))
def test_backward_fp32_matches_oracle(name):
    """fp32 layers: every gradient within max-abs 1e-4 * RMS of the oracle's (the forward's
    fp32 bar), on shapes without the bf16 path's tile constraints."""
    w = F32_CASES[name]
    inp = make_inputs(w, device=DEV, seed=3)
    dy = dy_for(w, 4)
    g, C = run_backward(w, inp, dy, d_aux=0.7, d_z=1.3)
    ref = oracle_backward(w, inp, dy, g["idx"], C, d_aux=0.7, d_z=1.3)
    names = ["dx", "dw_router", "dw1", "dw3", "dw2", "dgate", "dlogits", "d_router_bias"]
    if w.d_ff_shared:
        names += ["dw1s", "dw3s", "dw2s"]
    for n in names:
        got = g[n].double().cpu().numpy()
        rms = np.sqrt(np.mean(ref[n] ** 2))
        assert np.abs(got - ref[n]).max() <= 1e-4 * rms, (n, np.abs(got - ref[n]).max(), rms)
