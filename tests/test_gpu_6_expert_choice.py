"""GPU parity of expert-choice routing against the oracle.

The GPU ranks tokens by fp32 router probabilities, the oracle by fp64 ones: an expert's
chosen set must be identical unless its C-th and (C+1)-th oracle probabilities are a near
tie (relative gap < 1e-6). Layer outputs are checked with the oracle re-run on the GPU's own
choices (fp32 layers: max error <= 1e-4 RMS; bf16: relative L2 <= 2e-2)."""
import numpy as np
import pytest
import torch

import oracle as O
from moe_inputs import WORKLOADS, make_inputs, random_logits
from moe_testlib import host64, rel_l2
from mixture_experts_layer_92_b300 import _lib as L

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def near_tie_experts(p, C):
    T, E = p.shape
    out = set()
    if C >= T or C == 0:
        return out
    for e in range(E):
        s = np.sort(p[:, e])[::-1]
        if s[C - 1] - s[C] <= 1e-6 * s[C - 1]:
            out.add(e)
    return out


def run_ec(s, ws, T, E, C, **kw):
    Cp = min(C, T)
    perm = torch.full((max(E * Cp, 1),), -9, dtype=torch.int32, device=DEV)
    row_gate = torch.empty(max(E * Cp, 1), device=DEV)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    inv = torch.empty(max(T * E, 1), dtype=torch.int32, device=DEV)
    counts = torch.empty(E, dtype=torch.int32, device=DEV)
    unrouted = torch.empty(1, dtype=torch.int32, device=DEV)
    L.moe_expert_choice(s, ws, perm, offsets, row_gate, inv, counts, unrouted, **kw)
    torch.cuda.synchronize()
    assert L.moe_get_error(ws) == 0
    return dict(perm=perm.cpu().numpy()[:E * Cp], offsets=offsets.cpu().numpy(),
                gate=row_gate.cpu().numpy()[:E * Cp], inv=inv.cpu().numpy()[:T * E].reshape(T, E),
                counts=counts.cpu().numpy(), unrouted=int(unrouted.item()))


@pytest.mark.parametrize("T,E,C", [(300, 8, 75), (300, 8, 0), (64, 16, 64), (1000, 128, 8),
                                   (4097, 64, 130), (5, 4, 9), (2048, 256, 64),
                                   (300, 1, 50), (1, 3, 1)])   # one expert; one token
@pytest.mark.parametrize("ties", [False, True])
def test_expert_choice_matches_oracle(T, E, C, ties):
    l = random_logits(T, E, seed=T + E + C, ties=ties)
    s = L.make_shape(T, 16, E, 1, 16, gate="expert_choice", dtype=torch.float32, capacity=C)
    ws = L.alloc_workspace(s, DEV)
    g = run_ec(s, ws, T, E, C, logits_in=l.to(DEV))
    l64 = l.double().numpy()
    o = O.expert_choice(l64, C)
    Cp = min(C, T)
    np.testing.assert_array_equal(g["counts"], o["counts"])
    np.testing.assert_array_equal(g["offsets"], o["offsets"])
    skip = near_tie_experts(O.softmax_all(l64), Cp)
    for e in range(E):
        seg = slice(e * Cp, (e + 1) * Cp)
        assert np.all(np.diff(g["perm"][seg]) > 0)          # ascending tokens
        if e in skip:
            continue
        np.testing.assert_array_equal(g["perm"][seg], o["perm"][seg])
        np.testing.assert_array_equal(g["inv"][:, e], o["inv"][:, e])
    np.testing.assert_allclose(g["gate"], O.softmax_all(l64)[g["perm"], np.repeat(np.arange(E), Cp)],
                               rtol=2e-6, atol=1e-8)
    if not skip:
        assert g["unrouted"] == o["unrouted"]


def layer(w, C, dtype, seed=0):
    inp = make_inputs(w, device=DEV, seed=seed)
    s = L.make_shape(w.T, w.d, w.E, w.k, w.d_ff, gate="expert_choice", dtype=dtype, capacity=C,
                     d_ff_shared=w.d_ff_shared, alpha=w.alpha, beta=w.beta)
    ws = L.alloc_workspace(s, DEV)
    y = torch.empty_like(inp["x"])
    counts = torch.empty(w.E, dtype=torch.int32, device=DEV)
    unrouted = torch.empty(1, dtype=torch.int32, device=DEV)
    losses = torch.empty(2, device=DEV)
    L.moe_forward(s, ws, inp["x"], inp["w_router"], inp["w1"], inp["w3"], inp["w2"], y,
                  router_bias=inp["router_bias"], w1s=inp["w1s"], w3s=inp["w3s"], w2s=inp["w2s"],
                  counts=counts, dropped=unrouted, losses=losses)
    g = run_ec(s, ws, w.T, w.E, C, x=inp["x"], w_router=inp["w_router"],
               router_bias=inp["router_bias"])
    shared = {}
    if w.d_ff_shared:
        shared = dict(w1s=host64(inp["w1s"]), w3s=host64(inp["w3s"]), w2s=host64(inp["w2s"]))
    ref = O.expert_choice_forward(host64(inp["x"]), host64(inp["w_router"]), host64(inp["w1"]),
                                  host64(inp["w3"]), host64(inp["w2"]), C=C, k=w.k,
                                  router_bias=None if inp["router_bias"] is None
                                  else host64(inp["router_bias"]),
                                  alpha=w.alpha, beta=w.beta, choice=g, **shared)
    assert int(unrouted.item()) == g["unrouted"]
    np.testing.assert_array_equal(counts.cpu().numpy(), ref["ec"]["counts"])
    l = losses.cpu().numpy()
    assert l[0] == pytest.approx(ref["l_aux"], rel=1e-3)
    assert l[1] == pytest.approx(ref["l_z"], rel=1e-3)
    return y.double().cpu().numpy(), ref["y"]


def test_expert_choice_layer_fp32():
    w = WORKLOADS["tiny_fp32"].scaled(d_ff_shared=64)
    y, yref = layer(w, C=64, dtype=torch.float32)           # 8 * 64 = T * k: 2 per token on average
    assert np.abs(y - yref).max() <= 1e-4 * np.sqrt(np.mean(yref ** 2))


@pytest.mark.parametrize("T,d,E,F,C", [(600, 512, 8, 768, 150), (2048, 256, 16, 8192, 512)])
def test_expert_choice_layer_bf16(T, d, E, F, C):
    """bf16 tensor-core path; the second shape runs the 256-row down-projection tiles."""
    w = WORKLOADS["mixtral_prefill"].scaled(T=T, d=d, E=E, k=2, d_ff=F)
    y, yref = layer(w, C=C, dtype=torch.bfloat16, seed=4)
    assert rel_l2(y, yref) < 2e-2


def test_expert_choice_layer_bf16_pair_tiles_shared():
    """Expert-choice layers whose experts hold whole 256-row tiles run both expert GEMMs on CTA
    pairs (tcgen05 cta_group::2): here every expert takes C = 768 rows (three pair tiles),
    d_ff >= 8192, with the shared expert's 1500 rows (a last tile of 220) on the same pairs and
    a ragged K / N (d = 328 = 5 * 64 + 8)."""
    w = WORKLOADS["mixtral_prefill"].scaled(T=1500, d=328, E=4, k=2, d_ff=8192, d_ff_shared=200)
    y, yref = layer(w, C=768, dtype=torch.bfloat16, seed=8)
    assert rel_l2(y, yref) < 2e-2


def test_expert_choice_layer_bf16_pair_tiles_partial_last_tile():
    """C = 650 rows per expert: two whole pair tiles and a last one of 138 rows (more than
    half full, so the layer still runs on CTA pairs; CTA 1 holds 10 valid rows of it), in both
    expert GEMMs (d_ff >= 8192)."""
    w = WORKLOADS["mixtral_prefill"].scaled(T=1400, d=256, E=4, k=2, d_ff=8192)
    y, yref = layer(w, C=650, dtype=torch.bfloat16, seed=9)
    assert rel_l2(y, yref) < 2e-2
