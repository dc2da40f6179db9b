"""GPU parity of the dispatch a forward leaves in its workspace.

For every case the forward's own dispatch results -- perm, inv and offsets as moe_forward
leaves them in the workspace (moe_workspace_dispatch_offsets), counts and dropped as it returns
them -- are bit-identical to the dispatch kernel run through moe_dispatch and to the oracle's
counting sort ("Mixture of experts (MoE)", tirogla.com, How it works, step 3), both on the
forward's routing (moe_route_topk from x: the same fused router, the same bits); its losses
are bit-identical to moe_aux_loss on that routing's statistics and the counts. Shapes cover
router cluster splits of 1, 2, 4 and 8 (CTAs of 128, 64, 32 and 16 tokens, so the router's
statistic partials come in different counts), ragged token counts, k = 1 .. 8, E = 8 .. 256,
heavy drops (Zipf-biased router, cf < 1), C = 0, a batch of 36000 assignments and one of
160000 (two 32-wide pieces per dispatch warp); a second test runs forwards of different sizes
on one workspace (the dispatch's grid-barrier counters must return to zero after each)."""
import numpy as np
import pytest
import torch

import oracle as O
from moe_inputs import WORKLOADS, make_inputs
from mixture_experts_layer_92_b300 import _lib as L

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

CASES = [
    # name, base workload, T, d, E, k, gate, cf (None: no drop)
    ("mixtral_like_cs8", "mixtral_prefill", 1000, 512, 8, 2, "softmax_topk", None),
    ("switch_like_cs4_drops", "switch_top1", 4096, 256, 128, 1, "softmax_all", 1.0),
    ("switch_full_cs1", "switch_top1", 16384, 1024, 128, 1, "softmax_all", 1.0),
    ("cs2_drops", "switch_top1", 5000, 128, 32, 2, "softmax_topk", 1.0),
    ("k8_sigmoid_drops", "mixtral_prefill", 600, 256, 64, 8, "sigmoid_topk", 1.25),
    ("e256", "switch_top1", 256, 512, 256, 2, "softmax_topk", 1.0),
    ("c_zero", "mixtral_prefill", 700, 256, 16, 2, "softmax_topk", 0.0),
    ("ragged_tail", "switch_top1", 130, 384, 16, 4, "softmax_topk", 0.5),
    ("decode_empty_ctas", "mixtral_prefill", 32, 1024, 8, 2, "softmax_topk", None),
    ("large_batch", "mixtral_prefill", 18000, 128, 8, 2, "softmax_topk", 1.0),
    # 160000 assignments: more than 148 CTAs x 1024, so each dispatch warp walks two pieces
    ("two_pieces_per_warp", "switch_top1", 40000, 128, 16, 4, "softmax_topk", 1.0),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_forward_dispatch_equals_the_dispatch_kernel(case):
    name, base, T, d, E, k, gate, cf = case
    w = WORKLOADS[base].scaled(T=T, d=d, E=E, k=k, d_ff=64, gate=gate, cf=cf, d_ff_shared=0)
    C = T if cf is None else (0 if cf == 0.0 else O.capacity(cf, T, k, E))
    inp = make_inputs(w, device=DEV, seed=T + E + k)
    s = L.make_shape(T, d, E, k, 64, gate=gate, dtype=torch.bfloat16, capacity=C,
                     alpha=w.alpha, beta=w.beta)
    A = T * k

    # the forward, its dispatch results poisoned beforehand
    ws = L.alloc_workspace(s, device=DEV)
    perm_v, inv_v, off_v = L.workspace_dispatch(s, ws)
    perm_v.fill_(-9)
    inv_v.fill_(-9)
    off_v.fill_(-9)
    y = torch.empty_like(inp["x"])
    counts = torch.full((E,), -7, dtype=torch.int32, device=DEV)
    dropped = torch.full((1,), -7, dtype=torch.int32, device=DEV)
    losses = torch.full((2,), float("nan"), device=DEV)
    L.moe_forward(s, ws, inp["x"], inp["w_router"], inp["w1"], inp["w3"], inp["w2"], y,
                  router_bias=inp["router_bias"], counts=counts, dropped=dropped, losses=losses)
    torch.cuda.synchronize()
    assert L.moe_get_error(ws) == 0
    fperm, finv, foff = perm_v.clone(), inv_v.clone(), off_v.clone()

    # the same routing from the routing entry point, then the dispatch kernel on it
    ws2 = L.alloc_workspace(s, device=DEV)
    idx = torch.empty(T, k, dtype=torch.int32, device=DEV)
    gates = torch.empty(T, k, device=DEV)
    stats = torch.empty(E + 1, device=DEV)
    L.moe_route_topk(s, ws2, idx, gates, x=inp["x"], w_router=inp["w_router"],
                     router_bias=inp["router_bias"], stats=stats)
    cnt2 = torch.full((E,), -5, dtype=torch.int32, device=DEV)
    off2 = torch.full((E + 1,), -5, dtype=torch.int32, device=DEV)
    perm2 = torch.full((A,), -5, dtype=torch.int32, device=DEV)
    inv2 = torch.full((A,), -5, dtype=torch.int32, device=DEV)
    drp2 = torch.full((1,), -5, dtype=torch.int32, device=DEV)
    L.moe_dispatch(s, ws2, cnt2, off2, perm2, inv2, drp2, topk_idx=idx)
    losses2 = torch.full((2,), float("nan"), device=DEV)
    L.moe_aux_loss(s, stats, counts, losses2)
    torch.cuda.synchronize()
    assert L.moe_get_error(ws2) == 0

    R = int(off2[E].item())
    assert torch.equal(foff, off2)
    assert torch.equal(counts, cnt2)
    assert int(dropped.item()) == int(drp2.item()) == A - R
    assert torch.equal(finv, inv2)
    assert torch.equal(fperm[:R], perm2[:R])
    assert torch.equal(losses, losses2), (losses, losses2)

    o = O.dispatch(idx.cpu().numpy().astype(np.int64), E, C)
    np.testing.assert_array_equal(foff.cpu().numpy(), o["offsets"])
    np.testing.assert_array_equal(counts.cpu().numpy(), o["counts"])
    np.testing.assert_array_equal(fperm[:R].cpu().numpy(), o["perm"])
    np.testing.assert_array_equal(finv.cpu().numpy(), o["inv"])
    assert int(dropped.item()) == o["dropped"]


def test_forward_dispatch_repeats_on_one_workspace():
    """Forwards of different batches on one workspace each leave the oracle's dispatch (the
    dispatch kernel's grid-barrier counters live in the workspace header and must return to
    zero after every launch)."""
    E, k, d = 32, 2, 256
    w0 = WORKLOADS["switch_top1"].scaled(T=3000, d=d, E=E, k=k, d_ff=64, gate="softmax_topk",
                                         cf=1.0, d_ff_shared=0)
    s_max = L.make_shape(3000, d, E, k, 64, gate="softmax_topk", dtype=torch.bfloat16,
                         capacity=O.capacity(1.0, 3000, k, E))
    ws = L.alloc_workspace(s_max, device=DEV)
    for rep, T in enumerate((3000, 777, 3000, 64)):
        w = w0.scaled(T=T)
        C = O.capacity(1.0, T, k, E)
        s = L.make_shape(T, d, E, k, 64, gate="softmax_topk", dtype=torch.bfloat16, capacity=C)
        inp = make_inputs(w, device=DEV, seed=100 + rep)
        y = torch.empty_like(inp["x"])
        counts = torch.empty(E, dtype=torch.int32, device=DEV)
        dropped = torch.empty(1, dtype=torch.int32, device=DEV)
        L.moe_forward(s, ws, inp["x"], inp["w_router"], inp["w1"], inp["w3"], inp["w2"], y,
                      router_bias=inp["router_bias"], counts=counts, dropped=dropped)
        perm_v, inv_v, off_v = L.workspace_dispatch(s, ws)
        idx = torch.empty(T, k, dtype=torch.int32, device=DEV)
        L.moe_route_topk(s, L.alloc_workspace(s, device=DEV), idx, torch.empty(T, k, device=DEV),
                         x=inp["x"], w_router=inp["w_router"], router_bias=inp["router_bias"])
        torch.cuda.synchronize()
        assert L.moe_get_error(ws) == 0
        o = O.dispatch(idx.cpu().numpy().astype(np.int64), E, C)
        R = int(o["offsets"][E])
        np.testing.assert_array_equal(off_v.cpu().numpy(), o["offsets"])
        np.testing.assert_array_equal(perm_v[:R].cpu().numpy(), o["perm"])
        np.testing.assert_array_equal(inv_v.cpu().numpy(), o["inv"])
        np.testing.assert_array_equal(counts.cpu().numpy(), o["counts"])
        assert int(dropped.item()) == o["dropped"]
