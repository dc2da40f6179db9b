"""GPU parity of the top-1 bf16 path whose down projection writes y itself (no combine launch:
with one slot per token the combine is a copy; the token-major gather zeroes the rows of dropped
tokens), and of the router statistics and losses that ride in the dispatch launch.

y is filled with NaN before every forward, so a row that neither the GEMM's epilogue nor the
gather wrote shows up. Bar: every token's row against the oracle (relative L2 of y <= 2e-2 and
every kept row within 5 %), dropped tokens' rows exactly zero, counts and drops bit-exact, the
losses within 1e-3 of the oracle and bit-identical to moe_aux_loss on the forward's own
statistics and counts."""
import numpy as np
import pytest
import torch

import oracle as O
from moe_inputs import WORKLOADS, make_inputs
from moe_testlib import host64, oracle_y_for_tokens, rel_l2, routing_check
from mixture_experts_layer_92_b300 import _lib as L

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def forward_nan_filled(w, C):
    inp = make_inputs(w, device=DEV, seed=w.T + w.E)
    s = L.make_shape(w.T, w.d, w.E, w.k, w.d_ff, gate=w.gate, dtype=torch.bfloat16, capacity=C,
                     d_ff_shared=w.d_ff_shared, alpha=w.alpha, beta=w.beta)
    ws = L.alloc_workspace(s, device=DEV)
    y = torch.full_like(inp["x"], float("nan"))
    counts = torch.zeros(w.E, dtype=torch.int32, device=DEV)
    dropped = torch.zeros(1, dtype=torch.int32, device=DEV)
    losses = torch.zeros(2, device=DEV)
    L.moe_forward(s, ws, inp["x"], inp["w_router"], inp["w1"], inp["w3"], inp["w2"], y,
                  router_bias=inp["router_bias"], w1s=inp["w1s"], w3s=inp["w3s"], w2s=inp["w2s"],
                  counts=counts, dropped=dropped, losses=losses)
    idx = torch.empty(w.T, w.k, dtype=torch.int32, device=DEV)
    gate = torch.empty(w.T, w.k, device=DEV)
    L.moe_route_topk(s, ws, idx, gate, x=inp["x"], w_router=inp["w_router"],
                     router_bias=inp["router_bias"])
    torch.cuda.synchronize()
    assert L.moe_get_error(ws) == 0
    return inp, s, ws, y, counts, dropped, losses, idx


CASES = [
    # name, T, d, E, d_ff, cf, zipf, shared
    ("heavy_drops", 3000, 256, 32, 256, 0.5, 1.2, 0),
    ("no_drops_ragged", 1000, 384, 16, 320, None, None, 0),
    ("all_dropped", 600, 256, 16, 256, 0.0, None, 0),
    ("e512_unfused_router", 2048, 256, 512, 128, 1.0, 1.2, 0),
    ("with_shared_expert", 700, 256, 16, 256, 1.0, None, 128),   # keeps the combine launch
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_top1_layer_every_row_written(case):
    name, T, d, E, F, cf, zipf, Fs = case
    w = WORKLOADS["switch_top1"].scaled(T=T, d=d, E=E, k=1, d_ff=F, cf=cf, zipf_s=zipf,
                                        d_ff_shared=Fs)
    C = w.T if cf is None else (0 if cf == 0.0 else O.capacity(cf, w.T, 1, w.E))
    inp, s, ws, y, counts, dropped, losses, idx = forward_nan_filled(w, C)
    bias = None if inp["router_bias"] is None else host64(inp["router_bias"])
    logits64 = O.router_logits(host64(inp["x"]), host64(inp["w_router"]), bias)
    gidx = idx.cpu().numpy().astype(np.int64)
    bad, ties = routing_check(logits64, gidx, 1)
    assert set(bad.tolist()) <= set(ties.tolist())
    disp = O.dispatch(gidx, w.E, C)
    np.testing.assert_array_equal(counts.cpu().numpy(), disp["counts"])
    assert int(dropped.item()) == disp["dropped"]
    yh = y.double().cpu().numpy()
    assert np.isfinite(yh).all(), f"{name}: rows left unwritten"
    kept = disp["inv"].reshape(T) >= 0
    if Fs == 0:
        assert np.all(yh[~kept] == 0.0), f"{name}: a dropped token's row is not zero"
    yref = oracle_y_for_tokens(w, inp, logits64, gidx, disp["inv"], np.arange(T))
    if kept.any() or Fs:
        err = rel_l2(yh, yref)
        assert err < 2e-2, f"{name}: relative L2 {err:.3e}"
        rows = kept if Fs == 0 else np.ones(T, dtype=bool)
        num = np.linalg.norm(yh[rows] - yref[rows], axis=1)
        den = np.linalg.norm(yref[rows], axis=1)
        assert np.all(num <= 0.05 * den + 1e-6), f"{name}: worst row {np.max(num / den):.3e}"
    l = losses.cpu().numpy()
    assert l[0] == pytest.approx(O.aux_loss(logits64, gidx, w.alpha), rel=1e-3)
    assert l[1] == pytest.approx(O.z_loss(logits64, w.beta), rel=1e-3)
    # the statistics the dispatch left in the workspace give the same losses through
    # moe_aux_loss, bit for bit
    stats = torch.empty(E + 1, device=DEV)
    L.moe_route_topk(s, ws, torch.empty(T, 1, dtype=torch.int32, device=DEV),
                     torch.empty(T, 1, device=DEV), x=inp["x"], w_router=inp["w_router"],
                     router_bias=inp["router_bias"], stats=stats)
    losses2 = torch.full((2,), float("nan"), device=DEV)
    L.moe_aux_loss(s, stats, counts, losses2)
    torch.cuda.synchronize()
    assert torch.equal(losses, losses2), (losses, losses2)


def test_e1024_top2_layer_statistics_in_the_dispatch():
    """E = 1024 (the largest E, the unfused router): the dispatch runs 33 statistics CTAs beside
    its own, at one CTA per SM (its shared memory) -- the co-residency bound of its grid barrier
    in the tightest case. Every row against the oracle, losses bit-identical to moe_aux_loss."""
    w = WORKLOADS["deepseek_fine"].scaled(T=2048, d=128, E=1024, k=2, d_ff=128, d_ff_shared=0,
                                          gate="softmax_topk", cf=1.5)
    C = O.capacity(w.cf, w.T, w.k, w.E)
    inp, s, ws, y, counts, dropped, losses, idx = forward_nan_filled(w, C)
    logits64 = O.router_logits(host64(inp["x"]), host64(inp["w_router"]), None)
    gidx = idx.cpu().numpy().astype(np.int64)
    bad, ties = routing_check(logits64, gidx, w.k)
    assert set(bad.tolist()) <= set(ties.tolist())
    disp = O.dispatch(gidx, w.E, C)
    np.testing.assert_array_equal(counts.cpu().numpy(), disp["counts"])
    assert int(dropped.item()) == disp["dropped"]
    yh = y.double().cpu().numpy()
    assert np.isfinite(yh).all()
    yref = oracle_y_for_tokens(w, inp, logits64, gidx, disp["inv"], np.arange(w.T))
    assert rel_l2(yh, yref) < 2e-2
    l = losses.cpu().numpy()
    assert l[0] == pytest.approx(O.aux_loss(logits64, gidx, w.alpha), rel=1e-3)
    assert l[1] == pytest.approx(O.z_loss(logits64, w.beta), rel=1e-3)
    stats = torch.empty(w.E + 1, device=DEV)
    L.moe_route_topk(s, ws, torch.empty(w.T, w.k, dtype=torch.int32, device=DEV),
                     torch.empty(w.T, w.k, device=DEV), x=inp["x"], w_router=inp["w_router"],
                     stats=stats)
    losses2 = torch.full((2,), float("nan"), device=DEV)
    L.moe_aux_loss(s, stats, counts, losses2)
    torch.cuda.synchronize()
    assert torch.equal(losses, losses2), (losses, losses2)
