"""GPU parity of the fused router (bf16 layers with E <= 256: the logits are computed on the
tensor cores, split along d over the CTAs of a cluster, reduced on chip, and routed in the
same kernel).

For every case:
  * the logits it reports (logits_out) match the fp64 oracle on the same bf16 inputs to fp32
    accumulation accuracy;
  * its routing decisions are bit-identical to the top-k kernel run on those very logits
    (moe_route_topk with logits_in): the fused epilogue is the same routing step;
  * the statistics behind the balance losses agree with the top-k kernel's (different
    per-block partial sums, so to fp32 rounding);
  * a second run is bitwise identical (the cluster reduces in rank order).
Shapes cover every MMA width (E = 8 .. 256, full and ragged lane slots), every cluster size
(1, 2, 4, 8), a CTA whose K slice is empty (d = 320: 5 k-blocks over 4 CTAs), ragged token
tiles (T = 1, 127, 129, ...), ragged K (d = 200), the three gate modes, a router bias, and a
selection bias."""
import numpy as np
import pytest
import torch

import oracle as O
from moe_inputs import WORKLOADS, make_inputs, zipf_log_popularity
from moe_testlib import host64
from mixture_experts_layer_92_b300 import _lib as L

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

CASES = [
    # T, d, E, k, gate, router bias, selection bias
    (4096, 4096, 8, 2, "softmax_topk", False, False),     # the Mixtral-shaped prefill router
    (16384, 1024, 128, 1, "softmax_all", True, False),    # the Switch-shaped router (Zipf bias)
    (300, 256, 8, 2, "softmax_topk", False, False),
    (129, 200, 40, 3, "sigmoid_topk", False, False),      # ragged E, T and K
    (1, 64, 16, 4, "softmax_topk", False, False),         # one token
    (127, 320, 20, 2, "softmax_all", True, False),        # an empty K slice (5 k-blocks / 4 CTAs)
    (1000, 1024, 32, 2, "sigmoid_topk", False, True),     # selection bias
    (700, 512, 64, 6, "softmax_topk", True, False),
    (513, 768, 100, 5, "sigmoid_topk", False, False),
    (2048, 2048, 256, 8, "sigmoid_topk", False, False),   # N = 256 MMA, one CTA per SM
    (333, 7168, 200, 8, "softmax_topk", False, True),
]


def run(T, d, E, k, gate, bias, sel, seed):
    w = WORKLOADS["mixtral_prefill"].scaled(T=T, d=d, E=E, k=k, d_ff=8, gate=gate)
    inp = make_inputs(w, device=DEV, seed=seed)
    rb = zipf_log_popularity(E, 1.2).to(DEV) if bias else None
    sb = (torch.randn(E, generator=torch.Generator(device=DEV).manual_seed(seed + 1), device=DEV)
          * 0.05 if sel else None)
    s = L.make_shape(T, d, E, k, 8, gate=gate, dtype=torch.bfloat16)
    ws = L.alloc_workspace(s, DEV)
    out = []
    for rep in range(2):
        logits = torch.full((T, E), float("nan"), device=DEV)
        idx = torch.full((T, k), -1, dtype=torch.int32, device=DEV)
        g = torch.full((T, k), float("nan"), device=DEV)
        st = torch.full((E + 1,), float("nan"), device=DEV)
        if sel:
            L.moe_route_topk_balanced(s, ws, idx, g, sb, x=inp["x"], w_router=inp["w_router"],
                                      router_bias=rb, logits_out=logits, stats=st)
        else:
            L.moe_route_topk(s, ws, idx, g, x=inp["x"], w_router=inp["w_router"], router_bias=rb,
                             logits_out=logits, stats=st)
        out.append((logits, idx, g, st))
    # the top-k kernel on the fused router's own logits
    idx2 = torch.full((T, k), -1, dtype=torch.int32, device=DEV)
    g2 = torch.full((T, k), float("nan"), device=DEV)
    st2 = torch.full((E + 1,), float("nan"), device=DEV)
    if sel:
        L.moe_route_topk_balanced(s, ws, idx2, g2, sb, logits_in=out[0][0], stats=st2)
    else:
        L.moe_route_topk(s, ws, idx2, g2, logits_in=out[0][0], stats=st2)
    torch.cuda.synchronize()
    assert L.moe_get_error(ws) == 0
    return inp, rb, out, (idx2, g2, st2)


@pytest.mark.parametrize("case", CASES, ids=[f"T{c[0]}-d{c[1]}-E{c[2]}-k{c[3]}" for c in CASES])
def test_fused_router(case):
    T, d, E, k, gate, bias, sel = case
    inp, rb, out, ref = run(*case, seed=T + E)
    (logits, idx, g, st), (logits_b, idx_b, g_b, st_b) = out
    # logits against the fp64 oracle on the same bf16 values
    l64 = O.router_logits(host64(inp["x"]), host64(inp["w_router"]),
                          None if rb is None else host64(rb))
    np.testing.assert_allclose(logits.cpu().numpy(), l64, rtol=1e-5, atol=2e-5 * max(1, d / 1024))
    # the routing step is the top-k kernel's, bit for bit, on the same logits
    idx2, g2, st2 = ref
    np.testing.assert_array_equal(idx.cpu().numpy(), idx2.cpu().numpy())
    np.testing.assert_array_equal(g.cpu().numpy(), g2.cpu().numpy())
    np.testing.assert_allclose(st.cpu().numpy(), st2.cpu().numpy(), rtol=2e-6, atol=1e-6)
    # bitwise reproducible
    for a, b in ((logits, logits_b), (idx, idx_b), (g, g_b), (st, st_b)):
        assert torch.equal(a, b)
    # and the routing agrees with the oracle's except among near ties
    if not sel:
        o_idx = O.select_topk(l64, k)
        bad = np.nonzero(np.any(np.sort(o_idx, 1) != np.sort(idx.cpu().numpy(), 1), axis=1))[0]
        assert set(bad.tolist()) <= set(O.near_tie_tokens(l64, k).tolist())
