"""A seeded sweep of layer shapes through moe_forward, each checked against the fp64 oracle
run on the GPU's own routing decisions (top-k parity is tested bit for bit elsewhere; here a
mismatch may only fall on a near tie). The shapes are drawn, from a fixed seed, over what the
boundary accepts: ragged K and N (d and d_ff any multiple of 8, of 4 for fp32), 1..48
experts, k up to 6, the three gate modes, no drop / capacity factors that drop, a shared
expert, a Zipf-skewed router and batches from one token up; then the degenerate corners a
draw need not reach (a single expert, k = E with and without drops, one token over 256
experts, d = d_ff = 8, capacity 1, E = 1024). Bars: bf16 relative L2 <= 2e-2, fp32 max-abs
<= 1e-4 RMS; counts and drops exact; losses to 1e-3 (bf16) / 1e-5 (fp32)."""
import numpy as np
import pytest

import oracle as O
from moe_inputs import WORKLOADS, make_inputs
from moe_testlib import capacity_of, gpu_forward, host64, rel_l2, routing_check

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
GATES = ("softmax_all", "softmax_topk", "sigmoid_topk")


def draw(seed: int, dtype: str):
    r = np.random.default_rng(1000 + seed)
    step = 8 if dtype == "bf16" else 4
    E = int(r.integers(1, 49))
    return WORKLOADS["mixtral_prefill"].scaled(
        name=f"random{seed}_{dtype}",
        T=int(r.choice([1, int(r.integers(2, 64)), int(r.integers(64, 700))])),
        d=int(step * r.integers(1, 520 // step + 1)),
        E=E,
        k=int(r.integers(1, min(E, 6) + 1)),
        d_ff=int(step * r.integers(1, 640 // step + 1)),
        gate=str(r.choice(GATES)),
        dtype=dtype,
        cf=[None, 0.5, 1.0, 1.5][int(r.integers(0, 4))],
        d_ff_shared=int(step * r.integers(1, 256 // step + 1)) if r.random() < 0.3 else 0,
        zipf_s=1.2 if r.random() < 0.3 else None)


CASES = [draw(i, "bf16") for i in range(16)] + [draw(i, "f32") for i in range(16, 24)]


def edge(name, **kw):
    base = dict(gate="softmax_topk", dtype="bf16", cf=None, d_ff_shared=0, zipf_s=None)
    base.update(kw)
    return WORKLOADS["mixtral_prefill"].scaled(name=name, **base)


# the degenerate corners of the method, which a draw need not reach
EDGES = [
    edge("edge_single_expert", T=300, d=64, E=1, k=1, d_ff=48),
    edge("edge_single_expert_sigmoid_f32", T=77, d=32, E=1, k=1, d_ff=36, gate="sigmoid_topk",
         dtype="f32"),
    edge("edge_k_equals_E", T=200, d=128, E=8, k=8, d_ff=64),
    edge("edge_k_equals_E_shared_drop", T=150, d=64, E=4, k=4, d_ff=40, gate="softmax_all",
         cf=0.5, d_ff_shared=32),
    edge("edge_one_token_256_experts", T=1, d=256, E=256, k=8, d_ff=32, gate="sigmoid_topk"),
    edge("edge_smallest_dims", T=40, d=8, E=3, k=2, d_ff=8),
    edge("edge_capacity_one_E256", T=512, d=128, E=256, k=1, d_ff=32, gate="softmax_all",
         cf=0.25, zipf_s=1.2),
    edge("edge_unfused_router_E1024", T=96, d=64, E=1024, k=3, d_ff=16, cf=2.0),
]
CASES += EDGES


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_random_shape_matches_oracle(w):
    inp = make_inputs(w, device=DEV, seed=w.T + w.d)
    C = capacity_of(w)
    g = gpu_forward(w, inp, C=C)
    assert g["error"] == 0
    bias = None if inp["router_bias"] is None else host64(inp["router_bias"])
    x64 = host64(inp["x"])
    logits64 = O.router_logits(x64, host64(inp["w_router"]), bias)
    gidx = g["idx"].cpu().numpy().astype(np.int64)
    bad, ties = routing_check(logits64, gidx, w.k)
    assert set(bad.tolist()) <= set(ties.tolist()), (bad, ties)
    shared = {}
    if w.d_ff_shared:
        shared = dict(w1s=host64(inp["w1s"]), w3s=host64(inp["w3s"]), w2s=host64(inp["w2s"]))
    ref = O.forward(x64, host64(inp["w_router"]), host64(inp["w1"]), host64(inp["w3"]),
                    host64(inp["w2"]), k=w.k, mode=w.gate, C=C, router_bias=bias,
                    alpha=w.alpha, beta=w.beta, idx_override=gidx, **shared)
    y = g["y"].double().cpu().numpy()
    assert np.isfinite(y).all()
    if w.dtype == "bf16":
        assert rel_l2(y, ref["y"]) < 2e-2, rel_l2(y, ref["y"])
        ltol = 1e-3
    else:
        rms = np.sqrt(np.mean(ref["y"] ** 2))
        assert np.abs(y - ref["y"]).max() <= 1e-4 * rms
        ltol = 1e-5
    np.testing.assert_array_equal(g["counts"].cpu().numpy(), ref["dispatch"]["counts"])
    assert int(g["dropped"].item()) == ref["dispatch"]["dropped"]
    l = g["losses"].cpu().numpy()
    assert l[0] == pytest.approx(ref["l_aux"], rel=ltol, abs=1e-7)
    assert l[1] == pytest.approx(ref["l_z"], rel=ltol, abs=1e-7)
