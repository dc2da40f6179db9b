"""GPU parity of the block-scaled expert path (E4M3 / E2M1 weights with one power-of-two scale
per 32 values, activations quantized to E4M3 blocks on the GPU, tcgen05 kind::mxf8f6f4 MMAs)
against the oracle's forward_mx.

* The activation quantization is an integer decision taken from the same exact value on both
  sides (v * 2^-s of a bf16 input is exact in fp32 and in fp64), so codes and scales must be
  bit-identical.
* The layer: the oracle re-runs steps 3-6 on the GPU's own routing decisions (near ties may
  flip, see the full-size tests), quantizing x and H itself; the only other differences are
  fp32 accumulation, H computed in fp32 before its quantization (a different E4M3 code only
  when H sits within ~1e-6 of a rounding boundary), and the bf16 rounding of the expert rows
  and of y. Bar: relative L2 <= 2e-2 and every kept row within 5 %; losses to 1e-3 relative.
Shapes span 128-row tiles (several per expert, ragged), 32-row tiles (decode), drops, all
three gate modes and both weight formats."""
import numpy as np
import pytest
import torch

import oracle as O
from moe_inputs import WORKLOADS, make_inputs, quantize_weights_mx
from moe_testlib import host64, rel_l2
from mixture_experts_layer_92_b300 import _lib as L

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def test_mx_quantize_bitexact():
    g = torch.Generator(device=DEV).manual_seed(3)
    x = (torch.randn(70, 512, generator=g, device=DEV) *
         torch.exp2(torch.randint(-20, 20, (70, 1), generator=g, device=DEV).float()))
    x[0, :32] = 0.0                         # an all-zero block: the smallest scale
    x[1, :32] = -0.0
    x[2, 32:64] = 1e-30                     # tiny values
    x[3, 64:96] = 3.0e38                    # near the top of the range
    x[4, 5] = 448.0 * 2.0 ** -3             # exactly on a scale boundary
    x = x.to(torch.bfloat16)
    codes = torch.full((70, 512), 0xAA, dtype=torch.uint8, device=DEV)
    scales = torch.full((70, 16), 0xAA, dtype=torch.uint8, device=DEV)
    L.moe_mx_quantize(x, codes, scales)
    torch.cuda.synchronize()
    c_ref, s_ref = O.mx_quantize(host64(x), "e4m3")
    np.testing.assert_array_equal(codes.cpu().numpy(), c_ref)
    np.testing.assert_array_equal(scales.cpu().numpy().astype(np.int64), s_ref + 127)


def mx_layer(w, fmt, seed=0):
    inp = make_inputs(w, device=DEV, seed=seed)
    C = w.T if w.cf is None else O.capacity(w.cf, w.T, w.k, w.E)
    mx = {nm: quantize_weights_mx(inp[nm], fmt, host_codes=True) for nm in ("w1", "w3", "w2")}
    s = L.make_shape(w.T, w.d, w.E, w.k, w.d_ff, gate=w.gate, dtype=torch.bfloat16, capacity=C,
                     alpha=w.alpha, beta=w.beta)
    ws = L.alloc_workspace_mx(s, DEV)
    y = torch.full_like(inp["x"], float("nan"))
    counts = torch.zeros(w.E, dtype=torch.int32, device=DEV)
    dropped = torch.zeros(1, dtype=torch.int32, device=DEV)
    losses = torch.zeros(2, device=DEV)
    L.moe_forward_mx(s, ws, fmt, inp["x"], inp["w_router"], mx["w1"]["q"], mx["w1"]["sf"],
                     mx["w3"]["q"], mx["w3"]["sf"], mx["w2"]["q"], mx["w2"]["sf"], y,
                     router_bias=inp["router_bias"], counts=counts, dropped=dropped,
                     losses=losses)
    idx = torch.empty(w.T, w.k, dtype=torch.int32, device=DEV)
    gate = torch.empty(w.T, w.k, device=DEV)
    L.moe_route_topk(s, ws, idx, gate, x=inp["x"], w_router=inp["w_router"],
                     router_bias=inp["router_bias"])
    torch.cuda.synchronize()
    assert L.moe_get_error(ws) == 0
    mxw = dict(fmt=fmt)
    for nm in ("w1", "w3", "w2"):
        mxw[nm], mxw[nm + "_s"] = mx[nm]["codes"], mx[nm]["s"]
    bias = None if inp["router_bias"] is None else host64(inp["router_bias"])
    ref = O.forward_mx(host64(inp["x"]), host64(inp["w_router"]), mxw, k=w.k, mode=w.gate, C=C,
                       router_bias=bias, alpha=w.alpha, beta=w.beta,
                       idx_override=idx.cpu().numpy().astype(np.int64))
    return dict(y=y.double().cpu().numpy(), counts=counts.cpu().numpy(),
                dropped=int(dropped.item()), losses=losses.cpu().numpy(), ref=ref)


CASES = [
    # name, T, d, E, k, d_ff, gate, cf, fmt
    ("tiles128_e4m3", 300, 512, 8, 2, 384, "softmax_topk", None, "e4m3"),
    ("tiles128_e2m1", 300, 256, 4, 2, 256, "sigmoid_topk", None, "e2m1"),
    ("multi_tile_experts", 600, 256, 4, 1, 128, "softmax_topk", None, "e4m3"),
    ("decode_e4m3", 16, 512, 8, 2, 256, "softmax_topk", None, "e4m3"),
    ("decode_e2m1", 24, 256, 8, 2, 384, "softmax_topk", None, "e2m1"),
    ("drops_softmax_all", 400, 256, 16, 1, 128, "softmax_all", 1.0, "e4m3"),
    ("drops_e2m1", 333, 512, 8, 3, 256, "sigmoid_topk", 0.8, "e2m1"),
    # degenerate corners: one expert, k = E, one token, capacity 1
    ("single_expert_e4m3", 200, 256, 1, 1, 128, "softmax_topk", None, "e4m3"),
    ("k_equals_E_e2m1", 150, 256, 4, 4, 128, "softmax_all", None, "e2m1"),
    ("one_token_e4m3", 1, 512, 16, 4, 256, "sigmoid_topk", None, "e4m3"),
    ("capacity_one_e4m3", 256, 256, 32, 1, 128, "softmax_topk", 0.125, "e4m3"),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_mx_layer(case):
    name, T, d, E, k, F, gate, cf, fmt = case
    w = WORKLOADS["mixtral_prefill"].scaled(T=T, d=d, E=E, k=k, d_ff=F, gate=gate, cf=cf)
    out = mx_layer(w, fmt, seed=T + E)
    ref = out["ref"]
    np.testing.assert_array_equal(out["counts"], ref["dispatch"]["counts"])
    assert out["dropped"] == ref["dispatch"]["dropped"]
    err = rel_l2(out["y"], ref["y"])
    assert err < 2e-2, f"{name}: relative L2 {err:.3e}"
    # every token with a kept assignment within 5 %
    kept = np.any(ref["dispatch"]["inv"].reshape(T, k) >= 0, axis=1)
    num = np.linalg.norm(out["y"][kept] - ref["y"][kept], axis=1)
    den = np.linalg.norm(ref["y"][kept], axis=1)
    assert np.all(num <= 0.05 * den + 1e-6), f"{name}: worst row {np.max(num / den):.3e}"
    assert np.all(out["y"][~kept] == 0)
    assert out["losses"][0] == pytest.approx(ref["l_aux"], rel=1e-3)
    assert out["losses"][1] == pytest.approx(ref["l_z"], rel=1e-3)
    print(f"{name}: rel L2 {err:.2e}")


def test_mx_rejects_unsupported_shapes():
    s = L.make_shape(64, 200, 8, 2, 128, dtype=torch.bfloat16)       # d % 256 != 0
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device=DEV)
    dummy = torch.zeros(1 << 16, dtype=torch.uint8, device=DEV)
    x = torch.zeros(64, 200, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(L.MoeError) as ei:
        L.moe_forward_mx(s, ws, "e4m3", x, x, dummy, dummy, dummy, dummy, dummy, dummy, x)
    assert ei.value.status == -2


@pytest.mark.slow
@pytest.mark.parametrize("name,fmt", [("mixtral_decode", "e4m3"), ("mixtral_decode", "e2m1"),
                                      ("switch_top1", "e4m3")])
def test_mx_full_size_sampled(name, fmt):
    """The block-scaled layer at full size, in the launch configuration bench.py times, on
    sampled tokens that the oracle computes one expert at a time (weights decoded per expert),
    on the GPU's routing of the whole batch; counts and drops over all tokens."""
    w = WORKLOADS[name]
    inp = make_inputs(w, device=DEV)
    C = w.T if w.cf is None else O.capacity(w.cf, w.T, w.k, w.E)
    mx = {nm: quantize_weights_mx(inp[nm], fmt, host_codes=True) for nm in ("w1", "w3", "w2")}
    s = L.make_shape(w.T, w.d, w.E, w.k, w.d_ff, gate=w.gate, dtype=torch.bfloat16, capacity=C,
                     alpha=w.alpha, beta=w.beta)
    ws = L.alloc_workspace_mx(s, DEV)
    y = torch.empty_like(inp["x"])
    counts = torch.zeros(w.E, dtype=torch.int32, device=DEV)
    dropped = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.moe_forward_mx(s, ws, fmt, inp["x"], inp["w_router"], mx["w1"]["q"], mx["w1"]["sf"],
                     mx["w3"]["q"], mx["w3"]["sf"], mx["w2"]["q"], mx["w2"]["sf"], y,
                     router_bias=inp["router_bias"], counts=counts, dropped=dropped)
    idx = torch.empty(w.T, w.k, dtype=torch.int32, device=DEV)
    gate = torch.empty(w.T, w.k, device=DEV)
    L.moe_route_topk(s, ws, idx, gate, x=inp["x"], w_router=inp["w_router"],
                     router_bias=inp["router_bias"])
    torch.cuda.synchronize()
    assert L.moe_get_error(ws) == 0
    gidx = idx.cpu().numpy().astype(np.int64)
    disp = O.dispatch(gidx, w.E, C)
    np.testing.assert_array_equal(counts.cpu().numpy(), disp["counts"])
    assert int(dropped.item()) == disp["dropped"]
    bias = None if inp["router_bias"] is None else host64(inp["router_bias"])
    x64 = host64(inp["x"])
    logits = O.router_logits(x64, host64(inp["w_router"]), bias)
    tokens = np.sort(np.random.default_rng(9).choice(w.T, size=min(w.T, 32), replace=False))
    inv = disp["inv"].reshape(w.T, w.k)[tokens]
    g = O.gates(logits[tokens], gidx[tokens], w.gate)
    yref = np.zeros((len(tokens), w.d))
    for e in np.unique(gidx[tokens][inv >= 0]):
        W = {nm: O.mx_dequantize(mx[nm]["codes"][e], mx[nm]["s"][e], fmt) for nm in ("w1", "w3", "w2")}
        tl, sl = np.nonzero((gidx[tokens] == e) & (inv >= 0))
        rows = O.swiglu_ffn_mx(x64[tokens[tl]], W["w1"], W["w3"], W["w2"])
        for i, (t, sidx) in enumerate(zip(tl, sl)):
            yref[t] += g[t, sidx] * rows[i]
    got = y[torch.as_tensor(tokens, device=DEV)].double().cpu().numpy()
    err = rel_l2(got, yref)
    print(f"{name} {fmt}: sampled rel L2 {err:.3e}, dropped {disp['dropped']}")
    assert err < 2e-2
