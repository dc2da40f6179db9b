"""GPU parity of 8-bit (E4M3, per-row scale) expert weights against the oracle run on the
decoded weights: the tensor cores multiply exact fp16 copies of the codes by fp16 copies of
the activations (exact for these inputs) and the scales are applied to the fp32
accumulators; H is rounded to fp16 (finer than bf16), so the bf16 bound (relative L2 <=
2e-2, every kept row within 5%) applies unchanged. Activations beyond fp16's range are
reported through the error word, not silently turned into infinities."""
import numpy as np
import pytest
import torch

import oracle as O
from moe_inputs import WORKLOADS, make_inputs, quantize_rows_e4m3
from moe_testlib import capacity_of, host64, rel_l2, routing_check
from mixture_experts_layer_92_b300 import _lib as L

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def quantized(inp):
    q = {}
    for name in ("w1", "w3", "w2"):
        q[name + "q"], q[name + "s"] = quantize_rows_e4m3(inp[name])
    return q


def dequant_expert(q, name, e):
    return O.dequantize_rows(q[name + "q"][e].cpu().numpy(), q[name + "s"][e].cpu().numpy())


@pytest.mark.parametrize("T,d,E,k,F", [
    (64, 256, 8, 2, 1120),      # 224-wide gate/up tiles
    (700, 256, 6, 2, 384),      # 256-wide, several row tiles per expert
    (300, 208, 5, 1, 336),      # ragged K (208 = 3*64 + 16) and ragged N (336)
    (32, 256, 8, 2, 1120),      # decode-sized groups (<= 32 rows): 32-row A tiles
    (1, 256, 4, 2, 512),        # one token
    (20, 208, 5, 1, 336),       # short row tiles with ragged K and N
    (50, 256, 1, 1, 256),       # one expert
])
def test_grouped_swiglu_fp8_weights(T, d, E, k, F):
    w = WORKLOADS["mixtral_prefill"].scaled(T=T, d=d, E=E, k=k, d_ff=F)
    inp = make_inputs(w, device=DEV, seed=7)
    q = quantized(inp)
    l64 = np.random.default_rng(7).normal(size=(T, E))
    idx = O.select_topk(l64, k)
    g = O.gates(l64, idx, "softmax_topk")
    disp = O.dispatch(idx, E, T)
    s = L.make_shape(T, d, E, k, F, dtype=torch.bfloat16)
    ws = L.alloc_workspace(s, DEV)
    A, R = T * k, int(disp["offsets"][-1])
    perm = torch.zeros(A, dtype=torch.int32, device=DEV)
    perm[:R] = torch.from_numpy(disp["perm"].astype(np.int32)).to(DEV)
    offsets = torch.from_numpy(disp["offsets"].astype(np.int32)).to(DEV)
    y_perm = torch.full((A, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    L.moe_grouped_swiglu_fp8w(s, ws, inp["x"], perm, offsets, q["w1q"], q["w1s"], q["w3q"],
                              q["w3s"], q["w2q"], q["w2s"], y_perm,
                              topk_gate=torch.from_numpy(g.astype(np.float32)).to(DEV))
    torch.cuda.synchronize()
    assert L.moe_get_error(ws) == 0
    x64 = host64(inp["x"])
    W1 = np.stack([dequant_expert(q, "w1", e) for e in range(E)])
    W3 = np.stack([dequant_expert(q, "w3", e) for e in range(E)])
    W2 = np.stack([dequant_expert(q, "w2", e) for e in range(E)])
    ref = O.expert_outputs(x64, disp, k, W1, W3, W2) * g.reshape(-1)[disp["perm"]][:, None]
    got = y_perm[:R].double().cpu().numpy()
    assert rel_l2(got, ref) < 2e-2, rel_l2(got, ref)
    row_err = np.linalg.norm(got - ref, axis=1) / np.maximum(np.linalg.norm(ref, axis=1), 1e-30)
    assert row_err.max() < 5e-2
    assert torch.isnan(y_perm[R:].float()).all()


def test_forward_fp8_weights_decode_step():
    """The full Mixtral-shaped decode step (T = 32) on 8-bit weights, every token against
    the oracle on the decoded weights."""
    w = WORKLOADS["mixtral_decode"]
    inp = make_inputs(w, device=DEV)
    q = quantized(inp)
    s = L.make_shape(w.T, w.d, w.E, w.k, w.d_ff, gate=w.gate, dtype=torch.bfloat16)
    ws = L.alloc_workspace(s, DEV)
    y = torch.empty_like(inp["x"])
    counts = torch.empty(w.E, dtype=torch.int32, device=DEV)
    losses = torch.empty(2, device=DEV)
    L.moe_forward_fp8w(s, ws, inp["x"], inp["w_router"], q["w1q"], q["w1s"], q["w3q"], q["w3s"],
                       q["w2q"], q["w2s"], y, counts=counts, losses=losses)
    idx = torch.empty(w.T, w.k, dtype=torch.int32, device=DEV)
    gate = torch.empty(w.T, w.k, device=DEV)
    L.moe_route_topk(s, ws, idx, gate, x=inp["x"], w_router=inp["w_router"])
    torch.cuda.synchronize()
    assert L.moe_get_error(ws) == 0
    x64 = host64(inp["x"])
    logits64 = O.router_logits(x64, host64(inp["w_router"]))
    gidx = idx.cpu().numpy().astype(np.int64)
    bad, ties = routing_check(logits64, gidx, w.k)
    assert set(bad.tolist()) <= set(ties.tolist())
    disp = O.dispatch(gidx, w.E, w.T)
    np.testing.assert_array_equal(counts.cpu().numpy(), disp["counts"])
    rows = np.zeros((disp["perm"].shape[0], w.d))
    for e in range(w.E):
        lo, hi = int(disp["offsets"][e]), int(disp["offsets"][e + 1])
        if hi > lo:
            rows[lo:hi] = O.swiglu_ffn(x64[disp["perm"][lo:hi] // w.k], dequant_expert(q, "w1", e),
                                       dequant_expert(q, "w3", e), dequant_expert(q, "w2", e))
    yref = O.combine(O.gates(logits64, gidx, w.gate), disp["inv"], rows, w.T, w.k)
    assert rel_l2(y.double().cpu().numpy(), yref) < 2e-2
    assert losses[0].item() == pytest.approx(O.aux_loss(logits64, gidx, w.alpha), rel=1e-3)


def test_fp8_weights_flag_activations_beyond_fp16_range():
    """x holds one value (2^17, a bf16 number) that fp16 cannot represent: the call records
    MOE_ERR_NONFINITE instead of returning a silently wrong y; an in-range x leaves no error."""
    w = WORKLOADS["mixtral_decode"].scaled(T=16, d=256, d_ff=512)
    inp = make_inputs(w, device=DEV, seed=3)
    q = quantized(inp)
    s = L.make_shape(w.T, w.d, w.E, w.k, w.d_ff, gate=w.gate, dtype=torch.bfloat16)
    y = torch.empty_like(inp["x"])
    for big, want in ((False, 0), (True, L.MOE_ERR_NONFINITE)):
        ws = L.alloc_workspace(s, DEV)
        x = inp["x"].clone()
        if big:
            x[5, 17] = 2.0 ** 17
        L.moe_forward_fp8w(s, ws, x, inp["w_router"], q["w1q"], q["w1s"], q["w3q"], q["w3s"],
                           q["w2q"], q["w2s"], y)
        torch.cuda.synchronize()
        assert L.moe_get_error(ws) == want


def test_fp8_weights_subnormal_codes_are_not_flushed():
    """Every weight an E4M3 subnormal code (0x01..0x07, either sign; values 2^-9 .. 7*2^-9):
    the converters turn them into fp16 subnormals, which the tensor cores must use as they
    are (a flush to zero would make y = 0)."""
    T, d, E, k, F = 64, 256, 4, 2, 256
    w = WORKLOADS["mixtral_prefill"].scaled(T=T, d=d, E=E, k=k, d_ff=F)
    inp = make_inputs(w, device=DEV, seed=4)
    g = torch.Generator(device="cpu").manual_seed(4)
    q = {}
    for name, shape in (("w1", (E, F, d)), ("w3", (E, F, d)), ("w2", (E, d, F))):
        mag = torch.randint(1, 8, shape, generator=g, dtype=torch.uint8)
        sign = torch.randint(0, 2, shape, generator=g, dtype=torch.uint8) * 128
        q[name + "q"] = (mag | sign).to(DEV)
        q[name + "s"] = torch.full(shape[:2], 4.0, device=DEV)
    l64 = np.random.default_rng(4).normal(size=(T, E))
    idx = O.select_topk(l64, k)
    gt = O.gates(l64, idx, "softmax_topk")
    disp = O.dispatch(idx, E, T)
    s = L.make_shape(T, d, E, k, F, dtype=torch.bfloat16)
    ws = L.alloc_workspace(s, DEV)
    R = int(disp["offsets"][-1])
    perm = torch.zeros(T * k, dtype=torch.int32, device=DEV)
    perm[:R] = torch.from_numpy(disp["perm"].astype(np.int32)).to(DEV)
    offsets = torch.from_numpy(disp["offsets"].astype(np.int32)).to(DEV)
    y_perm = torch.zeros((T * k, d), dtype=torch.bfloat16, device=DEV)
    L.moe_grouped_swiglu_fp8w(s, ws, inp["x"], perm, offsets, q["w1q"], q["w1s"], q["w3q"],
                              q["w3s"], q["w2q"], q["w2s"], y_perm,
                              topk_gate=torch.from_numpy(gt.astype(np.float32)).to(DEV))
    torch.cuda.synchronize()
    assert L.moe_get_error(ws) == 0
    W = {n: np.stack([dequant_expert(q, n, e) for e in range(E)]) for n in ("w1", "w3", "w2")}
    assert np.abs(W["w1"]).max() < 2.0 ** -6 * 4.0          # all subnormal codes
    ref = O.expert_outputs(host64(inp["x"]), disp, k, W["w1"], W["w3"], W["w2"])
    ref *= gt.reshape(-1)[disp["perm"]][:, None]
    assert rel_l2(y_perm[:R].double().cpu().numpy(), ref) < 2e-2
