"""GPU parity of the bf16 path (tcgen05 grouped GEMMs, tcgen05 router) against the oracle.

Bar for bf16 workloads: relative L2 error of y <= 2e-2 and the balance loss within 1e-3
relative. The oracle sees the same bf16-rounded inputs in fp64; the GPU rounds the hidden
activations and the expert outputs to bf16, which the bound absorbs. Shapes span several
128-row tiles, several output-column tiles and ragged tails in rows, columns and K."""
import numpy as np
import pytest
import torch

import oracle as O
from moe_inputs import WORKLOADS, make_inputs
from moe_testlib import capacity_of, gpu_forward, host64, oracle_y_for_tokens, rel_l2, routing_check
from mixture_experts_layer_92_b300 import _lib as L

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

BF16_TOL = 2e-2


def dev_inputs(w, seed=0):
    return make_inputs(w, device=DEV, seed=seed)


def test_router_tcgen05_logits():
    """bf16 x . W_r^T with fp32 accumulation on the tensor cores vs fp64 on the same
    bf16 values; E = 8 (N = 16 tile), 128, 256 and a ragged E = 40."""
    for (T, d, E) in [(300, 256, 8), (1000, 1024, 128), (200, 7168, 256), (129, 200, 40)]:
        w = WORKLOADS["mixtral_prefill"].scaled(T=T, d=d, E=E, k=2, d_ff=64)
        inp = dev_inputs(w, seed=T)
        s = L.make_shape(T, d, E, 2, 64, dtype=torch.bfloat16)
        ws = L.alloc_workspace(s, DEV)
        logits = torch.empty(T, E, device=DEV)
        idx = torch.empty(T, 2, dtype=torch.int32, device=DEV)
        gate = torch.empty(T, 2, device=DEV)
        L.moe_route_topk(s, ws, idx, gate, x=inp["x"], w_router=inp["w_router"], logits_out=logits)
        torch.cuda.synchronize()
        assert L.moe_get_error(ws) == 0
        ref = O.router_logits(host64(inp["x"]), host64(inp["w_router"]))
        np.testing.assert_allclose(logits.cpu().numpy(), ref, rtol=1e-5, atol=2e-5)


def grouped_check(T, d, E, k, F, Fs=0, cf=None, gate="softmax_topk", seed=0, idx=None):
    """moe_grouped_swiglu alone, on the oracle's own dispatch of random routing (or of the
    given expert indices [T, k])."""
    w = WORKLOADS["mixtral_prefill"].scaled(T=T, d=d, E=E, k=k, d_ff=F, d_ff_shared=Fs, cf=cf,
                                            gate=gate)
    inp = dev_inputs(w, seed=seed)
    C = capacity_of(w)
    l64 = np.random.default_rng(seed).normal(size=(T, E))
    if idx is None:
        idx = O.select_topk(l64, k)
    g = O.gates(l64, idx, gate)
    disp = O.dispatch(idx, E, C)
    s = L.make_shape(T, d, E, k, F, gate=gate, dtype=torch.bfloat16, capacity=C, d_ff_shared=Fs)
    ws = L.alloc_workspace(s, DEV)
    A = T * k
    perm = torch.zeros(A, dtype=torch.int32, device=DEV)
    R = int(disp["offsets"][-1])
    perm[:R] = torch.from_numpy(disp["perm"].astype(np.int32)).to(DEV)
    offsets = torch.from_numpy(disp["offsets"].astype(np.int32)).to(DEV)
    gate_t = torch.from_numpy(g.astype(np.float32)).to(DEV)
    y_perm = torch.full((A, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    y_sh = torch.empty(T, d, dtype=torch.bfloat16, device=DEV) if Fs else None
    L.moe_grouped_swiglu(s, ws, inp["x"], perm, offsets, inp["w1"], inp["w3"], inp["w2"], y_perm,
                         topk_gate=gate_t, w1s=inp["w1s"], w3s=inp["w3s"], w2s=inp["w2s"],
                         y_shared=y_sh)
    torch.cuda.synchronize()
    assert L.moe_get_error(ws) == 0
    x64 = host64(inp["x"])
    rows = O.expert_outputs(x64, disp, k, host64(inp["w1"]), host64(inp["w3"]), host64(inp["w2"]))
    gflat = g.reshape(-1)[disp["perm"]]
    ref = rows * gflat[:, None]
    got = y_perm[:R].double().cpu().numpy()
    assert np.isfinite(got).all()
    assert rel_l2(got, ref) < BF16_TOL, rel_l2(got, ref)
    # row by row: every kept row is close (no tile or row mapping error hides in the mean)
    row_err = np.linalg.norm(got - ref, axis=1) / np.maximum(np.linalg.norm(ref, axis=1), 1e-30)
    assert row_err.max() < 5e-2, row_err.max()
    # rows past R untouched
    assert torch.isnan(y_perm[R:].float()).all()
    if Fs:
        sref = O.swiglu_ffn(x64, host64(inp["w1s"]), host64(inp["w3s"]), host64(inp["w2s"]))
        assert rel_l2(y_sh.double().cpu().numpy(), sref) < BF16_TOL


@pytest.mark.parametrize("T,d,E,k,F", [
    (700, 256, 6, 2, 384),      # ~233 rows per expert: 2-3 row tiles; 3 column tiles of H
    (300, 200, 5, 1, 328),      # ragged K (200 = 3*64 + 8) and ragged N (328)
    (64, 512, 8, 2, 512),       # ~16 rows per expert: tiles straddle expert boundaries
    (2048, 1024, 4, 2, 1024),   # 8 row tiles per expert, persistent loop over many tiles
    (64, 256, 8, 2, 1120),      # 1120 = 10 * 112: the 224-wide gate/up MMA (112 H columns)
])
def test_grouped_swiglu_tcgen05(T, d, E, k, F):
    grouped_check(T, d, E, k, F)


def test_grouped_swiglu_tcgen05_256_row_tiles():
    """The down projection runs 256-row CTA tiles (two MMAs per weight tile) when d_ff >= 8192
    and experts average >= 512 rows. Loads 612 / 1224 / 642 rows: last tiles with the second
    half empty (100 rows), partly valid (200 rows) and nearly empty (130 rows: 2 rows in the
    second half)."""
    counts = [612, 1224, 642]
    idx = np.concatenate([np.full(c, e) for e, c in enumerate(counts)])
    idx = idx[np.random.default_rng(5).permutation(idx.shape[0])][:, None]
    grouped_check(int(idx.shape[0]), 256, 3, 1, 8192, idx=idx, seed=5)


def test_grouped_swiglu_tcgen05_256_row_tiles_shared_ragged():
    """256-row tiles in both expert GEMMs (768 rows per expert, d_ff >= 8192) together with
    the shared expert's tiles (1536 rows, d_ff_shared = 200), on a ragged K of gate/up
    (d = 328 = 5 * 64 + 8) and a ragged N of the down projection (328 = 256 + 72)."""
    grouped_check(1536, 328, 2, 1, 8192, Fs=200, seed=6)


def test_grouped_swiglu_tcgen05_capacity_and_shared():
    grouped_check(500, 256, 8, 2, 256, Fs=128, cf=0.75, gate="sigmoid_topk", seed=3)


@pytest.mark.parametrize("T,d,E,k,F,Fs,cf", [
    (32, 256, 8, 2, 1120, 0, None),   # decode-sized: every expert <= 32 rows, 224-wide MMA
    (1, 256, 4, 2, 512, 0, None),     # one token: two 1-row groups, two empty ones
    (32, 512, 8, 2, 512, 128, None),  # with the shared expert (32 rows)
    (20, 200, 5, 1, 328, 0, None),    # ragged K (200) and N (328)
    (200, 256, 8, 2, 256, 0, 0.5),    # C = 25: many tokens, every group cut to <= 25 rows
])
def test_grouped_swiglu_tcgen05_short_row_tiles(T, d, E, k, F, Fs, cf):
    """No group above 32 rows: the GEMMs load 32-row A tiles (the MMA's other 96 rows read
    bytes of the same stage and are never stored)."""
    grouped_check(T, d, E, k, F, Fs=Fs, cf=cf, seed=T)


def layer_check(w, seed=0, sample=None):
    inp = dev_inputs(w, seed=seed)
    C = capacity_of(w)
    g = gpu_forward(w, inp, C=C)
    assert g["error"] == 0
    bias = None if inp["router_bias"] is None else host64(inp["router_bias"])
    logits64 = O.router_logits(host64(inp["x"]), host64(inp["w_router"]), bias)
    gidx = g["idx"].cpu().numpy().astype(np.int64)
    bad, ties = routing_check(logits64, gidx, w.k)
    assert set(bad.tolist()) <= set(ties.tolist())
    disp = O.dispatch(gidx, w.E, C)
    np.testing.assert_array_equal(g["counts"].cpu().numpy(), disp["counts"])
    assert int(g["dropped"].item()) == disp["dropped"]
    tokens = np.arange(w.T) if sample is None else sample
    yref = oracle_y_for_tokens(w, inp, logits64, gidx, disp["inv"], tokens)
    y = g["y"][torch.as_tensor(tokens, device=DEV)].double().cpu().numpy()
    assert rel_l2(y, yref) < BF16_TOL, rel_l2(y, yref)
    l = g["losses"].cpu().numpy()
    assert l[0] == pytest.approx(O.aux_loss(logits64, gidx, w.alpha), rel=1e-3)
    assert l[1] == pytest.approx(O.z_loss(logits64, w.beta), rel=1e-3)
    return g, disp, len(bad)


@pytest.mark.parametrize("name", ["mixtral_prefill", "mixtral_prefill_256", "switch_top1",
                                  "deepseek_fine", "mixtral_decode"])
def test_bf16_layer_scaled_workloads(name):
    """Each bf16 workload's recipe (gate mode, k, bias, capacity, shared expert) at reduced
    sizes that still span several tiles and ragged tails (mixtral_prefill_256: ~512 rows per
    expert, so the expert GEMMs run 256-row CTA tiles)."""
    base = WORKLOADS[name.replace("_256", "")]
    small = dict(mixtral_prefill=dict(T=600, d=512, d_ff=768),
                 mixtral_prefill_256=dict(T=2048, d=512, d_ff=768),
                 switch_top1=dict(T=1500, d=256, E=32, d_ff=384),
                 deepseek_fine=dict(T=400, d=384, E=24, k=4, d_ff=256, d_ff_shared=256),
                 mixtral_decode=dict(T=32, d=512, d_ff=1024))[name]
    g, disp, nflip = layer_check(base.scaled(**small), seed=1)
    if base.cf is not None:
        assert disp["dropped"] > 0


def test_bf16_deterministic():
    w = WORKLOADS["deepseek_fine"].scaled(T=300, d=256, E=16, k=4, d_ff=256, d_ff_shared=128)
    inp = dev_inputs(w)
    a = gpu_forward(w, inp)
    b = gpu_forward(w, inp)
    assert torch.equal(a["y"], b["y"]) and torch.equal(a["losses"], b["losses"])
    assert torch.equal(a["idx"], b["idx"]) and torch.equal(a["stats"], b["stats"])


def test_forward_host_stream_matches_device_forward():
    """MoELayer.forward_host_stream (the C ABI's host pipeline: uploads, layers and downloads
    on three streams over several batches, two device slots reused in turn) returns, batch by
    batch, exactly the y and losses of the device-resident forward; batches of several sizes,
    an empty one included, and two calls on the same pipeline."""
    import mixture_experts_layer_92_b300 as moe
    w = WORKLOADS["mixtral_prefill"].scaled(T=256, d=256, E=8, k=2, d_ff=384)
    inp = dev_inputs(w)
    layer = moe.MoELayer(inp["w_router"], inp["w1"], inp["w3"], inp["w2"], k=w.k, gate=w.gate,
                         max_tokens=w.T)
    sizes = [256, 200, 0, 256, 33, 256, 129]
    xs = [torch.randn(T, w.d, generator=torch.Generator().manual_seed(i)).to(torch.bfloat16)
          .pin_memory() for i, T in enumerate(sizes)]
    ys = [torch.full((T, w.d), float("nan"), dtype=torch.bfloat16).pin_memory() for T in sizes]
    ls = [torch.full((2,), float("nan")).pin_memory() for _ in sizes]
    layer.forward_host_stream(xs[:4], ys[:4], ls[:4])
    layer.forward_host_stream(xs[4:], ys[4:], ls[4:])
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    for xh, yh, lh in zip(xs, ys, ls):
        ref = layer.forward(xh.to(DEV))
        torch.cuda.synchronize()
        assert torch.equal(yh, ref.cpu())
        assert torch.equal(lh, layer.losses.cpu())


def test_forward_host_entry_point_matches_device_forward():
    """moe_forward_host (host x in, the layer, host y and losses out, on one stream) returns
    exactly what moe_forward returns on the same inputs, including a shared expert."""
    import mixture_experts_layer_92_b300 as moe
    w = WORKLOADS["deepseek_fine"].scaled(T=333, d=256, E=16, k=4, d_ff=256, d_ff_shared=128)
    inp = dev_inputs(w)
    layer = moe.MoELayer(inp["w_router"], inp["w1"], inp["w3"], inp["w2"], k=w.k, gate=w.gate,
                         router_bias=inp["router_bias"], w1s=inp["w1s"], w3s=inp["w3s"],
                         w2s=inp["w2s"], max_tokens=w.T)
    ref = layer.forward(inp["x"])
    torch.cuda.synchronize()
    x_host = inp["x"].cpu().pin_memory()
    y_host = torch.empty_like(x_host).pin_memory()
    losses_host = torch.empty(2, dtype=torch.float32).pin_memory()
    x_dev, y_dev = torch.empty_like(inp["x"]), torch.empty_like(inp["x"])
    ws = moe.alloc_workspace(layer.shape(w.T), device=DEV)
    moe.moe_forward_host(layer.shape(w.T), ws, x_host, inp["w_router"], inp["w1"], inp["w3"],
                         inp["w2"], y_host, x_dev, y_dev, router_bias=inp["router_bias"],
                         w1s=inp["w1s"], w3s=inp["w3s"], w2s=inp["w2s"],
                         losses_host=losses_host)
    torch.cuda.synchronize()
    assert moe.moe_get_error(ws) == 0
    assert torch.equal(y_host, ref.cpu())
    assert torch.equal(losses_host, layer.losses.cpu())
    # the same through MoELayer.forward_host
    y_host2 = torch.empty_like(x_host).pin_memory()
    losses_host2 = torch.empty(2, dtype=torch.float32).pin_memory()
    layer.forward_host(x_host, x_dev, y_dev, y_host2, losses_host2)
    torch.cuda.synchronize()
    assert layer.device_error() == 0
    assert torch.equal(y_host2, ref.cpu())
    assert torch.equal(losses_host2, losses_host)


@pytest.mark.parametrize("w", [
    WORKLOADS["mixtral_prefill"].scaled(T=1000, d=256, E=8, k=2, d_ff=256),
    WORKLOADS["switch_top1"].scaled(T=5000, d=256, E=128, k=1, d_ff=256),
    WORKLOADS["deepseek_fine"].scaled(T=600, d=256, E=256, k=8, d_ff=128, d_ff_shared=128),
    WORKLOADS["tiny_fp32"],
], ids=["mixtral_shaped", "switch_shaped", "deepseek_shaped", "tiny_fp32"])
def test_forward_losses_equal_step_by_step_losses(w):
    """The forward's balance losses (its statistics-and-losses kernel) and the step-by-step
    path (moe_route_topk's statistics fed to moe_aux_loss with the forward's counts) give the
    same two numbers bit for bit: the same reduction order over the same partial sums. The
    shapes reduce 9, 129 and 257 rows of partial sums, in bf16 and fp32."""
    import mixture_experts_layer_92_b300 as moe
    inp = dev_inputs(w)
    g = gpu_forward(w, inp)
    assert g["error"] == 0
    losses2 = torch.full((2,), float("nan"), device=DEV)
    moe.moe_aux_loss(g["shape"], g["stats"], g["counts"], losses2)
    torch.cuda.synchronize()
    assert torch.equal(g["losses"], losses2), (g["losses"], losses2)
