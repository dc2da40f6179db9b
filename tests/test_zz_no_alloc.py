"""moe_route_topk_noalloc: routing from precomputed logits for callers that cannot
allocate device memory (e.g. inside a framework that owns all device memory and forbids
cudaMalloc). Its scratch lives in a fixed array inside the library, so it takes no
workspace. It must return what moe_route_topk returns for the same logits, call after call,
and refuse sizes whose scratch would not fit.

This file is collected last on purpose; it passes on its own in a fresh process too."""
import numpy as np
import pytest
import torch

from moe_inputs import random_logits
from mixture_experts_layer_92_b300 import _lib as L

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def both(logits: torch.Tensor, k: int, mode: str):
    T, E = logits.shape
    s = L.make_shape(T, 16, E, k, 16, gate=mode, dtype=torch.float32)
    ws = L.alloc_workspace(s, DEV)
    l = logits.to(DEV)
    out = {}
    for name in ("workspace", "noalloc"):
        idx = torch.full((T, k), -7, dtype=torch.int32, device=DEV)
        gate = torch.full((T, k), -7.0, dtype=torch.float32, device=DEV)
        stats = torch.full((E + 1,), -7.0, dtype=torch.float32, device=DEV)
        if name == "workspace":
            L.moe_route_topk(s, ws, idx, gate, logits_in=l, stats=stats)
        else:
            L.moe_route_topk_noalloc(s, l, idx, gate, stats=stats)
        out[name] = (idx, gate, stats)
    torch.cuda.synchronize()
    assert L.moe_get_error(ws) == 0
    (i0, g0, s0), (i1, g1, s1) = out["workspace"], out["noalloc"]
    np.testing.assert_array_equal(i1.cpu().numpy(), i0.cpu().numpy())
    np.testing.assert_allclose(g1.cpu().numpy(), g0.cpu().numpy(), rtol=3e-6, atol=1e-7)
    np.testing.assert_allclose(s1.cpu().numpy(), s0.cpu().numpy(), rtol=2e-5, atol=1e-6)


def test_noalloc_matches_workspace_entry_on_consecutive_calls():
    # two calls in a row with different sizes share the library's scratch; a third call
    # repeats the first to show nothing stale is left behind
    both(random_logits(333, 64, seed=1), 6, "softmax_topk")
    both(random_logits(5000, 256, seed=2, ties=True), 8, "sigmoid_topk")
    both(random_logits(333, 64, seed=1), 6, "softmax_topk")
    both(random_logits(16384, 128, seed=3), 1, "softmax_all")


def test_noalloc_at_the_edge_of_its_scratch():
    # route_blocks(T) = min(ceil(T / 8), 592) blocks of (E + 1) partial sums, 4 bytes each:
    # E = 884 at 592 blocks fills the 2 MiB to within 1.2 KB, and E = 1024 fits while T
    # keeps the block count at 511 or below
    both(random_logits(4736, 884, seed=4), 4, "softmax_topk")
    both(random_logits(4000, 1024, seed=5), 2, "sigmoid_topk")


def test_noalloc_rejects_one_expert_past_the_edge():
    T, E, k = 4736, 885, 2                        # 592 * 886 * 4 bytes > 2 MiB
    s = L.make_shape(T, 16, E, k, 16, dtype=torch.float32)
    l = torch.zeros(T, E, device=DEV)
    idx = torch.empty(T, k, dtype=torch.int32, device=DEV)
    gate = torch.empty(T, k, device=DEV)
    with pytest.raises(L.MoeError) as ei:
        L.moe_route_topk_noalloc(s, l, idx, gate)
    assert ei.value.status == -2 and "scratch" in str(ei.value)


def test_noalloc_refuses_expert_choice_layers():
    # expert-choice layers have no top-k step; the workspace entry point refuses them too
    T, E = 64, 8
    s = L.make_shape(T, 16, E, 1, 16, gate="expert_choice", capacity=16, dtype=torch.float32)
    l = torch.zeros(T, E, device=DEV)
    idx = torch.empty(T, 1, dtype=torch.int32, device=DEV)
    gate = torch.empty(T, 1, device=DEV)
    with pytest.raises(L.MoeError) as ei:
        L.moe_route_topk_noalloc(s, l, idx, gate)
    assert ei.value.status == -2


def test_noalloc_rejects_sizes_beyond_its_scratch():
    T, E, k = 8192, 1024, 2                       # needs 1024 * 1025 * 4 bytes > 2 MiB
    s = L.make_shape(T, 16, E, k, 16, dtype=torch.float32)
    l = torch.zeros(T, E, device=DEV)
    idx = torch.empty(T, k, dtype=torch.int32, device=DEV)
    gate = torch.empty(T, k, device=DEV)
    with pytest.raises(L.MoeError) as ei:
        L.moe_route_topk_noalloc(s, l, idx, gate)
    assert ei.value.status == -2
    assert "scratch" in str(ei.value)
