"""The failure path on a real GPU, without a fault: a device wait that nothing completes runs
out its bound, the workspace error word reports MOE_ERR_TIMEOUT with the wait's site, and the
same context and workspace then run a layer normally."""
import time

import numpy as np
import pytest
import torch

import oracle as O
from moe_inputs import WORKLOADS, make_inputs
from moe_testlib import capacity_of, host64
from mixture_experts_layer_92_b300 import _lib as L

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
MOE_ERR_TIMEOUT = -5


def test_bounded_wait_times_out_and_the_context_stays_usable():
    w = WORKLOADS["tiny_fp32"]
    C = capacity_of(w)
    s = L.make_shape(w.T, w.d, w.E, w.k, w.d_ff, gate=w.gate, dtype=torch.float32, capacity=C,
                     alpha=w.alpha, beta=w.beta)
    ws = L.alloc_workspace(s, DEV)
    t0 = time.perf_counter()
    L.moe_selftest_wait_timeout(ws)
    status = L.moe_get_error(ws)          # synchronises
    waited = time.perf_counter() - t0
    assert status == MOE_ERR_TIMEOUT
    assert "site 40" in L.LIB.moe_last_error_detail().decode()
    assert 1.0 < waited < 60.0            # the 2 s bound, not a hang
    # sticky until cleared
    assert L.moe_get_error(ws) == MOE_ERR_TIMEOUT
    L.moe_clear_error(ws)
    assert L.moe_get_error(ws) == 0
    # the same context and workspace run the layer
    inp = make_inputs(w, device=DEV)
    y = torch.empty_like(inp["x"])
    L.moe_forward(s, ws, inp["x"], inp["w_router"], inp["w1"], inp["w3"], inp["w2"], y)
    torch.cuda.synchronize()
    assert L.moe_get_error(ws) == 0
    ref = O.forward(host64(inp["x"]), host64(inp["w_router"]), host64(inp["w1"]),
                    host64(inp["w3"]), host64(inp["w2"]), k=w.k, mode=w.gate, C=C,
                    alpha=w.alpha, beta=w.beta)
    yref = ref["y"]
    err = np.abs(y.double().cpu().numpy() - yref).max()
    assert err <= 1e-4 * np.sqrt(np.mean(yref ** 2))
