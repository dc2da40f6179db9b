"""Pins of the backward oracle (oracle/moe_backward.py) to things other than itself:
central finite differences of the forward oracle (itself pinned by test_oracle_pins.py)
along seeded random directions, with the routing decisions held fixed; closed forms; and
invariants that any correct gradient has (softmax shift invariance, a uniform load giving
no balance-loss gradient, a fully dropped batch giving no expert gradient)."""
import math

import numpy as np
import pytest

import oracle as O

GATES = ("softmax_all", "softmax_topk", "sigmoid_topk")


def make_case(seed, T=12, d=8, E=5, k=2, F=6, Fs=0, bias=False):
    rng = np.random.default_rng(seed)
    p = dict(x=rng.normal(size=(T, d)), w_router=rng.normal(size=(E, d)) / math.sqrt(d),
             w1=rng.normal(size=(E, F, d)) / math.sqrt(d), w3=rng.normal(size=(E, F, d)) / math.sqrt(d),
             w2=rng.normal(size=(E, d, F)) / math.sqrt(F),
             router_bias=rng.normal(size=E) * 0.5 if bias else None,
             w1s=None, w3s=None, w2s=None)
    if Fs:
        p.update(w1s=rng.normal(size=(Fs, d)) / math.sqrt(d), w3s=rng.normal(size=(Fs, d)) / math.sqrt(d),
                 w2s=rng.normal(size=(d, Fs)) / math.sqrt(Fs))
    dy = rng.normal(size=(T, d))
    return p, dy


def objective(p, dy, idx, *, k, mode, C, alpha, beta, d_aux, d_z):
    f = O.forward(p["x"], p["w_router"], p["w1"], p["w3"], p["w2"], k=k, mode=mode, C=C,
                  router_bias=p["router_bias"], w1s=p["w1s"], w3s=p["w3s"], w2s=p["w2s"],
                  alpha=alpha, beta=beta, idx_override=idx)
    return float((dy * f["y"]).sum() + d_aux * f["l_aux"] + d_z * f["l_z"])


GRAD_NAME = dict(x="dx", w_router="dw_router", router_bias="d_router_bias", w1="dw1", w3="dw3",
                 w2="dw2", w1s="dw1s", w3s="dw3s", w2s="dw2s")


@pytest.mark.parametrize("mode", GATES)
@pytest.mark.parametrize("C,Fs,bias", [(12, 0, False), (3, 0, True), (5, 4, True)])
def test_backward_matches_finite_differences(mode, C, Fs, bias):
    """Directional derivative of J along a random direction, for every input, equals the
    oracle's gradient contracted with that direction (central differences, h = 1e-5)."""
    k, alpha, beta, d_aux, d_z = 2, 0.3, 0.2, 0.7, 1.3
    p, dy = make_case(11 + C, Fs=Fs, bias=bias)
    g = O.backward(p["x"], p["w_router"], p["w1"], p["w3"], p["w2"], dy, k=k, mode=mode, C=C,
                   router_bias=p["router_bias"], w1s=p["w1s"], w3s=p["w3s"], w2s=p["w2s"],
                   alpha=alpha, beta=beta, d_aux=d_aux, d_z=d_z)
    idx = g["idx"]
    if C < 12:
        assert g["dispatch"]["dropped"] > 0            # the case really drops assignments
    rng = np.random.default_rng(5)
    h = 1e-5
    for name, gname in GRAD_NAME.items():
        if p[name] is None:
            assert g[gname] is None or name == "router_bias"
            continue
        v = rng.normal(size=p[name].shape)
        plus = dict(p, **{name: p[name] + h * v})
        minus = dict(p, **{name: p[name] - h * v})
        kw = dict(k=k, mode=mode, C=C, alpha=alpha, beta=beta, d_aux=d_aux, d_z=d_z)
        fd = (objective(plus, dy, idx, **kw) - objective(minus, dy, idx, **kw)) / (2 * h)
        an = float((g[gname] * v).sum())
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


def test_balance_terms_alone_match_finite_differences():
    """dy = 0 isolates the balance losses: the router gradient then comes only from
    P_i (aux) and lse (z-loss), and the experts get none."""
    p, _ = make_case(3)
    dy = np.zeros_like(p["x"])
    kw = dict(k=2, mode="softmax_topk", C=12, alpha=0.5, beta=0.25)
    g = O.backward(p["x"], p["w_router"], p["w1"], p["w3"], p["w2"], dy, **kw)
    assert np.all(g["dw1"] == 0) and np.all(g["dw2"] == 0) and np.all(g["dgate"] == 0)
    v = np.random.default_rng(1).normal(size=p["w_router"].shape)
    h = 1e-5
    J = lambda wr: objective(dict(p, w_router=wr), dy, g["idx"], d_aux=1.0, d_z=1.0, **kw)
    fd = (J(p["w_router"] + h * v) - J(p["w_router"] - h * v)) / (2 * h)
    assert fd == pytest.approx(float((g["dw_router"] * v).sum()), rel=1e-6, abs=1e-9)


def test_z_loss_gradient_closed_form_at_zero_logits():
    """l = 0: lse = ln E, p = 1/E, so dL_z/dl = 2 beta ln(E) / (T E) everywhere."""
    T, E, beta = 7, 5, 0.3
    np.testing.assert_allclose(O.z_loss_backward(np.zeros((T, E)), beta),
                               np.full((T, E), 2 * beta * math.log(E) / (T * E)), rtol=1e-14)


def test_aux_loss_gradient_vanishes_under_uniform_load():
    """With f_i = 1/E for every expert, a_i is constant and dL_aux/dl = p (a - a) = 0 for any
    logits: a perfectly balanced router feels no push from the aux loss."""
    E, k = 4, 2
    idx = np.array([[0, 1], [2, 3], [1, 0], [3, 2]])
    l = np.random.default_rng(0).normal(size=(4, E)) * 3
    np.testing.assert_allclose(O.aux_loss_backward(l, idx, 0.7), 0.0, atol=1e-16)


@pytest.mark.parametrize("mode", GATES)
def test_gate_gradient_invariants(mode):
    """Renormalised gates (softmax_topk, sigmoid_topk) sum to 1 over the selected experts,
    so a dgate that is the same for every slot moves nothing; softmax gates are unchanged by
    adding a constant to a token's logits, so their dl sums to 0 over the experts."""
    rng = np.random.default_rng(2)
    l = rng.normal(size=(9, 6))
    idx = O.select_topk(l, 3)
    const = np.full((9, 3), 0.37)
    if mode != "softmax_all":
        np.testing.assert_allclose(O.gate_backward(l, idx, mode, const), 0.0, atol=1e-15)
    dl = O.gate_backward(l, idx, mode, rng.normal(size=(9, 3)))
    if mode != "sigmoid_topk":
        np.testing.assert_allclose(dl.sum(axis=1), 0.0, atol=1e-15)
    else:
        # sigmoid gates: only the selected experts' logits move
        mask = np.zeros_like(dl, dtype=bool)
        np.put_along_axis(mask, idx, True, axis=1)
        assert np.all(dl[~mask] == 0.0)


def test_softmax_topk_with_k_equal_E_is_softmax_all():
    """k = E: the two softmax conventions are the same function, so are their gradients."""
    rng = np.random.default_rng(4)
    l = rng.normal(size=(6, 4))
    idx = O.select_topk(l, 4)
    dg = rng.normal(size=(6, 4))
    np.testing.assert_allclose(O.gate_backward(l, idx, "softmax_topk", dg),
                               O.gate_backward(l, idx, "softmax_all", dg), atol=1e-15)


def test_silu_gradient_values():
    """silu'(0) = 1/2; silu' -> 1 for large z and -> 0 for very negative z."""
    assert O.silu_grad(np.array([0.0]))[0] == 0.5
    assert O.silu_grad(np.array([40.0]))[0] == pytest.approx(1.0, abs=1e-12)
    assert abs(O.silu_grad(np.array([-40.0]))[0]) < 1e-12


def test_swiglu_backward_identity_weights_closed_form():
    """w1 = w3 = w2 = I (d = F): O = silu(x) * x elementwise, so
    dx = dout * (silu(x) + x silu'(x)) and dw2 = dout^T (silu(x) x)."""
    rng = np.random.default_rng(6)
    x = rng.normal(size=(5, 4))
    dout = rng.normal(size=(5, 4))
    I = np.eye(4)
    r = O.swiglu_ffn_backward(x, I, I, I, dout)
    sx = x / (1 + np.exp(-x))
    sig = 1 / (1 + np.exp(-x))
    np.testing.assert_allclose(r["dx"], dout * (sx + x * sig * (1 + x * (1 - sig))), rtol=1e-13)
    np.testing.assert_allclose(r["dw2"], dout.T @ (sx * x), rtol=1e-13)


def test_fully_dropped_batch_has_no_expert_gradient():
    """C = 0 drops every assignment: y = shared only, so the routed experts and the gates get
    no gradient; the router still gets the balance-loss gradient."""
    p, dy = make_case(8, Fs=3)
    g = O.backward(p["x"], p["w_router"], p["w1"], p["w3"], p["w2"], dy, k=2, mode="sigmoid_topk",
                   C=0, w1s=p["w1s"], w3s=p["w3s"], w2s=p["w2s"], alpha=0.1, beta=0.1)
    assert np.all(g["dw1"] == 0) and np.all(g["dw3"] == 0) and np.all(g["dw2"] == 0)
    assert np.all(g["dgate"] == 0)
    np.testing.assert_allclose(g["dlogits"], O.aux_loss_backward(O.router_logits(p["x"], p["w_router"]),
                                                                g["idx"], 0.1)
                               + O.z_loss_backward(O.router_logits(p["x"], p["w_router"]), 0.1),
                               rtol=1e-13, atol=1e-16)


def ec_objective(p, dy, choice, *, C, alpha, beta, d_aux, d_z):
    f = O.expert_choice_forward(p["x"], p["w_router"], p["w1"], p["w3"], p["w2"], C=C,
                                router_bias=p["router_bias"], w1s=p["w1s"], w3s=p["w3s"],
                                w2s=p["w2s"], alpha=alpha, beta=beta, k=2, choice=choice)
    return float((dy * f["y"]).sum() + d_aux * f["l_aux"] + d_z * f["l_z"])


@pytest.mark.parametrize("C,Fs,bias", [(5, 0, False), (2, 4, True), (12, 0, True)])
def test_expert_choice_backward_matches_finite_differences(C, Fs, bias):
    """Expert-choice layer: directional derivatives of J (choices held fixed) equal the
    oracle's gradients for every input; C = 2 (10 choices for 12 tokens) leaves tokens no
    expert chose, C = 12 (= T) lets every expert take every token."""
    alpha, beta, d_aux, d_z = 0.3, 0.2, 0.7, 1.3
    p, dy = make_case(31 + C, Fs=Fs, bias=bias)
    g = O.expert_choice_backward(p["x"], p["w_router"], p["w1"], p["w3"], p["w2"], dy, C=C,
                                 router_bias=p["router_bias"], w1s=p["w1s"], w3s=p["w3s"],
                                 w2s=p["w2s"], alpha=alpha, beta=beta, k=2, d_aux=d_aux, d_z=d_z)
    choice = dict(perm=g["ec"]["perm"], offsets=g["ec"]["offsets"], inv=g["ec"]["inv"])
    if C == 2:
        assert g["ec"]["unrouted"] > 0
    rng = np.random.default_rng(8)
    h = 1e-5
    kw = dict(C=C, alpha=alpha, beta=beta, d_aux=d_aux, d_z=d_z)
    for name, gname in GRAD_NAME.items():
        if p[name] is None:
            continue
        v = rng.normal(size=p[name].shape)
        fd = (ec_objective(dict(p, **{name: p[name] + h * v}), dy, choice, **kw)
              - ec_objective(dict(p, **{name: p[name] - h * v}), dy, choice, **kw)) / (2 * h)
        an = float((g[gname] * v).sum())
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


def test_expert_choice_aux_loss_has_no_gradient():
    """f_i = C'/(T k) for every expert and sum_i P_i = 1: L_aux is constant in the logits, so
    with dy = 0 and d_z = 0 the router gets no gradient at all."""
    p, _ = make_case(5)
    dy = np.zeros_like(p["x"])
    g = O.expert_choice_backward(p["x"], p["w_router"], p["w1"], p["w3"], p["w2"], dy, C=4,
                                 alpha=0.9, beta=0.3, d_aux=1.0, d_z=0.0)
    np.testing.assert_allclose(g["dlogits"], 0.0, atol=1e-16)
    np.testing.assert_allclose(g["dw_router"], 0.0, atol=1e-15)
