"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks one oracle function against something other than itself: the pages'
worked example, the demo's stated invariants, closed forms, or brute force on tiny
inputs. The cases are chosen so that a dropped term, a wrong sign, a wrong index or a
transposed operand in the oracle fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O


# ---------------------------------------------------------------- gating / selection
def test_worked_example_top2(golden_dir):
    """'DL S077' section 2: logits -> experts {2, 4}, gates 0.668 / 0.332."""
    g = json.load(open(os.path.join(golden_dir, "worked_example_top2.json")))
    l = np.array([g["logits"]])
    idx = O.select_topk(l, g["k"])
    assert idx[0].tolist() == g["experts"]
    gate = O.gates(l, idx, "softmax_topk")
    assert np.round(gate[0], 3).tolist() == g["gates_3dp"]


def test_softmax_all_closed_form():
    """Logits ln(1..4): probabilities 0.1..0.4; top-2 = experts 3, 2 with gates 0.4, 0.3."""
    l = np.log(np.array([[1.0, 2.0, 3.0, 4.0]]))
    p = O.softmax_all(l)
    np.testing.assert_allclose(p[0], [0.1, 0.2, 0.3, 0.4], rtol=0, atol=1e-15)
    idx = O.select_topk(l, 2)
    assert idx[0].tolist() == [3, 2]
    np.testing.assert_allclose(O.gates(l, idx, "softmax_all")[0], [0.4, 0.3], atol=1e-15)
    np.testing.assert_allclose(O.gates(l, idx, "softmax_topk")[0], [4 / 7, 3 / 7], atol=1e-15)


def test_sigmoid_topk_closed_form():
    """sigma(ln 3) = 0.75 and sigma(0) = 0.5 -> renormalised gates 0.6 / 0.4; k=1 -> 1."""
    l = np.array([[-30.0, 0.0, math.log(3.0), -20.0]])
    idx = O.select_topk(l, 2)
    assert idx[0].tolist() == [2, 1]
    np.testing.assert_allclose(O.gates(l, idx, "sigmoid_topk")[0], [0.6, 0.4], atol=1e-15)
    idx1 = O.select_topk(l, 1)
    np.testing.assert_allclose(O.gates(l, idx1, "sigmoid_topk")[0], [1.0], atol=0)


@pytest.mark.parametrize("E", [3, 8, 16])
def test_topk_softmax_equals_softmax_all_when_k_is_E(E):
    """With k = E the softmax over the selected logits is the softmax over all experts."""
    l = np.random.default_rng(E).normal(size=(40, E)) * 3
    idx = O.select_topk(l, E)
    np.testing.assert_allclose(O.gates(l, idx, "softmax_topk"), O.gates(l, idx, "softmax_all"),
                               rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("k", [1, 2, 5])
def test_topk_softmax_is_renormalised_softmax_all(k):
    l = np.random.default_rng(k).normal(size=(50, 8)) * 2
    idx = O.select_topk(l, k)
    p = O.gates(l, idx, "softmax_all")
    np.testing.assert_allclose(O.gates(l, idx, "softmax_topk"), p / p.sum(axis=1, keepdims=True),
                               rtol=1e-13)


def _brute_topk(row, k):
    """The unique k-subset S with every member beating every non-member (a larger logit,
    or an equal logit and a lower index); ordered by descending logit, then index."""
    E = len(row)
    found = []
    for S in itertools.combinations(range(E), k):
        rest = [i for i in range(E) if i not in S]
        if all(row[j] > row[i] or (row[j] == row[i] and j < i) for j in S for i in rest):
            found.append(S)
    assert len(found) == 1
    return sorted(found[0], key=lambda j: (-row[j], j))


@pytest.mark.parametrize("E", [4, 6, 8])
@pytest.mark.parametrize("kind", ["random", "tied", "equal"])
def test_topk_brute_force(E, kind):
    rng = np.random.default_rng(E * 7 + len(kind))
    if kind == "random":
        l = rng.normal(size=(12, E))
    elif kind == "tied":
        l = np.round(rng.normal(size=(12, E)) * 2) / 2
        l[0, :] = 0.0
        l[0, 1] = -0.0          # -0.0 and +0.0 compare equal: a tie
    else:
        l = np.full((3, E), 0.7)
    for k in range(1, E + 1):
        idx = O.select_topk(l, k)
        for t in range(l.shape[0]):
            assert idx[t].tolist() == _brute_topk(l[t].tolist(), k)
    if kind == "equal":
        assert O.select_topk(l, 3)[0].tolist() == [0, 1, 2]


def test_gates_sum_to_one_on_demo_logits(golden_dir):
    """'Mixture of experts (MoE)' (tirogla.com) demo: hashed logits, renormalised top-2
    gates sum to 1 within 1e-5; capacity at cf 1.25 is 20."""
    g = json.load(open(os.path.join(golden_dir, "demo_capacity.json")))
    T, E, k = g["T"], g["E"], g["k"]
    l = np.array([((i * 2654435761) >> 7) % 1000 / 250.0 for i in range(T * E)]).reshape(T, E)
    idx = O.select_topk(l, k)
    for mode in ("softmax_topk", "sigmoid_topk"):
        s = O.gates(l, idx, mode).sum(axis=1)
        assert np.all(np.abs(s - 1.0) < g["gate_sum_tol"])
    C = O.capacity(g["cf"], T, k, E)
    assert C == g["capacity"]
    d = O.dispatch(idx, E, C)
    kept = np.diff(d["offsets"])
    assert np.all(kept <= C)
    assert d["dropped"] == int(np.maximum(d["counts"] - C, 0).sum())


# ---------------------------------------------------------------- dispatch
def _brute_dispatch(flat, E, C):
    """Rank formulation: rank(a) = #earlier assignments to the same expert; a is kept
    iff rank < C, at row sum_{e' < e} min(n_e', C) + rank."""
    n = [sum(1 for v in flat if v == e) for e in range(E)]
    base = [sum(min(n[j], C) for j in range(e)) for e in range(E)]
    inv = []
    for a, e in enumerate(flat):
        rank = sum(1 for b in range(a) if flat[b] == e)
        inv.append(base[e] + rank if rank < C else -1)
    return n, inv


@pytest.mark.parametrize("seed", range(6))
def test_dispatch_brute_force(seed):
    rng = np.random.default_rng(seed)
    E = int(rng.integers(1, 9))
    k = int(rng.integers(1, E + 1))
    T = int(rng.integers(0, 40))
    l = rng.normal(size=(T, E))
    idx = O.select_topk(l, k) if T > 0 else np.zeros((0, k), dtype=np.int64)
    for C in (0, 1, 3, max(1, T * k // E), T):
        d = O.dispatch(idx, E, C)
        flat = idx.reshape(-1).tolist()
        n, inv = _brute_dispatch(flat, E, C)
        assert d["counts"].tolist() == n
        assert d["inv"].tolist() == inv
        assert d["dropped"] == sum(max(0, v - C) for v in n)
        # perm is the inverse of inv on the kept assignments and increasing per segment
        R = int(d["offsets"][-1])
        assert d["perm"].shape[0] == R == sum(1 for v in inv if v >= 0)
        for r in range(R):
            assert inv[d["perm"][r]] == r
        for e in range(E):
            seg = d["perm"][d["offsets"][e]:d["offsets"][e + 1]]
            assert np.all(np.diff(seg) > 0)
            assert all(flat[a] == e for a in seg)


def test_dispatch_collapse_closed_form():
    """All-equal logits send every token to experts 0..k-1: k*max(0, T-C) drops."""
    T, E, k = 50, 8, 2
    idx = O.select_topk(np.zeros((T, E)), k)
    assert np.all(idx == np.arange(k))
    for C in (0, 7, 50, 80):
        d = O.dispatch(idx, E, C)
        assert d["dropped"] == k * max(0, T - C)
        assert d["counts"].tolist() == [T] * k + [0] * (E - k)


def test_capacity_formula():
    assert O.capacity(1.25, 256, 2, 8) == 80
    assert O.capacity(1.0, 16384, 1, 128) == 128
    assert O.capacity(1.0, 10, 1, 3) == 4          # ceil(10/3)
    assert O.capacity(1.0, 12, 1, 3) == 4          # exact, no rounding up


# ---------------------------------------------------------------- losses
@pytest.mark.parametrize("E,k,m", [(8, 2, 3), (16, 1, 2), (4, 3, 5)])
def test_aux_loss_uniform_split_equals_alpha(E, k, m):
    """'Mixture of experts (MoE)' (tirogla.com): the balance loss equals alpha for a
    perfectly uniform split. Rows are the E cyclic rotations of one vector (m times),
    so every expert receives the same load and the same mean probability."""
    v = np.linspace(-1.0, 2.0, E)[np.random.default_rng(E).permutation(E)]
    l = np.stack([np.roll(v, s) for _ in range(m) for s in range(E)])
    idx = O.select_topk(l, k)
    np.testing.assert_allclose(O.load_fractions(idx, E), 1.0 / E, atol=1e-15)
    assert O.aux_loss(l, idx, 0.01) == pytest.approx(0.01, rel=1e-12)


def test_aux_loss_constant_logits():
    """Constant logits: P_i = 1/E, top-k = experts 0..k-1, f_i = 1/k there -> alpha."""
    for E, k in ((8, 2), (5, 1), (6, 6)):
        l = np.full((9, E), 0.3)
        idx = O.select_topk(l, k)
        assert O.aux_loss(l, idx, 0.02) == pytest.approx(0.02, rel=1e-12)


def test_aux_loss_collapse_closed_form():
    """k=1, expert 0 gets +L: f_0 = 1 and P_0 = e^L / (e^L + E - 1) -> alpha*E*P_0."""
    E, L = 8, 2.0
    l = np.zeros((11, E))
    l[:, 0] = L
    idx = O.select_topk(l, 1)
    P0 = math.exp(L) / (math.exp(L) + E - 1)
    assert O.aux_loss(l, idx, 0.01) == pytest.approx(0.01 * E * P0, rel=1e-12)


def test_losses_of_an_empty_batch_are_zero():
    l = np.zeros((0, 8))
    idx = np.zeros((0, 2), dtype=np.int64)
    assert O.aux_loss(l, idx, 0.01) == 0.0 and O.z_loss(l, 1e-3) == 0.0


def test_z_loss_closed_forms():
    """Zero logits: beta*(ln E)^2. Mixed rows: the mean of squares, not the square of
    the mean. Large constant logits do not overflow."""
    E, beta = 8, 1e-3
    assert O.z_loss(np.zeros((5, E)), beta) == pytest.approx(beta * math.log(E) ** 2, rel=1e-13)
    l = np.stack([np.zeros(E), np.full(E, 2.0)])
    a, b = math.log(E), 2.0 + math.log(E)
    assert O.z_loss(l, beta) == pytest.approx(beta * (a * a + b * b) / 2, rel=1e-13)
    assert O.z_loss(np.full((2, E), 1000.0), 1.0) == pytest.approx((1000 + math.log(E)) ** 2, rel=1e-13)


# ---------------------------------------------------------------- score and FFN
def test_router_logits_selects_components():
    """W_r rows are unit vectors e_{pi(e)}: logits[t, e] = x[t, pi(e)] + b[e] (E != d)."""
    d, E = 6, 4
    pi = [4, 0, 5, 2]
    W = np.zeros((E, d))
    W[np.arange(E), pi] = 1.0
    x = np.random.default_rng(0).normal(size=(7, d))
    b = np.array([0.5, -1.0, 0.0, 2.0])
    np.testing.assert_array_equal(O.router_logits(x, W, b), x[:, pi] + b)


def test_silu_closed_forms():
    np.testing.assert_allclose(O.silu([0.0, 1.0, -1.0]),
                               [0.0, 1 / (1 + math.exp(-1)), -1 / (1 + math.e)], atol=1e-16)
    assert O.silu([800.0])[0] == 800.0
    assert O.silu([-800.0])[0] == 0.0


def test_swiglu_structured_closed_form():
    """W1 = diag(a), W3 = diag(b), W2 = cyclic shift P (not symmetric):
    y = P (silu(a*x) * (b*x)). Swapping gate/up or transposing W2 fails."""
    n = 5
    a = np.array([1.0, -2.0, 0.5, 3.0, -1.0])
    b = np.array([2.0, 1.0, -1.0, 0.5, 4.0])
    P = np.roll(np.eye(n), 1, axis=0)          # (P v)[i] = v[i-1]
    x = np.array([[0.3, -1.2, 2.0, 0.7, -0.4]])
    h = (a * x) / (1 + np.exp(-(a * x))) * (b * x)
    expect = np.roll(h, 1, axis=1)
    np.testing.assert_allclose(O.swiglu_ffn(x, np.diag(a), np.diag(b), P), expect, atol=1e-15)


def test_swiglu_matches_torch_library():
    """Rectangular shapes against torch's own fp64 silu and matmul."""
    rng = np.random.default_rng(3)
    x, w1, w3, w2 = rng.normal(size=(9, 12)), rng.normal(size=(20, 12)), rng.normal(size=(20, 12)), rng.normal(size=(12, 20))
    tx, t1, t3, t2 = (torch.from_numpy(a) for a in (x, w1, w3, w2))
    ref = torch.nn.functional.linear(torch.nn.functional.silu(torch.nn.functional.linear(tx, t1))
                                     * torch.nn.functional.linear(tx, t3), t2)
    np.testing.assert_allclose(O.swiglu_ffn(x, w1, w3, w2), ref.numpy(), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- combine / forward
def test_combine_scale_experts_closed_form():
    """Experts that return (e+1)*x_t (the demo's stand-in experts): y_t is the sum over
    kept slots of g * (e+1) * x_t; dropped slots add nothing."""
    rng = np.random.default_rng(5)
    T, E, k, d = 20, 4, 2, 3
    x = rng.normal(size=(T, d))
    l = rng.normal(size=(T, E))
    idx = O.select_topk(l, k)
    g = O.gates(l, idx, "softmax_topk")
    disp = O.dispatch(idx, E, 6)
    rows = np.zeros((disp["perm"].shape[0], d))
    for r, a in enumerate(disp["perm"]):
        rows[r] = x[a // k] * (idx.reshape(-1)[a] + 1)
    y = O.combine(g, disp["inv"], rows, T, k)
    inv = disp["inv"].reshape(T, k)
    for t in range(T):
        s = sum(g[t, j] * (idx[t, j] + 1) for j in range(k) if inv[t, j] >= 0)
        np.testing.assert_allclose(y[t], s * x[t], atol=1e-14)
    assert disp["dropped"] > 0 and np.any(np.all(inv < 0, axis=1)) is not None


def _rand_weights(rng, E, F, d):
    return (rng.normal(size=(E, F, d)) / math.sqrt(d), rng.normal(size=(E, F, d)) / math.sqrt(d),
            rng.normal(size=(E, d, F)) / math.sqrt(F))


def test_identical_experts_reproduce_dense_ffn():
    """Identical experts, gates that sum to 1 and no drop give one dense SwiGLU FFN."""
    rng = np.random.default_rng(11)
    T, d, E, F, k = 32, 8, 6, 12, 3
    w1, w3, w2 = _rand_weights(rng, 1, F, d)
    W1, W3, W2 = (np.repeat(w, E, axis=0) for w in (w1, w3, w2))
    x = rng.normal(size=(T, d))
    wr = rng.normal(size=(E, d))
    for mode in ("softmax_topk", "sigmoid_topk"):
        out = O.forward(x, wr, W1, W3, W2, k=k, mode=mode, C=T)
        np.testing.assert_allclose(out["y"], O.swiglu_ffn(x, w1[0], w3[0], w2[0]), rtol=1e-12, atol=1e-12)


def test_shared_expert_only_when_everything_drops():
    """C = 0 drops every routed assignment: y is the shared expert's output alone."""
    rng = np.random.default_rng(12)
    T, d, E, F, k = 10, 8, 4, 6, 2
    w1, w3, w2 = _rand_weights(rng, E, F, d)
    s1, s3, s2 = (a[0] for a in _rand_weights(rng, 1, 5, d))
    x = rng.normal(size=(T, d))
    out = O.forward(x, rng.normal(size=(E, d)), w1, w3, w2, k=k, mode="sigmoid_topk", C=0,
                    w1s=s1, w3s=s3, w2s=s2)
    assert out["dispatch"]["dropped"] == T * k
    np.testing.assert_allclose(out["y"], O.swiglu_ffn(x, s1, s3, s2), atol=1e-14)


def test_forward_single_token_by_hand():
    """One token, E=3, k=2, d=F=1: y = sum_j g_j * w2_j silu(w1_j x) w3_j x."""
    x = np.array([[1.5]])
    wr = np.array([[1.0], [-1.0], [0.5]])        # logits 1.5, -1.5, 0.75 -> experts 0, 2
    w1 = np.array([[[2.0]], [[1.0]], [[-1.0]]])
    w3 = np.array([[[0.5]], [[1.0]], [[3.0]]])
    w2 = np.array([[[1.0]], [[1.0]], [[-2.0]]])
    out = O.forward(x, wr, w1, w3, w2, k=2, mode="softmax_topk", C=1)
    g0 = 1 / (1 + math.exp(0.75 - 1.5))
    f = lambda a, b, c: c * (a * 1.5) / (1 + math.exp(-a * 1.5)) * (b * 1.5)
    expect = g0 * f(2.0, 0.5, 1.0) + (1 - g0) * f(-1.0, 3.0, -2.0)
    assert out["idx"].tolist() == [[0, 2]]
    assert out["y"][0, 0] == pytest.approx(expect, rel=1e-14)


def test_near_tie_tokens():
    l = np.array([[3.0, 1.0, 0.9995, 0.0], [3.0, 1.0, 0.5, 0.0], [1.0, 1.0, 1.0, 1.0]])
    assert O.near_tie_tokens(l, 2).tolist() == [0, 2]
    assert O.near_tie_tokens(l, 4).tolist() == []


# ---------------------------------------------------------------- aux-loss-free balancing
@pytest.mark.parametrize("mode", ["softmax_all", "softmax_topk", "sigmoid_topk"])
def test_zero_selection_bias_is_plain_top_k(mode):
    """Affinity is monotone in the logit, so a zero bias selects exactly the top-k logits."""
    l = np.random.default_rng(21).normal(size=(60, 16)) * 2
    for k in (1, 3, 8):
        np.testing.assert_array_equal(O.select_topk_biased(l, k, mode, np.zeros(16)),
                                      O.select_topk(l, k))


def test_large_selection_bias_forces_expert_but_not_the_gate():
    """A bias of +10 on expert 5 puts it in every token's top-k (affinities are <= 1), while
    its gate is still sigma(l_5) / sum over the selected of sigma(l)."""
    l = np.random.default_rng(22).normal(size=(30, 8))
    b = np.zeros(8)
    b[5] = 10.0
    idx = O.select_topk_biased(l, 2, "sigmoid_topk", b)
    assert np.all(idx[:, 0] == 5)
    g = O.gates(l, idx, "sigmoid_topk")
    s = 1 / (1 + np.exp(-np.take_along_axis(l, idx, 1)))
    np.testing.assert_allclose(g, s / s.sum(1, keepdims=True), rtol=1e-14)
    # and the other slot is the best remaining expert by plain sigmoid (i.e. by logit)
    rest = np.where(np.arange(8)[None, :] == 5, -np.inf, l)
    np.testing.assert_array_equal(idx[:, 1], np.argmax(rest, axis=1))


def test_selection_bias_update_closed_form():
    """Mean load T*k/E = 6: loads 11, 6, 3, 4 -> -gamma, 0, +gamma, +gamma."""
    b = np.array([0.5, -0.25, 0.0, 1.0], dtype=np.float32)
    nb = O.update_select_bias(b, [11, 6, 3, 4], T=12, k=2, gamma=0.125)
    np.testing.assert_array_equal(nb, np.array([0.375, -0.25, 0.125, 1.125], dtype=np.float32))


def test_selection_bias_loop_balances_a_skewed_router():
    """Routing on a strongly skewed router (Zipf log-popularity added to the logits) with
    the bias nudged after every step drives the per-expert load towards uniform."""
    rng = np.random.default_rng(23)
    T, E, k = 512, 16, 2
    zipf = np.log(np.arange(1, E + 1) ** -1.2 / np.sum(np.arange(1, E + 1) ** -1.2))
    b = np.zeros(E, dtype=np.float32)
    spread = []
    for step in range(200):
        l = rng.normal(size=(T, E)) + zipf
        idx = O.select_topk_biased(l, k, "sigmoid_topk", b)
        n = np.bincount(idx.reshape(-1), minlength=E)
        spread.append(n.max() / (T * k / E))
        b = O.update_select_bias(b, n, T, k, 0.01)
    assert spread[0] > 3.0                      # starts badly unbalanced
    assert np.mean(spread[-20:]) < 1.5          # ends close to uniform


# ---------------------------------------------------------------- expert-choice routing
def test_expert_choice_brute_force():
    """Each expert's chosen set beats every unchosen token (higher probability, or equal
    and lower index); every expert takes exactly min(C, T) tokens."""
    rng = np.random.default_rng(31)
    for trial in range(6):
        T, E = int(rng.integers(1, 14)), int(rng.integers(1, 6))
        l = np.round(rng.normal(size=(T, E)) * 2) / 2         # frequent ties
        C = int(rng.integers(0, T + 3))
        ec = O.expert_choice(l, C)
        p = O.softmax_all(l)
        Cp = min(C, T)
        assert ec["counts"].tolist() == [Cp] * E
        for e in range(E):
            chosen = set(ec["perm"][e * Cp:(e + 1) * Cp].tolist())
            assert len(chosen) == Cp
            for t in chosen:
                for u in set(range(T)) - chosen:
                    assert p[t, e] > p[u, e] or (p[t, e] == p[u, e] and t < u)
            for j, t in enumerate(ec["perm"][e * Cp:(e + 1) * Cp]):
                assert ec["inv"][t, e] == e * Cp + j and ec["gate"][e * Cp + j] == p[t, e]
        assert ec["unrouted"] == sum(1 for t in range(T) if all(ec["inv"][t] < 0))


def test_expert_choice_single_expert_takes_the_first_tokens():
    """E = 1: every probability is 1 (a full tie), so the expert takes tokens 0..C-1."""
    ec = O.expert_choice(np.random.default_rng(32).normal(size=(10, 1)), 4)
    assert ec["perm"].tolist() == [0, 1, 2, 3] and ec["unrouted"] == 6


def test_expert_choice_everyone_chosen_with_identical_experts_is_the_dense_ffn():
    """C = T: every expert takes every token, the gates of a token sum to 1 (softmax), so
    identical experts give exactly one dense SwiGLU FFN."""
    rng = np.random.default_rng(33)
    T, d, E, F = 12, 6, 4, 10
    w1, w3, w2 = rng.normal(size=(F, d)), rng.normal(size=(F, d)), rng.normal(size=(d, F))
    W1, W3, W2 = (np.repeat(w[None], E, axis=0) for w in (w1, w3, w2))
    x = rng.normal(size=(T, d))
    out = O.expert_choice_forward(x, rng.normal(size=(E, d)), W1, W3, W2, C=T)
    np.testing.assert_allclose(out["y"], O.swiglu_ffn(x, w1, w3, w2), rtol=1e-12, atol=1e-12)
    assert out["ec"]["unrouted"] == 0


@pytest.mark.parametrize("T,E,C,k", [(12, 4, 5, 1), (12, 4, 12, 1), (7, 3, 20, 1), (9, 5, 0, 1),
                                     (16, 8, 3, 2), (10, 6, 4, 3), (1, 2, 1, 1)])
def test_expert_choice_balance_loss_closed_form(T, E, C, k):
    """Expert choice ([Starphix] "Router Variants") gives every expert exactly C' = min(C, T)
    rows, so f_i = C'/(T*k) for every i, and the all-E softmax makes sum_i P_i = 1: the
    balance loss alpha*E*sum_i f_i*P_i is alpha*E*C'/(T*k), whatever the logits. A
    normalisation by T instead of T*k, a dropped factor E, or f taken from the tokens
    instead of the rows each move it off this value."""
    rng = np.random.default_rng(T * 100 + E * 10 + C + k)
    d, F, alpha = 5, 6, 0.01
    x = rng.normal(size=(T, d))
    W1, W3 = rng.normal(size=(E, F, d)), rng.normal(size=(E, F, d))
    W2 = rng.normal(size=(E, d, F))
    out = O.expert_choice_forward(x, rng.normal(size=(E, d)) * 3, W1, W3, W2, C=C, k=k,
                                  alpha=alpha)
    assert out["l_aux"] == pytest.approx(alpha * E * min(C, T) / (T * k), rel=1e-12, abs=0)


# ---------------------------------------------------------------- 8-bit expert weights
def test_e4m3_decode_closed_forms():
    """Bit patterns of the E4M3 format: 1.0, 1.5, 2.0, the largest 448, the smallest normal
    2^-6, the smallest subnormal 2^-9, signed zero, -1 and NaN."""
    codes = np.array([0x38, 0x3C, 0x40, 0x7E, 0x08, 0x01, 0x00, 0x80, 0xB8, 0x7F, 0xFF],
                     dtype=np.uint8)
    v = O.decode_e4m3(codes)
    np.testing.assert_array_equal(v[:9], [1.0, 1.5, 2.0, 448.0, 2.0 ** -6, 2.0 ** -9, 0.0, -0.0, -1.0])
    assert np.signbit(v[7]) and np.isnan(v[9]) and np.isnan(v[10])


def test_e4m3_decode_matches_torch_float8_on_every_code():
    """All 256 codes against torch's own float8_e4m3fn -> float64 conversion."""
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.decode_e4m3(codes), ref)


def test_dequantize_rows_applies_one_scale_per_row():
    codes = np.array([[[0x38, 0x40], [0xB8, 0x3C]]], dtype=np.uint8)   # [1, 2, 2]
    w = O.dequantize_rows(codes, np.array([[0.5, 4.0]]))
    np.testing.assert_array_equal(w, [[[0.5, 1.0], [-4.0, 6.0]]])


# ---------------------------------------------------------------- block-scaled experts
def test_e2m1_decode_closed_forms():
    """The 16 E2M1 codes: 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives (sign bit 3)."""
    v = O.decode_e2m1(np.arange(16))
    np.testing.assert_array_equal(v[:8], [0, 0.5, 1, 1.5, 2, 3, 4, 6])
    np.testing.assert_array_equal(v[8:], -v[:8])
    assert np.signbit(v[8])


def test_e4m3_rounding_matches_torch_float8_conversion():
    """Round-to-nearest-even onto E4M3 against torch's float32 -> float8_e4m3fn conversion on
    float32 values: random magnitudes over every binade, the exact grid, the midpoints
    between neighbours (ties), subnormals and signed zeros."""
    rng = np.random.default_rng(41)
    grid = O.decode_e4m3(np.arange(0x7F)).astype(np.float32)            # 0 .. 448
    mids = ((grid[:-1].astype(np.float64) + grid[1:]) / 2).astype(np.float32)
    rand = (np.exp2(rng.uniform(-12, 8.8, 20000)) * rng.choice([-1, 1], 20000)).astype(np.float32)
    rand = rand[np.abs(rand) <= 448]
    v = np.concatenate([grid, -grid, mids, -mids, rand, np.float32([0.0, -0.0])])
    assert np.all(mids.astype(np.float64) == (grid[:-1].astype(np.float64) + grid[1:]) / 2)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(O.round_to_e4m3(v), ref)


@pytest.mark.parametrize("v,code", [(0.0, 0), (0.24, 0), (0.25, 0), (0.26, 1), (0.5, 1), (0.75, 2),
                                    (1.24, 2), (1.25, 2), (1.26, 3), (1.75, 4), (2.5, 4), (2.51, 5),
                                    (3.49, 5), (3.5, 6), (5.0, 6), (5.01, 7), (6.0, 7), (-0.3, 9),
                                    (-2.5, 12), (-6.0, 15)])
def test_e2m1_rounding_by_hand(v, code):
    """Nearest E2M1 value, ties to the even mantissa (0.25 -> 0, 0.75 -> 1, 1.25 -> 1,
    1.75 -> 2, 2.5 -> 2, 3.5 -> 4, 5 -> 4); the codes worked out by hand."""
    assert int(O.round_to_e2m1(np.array([v]))[0]) == code


def test_rounding_is_monotone_and_within_half_a_step():
    rng = np.random.default_rng(42)
    for fmt, qmax, n in (("e4m3", 448.0, 0x7F), ("e2m1", 6.0, 8)):
        v = np.sort(rng.uniform(-qmax, qmax, 5000))
        codes = O.round_to_e4m3(v) if fmt == "e4m3" else O.round_to_e2m1(v)
        q = O.mx_decode(codes, fmt)
        assert np.all(np.diff(q) >= 0)
        grid = np.sort(O.mx_decode(np.arange(n), fmt))
        gap = np.diff(grid)
        i = np.clip(np.searchsorted(grid, np.abs(v)) - 1, 0, len(gap) - 1)
        assert np.all(np.abs(np.abs(q) - np.abs(v)) <= gap[i] / 2 + 1e-12)


def test_mx_scale_exponent():
    """The smallest s with amax <= qmax * 2^s: brute force over s for random amax, and the
    closed cases (amax = qmax * 2^k gives k, a hair above gives k + 1, 0 gives -127)."""
    rng = np.random.default_rng(43)
    for qmax in (448.0, 6.0):
        a = np.exp2(rng.uniform(-100, 100, 300))
        s = O.mx_scale_exponent(a, qmax)
        for ai, si in zip(a, s):
            brute = next(t for t in range(-140, 140) if ai <= qmax * 2.0 ** t)
            assert si == max(-127, min(127, brute))
        k = np.arange(-20, 21)
        np.testing.assert_array_equal(O.mx_scale_exponent(qmax * np.exp2(k), qmax), k)
        np.testing.assert_array_equal(O.mx_scale_exponent(qmax * np.exp2(k) * (1 + 2.0 ** -40), qmax),
                                      k + 1)
        assert O.mx_scale_exponent(np.array([0.0]), qmax)[0] == -127
        assert O.mx_scale_exponent(np.array([1e-60]), qmax)[0] == -127


def test_mx_quantize_blocks():
    """Blocks of 32 along the last axis: values already on a block's grid come back exactly;
    each block's scale is set by its own maximum (a huge
    value in block 0 leaves block 1's small values at full E4M3 precision); the block
    maximum lands in (qmax / 2, qmax] before rounding, [qmax / 2, qmax] after; quantizing
    twice gives the values of quantizing once."""
    rng = np.random.default_rng(44)
    for fmt in ("e4m3", "e2m1"):
        n = 8 if fmt == "e2m1" else 0x7F
        codes = rng.integers(0, n, size=(5, 64)) | (rng.integers(0, 2, size=(5, 64)) << (3 if fmt == "e2m1" else 7))
        s = rng.integers(-20, 20, size=(5, 2))
        v = O.mx_dequantize(codes, s, fmt)
        v[:, 0] = O.MX_QMAX[fmt] * np.exp2(s[:, 0])                      # each block attains qmax
        v[:, 32] = -O.MX_QMAX[fmt] * np.exp2(s[:, 1])
        c2, s2 = O.mx_quantize(v, fmt)
        np.testing.assert_array_equal(s2, s)
        np.testing.assert_array_equal(O.mx_dequantize(c2, s2, fmt), v)
    x = np.concatenate([np.full(32, 1000.0), np.full(32, 1e-3)])[None]
    c, s = O.mx_quantize(x)
    xq = O.mx_dequantize(c, s)
    assert abs(xq[0, 40] - 1e-3) <= 1e-3 * 2.0 ** -4
    a = rng.normal(size=(7, 96)) * np.exp2(rng.integers(-30, 30, size=(7, 1)))
    c, s = O.mx_quantize(a)
    blk = np.abs(O.mx_dequantize(c, s)).reshape(7, 3, 32).max(-1) / np.exp2(s)
    assert np.all((blk >= 224) & (blk <= 448))
    # quantizing the quantized values again returns the same values (the codes may move one
    # binade when a block maximum rounded down to exactly qmax / 2)
    deq = O.mx_dequantize(c, s)
    np.testing.assert_array_equal(O.mx_dequantize(*O.mx_quantize(deq)), deq)


def test_swiglu_ffn_mx_by_hand():
    """d = F = 32, one row x = 1 (on the grid: x quantizes exactly), w1 = w3 = the first
    column of ones, so gate = up = 1 for every hidden unit and H = silu(1) = 0.7310586;
    the block's scale: 0.731 <= 448 * 2^-9 = 0.875 but > 448 * 2^-10, so s = -9 and
    0.7310586 * 2^9 = 374.3 rounds to 384 (E4M3 spacing 32 in [256, 448)): H is quantized to
    384 * 2^-9 = 0.75. w2 = all ones sums the 32 units: 24 (24.0, not 32 * 0.731 = 23.39)."""
    d = F = 32
    x = np.ones((1, d))
    w1 = np.zeros((F, d))
    w1[:, 0] = 1.0
    w2 = np.ones((d, F))
    y = O.swiglu_ffn_mx(x, w1, w1, w2)
    np.testing.assert_array_equal(y, np.full((1, d), 24.0))
    # x off the grid: 3.3 in a block whose maximum is 3.3: s = -7 (3.3 <= 448 / 128 = 3.5),
    # 3.3 * 128 = 422.4 rounds to 416 (spacing 32): x is quantized to 416 / 128 = 3.25
    x = np.zeros((1, d))
    x[0, 0] = 3.3
    w1 = np.zeros((F, d))
    w1[0, 0] = 1.0
    w3 = np.zeros((F, d))
    w3[0, 0] = 1.0 / 3.25
    w2 = np.zeros((d, F))
    w2[0, 0] = 1.0
    # gate = 3.25, up = 1: H_0 = silu(3.25) = 3.1271...; in its block: s = -7, *128 = 400.3,
    # spacing 32 -> 416 -> 3.25; everything else is 0
    y = O.swiglu_ffn_mx(x, w1, w3, w2)
    assert y[0, 0] == 3.25 and np.all(y[0, 1:] == 0)


def test_forward_mx_structure():
    """Identical experts and C = T: the layer is one dense FFN of the quantized operands
    (gates sum to 1); and against the same layer without any activation quantization the
    error stays at the E4M3 rounding level (neither zero nor gross)."""
    rng = np.random.default_rng(45)
    T, d, E, F, k = 24, 64, 4, 64, 2
    one = {nm: rng.normal(size=sh) / np.sqrt(sh[-1]) for nm, sh in
           (("w1", (F, d)), ("w3", (F, d)), ("w2", (d, F)))}
    mxw = dict(fmt="e4m3")
    for nm, w in one.items():
        c, s = O.mx_quantize(np.repeat(w[None], E, 0))
        mxw[nm], mxw[nm + "_s"] = c, s
    x = rng.normal(size=(T, d))
    wr = rng.normal(size=(E, d))
    out = O.forward_mx(x, wr, mxw, k=k, mode="softmax_topk", C=T)
    W = {nm: O.mx_dequantize(mxw[nm], mxw[nm + "_s"])[0] for nm in one}
    np.testing.assert_allclose(out["y"], O.swiglu_ffn_mx(x, W["w1"], W["w3"], W["w2"]),
                               rtol=1e-12, atol=1e-12)
    plain = O.forward(x, wr, *(O.mx_dequantize(mxw[nm], mxw[nm + "_s"]) for nm in ("w1", "w3", "w2")),
                      k=k, mode="softmax_topk", C=T)
    err = np.linalg.norm(out["y"] - plain["y"]) / np.linalg.norm(plain["y"])
    assert 0.005 < err < 0.08
