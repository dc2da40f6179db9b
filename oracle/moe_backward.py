"""CPU oracle for the backward pass of one Mixture-of-Experts layer (numpy, fp64).

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports this module: only the
tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg call it. It shares
no code with the CUDA library.

What is differentiated. The layer of ``moe_oracle.forward`` maps (x, W_r, b, W1, W3, W2 and
the shared expert's weights) to y and two scalar losses. The objective whose gradient this
module returns is

    J = sum_t dy_t . y_t  +  d_aux * L_aux  +  d_z * L_z

for a given upstream gradient dy [T, d] and loss weights d_aux, d_z. The pages fix which
parts carry a gradient: [Tirogla] "How it works", step 6 -- the load fraction f_i is not
differentiable, the mean router probability P_i is; the top-k selection and the dispatch
(which assignment is kept) are piecewise constant and pass no gradient either. So with the
routing decisions held fixed, J is a smooth function of every input, and each function
below is the chain rule through one forward step, in the forward's own order:

  score   l = x W_r^T + b                      -> dx += dl W_r, dW_r = dl^T x, db = sum_t dl
  gates   g = gate_mode(l, idx)                -> dl from dg (per-mode Jacobian)
  compute O_r = w2 (silu(w1 x) * w3 x)         -> SwiGLU backward per kept row
  combine y_t = sum_slots g O_r (+ shared)     -> dg = dy . O_r,  dO_r = g dy_t
  balance L_aux = alpha E sum f_i P_i, L_z = beta mean lse^2 -> dl through P_i and lse

Every function here is pinned by ``tests/test_oracle_backward_pins.py``: central finite
differences of the (separately pinned) forward oracle, closed forms and invariants.
"""
from __future__ import annotations

import numpy as np

from .moe_oracle import (_f64, dispatch, gates, load_fractions, logsumexp, router_logits,
                         select_topk, silu, softmax_all)


# ---------------------------------------------------------------------------------------
# Gates.  [Tirogla] "How it works", step 1: the three gate conventions; only the gate values
# of the selected experts depend on the logits (the selection itself is constant).
# ---------------------------------------------------------------------------------------
def gate_backward(logits, idx, mode: str, dgate) -> np.ndarray:
    """dJ/dl [T, E] given dJ/dg = ``dgate`` [T, k] for the gates of the selected ``idx``.

    softmax_all : g_s = p_{i_s}, p = softmax(l) over all E:
                  dl_j = p_j (a_j - sum_i p_i a_i), a = dgate scattered onto the experts.
    softmax_topk: g = softmax of the k selected logits:
                  dl_{i_s} = g_s (dgate_s - sum_r g_r dgate_r), other experts 0.
    sigmoid_topk: g_s = sig_s / S, S = sum_r sig_r:
                  dsig_s = (dgate_s - sum_r g_r dgate_r) / S, dl_{i_s} = dsig_s sig_s (1 - sig_s).
    """
    l = _f64(logits)
    idx = np.asarray(idx, dtype=np.int64)
    dg = _f64(dgate)
    T, E = l.shape
    out = np.zeros((T, E), dtype=np.float64)
    rows = np.arange(T)[:, None]
    if mode == "softmax_all":
        p = softmax_all(l)
        a = np.zeros((T, E), dtype=np.float64)
        np.add.at(a, (np.broadcast_to(rows, idx.shape), idx), dg)
        return p * (a - (p * a).sum(axis=1, keepdims=True))
    g = gates(l, idx, mode)
    centred = dg - (g * dg).sum(axis=1, keepdims=True)
    if mode == "softmax_topk":
        dsel = g * centred
    elif mode == "sigmoid_topk":
        sel = np.take_along_axis(l, idx, axis=1)
        sig = 1.0 / (1.0 + np.exp(-sel))
        S = sig.sum(axis=1, keepdims=True)
        dsel = centred / S * sig * (1.0 - sig)
    else:
        raise ValueError(f"unknown gate mode {mode!r}")
    np.add.at(out, (np.broadcast_to(rows, idx.shape), idx), dsel)
    return out


# ---------------------------------------------------------------------------------------
# Balance.  [Tirogla] "How it works", step 6 and "Code" (aux_loss, z_loss).
# ---------------------------------------------------------------------------------------
def aux_loss_backward(logits, idx, alpha: float) -> np.ndarray:
    """dL_aux/dl [T, E]. L_aux = alpha E sum_i f_i P_i with f constant and
    P_i = (1/T) sum_t p_{t,i}; so with a_i = alpha E f_i / T,
    dl_{t,j} = p_{t,j} (a_j - sum_i p_{t,i} a_i)."""
    l = _f64(logits)
    T, E = l.shape
    if T == 0:
        return np.zeros((0, E))
    a = alpha * E * load_fractions(idx, E) / T
    p = softmax_all(l)
    return p * (a[None, :] - (p * a[None, :]).sum(axis=1, keepdims=True))


def z_loss_backward(logits, beta: float) -> np.ndarray:
    """dL_z/dl [T, E]. L_z = (beta/T) sum_t lse_t^2 and d lse_t / d l_{t,j} = p_{t,j}:
    dl_{t,j} = (2 beta / T) lse_t p_{t,j}."""
    l = _f64(logits)
    T = l.shape[0]
    if T == 0:
        return np.zeros_like(l)
    return (2.0 * beta / T) * logsumexp(l)[:, None] * softmax_all(l)


# ---------------------------------------------------------------------------------------
# Compute.  [DL-S077] section 1.1: O = w2 (silu(w1 x) * w3 x); w1 = gate, w3 = up, w2 = down.
# ---------------------------------------------------------------------------------------
def silu_grad(z) -> np.ndarray:
    """d silu / dz = sigma(z) (1 + z (1 - sigma(z)))."""
    z = _f64(z)
    with np.errstate(over="ignore"):
        s = 1.0 / (1.0 + np.exp(-z))
    return s * (1.0 + z * (1.0 - s))


def swiglu_ffn_backward(x_rows, w1, w3, w2, dout) -> dict:
    """Gradients of sum(dout * swiglu_ffn(x_rows, w1, w3, w2)).

    Forward: G = x w1^T, U = x w3^T, H = silu(G) U, O = H w2^T.
    Backward: dH = dout w2, dw2 = dout^T H, dG = dH U silu'(G), dU = dH silu(G),
    dx = dG w1 + dU w3, dw1 = dG^T x, dw3 = dU^T x.  Returns dx, dw1, dw3, dw2, and the
    forward's H (used for the gate gradient)."""
    x, w1, w3, w2, dout = (_f64(a) for a in (x_rows, w1, w3, w2, dout))
    G = x @ w1.T
    U = x @ w3.T
    H = silu(G) * U
    dH = dout @ w2
    dG = dH * U * silu_grad(G)
    dU = dH * silu(G)
    return dict(dx=dG @ w1 + dU @ w3, dw1=dG.T @ x, dw3=dU.T @ x, dw2=dout.T @ H, H=H)


# ---------------------------------------------------------------------------------------
# The whole layer.
# ---------------------------------------------------------------------------------------
def backward(x, w_router, w1, w3, w2, dy, *, k: int, mode: str, C: int, router_bias=None,
             w1s=None, w3s=None, w2s=None, alpha: float = 0.01, beta: float = 1e-3,
             d_aux: float = 1.0, d_z: float = 1.0, idx_override=None) -> dict:
    """Gradient of J = sum(dy * y) + d_aux L_aux + d_z L_z with respect to every input of
    the layer, the routing decisions (top-k and dispatch) held at their forward values.

    Returns dx [T, d], dw_router [E, d], d_router_bias [E], dw1, dw3 [E, F, d], dw2 [E, d, F],
    dw1s, dw3s, dw2s (None without a shared expert), and the intermediates dgate [T, k]
    (0 for dropped assignments), dlogits [T, E], idx, gate and the dispatch dict."""
    x = _f64(x)
    dy = _f64(dy)
    T, d = x.shape
    E = np.asarray(w_router).shape[0]
    w1, w3, w2 = _f64(w1), _f64(w3), _f64(w2)
    logits = router_logits(x, w_router, router_bias)
    idx = (np.asarray(idx_override, dtype=np.int64) if idx_override is not None
           else select_topk(logits, k))
    g = gates(logits, idx, mode)
    disp = dispatch(idx, E, C)
    offsets, perm, inv = disp["offsets"], disp["perm"], disp["inv"]

    dx = np.zeros((T, d))
    dw1, dw3, dw2 = np.zeros_like(w1), np.zeros_like(w3), np.zeros_like(w2)
    dgate_flat = np.zeros(T * k)
    gflat = g.reshape(-1)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        a = perm[lo:hi]                       # assignments kept by expert e, token order
        toks = a // k
        # combine: y_t += g_a O_a, so dO_a = g_a dy_t and dg_a = dy_t . O_a
        dout = gflat[a][:, None] * dy[toks]
        r = swiglu_ffn_backward(x[toks], w1[e], w3[e], w2[e], dout)
        O = r["H"] @ w2[e].T
        dgate_flat[a] = (dy[toks] * O).sum(axis=1)
        np.add.at(dx, toks, r["dx"])
        dw1[e], dw3[e], dw2[e] = r["dw1"], r["dw3"], r["dw2"]
    dgate = dgate_flat.reshape(T, k)
    assert np.all(dgate_flat[inv < 0] == 0.0)   # dropped assignments carry no gradient

    dlogits = gate_backward(logits, idx, mode, dgate)
    dlogits = dlogits + d_aux * aux_loss_backward(logits, idx, alpha)
    dlogits = dlogits + d_z * z_loss_backward(logits, beta)
    wr = _f64(w_router)
    dx += dlogits @ wr
    out = dict(dw_router=dlogits.T @ x, d_router_bias=dlogits.sum(axis=0), dw1=dw1, dw3=dw3,
               dw2=dw2, dw1s=None, dw3s=None, dw2s=None, dgate=dgate, dlogits=dlogits,
               idx=idx, gate=g, dispatch=disp)
    if w1s is not None:
        r = swiglu_ffn_backward(x, w1s, w3s, w2s, dy)   # shared expert: gate 1, every token
        dx += r["dx"]
        out.update(dw1s=r["dw1"], dw3s=r["dw3"], dw2s=r["dw2"])
    out["dx"] = dx
    return out


# ---------------------------------------------------------------------------------------
# Expert-choice routing ([Starphix] "Router Variants": experts choose their tokens).
# ---------------------------------------------------------------------------------------
def expert_choice_backward(x, w_router, w1, w3, w2, dy, *, C: int, router_bias=None, w1s=None,
                           w3s=None, w2s=None, alpha: float = 0.01, beta: float = 1e-3,
                           k: int = 1, d_aux: float = 1.0, d_z: float = 1.0,
                           choice=None) -> dict:
    """Gradient of J = sum(dy * y) + d_aux L_aux + d_z L_z for the expert-choice layer of
    moe_oracle.expert_choice_forward, the experts' choices held fixed (``choice`` as there).

    Each row r of expert e holds token t = perm[r] with gate p[t, e] (softmax over all E), so
    dO_r = p[t, e] dy_t and dgate_r = dy_t . O_r; the gates' gradient reaches the logits
    through the softmax over all E: dl_t = p_t (a_t - sum_j p_tj a_tj), a[t, e] = dgate of the
    row (t, e) or 0. f_i = C'/(T k) is the same for every expert, so L_aux = alpha E f sum_i
    P_i = alpha E f is constant in the logits and has no gradient; the z-loss has its usual one.
    Returns dx, dw_router, d_router_bias, dw1, dw3, dw2 (+ shared), dgate_rows [rows],
    dlogits [T, E] and the choice dict ``ec``."""
    from .moe_oracle import expert_choice_forward
    x = _f64(x)
    dy = _f64(dy)
    T, d = x.shape
    fwd = expert_choice_forward(x, w_router, w1, w3, w2, C=C, router_bias=router_bias,
                                alpha=alpha, beta=beta, k=k, choice=choice)
    ec, logits = fwd["ec"], fwd["logits"]
    E = logits.shape[1]
    w1, w3, w2 = _f64(w1), _f64(w3), _f64(w2)
    dx = np.zeros((T, d))
    dw1, dw3, dw2 = np.zeros_like(w1), np.zeros_like(w3), np.zeros_like(w2)
    dgate_rows = np.zeros(ec["perm"].shape[0])
    for e in range(E):
        lo, hi = int(ec["offsets"][e]), int(ec["offsets"][e + 1])
        if hi == lo:
            continue
        toks = ec["perm"][lo:hi]
        r = swiglu_ffn_backward(x[toks], w1[e], w3[e], w2[e], ec["gate"][lo:hi][:, None] * dy[toks])
        O = r["H"] @ w2[e].T
        dgate_rows[lo:hi] = (dy[toks] * O).sum(axis=1)
        np.add.at(dx, toks, r["dx"])
        dw1[e], dw3[e], dw2[e] = r["dw1"], r["dw3"], r["dw2"]
    a = np.where(ec["inv"] >= 0, dgate_rows[np.maximum(ec["inv"], 0)], 0.0)
    p = softmax_all(logits)
    dlogits = p * (a - (p * a).sum(axis=1, keepdims=True))
    dlogits = dlogits + d_z * z_loss_backward(logits, beta)
    dx += dlogits @ _f64(w_router)
    out = dict(dw_router=dlogits.T @ x, d_router_bias=dlogits.sum(axis=0), dw1=dw1, dw3=dw3,
               dw2=dw2, dw1s=None, dw3s=None, dw2s=None, dgate_rows=dgate_rows,
               dlogits=dlogits, ec=ec)
    if w1s is not None:
        r = swiglu_ffn_backward(x, w1s, w3s, w2s, dy)
        dx += r["dx"]
        out.update(dw1s=r["dw1"], dw3s=r["dw3"], dw2s=r["dw2"])
    out["dx"] = dx
    return out
