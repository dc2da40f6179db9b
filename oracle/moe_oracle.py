"""CPU oracle for the forward pass of one Mixture-of-Experts layer (numpy, fp64).

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports this module: only the
tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg call it. It shares
no code with the CUDA library (no headers, tables, helpers or constants).

Every step is the plain definition, written in the order the pages give it. The pages:

* [Tirogla] "Mixture of experts (MoE)" (tirogla.com): section "How it works", steps 1-6
  (score, select, dispatch, compute, combine, balance), and section "Code".
* [DL-S077] "DL S077 - Mixture of Experts (MoE) Intuition" (dineshblog.com): section 1.1
  (the SwiGLU expert), section 2 (top-k gating, with a worked example).
* [Starphix] "Mixture of Experts (MoE)" (learn.starphix.com): "Key Equations",
  "Shared + Specialized".

Readings where the pages are silent or disagree:

* selection compares raw logits, descending, the lower expert index winning ties;
* gates: softmax over all E ("softmax_all"), softmax over the k selected logits
  ("softmax_topk"), or sigmoid affinities renormalised over the selected k ("sigmoid_topk");
* expert FFN is w2(silu(w1 x) * w3 x): w1 = gate, w3 = up, w2 = down, no biases;
* dispatch keeps, per expert, the first C assignments in token order (assignment
  a = t*k + slot), drops the rest, and gates are not renormalised after a drop;
* f_i = (assignments routed to i before the drop) / (T*k); P_i = mean softmax-over-all
  probability; L_aux = alpha*E*sum_i f_i*P_i; L_z = beta*mean_t(logsumexp(l_t)^2);
* capacity C = ceil(cf*T*k/E), computed in fp64; "no drop" is C = T;
* an empty batch (T = 0) has both losses 0 (f and P are undefined there);
* block-scaled experts (forward_mx): weights stored as E4M3 or E2M1 codes with one
  power-of-two scale per 32 values along K; the activations entering each expert GEMM
  (x and H) quantized to E4M3 blocks with the smallest scale that holds the block's
  maximum, rounding to nearest, ties to even.

Every function here is pinned by a ``-m "not gpu"`` test against closed forms, the
pages' worked example, or brute force; none is "parity unpinned".
"""
from __future__ import annotations

import math

import numpy as np

GATE_MODES = ("softmax_all", "softmax_topk", "sigmoid_topk")


def _f64(a) -> np.ndarray:
    a = np.asarray(a, dtype=np.float64)
    return a


# ---------------------------------------------------------------------------------------
# Step 1: score.  [Tirogla] "How it works", step 1; [Starphix] "Key Equations".
# ---------------------------------------------------------------------------------------
def router_logits(x, w_router, bias=None) -> np.ndarray:
    """Router logits l = x . W_r^T (+ b): x [T, d], W_r [E, d] (nn.Linear layout), b [E]."""
    l = _f64(x) @ _f64(w_router).T
    if bias is not None:
        l = l + _f64(bias)[None, :]
    return l


def softmax_all(logits) -> np.ndarray:
    """Softmax over all E experts per token (the Switch/GShard router probability)."""
    l = _f64(logits)
    assert np.all(np.isfinite(l)), "router logits must be finite"
    m = l.max(axis=1, keepdims=True)
    e = np.exp(l - m)
    return e / e.sum(axis=1, keepdims=True)


def logsumexp(logits) -> np.ndarray:
    """Per-token log(sum_j exp(l_j)), in the max-shifted form."""
    l = _f64(logits)
    m = l.max(axis=1)
    return m + np.log(np.exp(l - m[:, None]).sum(axis=1))


# ---------------------------------------------------------------------------------------
# Step 2: select.  [Tirogla] "How it works", step 2, and "Code" (route: a stable sort by
# descending logit, so among equal logits the lower index comes first).
# ---------------------------------------------------------------------------------------
def select_topk(logits, k: int) -> np.ndarray:
    """Indices [T, k] (int64) of the k largest logits per token, descending; ties -> lower
    index first (stable sort on the negated logits)."""
    l = _f64(logits)
    assert np.all(np.isfinite(l)), "router logits must be finite"
    E = l.shape[1]
    assert 1 <= k <= E
    order = np.argsort(-l, axis=1, kind="stable")
    return order[:, :k].astype(np.int64)


def gates(logits, idx, mode: str) -> np.ndarray:
    """Gate weights [T, k] for the selected experts ``idx`` under one of three conventions.

    softmax_all  -- [Tirogla] step 1 (Switch, GShard): the softmax-over-all probability of
                    each selected expert, kept as is.
    softmax_topk -- [Tirogla] step 1 (Mixtral), [DL-S077] section 2: softmax over the k
                    selected logits only.
    sigmoid_topk -- [Tirogla] step 1 (DeepSeek-V3): sigmoid affinities of the selected
                    experts divided by their sum.
    """
    l = _f64(logits)
    sel = np.take_along_axis(l, np.asarray(idx), axis=1)
    if mode == "softmax_all":
        return np.take_along_axis(softmax_all(l), np.asarray(idx), axis=1)
    if mode == "softmax_topk":
        m = sel.max(axis=1, keepdims=True)
        e = np.exp(sel - m)
        return e / e.sum(axis=1, keepdims=True)
    if mode == "sigmoid_topk":
        s = 1.0 / (1.0 + np.exp(-sel))
        return s / s.sum(axis=1, keepdims=True)
    raise ValueError(f"unknown gate mode {mode!r}")


# ---------------------------------------------------------------------------------------
# Step 3: dispatch.  [Tirogla] "How it works", step 3 (group the (token, expert)
# assignments by expert with a counting sort, keep at most C per expert) and "Code"
# (dispatch: one pass over assignments in token order, which is the priority).
# ---------------------------------------------------------------------------------------
def capacity(cf: float, T: int, k: int, E: int) -> int:
    """C = ceil(cf * T * k / E), evaluated in fp64. [Tirogla] "Code" (main) and
    "Complexity and constants" (capacity factor)."""
    return int(math.ceil(cf * T * k / E))


def dispatch(idx, E: int, C: int) -> dict:
    """Counting sort of the T*k assignments by expert, keeping the first C per expert.

    Assignment a = t*k + slot. Returns int64 arrays:
      counts  [E]    assignments routed to each expert before the drop (n_e),
      offsets [E+1]  exclusive prefix sum of kept_e = min(n_e, C),
      perm    [R]    assignment id held by each kept row, grouped by expert, token order,
      inv     [T*k]  kept row of each assignment, or -1 if dropped,
      dropped        number of dropped assignments.
    """
    flat = np.asarray(idx).reshape(-1)
    slots = [[] for _ in range(E)]
    counts = np.zeros(E, dtype=np.int64)
    dropped = 0
    for a in range(flat.shape[0]):           # token order = priority
        e = int(flat[a])
        counts[e] += 1
        if len(slots[e]) < C:
            slots[e].append(a)
        else:
            dropped += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + len(slots[e])
    perm = np.array([a for e in range(E) for a in slots[e]], dtype=np.int64)
    inv = np.full(flat.shape[0], -1, dtype=np.int64)
    inv[perm] = np.arange(perm.shape[0], dtype=np.int64)
    return dict(counts=counts, offsets=offsets, perm=perm, inv=inv, dropped=dropped)


# ---------------------------------------------------------------------------------------
# Step 4: compute.  [DL-S077] section 1.1: each expert is a SwiGLU MLP,
# w2(silu(w1 x) * w3 x), no biases; w1 = gate, w3 = up, w2 = down.
# ---------------------------------------------------------------------------------------
def silu(z) -> np.ndarray:
    """silu(z) = z * sigmoid(z)."""
    z = _f64(z)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def swiglu_ffn(x_rows, w1, w3, w2) -> np.ndarray:
    """SwiGLU FFN of row vectors: x [n, d], w1/w3 [F, d], w2 [d, F] -> [n, d]."""
    x = _f64(x_rows)
    g = x @ _f64(w1).T
    u = x @ _f64(w3).T
    return (silu(g) * u) @ _f64(w2).T


def expert_outputs(x, disp: dict, k: int, w1, w3, w2) -> np.ndarray:
    """Ungated FFN output of every kept row: row r holds FFN_e(x_t) for the assignment
    a = perm[r] (t = a // k) and its expert e (the segment r falls in). [R, d]."""
    x = _f64(x)
    offsets, perm = disp["offsets"], disp["perm"]
    E = offsets.shape[0] - 1
    out = np.zeros((perm.shape[0], x.shape[1]), dtype=np.float64)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            toks = perm[lo:hi] // k
            out[lo:hi] = swiglu_ffn(x[toks], w1[e], w3[e], w2[e])
    return out


# ---------------------------------------------------------------------------------------
# Step 5: combine.  [Tirogla] "How it works", step 5: y_t = sum over the token's selected
# experts of g_{t,e} * FFN_e(x_t); a dropped assignment contributes nothing.
# [Starphix] "Shared + Specialized": an always-active shared expert is added.
# ---------------------------------------------------------------------------------------
def combine(g, inv, rows, T: int, k: int, shared=None) -> np.ndarray:
    """y [T, d] = sum_{slot} [inv >= 0] g[t, slot] * rows[inv[t*k+slot]]  (+ shared[t]).

    ``rows`` are ungated expert outputs indexed by kept row; summed in slot order."""
    rows = _f64(rows)
    g = _f64(g).reshape(T, k)
    inv = np.asarray(inv).reshape(T, k)
    d = rows.shape[1] if rows.ndim == 2 and rows.shape[0] > 0 else (
        np.asarray(shared).shape[1] if shared is not None else 0)
    y = np.zeros((T, d), dtype=np.float64)
    for s in range(k):
        kept = inv[:, s] >= 0
        if np.any(kept):
            y[kept] += g[kept, s][:, None] * rows[inv[kept, s]]
    if shared is not None:
        y = y + _f64(shared)
    return y


# ---------------------------------------------------------------------------------------
# Step 6: balance.  [Tirogla] "How it works", step 6, and "Code" (aux_loss, z_loss).
# ---------------------------------------------------------------------------------------
def load_fractions(idx, E: int) -> np.ndarray:
    """f_i: fraction of all T*k routing decisions that chose expert i (before any drop)."""
    flat = np.asarray(idx).reshape(-1)
    return np.bincount(flat, minlength=E).astype(np.float64) / flat.shape[0]


def aux_loss(logits, idx, alpha: float) -> float:
    """Switch load-balancing loss alpha * E * sum_i f_i * P_i, with P_i the mean over tokens
    of the softmax-over-all probability of expert i."""
    l = _f64(logits)
    E = l.shape[1]
    if l.shape[0] == 0:          # no tokens: f and P are undefined; reported as 0
        return 0.0
    f = load_fractions(idx, E)
    P = softmax_all(l).mean(axis=0)
    return float(alpha * E * np.dot(f, P))


def z_loss(logits, beta: float) -> float:
    """Router z-loss beta * mean_t(logsumexp(l_t)^2) (ST-MoE form)."""
    if _f64(logits).shape[0] == 0:   # no tokens: reported as 0
        return 0.0
    lse = logsumexp(logits)
    return float(beta * np.mean(lse * lse))


# ---------------------------------------------------------------------------------------
# Auxiliary-loss-free balancing (DeepSeek-V3).  [Tirogla] "Implementation notes": a
# per-expert bias is added to the scores used for top-k selection only (not to the gates)
# and nudged up or down after each step by load. [DL-S077] section 8.2: up when an expert
# is under-used, down when over-used. Readings: the score is the gate affinity (sigmoid of
# the logit for sigmoid gating, the softmax-over-all probability otherwise); the nudge is a
# fixed step gamma by the sign of (mean load - load), loads counted before any drop.
# ---------------------------------------------------------------------------------------
def affinity(logits, mode: str) -> np.ndarray:
    """Per-expert routing score the gates are built from: sigmoid(l) or softmax_all(l)."""
    l = _f64(logits)
    if mode == "sigmoid_topk":
        return 1.0 / (1.0 + np.exp(-l))
    return softmax_all(l)


def select_topk_biased(logits, k: int, mode: str, select_bias) -> np.ndarray:
    """Top-k of affinity + bias per token (descending, ties -> lower index)."""
    key = affinity(logits, mode) + _f64(select_bias)[None, :]
    order = np.argsort(-key, axis=1, kind="stable")
    return order[:, :k].astype(np.int64)


def update_select_bias(select_bias, counts, T: int, k: int, gamma: float) -> np.ndarray:
    """b_i + gamma if expert i received fewer than T*k/E assignments, - gamma if more,
    unchanged at exactly the mean; evaluated in fp32 like the bias it updates."""
    b = np.asarray(select_bias, dtype=np.float32).copy()
    n = np.asarray(counts, dtype=np.int64)
    E = b.shape[0]
    g = np.float32(gamma)
    under = n * E < T * k           # n_i < T*k/E without rounding
    over = n * E > T * k
    b[under] = b[under] + g
    b[over] = b[over] - g
    return b


# ---------------------------------------------------------------------------------------
# Expert-choice routing.  [Starphix] "Router Variants": experts choose their tokens (rather
# than tokens choosing experts), which balances the load perfectly. Readings: the score is
# the softmax-over-all router probability; expert e takes the C tokens with the highest
# score for e (ties -> lower token index); the gate of that pair is the score; a token's
# output sums, in expert order, over the experts that chose it (possibly none).
# ---------------------------------------------------------------------------------------
def expert_choice(logits, C: int) -> dict:
    """Per-expert token choice. Returns
      perm    [E*C']  token of each row, expert-major, ascending tokens inside an expert,
      offsets [E+1]   e*C' (C' = min(C, T)),
      gate    [E*C']  router probability of (token, expert) for each row,
      inv     [T, E]  row of (t, e), or -1 when expert e did not choose token t,
      counts  [E]     C' each, unrouted: tokens no expert chose."""
    p = softmax_all(logits)
    T, E = p.shape
    Cp = min(C, T)
    perm = np.zeros(E * Cp, dtype=np.int64)
    gate = np.zeros(E * Cp, dtype=np.float64)
    inv = np.full((T, E), -1, dtype=np.int64)
    for e in range(E):
        chosen = np.sort(np.argsort(-p[:, e], kind="stable")[:Cp])
        rows = np.arange(e * Cp, (e + 1) * Cp)
        perm[rows] = chosen
        gate[rows] = p[chosen, e]
        inv[chosen, e] = rows
    return dict(perm=perm, offsets=np.arange(E + 1, dtype=np.int64) * Cp, gate=gate, inv=inv,
                counts=np.full(E, Cp, dtype=np.int64),
                unrouted=int(np.sum(np.all(inv < 0, axis=1))))


def expert_choice_forward(x, w_router, w1, w3, w2, *, C: int, router_bias=None, w1s=None,
                          w3s=None, w2s=None, alpha: float = 0.01, beta: float = 1e-3,
                          k: int = 1, choice=None) -> dict:
    """The layer with expert-choice routing, in fp64. The balance loss uses f_i = C'/(T*k).

    ``choice`` (perm, offsets, inv of another implementation) replaces the experts' choices;
    the gates are then this oracle's probabilities of the given pairs."""
    x = _f64(x)
    T = x.shape[0]
    logits = router_logits(x, w_router, router_bias)
    ec = expert_choice(logits, C)
    E = logits.shape[1]
    if choice is not None:
        p = softmax_all(logits)
        ec = dict(ec)
        ec["perm"] = np.asarray(choice["perm"], dtype=np.int64)
        ec["offsets"] = np.asarray(choice["offsets"], dtype=np.int64)
        ec["inv"] = np.asarray(choice["inv"], dtype=np.int64).reshape(T, E)
        owner = np.repeat(np.arange(E), np.diff(ec["offsets"]))
        ec["gate"] = p[ec["perm"], owner]
    rows = np.zeros((ec["perm"].shape[0], x.shape[1]), dtype=np.float64)
    for e in range(E):
        lo, hi = int(ec["offsets"][e]), int(ec["offsets"][e + 1])
        if hi > lo:
            rows[lo:hi] = swiglu_ffn(x[ec["perm"][lo:hi]], w1[e], w3[e], w2[e])
    y = np.zeros_like(x)
    for e in range(E):                      # expert order
        sel = ec["inv"][:, e] >= 0
        r = ec["inv"][sel, e]
        y[sel] += ec["gate"][r][:, None] * rows[r]
    if w1s is not None:
        y = y + swiglu_ffn(x, w1s, w3s, w2s)
    P = softmax_all(logits).mean(axis=0) if T else np.zeros(E)
    f = ec["counts"] / float(T * k) if T else np.zeros(E)
    l_aux = float(alpha * E * np.dot(f, P)) if T else 0.0
    return dict(y=y, logits=logits, ec=ec, l_aux=l_aux, l_z=z_loss(logits, beta))


# ---------------------------------------------------------------------------------------
# Low-precision expert weights (weight streaming): each expert weight row n is stored as
# 8-bit E4M3 codes q[n, :] and one scale s[n], W[n, k] = decode(q[n, k]) * s[n]. The FFN
# is then the plain SwiGLU FFN of the decoded weights.
# E4M3 (the OCP 8-bit float "E4M3FN"): sign bit, 4 exponent bits with bias 7, 3 mantissa
# bits; exponent 0 encodes subnormals m/8 * 2^-6; exponent 15 with mantissa 7 is NaN; no
# infinities; the largest finite value is 448.
# ---------------------------------------------------------------------------------------
def decode_e4m3(codes) -> np.ndarray:
    """E4M3 byte codes (uint8 array) -> fp64 values."""
    b = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(b >> 7, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    sub = (m / 8.0) * 2.0 ** -6
    v = sign * np.where(e == 0, sub, normal)
    return np.where((e == 15) & ((b & 7) == 7), np.nan, v)


def dequantize_rows(codes, scales) -> np.ndarray:
    """W[..., n, k] = decode(codes[..., n, k]) * scales[..., n]."""
    return decode_e4m3(codes) * _f64(scales)[..., None]


# ---------------------------------------------------------------------------------------
# Block-scaled ("microscaling") experts: [Starphix] "Inference Optimization", Quantization
# (experts stored in 8 or 4 bits, the router kept in 16 bits) and [DL-S077] section 8.2
# (DeepSeek-V3 computes in FP8). The pages fix no format; the reading taken here:
#   * every 32 consecutive values along a row (the reduction axis K of a GEMM operand) share
#     one power-of-two scale 2^s, and each value is stored as an 8-bit E4M3 code or a 4-bit
#     E2M1 code: value = decode(code) * 2^s;
#   * expert weights are stored this way (E4M3 or E2M1 codes);
#   * the activations entering each expert GEMM -- the token rows x and the hidden rows
#     H = silu(x W1^T) * (x W3^T) -- are quantized to E4M3 blocks the same way, with
#     s = the smallest integer such that amax <= qmax * 2^s (qmax = 448 for E4M3, 6 for
#     E2M1; amax = 0 gives the smallest scale), s clamped to [-127, 127], and codes rounded to
#     the nearest value, ties to even (no value ever exceeds qmax, so nothing saturates);
#   * products of decoded values are exact and summed; the router, the gates and the combine
#     are those of the plain layer. There is no shared expert in this form.
# E2M1 (4 bits): sign bit 3, exponent bits 2..1 with bias 1, mantissa bit 0; exponent 0
# encodes m * 0.5; the values are 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives.
# ---------------------------------------------------------------------------------------
MX_BLOCK = 32
MX_QMAX = {"e4m3": 448.0, "e2m1": 6.0}


def decode_e2m1(codes) -> np.ndarray:
    """E2M1 codes (integers 0..15, one per value) -> fp64 values."""
    b = np.asarray(codes).astype(np.int64) & 0xF
    sign = np.where(b >> 3, -1.0, 1.0)
    e = (b >> 1) & 0x3
    m = (b & 1).astype(np.float64)
    return sign * np.where(e == 0, m * 0.5, (1.0 + m / 2.0) * np.exp2(e.astype(np.float64) - 1.0))


def mx_decode(codes, fmt: str) -> np.ndarray:
    return decode_e4m3(codes) if fmt == "e4m3" else decode_e2m1(codes)


def mx_scale_exponent(amax, qmax: float) -> np.ndarray:
    """The smallest integer s with amax <= qmax * 2^s, clamped to [-127, 127]; -127 for
    amax = 0. (Exact: qmax * 2^s is exact in fp64, and the candidate from log2 is moved to
    the smallest integer that satisfies the inequality.)"""
    a = _f64(amax)
    pos = a > 0
    s = np.zeros(a.shape, dtype=np.int64)
    with np.errstate(divide="ignore"):
        s[pos] = np.ceil(np.log2(a[pos] / qmax)).astype(np.int64)
    s[pos] = np.where(a[pos] > qmax * np.exp2(s[pos].astype(np.float64)), s[pos] + 1, s[pos])
    s[pos] = np.where(a[pos] <= qmax * np.exp2(s[pos].astype(np.float64) - 1.0), s[pos] - 1, s[pos])
    s[~pos] = -127
    return np.clip(s, -127, 127)


def round_to_e4m3(v) -> np.ndarray:
    """Codes of the E4M3 values nearest to v (|v| <= 448), ties to the even mantissa."""
    v = _f64(v)
    a = np.abs(v)
    f, e = np.frexp(np.where(a > 0, a, 1.0))               # a = f * 2^e, f in [0.5, 1)
    k = np.maximum(e - 1, -6)                              # binade; subnormals share 2^-6's ulp
    ulp = np.exp2(k.astype(np.float64) - 3.0)
    q = np.rint(a / ulp) * ulp                             # np.rint: half to even
    # encode q: normal when q >= 2^-6 (exponent field k + 7, mantissa (q / 2^k - 1) * 8)
    f2, e2 = np.frexp(np.where(q > 0, q, 1.0))
    k2 = e2 - 1
    normal = q >= 2.0 ** -6
    mant = np.where(normal, (q / np.exp2(k2.astype(np.float64)) - 1.0) * 8.0, q / 2.0 ** -9)
    code = np.where(normal, ((k2 + 7) << 3) | np.rint(mant).astype(np.int64),
                    np.rint(mant).astype(np.int64))
    code = np.where(q == 0, 0, code)
    assert np.all(a <= 448.0), "E4M3 rounding expects |v| <= 448"
    return (code | np.where(np.signbit(v), 0x80, 0)).astype(np.uint8)


def round_to_e2m1(v) -> np.ndarray:
    """Codes of the E2M1 values nearest to v (|v| <= 6), ties to the even mantissa: each
    magnitude is compared with the 8 grid values."""
    v = _f64(v)
    a = np.abs(v)
    assert np.all(a <= 6.0), "E2M1 rounding expects |v| <= 6"
    grid = decode_e2m1(np.arange(8))
    d = np.abs(a[..., None] - grid)
    best = np.min(d, axis=-1, keepdims=True)
    cand = d == best
    # among the (at most two) nearest grid values, the one with mantissa bit 0 (even code)
    even = cand & (np.arange(8) % 2 == 0)
    code = np.where(np.any(even, axis=-1), np.argmax(even, axis=-1), np.argmax(cand, axis=-1))
    return (code | np.where(np.signbit(v), 8, 0)).astype(np.uint8)


def mx_quantize(v, fmt: str = "e4m3"):
    """Blocks of 32 along the last axis -> (codes [..., n] uint8, s [..., n / 32] int64)."""
    v = _f64(v)
    n = v.shape[-1]
    assert n % MX_BLOCK == 0
    blocks = v.reshape(v.shape[:-1] + (n // MX_BLOCK, MX_BLOCK))
    s = mx_scale_exponent(np.max(np.abs(blocks), axis=-1), MX_QMAX[fmt])
    scaled = blocks / np.exp2(s.astype(np.float64))[..., None]
    codes = round_to_e4m3(scaled) if fmt == "e4m3" else round_to_e2m1(scaled)
    return codes.reshape(v.shape), s


def mx_dequantize(codes, s, fmt: str = "e4m3") -> np.ndarray:
    """decode(codes) * 2^s, one s per block of 32 along the last axis."""
    vals = mx_decode(codes, fmt)
    n = vals.shape[-1]
    blocks = vals.reshape(vals.shape[:-1] + (n // MX_BLOCK, MX_BLOCK))
    return (blocks * np.exp2(_f64(s))[..., None]).reshape(vals.shape)


def swiglu_ffn_mx(x_rows, w1, w3, w2) -> np.ndarray:
    """The expert FFN on block-scaled activations: x rows and the hidden rows H are each
    quantized to E4M3 blocks before their GEMM; w1, w3, w2 are the decoded weights."""
    xq = mx_dequantize(*mx_quantize(x_rows, "e4m3"), "e4m3")
    g = xq @ _f64(w1).T
    u = xq @ _f64(w3).T
    h = silu(g) * u
    hq = mx_dequantize(*mx_quantize(h, "e4m3"), "e4m3")
    return hq @ _f64(w2).T


def forward_mx(x, w_router, mxw: dict, *, k: int, mode: str, C: int, router_bias=None,
               alpha: float = 0.01, beta: float = 1e-3, idx_override=None) -> dict:
    """The layer with block-scaled experts. mxw: fmt ("e4m3" | "e2m1") and, for each of
    w1, w3 ([E, F, d]) and w2 ([E, d, F]), its codes and block exponents (keys "w1", "w1_s",
    ...). Steps 1-3, 5 and 6 as in forward(); step 4 is swiglu_ffn_mx."""
    x = _f64(x)
    T = x.shape[0]
    E = np.asarray(w_router).shape[0]
    fmt = mxw["fmt"]
    W = {nm: mx_dequantize(mxw[nm], mxw[nm + "_s"], fmt) for nm in ("w1", "w3", "w2")}
    logits = router_logits(x, w_router, router_bias)
    idx = select_topk(logits, k) if idx_override is None else np.asarray(idx_override, np.int64)
    g = gates(logits, idx, mode)
    disp = dispatch(idx, E, C)
    rows = np.zeros((disp["perm"].shape[0], x.shape[1]), dtype=np.float64)
    for e in range(E):
        lo, hi = int(disp["offsets"][e]), int(disp["offsets"][e + 1])
        if hi > lo:
            rows[lo:hi] = swiglu_ffn_mx(x[disp["perm"][lo:hi] // k], W["w1"][e], W["w3"][e],
                                        W["w2"][e])
    y = combine(g, disp["inv"], rows, T, k)
    return dict(y=y, logits=logits, idx=idx, gate=g, dispatch=disp,
                l_aux=aux_loss(logits, idx, alpha), l_z=z_loss(logits, beta))


# ---------------------------------------------------------------------------------------
# The whole layer, for inputs small enough to hold in fp64.
# ---------------------------------------------------------------------------------------
def route(logits, k: int, mode: str) -> dict:
    """Steps 1-2 on given logits: top-k indices and gates."""
    idx = select_topk(logits, k)
    return dict(idx=idx, gate=gates(logits, idx, mode))


def forward(x, w_router, w1, w3, w2, *, k: int, mode: str, C: int, router_bias=None,
            w1s=None, w3s=None, w2s=None, alpha: float = 0.01, beta: float = 1e-3,
            idx_override=None, select_bias=None) -> dict:
    """Full forward of one MoE layer in fp64.

    ``idx_override`` replaces the selected experts (the gates are then taken for those
    experts from the same logits); it lets a test recompute steps 3-6 on another
    implementation's routing decisions. ``select_bias`` [E] selects on affinity + bias
    (auxiliary-loss-free balancing); gates never include it.
    Returns y, logits, idx, gate, the dispatch dict, l_aux, l_z."""
    x = _f64(x)
    T = x.shape[0]
    E = np.asarray(w_router).shape[0]
    logits = router_logits(x, w_router, router_bias)
    if idx_override is not None:
        idx = np.asarray(idx_override, dtype=np.int64)
    elif select_bias is not None:
        idx = select_topk_biased(logits, k, mode, select_bias)
    else:
        idx = select_topk(logits, k)
    g = gates(logits, idx, mode)
    disp = dispatch(idx, E, C)
    rows = expert_outputs(x, disp, k, w1, w3, w2)
    shared = swiglu_ffn(x, w1s, w3s, w2s) if w1s is not None else None
    y = combine(g, disp["inv"], rows, T, k, shared)
    return dict(y=y, logits=logits, idx=idx, gate=g, dispatch=disp,
                l_aux=aux_loss(logits, idx, alpha), l_z=z_loss(logits, beta))


def near_tie_tokens(logits, k: int, eps: float = 1e-3) -> np.ndarray:
    """Tokens whose k-th and (k+1)-th largest logits differ by less than ``eps``: the only
    tokens whose expert set may legitimately differ between two implementations that
    round the router differently."""
    l = _f64(logits)
    E = l.shape[1]
    if k >= E:
        return np.zeros(0, dtype=np.int64)
    s = -np.sort(-l, axis=1)
    return np.nonzero(s[:, k - 1] - s[:, k] < eps)[0]
