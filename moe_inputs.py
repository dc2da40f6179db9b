"""Seeded synthetic inputs for the MoE layer forward: workload presets and generators.

This module is shared by the CPU oracle's tests, the GPU parity tests and ``bench.py``.
It holds no step of the layer's arithmetic (no routing, capacity, FFN or loss): it only
names workload shapes and draws the tensors both sides consume.

Recipe (the same for every workload):

* ``x`` ~ N(0, 1), shape [T, d].
* router weight ``w_router`` ~ N(0, 1/d), shape [E, d] (an ``nn.Linear(d, E)`` weight,
  used as ``x @ w_router.T``).
* expert weights per expert e: ``w1[e]`` (gate) and ``w3[e]`` (up) ~ N(0, 1/d), shape
  [d_ff, d]; ``w2[e]`` (down) ~ N(0, 1/d_ff), shape [d, d_ff] (fan-in scaling).
* optional shared expert ``w1s, w3s`` [d_ff_shared, d] and ``w2s`` [d, d_ff_shared], same laws.
* optional per-expert router logit bias (Switch-style skewed load): a Zipf(s) popularity
  ranking with expert 0 the most popular, ``b_e = ln(r^-s / sum_{r'=1..E} r'^-s)``, r = e+1.
* draws are fp32 from ``torch.Generator(device).manual_seed(seed)`` in the fixed order
  x, w_router, w1, w3, w2, w1s, w3s, w2s (expert by expert), then rounded to nearest-even
  bf16 for bf16 workloads. The same realised tensors are handed to both the CUDA path and
  the oracle (the oracle receives fp64 copies of them).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int            # tokens
    d: int            # model width
    E: int            # routed experts
    k: int            # experts per token
    d_ff: int         # routed expert hidden width
    gate: str         # "softmax_all" | "softmax_topk" | "sigmoid_topk"
    dtype: str        # "f32" | "bf16"
    cf: Optional[float] = None   # capacity factor; None = no drop (capacity = T)
    d_ff_shared: int = 0         # 0 = no shared expert
    zipf_s: Optional[float] = None  # router logit bias from a Zipf(s) popularity ranking
    alpha: float = 0.01          # load-balancing loss coefficient
    beta: float = 1e-3           # router z-loss coefficient
    seed: int = 0

    def scaled(self, **kw) -> "Workload":
        """Same recipe with some sizes replaced (for small parity cases)."""
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    # Tiny fp32 layer, Mixtral gating, capacity factor 1.25 with drop.
    "tiny_fp32": Workload("tiny_fp32", T=256, d=128, E=8, k=2, d_ff=256,
                          gate="softmax_topk", dtype="f32", cf=1.25),
    # Mixtral-8x7B-shaped prefill layer, no drop.
    "mixtral_prefill": Workload("mixtral_prefill", T=4096, d=4096, E=8, k=2, d_ff=14336,
                                gate="softmax_topk", dtype="bf16"),
    # Switch-style top-1 layer with skewed load (Zipf 1.2 bias) and capacity factor 1.0.
    "switch_top1": Workload("switch_top1", T=16384, d=1024, E=128, k=1, d_ff=4096,
                            gate="softmax_all", dtype="bf16", cf=1.0, zipf_s=1.2),
    # DeepSeek-style fine-grained layer: 256 routed + 1 shared, sigmoid gates, top-8, no drop.
    "deepseek_fine": Workload("deepseek_fine", T=8192, d=7168, E=256, k=8, d_ff=2048,
                              gate="sigmoid_topk", dtype="bf16", d_ff_shared=2048),
    # Mixtral-shaped decode step (32 tokens): weight streaming.
    "mixtral_decode": Workload("mixtral_decode", T=32, d=4096, E=8, k=2, d_ff=14336,
                               gate="softmax_topk", dtype="bf16"),
}


def torch_dtype(w: Workload) -> torch.dtype:
    return torch.float32 if w.dtype == "f32" else torch.bfloat16


def zipf_log_popularity(E: int, s: float) -> torch.Tensor:
    """ln of Zipf(s) popularity over ranks 1..E (expert 0 = rank 1), fp32 [E]."""
    r = torch.arange(1, E + 1, dtype=torch.float64)
    p = r.pow(-s)
    p = p / p.sum()
    return p.log().to(torch.float32)


def _normal(gen, shape, std, device, out_dtype):
    t = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(out_dtype)


def _expert_stack(gen, E, rows, cols, std, device, out_dtype):
    out = torch.empty((E, rows, cols), device=device, dtype=out_dtype)
    for e in range(E):
        out[e].copy_(_normal(gen, (rows, cols), std, device, out_dtype))
    return out


def make_inputs(w: Workload, device="cpu", seed: Optional[int] = None) -> dict:
    """Draw every input of one workload on ``device``; returns a dict of tensors.

    Keys: x, w_router, router_bias (None unless zipf_s), w1, w3, w2, and w1s, w3s, w2s
    (None unless d_ff_shared > 0).
    """
    seed = w.seed if seed is None else seed
    dt = torch_dtype(w)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = _normal(g, (w.T, w.d), 1.0, device, dt)
    w_router = _normal(g, (w.E, w.d), 1.0 / math.sqrt(w.d), device, dt)
    w1 = _expert_stack(g, w.E, w.d_ff, w.d, 1.0 / math.sqrt(w.d), device, dt)
    w3 = _expert_stack(g, w.E, w.d_ff, w.d, 1.0 / math.sqrt(w.d), device, dt)
    w2 = _expert_stack(g, w.E, w.d, w.d_ff, 1.0 / math.sqrt(w.d_ff), device, dt)
    w1s = w3s = w2s = None
    if w.d_ff_shared > 0:
        fs = w.d_ff_shared
        w1s = _normal(g, (fs, w.d), 1.0 / math.sqrt(w.d), device, dt)
        w3s = _normal(g, (fs, w.d), 1.0 / math.sqrt(w.d), device, dt)
        w2s = _normal(g, (w.d, fs), 1.0 / math.sqrt(fs), device, dt)
    bias = None
    if w.zipf_s is not None:
        bias = zipf_log_popularity(w.E, w.zipf_s).to(device)
    return dict(x=x, w_router=w_router, router_bias=bias, w1=w1, w3=w3, w2=w2,
                w1s=w1s, w3s=w3s, w2s=w2s)


def random_logits(T: int, E: int, seed: int = 0, device="cpu", ties: bool = False) -> torch.Tensor:
    """fp32 router logits [T, E] ~ N(0,1); with ``ties`` they are rounded to multiples of
    0.25 in [-1, 1] so that equal logits are frequent."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    l = torch.randn((T, E), generator=g, device=device, dtype=torch.float32)
    if ties:
        l = (l * 4).round().clamp(-4, 4) / 4
    return l


def logits_with_popularity_bias(T: int, E: int, s: float, seed: int = 0, device="cpu") -> torch.Tensor:
    """fp32 logits N(0,1) plus a Zipf(s) log-popularity bias: a skewed, heavy-drop load."""
    return random_logits(T, E, seed, device) + zipf_log_popularity(E, s).to(device)


def quantize_rows_e4m3(w: torch.Tensor):
    """8-bit expert weights for weight streaming: per output row n, scale = max|w[n, :]| / 448
    and codes = round-to-nearest E4M3 of w / scale (torch's float8_e4m3fn cast). Returns
    (codes uint8, same shape as w; scales fp32, w.shape[:-1]). Works on any device."""
    wf = w.float()
    scale = wf.abs().amax(dim=-1).clamp_min(1e-12) / 448.0
    codes = (wf / scale.unsqueeze(-1)).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scale.contiguous()


_E2M1_MAGNITUDES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def quantize_weights_mx(w: torch.Tensor, fmt: str = "e4m3", host_codes: bool = False) -> dict:
    """Block-scaled expert weights: every 32 values along the last axis (K) share a power-of-two
    scale 2^s with s the smallest integer such that the block maximum fits the element format
    (448 for E4M3, 6 for E2M1); the elements are E4M3 codes (torch's float8_e4m3fn cast) or
    E2M1 codes (the nearest of the 8 magnitudes). Input preparation only: any valid codes
    would do.

    Returns on w's device:
      q  : E4M3 codes uint8 [E, N, K], or E2M1 codes packed two per byte [E, N, K / 2] (the even
           K index in the low nibble);
      sf : scale bytes s + 127 in 512-byte atoms [E, N / 128, K / 128, 512]: the scale of row n,
           columns 32j.. at byte (n % 32) * 16 + ((n % 128) / 32) * 4 + j % 4 of atom
           (n / 128, j / 4);
    and with host_codes, the same weights as numpy arrays for the CPU oracle: codes [E, N, K]
    (one code per value) and s [E, N, K / 32]."""
    E, N, K = w.shape
    assert N % 128 == 0 and K % 128 == 0
    qmax = 448.0 if fmt == "e4m3" else 6.0
    mags = torch.tensor(_E2M1_MAGNITUDES, device=w.device)
    qs, sfs, codes_h, s_h = [], [], [], []
    for e in range(E):                                 # one expert at a time: bounded memory
        blocks = w[e].double().reshape(N, K // 32, 32)
        amax = blocks.abs().amax(dim=-1)
        s = torch.ceil(torch.log2(amax.clamp_min(1e-300) / qmax))
        s = torch.where(amax > qmax * torch.exp2(s), s + 1, s)
        s = torch.where(amax <= qmax * torch.exp2(s - 1), s - 1, s)
        s = torch.where(amax > 0, s, torch.full_like(s, -127.0)).clamp(-127, 127)
        scaled = (blocks / torch.exp2(s).unsqueeze(-1)).float()
        del blocks
        if fmt == "e4m3":
            codes = scaled.to(torch.float8_e4m3fn).view(torch.uint8).reshape(N, K)
            q = codes
        else:
            idx = torch.empty(scaled.shape, dtype=torch.uint8, device=w.device)
            for r0 in range(0, N, 1024):
                a = scaled[r0:r0 + 1024].abs().unsqueeze(-1)
                idx[r0:r0 + 1024] = (a - mags).abs().argmin(dim=-1).to(torch.uint8)
            codes = (idx | (torch.signbit(scaled).to(torch.uint8) << 3)).reshape(N, K)
            q = (codes[:, 0::2] | (codes[:, 1::2] << 4)).contiguous()
        b = (s + 127).to(torch.uint8)                               # [N, K / 32]
        sfs.append(b.reshape(N // 128, 4, 32, K // 128, 4)          # n1, n0, ka, j
                   .permute(0, 3, 2, 1, 4).reshape(N // 128, K // 128, 512).contiguous())
        qs.append(q)
        if host_codes:
            codes_h.append(codes.cpu())
            s_h.append(s.to(torch.int64).cpu())
    out = dict(fmt=fmt, q=torch.stack(qs).contiguous(), sf=torch.stack(sfs).contiguous())
    if host_codes:
        out.update(codes=torch.stack(codes_h).numpy(), s=torch.stack(s_h).numpy())
    return out
