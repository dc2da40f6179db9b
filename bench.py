"""Benchmark of the MoE layer forward on B300: tokens/s and roofline fractions.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one moe_forward (router GEMM, gates/top-k, dispatch, gather, gate/up GEMM +
SwiGLU, down GEMM + gate scale, combine, balance losses) over one batch of the workload
(default: the Mixtral-shaped prefill layer, T=4096, d=4096, E=8, d_ff=14336, top-2, bf16).
Inputs are synthetic and seeded (moe_inputs.py), resident in HBM before the timed region.
L2 is flushed (a 256 MiB write) between timed steps, outside the timed events.

Under torchrun (N > 1) every rank runs an independent replica of the layer on its own GPU:
the layer has no cross-GPU exchange on one node's data-parallel path, so `value` is the sum
of all ranks' tokens divided by the slowest rank's time (weak scaling).

--impl reference times the CPU oracle (fp64 numpy, oracle/) on bounded samples of the same
workload on this host's cores; under torchrun only rank 0 runs it.

--backward times a training step instead: moe_forward followed by moe_backward (all input
and weight gradients of sum(dy*y) + L_aux + L_z, dy synthetic and seeded), with the per-stage
events of both and the roofline of the dominant backward kernel.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from moe_inputs import WORKLOADS, make_inputs  # noqa: E402

METRIC = "MoE layer fwd tokens/sec (1 B300) + % of BF16 tensor / HBM roofline"
UNIT = "tokens/s"
STAGES = ("router_gemm", "gates_topk", "dispatch", "gather", "gemm_gateup_swiglu",
          "gemm_down_scale", "combine", "aux_loss")
DOMINANT = "gemm_gateup_swiglu"
FLUSH_BYTES = 256 << 20


# ------------------------------------------------------------------------------ helpers
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained"), source="measured")
    return dict(hbm_gbs=6400.0, bf16_tflops=1800.0, bf16_tflops_sustained=1400.0, source="fallback")


def capacity(w):
    # the C ABI's own capacity helper (ceil(cf*T*k/E), clamped to T)
    from mixture_experts_layer_92_b300 import moe_capacity
    return w.T if w.cf is None else moe_capacity(w.cf, w.T, w.k, w.E)


def algorithmic_work(w, R: int, touched: int, wb=None, block_scales: bool = False):
    """FLOPs and bytes the method itself must compute and move for one forward.

    Layer: FLOPs = router 2*T*d*E + 6*d*d_ff per kept assignment (three GEMMs) + 6*d*d_ff_s
    per token for the shared expert; bytes = x + W_r + weights of the experts that received
    at least one token (3*d*d_ff each) + shared expert weights + y.
    Per kernel (one launch): gate/up GEMM 4*R*d*d_ff FLOPs over W1+W3 of the touched
    experts + its rows in and out; down GEMM 2*R*d*d_ff FLOPs over W2 + rows; the
    bandwidth kernels their rows in and out."""
    es = 4 if w.dtype == "f32" else 2
    wb = es if wb is None else wb          # bytes per routed-expert weight (1: 8-bit, 0.5: 4-bit)
    T, d, E, F, Fs, k = w.T, w.d, w.E, w.d_ff, w.d_ff_shared, w.k
    flops_router = 2.0 * T * d * E
    flops_gateup = 4.0 * R * d * F + 4.0 * T * d * Fs
    flops_down = 2.0 * R * d * F + 2.0 * T * d * Fs
    # weight scales: one byte per 32 weights (block-scaled), or an fp32 per row (8-bit rows)
    def wbytes(rows, K):
        if block_scales:
            return rows * K * (wb + 1.0 / 32)
        return rows * (K * wb + (4.0 if wb != es else 0.0))
    ab = 1.0 if block_scales else es       # bytes per activation element in the expert GEMMs
    bytes_gateup = (touched * wbytes(2.0 * F, d) + R * d * ab + R * F * ab
                    + (2.0 * Fs * d + T * d + T * Fs) * es)
    bytes_down = touched * wbytes(1.0 * d, F) + R * F * ab + R * d * es + (Fs * d + T * Fs + T * d) * es
    bytes_total = ((T * d + E * d + 3.0 * d * Fs + T * d) * es
                   + touched * (wbytes(2.0 * F, d) + wbytes(1.0 * d, F)))
    return dict(flops=flops_router + flops_gateup + flops_down, bytes=bytes_total,
                per_stage=dict(
                    router_gemm=(flops_router, (T * d + E * d) * es + T * E * 4.0),
                    gates_topk=(0.0, T * E * 4.0 + T * k * 8.0),
                    dispatch=(0.0, T * k * 4.0 * 3 + R * 4.0),
                    gather=(0.0, R * d * (es + (ab + ab / 32 if block_scales else es))),
                    gemm_gateup_swiglu=(flops_gateup, bytes_gateup),
                    gemm_down_scale=(flops_down, bytes_down),
                    combine=(0.0, (R * d + T * d * (2 if Fs else 1)) * es),
                    aux_loss=(0.0, 0.0)))


def slowest_rank_ms(times_ms, dist=None, device="cpu"):
    """The timing of the slowest rank: every rank passes its own [total_ms, e2e_ms, ...], all
    ranks get the element-wise maximum (a no-op with one process)."""
    t = torch.tensor([float(v) for v in times_ms], dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(tokens_per_step, steps, world, total_ms):
    """Replicas: every rank processes its own batch of tokens_per_step per step, so the job
    processes world times as many tokens in the slowest rank's time."""
    return tokens_per_step * steps * world / (total_ms / 1e3)


def tensor_peak(pk):
    """bf16 denominator: the burst figure (cuBLAS timed alone). Every kernel here is timed
    inside millisecond-scale steps, not inside a loop that runs for seconds, so the burst
    figure applies; the clocks the run saw are reported beside it, not folded into it."""
    return pk["bf16_tflops"], "bf16 burst"


def stage_roofline(flops, nbytes, ms, pk):
    """Achieved rate of one kernel against whichever roofline binds it (burst bf16 peak or
    HBM copy bandwidth, both measured)."""
    peak, _ = tensor_peak(pk)
    t_tensor = flops / (peak * 1e12)
    t_hbm = nbytes / (pk["hbm_gbs"] * 1e9)
    if flops > 0 and t_tensor >= t_hbm:
        ach = flops / (ms / 1e3) / 1e12
        return dict(ms=ms, bound="tensor", achieved=ach, unit="TFLOP/s", peak=peak,
                    frac=ach / peak, algorithmic=flops)
    ach = nbytes / (ms / 1e3) / 1e9 if ms > 0 else 0.0
    return dict(ms=ms, bound="hbm", achieved=ach, unit="GB/s", peak=pk["hbm_gbs"],
                frac=ach / pk["hbm_gbs"], algorithmic=nbytes)


def source_sha(path):
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def traffic_from_profile(workload: str, kernel: str):
    """dram bytes per launch from a committed ncu summary, or None if there is none or the
    kernel's source changed since it was captured."""
    p = os.path.join(ROOT, "profiles", f"{kernel}__{workload}.txt")
    if not os.path.exists(p):
        return None
    vals = {}
    for line in open(p):
        if ":" in line:
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    src = os.path.join(ROOT, "mixture_experts_layer_92_b300", "csrc", vals.get("source_file", ""))
    if "dram_bytes_per_launch" not in vals or not os.path.exists(src):
        return None
    if source_sha(src) != vals.get("source_sha256_16"):
        return None
    return float(vals["dram_bytes_per_launch"].split()[0])


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms while running."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.times = []                 # host clock (perf_counter) of each sample
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 8:
                self.rows.append(parts)
                self.times.append(time.perf_counter())

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, window=None):
        """Clocks of the samples taken inside `window` = (t0, t1) on the host clock (widened
        by one sampling period on each side, so that a timed region shorter than the period
        still gets its nearest samples); all samples when there is no window."""
        rows = self.rows
        if window is not None and self.times:
            t0, t1 = window[0] - 0.2, window[1] + 0.2
            rows = [r for r, t in zip(self.rows, self.times) if t0 <= t <= t1]
        if not rows:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=[], samples=0)
        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        pw = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in rows for n, v in zip(names, r[4:8]) if v == "Active"})
        return dict(sm_mhz=statistics.median(sm) if sm else None,
                    sm_max_mhz=max(mx) if mx else None, reasons=reasons, samples=len(rows),
                    power_w_max=max(pw) if pw else None)


# ------------------------------------------------------------------------------ CPU oracle arm
def oracle_sample(w, inp_host: dict, n_tokens: int, seed: int = 0):
    """Run the CPU oracle (as it stands) on a batch of n_tokens tokens of the workload;
    returns seconds."""
    import oracle as O
    C = w.T if w.cf is None else O.capacity(w.cf, n_tokens, w.k, w.E)
    x = inp_host["x"][:n_tokens]
    t0 = time.perf_counter()
    O.forward(x, inp_host["w_router"], inp_host["w1"], inp_host["w3"], inp_host["w2"], k=w.k,
              mode=w.gate, C=min(C, n_tokens), router_bias=inp_host["router_bias"],
              w1s=inp_host["w1s"], w3s=inp_host["w3s"], w2s=inp_host["w2s"], alpha=w.alpha,
              beta=w.beta)
    return time.perf_counter() - t0


def host_inputs(inp: dict) -> dict:
    return {k: (None if v is None else v.float().cpu().numpy()) for k, v in inp.items()}


def oracle_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        return max([i.get("num_threads", 1) for i in threadpool_info()] or [1])
    except Exception:
        return os.cpu_count() or 1


def grow_sample(n, t, n_max, target_s):
    """The next sample size when a sample of n tokens took t seconds, aiming at target_s;
    None once the sample is long enough (half the target) or the whole batch. The oracle has
    a per-call cost that does not scale with n, so one extrapolation can fall well short."""
    if t >= 0.5 * target_s or n >= n_max:
        return None
    return int(min(n_max, max(2 * n, n * target_s / max(t, 1e-3) * 0.8)))


def cpu_baseline(w, inp_host: dict, target_s: float = 15.0):
    n = min(w.T, 16)
    t = oracle_sample(w, inp_host, n)
    for _ in range(5):
        n2 = grow_sample(n, t, w.T, target_s)
        if n2 is None:
            break
        t = oracle_sample(w, inp_host, n2)
        n = n2
    return dict(value=n / t, unit=UNIT, cores=oracle_threads(), kind="oracle",
                sample=f"first {n} tokens of {w.name} (full routing/dispatch/FFN/combine/losses of "
                       f"that batch, fp64 numpy), {t:.2f} s")


def routing_report(w, ih: dict, gpu_idx: np.ndarray, y_gpu, C: int, fp8: bool = False,
                   n_sample: int = 32, seed: int = 7):
    """The routing comparison with the fp64 oracle on the whole batch (part of the CPU
    baseline leg: the oracle runs on the host, outside every timed region).

    near_ties: tokens whose k-th and (k+1)-th oracle logits differ by less than 1e-3;
    routed_differently: tokens whose GPU expert set differs from the oracle's (allowed only
    among near ties). On a seeded sample of tokens, y from the GPU is compared with the
    oracle's output under (a) the oracle's own routing of the whole batch (the direct end to
    end comparison: a routing flip also moves capacity drops of later tokens) and (b) the
    GPU's routing decisions (the FFN and combine numerics alone)."""
    import oracle as O
    t0 = time.perf_counter()
    logits = O.router_logits(ih["x"], ih["w_router"], ih["router_bias"])
    o_idx = O.select_topk(logits, w.k)
    ties = O.near_tie_tokens(logits, w.k)
    diff = np.nonzero(np.any(np.sort(o_idx, 1) != np.sort(gpu_idx, 1), axis=1))[0]
    rep = dict(eps=1e-3, tokens=w.T, near_ties=int(len(ties)),
               routed_differently=int(len(diff)),
               all_differences_among_near_ties=bool(set(diff.tolist()) <= set(ties.tolist())))
    if not fp8:
        tokens = np.sort(np.random.default_rng(seed).choice(w.T, size=min(n_sample, w.T),
                                                            replace=False))
        y = y_gpu[torch.as_tensor(tokens, device=y_gpu.device)].double().cpu().numpy()
        ref = {}
        for name, idx in (("oracle_routing", o_idx), ("gpu_routing", gpu_idx)):
            inv = O.dispatch(idx, w.E, C)["inv"].reshape(w.T, w.k)[tokens]
            g = O.gates(logits[tokens], idx[tokens], w.gate)
            rows = np.zeros((len(tokens) * w.k, w.d))
            for e in np.unique(idx[tokens]):
                sel = (idx[tokens] == e) & (inv >= 0)
                tl, sl = np.nonzero(sel)
                if len(tl):
                    rows[tl * w.k + sl] = O.swiglu_ffn(ih["x"][tokens[tl]], ih["w1"][e],
                                                       ih["w3"][e], ih["w2"][e])
            inv_l = np.where(inv >= 0, np.arange(len(tokens) * w.k).reshape(-1, w.k), -1)
            shared = (O.swiglu_ffn(ih["x"][tokens], ih["w1s"], ih["w3s"], ih["w2s"])
                      if ih.get("w1s") is not None else None)
            ref[name] = O.combine(g, inv_l, rows, len(tokens), w.k, shared)
        rl2 = lambda a, b: float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))
        rep.update(sample_tokens=int(len(tokens)),
                   rel_l2_direct=rl2(y, ref["oracle_routing"]),
                   rel_l2_gpu_routing=rl2(y, ref["gpu_routing"]))
    rep["host_seconds"] = round(time.perf_counter() - t0, 2)
    return rep


def oracle_train_sample(w, inp_host: dict, dy_host, n_tokens: int):
    """The CPU oracle's forward and backward on the first n_tokens tokens; returns seconds."""
    import oracle as O
    C = w.T if w.cf is None else O.capacity(w.cf, n_tokens, w.k, w.E)
    t0 = time.perf_counter()
    O.forward(inp_host["x"][:n_tokens], inp_host["w_router"], inp_host["w1"], inp_host["w3"],
              inp_host["w2"], k=w.k, mode=w.gate, C=min(C, n_tokens),
              router_bias=inp_host["router_bias"], w1s=inp_host["w1s"], w3s=inp_host["w3s"],
              w2s=inp_host["w2s"], alpha=w.alpha, beta=w.beta)
    O.backward(inp_host["x"][:n_tokens], inp_host["w_router"], inp_host["w1"], inp_host["w3"],
               inp_host["w2"], dy_host[:n_tokens], k=w.k, mode=w.gate, C=min(C, n_tokens),
               router_bias=inp_host["router_bias"], w1s=inp_host["w1s"], w3s=inp_host["w3s"],
               w2s=inp_host["w2s"], alpha=w.alpha, beta=w.beta)
    return time.perf_counter() - t0


def step_tokens(n1, t1, n2, t2, n_max, target_s=3.0):
    """Tokens per reference step from two timed samples, on the fit t(n) = a + b*n (a: the
    oracle's per-call cost that does not depend on the tokens, b: per token). A step is sized
    to max(target_s, 2a) seconds, so that at least half of it is per-token work; clamped to
    [n1, n_max]."""
    b = max((t2 - t1) / max(n2 - n1, 1), 1e-9)
    a = max(t1 - b * n1, 0.0)
    n = int(round((max(target_s, 2.0 * a) - a) / b))
    return max(n1, min(n_max, n))


def run_reference(args, w, rank):
    if rank != 0:
        return
    inp = make_inputs(w, device="cuda" if torch.cuda.is_available() else "cpu")
    ih = host_inputs(inp)
    del inp
    # size one step to a few seconds, from two samples
    n1 = min(w.T, 8)
    t1 = oracle_sample(w, ih, n1)
    n2 = min(w.T, 72)
    t2 = oracle_sample(w, ih, n2) if n2 > n1 else t1
    n = step_tokens(n1, t1, n2, t2, w.T)
    for _ in range(args.warmup):
        oracle_sample(w, ih, n)
    total = 0.0
    for _ in range(args.steps):
        total += oracle_sample(w, ih, n)
    val = n * args.steps / total
    cores = oracle_threads()
    sample = f"first {n} tokens of {w.name} per step (fp64 numpy oracle)"
    print(json.dumps(dict(
        impl="reference", metric=METRIC, value=val, unit=UNIT, n_gpus=args.gpus,
        steps=args.steps, warmup=args.warmup, ms_per_step=1e3 * total / args.steps,
        higher_is_better=True, scaling="weak", vs_baseline=None, dtype="f64", data="synthetic",
        config=dict(workload=w.name, tokens_per_step=n),
        cpu_baseline=dict(value=val, unit=UNIT, cores=cores, kind="oracle", sample=sample),
        e2e=dict(value=val, unit=UNIT, h2d_bytes_per_step=0, d2h_bytes_per_step=0))), flush=True)


# ------------------------------------------------------------------------------ GPU arm
def launches_per_forward(w, quantized=False) -> int:
    # router (bf16 with E <= 256: the fused router, which also routes; else the router GEMM
    # and the top-k kernel); top-k layers: dispatch (it also reduces the router statistics
    # to the losses), gather, gate/up GEMM, down GEMM, combine -- none for top-1 bf16 layers
    # without a shared expert, whose down projection writes y itself; the fp32 path launches
    # the shared expert's two GEMMs separately; expert choice: a selection and an
    # unrouted-token count in place of the dispatch, and the statistics kernel
    fused = w.dtype == "bf16" and w.E <= 256
    n = (1 if fused else 2) + 3 + (2 if (w.dtype == "f32" and w.d_ff_shared) else 0)
    if w.gate == "expert_choice":
        return n + 2 + 1 + 1
    direct = w.k == 1 and w.d_ff_shared == 0 and w.dtype == "bf16" and not quantized
    return n + 1 + (0 if direct else 1)


def run_ours(args, w, rank, world, local_rank):
    import mixture_experts_layer_92_b300 as moe
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    inp = make_inputs(w, device=dev)
    C = capacity(w)
    fp8 = None
    if args.fp8_weights:
        from moe_inputs import quantize_rows_e4m3
        fp8 = {}
        for nm in ("w1", "w3", "w2"):
            fp8[nm + "q"], fp8[nm + "s"] = quantize_rows_e4m3(inp[nm])
            inp[nm] = None                         # only the 8-bit copy stays resident
        torch.cuda.empty_cache()
    mx = None
    if args.mx_weights:
        from moe_inputs import quantize_weights_mx
        mx = dict(fmt=args.mx_weights)
        for nm in ("w1", "w3", "w2"):
            qw = quantize_weights_mx(inp[nm], args.mx_weights)
            mx[nm + "q"], mx[nm + "sf"] = qw["q"], qw["sf"]
            inp[nm] = None                         # only the block-scaled copy stays resident
        torch.cuda.empty_cache()
    layer = moe.MoELayer(inp["w_router"], inp["w1"], inp["w3"], inp["w2"], k=w.k, gate=w.gate,
                         capacity=C, router_bias=inp["router_bias"], w1s=inp["w1s"],
                         w3s=inp["w3s"], w2s=inp["w2s"], alpha=w.alpha, beta=w.beta, max_tokens=w.T,
                         balance_gamma=args.balance_gamma, fp8=fp8, mx=mx)
    x = inp["x"]
    y = torch.empty_like(x)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(STAGES) + 1)]
           for _ in range(args.steps)]
    ev_step = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    visible = [v for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    sampler = ClockSampler(visible[local_rank] if local_rank < len(visible) else local_rank)
    sampler.start()
    spread = []
    for i in range(args.warmup):
        flush.zero_()
        layer.forward(x, y)
        if i == 0:
            spread.append(float(layer.counts.max().item()) / (w.T * w.k / w.E))
    barrier()
    # timed steps: one event before and one after each forward, and one pair around the
    # dominant kernel (the gate/up GEMM) only; the other kernel boundaries carry no event, so
    # each launch still overlaps the previous kernel's tail
    ev_dom = [[None] * (len(STAGES) + 1) for _ in range(args.steps)]
    j_dom = STAGES.index(DOMINANT)
    for i in range(args.steps):
        ev_dom[i][j_dom] = torch.cuda.Event(enable_timing=True)
        ev_dom[i][j_dom + 1] = torch.cuda.Event(enable_timing=True)
    t_wall = time.perf_counter()
    t_timed0 = t_wall
    for i in range(args.steps):
        flush.zero_()
        ev_step[i][0].record(stream)
        layer.forward(x, y, events=ev_dom[i])
        ev_step[i][1].record(stream)
    barrier()
    t_timed1 = time.perf_counter()
    t_wall = t_timed1 - t_wall
    # the per-stage breakdown: the same steps again with an event at every stage boundary
    for i in range(args.steps):
        flush.zero_()
        layer.forward(x, y, events=evs[i])
    barrier()
    err = moe.moe_get_error(layer.ws)
    if err != 0:
        raise RuntimeError(f"device error {moe.moe_status_string(err)}")
    step_ms = [ev_step[i][0].elapsed_time(ev_step[i][1]) for i in range(args.steps)]
    dom_ms = [ev_dom[i][j_dom].elapsed_time(ev_dom[i][j_dom + 1]) for i in range(args.steps)]
    stage_ms = {name: [evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(args.steps)]
                for j, name in enumerate(STAGES)}
    total_ms = sum(step_ms)
    # for the routing report: the GPU's own top-k of the whole batch (the same routing
    # kernels moe_forward runs), read back once, outside every timed region
    gpu_idx = None
    if w.gate != "expert_choice" and args.balance_gamma is None:
        gpu_idx = layer.route(x).cpu().numpy().astype(np.int64)

    # end to end through the public API from pinned host memory: every step copies its own
    # x in and its y out; MoELayer.forward_host_stream overlaps those copies with the layer
    x_host = x.cpu().pin_memory()
    y_hosts = [torch.empty(y.shape, dtype=y.dtype, pin_memory=True) for _ in range(2)]
    layer.forward_host_stream([x_host] * args.warmup, [y_hosts[i % 2] for i in range(args.warmup)])
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    layer.forward_host_stream([x_host] * args.steps, [y_hosts[i % 2] for i in range(args.steps)])
    e1.record(stream)
    barrier()
    sampler.stop()
    e2e_ms = e0.elapsed_time(e1)
    err = layer.device_error()
    if err != 0:
        raise RuntimeError(f"device error {moe.moe_status_string(err)} in the host-memory steps")

    # the slowest rank sets the time
    total_ms, e2e_ms = slowest_rank_ms([total_ms, e2e_ms], dist, dev)
    counts = layer.counts.cpu().numpy()
    spread.append(float(counts.max()) / (w.T * w.k / w.E))
    R = int(np.minimum(counts, C).sum())
    touched = int((counts > 0).sum())
    if rank != 0:
        if dist is not None:
            dist.barrier()
            dist.destroy_process_group()
        return
    pk = peaks()
    wb = 1 if (args.fp8_weights or args.mx_weights == "e4m3") else (
        0.5 if args.mx_weights == "e2m1" else None)
    work = algorithmic_work(w, R, touched, wb=wb, block_scales=bool(args.mx_weights))
    tokens = w.T * args.steps * world
    value = whole_job_rate(w.T, args.steps, world, total_ms)
    ms_per_step = total_ms / args.steps
    clk = sampler.summary(window=(t_timed0, t_timed1))
    tpeak, tpeak_name = tensor_peak(pk)
    stages = {}
    for name in STAGES:
        flops, nbytes = work["per_stage"][name]
        stages[name] = stage_roofline(flops, nbytes, statistics.mean(stage_ms[name]), pk)
    roofline = None
    if w.dtype == "bf16":
        # the dominant kernel as timed inside the timed steps themselves (its own event pair)
        dom = stage_roofline(*work["per_stage"][DOMINANT], statistics.mean(dom_ms), pk)
        tr = traffic_from_profile(w.name, DOMINANT)
        roofline = dict(bound=dom["bound"], kernel=DOMINANT, achieved=dom["achieved"],
                        peak=dom["peak"], unit=dom["unit"], frac=dom["frac"], traffic=tr,
                        peak_source=f"{pk['source']} " + (
                            tpeak_name if dom["bound"] == "tensor" else "HBM copy"),
                        kernel_ms=dom["ms"], algorithmic_per_launch=dom["algorithmic"],
                        timing="CUDA events around this kernel's launch inside the timed steps")
        if clk.get("sm_mhz") and clk.get("sm_max_mhz"):
            roofline["clock_note"] = (
                f"median SM clock {clk['sm_mhz']:.0f} of {clk['sm_max_mhz']:.0f} MHz around the "
                f"timed steps; at the maximum clock this kernel time would be "
                f"{dom['ms'] * clk['sm_mhz'] / clk['sm_max_mhz']:.4f} ms")
    t_roof = max(work["flops"] / (tpeak * 1e12), work["bytes"] / (pk["hbm_gbs"] * 1e9))
    layer_roof = dict(flops=work["flops"], bytes=work["bytes"], roofline_ms=t_roof * 1e3,
                      measured_ms=ms_per_step, frac=t_roof * 1e3 / ms_per_step,
                      note=f"max(FLOPs / {tpeak_name} peak, bytes / HBM peak), measured peaks")
    cpu = None
    report = None
    quantized = bool(args.fp8_weights or args.mx_weights)
    if world == 1 and not args.no_cpu_baseline and not quantized:
        ih = host_inputs(inp)
        cpu = cpu_baseline(w, ih, target_s=args.cpu_seconds)
        if gpu_idx is not None:
            report = routing_report(w, ih, gpu_idx, y, C)
    es = x.element_size()
    line = dict(
        metric=METRIC, value=value, unit=UNIT, n_gpus=world, steps=args.steps,
        warmup=args.warmup, ms_per_step=ms_per_step, higher_is_better=True, scaling="weak",
        vs_baseline=None, dtype=w.dtype, data="synthetic (seeded; random-init weights)",
        config=dict(workload=w.name, T=w.T, d=w.d, E=w.E, k=w.k, d_ff=w.d_ff,
                    d_ff_shared=w.d_ff_shared, gate=w.gate, capacity=C,
                    l2="flushed between timed steps (256 MiB write, outside the events); "
                       "expert weights also exceed L2",
                    kept_assignments=R, experts_touched=touched,
                    wall_s=t_wall),
        roofline=roofline, layer_roofline=layer_roof, stages=stages,
        cpu_baseline=cpu, routing_report=report,
        e2e=dict(value=whole_job_rate(w.T, args.steps, world, e2e_ms), unit=UNIT,
                 h2d_bytes_per_step=w.T * w.d * es,
                 d2h_bytes_per_step=w.T * w.d * es,
                 note="MoELayer.forward_host_stream: for plain bf16/fp32 layers one "
                      "moe_host_pipeline_forward C-ABI call per step (x pinned host -> device on "
                      "the pipeline's upload stream, the layer on the compute stream, y -> pinned "
                      "host on its download stream; copies of neighbouring steps overlap the "
                      "layer); 8-bit and balanced layers copy through torch around the call"),
        gpu_launches=(launches_per_forward(w, quantized)
                      + (1 if args.balance_gamma is not None else 0))
        * args.steps,
        clocks=dict(sm_mhz=clk["sm_mhz"], sm_max_mhz=clk["sm_max_mhz"], reasons=clk["reasons"],
                    samples=clk["samples"],
                    window="nvidia-smi samples (every 200 ms) from 0.2 s before the timed steps "
                           "to 0.2 s after them"))
    if args.balance_gamma is not None:
        line["balance"] = dict(gamma=args.balance_gamma, load_spread_first_step=spread[0],
                               load_spread_last_step=spread[-1],
                               note="max expert load / mean load (pre-drop); the selection "
                                    "bias is nudged after every forward, warm-up included")
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


# ------------------------------------------------------------------------------ training step
TRAIN_METRIC = "MoE layer fwd+bwd (training step) tokens/sec (1 B300) + % of BF16 tensor / HBM roofline"
BWD_STAGES = ("route_dispatch", "gather_x_dy", "recompute_gu", "gemm_dh_swiglu_bwd",
              "gate_logit_grads", "gemm_dx", "dx_combine", "gemm_wgrad")
BWD_DOMINANT = "gemm_wgrad"


def backward_work(w, R: int, touched: int):
    """FLOPs and bytes of one moe_backward, per stage (the same conventions as
    algorithmic_work). GEMM FLOPs: recomputed G|U 4RdF, dH 2RdF, dX 4RdF, weight gradients
    6RdF (+ the shared expert's over T rows, + router dx and dW_r 2TdE each)."""
    es = 2
    T, d, E, F, Fs, k = w.T, w.d, w.E, w.d_ff, w.d_ff_shared, w.k
    wts = touched * 3.0 * d * F * es + 3.0 * d * Fs * es
    per = dict(
        route_dispatch=(2.0 * T * d * E, (T * d + E * d) * es + T * E * 8.0 + T * k * 16.0),
        gather_x_dy=(0.0, (2 * R * d + 3 * R * d) * es),
        recompute_gu=(4.0 * d * (R * F + T * Fs),
                      touched * 2.0 * F * d * es + 2.0 * Fs * d * es + (R * d + 2 * R * F
                                                                        + T * d + 2 * T * Fs) * es),
        gemm_dh_swiglu_bwd=(2.0 * d * (R * F + T * Fs),
                            touched * d * F * es + Fs * d * es + (R * d + 5 * R * F
                                                                  + T * d + 5 * T * Fs) * es),
        gate_logit_grads=(0.0, T * k * 8.0 + T * E * 14.0),
        gemm_dx=(4.0 * d * (R * F + T * Fs) + 2.0 * T * E * d,
                 touched * 2.0 * F * d * es + 2.0 * Fs * d * es + (2 * R * F + R * d + 2 * T * Fs
                                                                   + 2 * T * d) * es),
        dx_combine=(0.0, (R * d + 3 * T * d) * es),
        gemm_wgrad=(6.0 * d * (R * F + T * Fs) + 2.0 * T * E * d,
                    (R * (2 * F + 2 * d + F) + T * (3 * Fs + 2 * d)) * es + (E * 3.0 * d * F
                                                                              + 3.0 * d * Fs + E * d) * 4.0))
    flops = sum(v[0] for v in per.values())
    nbytes = wts + (2 * T * d * es) + (E * 3.0 * d * F + 3.0 * d * Fs + E * d) * 4.0
    return dict(flops=flops, bytes=nbytes, per_stage=per)


def run_train(args, w, rank, world, local_rank):
    import mixture_experts_layer_92_b300 as moe
    from mixture_experts_layer_92_b300 import _lib as L
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    inp = make_inputs(w, device=dev)
    C = capacity(w)
    gen = torch.Generator(device=dev).manual_seed(1)
    dy = torch.randn(inp["x"].shape, generator=gen, device=dev).to(inp["x"].dtype)
    layer = moe.MoELayer(inp["w_router"], inp["w1"], inp["w3"], inp["w2"], k=w.k, gate=w.gate,
                         capacity=C, router_bias=inp["router_bias"], w1s=inp["w1s"],
                         w3s=inp["w3s"], w2s=inp["w2s"], alpha=w.alpha, beta=w.beta, max_tokens=w.T)
    s = layer.shape(w.T)
    bws = L.alloc_workspace_backward(s, dev)
    f32 = dict(device=dev, dtype=torch.float32)
    grads = dict(dx=torch.empty_like(inp["x"]), dw_router=torch.empty((w.E, w.d), **f32),
                 dw1=torch.empty((w.E, w.d_ff, w.d), **f32), dw3=torch.empty((w.E, w.d_ff, w.d), **f32),
                 dw2=torch.empty((w.E, w.d, w.d_ff), **f32))
    if w.d_ff_shared:
        grads.update(dw1s=torch.empty((w.d_ff_shared, w.d), **f32),
                     dw3s=torch.empty((w.d_ff_shared, w.d), **f32),
                     dw2s=torch.empty((w.d, w.d_ff_shared), **f32))
    x = inp["x"]
    y = torch.empty_like(x)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def backward(xx, dyy, events=None):
        L.moe_backward(s, bws, xx, inp["w_router"], inp["w1"], inp["w3"], inp["w2"], dyy,
                       grads["dx"], grads["dw_router"], grads["dw1"], grads["dw3"], grads["dw2"],
                       router_bias=inp["router_bias"], w1s=inp["w1s"], w3s=inp["w3s"],
                       w2s=inp["w2s"], dw1s=grads.get("dw1s"), dw3s=grads.get("dw3s"),
                       dw2s=grads.get("dw2s"), events=events)

    fevs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(STAGES) + 1)]
            for _ in range(args.steps)]
    bevs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(BWD_STAGES) + 1)]
            for _ in range(args.steps)]
    ev_step = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    visible = [v for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    sampler = ClockSampler(visible[local_rank] if local_rank < len(visible) else local_rank)
    sampler.start()
    for _ in range(args.warmup):
        flush.zero_()
        layer.forward(x, y)
        backward(x, dy)
    barrier()
    t_timed0 = time.perf_counter()
    for i in range(args.steps):                 # timed: start and end events only
        flush.zero_()
        ev_step[i][0].record(stream)
        layer.forward(x, y)
        backward(x, dy)
        ev_step[i][1].record(stream)
    barrier()
    t_timed1 = time.perf_counter()
    for i in range(args.steps):                 # per-stage breakdown
        flush.zero_()
        layer.forward(x, y, events=fevs[i])
        backward(x, dy, events=bevs[i])
    barrier()
    for ws in (layer.ws, bws):
        if moe.moe_get_error(ws) != 0:
            raise RuntimeError("device error")
    step_ms = [ev_step[i][0].elapsed_time(ev_step[i][1]) for i in range(args.steps)]
    fwd_ms = [fevs[i][0].elapsed_time(fevs[i][-1]) for i in range(args.steps)]
    bwd_ms = [bevs[i][0].elapsed_time(bevs[i][-1]) for i in range(args.steps)]
    bstage_ms = {name: [bevs[i][j].elapsed_time(bevs[i][j + 1]) for i in range(args.steps)]
                 for j, name in enumerate(BWD_STAGES)}
    total_ms = sum(step_ms)

    # end to end: x and dy from pinned host memory in, y and dx out, every step
    xh, dyh = x.cpu().pin_memory(), dy.cpu().pin_memory()
    yh = torch.empty(y.shape, dtype=y.dtype, pin_memory=True)
    dxh = torch.empty(y.shape, dtype=y.dtype, pin_memory=True)
    xd, dyd = torch.empty_like(x), torch.empty_like(dy)

    def e2e_step():
        xd.copy_(xh, non_blocking=True)
        dyd.copy_(dyh, non_blocking=True)
        layer.forward(xd, y)
        backward(xd, dyd)
        yh.copy_(y, non_blocking=True)
        dxh.copy_(grads["dx"], non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    barrier()
    sampler.stop()
    e2e_ms = e0.elapsed_time(e1)
    total_ms, e2e_ms = slowest_rank_ms([total_ms, e2e_ms], dist, dev)
    counts = layer.counts.cpu().numpy()
    R = int(np.minimum(counts, C).sum())
    touched = int((counts > 0).sum())
    if rank != 0:
        if dist is not None:
            dist.barrier()
            dist.destroy_process_group()
        return
    pk = peaks()
    fw = algorithmic_work(w, R, touched)
    bw = backward_work(w, R, touched)
    tokens = w.T * args.steps * world
    clk = sampler.summary(window=(t_timed0, t_timed1))
    tpeak, tpeak_name = tensor_peak(pk)
    stages = {name: stage_roofline(*bw["per_stage"][name], statistics.mean(bstage_ms[name]), pk)
              for name in BWD_STAGES}
    dom = stages[BWD_DOMINANT]
    roofline = dict(bound=dom["bound"], kernel=BWD_DOMINANT, achieved=dom["achieved"],
                    peak=dom["peak"], unit=dom["unit"], frac=dom["frac"],
                    traffic=traffic_from_profile(w.name + "+train", BWD_DOMINANT),
                    peak_source=f"{pk['source']} " + (
                        tpeak_name if dom["bound"] == "tensor" else "HBM copy"),
                    algorithmic_per_step=dom["algorithmic"],
                    note="gemm_wgrad = all weight-gradient GEMM launches of one backward")
    flops = fw["flops"] + bw["flops"]
    nbytes = fw["bytes"] + bw["bytes"]
    ms_per_step = total_ms / args.steps
    t_roof = max(flops / (tpeak * 1e12), nbytes / (pk["hbm_gbs"] * 1e9))
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        ih = host_inputs(inp)
        dyh64 = dy.float().cpu().numpy()
        n = min(w.T, 4)
        tt = oracle_train_sample(w, ih, dyh64, n)
        for _ in range(5):
            n2 = grow_sample(n, tt, w.T, args.cpu_seconds)
            if n2 is None:
                break
            tt = oracle_train_sample(w, ih, dyh64, n2)
            n = n2
        cpu = dict(value=n / tt, unit=UNIT, cores=oracle_threads(), kind="oracle",
                   sample=f"first {n} tokens of {w.name}: oracle forward + backward (fp64 numpy), "
                          f"{tt:.2f} s")
    es = x.element_size()
    line = dict(
        metric=TRAIN_METRIC, value=whole_job_rate(w.T, args.steps, world, total_ms), unit=UNIT,
        n_gpus=world,
        steps=args.steps, warmup=args.warmup, ms_per_step=ms_per_step, higher_is_better=True,
        scaling="weak", vs_baseline=None, dtype=w.dtype,
        data="synthetic (seeded; random-init weights; dy ~ N(0,1))",
        config=dict(workload=w.name + "+train", T=w.T, d=w.d, E=w.E, k=w.k, d_ff=w.d_ff,
                    d_ff_shared=w.d_ff_shared, gate=w.gate, capacity=C,
                    l2="flushed between timed steps (256 MiB write, outside the events)",
                    kept_assignments=R, experts_touched=touched,
                    forward_ms=statistics.mean(fwd_ms), backward_ms=statistics.mean(bwd_ms)),
        roofline=roofline,
        layer_roofline=dict(flops=flops, bytes=nbytes, roofline_ms=t_roof * 1e3,
                            measured_ms=ms_per_step, frac=t_roof * 1e3 / ms_per_step,
                            note=f"max(FLOPs / {tpeak_name} peak, bytes / HBM peak), "
                                 "measured peaks"),
        stages=stages, cpu_baseline=cpu,
        e2e=dict(value=whole_job_rate(w.T, args.steps, world, e2e_ms), unit=UNIT,
                 h2d_bytes_per_step=2 * w.T * w.d * es,
                 d2h_bytes_per_step=2 * w.T * w.d * es,
                 note="per step: x and dy (pinned) -> device, forward, backward, y and dx -> host; "
                      "the weight gradients stay on the device"),
        gpu_launches=(launches_per_forward(w) + 15 + (4 if w.d_ff_shared else 0)) * args.steps,
        clocks=dict(sm_mhz=clk["sm_mhz"], sm_max_mhz=clk["sm_max_mhz"], reasons=clk["reasons"],
                    samples=clk["samples"]))
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="mixtral_prefill", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--balance-gamma", type=float, default=None,
                    help="auxiliary-loss-free balancing: nudge a selection bias by this step")
    ap.add_argument("--expert-choice", action="store_true",
                    help="expert-choice routing: each expert takes C = ceil(cf*T*k/E) tokens "
                         "(cf = 1 when the workload has none)")
    ap.add_argument("--fp8-weights", action="store_true",
                    help="8-bit (E4M3, per-row scale) routed expert weights (weight streaming)")
    ap.add_argument("--mx-weights", default=None, choices=["e4m3", "e2m1"],
                    help="block-scaled routed expert weights (one power-of-two scale per 32 "
                         "values) on the block-scaled tensor-core MMAs; activations quantized "
                         "to E4M3 blocks on the GPU")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override the workload's token count (smaller cases for profiling)")
    ap.add_argument("--experts", type=int, default=None,
                    help="override the number of routed experts (smaller profiling cases)")
    ap.add_argument("--d-ff", type=int, default=None,
                    help="override the workload's expert width d_ff (smaller cases for profiling)")
    ap.add_argument("--backward", action="store_true",
                    help="time a training step: moe_forward + moe_backward")
    ap.add_argument("--zipf", type=float, default=None,
                    help="add a Zipf(s) log-popularity bias to the router logits (skewed load)")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)          # timing rule: at least 3 warm-up steps
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    w = WORKLOADS[args.workload]
    if args.tokens is not None:
        w = w.scaled(T=args.tokens, name=f"{w.name}+T{args.tokens}")
    if args.d_ff is not None:
        w = w.scaled(d_ff=args.d_ff, name=f"{w.name}+F{args.d_ff}")
    if args.experts is not None:
        w = w.scaled(E=args.experts, name=f"{w.name}+E{args.experts}")
    if args.zipf is not None:
        w = w.scaled(zipf_s=args.zipf, name=f"{w.name}+zipf{args.zipf}")
    if args.balance_gamma is not None:
        w = w.scaled(name=f"{w.name}+balanced")
    if args.fp8_weights:
        w = w.scaled(name=f"{w.name}+fp8w")
    if args.mx_weights:
        w = w.scaled(name=f"{w.name}+mx_{args.mx_weights}")
    if args.expert_choice:
        w = w.scaled(gate="expert_choice", cf=w.cf if w.cf is not None else 1.0,
                     name=f"{w.name}+expert_choice")
    if args.impl == "reference":
        run_reference(args, w, rank)
        return
    if args.backward:
        run_train(args, w, rank, world, local_rank)
        return
    run_ours(args, w, rank, world, local_rank)


if __name__ == "__main__":
    main()
