#!/usr/bin/env python
"""Throughput of one forward+backward step of the MoE expert layer on GB300.

A step is the whole hot path over one batch of synthetic tokens: routing
(top-k, counts, offsets, stable row table), dispatch, GroupGEMM -> SwiGLU ->
GroupGEMM, gated combine, combine backward, both dgrad GroupGEMMs, the
weight-gradient Transposed GroupGEMMs and the dispatch backward.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 4] [--impl ours|reference]

Prints one JSON line (rank 0).  `value` is tokens/s over all ranks with the
inputs resident in HBM; `e2e` is the same metric through the C ABI with the
step's inputs copied from pinned host memory and its outputs copied back inside
the timed region.  Under torchrun every rank runs an independent replica of the
layer on its own tokens (weak scaling, no collective on the data path).

`--impl reference` times the CPU oracle instead (rank 0 only), on a bounded
sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s fwd+bwd; GEMM % BF16 peak; permute GB/s % HBM"
UNIT = "tokens/s"

FWD_KERNELS = ["gather_rows", "gemm_fwd1_swiglu", "gemm_fwd2", "combine"]
FWD_KERNELS_COMBINE_FUSED = ["gather_rows", "gemm_fwd1_swiglu", "gemm_fwd2_combine"]
FWD_KERNELS_FUSED = ["fused_forward", "combine"]
FWD_KERNELS_GATHER = ["gemm_fwd1_gather_swiglu", "gemm_fwd2", "combine"]
FWD_KERNELS_GATHER_COMBINE = ["gemm_fwd1_gather_swiglu", "gemm_fwd2_combine"]
BWD_KERNELS = ["combine_bwd", "gemm_dgrad2_swiglu_bwd", "gemm_dgrad1", "unpermute", "gemm_wgrad13", "gemm_wgrad2"]
BWD_KERNELS_FUSED = ["combine_bwd", "fused_backward", "unpermute"]
BWD_KERNELS_ROUTER = ["router_transpose", "combine_bwd", "gemm_dgrad2_swiglu_bwd", "gemm_dgrad1", "gemm_router_wgrad",
                      "router_reduce", "unpermute", "gemm_wgrad13", "gemm_wgrad2"]
# The non-bitwise weight-gradient variant (--wgrad-subbatches 2): each weight
# gradient GEMM runs once per token sub-batch, the second adding onto the first.
NB_TAIL = ["subbatch_rows", "gemm_wgrad13_sb0", "gemm_wgrad2_sb0", "gemm_wgrad13_sb1", "gemm_wgrad2_sb1"]
BWD_KERNELS_NB = BWD_KERNELS[:4] + NB_TAIL
BWD_KERNELS_ROUTER_NB = BWD_KERNELS_ROUTER[:7] + NB_TAIL
N_PLAN_KERNELS = 2


def work_per_kernel(T, H, F, E, k):
    """Algorithmic FLOPs and HBM bytes of one launch of each kernel (padding and re-reads not counted)."""
    R = T * k
    b = {
        "plan": 4 * T * E + 12 * T * k + 4 * R,
        "gather_rows": 2 * T * H + 2 * R * H + 4 * R,
        "gemm_fwd1_swiglu": 2 * R * H + 4 * E * H * F + 6 * R * F,
        "gemm_fwd2": 2 * R * F + 2 * E * F * H + 2 * R * H,
        "combine": 2 * R * H + 2 * T * H + 8 * R,
        "combine_bwd": 2 * T * H + 4 * R * H + 12 * R,
        "gemm_dgrad2_swiglu_bwd": 2 * R * H + 2 * E * F * H + 8 * R * F,
        "gemm_dgrad1": 4 * R * F + 4 * E * H * F + 2 * R * H,
        "gemm_wgrad13": 2 * R * H + 4 * R * F + 8 * E * H * F,
        "gemm_wgrad2": 2 * R * F + 2 * R * H + 4 * E * H * F,
        "unpermute": 2 * R * H + 2 * T * H + 4 * R,
    }
    # GEMM1 with the dispatch in its A-operand load: reads x (and row_src) instead of Xp, writes Xp.
    b["gemm_fwd1_gather_swiglu"] = 2 * T * H + 4 * R + 2 * R * H + 4 * E * H * F + 6 * R * F
    # GEMM2 with the gated combine in its epilogue: also reads the k rows of Y per token and writes out.
    b["gemm_fwd2_combine"] = b["gemm_fwd2"] + b["combine"]
    # Fused forward: reads x, row_src and every weight once; writes Xp, GU, h and Y.
    b["fused_forward"] = 2 * T * H + 4 * R + 6 * E * H * F + 2 * R * H + 6 * R * F + 2 * R * H
    # Fused backward: reads dY, GU, Xp, h and every weight once; writes dGU, dXp and dW1, dW3, dW2 (fp32).
    b["fused_backward"] = (2 * R * H + 4 * R * F + 2 * R * H + 2 * R * F + 6 * E * H * F
                           + 4 * R * F + 2 * R * H + 12 * E * H * F)
    # The router (--router): logits GEMM; Wr^T; dWr GEMM over token splits (dense
    # in the experts) and the fixed-order reduction of its partials.
    sp = router_splits(T, H, E)
    b["gemm_router_fwd"] = 2 * T * H + 2 * H * E + 4 * T * E
    b["router_transpose"] = 4 * H * E
    b["gemm_router_wgrad"] = 2 * T * H + 2 * T * E + 4 * sp * H * E
    b["router_reduce"] = 4 * sp * H * E + 4 * H * E
    # NB sub-batch passes: sub-batch 0 writes dW, sub-batch 1 reads it back and adds.
    R0 = k * ((T + 1) // 2)
    R1 = R - R0
    b["subbatch_rows"] = 12 * E
    b["gemm_wgrad13_sb0"] = 2 * R0 * H + 4 * R0 * F + 8 * E * H * F
    b["gemm_wgrad2_sb0"] = 2 * R0 * F + 2 * R0 * H + 4 * E * H * F
    b["gemm_wgrad13_sb1"] = 2 * R1 * H + 4 * R1 * F + 16 * E * H * F
    b["gemm_wgrad2_sb1"] = 2 * R1 * F + 2 * R1 * H + 8 * E * H * F
    f = {
        "gemm_router_fwd": 2 * T * H * E,
        "gemm_router_wgrad": 2 * T * H * E,
        "fused_forward": 6 * R * H * F,
        "fused_backward": 12 * R * H * F,
        "gemm_fwd1_swiglu": 4 * R * H * F,
        "gemm_fwd1_gather_swiglu": 4 * R * H * F,
        "gemm_fwd2": 2 * R * H * F,
        "gemm_fwd2_combine": 2 * R * H * F,
        "gemm_dgrad2_swiglu_bwd": 2 * R * H * F,
        "gemm_dgrad1": 4 * R * H * F,
        "gemm_wgrad13": 4 * R * H * F,
        "gemm_wgrad2": 2 * R * H * F,
        "gemm_wgrad13_sb0": 4 * R0 * H * F,
        "gemm_wgrad2_sb0": 2 * R0 * H * F,
        "gemm_wgrad13_sb1": 4 * R1 * H * F,
        "gemm_wgrad2_sb1": 2 * R1 * H * F,
    }
    return f, b


def router_splits(T, H, E):
    """Token splits of the router's dWr GEMM (the library's rule: ~304 tiles, a function of the dims)."""
    tiles = (H // 128) * ((E + 255) // 256)
    nkb = (T + 63) // 64
    sp = max(1, min(nkb, (304 + tiles - 1) // tiles))
    ks = ((nkb + sp - 1) // sp) * 64
    return max(1, (T + ks - 1) // ks)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of a kernel from the committed ncu summary, or None.

    profiles/traffic.txt holds lines `kernel source_sha dram_bytes_per_launch workload`;
    a line counts only for its own workload and while the kernel's source file
    is unchanged.
    """
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    if kernel.startswith(("gemm", "fused")):
        name = "gemm.cu"
    elif kernel.startswith("route") or kernel == "plan":
        name = "plan.cu"
    else:
        name = "rows.cu"
    src = os.path.join(ROOT, "mixture_experts_layer_gb300", "csrc", name)
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    for line in open(path):
        parts = line.split()
        if (len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel and parts[1] == sha
                and parts[3] == workload):
            return float(parts[2])
    return None


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons, pw = [], 0.0, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = max(mx, float(parts[1]))
            except ValueError:
                continue
            try:
                pw.append(float(parts[2]))
            except ValueError:
                pass
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}
        if pw:
            out["power_w"] = statistics.median(pw)
        return out


class HostBuffers:
    """Page-locked host tensors for the end-to-end copies.

    Each buffer is an anonymous mapping advised for transparent huge pages and
    then page-locked with cudaHostRegister, so a 1 GB buffer is a few large
    pages for the copy engines to translate instead of tens of thousands of
    base pages (on some machines a 1 GB upload from torch's
    pin_memory ran at 24 GB/s against 166 GB/s for a 17 MB one).  Where the
    mapping or the registration fails, torch's pin_memory is used instead."""

    def __init__(self):
        self.keep = []       # the mappings (and the ctypes views that pin their addresses)
        self.registered = []
        self.fallbacks = 0   # buffers that fell back to torch's pin_memory

    def _page(self) -> int:
        try:
            return int(open("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size").read())
        except (OSError, ValueError):
            return 2 << 20

    def empty_like(self, t):
        import ctypes
        import mmap
        import torch
        nbytes = t.numel() * t.element_size()
        try:
            align = self._page()
            mm = mmap.mmap(-1, nbytes + align, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
            if hasattr(mmap, "MADV_HUGEPAGE"):
                mm.madvise(mmap.MADV_HUGEPAGE)
            base = (ctypes.c_char * 1).from_buffer(mm)
            off = (-ctypes.addressof(base)) % align
            h = torch.frombuffer(mm, dtype=t.dtype, count=t.numel(), offset=off).view(t.shape)
            h.zero_()  # touch every page before it is locked
            rc = torch.cuda.cudart().cudaHostRegister(h.data_ptr(), nbytes, 0)
            if int(rc) != 0:
                raise RuntimeError(f"cudaHostRegister: {rc}")
            self.keep.append((mm, base))
            self.registered.append(h.data_ptr())
            return h
        except (OSError, ValueError, RuntimeError, AttributeError):
            self.fallbacks += 1
            return torch.empty(t.shape, dtype=t.dtype).pin_memory()

    def copy_of(self, t):
        h = self.empty_like(t)
        h.copy_(t)
        return h

    def close(self):
        import torch
        for ptr in self.registered:
            torch.cuda.cudart().cudaHostUnregister(ptr)
        self.registered.clear()


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def max_over_ranks(v: float, world: int) -> float:
    if world <= 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# CPU oracle leg
# ---------------------------------------------------------------------------
# Workloads whose float64 weights and weight gradients (6 E H F doubles) fit in
# this much host memory run the oracle's whole step on a prefix of the tokens;
# larger ones (large-expert, skewed, long-sequence) run its sampled form.
ORACLE_FULL_BYTES = 12e9


class OracleWorkload:
    """The workload's inputs (generated on the GPU when there is one) and the
    oracle's routing of all of its tokens.  Inputs reach the oracle as float64
    arrays through the accessors below, whose conversion time is recorded in
    `conv_s` so the timed oracle work can leave it out."""

    def __init__(self, shape, seed):
        import torch

        import moe_synth as S
        self.shape = shape
        self.dev = "cuda" if torch.cuda.is_available() else "cpu"
        self.inp = S.layer_inputs(shape, seed, device=self.dev)
        self.logits = self.inp["logits"].cpu().numpy()
        self.conv_s = 0.0
        self.full = 6.0 * shape.E * shape.H * shape.F * 8 <= ORACLE_FULL_BYTES
        if self.full:
            self.W = tuple(self._f64(self.inp[n]) for n in ("W1", "W3", "W2"))

    def _f64(self, t):
        import torch
        t0 = time.perf_counter()
        a = t.detach().to("cpu", torch.float64).numpy()
        self.conv_s += time.perf_counter() - t0
        return a

    def weights(self, e):
        return tuple(self._f64(self.inp[n][e]) for n in ("W1", "W3", "W2"))

    def rows(self, name, toks):
        import torch
        return self._f64(self.inp[name][torch.as_tensor(toks, device=self.dev)])

    def close(self):
        del self.inp
        import torch
        if torch.cuda.is_available():
            torch.cuda.empty_cache()


def oracle_prefix_step(ow, T_s):
    """The oracle's whole step (plan, forward, backward with every weight
    gradient) on the first T_s tokens; returns the oracle's seconds."""
    import oracle.moe_oracle as O
    sh = ow.shape
    x = ow._f64(ow.inp["x"][:T_s])
    dout = ow._f64(ow.inp["dout"][:T_s])
    t0 = time.perf_counter()
    O.layer_step(x, ow.logits[:T_s], dout, ow.W, sh.k, sh.E, mirror=True)
    return time.perf_counter() - t0


def oracle_sampled_step(ow, toks, experts):
    """The oracle's sampled step: routing of all T tokens, out/dx/dgate of the
    tokens `toks` from their own k rows, and the full weight gradients of the
    experts `experts` over all of their rows.  Returns (oracle seconds, GEMM
    FLOPs of the sample); input conversion to float64 is not counted."""
    import oracle.moe_oracle as O
    sh = ow.shape
    c0 = ow.conv_s
    t0 = time.perf_counter()
    ids, w = O.route(ow.logits, sh.k)
    perm = O.permutation(ids, sh.E)
    xr, dr = ow.rows("x", toks), ow.rows("dout", toks)
    O.token_rows(toks, xr, dr, ids, w, ow.weights, mirror=True)
    rows = 0
    for e in experts:
        O.expert_grads(e, lambda t: ow.rows("x", t), lambda t: ow.rows("dout", t), ids, w, perm, ow.weights,
                       mirror=True)
        rows += int(perm.counts[e])
    t = time.perf_counter() - t0 - (ow.conv_s - c0)
    # token_rows: forward and dgrad of the tokens' k rows (12 R H F); expert_grads:
    # forward, dgrad and weight gradients of each expert's rows (18 n_e H F).
    flops = 12 * len(toks) * sh.k * sh.H * sh.F + 18 * rows * sh.H * sh.F
    return t, flops


def oracle_threads():
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(v):
            try:
                return int(os.environ[v])
            except ValueError:
                pass
    return os.cpu_count() or 1


def _sample_tokens(shape, n, seed):
    import numpy as np
    rng = np.random.default_rng(seed)
    return sorted(rng.choice(shape.T, size=min(n, shape.T), replace=False).tolist())


def oracle_rate(ow, budget_s, steps=1, warm=0):
    """Times `steps` oracle steps, each a bounded sample of about budget_s seconds.

    Returns (tokens/s, seconds per step, description of the sample).  Small
    workloads run the whole step on a token prefix (tokens/s = prefix / time);
    large ones run the sampled step, whose tokens/s is the step's T scaled by
    the sample's share of the step's GEMM FLOPs (18 T k H F)."""
    import numpy as np
    sh = ow.shape
    if ow.full:
        # A fixed cost plus a part linear in the tokens, fitted from two probes.
        t_a = oracle_prefix_step(ow, 16)
        t_b = oracle_prefix_step(ow, 64)
        slope = max((t_b - t_a) / 48.0, 1e-9)
        T_s = int(max(16, min(sh.T, 64 + (budget_s - t_b) / slope)))
        for _ in range(warm):
            oracle_prefix_step(ow, T_s)
        t = sum(oracle_prefix_step(ow, T_s) for _ in range(steps))
        return (T_s * steps / t, t / steps,
                f"first {T_s} of {sh.T} tokens per step: plan, forward and backward (every weight gradient over "
                f"those tokens' rows), numpy float64 oracle")
    step_flops = 18.0 * sh.T * sh.k * sh.H * sh.F
    counts = np.bincount(np.asarray(ow.logits.argmax(axis=1)), minlength=sh.E)  # probe only: an expert order
    order = [int(e) for e in np.argsort(-counts, kind="stable")]
    # Probe: 32 tokens and one expert, then 96 tokens and the same expert.
    t_a, f_a = oracle_sampled_step(ow, _sample_tokens(sh, 32, 1), order[:1])
    t_b, f_b = oracle_sampled_step(ow, _sample_tokens(sh, 96, 2), order[:1])
    slope = max((t_b - t_a) / 64.0, 1e-9)
    n_tok = int(max(32, min(sh.T, 96 + (budget_s - t_b) / slope)))
    for i in range(warm):
        oracle_sampled_step(ow, _sample_tokens(sh, n_tok, 100 + i), order[i % len(order): i % len(order) + 1])
    t = fl = 0.0
    for i in range(steps):
        dt, df = oracle_sampled_step(ow, _sample_tokens(sh, n_tok, 200 + i),
                                     order[(i + 1) % len(order): (i + 1) % len(order) + 1])
        t += dt
        fl += df
    value = sh.T * (fl / step_flops) / t
    return (value, t / steps,
            f"sampled step: routing of all {sh.T} tokens, out/dx/dgate of {n_tok} seeded tokens from their own "
            f"{sh.k} rows, and the full weight gradients of one expert per step (forward, dgrad and weight "
            f"gradients over all its rows); tokens/s = T x (sample GEMM FLOPs / step GEMM FLOPs 18 T k H F) / "
            f"oracle seconds; numpy float64 oracle, float64 input conversion not timed")


def run_reference(args):
    import moe_synth as S
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    shape = S.CONFIGS[args.config]
    steps, warm = args.steps, args.warmup
    # Size the sample so the whole run stays within a few minutes.
    budget = min(8.0, 150.0 / max(1, steps + warm))
    ow = OracleWorkload(shape, S.config_seed(args.config))
    value, sec, sample = oracle_rate(ow, budget, steps=steps, warm=warm)
    ow.close()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": warm, "ms_per_step": 1000.0 * sec, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(shape, args.config),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(shape, idx):
    return {"workload": f"{shape.name} MoE expert layer fwd+bwd, T={shape.T} H={shape.H} F={shape.F} "
                        f"E={shape.E} k={shape.k}, bf16 in / fp32 accumulate, all experts on one GPU",
            "config_index": idx, "T": shape.T, "H": shape.H, "F": shape.F, "E": shape.E, "k": shape.k,
            "l2": "inputs larger than L2 (expert weights alone exceed the 129 MB L2)"}


# ---------------------------------------------------------------------------
# GPU leg
# ---------------------------------------------------------------------------
def run_ours(args):
    import torch

    import moe_synth as S
    import mixture_experts_layer_gb300 as M
    from mixture_experts_layer_gb300.layer import MoELayer

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    shape = S.CONFIGS[args.config]
    if args.shape:
        if not args.profile:
            raise SystemExit("--shape is for profiler captures (with --profile)")
        T, H, F, E, k = (int(v) for v in args.shape.split(","))
        shape = S.LayerShape(T, H, F, E, k, f"shape-T{T}-H{H}-F{F}-E{E}-k{k}")
    T, H, F, E, k = shape.T, shape.H, shape.F, shape.E, shape.k
    seed = S.config_seed(args.config) + 1000 * rank  # each replica its own tokens
    M.lib()
    if args.profile and args.part == "plan":
        # Routing only: the logits and the plan's tables are all that is allocated.
        lg = S.layer_inputs(shape, seed, device=dev, with_weights=False)["logits"]
        layer = MoELayer(T, H, F, E, k, device=dev, plan_only=True, pad=args.pad)
        for _ in range(args.warmup + 1):
            layer.plan(lg)
        torch.cuda.synchronize()
        st = layer.status()
        if st[0] != 0:
            raise RuntimeError(f"device status {st}")
        if rank == 0:
            print(json.dumps({"profile_step": "done", "part": "plan", "config": workload_config(shape, args.config),
                              "kernels_per_step": N_PLAN_KERNELS}), flush=True)
        return
    inp = S.layer_inputs(shape, seed, device=dev)
    layer = MoELayer(T, H, F, E, k, device=dev, with_router=args.router, pad=args.pad)
    stream = torch.cuda.current_stream(dev)
    gather_fused = args.dispatch == 2 and args.schedule == 0 and args.cta_pair != 1 and args.pad <= 1
    if gather_fused:
        fwd_names = FWD_KERNELS_GATHER_COMBINE if args.combine == 1 else FWD_KERNELS_GATHER
    else:
        fwd_names = (FWD_KERNELS_FUSED if args.schedule in (1, 2)
                     else FWD_KERNELS_COMBINE_FUSED if args.combine == 1 else FWD_KERNELS)
    nb_variant = args.wgrad_subbatches == 2
    if nb_variant and args.schedule == 2:
        raise SystemExit("--wgrad-subbatches 2 runs with schedules 0 and 1")
    bwd_names = BWD_KERNELS_FUSED if args.schedule == 2 else BWD_KERNELS_NB if nb_variant else BWD_KERNELS
    if args.router:
        if args.schedule == 2:
            raise SystemExit("--router is measured with schedules 0 and 1")
        bwd_names = BWD_KERNELS_ROUTER_NB if nb_variant else BWD_KERNELS_ROUTER
    nf, nb = len(fwd_names), len(bwd_names)
    router_arg = (inp["x"], inp["Wr"]) if args.router else None
    opt_kw = dict(schedule=args.schedule, cta_pair=args.cta_pair, combine=args.combine,
                  wgrad_subbatches=args.wgrad_subbatches, dispatch=args.dispatch, grid=args.grid)
    base_opts = layer.opts(**opt_kw)

    def step(opts_f=None, opts_b=None, ev_plan=None, opts_r=None):
        opts_f = opts_f if opts_f is not None else base_opts
        opts_b = opts_b if opts_b is not None else base_opts
        if args.router:
            layer.router_forward(inp["x"], inp["Wr"], opts=opts_r if opts_r is not None else base_opts)
        if ev_plan is not None:
            ev_plan[0].record(stream)
        layer.plan(layer.logits if args.router else inp["logits"])
        if ev_plan is not None:
            ev_plan[1].record(stream)
        layer.forward(inp["x"], inp["W1"], inp["W3"], inp["W2"], opts=opts_f)
        layer.backward(inp["dout"], inp["W1"], inp["W3"], inp["W2"], opts=opts_b, router=router_arg)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = layer.status()
    if st[0] != 0:
        raise RuntimeError(f"device status {st}")
    if args.profile:
        # One more step and nothing else: the launch sequence a profiler captures.
        step()
        torch.cuda.synchronize()
        st = layer.status()
        if st[0] != 0:
            raise RuntimeError(f"device status {st}")
        if rank == 0:
            print(json.dumps({"profile_step": "done", "config": workload_config(shape, args.config),
                              "kernels_per_step": N_PLAN_KERNELS + nf + nb}), flush=True)
        return

    # Per-kernel events of every timed step (recorded on the launching stream).
    evs_f = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * nf)] for _ in range(args.steps)]
    evs_b = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * nb)] for _ in range(args.steps)]
    evs_p = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    evs_r = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for e in [e for row in evs_f + evs_b + evs_p + evs_r for e in row]:
        e.record(stream)  # torch creates the CUDA event on first record
    torch.cuda.synchronize()
    opts_f = []
    keep = []
    for e in evs_f:
        o = layer.opts(events=e, **opt_kw)
        keep.append(layer._ev_keep)
        opts_f.append(o)
    opts_b = []
    for e in evs_b:
        o = layer.opts(events=e, **opt_kw)
        keep.append(layer._ev_keep)
        opts_b.append(o)
    opts_r = []
    for e in evs_r:
        o = layer.opts(events=e, **opt_kw)
        keep.append(layer._ev_keep)
        opts_r.append(o)

    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    # Timed region: K whole steps, nothing but the layer's own launches in it.  By
    # default the step's launches (plan, forward, backward: all stream-ordered, no
    # host synchronisation) are captured once in a CUDA graph and the graph is
    # replayed K times, which removes the host launch gaps between the kernels.
    graph = None
    if not args.no_graph:
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        l0 = M.moe_launch_count()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            step()
        per_step_launches = M.moe_launch_count() - l0
        stream.wait_stream(side)
        torch.cuda.synchronize()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
    l0 = M.moe_launch_count()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        if graph is not None:
            graph.replay()
        else:
            step()
    t_end.record(stream)
    torch.cuda.synchronize()
    launches = M.moe_launch_count() - l0 if graph is None else per_step_launches * args.steps
    barrier(world)
    ms_local = t_start.elapsed_time(t_end)
    ms_total = max_over_ranks(ms_local, world)
    # Second timed pass of K steps with a CUDA event pair around every kernel (on the
    # launching stream) for the per-kernel durations; the events themselves cost a
    # few percent of a short step, so the headline value comes from the pass above.
    k_start = torch.cuda.Event(enable_timing=True)
    k_end = torch.cuda.Event(enable_timing=True)
    k_start.record(stream)
    for i in range(args.steps):
        step(opts_f[i], opts_b[i], evs_p[i], opts_r[i])
    k_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    ms_events = k_start.elapsed_time(k_end) / args.steps
    st = layer.status()
    if st[0] != 0:
        raise RuntimeError(f"device status {st}")
    # Load imbalance of the routed batch: the busiest expert's rows over the mean, minus one.
    maxvio = float(layer.counts.max().item()) / (T * k / E) - 1.0

    # Per-kernel average durations.
    names = (["gemm_router_fwd"] if args.router else []) + ["plan"] + fwd_names + bwd_names
    per = {n: 0.0 for n in names}
    for i in range(args.steps):
        if args.router:
            per["gemm_router_fwd"] += evs_r[i][0].elapsed_time(evs_r[i][1])
        per["plan"] += evs_p[i][0].elapsed_time(evs_p[i][1])
        for j, n in enumerate(fwd_names):
            per[n] += evs_f[i][2 * j].elapsed_time(evs_f[i][2 * j + 1])
        for j, n in enumerate(bwd_names):
            per[n] += evs_b[i][2 * j].elapsed_time(evs_b[i][2 * j + 1])
    per = {n: v / args.steps for n, v in per.items()}
    flops, bytes_ = work_per_kernel(T, H, F, E, k)
    peaks = load_peaks()
    long_region = ms_total > 1000.0
    tc_peak = peaks["bf16_tflops_sustained"] if long_region else peaks["bf16_tflops"]
    kern = {}
    for n, ms in per.items():
        ent = {"ms": round(ms, 4), "gbs": round(bytes_[n] / (ms * 1e-3) / 1e9, 1),
               "hbm_frac": round(bytes_[n] / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 3)}
        if n in flops:
            tf = flops[n] / (ms * 1e-3) / 1e12
            ent["tflops"] = round(tf, 1)
            ent["tensor_frac"] = round(tf / tc_peak, 3)
        kern[n] = ent
    dom = max(per, key=per.get)
    # Judge the dominant kernel against its binding roof: the tensor-core peak
    # when its FLOPs take longer at peak than its algorithmic bytes at the
    # copy bandwidth, HBM otherwise.
    t_tc = flops.get(dom, 0) / (tc_peak * 1e12)
    t_hbm = bytes_[dom] / (peaks["hbm_gbs"] * 1e9)
    if dom in flops and t_tc >= t_hbm:
        ach = flops[dom] / (per[dom] * 1e-3) / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": round(ach, 1), "peak": tc_peak, "unit": "TFLOP/s",
                "frac": round(ach / tc_peak, 4), "traffic": profiled_traffic(dom, shape.name),
                "peak_kind": ("sustained" if long_region else "burst") + f" bf16 of {peaks['source']}"}
    else:
        ach = bytes_[dom] / (per[dom] * 1e-3) / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(ach / peaks["hbm_gbs"], 4), "traffic": profiled_traffic(dom, shape.name),
                "peak_kind": f"copy bandwidth of {peaks['source']}"}
    roof["algorithmic_per_launch"] = flops[dom] if roof["bound"] == "tensor" else bytes_[dom]
    for n, ent in kern.items():
        tt = flops.get(n, 0) / (tc_peak * 1e12)
        th = bytes_[n] / (peaks["hbm_gbs"] * 1e9)
        ent["bound"] = "tensor" if tt >= th else "hbm"
        ent["roof_frac"] = round(max(tt, th) / (per[n] * 1e-3), 3)

    # End-to-end through the C ABI: every step copies its inputs from pinned host
    # memory and reads its results (out, dx) back to pinned host memory.  The copies
    # run on copy streams, double-buffered, the way a training loop overlaps its
    # data movement with compute: step i+1's inputs are uploaded while step i
    # computes, and step i's results (written by the layer straight into buffer set
    # i mod 2: the C ABI takes out and dx per call) download while step i+1 computes.
    # The timed region ends when the last download is done.
    hb = HostBuffers()
    h_x = hb.copy_of(inp["x"])
    h_lg = hb.copy_of(inp["logits"])
    h_do = hb.copy_of(inp["dout"])
    h_out = hb.empty_like(inp["x"])
    h_dx = hb.empty_like(inp["x"])
    d_in = [(torch.empty_like(inp["x"]), torch.empty_like(inp["logits"]), torch.empty_like(inp["dout"]))
            for _ in range(2)]
    d_res = [(torch.empty_like(layer.out), torch.empty_like(layer.dx)) for _ in range(2)]  # out, dx per buffer set
    # NS upload and NS download streams: every tensor moves as NS row slices, one per
    # stream, so the copies spread over several copy engines each way.
    NS = 4
    ups = [torch.cuda.Stream(dev) for _ in range(NS)]
    downs = [torch.cuda.Stream(dev) for _ in range(NS)]
    bounds = [T * q // NS for q in range(NS + 1)]
    rows = [(bounds[q], bounds[q + 1]) for q in range(NS)]  # token rows of slice q
    ev_in = [[torch.cuda.Event() for _ in range(NS)] for _ in range(2)]   # slice q of inputs j uploaded
    ev_used = [torch.cuda.Event() for _ in range(2)]                       # compute done with inputs j
    ev_staged = [torch.cuda.Event() for _ in range(2)]                     # results j written
    ev_out = [[torch.cuda.Event() for _ in range(NS)] for _ in range(2)]  # slice q of results j downloaded
    for j in range(2):
        ev_used[j].record(stream)
        for q in range(NS):
            ev_out[j][q].record(stream)

    # With `windows` set, every copy slice is bracketed by timing events, so the timed
    # region also reports the copy rates it got (other work on the machine can slow
    # host memory down while the region runs).
    windows = None

    def bracket(st):
        if windows is None:
            return None
        a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_ev.record(st)
        return a_ev, b_ev

    def upload(j):
        d_x, d_lg, d_do = d_in[j]
        evs = []
        for q, st in enumerate(ups):
            a_, b_ = rows[q]
            st.wait_event(ev_used[j])
            br = bracket(st)
            with torch.cuda.stream(st):
                d_x[a_:b_].copy_(h_x[a_:b_], non_blocking=True)
                d_do[a_:b_].copy_(h_do[a_:b_], non_blocking=True)
                if not args.router:
                    d_lg[a_:b_].copy_(h_lg[a_:b_], non_blocking=True)
            if br is not None:
                br[1].record(st)
                evs.append(br)
            ev_in[j][q].record(st)
        if windows is not None:
            windows["h2d"].append(evs)

    def download(j):
        evs = []
        for q, st in enumerate(downs):
            a_, b_ = rows[q]
            st.wait_event(ev_staged[j])
            br = bracket(st)
            with torch.cuda.stream(st):
                h_out[a_:b_].copy_(d_res[j][0][a_:b_], non_blocking=True)
                h_dx[a_:b_].copy_(d_res[j][1][a_:b_], non_blocking=True)
            if br is not None:
                br[1].record(st)
                evs.append(br)
            ev_out[j][q].record(st)
        if windows is not None:
            windows["d2h"].append(evs)

    def compute(j):
        d_x, d_lg, d_do = d_in[j]
        if args.router:
            layer.router_forward(d_x, inp["Wr"], opts=base_opts)
        layer.plan(layer.logits if args.router else d_lg)
        # out and dx go straight to buffer set j (the ABI takes them per call), which is
        # downloaded while the next step computes into set j ^ 1.
        layer.forward(d_x, inp["W1"], inp["W3"], inp["W2"], opts=base_opts, out=d_res[j][0])
        layer.backward(d_do, inp["W1"], inp["W3"], inp["W2"], opts=base_opts,
                       router=(d_x, inp["Wr"]) if args.router else None, dx=d_res[j][1])

    # One graph per input/staging buffer set, as in the device-timed region.
    e2e_graphs = [None, None]
    if graph is not None:
        side = torch.cuda.Stream(dev)
        for j in range(2):
            side.wait_stream(stream)
            e2e_graphs[j] = torch.cuda.CUDAGraph()
            with torch.cuda.graph(e2e_graphs[j], stream=side):
                compute(j)
            stream.wait_stream(side)
        torch.cuda.synchronize()

    def e2e_step(i, last):
        j = i & 1
        for q in range(NS):
            stream.wait_event(ev_in[j][q])
            stream.wait_event(ev_out[j][q])  # results j downloaded (two steps ago)
        if e2e_graphs[j] is not None:
            e2e_graphs[j].replay()
        else:
            compute(j)
        ev_used[j].record(stream)
        ev_staged[j].record(stream)
        if not last:
            upload(j ^ 1)
        download(j)

    def e2e_run(n):
        upload(0)
        for i in range(n):
            e2e_step(i, i == n - 1)
        for q in range(NS):
            stream.wait_event(ev_out[(n - 1) & 1][q])

    e2e_run(max(3, args.warmup))
    torch.cuda.synchronize()
    # This machine's host copy rates for one x-sized tensor each way, on one stream
    # and as NS row slices on NS streams: a reference for the end-to-end number,
    # whose copies must hide behind the step.
    probe = {}
    for name, dst, src in (("h2d", d_in[0][0], h_x), ("d2h", h_out, d_res[0][0])):
        for nst in (1, NS):
            c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            c0.record(stream)
            for q in range(nst):
                st = (ups if name == "h2d" else downs)[q]
                st.wait_event(c0)
                a_, b_ = (T * q // nst, T * (q + 1) // nst)
                with torch.cuda.stream(st):
                    dst[a_:b_].copy_(src[a_:b_], non_blocking=True)
                stream.wait_stream(st)
            c1.record(stream)
            c1.synchronize()
            key = name if nst == 1 else f"{name}_{nst}_streams"
            probe[key] = round(src.numel() * src.element_size() / (c0.elapsed_time(c1) * 1e-3) / 1e9, 1)
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e2e_clocks = ClockSampler(local)
    e2e_clocks.start()
    time.sleep(0.3)
    e0.record(stream)
    for c in ups + downs:
        c.wait_event(e0)
    windows = {"h2d": [], "d2h": []}
    e2e_run(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_clk = e2e_clocks.stop()
    # Each step's upload (download) window: first slice start to last slice end.
    in_region = {}
    for name, nbytes in (("h2d", (h_x.numel() + h_do.numel()) * 2 + (0 if args.router else h_lg.numel() * 4)),
                         ("d2h", (h_out.numel() + h_dx.numel()) * 2)):
        spans = []
        for evs in windows[name]:
            t0_ = min(range(len(evs)), key=lambda q: e0.elapsed_time(evs[q][0]))
            start = e0.elapsed_time(evs[t0_][0])
            end = max(e0.elapsed_time(b_) for _, b_ in evs)
            spans.append(end - start)
        if spans:
            in_region[name] = round(nbytes / (statistics.median(spans) * 1e-3) / 1e9, 1)
            in_region[name + "_ms_median"] = round(statistics.median(spans), 3)
    windows = None
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    h2d = h_x.numel() * 2 + (0 if args.router else h_lg.numel() * 4) + h_do.numel() * 2
    d2h = h_out.numel() * 2 + h_dx.numel() * 2

    ms_step = ms_total / args.steps
    value = world * T * args.steps / (ms_total * 1e-3)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(workload_config(shape, args.config), parallelism=f"replicas x{world}" if world > 1 else "1 GPU",
                       grid=args.grid if args.grid else "one CTA per SM",
                       schedule={0: "one persistent launch per phase", 1: "fused persistent forward, per-GEMM backward",
                                 2: "fused forward, fused backward"}[args.schedule],
                       gemm_tiles={0: "two-CTA 256x256 pair tiles (cta_group::2); dgrad2 on 128x256 single-CTA "
                                      "tiles unless experts average >= 2048 rows",
                                   1: "single-CTA 128x256 tiles (cta_group::1)",
                                   2: "two-CTA 256x256 pair tiles (cta_group::2)"}[args.cta_pair],
                       router="on the path: logits = x Wr on the GPU, gradient through the gating (dlogits, dWr, "
                              "dx share)" if args.router else "off (logits given; the pages time the layer "
                                                               "excluding gating)",
                       dispatch=("inside GEMM1's A-operand load (cp.async row copies, Xp stored from the stages)"
                                 if gather_fused else "its own kernel" if args.schedule == 0
                                 else "gather tasks of the fused forward"),
                       rows=("padding-free GroupGEMM (R = T*k rows)" if args.pad <= 1 else
                             f"static-shape: each expert's rows padded to a multiple of {args.pad} "
                             f"({int(layer.offsets[-1].item())} rows in use of {layer.R}; the algorithmic "
                             "work counts the T*k routed rows)"),
                       weight_gradients="non-bitwise: two token sub-batches, the second added onto the first"
                       if args.wgrad_subbatches == 2 else "bitwise-reproducible: one reduction chain per tile",
                       maxvio=round(maxvio, 4)),
        "roofline": roof,
        "e2e": {"value": round(world * T * args.steps / (e2e_ms * 1e-3), 1), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "copies": f"pinned host <-> device as {NS} row slices on {NS} upload and {NS} download streams, "
                          "double-buffered: step i+1's upload and step i's download overlap compute",
                "launch": "CUDA graph per buffer set" if graph is not None else "eager launches",
                "host_buffers": ("anonymous mappings advised for transparent huge pages, page-locked with "
                                 "cudaHostRegister") if hb.fallbacks == 0 else "torch pin_memory (in part)",
                "host_copy_gbs": probe, "copy_gbs_in_region": in_region, "clocks": e2e_clk},
        "gpu_launches": int(launches),
        "kernel_timing": {"how": "CUDA event pair around each kernel on its launching stream, second timed pass of "
                                 "the same K steps (eager launches)", "ms_per_step_with_events": round(ms_events, 4)},
        "launch": ("CUDA graph of one step (plan + forward + backward) replayed K times" if graph is not None
                   else "eager launches"),
        "clocks": clk,
        "kernels": kern,
        "step_gemm_tflops": round((18 * T * k * H * F + (4 * T * H * E if args.router else 0))
                                  / (ms_step * 1e-3) / 1e12, 1),
    }

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(shape, args.config)
    extra = [int(c) for c in args.also.split(",") if c.strip()] if args.also else []
    if world == 1 and extra and not args.router and args.pad <= 1:
        # Free this workload's buffers, then time the other workloads the same way.
        del layer, inp, graph, e2e_graphs, d_in, d_res, h_x, h_lg, h_do, h_out, h_dx, opts_f, opts_b, opts_r, keep
        hb.close()
        import gc
        gc.collect()
        torch.cuda.empty_cache()
        line["other_workloads"] = {S.CONFIGS[c].name: time_other_workload(c, args, dev, opt_kw) for c in extra}
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def time_other_workload(idx, args, dev, opt_kw):
    """ms/step, tokens/s and per-kernel rates of another workload, timed as the headline one
    (a CUDA graph of one step replayed K times, then a pass with an event pair around every
    kernel), for the record beside the headline line."""
    import torch

    import moe_synth as S
    from mixture_experts_layer_gb300.layer import MoELayer
    shape = S.CONFIGS[idx]
    T, H, F, E, k = shape.T, shape.H, shape.F, shape.E, shape.k
    inp = S.layer_inputs(shape, S.config_seed(idx), device=dev)
    layer = MoELayer(T, H, F, E, k, device=dev)
    stream = torch.cuda.current_stream(dev)
    opts = layer.opts(**opt_kw)

    def step(of=None, ob=None, ep=None):
        if ep is not None:
            ep[0].record(stream)
        layer.plan(inp["logits"])
        if ep is not None:
            ep[1].record(stream)
        layer.forward(inp["x"], inp["W1"], inp["W3"], inp["W2"], opts=of or opts)
        layer.backward(inp["dout"], inp["W1"], inp["W3"], inp["W2"], opts=ob or opts)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        step()
    stream.wait_stream(side)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    fwd_names, bwd_names = FWD_KERNELS, BWD_KERNELS
    evf = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * len(fwd_names))] for _ in range(args.steps)]
    evb = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * len(bwd_names))] for _ in range(args.steps)]
    evp = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for e in [e for row in evf + evb + evp for e in row]:
        e.record(stream)
    torch.cuda.synchronize()
    keep, of, ob = [], [], []
    for i in range(args.steps):
        of.append(layer.opts(events=evf[i], **opt_kw))
        keep.append(layer._ev_keep)
        ob.append(layer.opts(events=evb[i], **opt_kw))
        keep.append(layer._ev_keep)
    for i in range(args.steps):
        step(of[i], ob[i], evp[i])
    torch.cuda.synchronize()
    clk = clocks.stop()
    st = layer.status()
    if st[0] != 0:
        raise RuntimeError(f"device status {st}")
    per = {"plan": sum(evp[i][0].elapsed_time(evp[i][1]) for i in range(args.steps)) / args.steps}
    for names, evs in ((fwd_names, evf), (bwd_names, evb)):
        for j, n in enumerate(names):
            per[n] = sum(evs[i][2 * j].elapsed_time(evs[i][2 * j + 1]) for i in range(args.steps)) / args.steps
    flops, bytes_ = work_per_kernel(T, H, F, E, k)
    peaks = load_peaks()
    kern = {}
    for n, t in per.items():
        ent = {"ms": round(t, 4), "gbs": round(bytes_[n] / (t * 1e-3) / 1e9, 1),
               "hbm_frac": round(bytes_[n] / (t * 1e-3) / 1e9 / peaks["hbm_gbs"], 3)}
        if n in flops:
            tf = flops[n] / (t * 1e-3) / 1e12
            ent["tflops"] = round(tf, 1)
            ent["tensor_frac"] = round(tf / peaks["bf16_tflops"], 3)
        tt = flops.get(n, 0) / (peaks["bf16_tflops"] * 1e12)
        th = bytes_[n] / (peaks["hbm_gbs"] * 1e9)
        ent["bound"] = "tensor" if tt >= th else "hbm"
        ent["roof_frac"] = round(max(tt, th) / (t * 1e-3), 3)
        kern[n] = ent
    maxvio = float(layer.counts.max().item()) / (T * k / E) - 1.0
    out = {"workload": workload_config(shape, idx)["workload"], "ms_per_step": round(ms, 4),
           "value": round(T / (ms * 1e-3), 1), "unit": UNIT, "steps": args.steps,
           "timing": "CUDA graph of one step replayed K times; per-kernel times from an event pass",
           "tensor_peak": "burst bf16 of " + peaks["source"], "maxvio": round(maxvio, 4), "clocks": clk,
           "kernels": kern}
    del layer, inp, graph
    import gc
    gc.collect()
    torch.cuda.empty_cache()
    return out


def cpu_baseline(shape, idx):
    """The oracle, as it stands, on a bounded sample of the same workload (~10-30 s)."""
    import moe_synth as S
    ow = OracleWorkload(shape, S.config_seed(idx))
    value, sec, sample = oracle_rate(ow, 12.0)
    ow.close()
    return {"value": round(value, 2), "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
            "sample": f"{sample}; {sec:.1f} s"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=4,
                    help="workload index: 0 tiny, 1 fine-grained, 2 large-expert, 3 skewed, 4 long-sequence "
                         "(default: the largest that fits one GPU)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--also", default=None,
                    help="comma-separated workload indices timed after the headline one and reported under "
                         "other_workloads (default with the long-sequence headline: 2,3, the large-expert and "
                         "skewed workloads; '' for none)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--schedule", type=int, default=0, choices=[0, 1, 2],
                    help="0: one persistent launch per phase; 1: fused persistent forward, one persistent "
                         "kernel per backward GEMM; 2: fused forward and fused backward")
    ap.add_argument("--cta-pair", type=int, default=0, choices=[0, 1, 2],
                    help="grouped GEMMs that run as their own kernels: 0 library default (pair tiles but for "
                         "dgrad2), 1 one CTA per tile, 2 two-CTA pair tiles")
    ap.add_argument("--grid", type=int, default=0,
                    help="CTAs of the persistent kernels (0: one per SM); results do not depend on it")
    ap.add_argument("--combine", type=int, default=0, choices=[0, 1],
                    help="schedule 0: 0 a separate gated-combine kernel, 1 the combine in GEMM2's epilogue")
    ap.add_argument("--dispatch", type=int, default=0, choices=[0, 1, 2],
                    help="schedule 0: 0 library default, 1 a dispatch kernel, 2 the dispatch inside GEMM1's "
                         "A-operand load (cp.async row copies)")
    ap.add_argument("--wgrad-subbatches", type=int, default=0, choices=[0, 2],
                    help="0: bitwise-reproducible weight gradients (one reduction chain); 2: the non-bitwise "
                         "variant (two token sub-batches, the second added onto the first)")
    ap.add_argument("--pad", type=int, default=0,
                    help="token padding granule: 0 padding-free (default); P >= 2 pads every expert's rows to a "
                         "multiple of P (static-shape variant)")
    ap.add_argument("--router", action="store_true",
                    help="put the router on the timed path: logits = x Wr on the GPU and its backward")
    ap.add_argument("--no-graph", action="store_true",
                    help="time the steps as eager launches instead of replaying a CUDA graph of one step")
    ap.add_argument("--profile", action="store_true",
                    help="run the warm-up steps and one more step only (for ncu captures)")
    ap.add_argument("--shape", default="",
                    help="with --profile: a layer shape T,H,F,E,k of its own instead of a workload (small "
                         "profiler captures with a workload's expert shapes)")
    ap.add_argument("--part", default="step", choices=["step", "plan"],
                    help="with --profile: the whole step, or the routing kernels alone (plan buffers only)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.also is None:
        args.also = "2,3" if args.config == 4 and not args.profile else ""
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
