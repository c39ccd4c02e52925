"""Per-k-block timeline of one pair-tile GroupGEMM launch (diagnosis only).

    python -m mixture_experts_layer_gb300.timeline [--config 1] [--mode 0] [--cap 512]

Builds a diagnosis copy of the library with -DMOE_TIMELINE
(libmoe_timeline.so, never loaded by the product), runs one step of the
workload, then runs the forward or backward again with the pair kernel of the
chosen GEMM mode stamping its SM's cycle counter (clock64) at five points of
its pipeline, for every k-block of every CTA (the points of one k-block are all
taken in the same CTA, so they share a clock):

    0  the producer warp found the shared-memory stage free (its TMA loads follow)
    1  the MMA warp saw the stage land (both operands of this CTA's half)
    2  the leader CTA saw the partner's stage land (relay), or the odd CTA relayed it
    3  the leader issued the k-block's MMAs and their commit
    4  (first k-block of a tile) the leader got a free accumulator

and prints a summary in SM cycles: the k-block cadence of the MMA issue
against the cycles the tensor cores need for a pair k-block (256 x 256 x 64 on
two SMs: 512 cycles), the load latency (issue to landing), and where the MMA
thread waits.  Modes: 0 fwd1, 1 fwd2,
2 dgrad2, 3 dgrad1, 4 wgrad13, 5 wgrad2.  Needs a GB300.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

MODES = {0: "gemm_fwd1_swiglu", 1: "gemm_fwd2", 2: "gemm_dgrad2_swiglu_bwd", 3: "gemm_dgrad1", 4: "gemm_wgrad13",
         5: "gemm_wgrad2"}


def _pct(v, q):
    v = sorted(v)
    return v[min(len(v) - 1, int(q * (len(v) - 1)))] if v else float("nan")


def summarise(stamps, ncta, cap, mma_cycles):
    """stamps: list of ncta*cap*5 integers (SM cycles, 0 = not recorded)."""
    cad, lat, wait_full, wait_relay, issue_gap = [], [], [], [], []
    kblocks = []
    for c in range(ncta):
        rec = [stamps[(c * cap + n) * 5:(c * cap + n) * 5 + 5] for n in range(cap)]
        n_rec = sum(1 for r in rec if r[0] or r[1] or r[3])
        kblocks.append(n_rec)
        leader = c % 2 == 0
        for n in range(1, n_rec):
            a, b = rec[n - 1], rec[n]
            if b[0] and b[1] and b[1] >= b[0]:
                lat.append(b[1] - b[0])
            if leader and a[3] and b[3]:
                cad.append(b[3] - a[3])
                if b[1]:
                    wait_full.append(max(0, b[1] - a[3]))
                if b[2] and b[1]:
                    wait_relay.append(max(0, b[2] - b[1]))
                if b[2]:
                    issue_gap.append(max(0, b[3] - b[2]))
    return {
        "ctas": ncta, "kblocks_recorded_per_cta_median": statistics.median(kblocks) if kblocks else 0,
        "unit": "SM cycles",
        "mma_issue_cadence": {"p10": _pct(cad, 0.1), "median": _pct(cad, 0.5), "p90": _pct(cad, 0.9)},
        "mma_cycles_per_kblock": mma_cycles,
        "load_latency_issue_to_land": {"p10": _pct(lat, 0.1), "median": _pct(lat, 0.5), "p90": _pct(lat, 0.9)},
        "mma_thread_wait_for_own_stage": {"median": _pct(wait_full, 0.5), "p90": _pct(wait_full, 0.9)},
        "leader_wait_for_partner_stage": {"median": _pct(wait_relay, 0.5), "p90": _pct(wait_relay, 0.9)},
        "relay_to_mma_issued": {"median": _pct(issue_gap, 0.5), "p90": _pct(issue_gap, 0.9)},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--config", type=int, default=1)
    ap.add_argument("--mode", type=int, default=0, choices=sorted(MODES))
    ap.add_argument("--cap", type=int, default=512, help="k-blocks recorded per CTA")
    args = ap.parse_args()

    from mixture_experts_layer_gb300 import build as B
    path = B.build(defines=("MOE_TIMELINE",), out=os.path.join(os.path.dirname(B.LIB), "libmoe_timeline.so"))
    import torch

    import mixture_experts_layer_gb300 as M
    import moe_synth as S
    from mixture_experts_layer_gb300.layer import MoELayer
    L = M.lib(path)
    L.moe_debug_timeline.restype = ctypes.c_int
    L.moe_debug_timeline.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int]

    shape = S.CONFIGS[args.config]
    inp = S.layer_inputs(shape, S.config_seed(args.config), device="cuda")
    layer = MoELayer(shape.T, shape.H, shape.F, shape.E, shape.k)
    fwd = args.mode in (0, 1)

    def step():
        layer.plan(inp["logits"])
        layer.forward(inp["x"], inp["W1"], inp["W3"], inp["W2"])
        layer.backward(inp["dout"], inp["W1"], inp["W3"], inp["W2"])

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    ncta = torch.cuda.get_device_properties(0).multi_processor_count
    buf = torch.zeros(ncta * args.cap * 5, dtype=torch.int64, device="cuda")
    M.check(L.moe_debug_timeline(buf.data_ptr(), args.cap, args.mode), "moe_debug_timeline")
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    layer.plan(inp["logits"])
    ev[0].record()
    if fwd:
        layer.forward(inp["x"], inp["W1"], inp["W3"], inp["W2"])
    else:
        layer.forward(inp["x"], inp["W1"], inp["W3"], inp["W2"])
        layer.backward(inp["dout"], inp["W1"], inp["W3"], inp["W2"])
    ev[1].record()
    torch.cuda.synchronize()
    M.check(L.moe_debug_timeline(None, 0, -1), "moe_debug_timeline")
    st = layer.status()
    if st[0] != 0:
        raise RuntimeError(f"device status {st}")
    # One pair k-block: 2 * 256 * 256 * 64 FLOP on two SMs at 8192 dense bf16 FLOP per SM per cycle.
    mma_cycles = 2 * 256 * 256 * 64 // (2 * 8192)
    out = summarise(buf.cpu().tolist(), ncta, args.cap, mma_cycles)
    out.update({"workload": shape.name, "mode": MODES[args.mode], "pass_ms": round(ev[0].elapsed_time(ev[1]), 4)})
    print(json.dumps(out, indent=1))


if __name__ == "__main__":
    main()
