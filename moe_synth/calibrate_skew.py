"""Find the skewed workload's bias scale BETA by bisection.

The skewed layer adds bias_e = BETA * ln(z_rank(e) / sum z) (z_i = i**-1.2) to
the router logits, plus a large negative bias on the lowest-ranked experts.
This script bisects BETA until the routed load's
maxvio = max_e n_e / (T k / E) - 1 lies in [2.9, 3.1] and prints it; the value is
stored as SKEW_BETA in moe_synth.  The loads are counted with torch.topk on
the float32 logits (the routing's ties play no part in a load count).

    python -m moe_synth.calibrate_skew
"""
import torch

import moe_synth as S


def maxvio_for(beta: float, x, Wr, shape) -> tuple[float, int]:
    lg = S.router_logits(x, Wr, S.skew_bias(S.config_seed(3), shape.E, beta))
    ids = torch.topk(lg, shape.k, dim=1).indices.reshape(-1)
    n = torch.bincount(ids, minlength=shape.E).double()
    return float(n.max() / (shape.T * shape.k / shape.E) - 1.0), int((n == 0).sum())


def main():
    sh = S.CONFIGS[3]
    seed = S.config_seed(3)
    x = S.normal_bf16(seed, S.STREAM_X, (sh.T, sh.H), 1.0)
    Wr = S.normal_bf16(seed, S.STREAM_WR, (sh.H, sh.E), 1.0 / sh.H ** 0.5)
    lo, hi = 0.0, 1.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        mv, _ = maxvio_for(mid, x, Wr, sh)
        if 2.9 <= mv <= 3.1:
            lo = hi = mid
            break
        if mv < 3.0:
            lo = mid
        else:
            hi = mid
    beta = round(lo, 3)
    mv, empty = maxvio_for(beta, x, Wr, sh)
    print(f"BETA={beta} maxvio={mv:.3f} empty_experts={empty}")


if __name__ == "__main__":
    main()
