"""GPU path vs the oracle on seeded random layers and random option mixes.

Each case draws a shape (T tokens, H and F multiples of 128, E experts, k <= min(E, 8)),
optionally a skewing logit bias that empties some experts, and a combination of the
library's options (tile shape, schedule, combine in GEMM2's epilogue, dispatch inside
GEMM1's A-operand load, grid size).  Every option must give the oracle's results within
the agreement bar: routing tables bit-exact, floats per element within 1e-2 of the
largest reference value and within 5e-3 relative L2 error.  The draws are fixed by the
seed, so a failure reproduces.  A second set draws wide expert counts (41 to 256, among
them row widths such as 48, 96 and 192 that leave value slots of the four-thread top-k
past the row's end) with small H and F.
"""
import numpy as np
import pytest
import torch

import moe_synth as S
from helpers import check_backward, check_forward, check_tables, poison, run_gpu, run_oracle, shape_inputs

pytestmark = pytest.mark.gpu

N_CASES = 32


def _draw(i):
    rng = np.random.default_rng(7000 + i)
    E = int(rng.integers(1, 41))
    k = int(rng.integers(1, min(E, 8) + 1))
    T = int(rng.choice([1, 2, 63, 64, 65, 255, 256, 257, int(rng.integers(3, 900))]))
    H = int(rng.choice([128, 256, 384, 512]))
    F = int(rng.choice([128, 256, 384, 640]))
    skew = bool(rng.random() < 0.4) and E > 2
    opts = dict(cta_pair=int(rng.integers(0, 3)), schedule=int(rng.integers(0, 3)),
                combine=int(rng.integers(0, 2)), dispatch=int(rng.choice([0, 2])),
                grid=int(rng.choice([0, 0, 2, 38, 74])))
    return S.LayerShape(T, H, F, E, k), skew, opts


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_layer_matches_oracle(i):
    from mixture_experts_layer_gb300.layer import MoELayer
    shape, skew, opts = _draw(i)
    bias = None
    if skew:
        bias = torch.zeros(shape.E)
        bias[: max(1, shape.E // 3)] = -30.0  # a third of the experts receive no token
    inp = shape_inputs(shape, 8000 + i, bias)
    layer = MoELayer(shape.T, shape.H, shape.F, shape.E, shape.k)
    poison(layer)
    run_gpu(layer, inp, opts=layer.opts(**opts))
    ref = run_oracle(inp, shape.k, shape.E)
    check_tables(layer, ref)
    check_forward(layer, ref)
    check_backward(layer, ref)


N_WIDE = 16


def _draw_wide(i):
    rng = np.random.default_rng(9000 + i)
    E = int(rng.choice([41, 44, 48, 60, 64, 80, 96, 100, 112, 128, 144, 160, 192, 200, 240, 256]))
    k = int(rng.integers(1, 9))
    T = int(rng.choice([1, 64, 65, 257, int(rng.integers(3, 700))]))
    H = int(rng.choice([128, 256]))
    F = int(rng.choice([128, 256]))
    skew = bool(rng.random() < 0.4)
    opts = dict(cta_pair=int(rng.integers(0, 3)), schedule=int(rng.integers(0, 3)),
                combine=int(rng.integers(0, 2)), dispatch=int(rng.choice([0, 2])),
                grid=int(rng.choice([0, 0, 38, 74])))
    return S.LayerShape(T, H, F, E, k), skew, opts


@pytest.mark.parametrize("i", range(N_WIDE))
def test_random_wide_layer_matches_oracle(i):
    from mixture_experts_layer_gb300.layer import MoELayer
    shape, skew, opts = _draw_wide(i)
    bias = None
    if skew:
        bias = torch.zeros(shape.E)
        bias[: shape.E // 3] = -30.0  # a third of the experts receive no token
    inp = shape_inputs(shape, 9500 + i, bias)
    layer = MoELayer(shape.T, shape.H, shape.F, shape.E, shape.k)
    poison(layer)
    run_gpu(layer, inp, opts=layer.opts(**opts))
    ref = run_oracle(inp, shape.k, shape.E)
    check_tables(layer, ref)
    check_forward(layer, ref)
    check_backward(layer, ref)
