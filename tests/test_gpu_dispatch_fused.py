"""The dispatch inside GEMM1's A-operand load (moe_opts.dispatch = 2): the
producer warp copies each tile's rows of x into the swizzled stage with 16-byte
cp.async copies, and the first N tile of each row block stores them to Xp for
the backward ("UniEP", section
3: the dispatch workers deliver the GEMM's operand rows; "MoonEP": zero-copy
dispatch into the expert-grouped layout).

Bitwise against the separate dispatch kernel (which the oracle pins), for Xp,
every saved tensor, out and the whole backward, over shapes with ragged and
empty experts, a single token, an x too large for the gather-by-row kernel,
grids of 2, 74 and one CTA per SM, and the combine in GEMM2's epilogue; and
against the oracle on one shape.  Where the fused form does not apply (padded
layout, single-CTA tiles) the separate kernel runs, with the same bits.
"""
import numpy as np
import pytest
import torch

import moe_synth as S
from helpers import check_backward, check_forward, check_tables, poison, run_gpu, run_oracle, shape_inputs

pytestmark = pytest.mark.gpu

CASES = {
    "fine_grained": (S.CONFIGS[1], S.config_seed(1), 0),
    "ragged": (S.LayerShape(300, 256, 384, 5, 3), 91, 0),
    "odd_extents": (S.LayerShape(700, 384, 640, 6, 2), 92, 0),
    "empty_experts": (S.LayerShape(512, 256, 256, 32, 4), 93, 8),
    "one_token": (S.LayerShape(1, 256, 128, 6, 2), 94, 0),
    "k1_E1": (S.LayerShape(200, 128, 128, 1, 1), 95, 0),
    "large_x": (S.LayerShape(2100, 8192, 128, 8, 2), 96, 0),
}
SAVED = ("Xp", "GU", "h", "Y")
OUTS = ("out", "dx", "dgate", "dW1", "dW3", "dW2", "dY", "dGU", "dXp")


def _inputs(shape, seed, n_empty):
    inp = shape_inputs(shape, seed)
    if n_empty:
        inp["logits"][:, :n_empty] -= 40.0
    return inp


def _run(shape, inp, pad=0, **kw):
    from mixture_experts_layer_gb300.layer import MoELayer
    L = MoELayer(shape.T, shape.H, shape.F, shape.E, shape.k, pad=pad)
    poison(L)
    run_gpu(L, inp, opts=L.opts(**kw))
    return L


def _same(a, b):
    for n in SAVED:
        assert torch.equal(getattr(a, n)[: a.R], getattr(b, n)[: b.R]), n
    for n in OUTS:
        assert torch.equal(getattr(a, n), getattr(b, n)), n


@pytest.mark.parametrize("name", list(CASES))
def test_fused_dispatch_same_bits(name):
    shape, seed, n_empty = CASES[name]
    inp = _inputs(shape, seed, n_empty)
    ref = _run(shape, inp, dispatch=1)
    _same(_run(shape, inp, dispatch=2), ref)


@pytest.mark.parametrize("kw", [dict(grid=2), dict(grid=74), dict(grid=-1), dict(combine=1)])
def test_fused_dispatch_grids_and_combine(kw):
    shape, seed, _ = CASES["odd_extents"]
    inp = _inputs(shape, seed, 0)
    if kw.get("grid") == -1:
        kw = dict(grid=torch.cuda.get_device_properties(0).multi_processor_count)
    ref = _run(shape, inp, dispatch=1)
    _same(_run(shape, inp, dispatch=2, **kw), ref)


def test_fused_dispatch_falls_back_with_the_same_bits():
    shape, seed, _ = CASES["ragged"]
    inp = _inputs(shape, seed, 0)
    _same(_run(shape, inp, dispatch=2, cta_pair=1), _run(shape, inp, dispatch=1, cta_pair=1))
    a, b = _run(shape, inp, pad=64, dispatch=2), _run(shape, inp, pad=64, dispatch=1)
    used = int(a.offsets[-1])  # rows past the ones in use keep their poison in both
    for n in SAVED + ("dY", "dGU", "dXp"):
        assert torch.equal(getattr(a, n)[:used], getattr(b, n)[:used]), n
    for n in ("out", "dx", "dgate", "dW1", "dW3", "dW2"):
        assert torch.equal(getattr(a, n), getattr(b, n)), n


def test_fused_dispatch_matches_oracle():
    shape, seed, n_empty = CASES["ragged"]
    inp = _inputs(shape, seed, n_empty)
    L = _run(shape, inp, dispatch=2)
    ref = run_oracle(inp, shape.k, shape.E)
    check_tables(L, ref)
    check_forward(L, ref)
    check_backward(L, ref)
