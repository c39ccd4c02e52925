"""Two-SM pair tiles (tcgen05 cta_group::2) vs the CPU oracle and vs themselves.

The pair kernels run whenever a grouped GEMM is its own launch and
moe_opts.cta_pair = 2: here schedule 0 (one launch per phase), so all six GEMM
modes take the pair path.  Shapes cover an odd number of 128-row tiles per
expert (a pair whose second half has no rows), N extents that are odd
multiples of 128 (128-wide tail tiles, 64 columns per CTA), weight-gradient
extents that are odd multiples of 128 (a pair whose second CTA lies past the
weight), ragged K tails, and empty experts.
"""
import pytest
import torch

import moe_synth as S
from helpers import check_backward, check_forward, check_tables, poison, run_gpu, run_oracle, shape_inputs
from test_gpu_determinism import _diff

pytestmark = pytest.mark.gpu

CASES = {
    "tiny": (S.CONFIGS[0], 20260000, 0),
    "ragged": (S.LayerShape(300, 256, 384, 5, 3), 11, 0),
    "odd_extents": (S.LayerShape(700, 384, 640, 6, 2), 41, 0),
    "multi_tile": (S.LayerShape(1000, 512, 256, 16, 4), 12, 0),
    "k1_E1": (S.LayerShape(200, 128, 128, 1, 1), 13, 0),
    "one_token": (S.LayerShape(1, 256, 128, 6, 2), 15, 0),
    "empty_experts": (S.LayerShape(512, 256, 256, 32, 4), 16, 8),
}
OUTS = ("out", "dx", "dgate", "dW1", "dW3", "dW2", "Y", "h", "GU", "dGU", "dXp")


def _inputs(shape, seed, n_empty):
    inp = shape_inputs(shape, seed)
    if n_empty:
        inp["logits"][:, :n_empty] -= 40.0
    return inp


@pytest.mark.parametrize("name", list(CASES))
def test_pair_tiles_match_oracle(name):
    from mixture_experts_layer_gb300.layer import MoELayer
    shape, seed, n_empty = CASES[name]
    inp = _inputs(shape, seed, n_empty)
    layer = MoELayer(shape.T, shape.H, shape.F, shape.E, shape.k)
    poison(layer)
    run_gpu(layer, inp, opts=layer.opts(schedule=0, cta_pair=2))
    ref = run_oracle(inp, shape.k, shape.E)
    check_tables(layer, ref)
    check_forward(layer, ref)
    check_backward(layer, ref)


@pytest.mark.parametrize("shape,seed", [(S.CONFIGS[1], S.config_seed(1)), (S.LayerShape(700, 384, 640, 6, 2), 42)])
def test_pair_tiles_bitwise_over_runs_and_grids(shape, seed):
    """Same bits over repeated runs and over grids of 2, 74 and one CTA per SM
    (each pair tile has one owning pair and a fixed reduction order)."""
    from mixture_experts_layer_gb300.layer import MoELayer
    inp = shape_inputs(shape, seed)
    layer = MoELayer(shape.T, shape.H, shape.F, shape.E, shape.k)
    run_gpu(layer, inp, opts=layer.opts(schedule=0, cta_pair=2))
    ref = {n: getattr(layer, n).clone() for n in OUTS}
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for g in (0, 0, 74, sms, 2):
        for n in OUTS:
            getattr(layer, n).fill_(float("nan"))
        run_gpu(layer, inp, opts=layer.opts(grid=g, schedule=0, cta_pair=2))
        for n in OUTS:
            md, frac = _diff(getattr(layer, n), ref[n])
            assert md == 0 and frac == 0, f"{n} differs at grid {g or sms}: max_diff={md} non-bw={frac:.2%}"


@pytest.mark.parametrize("shape,seed", [(S.CONFIGS[1], S.config_seed(1)), (S.LayerShape(700, 384, 640, 6, 2), 43)])
def test_pair_tiles_give_the_bits_of_single_tiles(shape, seed):
    """A pair tile's rows are computed by the same K-ordered MMA chain as a
    single-CTA tile's, so both tile shapes give the same bits."""
    from mixture_experts_layer_gb300.layer import MoELayer
    inp = shape_inputs(shape, seed)
    a = MoELayer(shape.T, shape.H, shape.F, shape.E, shape.k)
    b = MoELayer(shape.T, shape.H, shape.F, shape.E, shape.k)
    run_gpu(a, inp, opts=a.opts(schedule=0, cta_pair=1))
    run_gpu(b, inp, opts=b.opts(schedule=0, cta_pair=2))
    for n in OUTS:
        md, frac = _diff(getattr(a, n), getattr(b, n))
        assert md == 0 and frac == 0, f"{n}: max_diff={md} non-bw={frac:.2%}"


@pytest.mark.parametrize("shape,seed", [(S.CONFIGS[1], S.config_seed(1)), (S.LayerShape(700, 384, 640, 6, 2), 44),
                                        (S.LayerShape(900, 256, 256, 24, 4), 45)])
def test_fused_forward_pair_tiles_bitwise(shape, seed):
    """The fused persistent forward on pair tiles (task ring shared by a CTA pair)
    gives the bits of the phased pair-tile forward, over grids of 2, 74 and one
    CTA per SM, and of the single-CTA fused forward."""
    from mixture_experts_layer_gb300.layer import MoELayer
    inp = shape_inputs(shape, seed)
    if shape.E == 24:
        inp["logits"][:, :5] -= 40.0  # a few empty experts
    ref = MoELayer(shape.T, shape.H, shape.F, shape.E, shape.k)
    run_gpu(ref, inp, opts=ref.opts(schedule=0))
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    L = MoELayer(shape.T, shape.H, shape.F, shape.E, shape.k)
    for g, pair in ((0, 2), (2, 2), (74, 2), (sms, 2), (0, 1)):
        for n in ("Xp", "GU", "h", "Y", "out"):
            getattr(L, n).fill_(float("nan"))
        run_gpu(L, inp, opts=L.opts(grid=g, schedule=1, cta_pair=pair))
        for n in ("Xp", "GU", "h", "Y", "out", "dx", "dW1"):
            a, b = getattr(L, n), getattr(ref, n)
            if n in ("Xp", "GU", "h", "Y"):
                a, b = a[: L.R], b[: L.R]
            assert torch.equal(a, b), f"{n} differs (grid {g}, cta_pair {pair})"
