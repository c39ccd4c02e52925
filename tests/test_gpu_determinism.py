"""Bitwise reproducibility of the GPU path.

Outputs, weight gradients and tables must be bitwise identical over 10
repeated runs and across persistent grid sizes (74 and 148 CTAs, one per SM
of this GPU, and a single CTA):
every output tile has one owner and a fixed reduction order ("UniEP: Unified
Expert-Parallel MoE MegaKernel for LLM Training", section 6, Bitwise
Equivalence Verification: max_diff = 0 and 0% non-bitwise elements).
"""
import pytest
import torch

import moe_synth as S
from helpers import check_backward, check_forward, check_tables, poison, run_gpu, run_oracle, shape_inputs

pytestmark = pytest.mark.gpu

OUTS = ("ids", "w", "dest", "row_src", "out", "dx", "dgate", "dW1", "dW3", "dW2", "Y", "h", "dXp")


def _snapshot(layer):
    return {n: getattr(layer, n).clone() for n in OUTS}


def _diff(a, b):
    """(max_diff, fraction of non-bitwise-equal elements) as in the pages' Table 6."""
    if a.dtype in (torch.int32, torch.uint8):
        ne = (a != b)
        return float(ne.any()), float(ne.float().mean())
    ne = a.view(torch.int16 if a.element_size() == 2 else torch.int32) != \
        b.view(torch.int16 if b.element_size() == 2 else torch.int32)
    return float((a.float() - b.float()).abs().max()), float(ne.float().mean())


@pytest.mark.parametrize("shape,seed", [(S.CONFIGS[1], S.config_seed(1)), (S.LayerShape(1000, 512, 384, 12, 3), 31)])
def test_bitwise_over_runs_and_grids(shape, seed):
    from mixture_experts_layer_gb300.layer import MoELayer
    import mixture_experts_layer_gb300 as M
    inp = shape_inputs(shape, seed)
    layer = MoELayer(shape.T, shape.H, shape.F, shape.E, shape.k)
    run_gpu(layer, inp)
    ref = _snapshot(layer)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    runs = [0] * 9 + [74, 148, sms, 1]
    for g in runs:
        opts = layer.opts(grid=g) if g else None
        for n in OUTS:  # poison: a kernel that skipped work cannot pass
            getattr(layer, n).fill_(0 if getattr(layer, n).dtype != torch.float32 else float("nan"))
        run_gpu(layer, inp, opts=opts)
        for n in OUTS:
            md, frac = _diff(getattr(layer, n), ref[n])
            assert md == 0 and frac == 0, f"{n} differs at grid {g or sms}: max_diff={md} non-bw={frac:.2%}"


@pytest.mark.parametrize("shape,seed", [(S.CONFIGS[1], S.config_seed(1)), (S.LayerShape(777, 256, 384, 9, 3), 32),
                                        (S.LayerShape(1, 128, 128, 3, 2), 33),
                                        (S.LayerShape(900, 256, 256, 24, 4), 34)])
def test_schedules_give_the_same_bits(shape, seed):
    """The persistent fused kernels (task cursor + readiness counters) and the
    one-launch-per-phase kernels compute every tile identically: same bits
    for schedules 0, 1 and 2, starting from NaN-poisoned buffers."""
    from mixture_experts_layer_gb300.layer import MoELayer
    inp = shape_inputs(shape, seed)
    if shape.E == 24:  # a few empty experts
        inp["logits"][:, :5] -= 40.0
    layers = []
    for sched in (0, 1, 2):
        L = MoELayer(shape.T, shape.H, shape.F, shape.E, shape.k)
        poison(L)
        run_gpu(L, inp, opts=L.opts(schedule=sched))
        layers.append(L)
    rows = ("Xp", "GU", "h", "Y", "dY", "dGU", "dXp")
    for n in ("Xp", "GU", "h", "Y", "out", "dY", "dGU", "dXp", "dx", "dW1", "dW3", "dW2", "dgate"):
        ref = getattr(layers[0], n)[: layers[0].R if n in rows else None]
        assert not torch.isnan(ref.float()).any(), n
        for L in layers[1:]:
            assert torch.equal(getattr(L, n)[: L.R if n in rows else None], ref), n


@pytest.mark.parametrize("shape,seed", [(S.CONFIGS[1], S.config_seed(1)), (S.LayerShape(700, 384, 640, 6, 2), 35),
                                        (S.LayerShape(300, 256, 128, 4, 4), 36), (S.LayerShape(200, 128, 128, 8, 1), 37)])
def test_combine_in_gemm2_epilogue_is_bitwise(shape, seed):
    """The gated combine run in GEMM2's epilogue (per-token arrival counters,
    the warp completing a token sums its k rows in slot order) gives the bits of
    the separate combine kernel, over runs and grids."""
    from mixture_experts_layer_gb300.layer import MoELayer
    inp = shape_inputs(shape, seed)
    ref = MoELayer(shape.T, shape.H, shape.F, shape.E, shape.k)
    run_gpu(ref, inp, opts=ref.opts(combine=0))
    L = MoELayer(shape.T, shape.H, shape.F, shape.E, shape.k)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for g in (0, 0, 74, sms, 2):
        L.out.fill_(float("nan"))
        run_gpu(L, inp, opts=L.opts(grid=g, combine=1))
        assert torch.equal(L.out, ref.out), f"out differs at grid {g}"


@pytest.mark.parametrize("shape,seed", [(S.LayerShape(700, 384, 640, 6, 2), 35), (S.LayerShape(300, 256, 128, 4, 4), 36),
                                        (S.LayerShape(512, 256, 256, 32, 4), 38)])
def test_combine_in_gemm2_epilogue_matches_oracle(shape, seed):
    """The gated combine run in GEMM2's epilogue against the oracle's combine
    (out[t] = sum over the k slots, in slot order, of w[t,j] Y[dest[t,j]];
    "UniEP", section 3, Top-k accumulation constraint), on its own: tables,
    the forward's saved tensors and out, and the backward that reads them,
    from NaN-poisoned buffers, on shapes with ragged and empty experts."""
    from mixture_experts_layer_gb300.layer import MoELayer
    inp = shape_inputs(shape, seed)
    if shape.E == 32:
        inp["logits"][:, :8] -= 40.0  # eight empty experts
    L = MoELayer(shape.T, shape.H, shape.F, shape.E, shape.k)
    poison(L)
    run_gpu(L, inp, opts=L.opts(combine=1))
    ref = run_oracle(inp, shape.k, shape.E)
    check_tables(L, ref)
    check_forward(L, ref)
    check_backward(L, ref)
