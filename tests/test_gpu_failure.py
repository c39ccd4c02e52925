"""Failure detection without a GPU fault: every wait in the kernels is bounded.

With moe_opts.debug_drop_task, the fused persistent forward withholds the
completion signal of one gather task, so the GEMM tile that needs those rows
waits out its bound.  The kernel must record MOE_ERR_TIMEOUT in the status word
and return (no hang, no fault), and the context must stay usable: the next
step, without the injection, must succeed and match the oracle's tables.
"""
import numpy as np
import pytest
import torch

import moe_synth as S
from helpers import run_gpu, run_oracle, check_forward, shape_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cta_pair", [1, 2])
def test_withheld_signal_times_out_and_recovers(cta_pair):
    from mixture_experts_layer_gb300.layer import MoELayer
    shape = S.LayerShape(600, 256, 256, 6, 2)
    inp = shape_inputs(shape, 61)
    L = MoELayer(shape.T, shape.H, shape.F, shape.E, shape.k)
    L.plan(inp["logits"])
    L.forward(inp["x"], inp["W1"], inp["W3"], inp["W2"], opts=L.opts(schedule=1, cta_pair=cta_pair, debug_drop_task=1))
    torch.cuda.synchronize()
    st, where, detail = L.status()  # reading the status clears it
    assert st == 1, f"expected MOE_ERR_TIMEOUT, got status {st} at {where}"
    # the context is usable and the layer is correct again without the injection
    run_gpu(L, inp, opts=L.opts(schedule=1, cta_pair=cta_pair))
    ref = run_oracle(inp, shape.k, shape.E)
    check_forward(L, ref)
