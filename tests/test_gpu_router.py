"""The router on the GPU (tcgen05 logits GEMM, gradient through the gating,
dWr GEMM over token splits, dx's router share) vs the CPU oracle.

Routing is decided on the float32 logits.  The GPU's logits are checked against
the oracle's, and the rest of the step is checked against the oracle run on the
GPU's own logits, so that a last-bit difference between two correct fp32 sums
cannot flip a near-tie and make the tables differ for the wrong reason.
"""
import numpy as np
import pytest
import torch

import moe_synth as S
import oracle.moe_oracle as O
from helpers import ELEM_TOL, RELL2_TOL, assert_close, check_backward, check_forward, f64, shape_inputs

pytestmark = pytest.mark.gpu

SHAPES = {
    "small": (S.LayerShape(300, 256, 128, 16, 2), 51),
    "E8": (S.LayerShape(200, 128, 128, 8, 2), 52),          # fewer experts than a 64-column panel
    "E72": (S.LayerShape(257, 384, 256, 72, 3), 53),        # MMA N rounded up to 80
    "E320": (S.LayerShape(130, 128, 128, 320, 4), 54),      # two N tiles
    "fine_grained": (S.CONFIGS[1], S.config_seed(1)),
}


def _run(shape, seed, grid=0):
    from mixture_experts_layer_gb300.layer import MoELayer
    inp = shape_inputs(shape, seed)
    L = MoELayer(shape.T, shape.H, shape.F, shape.E, shape.k, with_router=True)
    for n in ("logits", "dlogits", "dWr", "dx", "dW1"):
        getattr(L, n).fill_(float("nan"))
    opts = L.opts(grid=grid) if grid else None
    L.router_forward(inp["x"], inp["Wr"], opts=opts)
    L.plan(L.logits)
    L.forward(inp["x"], inp["W1"], inp["W3"], inp["W2"], opts=opts)
    L.backward(inp["dout"], inp["W1"], inp["W3"], inp["W2"], opts=opts, router=(inp["x"], inp["Wr"]))
    torch.cuda.synchronize()
    st, where, detail = L.status()
    assert st == 0, f"device status {st} at {where} ({detail})"
    return L, inp


def _reference(L, inp, shape):
    x, Wr = f64(inp["x"]), f64(inp["Wr"])
    W = (f64(inp["W1"]), f64(inp["W3"]), f64(inp["W2"]))
    logits = L.logits.cpu().numpy()
    ids, w = O.route(logits, shape.k)
    perm = O.permutation(ids, shape.E)
    fwd = O.forward(x, W, ids, w, perm)
    bwd = O.backward(f64(inp["dout"]), W, fwd, w, perm)
    r = O.router_grads(x, Wr, ids, w, bwd["dgate"], shape.E)
    dx = O.bf16_round(O.unpermute_sum(bwd["dXp"], perm.dest, mirror=False) + r["dx_router"])
    ref = {"ids": ids, "w": w, "perm": perm, **fwd, **bwd, "dx": dx, "dlogits": r["dlogits"], "dWr": r["dWr"]}
    return ref, O.router_logits(x, Wr)


@pytest.mark.parametrize("name", list(SHAPES))
def test_router_step_matches_oracle(name):
    shape, seed = SHAPES[name]
    L, inp = _run(shape, seed)
    ref, ref_logits = _reference(L, inp, shape)
    # logits: an fp32 sum of exact bf16 products; tighter than the layer's bar
    g = L.logits.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(g - ref_logits)) <= 1e-5 * np.max(np.abs(ref_logits)), "logits"
    assert np.array_equal(L.ids.cpu().numpy(), ref["ids"]), "topk ids"
    assert np.array_equal(L.dest.cpu().numpy(), ref["perm"].dest), "dest"
    check_forward(L, ref)
    check_backward(L, ref)
    assert_close("dlogits", L.dlogits, ref["dlogits"])
    assert_close("dWr", L.dWr, ref["dWr"])
    # only the k chosen logits carry a gradient, and each token's sum is ~0
    nz = (L.dlogits != 0).sum(dim=1)
    assert int(nz.max()) <= shape.k


def test_router_k1_has_no_gradient():
    shape = S.LayerShape(100, 128, 128, 8, 1)
    L, inp = _run(shape, 55)
    assert float(L.dlogits.abs().max()) == 0.0 and float(L.dWr.abs().max()) == 0.0


def test_router_bitwise_over_runs_and_grids():
    shape, seed = SHAPES["small"]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    runs = [_run(shape, seed, grid=g)[0] for g in (0, 0, 74, sms, 3)]
    for n in ("logits", "dlogits", "dWr", "dx"):
        ref = getattr(runs[0], n)
        for L in runs[1:]:
            assert torch.equal(getattr(L, n), ref), n
