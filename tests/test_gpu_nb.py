"""The non-bitwise (NB) weight-gradient variant on the GPU
(moe_opts.wgrad_subbatches = 2: two token sub-batches, "UniEP", section 6,
Performance Cost of Bitwise Reproducibility).

* vs the CPU oracle's two-sub-batch step, at the layer's tolerance;
* structure, bit for bit: the NB weight gradients are the float32 sum of the
  weight gradients the GPU computes for each sub-batch run as a batch of its
  own, and every other output equals the bitwise-reproducible (BW) step;
* NB is reproducible from run to run and over grids, and differs from BW in
  the last bits (max_diff and the fraction of non-bitwise elements, the
  pages' Table 6 measures, are reported);
* with one token there is a single sub-batch and NB equals BW.
"""
import pytest
import torch

import moe_synth as S
import oracle.moe_oracle as O
from helpers import assert_close, f64, poison, run_gpu, shape_inputs
from test_gpu_determinism import _diff

pytestmark = pytest.mark.gpu

CASES = {
    "fine_grained": (S.CONFIGS[1], S.config_seed(1), 0),
    "ragged_odd_T": (S.LayerShape(777, 256, 384, 9, 3), 71, 0),
    "empty_experts": (S.LayerShape(900, 256, 256, 24, 4), 72, 5),
    "k1_E1": (S.LayerShape(301, 128, 128, 1, 1), 73, 0),
}
DW = ("dW1", "dW3", "dW2")


def _inputs(shape, seed, n_empty):
    inp = shape_inputs(shape, seed)
    if n_empty:
        inp["logits"][:, :n_empty] -= 40.0
    return inp


def _layer(shape, inp, **kw):
    from mixture_experts_layer_gb300.layer import MoELayer
    L = MoELayer(shape.T, shape.H, shape.F, shape.E, shape.k)
    poison(L)
    run_gpu(L, inp, opts=L.opts(**kw))
    return L


def _half(inp, a, b):
    return {n: (v[a:b].clone() if n in ("x", "logits", "dout") else v) for n, v in inp.items()}


@pytest.mark.parametrize("name", list(CASES))
def test_nb_matches_oracle(name):
    shape, seed, n_empty = CASES[name]
    inp = _inputs(shape, seed, n_empty)
    L = _layer(shape, inp, wgrad_subbatches=2)
    W = (f64(inp["W1"]), f64(inp["W3"]), f64(inp["W2"]))
    ref = O.layer_step_subbatches(f64(inp["x"]), inp["logits"].cpu().numpy(), f64(inp["dout"]), W, shape.k, shape.E,
                                  mirror=True)
    for n in ("out", "dx", "dgate") + DW:
        assert_close(n, getattr(L, n), ref[n])


@pytest.mark.parametrize("name", ["fine_grained", "ragged_odd_T", "empty_experts"])
@pytest.mark.parametrize("cta_pair", [1, 2])
def test_nb_is_the_sum_of_the_sub_batches(name, cta_pair):
    shape, seed, n_empty = CASES[name]
    inp = _inputs(shape, seed, n_empty)
    nb = _layer(shape, inp, wgrad_subbatches=2, cta_pair=cta_pair)
    bw = _layer(shape, inp, cta_pair=cta_pair)
    t0 = (shape.T + 1) // 2
    parts = [_layer(S.LayerShape(b - a, shape.H, shape.F, shape.E, shape.k), _half(inp, a, b), cta_pair=cta_pair)
             for a, b in ((0, t0), (t0, shape.T))]
    for n in DW:
        want = getattr(parts[0], n) + getattr(parts[1], n)  # float32 adds, sub-batch 0 first
        assert torch.equal(getattr(nb, n), want), n
    for n in ("out", "dx", "dgate", "dXp", "dGU", "dY"):
        assert torch.equal(getattr(nb, n), getattr(bw, n)), n


def test_nb_reproducible_and_not_bitwise_equal_to_bw():
    shape, seed, _ = CASES["fine_grained"]
    inp = shape_inputs(shape, seed)
    bw = _layer(shape, inp)
    ref = _layer(shape, inp, wgrad_subbatches=2)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for g in (0, 74, sms, 2):
        L = _layer(shape, inp, wgrad_subbatches=2, grid=g)
        for n in DW:
            assert torch.equal(getattr(L, n), getattr(ref, n)), f"{n} differs at grid {g}"
    report = {}
    for n in DW:
        md, frac = _diff(getattr(ref, n), getattr(bw, n))
        report[n] = (md, frac)
        assert frac > 0, f"{n}: NB gave the bits of BW"
        assert_close(n, getattr(ref, n), f64(getattr(bw, n)))
    print("NB vs BW (max_diff, non-bitwise fraction):", report)


def test_one_token_nb_equals_bw():
    shape = S.LayerShape(1, 256, 128, 6, 2)
    inp = shape_inputs(shape, 74)
    nb = _layer(shape, inp, wgrad_subbatches=2)
    bw = _layer(shape, inp)
    for n in DW + ("dx", "out"):
        assert torch.equal(getattr(nb, n), getattr(bw, n)), n
