"""The static-shape (padded) layout on the GPU (moe_dims.pad = P >= 2: every
expert's rows padded to a multiple of P, "MoonEP", The Buffer API,
token_padding), against the oracle's padded tables and against the
padding-free layer.

* routing tables bit-exact vs the oracle's padded permutation (padding rows
  row_src = -1, row_slot = 255), for granules 8 .. 128, empty experts, one
  token, and the scatter dispatch (x above 32 MB);
* the whole step, bit for bit, equals the padding-free step: out, dx, dgate,
  dW1, dW3, dW2, and every stored row tensor on its real rows, with zeros on
  the padding rows; under schedules 0 and 1, both tile shapes, the combine in
  GEMM2's epilogue and the non-bitwise weight gradients;
* one case through the oracle's padded step at the layer's tolerance.
"""
import numpy as np
import pytest
import torch

import moe_synth as S
import oracle.moe_oracle as O
from helpers import assert_close, f64, poison, run_gpu, shape_inputs

pytestmark = pytest.mark.gpu

CASES = {
    "tiny_P128": (S.CONFIGS[0], 20260000, 0, 128),
    "ragged_P64": (S.LayerShape(300, 256, 384, 5, 3), 81, 0, 64),
    "multi_tile_P8": (S.LayerShape(1000, 512, 256, 16, 4), 82, 0, 8),
    "odd_P5": (S.LayerShape(257, 256, 256, 9, 3), 83, 0, 5),
    "empty_experts_P128": (S.LayerShape(512, 256, 256, 32, 4), 84, 8, 128),
    "one_token_P128": (S.LayerShape(1, 256, 128, 6, 2), 85, 0, 128),
    "scatter_P128": (S.LayerShape(2100, 8192, 128, 8, 2), 86, 0, 128),
    # the largest granule the ABI accepts: nearly every grouped row is padding
    "max_pad_P4096": (S.LayerShape(64, 128, 128, 4, 2), 87, 0, 4096),
}
ROWS = ("Xp", "GU", "h", "Y", "dY", "dGU", "dXp")
TOKEN = ("out", "dx", "dgate", "dW1", "dW3", "dW2")


def _inputs(shape, seed, n_empty):
    inp = shape_inputs(shape, seed)
    if n_empty:
        inp["logits"][:, :n_empty] -= 40.0
    return inp


def _run(shape, inp, pad, **kw):
    from mixture_experts_layer_gb300.layer import MoELayer
    L = MoELayer(shape.T, shape.H, shape.F, shape.E, shape.k, pad=pad)
    poison(L)
    run_gpu(L, inp, opts=L.opts(**kw) if kw else None)
    return L


def _check_tables(L, inp, shape, pad):
    ids, _ = O.route(inp["logits"].cpu().numpy(), shape.k)
    p = O.permutation(ids, shape.E, pad)
    used = int(L.offsets[-1])
    assert used == p.row_src.shape[0] <= L.R
    assert np.array_equal(L.ids.cpu().numpy(), ids), "topk ids"
    assert np.array_equal(L.counts.cpu().numpy(), p.counts), "counts"
    assert np.array_equal(L.offsets.cpu().numpy(), p.offsets), "offsets"
    assert np.array_equal(L.dest.cpu().numpy(), p.dest), "dest"
    assert np.array_equal(L.row_src[:used].cpu().numpy(), p.row_src), "row_src"
    assert np.array_equal(L.row_slot[:used].cpu().numpy().astype(np.int64), p.row_slot), "row_slot"


def _check_same_bits(P, F):
    """P padded, F padding-free: identical per-token outputs and weight gradients;
    the real rows of every row tensor identical, the padding rows zero."""
    for n in TOKEN:
        assert torch.equal(getattr(P, n), getattr(F, n)), n
    used = int(P.offsets[-1])
    src = P.row_src[:used]
    real = src >= 0
    for n in ROWS:
        a = getattr(P, n)[:used]
        assert torch.equal(a[real], getattr(F, n)[: F.R]), n
        assert not a[~real].any(), f"{n}: padding rows are not zero"


@pytest.mark.parametrize("name", list(CASES))
def test_padded_tables_and_bits(name):
    shape, seed, n_empty, pad = CASES[name]
    inp = _inputs(shape, seed, n_empty)
    P = _run(shape, inp, pad)
    _check_tables(P, inp, shape, pad)
    F = _run(shape, inp, 0)
    _check_same_bits(P, F)


@pytest.mark.parametrize("kw", [dict(schedule=1), dict(schedule=1, cta_pair=1), dict(cta_pair=1), dict(cta_pair=2),
                                dict(combine=1), dict(wgrad_subbatches=2), dict(schedule=2)])
def test_padded_variants_same_bits(kw):
    shape, seed, n_empty, pad = CASES["multi_tile_P8"]
    inp = _inputs(shape, seed, n_empty)
    F = _run(shape, inp, 0, **kw)
    for p in (8, 128):
        _check_same_bits(_run(shape, inp, p, **kw), F)


def test_fine_grained_padded_same_bits():
    shape, seed = S.CONFIGS[1], S.config_seed(1)
    inp = shape_inputs(shape, seed)
    _check_same_bits(_run(shape, inp, 128), _run(shape, inp, 0))


def test_padded_vs_oracle():
    shape, seed, n_empty, pad = CASES["ragged_P64"]
    inp = _inputs(shape, seed, n_empty)
    L = _run(shape, inp, pad)
    W = (f64(inp["W1"]), f64(inp["W3"]), f64(inp["W2"]))
    ref = O.layer_step(f64(inp["x"]), inp["logits"].cpu().numpy(), f64(inp["dout"]), W, shape.k, shape.E,
                       mirror=True, pad=pad)
    used = ref["perm"].row_src.shape[0]
    assert np.array_equal(f64(L.Xp[:used]), ref["Xp"])
    F = shape.F
    assert_close("G", L.GU[:used, :F], ref["G"])
    assert_close("h", L.h[:used], ref["h"])
    assert_close("Y", L.Y[:used], ref["Y"])
    assert_close("dG", L.dGU[:used, :F], ref["dG"])
    assert_close("dXp", L.dXp[:used], ref["dXp"])
    for n in TOKEN:
        assert_close(n, getattr(L, n), ref[n])
