"""Pins of the oracle's non-bitwise (two token sub-batch) step (CPU only).

* Linearity: in float64 the weight gradient of the whole batch is the sum of
  the two sub-batches' gradients, to rounding (any dropped or doubled token
  rows would fail it);
* per-token outputs (out, dx, dgate, the routing) of the sub-batch step equal
  the whole-batch step exactly, in the layer's own rounding;
* the rounded NB weight gradient is within a few float32 ulps of the
  whole-batch one and is the float32 sum of the two parts;
* a planted mistake (the second sub-batch's gradient left out) is caught.
"""
import numpy as np
import pytest

import oracle.moe_oracle as O


def _case(T, H=16, F=24, E=6, k=2, seed=0):
    rng = np.random.default_rng(seed)
    bf = O.bf16_round
    return dict(x=bf(rng.standard_normal((T, H))), logits=rng.standard_normal((T, E)).astype(np.float32),
                W=(bf(rng.standard_normal((E, H, F)) / np.sqrt(H)), bf(rng.standard_normal((E, H, F)) / np.sqrt(H)),
                   bf(rng.standard_normal((E, F, H)) / np.sqrt(F))),
                dout=bf(rng.standard_normal((T, H))), k=k, E=E)


def _full(c, mirror):
    return O.layer_step(c["x"], c["logits"], c["dout"], c["W"], c["k"], c["E"], mirror=mirror)


def _nb(c, mirror):
    return O.layer_step_subbatches(c["x"], c["logits"], c["dout"], c["W"], c["k"], c["E"], mirror=mirror)


@pytest.mark.parametrize("T,seed", [(40, 1), (37, 2), (2, 3)])
def test_weight_gradient_is_linear_in_the_batch(T, seed):
    c = _case(T, seed=seed)
    full, nb = _full(c, False), _nb(c, False)
    for n in ("dW1", "dW3", "dW2"):
        scale = np.max(np.abs(full[n]))
        assert np.max(np.abs(nb[n] - full[n])) <= 1e-12 * scale, n
    assert len(nb["parts"]) == 2
    assert nb["parts"][0]["out"].shape[0] == (T + 1) // 2  # the first sub-batch takes ceil(T/2) tokens


@pytest.mark.parametrize("T,seed", [(40, 4), (33, 5)])
def test_per_token_outputs_are_unchanged(T, seed):
    c = _case(T, seed=seed)
    full, nb = _full(c, True), _nb(c, True)
    for n in ("ids", "w", "out", "dx", "dgate"):
        assert np.array_equal(nb[n], full[n]), n


def test_rounded_nb_gradient_is_the_float32_sum_of_the_parts():
    c = _case(50, seed=6)
    full, nb = _full(c, True), _nb(c, True)
    for n in ("dW1", "dW3", "dW2"):
        p0, p1 = (q[n].astype(np.float32) for q in nb["parts"])
        assert np.array_equal(nb[n], (p0 + p1).astype(np.float64)), n
        # three float32 roundings (each part, their sum) against one (the whole batch's),
        # each within half an ulp of its own value
        ulp = lambda a: np.spacing(np.abs(a).astype(np.float32)).astype(np.float64)
        bound = 0.5 * (ulp(p0) + ulp(p1) + ulp(nb[n]) + ulp(full[n]))
        assert np.all(np.abs(nb[n] - full[n]) <= bound * (1 + 1e-9)), n
        assert np.any(nb[n] != full[n]), n  # a different order of the reduction: not bitwise the same


def test_one_token_has_one_sub_batch():
    c = _case(1, seed=7)
    full, nb = _full(c, True), _nb(c, True)
    assert len(nb["parts"]) == 1
    for n in ("dW1", "dW3", "dW2", "out", "dx"):
        assert np.array_equal(nb[n], full[n]), n


def test_planted_mistake_is_caught():
    """Leaving out the second sub-batch's gradient must fail the linearity pin."""
    c = _case(40, seed=8)
    full, nb = _full(c, False), _nb(c, False)
    wrong = nb["parts"][0]["dW1"]
    assert np.max(np.abs(wrong - full["dW1"])) > 1e-3 * np.max(np.abs(full["dW1"]))
