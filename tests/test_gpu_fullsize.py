"""GPU path vs the oracle at the workloads' full sizes, in the launch
configuration the benchmark times (one persistent CTA per SM).

* fine-grained (T=4096, H=2048, F=1408, E=64, k=6): every element of every
  output against the full oracle;
* large-expert and skewed (T=4096, H=7168, F=2048, E=256, k=8): routing tables
  bit-exact, 512 seeded tokens' out/dx/dgate, and the full weight gradients of
  at least four experts: the hottest, the coldest non-empty one and two seeded
  ones (plus, on the skewed layer, two of its empty experts, whose gradients
  must be exact zeros);
* long-sequence (T=131072, H=4096, F=1536, E=128, k=8): tables bit-exact, 512
  seeded tokens' out/dx/dgate and the full weight gradients of 4 seeded experts.
"""
import numpy as np
import pytest
import torch

import moe_synth as S
import oracle.moe_oracle as O
from helpers import (assert_close, check_backward, check_forward, check_tables, f64, run_gpu, run_oracle,
                     shape_inputs)

pytestmark = pytest.mark.gpu


def _layer(shape):
    from mixture_experts_layer_gb300.layer import MoELayer
    return MoELayer(shape.T, shape.H, shape.F, shape.E, shape.k)


def test_fine_grained_full_oracle():
    shape = S.CONFIGS[1]
    inp = shape_inputs(shape, S.config_seed(1))
    layer = _layer(shape)
    run_gpu(layer, inp)
    ref = run_oracle(inp, shape.k, shape.E)
    check_tables(layer, ref)
    check_forward(layer, ref)
    check_backward(layer, ref)


def _sampled(idx, n_tokens, experts_fn):
    shape = S.CONFIGS[idx]
    inp = shape_inputs(shape, S.config_seed(idx))
    layer = _layer(shape)
    run_gpu(layer, inp)
    # Routing tables, bit-exact, for every token.
    lg = inp["logits"].cpu().numpy()
    ids, w = O.route(lg, shape.k)
    perm = O.permutation(ids, shape.E)
    assert np.array_equal(layer.ids.cpu().numpy(), ids)
    assert np.array_equal(layer.counts.cpu().numpy(), perm.counts)
    assert np.array_equal(layer.offsets.cpu().numpy(), perm.offsets)
    assert np.array_equal(layer.dest.cpu().numpy(), perm.dest)
    assert np.array_equal(layer.row_src.cpu().numpy(), perm.row_src)
    assert np.array_equal(layer.row_slot.cpu().numpy().astype(np.int64), perm.row_slot)
    assert np.max(np.abs(layer.w.cpu().numpy().astype(np.float64) - w)) <= 4 * 2.0 ** -24

    W = lambda e: (f64(inp["W1"][e]), f64(inp["W3"][e]), f64(inp["W2"][e]))
    rng = np.random.default_rng(1000 + idx)
    # Dispatched rows: a copy, bit-exact (sampled rows of Xp against x[row_src]).
    rs = torch.as_tensor(rng.choice(layer.R, size=min(layer.R, 4096), replace=False), device="cuda")
    assert torch.equal(layer.Xp[rs], inp["x"][torch.as_tensor(perm.row_src, device="cuda")[rs]]), "Xp rows"
    toks = sorted(rng.choice(shape.T, size=n_tokens, replace=False).tolist())
    tk = torch.tensor(toks, device="cuda")
    s = O.token_rows(toks, f64(inp["x"][tk]), f64(inp["dout"][tk]), ids, w, W, mirror=True)
    assert_close("out[sample]", layer.out[tk], s["out"])
    assert_close("dx[sample]", layer.dx[tk], s["dx"])
    assert_close("dgate[sample]", layer.dgate[tk], s["dgate"])

    xs = lambda t: f64(inp["x"][torch.as_tensor(t, device="cuda")])
    ds = lambda t: f64(inp["dout"][torch.as_tensor(t, device="cuda")])
    for e in experts_fn(perm.counts, rng):
        g = O.expert_grads(e, xs, ds, ids, w, perm, W, mirror=True)
        if perm.counts[e] == 0:
            for n in ("dW1", "dW3", "dW2"):
                assert float(getattr(layer, n)[e].abs().max()) == 0.0
            continue
        assert_close(f"dW1[{e}]", layer.dW1[e], g["dW1"])
        assert_close(f"dW3[{e}]", layer.dW3[e], g["dW3"])
        assert_close(f"dW2[{e}]", layer.dW2[e], g["dW2"])


def _hot_cold_and_seeded(c, rng, n_seeded=2):
    """The hottest expert, the coldest non-empty one and n_seeded other non-empty ones."""
    live = np.flatnonzero(c > 0)
    hot = int(live[np.argmax(c[live])])
    cold = int(live[np.argmin(c[live])])
    rest = [int(e) for e in live if e not in (hot, cold)]
    return [hot, cold] + sorted(rng.choice(rest, n_seeded, replace=False).tolist())


def test_large_expert_sampled():
    _sampled(2, 512, _hot_cold_and_seeded)


def test_skewed_sampled():
    def pick(c, rng):
        assert (c == 0).sum() >= 16
        empty = np.flatnonzero(c == 0)
        return _hot_cold_and_seeded(c, rng) + [int(empty[0]), int(empty[-1])]
    _sampled(3, 512, pick)


def test_long_sequence_sampled():
    _sampled(4, 512, lambda c, rng: sorted(rng.choice(len(c), 4, replace=False).tolist()))
