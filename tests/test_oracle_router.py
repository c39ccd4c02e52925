"""Pins of the oracle's router forward and backward (CPU only).

* logits against a brute-force triple loop;
* dlogits against torch autograd of the renormalised top-k softmax, routing
  held fixed (independent of the hand-derived formula);
* the whole step with the router on the path -- logits = x Wr, gating, experts,
  combine -- differentiated by torch autograd (dx, dWr) and by central finite
  differences of <dout, out> in Wr and in x;
* invariants: each token's dlogits sum to zero; k = 1 gives no router gradient;
* a planted mistake (the shared term of the softmax Jacobian dropped) is caught.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as Fn

import oracle.moe_oracle as O


def _case(T=20, H=12, F=16, E=6, k=2, seed=0):
    rng = np.random.default_rng(seed)
    bf = O.bf16_round
    return dict(x=bf(rng.standard_normal((T, H))), Wr=bf(rng.standard_normal((H, E)) / np.sqrt(H)),
                W1=bf(rng.standard_normal((E, H, F)) / np.sqrt(H)), W3=bf(rng.standard_normal((E, H, F)) / np.sqrt(H)),
                W2=bf(rng.standard_normal((E, F, H)) / np.sqrt(F)), dout=bf(rng.standard_normal((T, H))), k=k, E=E)


def _step(c, mirror=False):
    return O.layer_step_router(c["x"], c["Wr"], c["dout"], (c["W1"], c["W3"], c["W2"]), c["k"], c["E"], mirror=mirror)


def test_logits_brute_force():
    c = _case(T=5, H=7, E=3)
    l = O.router_logits(c["x"], c["Wr"], mirror=False)
    for t in range(5):
        for e in range(3):
            acc = 0.0
            for h in range(7):
                acc += float(c["x"][t, h]) * float(c["Wr"][h, e])
            assert abs(l[t, e] - acc) <= 1e-12 * max(1.0, abs(acc))


@pytest.mark.parametrize("k,E", [(2, 6), (3, 5), (4, 4), (1, 5)])
def test_dlogits_match_autograd_of_gating(k, E):
    rng = np.random.default_rng(10 + k)
    T = 17
    logits = rng.standard_normal((T, E))
    ids, _ = O.route(logits.astype(np.float32), k)
    dgate = rng.standard_normal((T, k))
    lt = torch.tensor(logits, requires_grad=True)
    sel = torch.gather(lt, 1, torch.tensor(ids.astype(np.int64)))
    w = torch.softmax(sel, dim=1)  # renormalised over the chosen k
    (w * torch.tensor(dgate)).sum().backward()
    r = O.router_grads(np.zeros((T, 3)), np.zeros((3, E)), ids, w.detach().numpy(), dgate, E, mirror=False)
    assert np.allclose(r["dlogits"], lt.grad.numpy(), rtol=1e-12, atol=1e-14)


def _autograd_step(c, ids):
    """Every token through every expert, gated by the renormalised softmax of the
    router's logits over the (fixed) chosen experts; torch float64 autograd."""
    t = lambda a: torch.tensor(np.asarray(a, np.float64), requires_grad=True)
    x, Wr, W1, W3, W2 = t(c["x"]), t(c["Wr"]), t(c["W1"]), t(c["W3"]), t(c["W2"])
    ids_t = torch.tensor(ids.astype(np.int64))
    l = x @ Wr
    w = torch.softmax(torch.gather(l, 1, ids_t), dim=1)
    out = torch.zeros_like(x)
    for e in range(c["E"]):
        we = ((ids_t == e).to(torch.float64) * w).sum(dim=1, keepdim=True)
        out = out + we * ((Fn.silu(x @ W1[e]) * (x @ W3[e])) @ W2[e])
    (out * torch.tensor(c["dout"])).sum().backward()
    return dict(out=out.detach().numpy(), dx=x.grad.numpy(), dWr=Wr.grad.numpy(), dW1=W1.grad.numpy())


@pytest.mark.parametrize("shape", [dict(), dict(T=23, H=8, F=12, E=5, k=3, seed=1), dict(T=11, H=16, F=8, E=4, k=4, seed=2)])
def test_step_with_router_matches_autograd(shape):
    c = _case(**shape)
    r = _step(c)
    d = _autograd_step(c, r["ids"])
    for name in ("out", "dx", "dWr", "dW1"):
        assert np.allclose(r[name], d[name], rtol=1e-9, atol=1e-12), name


def _loss(c, x=None, Wr=None):
    x = c["x"] if x is None else x
    Wr = c["Wr"] if Wr is None else Wr
    r = O.layer_step_router(x, Wr, c["dout"], (c["W1"], c["W3"], c["W2"]), c["k"], c["E"], mirror=False)
    return float(np.sum(r["out"] * c["dout"])), r["ids"]


def test_finite_differences_in_Wr_and_x():
    c = _case(T=10, H=6, F=8, E=4, k=2, seed=5)
    r = _step(c)
    eps = 1e-6
    rng = np.random.default_rng(0)
    for _ in range(6):
        h, e = rng.integers(6), rng.integers(4)
        Wp, Wm = c["Wr"].copy(), c["Wr"].copy()
        Wp[h, e] += eps
        Wm[h, e] -= eps
        (lp, ip), (lm, im) = _loss(c, Wr=Wp), _loss(c, Wr=Wm)
        assert np.array_equal(ip, r["ids"]) and np.array_equal(im, r["ids"])  # routing unchanged
        assert abs((lp - lm) / (2 * eps) - r["dWr"][h, e]) <= 1e-6 * max(1.0, abs(r["dWr"][h, e]))
    for _ in range(6):
        t, h = rng.integers(10), rng.integers(6)
        xp, xm = c["x"].copy(), c["x"].copy()
        xp[t, h] += eps
        xm[t, h] -= eps
        (lp, ip), (lm, im) = _loss(c, x=xp), _loss(c, x=xm)
        assert np.array_equal(ip, r["ids"]) and np.array_equal(im, r["ids"])
        assert abs((lp - lm) / (2 * eps) - r["dx"][t, h]) <= 1e-6 * max(1.0, abs(r["dx"][t, h]))


def test_invariants():
    c = _case(T=30, E=7, k=3, seed=7)
    r = _step(c)
    assert np.max(np.abs(r["dlogits"].sum(axis=1))) <= 1e-12
    nz = (r["dlogits"] != 0).sum(axis=1)
    assert np.all(nz <= 3)
    c1 = _case(T=30, E=7, k=1, seed=8)
    r1 = _step(c1)
    assert np.all(r1["dlogits"] == 0.0) and np.all(r1["dWr"] == 0.0)


def test_planted_mistake_is_caught():
    """Dropping the shared term (w_m * sum_j w_j dgate_j) of the gating gradient
    must fail the autograd pin."""
    c = _case(seed=3)
    r = _step(c)
    d = _autograd_step(c, r["ids"])
    T, k = r["ids"].shape
    wrong = np.zeros_like(r["dlogits"])
    for j in range(k):
        wrong[np.arange(T), r["ids"][:, j]] = r["w"][:, j] * r["dgate"][:, j]
    assert not np.allclose(c["x"].T @ wrong, d["dWr"], rtol=1e-6, atol=1e-9)
    assert np.allclose(r["dWr"], d["dWr"], rtol=1e-9, atol=1e-12)
