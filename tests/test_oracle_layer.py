"""Pins of the oracle's forward and backward (CPU only).

* a dense evaluation -- every token through every expert, masked by its gate
  weight -- differentiated by torch autograd in float64 (independent of the
  oracle's permutation plumbing and of its hand-derived backward formulas);
* central finite differences of every gradient;
* the E = 1, k = 1 special case, a plain SwiGLU MLP built from torch.nn.functional;
* identity experts, exact power-of-two scalings, expert relabelling;
* planted mistakes, to show the pins above catch them.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as Fn

import oracle.moe_oracle as O


def _case(T=24, H=12, F=20, E=5, k=2, seed=0):
    rng = np.random.default_rng(seed)
    bf = O.bf16_round
    x = bf(rng.standard_normal((T, H)))
    W1 = bf(rng.standard_normal((E, H, F)) / np.sqrt(H))
    W3 = bf(rng.standard_normal((E, H, F)) / np.sqrt(H))
    W2 = bf(rng.standard_normal((E, F, H)) / np.sqrt(F))
    dout = bf(rng.standard_normal((T, H)))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    return dict(x=x, W1=W1, W3=W3, W2=W2, dout=dout, logits=logits, k=k, E=E)


def _run(c, mirror):
    return O.layer_step(c["x"], c["logits"], c["dout"], (c["W1"], c["W3"], c["W2"]),
                        c["k"], c["E"], mirror=mirror)


def _dense_autograd(c, ids, w):
    t = lambda a: torch.tensor(np.asarray(a, np.float64), requires_grad=True)
    x, W1, W3, W2, wt = t(c["x"]), t(c["W1"]), t(c["W3"]), t(c["W2"]), t(w)
    ids_t = torch.tensor(ids.astype(np.int64))
    out = torch.zeros_like(x)
    for e in range(c["E"]):
        we = ((ids_t == e).to(torch.float64) * wt).sum(dim=1, keepdim=True)
        Y = (Fn.silu(x @ W1[e]) * (x @ W3[e])) @ W2[e]
        out = out + we * Y
    (out * torch.tensor(c["dout"])).sum().backward()
    g = lambda a: a.grad.numpy()
    return dict(out=out.detach().numpy(), dx=g(x), dW1=g(W1), dW3=g(W3), dW2=g(W2), dgate=g(wt))


@pytest.mark.parametrize("shape", [dict(), dict(T=31, H=8, F=16, E=4, k=3, seed=1),
                                   dict(T=9, H=16, F=8, E=7, k=7, seed=2),
                                   dict(T=40, H=8, F=12, E=6, k=1, seed=3)])
def test_matches_dense_autograd(shape):
    c = _case(**shape)
    r = _run(c, mirror=False)
    d = _dense_autograd(c, r["ids"], r["w"])
    for name in ("out", "dx", "dW1", "dW3", "dW2", "dgate"):
        assert np.allclose(r[name], d[name], rtol=1e-10, atol=1e-12), name


def test_finite_differences():
    c = _case(T=10, H=6, F=8, E=4, k=2, seed=7)
    r = _run(c, mirror=False)
    ids, w, perm = r["ids"], r["w"].astype(np.float64), r["perm"]
    Wt = (c["W1"], c["W3"], c["W2"])

    def loss(x, W, wv):
        return float((O.forward(x, W, ids, wv, perm, mirror=False)["out"] * c["dout"]).sum())

    eps = 1e-6
    rng = np.random.default_rng(8)
    for name, arr_i in (("x", None), ("W1", 0), ("W3", 1), ("W2", 2), ("w", None)):
        for _ in range(4):
            if name == "x":
                base = c["x"]
            elif name == "w":
                base = w
            else:
                base = Wt[arr_i]
            idx = tuple(int(rng.integers(0, s)) for s in base.shape)
            vals = []
            for sgn in (1, -1):
                p = base.copy()
                p[idx] += sgn * eps
                xs = p if name == "x" else c["x"]
                ws = p if name == "w" else w
                W = list(Wt)
                if arr_i is not None:
                    W[arr_i] = p
                vals.append(loss(xs, tuple(W), ws))
            fd = (vals[0] - vals[1]) / (2 * eps)
            an = {"x": r["dx"], "W1": r["dW1"], "W3": r["dW3"], "W2": r["dW2"], "w": r["dgate"]}[name][idx]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, idx, fd, an)


def test_single_expert_is_a_swiglu_mlp():
    c = _case(T=16, H=8, F=12, E=1, k=1, seed=4)
    c["logits"] = np.zeros((16, 1), np.float32)
    r = _run(c, mirror=False)
    assert np.all(r["w"] == 1.0)
    x = torch.tensor(c["x"])
    ref = Fn.linear(Fn.silu(Fn.linear(x, torch.tensor(c["W1"][0]).T)) * Fn.linear(x, torch.tensor(c["W3"][0]).T),
                    torch.tensor(c["W2"][0]).T)
    assert np.allclose(r["out"], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_identity_experts_return_the_input():
    c = _case(T=30, H=8, E=6, k=3, seed=5)
    ids, w = O.route(c["logits"], 3)
    p = O.permutation(ids, 6)
    out = O.combine(O.gather(c["x"], p.row_src), w, p.dest, mirror=False)
    assert np.allclose(out, c["x"], rtol=4e-7, atol=0)


def test_power_of_two_scalings_are_exact_in_mirror_mode():
    c = _case(T=40, H=16, F=24, E=5, k=2, seed=6)
    r = _run(c, mirror=True)
    c2 = dict(c, W2=c["W2"] * 2.0)
    r2 = _run(c2, mirror=True)
    for n in ("out", "dx", "dW1", "dW3", "dgate"):
        assert np.array_equal(r2[n], 2.0 * r[n]), n
    assert np.array_equal(r2["dW2"], r["dW2"])
    c3 = dict(c, dout=c["dout"] * 0.5)
    r3 = _run(c3, mirror=True)
    for n in ("dx", "dW1", "dW3", "dW2", "dgate"):
        assert np.array_equal(r3[n], 0.5 * r[n]), n
    assert np.array_equal(r3["out"], r["out"])


def test_expert_relabelling_changes_nothing():
    c = _case(T=50, H=8, F=12, E=6, k=2, seed=9)
    r = _run(c, mirror=True)
    pi = np.array([3, 0, 5, 1, 4, 2])  # expert e becomes pi[e]
    c2 = dict(c)
    c2["logits"] = np.empty_like(c["logits"]); c2["logits"][:, pi] = c["logits"]
    for n in ("W1", "W3", "W2"):
        c2[n] = np.empty_like(c[n]); c2[n][pi] = c[n]
    r2 = _run(c2, mirror=True)
    assert np.array_equal(r2["ids"], pi[r["ids"]])
    for n in ("out", "dx", "dgate"):
        assert np.array_equal(r2[n], r[n]), n
    for n in ("dW1", "dW3", "dW2"):
        assert np.array_equal(r2[n][pi], r[n]), n


def test_sampled_rows_and_experts_match_the_full_layer():
    c = _case(T=64, H=16, F=24, E=6, k=3, seed=10)
    W = (c["W1"], c["W3"], c["W2"])
    for mirror, tol in ((False, 1e-12), (True, 1e-2)):
        r = _run(c, mirror)
        toks = [0, 5, 17, 63]
        s = O.token_rows(toks, c["x"][toks], c["dout"][toks], r["ids"], r["w"], W, mirror)
        for n in ("out", "dx", "dgate"):
            assert np.allclose(s[n], r[n][toks], rtol=tol, atol=tol * 1e-2), (mirror, n)
        for e in (0, 4):
            g = O.expert_grads(e, c["x"], c["dout"], r["ids"], r["w"], r["perm"], W, mirror)
            for n in ("dW1", "dW3", "dW2"):
                assert np.allclose(g[n], r[n][e], rtol=tol, atol=tol * 1e-2), (mirror, n)


# ------------------------------------------------------------ planted mistakes
_GOOD_BACKWARD = O.expert_backward


def _bad_backward_dropped_term(dY, G, U, W1e, W3e, W2e, mirror=True):
    dH = dY @ W2e.T
    s = O.sigmoid(G)
    dG = dH * U * s                      # the G * (1 - s) term is missing
    dU = dH * G * s
    return dG, dU, dG @ W1e.T + dU @ W3e.T


def _bad_backward_swapped(dY, G, U, W1e, W3e, W2e, mirror=True):
    dG, dU, _ = _GOOD_BACKWARD(dY, G, U, W1e, W3e, W2e, mirror)
    return dG, dU, dG @ W3e.T + dU @ W1e.T  # W1 and W3 exchanged


def _bad_combine_slots(Y, w, dest, mirror=True):
    out = np.zeros((dest.shape[0], Y.shape[1]))
    k = dest.shape[1]
    for j in range(k):
        out += w[:, j:j + 1] * Y[dest[:, k - 1 - j]]  # weight of the wrong slot
    return out


@pytest.mark.parametrize("target,bad", [("expert_backward", _bad_backward_dropped_term),
                                        ("expert_backward", _bad_backward_swapped),
                                        ("combine", _bad_combine_slots)])
def test_planted_mistakes_are_caught(monkeypatch, target, bad):
    c = _case(T=20, H=8, F=12, E=4, k=2, seed=11)
    monkeypatch.setattr(O, target, bad)
    r = _run(c, mirror=False)
    d = _dense_autograd(c, r["ids"], r["w"])
    ok = all(np.allclose(r[n], d[n], rtol=1e-8, atol=1e-10)
             for n in ("out", "dx", "dW1", "dW3", "dW2", "dgate"))
    assert not ok
