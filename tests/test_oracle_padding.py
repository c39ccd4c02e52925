"""Pins of the oracle's static-shape (padded) layout (CPU only).

* pad 0 and 1 are the padding-free tables;
* every expert's segment starts at a multiple of the granule and holds its
  rows, in token order, then padding rows (row_src = -1, row_slot = 255) up to
  the next multiple; removing the padding rows gives the padding-free tables,
  and dest moves by the same segment shift;
* the whole step on the padded layout equals the padding-free step exactly,
  output by output (padding rows carry zeros through every stage), and its
  stored row tensors are the padding-free rows plus zero rows;
* a hand-worked fixture: T = 3, k = 2, E = 3, pad = 4.
"""
import numpy as np
import pytest

import oracle.moe_oracle as O


def _ids(T, E, k, seed):
    rng = np.random.default_rng(seed)
    return np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int64)


@pytest.mark.parametrize("pad", [0, 1])
def test_no_padding(pad):
    ids = _ids(50, 7, 3, 0)
    a, b = O.permutation(ids, 7, pad), O.permutation(ids, 7)
    for n in ("counts", "offsets", "dest", "row_src", "row_slot"):
        assert np.array_equal(getattr(a, n), getattr(b, n)), n


@pytest.mark.parametrize("T,E,k,pad,seed", [(50, 7, 3, 8, 1), (200, 16, 2, 128, 2), (9, 12, 4, 5, 3), (1, 4, 1, 64, 4)])
def test_padded_tables(T, E, k, pad, seed):
    ids = _ids(T, E, k, seed)
    p, q = O.permutation(ids, E, pad), O.permutation(ids, E)
    assert np.array_equal(p.counts, q.counts)
    seg = np.diff(p.offsets)
    assert np.all(p.offsets % pad == 0)
    assert np.array_equal(seg, -(-q.counts // pad) * pad)
    assert p.row_src.shape[0] == p.offsets[E] <= T * k + min(E, T * k) * (pad - 1)
    for e in range(E):
        a, n = p.offsets[e], p.counts[e]
        assert np.all(p.row_src[a + n:p.offsets[e + 1]] == -1) and np.all(p.row_slot[a + n:p.offsets[e + 1]] == 255)
        assert np.all(p.row_src[a:a + n] >= 0)
    real = p.row_src >= 0
    assert np.array_equal(p.row_src[real], q.row_src) and np.array_equal(p.row_slot[real], q.row_slot)
    shift = (p.offsets[:-1] - q.offsets[:-1])[ids]
    assert np.array_equal(p.dest - shift, q.dest)


def test_hand_worked_fixture():
    # token 0 -> experts (2, 0), token 1 -> (0, 1), token 2 -> (2, 1); pad 4
    ids = np.array([[2, 0], [0, 1], [2, 1]])
    p = O.permutation(ids, 3, 4)
    assert p.counts.tolist() == [2, 2, 2]
    assert p.offsets.tolist() == [0, 4, 8, 12]
    assert p.dest.tolist() == [[8, 0], [1, 4], [9, 5]]
    assert p.row_src.tolist() == [0, 1, -1, -1, 1, 2, -1, -1, 0, 2, -1, -1]
    assert p.row_slot.tolist() == [1, 0, 255, 255, 1, 1, 255, 255, 0, 0, 255, 255]


@pytest.mark.parametrize("pad,mirror", [(8, True), (3, False), (16, True)])
def test_padded_step_equals_padding_free(pad, mirror):
    rng = np.random.default_rng(5)
    T, H, F, E, k = 30, 12, 16, 5, 2
    bf = O.bf16_round
    x = bf(rng.standard_normal((T, H)))
    logits = rng.standard_normal((T, E)).astype(np.float32)
    W = (bf(rng.standard_normal((E, H, F)) / 4), bf(rng.standard_normal((E, H, F)) / 4),
         bf(rng.standard_normal((E, F, H)) / 4))
    dout = bf(rng.standard_normal((T, H)))
    a = O.layer_step(x, logits, dout, W, k, E, mirror=mirror, pad=pad)
    b = O.layer_step(x, logits, dout, W, k, E, mirror=mirror)
    for n in ("out", "dx", "dgate", "dW1", "dW3", "dW2"):
        assert np.array_equal(a[n], b[n]), n
    real = a["perm"].row_src >= 0
    for n in ("Xp", "G", "U", "h", "Y", "dY", "dG", "dU", "dXp"):
        assert np.array_equal(a[n][real], b[n]), n
        assert np.all(a[n][~real] == 0), n
