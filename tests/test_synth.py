"""The seeded input generator: published SplitMix64 words, slice consistency, scale."""
import numpy as np
import torch

import moe_synth as S


def test_splitmix64_published_words():
    # SplitMix64 from state 0 (Steele, Lea, Flood 2014; the generator Java's
    # SplittableRandom and the xoshiro authors' seeding use).
    expect = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    got = [int(v) & S.MASK64 for v in S.words(0, 0, 3)]
    assert got == expect
    assert [S.mix64(S.GOLDEN * (i + 1)) for i in range(3)] == expect


def test_words_match_numpy_uint64():
    key = S.stream_key(1234, 5)
    n = 4096
    z = (np.arange(n, dtype=np.uint64) + np.uint64(1)) * np.uint64(S.GOLDEN) + np.uint64(key)
    z = (z ^ (z >> np.uint64(30))) * np.uint64(S.MIX1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(S.MIX2)
    z = z ^ (z >> np.uint64(31))
    got = S.words(key, 0, n).numpy().view(np.uint64)
    assert np.array_equal(got, z)


def test_slices_regenerate_the_same_bits():
    sh = S.LayerShape(8, 16, 24, 5, 2)
    full = S.layer_inputs(sh, 77)
    for e in range(sh.E):
        ew = S.expert_weights(sh, 77, e)
        for n in ("W1", "W3", "W2"):
            assert torch.equal(ew[n], full[n][e])
    part = S.normal_bf16(77, S.STREAM_X, (3, 16), 1.0, start=5 * 16)
    assert torch.equal(part, full["x"][5:8])


def test_scale_and_shape():
    x = S.normal_bf16(9, 0, (512, 512), 0.25).float()
    assert abs(x.mean().item()) < 0.01
    assert abs(x.std().item() - 0.25) < 0.005
    assert x.abs().max().item() <= 0.25 * 2 * 3 ** 0.5 + 1e-3  # Irwin-Hall(4) support


def test_skew_bias_shape():
    b = S.skew_bias(S.config_seed(3), 256)
    assert b.shape == (256,)
    assert int((b < -20).sum()) == S.SKEW_EMPTY
