"""Routing tables on the GPU vs the CPU oracle, bit-exact, over many (T, E, k).

Covers both top-k kernels (four threads per token where E % 4 == 0, E <= 256
and k <= 8; one warp per token otherwise), ragged token counts (not multiples
of the 64-token CTA or the 256-token chunk), logits with many exact ties (values
drawn from a few levels, every logit equal, and -0 next to +0) and logits that
differ only in their last bits (distinct values a few ulps apart).  Row widths
E that are multiples of 16 without being 16 times a power of two leave value
slots of the four-thread kernel past the row's end.  Ties must go to the
lower expert id ("UniEP", section 3.1: a deterministic mapping; the gating reading
of the layer: descending logit, ties to the lower id).
"""
import numpy as np
import pytest
import torch

import oracle.moe_oracle as O

pytestmark = pytest.mark.gpu

# (T, E, k): E % 4 == 0 and k <= 8 take the four-threads-per-token kernel.
SHAPES = [
    (1, 4, 4), (63, 8, 2), (300, 12, 3), (1000, 20, 5), (777, 64, 6), (1500, 100, 8), (2049, 128, 8),
    (520, 256, 8), (333, 256, 1), (4000, 32, 8), (100, 32, 1), (700, 128, 3), (65, 64, 8),
    # several 8192-token super-chunks (the coarse level of the prefix over chunks), ragged tails;
    # 32768 tokens: chunk and super-chunk counts both a multiple of 4 (the rank kernel's 16-byte loads)
    (20000, 64, 6), (17000, 128, 8), (32768, 64, 8), (32768, 128, 3),
    # E a multiple of 16 but not 16 times a power of two: the row is narrower than the value slots
    (700, 48, 8), (1000, 80, 4), (900, 96, 6), (5000, 112, 8), (300, 192, 8), (257, 240, 5),
    # the warp-per-token kernel
    (500, 6, 2), (400, 260, 4), (300, 64, 9), (129, 1, 1), (9000, 6, 2),
]
KINDS = ["normal", "levels", "equal", "close", "zeros"]


def _logits(T, E, kind, seed):
    g = torch.Generator().manual_seed(seed)
    if kind == "normal":
        return torch.randn(T, E, generator=g)
    if kind == "levels":  # five levels: most rows hold ties at the threshold
        return torch.randint(0, 5, (T, E), generator=g).float() * 0.5 - 1.0
    if kind == "close":  # 0.5 plus a few multiples of 2^-21: distinct values 8 ulps apart, some exact ties
        return 0.5 + torch.randint(0, 6, (T, E), generator=g).float() * 2.0 ** -21
    if kind == "zeros":  # -0 and +0 (equal values: ids decide), the smallest subnormals of both signs, one level
        levels = torch.tensor([-0.0, 0.0, -1e-45, 1e-45, 0.25])
        return levels[torch.randint(0, 5, (T, E), generator=g)]
    return torch.full((T, E), 0.75)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("T,E,k", SHAPES)
def test_routing_tables_match_oracle(T, E, k, kind):
    import mixture_experts_layer_gb300 as M
    from mixture_experts_layer_gb300.layer import MoELayer
    M.lib()
    lg = _logits(T, E, kind, 1000 * T + 10 * E + k)
    layer = MoELayer(T, 128, 128, E, k, with_backward=False)
    layer.w.fill_(float("nan"))
    layer.plan(lg.cuda().contiguous())
    torch.cuda.synchronize()
    st, where, detail = layer.status()
    assert st == 0, f"device status {st} at {where} ({detail})"
    ids, w = O.route(lg.numpy(), k)
    perm = O.permutation(ids, E)
    assert np.array_equal(layer.ids.cpu().numpy(), ids), "topk ids"
    assert np.array_equal(layer.counts.cpu().numpy(), perm.counts), "counts"
    assert np.array_equal(layer.offsets.cpu().numpy(), perm.offsets), "offsets"
    assert np.array_equal(layer.dest.cpu().numpy(), perm.dest), "dest"
    assert np.array_equal(layer.row_src.cpu().numpy(), perm.row_src), "row_src"
    assert np.array_equal(layer.row_slot.cpu().numpy().astype(np.int64), perm.row_slot), "row_slot"
    gw = layer.w.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(gw - w.astype(np.float64))) <= 4 * 2.0 ** -24, "gate weights"
