"""moe_plan_noalloc: routing for callers that cannot allocate device memory.

Some callers run this library inside code that must not call cudaMalloc: an
inference engine or plugin whose device memory is planned before it runs, a
latency-critical path where an allocation could block, or a process that has no
device allocator of its own.  They pass inputs and outputs but no workspace;
the entry point keeps its scratch in a fixed device array inside the library.

Checked here through the C ABI, on two calls in a row with different inputs
(the shared array keeps the first call's contents): the tables and weights
equal those of moe_plan, which uses a caller-provided workspace, at the same
agreement bar as the other routing tests (tables bit-exact, weights within
4 float32 ulps).  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import moe_synth as S

pytestmark = pytest.mark.gpu


def _tables(layer):
    return {n: getattr(layer, n).cpu().numpy() for n in
            ("ids", "counts", "offsets", "dest", "row_src", "row_slot")}


@pytest.mark.parametrize("calls", [[(S.LayerShape(4096, 2048, 1408, 64, 6), 101, None),
                                    (S.LayerShape(1000, 128, 128, 256, 8), 102, "skew")]])
def test_noalloc_plan_matches_moe_plan(calls):
    import mixture_experts_layer_gb300 as M
    from mixture_experts_layer_gb300.layer import MoELayer

    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    for shape, seed, kind in calls:
        inp = S.layer_inputs(shape, seed, device="cuda", with_weights=False)
        lg = inp["logits"]
        if kind == "skew":
            lg = (lg + S.skew_bias(seed, shape.E).cuda()).contiguous()
        ref = MoELayer(shape.T, shape.H, shape.F, shape.E, shape.k, with_backward=False)
        got = MoELayer(shape.T, shape.H, shape.F, shape.E, shape.k, with_backward=False)
        # Poison every output of both calls the same way, so stale or unwritten
        # values cannot pass for results and the whole tile table compares equal
        # only where both calls wrote the same words.
        for L in (ref, got):
            for n in ("ids", "dest", "row_src", "counts", "offsets", "tiles"):
                getattr(L, n).fill_(-7)
            L.row_slot.fill_(0xAB)
            L.w.fill_(float("nan"))
        ref.plan(lg)
        rc = M.moe_plan_noalloc(got.dims, lg.data_ptr(), got.plan_s, status.data_ptr(),
                                torch.cuda.current_stream().cuda_stream)
        M.check(rc, "moe_plan_noalloc")
        torch.cuda.synchronize()
        rc, st, where, detail = M.moe_get_status(status.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert rc == 0 and st == 0, (st, where, detail)
        assert ref.status()[0] == 0
        a, b = _tables(ref), _tables(got)
        for n in a:
            assert np.array_equal(a[n], b[n]), n
        wa = ref.w.cpu().numpy().astype(np.float64)
        wb = got.w.cpu().numpy().astype(np.float64)
        assert np.max(np.abs(wa - wb)) <= 4 * 2.0 ** -24
        # The whole tile table: counts, per-expert first tiles, the 128-row tile
        # entries, the pair prefix and the per-expert GEMM row counts.
        assert torch.equal(ref.tiles, got.tiles), "tile table"
        assert int(got.tiles[0].item()) > 0


def test_noalloc_rejects_dims_beyond_its_buffer():
    import mixture_experts_layer_gb300 as M
    big = M.moe_dims(1 << 20, 128, 128, 1024, 8)  # ~4096 chunks x 1024 experts x 40 B >> 4 MiB
    plan = M.moe_plan_t()
    assert M.moe_plan_noalloc(big, 0, plan, 0) == M.MOE_ERR_TOO_LARGE
    assert "MOE_NOALLOC_SCRATCH_BYTES" in M.moe_strerror(M.MOE_ERR_TOO_LARGE)
    fits = M.moe_dims(131072, 4096, 1536, 128, 8)  # the long-sequence layer fits
    assert M.moe_plan_noalloc(fits, 0, plan, 0) == M.MOE_ERR_ARG  # rejected only for its null pointers


def test_clear_status_touches_only_the_status_words():
    """moe_clear_status and moe_get_status are documented as safe on the 16-byte
    status buffer of moe_plan_noalloc: neither may write past its first three words."""
    import mixture_experts_layer_gb300 as M
    buf = torch.full((16,), 12345, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    M.check(M.moe_clear_status(buf.data_ptr(), s), "moe_clear_status")
    torch.cuda.synchronize()
    assert buf[:3].tolist() == [0, 0, 0]
    assert (buf[3:] == 12345).all(), buf.tolist()
    buf[:3] = torch.tensor([2, 7, 9], dtype=torch.int32, device="cuda")
    rc, st, where, detail = M.moe_get_status(buf.data_ptr(), s)
    assert rc == 0 and (st, where, detail) == (2, 7, 9)
    assert buf[:3].tolist() == [0, 0, 0]
    assert (buf[3:] == 12345).all(), buf.tolist()
