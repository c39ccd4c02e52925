"""Shared helpers of the GPU parity tests: run the layer through the C ABI and
compare with the CPU oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import moe_synth as S
import oracle.moe_oracle as O

# Agreement bar for floating-point tensors: per element
# |gpu - ref| <= 1e-2 * max|ref| and relative L2 error <= 5e-3.
ELEM_TOL = 1e-2
RELL2_TOL = 5e-3


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def assert_close(name, gpu, ref, elem_tol=ELEM_TOL, rel_l2_tol=RELL2_TOL):
    g = f64(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (name, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{name}: non-finite values on the GPU"
    scale = float(np.max(np.abs(r))) if r.size else 0.0
    err = float(np.max(np.abs(g - r))) if r.size else 0.0
    den = float(np.linalg.norm(r))
    rel = float(np.linalg.norm(g - r)) / den if den > 0 else float(np.linalg.norm(g - r))
    assert err <= elem_tol * max(scale, 1e-30), f"{name}: max |gpu-ref| = {err:.3e} > {elem_tol} * {scale:.3e}"
    assert rel <= rel_l2_tol, f"{name}: relative L2 error {rel:.3e} > {rel_l2_tol}"
    return err / max(scale, 1e-30), rel


def shape_inputs(shape: S.LayerShape, seed: int, bias=None, device="cuda"):
    d = S.layer_inputs(shape, seed, device=device)
    if bias is not None:
        d["logits"] = (d["logits"] + bias.to(d["logits"].device)).contiguous()
    return d


def poison(layer):
    """Fill every intermediate and output buffer with NaN, so a kernel that reads
    a value before it is written, or skips a write, cannot go unnoticed."""
    for n in ("Xp", "GU", "h", "Y", "out", "dY", "dGU", "dXp", "dx", "dW1", "dW3", "dW2", "dgate", "w"):
        if hasattr(layer, n):
            getattr(layer, n).fill_(float("nan"))


def run_gpu(layer, inp, opts=None):
    layer.plan(inp["logits"])
    layer.forward(inp["x"], inp["W1"], inp["W3"], inp["W2"], opts=opts)
    layer.backward(inp["dout"], inp["W1"], inp["W3"], inp["W2"], opts=opts)
    torch.cuda.synchronize()
    st, where, detail = layer.status()
    assert st == 0, f"device status {st} at {where} ({detail})"


def run_oracle(inp, k, E):
    W = (f64(inp["W1"]), f64(inp["W3"]), f64(inp["W2"]))
    return O.layer_step(f64(inp["x"]), inp["logits"].cpu().numpy(), f64(inp["dout"]), W, k, E, mirror=True)


def check_tables(layer, ref):
    assert np.array_equal(layer.ids.cpu().numpy(), ref["ids"]), "topk ids"
    p = ref["perm"]
    assert np.array_equal(layer.counts.cpu().numpy(), p.counts), "counts"
    assert np.array_equal(layer.offsets.cpu().numpy(), p.offsets), "offsets"
    assert np.array_equal(layer.dest.cpu().numpy(), p.dest), "dest"
    assert np.array_equal(layer.row_src.cpu().numpy(), p.row_src), "row_src"
    assert np.array_equal(layer.row_slot.cpu().numpy().astype(np.int64), p.row_slot), "row_slot"
    w = layer.w.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(w - ref["w"])) <= 4 * 2.0 ** -24, "gate weights"


def check_forward(layer, ref):
    assert np.array_equal(f64(layer.Xp), ref["Xp"]), "Xp (a copy) must be bit-exact"
    F = layer.F
    assert_close("G", layer.GU[:, :F], ref["G"])
    assert_close("U", layer.GU[:, F:], ref["U"])
    assert_close("h", layer.h, ref["h"])
    assert_close("Y", layer.Y, ref["Y"])
    assert_close("out", layer.out, ref["out"])


def check_backward(layer, ref):
    F = layer.F
    assert_close("dY", layer.dY, ref["dY"])
    assert_close("dgate", layer.dgate, ref["dgate"])
    assert_close("dG", layer.dGU[:, :F], ref["dG"])
    assert_close("dU", layer.dGU[:, F:], ref["dU"])
    assert_close("dXp", layer.dXp, ref["dXp"])
    assert_close("dx", layer.dx, ref["dx"])
    assert_close("dW1", layer.dW1, ref["dW1"])
    assert_close("dW3", layer.dW3, ref["dW3"])
    assert_close("dW2", layer.dW2, ref["dW2"])
