"""Seeded synthetic inputs for the MoE expert layer.

This module is the one place both sides of every parity check draw their inputs
from: the CUDA library's callers (tests, benchmark) and the CPU oracle's tests.
It holds none of the layer's arithmetic (no gating, no permutation, no expert
math); it only makes random tensors of the workloads' shapes and scales.

Random numbers
--------------
Every element is a pure function of (seed, stream, flat index), so any slice of
any tensor can be regenerated on its own (a few experts' weights, a few
tokens' rows) and the generator gives the same bits on the CPU and on a CUDA
device.  The word generator is SplitMix64 (Steele, Lea and Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014): the i-th word of a
stream whose state starts at ``key`` is ``mix64(key + (i + 1) * GOLDEN)``.

Each 64-bit word is split into four 16-bit uniforms whose centred sum
(Irwin-Hall with n = 4, variance matched to 1) stands in for a N(0, 1) draw:

    v = (u0 + u1 + u2 + u3 - 131070) * float32(sigma * sqrt(3) / 65536)

The centred sum is an integer below 2**24, so it is exact in float32; the
single float32 multiply is correctly rounded by IEEE 754 on every device, and
the final bfloat16 conversion rounds to nearest-even.  The result is therefore
bit-identical wherever it is computed.

Workloads
---------
``CONFIGS`` lists the five layer shapes the library is measured and checked on
(tokens T, hidden H, per-expert FFN width F, experts E, top-k k).  Router logits
are x @ W_r in float32 (plus, for the skewed workload, a per-expert bias that
follows a Zipf ranking); they are an input to the layer's planning step.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

MASK64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB

# One stream per tensor, in a fixed order.
STREAM_X, STREAM_WR, STREAM_W1, STREAM_W3, STREAM_W2, STREAM_DOUT, STREAM_PERM = range(7)

_CHUNK = 1 << 24


def _s64(v: int) -> int:
    """Python int -> the int64 with the same 64 bits."""
    v &= MASK64
    return v - (1 << 64) if v >> 63 else v


def mix64(z: int) -> int:
    """SplitMix64 output function on a Python int (reference form)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * MIX1) & MASK64
    z = ((z ^ (z >> 27)) * MIX2) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, stream: int) -> int:
    """Initial SplitMix64 state of one tensor's stream."""
    return mix64(((seed & ((1 << 56) - 1)) << 8) | (stream & 0xFF))


def _mix64_t(z: torch.Tensor) -> torch.Tensor:
    # int64 tensors: multiplication wraps mod 2**64; right shifts are
    # arithmetic, so the shifted-in sign bits are masked off.
    z = z ^ ((z >> 30) & ((1 << 34) - 1))
    z = z * _s64(MIX1)
    z = z ^ ((z >> 27) & ((1 << 37) - 1))
    z = z * _s64(MIX2)
    z = z ^ ((z >> 31) & ((1 << 33) - 1))
    return z


def words(key: int, start: int, count: int, device="cpu") -> torch.Tensor:
    """SplitMix64 words start .. start+count-1 of the stream at ``key`` (int64 bits)."""
    idx = torch.arange(start, start + count, dtype=torch.int64, device=device)
    z = idx * _s64(GOLDEN) + _s64(key + GOLDEN)
    return _mix64_t(z)


def _scale(sigma: float) -> float:
    return sigma * math.sqrt(3.0) / 65536.0


def normal_bf16(seed: int, stream: int, shape, sigma: float = 1.0, device="cpu",
                start: int = 0) -> torch.Tensor:
    """bf16 tensor of ``shape`` holding elements start .. start+numel-1 of a stream."""
    n = 1
    for s in shape:
        n *= int(s)
    key = stream_key(seed, stream)
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    c = torch.tensor(_scale(sigma), dtype=torch.float32, device=device)
    for a in range(0, n, _CHUNK):
        m = min(_CHUNK, n - a)
        z = words(key, start + a, m, device)
        s = ((z & 0xFFFF) + ((z >> 16) & 0xFFFF) + ((z >> 32) & 0xFFFF)
             + ((z >> 48) & 0xFFFF) - 131070)
        out[a:a + m] = (s.to(torch.float32) * c).to(torch.bfloat16)
    return out.view(*shape)


@dataclass(frozen=True)
class LayerShape:
    T: int
    H: int
    F: int
    E: int
    k: int
    name: str = ""
    skew: bool = False

    @property
    def R(self) -> int:
        return self.T * self.k


CONFIGS = {
    0: LayerShape(256, 128, 256, 8, 2, "tiny"),
    1: LayerShape(4096, 2048, 1408, 64, 6, "fine-grained"),
    2: LayerShape(4096, 7168, 2048, 256, 8, "large-expert"),
    3: LayerShape(4096, 7168, 2048, 256, 8, "skewed", skew=True),
    4: LayerShape(131072, 4096, 1536, 128, 8, "long-seq"),
}


def config_seed(index: int) -> int:
    return 20260000 + index


# Skewed workload: bias_e = BETA * ln(z_rank(e) / sum z) with z_i = i**-ZIPF_S, plus
# SKEW_EMPTY_BIAS on the SKEW_EMPTY lowest-ranked experts.  BETA was found by
# bisection with moe_synth/calibrate_skew.py so that the routed load has
# maxvio = max_e n_e / (T k / E) - 1 close to 3.
ZIPF_S = 1.2
SKEW_EMPTY = 16
SKEW_EMPTY_BIAS = -30.0
SKEW_BETA = 0.125


def skew_bias(seed: int, E: int, beta: float = SKEW_BETA) -> torch.Tensor:
    """Per-expert additive logit bias (float32 [E]) of the skewed workload."""
    key = stream_key(seed, STREAM_PERM)
    rank = torch.argsort(words(key, 0, E), stable=True)  # expert -> 0-based Zipf rank
    rank = torch.argsort(rank, stable=True).tolist()
    z = [(i + 1) ** (-ZIPF_S) for i in range(E)]
    zs = sum(z)
    bias = []
    for e in range(E):
        b = beta * math.log(z[rank[e]] / zs)
        if rank[e] >= E - SKEW_EMPTY:
            b += SKEW_EMPTY_BIAS
        bias.append(b)
    return torch.tensor(bias, dtype=torch.float64).to(torch.float32)


def router_logits(x: torch.Tensor, Wr: torch.Tensor, bias: torch.Tensor | None = None) -> torch.Tensor:
    """float32 logits [T, E] = x @ W_r (+ bias), computed where x lives, TF32 off."""
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        lg = torch.matmul(x.to(torch.float32), Wr.to(torch.float32))
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    if bias is not None:
        lg = lg + bias.to(lg.device)
    return lg.contiguous()


def layer_inputs(shape: LayerShape, seed: int, device="cpu", weights_device=None,
                 with_weights: bool = True) -> dict:
    """All inputs of one forward+backward step of the layer.

    x ~ N(0,1) [T,H]; W_r ~ N(0,1/H) [H,E]; W1, W3 ~ N(0,1/H) [E,H,F];
    W2 ~ N(0,1/F) [E,F,H]; dout ~ N(0,1) [T,H]; all bf16; logits float32 [T,E].
    """
    T, H, F, E = shape.T, shape.H, shape.F, shape.E
    wdev = device if weights_device is None else weights_device
    d = {}
    d["x"] = normal_bf16(seed, STREAM_X, (T, H), 1.0, device)
    d["Wr"] = normal_bf16(seed, STREAM_WR, (H, E), 1.0 / math.sqrt(H), device)
    bias = skew_bias(seed, E) if shape.skew else None
    d["logits"] = router_logits(d["x"], d["Wr"], bias)
    d["dout"] = normal_bf16(seed, STREAM_DOUT, (T, H), 1.0, device)
    if with_weights:
        d["W1"] = normal_bf16(seed, STREAM_W1, (E, H, F), 1.0 / math.sqrt(H), wdev)
        d["W3"] = normal_bf16(seed, STREAM_W3, (E, H, F), 1.0 / math.sqrt(H), wdev)
        d["W2"] = normal_bf16(seed, STREAM_W2, (E, F, H), 1.0 / math.sqrt(F), wdev)
    return d


def expert_weights(shape: LayerShape, seed: int, e: int, device="cpu") -> dict:
    """W1[e], W3[e], W2[e] alone (same bits as the slices of the full tensors)."""
    H, F = shape.H, shape.F
    n = H * F
    return {
        "W1": normal_bf16(seed, STREAM_W1, (H, F), 1.0 / math.sqrt(H), device, start=e * n),
        "W3": normal_bf16(seed, STREAM_W3, (H, F), 1.0 / math.sqrt(H), device, start=e * n),
        "W2": normal_bf16(seed, STREAM_W2, (F, H), 1.0 / math.sqrt(F), device, start=e * n),
    }
