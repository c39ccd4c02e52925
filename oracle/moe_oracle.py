"""Plain CPU oracle of the single-GPU MoE expert layer, forward and backward.

TEST INFRASTRUCTURE ONLY.  It is imported by ``tests/``, by
``__graft_entry__.smoke()`` and by the CPU-baseline and reference legs of
``bench.py``; the library never imports it and has no CPU fallback.  It shares
no code with the CUDA path: it is written from the definitions below with
numpy, in float64, and uses library routines (matmul, exp, a stable argsort)
only as single steps.

What it computes (sources are named by page title and section):

* Gating -- "UniEP: Unified Expert-Parallel MoE MegaKernel for LLM Training",
  background, Forward Propagation (Figure 1): a router gives each token a
  probability distribution over the E experts and the token goes to its top-k.
  Reading taken: softmax over E, keep the k largest, renormalise over the k.
  The k are chosen on the float32 logits (softmax is monotone), ordered by
  descending logit, ties to the lower expert id.
* Permutation -- same page, Forward Propagation and section 3.1 Deterministic
  Token Mapping (Algorithm 1): rows are grouped by expert, experts in ascending
  order, and inside an expert by original token order (a stable sort).  With a
  single source the global offsets of Algorithm 1 reduce to the exclusive
  prefix sum of the per-expert counts, so this is a counting sort.
* Dispatch -- "MoonEP: Balanced Expert Parallelism for MoE Training via Dynamic
  Redundant Experts", How Redundant Expert Planning Achieves Perfect Balance
  (zero-copy dispatch): each token row is written straight to its final
  expert-grouped position.
* Experts -- UniEP, Forward Propagation: GroupGEMM, SwiGLU, GroupGEMM.  Reading:
  h = silu(x W1) * (x W3), y = h W2 with W1, W3 [E,H,F] and W2 [E,F,H].
* Combine -- UniEP, Forward Propagation and the GroupGEMM+Combine paragraph of
  section 3 (Top-k accumulation constraint): out[t] = sum over the k slots, in
  slot order, of w[t,j] * Y[dest[t,j]].
* Backward -- UniEP, Backward Propagation and Numerical Stability: output
  gradients are dispatched to the experts, the input gradients come from the
  dgrad GroupGEMMs and the weight gradients from a Transposed GroupGEMM whose
  reduction runs over the token rows; MoonEP, same section as above: the
  gradient of dispatch sums each token's k row gradients back to token order.
  The router is outside the timed layer (UniEP, section 6, Figure 4 "excluding
  gating"), so routing is held fixed and the gate weights w are an input whose
  gradient dgate is returned.
* Non-bitwise variant (``layer_step_subbatches``) -- UniEP, section 6,
  Performance Cost of Bitwise Reproducibility: two token sub-batches, weight
  gradients summed over them.
* Router (optional, ``router_logits`` / ``router_grads`` / ``layer_step_router``):
  logits = x Wr and the gradient through the renormalised top-k softmax with
  routing held fixed: dlogits, dWr = x^T dlogits and the router's share of dx.

Precision policy.  ``mirror=True`` rounds where the layer stores a tensor:
bf16 (round to nearest even) for Xp, G, U, h, Y, out, dY, dG, dU, dXp, dx and
float32 for w, dgate, dW1, dW3, dW2; everything between those points is
float64.  h is formed from the unrounded G and U; the backward reads the stored
(bf16) G and U.  ``mirror=False`` keeps float64 everywhere; the finite-difference
and dense pins use it.

Pinned by tests/test_oracle_*.py (all ``-m "not gpu"``): published SplitMix64
words, brute-force top-k and stable sort, closed forms (E = k, k = 1, E = 1),
a dense every-token-through-every-expert evaluation, identity experts,
exact power-of-two scalings, relabelling invariance, central finite
differences of every gradient, and a hand-worked permutation fixture.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

BF16_MAX_EXP = 128  # values rounding to 2**128 or beyond overflow to inf


# --------------------------------------------------------------------------
# rounding
# --------------------------------------------------------------------------
def bf16_round(a) -> np.ndarray:
    """Nearest bfloat16 value of each element (ties to even), as float64.

    bfloat16 has 8 significant bits: with a = m * 2**e (0.5 <= |m| < 1) the
    spacing is 2**(e-8), but never finer than 2**-133 (the subnormal spacing).
    Scaling by a power of two is exact, so ``rint`` does the only rounding.
    """
    a = np.asarray(a, dtype=np.float64)
    finite = np.isfinite(a)
    af = np.where(finite, a, 0.0)
    _, e = np.frexp(af)
    q = np.maximum(e - 8, -133)
    r = np.ldexp(np.rint(np.ldexp(af, -q)), q)
    r = np.where(np.abs(r) >= 2.0 ** BF16_MAX_EXP, np.copysign(np.inf, af), r)
    return np.where(finite, r, a)


def f32_round(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64).astype(np.float32).astype(np.float64)


def _store_bf16(a, mirror):
    return bf16_round(a) if mirror else np.asarray(a, dtype=np.float64)


def _store_f32(a, mirror):
    return f32_round(a) if mirror else np.asarray(a, dtype=np.float64)


# --------------------------------------------------------------------------
# gating
# --------------------------------------------------------------------------
def route(logits, k: int):
    """Top-k experts and renormalised gate weights of every token.

    Returns ids int32 [T,k] (descending logit, ties to the lower id) and
    w float32 [T,k] with w[t,j] = exp(l_j - l_max) / sum_{i in top-k} exp(l_i - l_max),
    which equals softmax over all E followed by renormalisation over the k
    (the full denominator cancels).
    """
    l = np.asarray(logits, dtype=np.float32)
    if l.ndim != 2:
        raise ValueError("logits must be [T, E]")
    if not np.all(np.isfinite(l)):
        raise ValueError("non-finite router logit")
    T, E = l.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    order = np.argsort(-l, axis=1, kind="stable")  # descending; equal logits keep id order
    ids = order[:, :k]
    sel = np.take_along_axis(l, ids, axis=1).astype(np.float64)
    ex = np.exp(sel - sel[:, :1])
    w = ex / ex.sum(axis=1, keepdims=True)
    return ids.astype(np.int32), w.astype(np.float32)


# --------------------------------------------------------------------------
# permutation
# --------------------------------------------------------------------------
@dataclass
class Permutation:
    counts: np.ndarray    # int64 [E]    rows per expert n_e
    offsets: np.ndarray   # int64 [E+1]  exclusive prefix of counts
    dest: np.ndarray      # int64 [T,k]  row of slot (t, j) in the grouped buffer
    row_src: np.ndarray   # int64 [R]    token of each grouped row
    row_slot: np.ndarray  # int64 [R]    slot j of each grouped row


def permutation(ids, E: int, pad: int = 0) -> Permutation:
    """Stable counting sort of the (token, slot) pairs by expert.

    Histogram, exclusive scan, then one pass over tokens in order (slots in
    order) handing out consecutive rows of each expert's segment.

    pad >= 2 is the static-shape layout ("MoonEP: Balanced Expert Parallelism
    for MoE Training via Dynamic Redundant Experts", The Buffer API, the
    token_padding parameter): each expert's segment is its count rounded up to
    a multiple of pad; the rows past the count are padding rows, marked with
    row_src = -1 and row_slot = 255.  counts stay the routed rows.
    """
    ids = np.asarray(ids)
    T, k = ids.shape
    counts = np.zeros(E, dtype=np.int64)
    for e in ids.reshape(-1).tolist():
        counts[e] += 1
    seg = -(-counts // pad) * pad if pad > 1 else counts
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(seg)
    cursor = offsets[:-1].copy()
    R = int(offsets[E])
    dest = np.empty((T, k), dtype=np.int64)
    row_src = np.full(R, -1, dtype=np.int64)
    row_slot = np.full(R, 255, dtype=np.int64)
    idl = ids.tolist()
    for t in range(T):
        for j in range(k):
            e = idl[t][j]
            r = cursor[e]
            cursor[e] = r + 1
            dest[t, j] = r
            row_src[r] = t
            row_slot[r] = j
    return Permutation(counts, offsets, dest, row_src, row_slot)


def gather(x, row_src) -> np.ndarray:
    """Dispatch: Xp[r] = x[row_src[r]] (a copy; exact); padding rows (row_src = -1) are zero."""
    row_src = np.asarray(row_src)
    real = row_src >= 0
    Xp = np.zeros((row_src.shape[0], np.asarray(x).shape[1]), dtype=np.float64)
    Xp[real] = np.asarray(x, dtype=np.float64)[row_src[real]]
    return Xp


def combine(Y, w, dest, mirror=True) -> np.ndarray:
    """out[t] = sum_j w[t,j] * Y[dest[t,j]], slots in ascending order."""
    Y = np.asarray(Y, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    T, k = dest.shape
    out = np.zeros((T, Y.shape[1]), dtype=np.float64)
    for j in range(k):
        out += w[:, j:j + 1] * Y[dest[:, j]]
    return _store_bf16(out, mirror)


def unpermute_sum(dXp, dest, mirror=True) -> np.ndarray:
    """Gradient of dispatch: dx[t] = sum_j dXp[dest[t,j]], slots in ascending order."""
    dXp = np.asarray(dXp, dtype=np.float64)
    T, k = dest.shape
    dx = np.zeros((T, dXp.shape[1]), dtype=np.float64)
    for j in range(k):
        dx += dXp[dest[:, j]]
    return _store_bf16(dx, mirror)


# --------------------------------------------------------------------------
# one expert
# --------------------------------------------------------------------------
def silu(a):
    with np.errstate(over="ignore"):
        return a / (1.0 + np.exp(-a))


def sigmoid(a):
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-a))


def expert_forward(X, W1e, W3e, W2e, mirror=True):
    """Rows X [n,H] through one SwiGLU expert.  Returns stored G, U, h, Y."""
    X = np.asarray(X, dtype=np.float64)
    G = X @ np.asarray(W1e, dtype=np.float64)
    U = X @ np.asarray(W3e, dtype=np.float64)
    h = _store_bf16(silu(G) * U, mirror)
    Y = _store_bf16(h @ np.asarray(W2e, dtype=np.float64), mirror)
    return _store_bf16(G, mirror), _store_bf16(U, mirror), h, Y


def expert_backward(dY, G, U, W1e, W3e, W2e, mirror=True):
    """Row gradients of one expert: dG, dU (SwiGLU backward) and dXp."""
    dY = np.asarray(dY, dtype=np.float64)
    dH = dY @ np.asarray(W2e, dtype=np.float64).T
    s = sigmoid(G)
    dG = _store_bf16(dH * U * s * (1.0 + G * (1.0 - s)), mirror)
    dU = _store_bf16(dH * G * s, mirror)
    dXp = dG @ np.asarray(W1e, dtype=np.float64).T + dU @ np.asarray(W3e, dtype=np.float64).T
    return dG, dU, _store_bf16(dXp, mirror)


def expert_wgrad(X, h, dY, dG, dU, mirror=True):
    """Transposed GroupGEMM of one expert: reductions over its token rows."""
    X = np.asarray(X, dtype=np.float64)
    dW1 = X.T @ dG
    dW3 = X.T @ dU
    dW2 = np.asarray(h, dtype=np.float64).T @ np.asarray(dY, dtype=np.float64)
    return _store_f32(dW1, mirror), _store_f32(dW3, mirror), _store_f32(dW2, mirror)


def dispatch_grad(dout, w, row_src, row_slot, mirror=True):
    """dY[r] = w[t,j] * dout[t] for the grouped row r of slot (t, j); zero on padding rows."""
    dout = np.asarray(dout, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    row_src, row_slot = np.asarray(row_src), np.asarray(row_slot)
    real = row_src >= 0
    dY = np.zeros((row_src.shape[0], dout.shape[1]), dtype=np.float64)
    dY[real] = w[row_src[real], row_slot[real]][:, None] * dout[row_src[real]]
    return _store_bf16(dY, mirror)


def gate_grad(dout, Y, dest, mirror=True):
    """dgate[t,j] = <dout[t], Y[dest[t,j]]>."""
    dout = np.asarray(dout, dtype=np.float64)
    Y = np.asarray(Y, dtype=np.float64)
    T, k = dest.shape
    g = np.empty((T, k), dtype=np.float64)
    for j in range(k):
        g[:, j] = np.einsum("th,th->t", dout, Y[dest[:, j]])
    return _store_f32(g, mirror)


# --------------------------------------------------------------------------
# the whole layer
# --------------------------------------------------------------------------
def _weights_getter(W):
    if callable(W):
        return W
    W1, W3, W2 = W
    return lambda e: (W1[e], W3[e], W2[e])


def forward(x, W, ids, w, perm: Permutation, mirror=True) -> dict:
    """Forward pass over all tokens.  W = (W1, W3, W2) arrays or a callable e -> (W1e, W3e, W2e)."""
    get = _weights_getter(W)
    x = np.asarray(x, dtype=np.float64)
    T, H = x.shape
    E = perm.counts.shape[0]
    R = perm.row_src.shape[0]
    Xp = gather(x, perm.row_src)
    G = U = h = None
    Y = np.zeros((R, H), dtype=np.float64)
    for e in range(E):
        a, b = int(perm.offsets[e]), int(perm.offsets[e + 1])
        W1e, W3e, W2e = get(e)
        Ge, Ue, he, Ye = expert_forward(Xp[a:b], W1e, W3e, W2e, mirror)
        if G is None:
            F = Ge.shape[1] if b > a else np.asarray(W1e).shape[1]
            G = np.zeros((R, F)); U = np.zeros((R, F)); h = np.zeros((R, F))
        G[a:b], U[a:b], h[a:b], Y[a:b] = Ge, Ue, he, Ye
    out = combine(Y, w, perm.dest, mirror)
    return {"Xp": Xp, "G": G, "U": U, "h": h, "Y": Y, "out": out}


def backward(dout, W, fwd: dict, w, perm: Permutation, mirror=True) -> dict:
    """Backward pass over all tokens given the forward's stored tensors."""
    get = _weights_getter(W)
    dY = dispatch_grad(dout, w, perm.row_src, perm.row_slot, mirror)
    dgate = gate_grad(dout, fwd["Y"], perm.dest, mirror)
    E = perm.counts.shape[0]
    R, F = fwd["G"].shape
    H = fwd["Xp"].shape[1]
    dG = np.zeros((R, F)); dU = np.zeros((R, F)); dXp = np.zeros((R, H))
    dW1 = np.zeros((E, H, F)); dW3 = np.zeros((E, H, F)); dW2 = np.zeros((E, F, H))
    for e in range(E):
        a, b = int(perm.offsets[e]), int(perm.offsets[e + 1])
        W1e, W3e, W2e = get(e)
        dG[a:b], dU[a:b], dXp[a:b] = expert_backward(dY[a:b], fwd["G"][a:b], fwd["U"][a:b],
                                                     W1e, W3e, W2e, mirror)
        dW1[e], dW3[e], dW2[e] = expert_wgrad(fwd["Xp"][a:b], fwd["h"][a:b], dY[a:b],
                                              dG[a:b], dU[a:b], mirror)
    dx = unpermute_sum(dXp, perm.dest, mirror)
    return {"dY": dY, "dgate": dgate, "dG": dG, "dU": dU, "dXp": dXp, "dx": dx,
            "dW1": dW1, "dW3": dW3, "dW2": dW2}


def layer_step(x, logits, dout, W, k: int, E: int, mirror=True, pad: int = 0) -> dict:
    """Plan, forward and backward of one step (everything the layer computes);
    pad >= 2: the static-shape layout with padded expert segments."""
    ids, w = route(logits, k)
    perm = permutation(ids, E, pad)
    fwd = forward(x, W, ids, w, perm, mirror)
    bwd = backward(dout, W, fwd, w, perm, mirror)
    return {"ids": ids, "w": w, "perm": perm, **fwd, **bwd}


def layer_step_subbatches(x, logits, dout, W, k: int, E: int, mirror=True) -> dict:
    """The non-bitwise (NB) variant of one step: the tokens form two sub-batches,
    [0, ceil(T/2)) and [ceil(T/2), T), each runs the whole step on its own, and
    the weight gradients are the sum of the two sub-batches' gradients, the
    second added onto the first in float32 (UniEP, section 6, Performance Cost of
    Bitwise Reproducibility: splitting the tokens into two sub-batches changes
    the accumulation order of the weight-gradient reduction).  Every other output
    is per token, so it is the two sub-batches' rows in token order."""
    x = np.asarray(x)
    T = x.shape[0]
    t0 = (T + 1) // 2
    parts = [layer_step(x[a:b], logits[a:b], dout[a:b], W, k, E, mirror) for a, b in ((0, t0), (t0, T)) if b > a]
    res = {n: np.concatenate([q[n] for q in parts]) for n in ("ids", "w", "out", "dx", "dgate")}
    for n in ("dW1", "dW3", "dW2"):
        res[n] = _store_f32(sum(q[n] for q in parts), mirror)  # one sub-batch (T = 1): its own gradient
    res["parts"] = parts
    return res


# --------------------------------------------------------------------------
# the router (gating) forward and backward
# --------------------------------------------------------------------------
def router_logits(x, Wr, mirror=True) -> np.ndarray:
    """l[t,e] = sum_h x[t,h] Wr[h,e]: the router's score of token t for expert e
    (UniEP, background, Forward Propagation: the router maps each token to a
    distribution over the experts).  Stored as float32."""
    x = np.asarray(x, dtype=np.float64)
    Wr = np.asarray(Wr, dtype=np.float64)
    return _store_f32(x @ Wr, mirror)


def router_grads(x, Wr, ids, w, dgate, E: int, mirror=True) -> dict:
    """Gradient of the loss through the gating, routing held fixed.

    With w_j = exp(l_j) / sum_{i in top-k} exp(l_i) (softmax over the experts,
    renormalised over the k chosen ones), dw_j / dl_m = w_j (delta_jm - w_m) for
    m among the chosen experts and 0 otherwise (the choice is piecewise
    constant in l), so
        dl_m = w_m (dgate_m - sum_j w_j dgate_j)   for the k chosen experts,
        dl_m = 0                                  for the others.
    dWr = x^T dl and the router's share of dx is dl Wr^T.

    Rounding points of the layer (mirror=True): dl in float32 (``dlogits``);
    the weight gradient dWr (float32) is formed from dl rounded to bf16, the
    stored row gradient the tensor cores read; the router's dx share is
    returned unrounded and is added to the experts' share before dx's single
    bf16 rounding.
    """
    x = np.asarray(x, dtype=np.float64)
    Wr = np.asarray(Wr, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    dgate = np.asarray(dgate, dtype=np.float64)
    ids = np.asarray(ids)
    T, k = ids.shape
    s = np.zeros(T)
    for j in range(k):
        s += w[:, j] * dgate[:, j]
    dl_slot = _store_f32(w * (dgate - s[:, None]), mirror)
    dlogits = np.zeros((T, E))
    for j in range(k):
        dlogits[np.arange(T), ids[:, j]] = dl_slot[:, j]
    dl_gemm = _store_bf16(dlogits, mirror)
    dWr = _store_f32(x.T @ dl_gemm, mirror)
    dx_router = dlogits @ Wr.T
    return {"dl_slot": dl_slot, "dlogits": dlogits, "dWr": dWr, "dx_router": dx_router}


def layer_step_router(x, Wr, dout, W, k: int, E: int, mirror=True) -> dict:
    """One step with the router on the path: logits = x Wr, then plan, forward
    and backward as in layer_step; dx gains the router's share (one bf16
    rounding of the sum of both shares).

    The experts are chosen on the float32 logits as in ``route``; the gate
    weights come from the float32 logits in mirror mode (as the layer stores
    them) and from the float64 logits otherwise."""
    logits = router_logits(x, Wr, mirror)
    ids, w = route(logits, k)
    if not mirror:
        sel = np.take_along_axis(np.asarray(logits, dtype=np.float64), ids.astype(np.int64), axis=1)
        ex = np.exp(sel - sel[:, :1])
        w = ex / ex.sum(axis=1, keepdims=True)
    perm = permutation(ids, E)
    fwd = forward(x, W, ids, w, perm, mirror)
    bwd = backward(dout, W, fwd, w, perm, mirror)
    r = router_grads(x, Wr, ids, w, bwd["dgate"], E, mirror)
    dx_experts = unpermute_sum(bwd["dXp"], perm.dest, mirror=False)
    step = {"ids": ids, "w": w, "perm": perm, **fwd, **bwd}
    step["logits"] = logits
    step["dlogits"] = r["dlogits"]
    step["dWr"] = r["dWr"]
    step["dx"] = _store_bf16(dx_experts + r["dx_router"], mirror)
    return step


# --------------------------------------------------------------------------
# sampled evaluation for layers too large to run whole on a CPU
# --------------------------------------------------------------------------
def token_rows(tokens, x_rows, dout_rows, ids, w, W, mirror=True) -> dict:
    """out, dx and dgate of selected tokens, computed from their own k rows.

    Every quantity except the weight gradients is row-local, so a token's
    outputs need only its own row of x, its row of dout and its k experts.
    x_rows / dout_rows are [len(tokens), H] (the rows of those tokens).
    """
    get = _weights_getter(W)
    tokens = list(tokens)
    ids = np.asarray(ids)
    w = np.asarray(w, dtype=np.float64)
    x_rows = np.asarray(x_rows, dtype=np.float64)
    dout_rows = np.asarray(dout_rows, dtype=np.float64)
    n, H = x_rows.shape
    k = ids.shape[1]
    Y = np.zeros((n, k, H)); dXp = np.zeros((n, k, H))
    dgate = np.zeros((n, k))
    by_e = {}
    for i, t in enumerate(tokens):
        for j in range(k):
            by_e.setdefault(int(ids[t, j]), []).append((i, j))
    for e, pairs in sorted(by_e.items()):
        W1e, W3e, W2e = get(e)
        ii = [p[0] for p in pairs]
        jj = [p[1] for p in pairs]
        G, U, h, Ye = expert_forward(x_rows[ii], W1e, W3e, W2e, mirror)
        tk = [tokens[i] for i in ii]
        dYe = _store_bf16(w[tk, jj][:, None] * dout_rows[ii], mirror)
        _, _, dXe = expert_backward(dYe, G, U, W1e, W3e, W2e, mirror)
        Y[ii, jj] = Ye
        dXp[ii, jj] = dXe
    out = np.zeros((n, H)); dx = np.zeros((n, H))
    for j in range(k):
        out += w[tokens, j][:, None] * Y[:, j]
        dx += dXp[:, j]
        dgate[:, j] = np.einsum("th,th->t", dout_rows, Y[:, j])
    return {"out": _store_bf16(out, mirror), "dx": _store_bf16(dx, mirror),
            "dgate": _store_f32(dgate, mirror)}


def expert_grads(e, x, dout, ids, w, perm: Permutation, W, mirror=True) -> dict:
    """dW1[e], dW3[e], dW2[e] from the rows of expert e alone.

    x and dout may be arrays or callables t_list -> rows.
    """
    get = _weights_getter(W)
    a, b = int(perm.offsets[e]), int(perm.offsets[e + 1])
    toks = perm.row_src[a:b]
    slots = perm.row_slot[a:b]
    X = x(toks) if callable(x) else np.asarray(x, dtype=np.float64)[toks]
    D = dout(toks) if callable(dout) else np.asarray(dout, dtype=np.float64)[toks]
    W1e, W3e, W2e = get(e)
    G, U, h, Y = expert_forward(X, W1e, W3e, W2e, mirror)
    dY = _store_bf16(np.asarray(w, dtype=np.float64)[toks, slots][:, None] * D, mirror)
    dG, dU, _ = expert_backward(dY, G, U, W1e, W3e, W2e, mirror)
    dW1, dW3, dW2 = expert_wgrad(X, h, dY, dG, dU, mirror)
    return {"dW1": dW1, "dW3": dW3, "dW2": dW2}
