"""Plain, slow fp64 CPU oracle of the Mixtral sparse-MoE feed-forward layer.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.  It
shares no code with the CUDA library; the only thing both sides use is the
seeded input generator in ``moe_workloads``.

What it computes (per token t, independently), following the pages:

  * "The Evolving Transformer - 05 Mixtral", section 05 (MoE router + MoE):
    the layer output is the gate-weighted sum over the top-k experts,
    y = sum_j w_j * E_{i_j}(x), with (w, i) from the router.
  * Same page, section 05, class MoERouter: logits G(x) = x Wg^T (bias-free
    linear d -> E), a softmax over all E logits, top-k of the probabilities
    (sorted descending), then the k weights renormalised to sum to 1.
  * Same page, section 04 (SwiGLU): each expert is three bias-free linear
    maps, down(silu(gate(x)) * up(x)).  The tutorial names them w1 (gate),
    w2 (up), w3 (down); this library names them W1 (gate), W3 (up), W2 (down).
  * Same page, section 05, class MoE: the output starts at zero; for each
    slot j and each expert e, the tokens whose slot-j expert is e are passed
    through expert e and added with their slot-j weight.
  * Same page, section 03 (RMSNorm) and section 06 (Block): the block form is
    x + MoE(RMSNorm(x)) with RMSNorm(x) = x * (mean(x^2) + eps)^-1/2 * gamma.

Readings where the pages are silent:
  * Equal router probabilities keep the lower expert index first.
  * In the block form the normalised activation is rounded once to bf16
    (round to nearest even) before the router and the experts, as a bf16
    layer stores it.  That rounding is a quantisation decision, so it is
    taken from an fp32 value, the precision the block workload fixes for
    its norm ("fp32 norm"); everything else stays in fp64.

Parity pins for every function here live in tests/test_oracle_pins.py.
"""
from __future__ import annotations

import numpy as np

try:  # torch tensors are accepted as inputs; the arithmetic is numpy fp64.
    import torch
except ImportError:  # pragma: no cover
    torch = None


def f64(a) -> np.ndarray:
    """Exact fp64 copy of a numpy array or a CPU torch tensor (any float dtype)."""
    if torch is not None and isinstance(a, torch.Tensor):
        return a.detach().to("cpu", torch.float64).numpy()
    return np.asarray(a, dtype=np.float64)


def round_to_bf16(v) -> np.ndarray:
    """Round fp64 values to the nearest bfloat16 value, ties to even.

    bfloat16 keeps 8 significant bits and fp32's exponent range; below the
    smallest normal (2^-126) the spacing stays 2^-133.
    """
    v = np.asarray(v, dtype=np.float64)
    m, e = np.frexp(v)  # v = m * 2^e, 0.5 <= |m| < 1
    e = np.maximum(e, -125)  # subnormal range: fixed spacing
    scale = np.ldexp(1.0, 8 - e)  # spacing of 8-bit significands at this binade
    return np.rint(v * scale) / scale  # np.rint rounds half to even


# ---------------------------------------------------------------- RMSNorm
def rmsnorm(x, gamma, eps) -> np.ndarray:
    """Section 03 (RMSNorm): x * (mean over features of x^2 + eps)^-1/2 * gamma."""
    x = f64(x)
    g = f64(gamma)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * g


def rmsnorm_fp32(x, gamma, eps) -> np.ndarray:
    """Section 03 (RMSNorm) in fp32 arithmetic: mean of squares, then
    (x * (mean + eps)^-1/2) * gamma, every operation rounded to fp32."""
    x32 = f64(x).astype(np.float32)
    g32 = f64(gamma).astype(np.float32)
    ms = np.mean(x32 * x32, axis=-1, keepdims=True, dtype=np.float32)
    r = np.float32(1.0) / np.sqrt(ms + np.float32(eps))
    return (x32 * r) * g32


# ---------------------------------------------------------------- router
def router_logits(x, Wg) -> np.ndarray:
    """Section 05, MoERouter: the bias-free gate, l[t, e] = sum_c x[t, c] Wg[e, c]."""
    return f64(x) @ f64(Wg).T


def softmax(l, axis=-1) -> np.ndarray:
    z = l - np.max(l, axis=axis, keepdims=True)
    p = np.exp(z)
    return p / np.sum(p, axis=axis, keepdims=True)


def router(x, Wg, k):
    """Section 05, MoERouter.forward.

    Returns (w[T,k], idx[T,k], logits[T,E]): softmax over all E logits, the k
    largest probabilities in descending order (equal ones: lower index
    first), and those k probabilities divided by their sum.
    """
    logits = router_logits(x, Wg)
    prob = softmax(logits)
    order = np.argsort(-prob, axis=-1, kind="stable")[:, :k]
    w = np.take_along_axis(prob, order, axis=-1)
    w = w / np.sum(w, axis=-1, keepdims=True)
    return w, order.astype(np.int64), logits


# ---------------------------------------------------------------- experts
def silu(a) -> np.ndarray:
    """SiLU (swish): a * sigmoid(a) = a / (1 + exp(-a))."""
    return a / (1.0 + np.exp(-a))


def gate_up_preactivations(x, W1e, W3e):
    """Section 04, SwiGLUFeedForward: the two projections a = W1 x (gate) and
    b = W3 x (up) that the SwiGLU combines, each [n,F]."""
    x = f64(x)
    return x @ f64(W1e).T, x @ f64(W3e).T


def swiglu_hidden(x, W1e, W3e) -> np.ndarray:
    """Section 04, SwiGLUFeedForward: the hidden activation silu(W1 x) * (W3 x), [n,F]."""
    a, b = gate_up_preactivations(x, W1e, W3e)
    return silu(a) * b


def swiglu_expert(x, W1e, W3e, W2e) -> np.ndarray:
    """Section 04, SwiGLUFeedForward.forward: W2 (silu(W1 x) * (W3 x)).

    x[n,d]; W1e, W3e [F,d] (gate, up); W2e [d,F] (down).  Returns [n,d].
    """
    return swiglu_hidden(x, W1e, W3e) @ f64(W2e).T


# ---------------------------------------------------------------- dispatch
def dispatch(idx, E):
    """Group the (token, slot) pairs by expert, as section 05's MoE loop does
    when it selects the tokens routed to each expert.

    The flat pair index is f = t*k + j.  Returns (counts[E], offsets[E+1],
    row_src[T*k], slot_pos[T*k]): pairs sorted by expert with ties in
    ascending f (a stable sort), row_src[p] the source token of row p, and
    slot_pos[f] the row that pair f moved to.
    """
    idx = np.asarray(idx)
    k = idx.shape[1]
    flat = idx.reshape(-1)
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    order = np.argsort(flat, kind="stable")  # order[p] = pair at row p
    row_src = order // k
    slot_pos = np.empty_like(order)
    slot_pos[order] = np.arange(order.size)
    return counts, offsets, row_src, slot_pos


# ---------------------------------------------------------------- grouped steps
# The layer's steps on rows already grouped by expert (the order `dispatch`
# gives): rows offsets[e] .. offsets[e+1]-1 belong to expert e.  Section 05's
# MoE loop applies each expert to the tokens routed to it; these functions
# apply the same per-expert maps to those rows, one expert at a time.
def gate_up_projection(x_perm, offsets, W1, W3) -> np.ndarray:
    """Section 04, SwiGLUFeedForward, first half, per expert segment:
    h[p] = silu(W1_e x_perm[p]) * (W3_e x_perm[p]) for the rows p of expert e.
    Returns h[Tk,F]."""
    x_perm = f64(x_perm)
    offsets = np.asarray(offsets)
    out = np.zeros((x_perm.shape[0], W1.shape[1]))
    for e in range(W1.shape[0]):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            out[a:b] = swiglu_hidden(x_perm[a:b], W1[e], W3[e])
    return out


def down_projection(h, offsets, W2) -> np.ndarray:
    """Section 04, SwiGLUFeedForward, the down projection, per expert
    segment: y[p] = W2_e h[p] for the rows p of expert e.  h[Tk,F],
    W2[E,d,F]; returns y[Tk,d]."""
    h = f64(h)
    offsets = np.asarray(offsets)
    out = np.zeros((h.shape[0], W2.shape[1]))
    for e in range(W2.shape[0]):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            out[a:b] = h[a:b] @ f64(W2[e]).T
    return out


def combine(y_perm, slot_pos, w, residual=None) -> np.ndarray:
    """Section 05, class MoE: each token's output is the sum over its k
    slots of the slot's gate weight times the output of the slot's expert;
    section 06 (Block) adds the residual.  The output of pair (t, j) is row
    slot_pos[t*k + j] of y_perm.  Returns out[T,d]."""
    y = f64(y_perm)
    w = np.asarray(w, dtype=np.float64)
    T, k = w.shape
    pos = np.asarray(slot_pos).reshape(T, k)
    out = np.zeros((T, y.shape[1]))
    for j in range(k):
        out += w[:, j][:, None] * y[pos[:, j]]
    if residual is not None:
        out += f64(residual)
    return out


# ---------------------------------------------------------------- layer
def moe_forward_with_routing(x, W1, W3, W2, w, idx) -> np.ndarray:
    """Section 05, MoE.forward given the router's (w, idx).

    Output starts at zero; for each slot j, for each expert e, the tokens
    whose slot-j expert is e go through expert e and are added with weight
    w[:, j].  Experts that no token picked in a slot are skipped.
    """
    x = f64(x)
    w = np.asarray(w, dtype=np.float64)
    idx = np.asarray(idx)
    T = x.shape[0]
    E = W1.shape[0]
    d = W2.shape[1]
    out = np.zeros((T, d), dtype=np.float64)
    for j in range(idx.shape[1]):
        for e in range(E):
            mask = idx[:, j] == e
            if mask.any():
                y = swiglu_expert(x[mask], W1[e], W3[e], W2[e])
                out[mask] += w[mask, j][:, None] * y
    return out


def moe_forward(x, Wg, W1, W3, W2, k):
    """The sparse MoE layer: returns (out[T,d], w[T,k], idx[T,k], logits[T,E])."""
    w, idx, logits = router(x, Wg, k)
    return moe_forward_with_routing(x, W1, W3, W2, w, idx), w, idx, logits


def block_normed_input(x, gamma, eps) -> np.ndarray:
    """Section 06 (Block), MoE half: the bf16-rounded RMSNorm(x) fed to the MoE
    (the fp32 norm, rounded once)."""
    return round_to_bf16(rmsnorm_fp32(x, gamma, eps).astype(np.float64))


def block_forward(x, gamma, eps, Wg, W1, W3, W2, k):
    """Section 06 (Block), MoE half: x + MoE(RMSNorm(x)).

    Returns (out[T,d], w, idx, logits, xn); logits and routing are those of
    the normalised input xn.
    """
    xn = block_normed_input(x, gamma, eps)
    delta, w, idx, logits = moe_forward(xn, Wg, W1, W3, W2, k)
    return f64(x) + delta, w, idx, logits, xn


# ---------------------------------------------------------------- shapes
def expert_param_shapes(d, F):
    """Shapes of one expert's three bias-free matrices: gate, up, down."""
    return [(F, d), (F, d), (d, F)]


def moe_layer_param_count(d, F, E) -> int:
    """Parameters of one MoE layer: E experts plus the bias-free d->E gate."""
    per_expert = sum(a * b for a, b in expert_param_shapes(d, F))
    return E * per_expert + d * E


def moe_layer_active_param_count(d, F, E, k) -> int:
    """Parameters one token touches in an MoE layer: k experts and the gate."""
    per_expert = sum(a * b for a, b in expert_param_shapes(d, F))
    return k * per_expert + d * E


# ---------------------------------------------------------------- int8 weight-only experts
# KerasFormers Mixtral docs, "Lower memory": checkpoints may be loaded with
# the weights alone quantized to int8 while activations stay bf16.  The docs
# do not spell the scheme out; the reading taken here is the plain one for a
# weight-only int8 linear map: symmetric, one fp32 scale per output channel
# (per row of the nn.Linear weight), scale = max|row| / 127, codes rounded to
# nearest (ties to even) and clamped to [-127, 127].  The codes are integers
# decided by floating point, so they are decided in fp32 (IEEE division, as a
# GPU kernel computes them): s = fl32(amax / 127), q = rint(fl32(w / s)).
# A row of zeros has scale 0 and codes 0.
def quantize_int8_rows(W):
    """Per-row symmetric int8 quantisation of W[..., cols].

    Returns (q int8 with W's shape, s float32 with W's shape minus the last
    axis)."""
    w32 = f64(W).astype(np.float32)
    amax = np.max(np.abs(w32), axis=-1)
    s = (amax / np.float32(127.0)).astype(np.float32)
    safe = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
    q = np.rint((w32 / safe[..., None]).astype(np.float32))
    q = np.clip(q, -127, 127)
    q = np.where(s[..., None] > 0, q, 0.0)
    return q.astype(np.int8), s


def dequantize_int8_rows(q, s) -> np.ndarray:
    """The weight a quantised layer multiplies by: s[row] * q[row, col], exact in fp64."""
    return np.asarray(q, dtype=np.float64) * np.asarray(s, dtype=np.float64)[..., None]


def moe_forward_w8(x, Wg, q1, s1, q3, s3, q2, s2, k):
    """The sparse MoE layer with int8 expert weights: the router uses Wg as
    given; every expert matrix is its dequantised value s * q.  Returns
    (out[T,d], w[T,k], idx[T,k], logits[T,E])."""
    W1 = dequantize_int8_rows(q1, s1)
    W3 = dequantize_int8_rows(q3, s3)
    W2 = dequantize_int8_rows(q2, s2)
    return moe_forward(x, Wg, W1, W3, W2, k)


# ---------------------------------------------------------------- backward
# Mixtral 8x7B model reference page, Training: the experts and the router are
# trained together, so the layer is differentiated with respect to its input,
# the gate and every expert matrix.  The top-k choice is piecewise constant in
# the logits, so gradients flow through the k chosen logits only (through the
# softmax over them) and through the chosen experts.
def silu_grad(a) -> np.ndarray:
    """d/da [a * sigmoid(a)] = sigmoid(a) * (1 + a * (1 - sigmoid(a)))."""
    s = 1.0 / (1.0 + np.exp(-a))
    return s * (1.0 + a * (1.0 - s))


def moe_backward(x, Wg, W1, W3, W2, k, dout, idx=None, experts=None, with_scale=False, weight_grads=True):
    """Gradients of L = sum(out * dout) for out = moe_forward(x, ...).

    ``idx`` replaces the router's choice (the weights are then the softmax
    over the chosen logits), for scoring near-tie tokens; ``experts`` limits
    the expert weight gradients to those experts (the others stay zero), to
    bound memory at full size; ``weight_grads=False`` skips dW1, dW3 and dW2
    (returned as None), for the input gradient of a few tokens at full size
    (a token's dx depends on that token alone).  ``with_scale`` also returns, under the same
    keys with a "_scale" suffix, each output's sum of the absolute values of
    the terms it is summed from (through the chain), the quantity rounding-
    error bounds of a computation with rounded factors are proportional to.

    Returns dict(dx[T,d], dWg[E,d], dW1[E,F,d], dW3[E,F,d], dW2[E,d,F]) in fp64,
    following the chain rule step by step:
      dy_j = w_j dout             (each chosen expert's output gradient)
      dw_j = <dout, y_j>          (gate weight gradient)
      dl_j = w_j (dw_j - sum_i w_i dw_i)   (softmax over the k chosen logits)
      dh   = dy W2_e,  da = dh * b * silu'(a),  db = dh * silu(a)
      dx  += da W1_e + db W3_e + sum_j dl_j Wg[i_j]
      dW2_e += dy^T h,  dW1_e += da^T x,  dW3_e += db^T x,  dWg[i_j] += dl_j x
    """
    x = f64(x)
    dout = f64(dout)
    Wg = f64(Wg)
    T, d = x.shape
    E, F = W1.shape[0], W1.shape[1]
    if idx is None:
        w, idx, _ = router(x, Wg, k)
    else:
        idx = np.asarray(idx)
        w = softmax(np.take_along_axis(router_logits(x, Wg), idx, axis=1))
    keep = set() if not weight_grads else set(range(E)) if experts is None else set(experts)
    dx = np.zeros_like(x)
    dWg = np.zeros_like(Wg)
    dW1 = dW3 = dW2 = None
    if weight_grads:
        dW1, dW3, dW2 = np.zeros((E, F, d)), np.zeros((E, F, d)), np.zeros((E, d, F))
    dw = np.zeros((T, k))
    if with_scale:
        sx, sWg = np.zeros_like(x), np.zeros_like(Wg)
        s1 = s3 = s2 = None
        if weight_grads:
            s1, s3, s2 = np.zeros((E, F, d)), np.zeros((E, F, d)), np.zeros((E, d, F))
        sdw = np.zeros((T, k))
    for j in range(k):
        for e in range(E):
            rows = np.nonzero(idx[:, j] == e)[0]
            if rows.size == 0:
                continue
            xe = x[rows]
            W1e, W3e, W2e = f64(W1[e]), f64(W3[e]), f64(W2[e])
            a = xe @ W1e.T
            b = xe @ W3e.T
            h = silu(a) * b
            y = h @ W2e.T
            dw[rows, j] = np.sum(dout[rows] * y, axis=1)
            dy = w[rows, j][:, None] * dout[rows]
            dh = dy @ W2e
            da = dh * b * silu_grad(a)
            db = dh * silu(a)
            dx[rows] += da @ W1e + db @ W3e
            if e in keep:
                dW2[e] += dy.T @ h
                dW1[e] += da.T @ xe
                dW3[e] += db.T @ xe
            if with_scale:
                sdw[rows, j] = np.sum(np.abs(dout[rows] * y), axis=1)
                ada, adb, axe = np.abs(da), np.abs(db), np.abs(xe)
                sx[rows] += ada @ np.abs(W1e) + adb @ np.abs(W3e)
                if e in keep:
                    s2[e] += np.abs(dy).T @ np.abs(h)
                    s1[e] += ada.T @ axe
                    s3[e] += adb.T @ axe
    dl = w * (dw - np.sum(w * dw, axis=1, keepdims=True))
    for j in range(k):
        dx += dl[:, j][:, None] * Wg[idx[:, j]]
        np.add.at(dWg, idx[:, j], dl[:, j][:, None] * x)
    out = {"dx": dx, "dWg": dWg, "dW1": dW1, "dW3": dW3, "dW2": dW2}
    if with_scale:
        sdl = w * (sdw + np.sum(w * sdw, axis=1, keepdims=True))
        for j in range(k):
            sx += sdl[:, j][:, None] * np.abs(Wg[idx[:, j]])
            np.add.at(sWg, idx[:, j], sdl[:, j][:, None] * np.abs(x))
        out.update({"dx_scale": sx, "dWg_scale": sWg, "dW1_scale": s1, "dW3_scale": s3, "dW2_scale": s2})
    return out


def expert_grad_hidden_unit(xe, doute, we, W1e, W3e, W2e, f):
    """The expert weight gradients that touch one hidden unit f of one
    expert, from the rows routed to it: xe [n,d] (the tokens), doute [n,d]
    (their output gradients) and we [n] (their gate weights for this expert).
    The same chain rule as moe_backward, restricted to column f of h:
      a = xe W1e[f],  b = xe W3e[f],  h = silu(a) b          (each [n])
      dy = we dout,   dh = dy W2e[:, f]
      da = dh b silu'(a),  db = dh silu(a)
      dW1e[f, :] = da^T xe,  dW3e[f, :] = db^T xe,  dW2e[:, f] = dy^T h
    Each with its sum of absolute terms ("_scale"), as moe_backward's.  A
    hidden unit costs O(n d), so single rows and columns of the gradients can
    be checked at full size."""
    xe, doute = f64(xe), f64(doute)
    we = np.asarray(we, dtype=np.float64)
    a = xe @ f64(W1e[f])
    b = xe @ f64(W3e[f])
    h = silu(a) * b
    dy = we[:, None] * doute
    dh = dy @ f64(W2e[:, f])
    da = dh * b * silu_grad(a)
    db = dh * silu(a)
    axe = np.abs(xe)
    return {"dW1": da @ xe, "dW3": db @ xe, "dW2": dy.T @ h,
            "dW1_scale": np.abs(da) @ axe, "dW3_scale": np.abs(db) @ axe, "dW2_scale": np.abs(dy).T @ np.abs(h)}
