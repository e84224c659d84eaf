"""Checks that pin the fp64 oracle to facts other than itself.

Each ``pin_*`` takes an oracle namespace ``o`` (the real ``oracle.moe_oracle``
module, or a copy with a planted mistake) and raises on a mismatch.  The
expected values come from brute force on tiny inputs, pure-Python textbook
loops, closed forms, invariants of the layer, library routines for special
cases, and the parameter counts printed on the pages — never from the
oracle's own formulas retyped.

Sources (page title, section):
  * "The Evolving Transformer - 05 Mixtral", section 05 (MoE router + MoE),
    section 04 (SwiGLU), section 03 (RMSNorm), section 06 (Block),
    section 00 (Config).
  * KerasFormers Mixtral docs, MixtralModel argument table.
  * Mixtral 8x7B model reference page (46.7B total / 12.9B active).
"""
from __future__ import annotations

import itertools
import json
import math
import os

import mpmath
import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

mpmath.mp.dps = 40


def _rng(seed):
    return np.random.default_rng(seed)


def _tiny_layer(seed, T=40, d=12, F=10, E=8, scale=1.0):
    r = _rng(seed)
    return dict(
        x=r.standard_normal((T, d)) * scale,
        Wg=r.standard_normal((E, d)) / math.sqrt(d),
        W1=r.standard_normal((E, F, d)) / math.sqrt(d),
        W3=r.standard_normal((E, F, d)) / math.sqrt(d),
        W2=r.standard_normal((E, d, F)) / math.sqrt(F),
    )


def _py_dot(a, b):
    return math.fsum(float(u) * float(v) for u, v in zip(a, b))


def _py_silu(a):
    return a / (1.0 + math.exp(-a))


def _py_swiglu(xrow, W1e, W3e, W2e):
    """Textbook SwiGLU for one token with pure-Python loops (gate W1, up W3, down W2)."""
    F = len(W1e)
    h = []
    for f in range(F):
        a = _py_dot(xrow, W1e[f])
        b = _py_dot(xrow, W3e[f])
        h.append(_py_silu(a) * b)
    return [_py_dot(W2e[o], h) for o in range(len(W2e))]


# ------------------------------------------------------------------ router
def pin_router_logits_brute_force(o):
    """Gate logits equal the per-(token, expert) dot product, summed exactly."""
    L = _tiny_layer(1, T=6, d=7, E=5)
    got = o.router_logits(L["x"], L["Wg"])
    for t in range(6):
        for e in range(5):
            want = _py_dot(L["x"][t], L["Wg"][e])
            assert abs(got[t, e] - want) <= 1e-13 * max(1.0, abs(want)), (t, e)


def pin_topk_set_brute_force(o):
    """The chosen set maximises the sum of logits over all C(E,k) subsets."""
    for k in (1, 2, 3):
        L = _tiny_layer(2 + k, T=60)
        _, idx, _ = o.router(L["x"], L["Wg"], k)
        logits = L["x"] @ L["Wg"].T  # exact enough: subsets differ by >> 1e-12 here
        for t in range(60):
            best = max(itertools.combinations(range(8), k), key=lambda s: sum(logits[t, list(s)]))
            assert set(int(i) for i in idx[t]) == set(best), (k, t)


def pin_slot_order_descending(o):
    """Slot 0 carries the largest weight (top-k output is sorted)."""
    L = _tiny_layer(7, T=80)
    w, idx, _ = o.router(L["x"], L["Wg"], 3)
    assert np.all(w[:, 0] >= w[:, 1]) and np.all(w[:, 1] >= w[:, 2])
    logits = L["x"] @ L["Wg"].T
    sel = np.take_along_axis(logits, idx, axis=1)
    assert np.all(sel[:, 0] >= sel[:, 1]) and np.all(sel[:, 1] >= sel[:, 2])


def pin_gate_weights_top2_sigmoid(o):
    """k=2: renormalised softmax over the pair is sigmoid of the logit gap.

    softmax(l)_i / (softmax(l)_i + softmax(l)_j) = 1 / (1 + exp(l_j - l_i)):
    the normaliser over all E cancels.  Checked to 40 digits with mpmath.
    """
    L = _tiny_layer(11, T=50)
    w, idx, _ = o.router(L["x"], L["Wg"], 2)
    for t in range(50):
        li = [mpmath.fsum(mpmath.mpf(float(a)) * mpmath.mpf(float(b)) for a, b in zip(L["x"][t], L["Wg"][e]))
              for e in (int(idx[t, 0]), int(idx[t, 1]))]
        w0 = 1 / (1 + mpmath.exp(li[1] - li[0]))
        assert abs(w[t, 0] - float(w0)) < 1e-14, t
        assert abs(w[t, 1] - float(1 - w0)) < 1e-14, t


def pin_gate_weights_invariants(o):
    """Weights are positive and sum to one for every k."""
    for k in (1, 2, 4, 8):
        L = _tiny_layer(13 + k, T=30)
        w, _, _ = o.router(L["x"], L["Wg"], k)
        assert np.all(w > 0)
        assert np.allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-15)


def pin_k1_weight_is_one(o):
    """k=1: the single weight is exactly 1 and the layer is the argmax expert."""
    L = _tiny_layer(17, T=20)
    out, w, idx, _ = o.moe_forward(L["x"], L["Wg"], L["W1"], L["W3"], L["W2"], 1)
    assert np.all(w == 1.0)
    logits = L["x"] @ L["Wg"].T
    for t in range(20):
        e = int(np.argmax(logits[t]))
        assert int(idx[t, 0]) == e
        want = _py_swiglu(L["x"][t], L["W1"][e], L["W3"][e], L["W2"][e])
        assert np.allclose(out[t], want, rtol=1e-12, atol=1e-14)


def pin_equal_logits_split_evenly(o):
    """Two identical, dominant gate rows: weights 0.5/0.5, lower index first."""
    L = _tiny_layer(19, T=16)
    Wg = L["Wg"].copy()
    Wg[2] = Wg[5] = 1.0  # the same row twice
    x = np.abs(L["x"]) + 0.5  # logits of rows 2/5 are the largest
    w, idx, _ = o.router(x, Wg, 2)
    assert np.all(idx[:, 0] == 2) and np.all(idx[:, 1] == 5)
    assert np.all(w == 0.5)


def pin_two_experts_select_both(o):
    """E=2, k=2 selects both experts, larger logit first."""
    L = _tiny_layer(23, T=25, E=2)
    w, idx, _ = o.router(L["x"], L["Wg"], 2)
    assert np.all(np.sort(idx, axis=1) == np.array([0, 1]))


def pin_router_topk_softmax_restatement(o):
    """Top-k of the logits, then a softmax over the k chosen (this library's
    GPU formulation) equals softmax-over-all, top-k, renormalise."""
    L = _tiny_layer(29, T=200)
    for k in (2, 3):
        w, idx, _ = o.router(L["x"], L["Wg"], k)
        logits = L["x"] @ L["Wg"].T
        for t in range(200):
            order = sorted(range(8), key=lambda e: (-logits[t, e], e))[:k]
            m = logits[t, order[0]]
            ex = [math.exp(logits[t, e] - m) for e in order]
            s = math.fsum(ex)
            assert [int(i) for i in idx[t]] == order
            assert np.allclose(w[t], [v / s for v in ex], rtol=0, atol=1e-14)


def pin_dispatch_brute_force(o):
    """Rows grouped per expert in ascending (token, slot), by plain loops."""
    r = _rng(5)
    for k, E, T in ((2, 8, 37), (1, 3, 10), (3, 5, 0), (2, 8, 1)):
        idx = np.stack([r.permutation(E)[:k] for _ in range(T)]) if T else np.zeros((0, k), dtype=np.int64)
        counts, offsets, row_src, slot_pos = o.dispatch(idx, E)
        rows = []
        for e in range(E):
            for t in range(T):
                for j in range(k):
                    if idx[t, j] == e:
                        rows.append((t, j))
        assert list(counts) == [sum(1 for t in range(T) for j in range(k) if idx[t, j] == e) for e in range(E)]
        assert list(offsets) == [sum(counts[:e]) for e in range(E + 1)]
        assert [int(v) for v in row_src] == [t for t, _ in rows]
        for p, (t, j) in enumerate(rows):
            assert slot_pos[t * k + j] == p


def _segments(counts):
    """Offsets of consecutive expert segments with the given row counts, and
    the expert of every row, by plain loops."""
    offsets, owner = [0], []
    for e, n in enumerate(counts):
        offsets.append(offsets[-1] + n)
        owner += [e] * n
    return offsets, owner


def pin_gate_up_projection_brute_force(o):
    """Grouped gate/up: each row meets its own expert's W1 and W3 only, by
    pure-Python loops; empty segments and a segment at the end included."""
    r = _rng(34)
    counts = [2, 0, 3, 1, 0]
    offsets, owner = _segments(counts)
    E, F, d = len(counts), 4, 3
    x = r.standard_normal((offsets[-1], d))
    W1, W3 = r.standard_normal((E, F, d)), r.standard_normal((E, F, d))
    got = o.gate_up_projection(x, offsets, W1, W3)
    assert got.shape == (offsets[-1], F)
    for p, e in enumerate(owner):
        for f in range(F):
            want = _py_silu(_py_dot(x[p], W1[e][f])) * _py_dot(x[p], W3[e][f])
            assert abs(got[p, f] - want) < 1e-13 * max(1.0, abs(want)), (p, f)


def pin_down_projection_brute_force(o):
    """Grouped down projection: y[p][c] = sum_f h[p][f] W2[e][c][f] with e the
    expert owning row p, by pure-Python loops (W2 is [E, d, F]: output
    channel first)."""
    r = _rng(35)
    counts = [0, 3, 2, 0, 1]
    offsets, owner = _segments(counts)
    E, F, d = len(counts), 5, 3
    h = r.standard_normal((offsets[-1], F))
    W2 = r.standard_normal((E, d, F))
    got = o.down_projection(h, offsets, W2)
    assert got.shape == (offsets[-1], d)
    for p, e in enumerate(owner):
        for c in range(d):
            want = _py_dot(h[p], W2[e][c])
            assert abs(got[p, c] - want) < 1e-13 * max(1.0, abs(want)), (p, c)


def pin_combine_brute_force(o):
    """Combine: out[t] = sum_j w[t][j] y[slot_pos[t*k+j]] (+ residual[t]), by
    pure-Python loops over tokens and slots, with a shuffled slot_pos."""
    r = _rng(36)
    T, k, d = 5, 3, 4
    y = r.standard_normal((T * k, d))
    pos = r.permutation(T * k)
    w = r.uniform(0.1, 1.0, (T, k))
    res = r.standard_normal((T, d))
    for residual in (None, res):
        got = o.combine(y, pos, w, residual)
        for t in range(T):
            for c in range(d):
                terms = [w[t][j] * y[pos[t * k + j]][c] for j in range(k)]
                if residual is not None:
                    terms.append(residual[t][c])
                want = math.fsum(terms)
                assert abs(got[t, c] - want) < 1e-13 * max(1.0, abs(want)), (t, c)


def pin_grouped_steps_compose_to_layer(o):
    """dispatch -> gather -> gate_up_projection -> down_projection -> combine
    with the router's (w, idx) gives the layer by brute force: the grouped
    steps are the layer of section 05, reordered."""
    L = _tiny_layer(61, T=14, d=6, F=5)
    k = 2
    w, idx, _ = o.router(L["x"], L["Wg"], k)
    counts, offsets, row_src, slot_pos = o.dispatch(idx, 8)
    h = o.gate_up_projection(L["x"][row_src], offsets, L["W1"], L["W3"])
    y = o.down_projection(h, offsets, L["W2"])
    out = o.combine(y, slot_pos, w)
    for t in range(14):
        lg = [_py_dot(L["x"][t], L["Wg"][e]) for e in range(8)]
        i0, i1 = sorted(max(itertools.combinations(range(8), 2), key=lambda s: lg[s[0]] + lg[s[1]]),
                        key=lambda e: -lg[e])
        w0 = 1.0 / (1.0 + math.exp(lg[i1] - lg[i0]))
        y0 = _py_swiglu(L["x"][t], L["W1"][i0], L["W3"][i0], L["W2"][i0])
        y1 = _py_swiglu(L["x"][t], L["W1"][i1], L["W3"][i1], L["W2"][i1])
        assert np.allclose(out[t], [w0 * a + (1.0 - w0) * b for a, b in zip(y0, y1)], rtol=1e-12, atol=1e-14), t


def pin_swiglu_hidden_textbook(o):
    """The hidden activation silu(W1 x) * (W3 x) by pure-Python loops."""
    r = _rng(33)
    x = r.standard_normal((3, 4))
    W1, W3 = r.standard_normal((5, 4)), r.standard_normal((5, 4))
    got = o.swiglu_hidden(x, W1, W3)
    for n in range(3):
        for f in range(5):
            want = _py_silu(_py_dot(x[n], W1[f])) * _py_dot(x[n], W3[f])
            assert abs(got[n, f] - want) < 1e-13 * max(1.0, abs(want))


# ------------------------------------------------------------------ experts
def pin_silu_closed_form(o):
    """silu(0)=0, silu(ln 3) = 0.75 ln 3, silu(-ln 3) = -0.25 ln 3."""
    l3 = math.log(3.0)
    got = o.silu(np.array([0.0, l3, -l3, 40.0]))
    assert got[0] == 0.0
    assert abs(got[1] - 0.75 * l3) < 1e-15
    assert abs(got[2] + 0.25 * l3) < 1e-15
    assert abs(got[3] - 40.0) < 1e-12


def pin_swiglu_textbook(o):
    """SwiGLU on 2 tokens x d=3 x F=4 against pure-Python loops."""
    r = _rng(31)
    x = r.standard_normal((2, 3))
    W1, W3, W2 = r.standard_normal((4, 3)), r.standard_normal((4, 3)), r.standard_normal((3, 4))
    got = o.swiglu_expert(x, W1, W3, W2)
    for n in range(2):
        assert np.allclose(got[n], _py_swiglu(x[n], W1, W3, W2), rtol=1e-13, atol=1e-15)


def pin_swiglu_hand_values(o):
    """A hand-worked SwiGLU: gate pre-activations ln 3 and 0, up 2 and 5.

    x = [1, 0]; W1 rows give a = [ln 3, 0]; W3 rows give b = [2, 5];
    h = [0.75 ln 3 * 2, 0 * 5] = [1.5 ln 3, 0]; W2 = [[1, 7], [-2, 3]]
    gives y = [1.5 ln 3, -3 ln 3].
    """
    l3 = math.log(3.0)
    x = np.array([[1.0, 0.0]])
    W1 = np.array([[l3, 9.0], [0.0, -4.0]])
    W3 = np.array([[2.0, 1.0], [5.0, 8.0]])
    W2 = np.array([[1.0, 7.0], [-2.0, 3.0]])
    y = o.swiglu_expert(x, W1, W3, W2)[0]
    assert abs(y[0] - 1.5 * l3) < 1e-14 and abs(y[1] + 3.0 * l3) < 1e-14


def pin_dense_reduction(o):
    """E=1, k=1 is exactly the dense SwiGLU block of Mistral (section 04)."""
    L = _tiny_layer(37, T=9, d=5, F=6, E=1)
    out, w, idx, _ = o.moe_forward(L["x"], L["Wg"], L["W1"], L["W3"], L["W2"], 1)
    assert np.all(idx == 0) and np.all(w == 1.0)
    for t in range(9):
        assert np.allclose(out[t], _py_swiglu(L["x"][t], L["W1"][0], L["W3"][0], L["W2"][0]),
                           rtol=1e-12, atol=1e-14)


def pin_identical_experts_reduce_to_one(o):
    """All experts equal: any routing gives the single SwiGLU (weights sum to 1)."""
    L = _tiny_layer(41, T=30, d=6, F=5)
    for k in (2, 3):
        W1 = np.repeat(L["W1"][:1], 8, axis=0)
        W3 = np.repeat(L["W3"][:1], 8, axis=0)
        W2 = np.repeat(L["W2"][:1], 8, axis=0)
        out, _, _, _ = o.moe_forward(L["x"], L["Wg"], W1, W3, W2, k)
        for t in range(30):
            assert np.allclose(out[t], _py_swiglu(L["x"][t], W1[0], W3[0], W2[0]), rtol=1e-12, atol=1e-14)


def pin_zero_input_zero_output(o):
    L = _tiny_layer(43, T=5)
    out, _, _, _ = o.moe_forward(np.zeros_like(L["x"]), L["Wg"], L["W1"], L["W3"], L["W2"], 2)
    assert np.all(out == 0.0)


def pin_down_projection_linear(o):
    """Scaling every W2 by c scales the output by c; the routing does not move."""
    L = _tiny_layer(47, T=40)
    a, wa, ia, _ = o.moe_forward(L["x"], L["Wg"], L["W1"], L["W3"], L["W2"], 2)
    b, wb, ib, _ = o.moe_forward(L["x"], L["Wg"], L["W1"], L["W3"], -3.5 * L["W2"], 2)
    assert np.array_equal(ia, ib) and np.array_equal(wa, wb)
    assert np.allclose(b, -3.5 * a, rtol=1e-13, atol=1e-15)


def pin_token_permutation_equivariance(o):
    """Permuting the tokens permutes the output rows the same way."""
    L = _tiny_layer(53, T=64)
    perm = _rng(54).permutation(64)
    a, _, _, _ = o.moe_forward(L["x"], L["Wg"], L["W1"], L["W3"], L["W2"], 2)
    b, _, _, _ = o.moe_forward(L["x"][perm], L["Wg"], L["W1"], L["W3"], L["W2"], 2)
    assert np.allclose(b, a[perm], rtol=1e-13, atol=1e-15)


def pin_layer_brute_force(o):
    """Whole layer on tiny inputs: top-2 by brute force, weights by the sigmoid
    form, experts by textbook loops, summed per token."""
    L = _tiny_layer(59, T=12, d=6, F=5)
    out, _, _, _ = o.moe_forward(L["x"], L["Wg"], L["W1"], L["W3"], L["W2"], 2)
    for t in range(12):
        lg = [_py_dot(L["x"][t], L["Wg"][e]) for e in range(8)]
        pair = max(itertools.combinations(range(8), 2), key=lambda s: lg[s[0]] + lg[s[1]])
        i0, i1 = sorted(pair, key=lambda e: -lg[e])
        w0 = 1.0 / (1.0 + math.exp(lg[i1] - lg[i0]))
        y0 = _py_swiglu(L["x"][t], L["W1"][i0], L["W3"][i0], L["W2"][i0])
        y1 = _py_swiglu(L["x"][t], L["W1"][i1], L["W3"][i1], L["W2"][i1])
        want = [w0 * a + (1.0 - w0) * b for a, b in zip(y0, y1)]
        assert np.allclose(out[t], want, rtol=1e-12, atol=1e-14), t


# ------------------------------------------------------------------ norm / block
def pin_rmsnorm_closed_form(o):
    """Constant row c with gamma=1: every output is c / sqrt(c^2 + eps)."""
    for c in (0.3, -2.0, 1e-3):
        x = np.full((1, 16), c)
        got = o.rmsnorm(x, np.ones(16), 1e-5)
        assert np.allclose(got, c / math.sqrt(c * c + 1e-5), rtol=1e-15, atol=0)


def pin_rmsnorm_mpmath(o):
    """Random rows and gamma against a 40-digit evaluation of the definition."""
    r = _rng(61)
    x = r.standard_normal((3, 10))
    g = 1.0 + 0.02 * r.standard_normal(10)
    got = o.rmsnorm(x, g, 1e-5)
    for t in range(3):
        ms = mpmath.fsum(mpmath.mpf(float(v)) ** 2 for v in x[t]) / 10
        inv = 1 / mpmath.sqrt(ms + mpmath.mpf(1e-5))
        for c in range(10):
            assert abs(got[t, c] - float(mpmath.mpf(float(x[t, c])) * inv * mpmath.mpf(float(g[c])))) < 1e-15


def pin_rmsnorm_fp32_within_rounding(o):
    """The fp32 norm agrees with the exact (fp64) one: after the bf16 rounding
    the two differ by at most one bf16 step, in a tiny fraction of elements."""
    r = _rng(63)
    x = torch.from_numpy(r.standard_normal((64, 512))).to(torch.bfloat16)
    g = torch.from_numpy(1.0 + 0.02 * r.standard_normal(512)).to(torch.bfloat16)
    exact = o.rmsnorm(x, g, 1e-5)
    f32 = o.rmsnorm_fp32(x, g, 1e-5).astype(np.float64)
    assert np.max(np.abs(f32 - exact) / np.abs(exact)) < 2e-6  # a few fp32 rounding steps
    a, b = o.round_to_bf16(exact), o.block_normed_input(x, g, 1e-5)
    step = np.ldexp(1.0, np.frexp(np.abs(a))[1] - 8)
    assert np.all(np.abs(a - b) <= step) and np.mean(a != b) < 1e-3


def pin_round_to_bf16(o):
    """fp64 -> bf16 rounding: hand ties, and torch's fp32 -> bf16 on fp32 inputs."""
    one = 1.0
    cases = {
        one + 2.0 ** -8: 1.0,  # tie, keep even significand
        one + 3 * 2.0 ** -8: one + 2.0 ** -6,  # tie, round up to even
        one + 2.0 ** -8 + 2.0 ** -30: one + 2.0 ** -7,  # just above the tie
        -(one + 2.0 ** -8): -1.0,
        0.0: 0.0,
    }
    for v, want in cases.items():
        assert o.round_to_bf16(np.array([v]))[0] == want, v
    r = _rng(67)
    v32 = (r.standard_normal(20000) * np.exp(r.uniform(-20, 20, 20000))).astype(np.float32)
    want = torch.from_numpy(v32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(o.round_to_bf16(v32.astype(np.float64)), want)


def pin_block_residual(o):
    """gamma = 0 makes the normalised input zero, so the block returns x."""
    L = _tiny_layer(71, T=10)
    out, _, _, _, xn = o.block_forward(L["x"], np.zeros(12), 1e-5, L["Wg"], L["W1"], L["W3"], L["W2"], 2)
    assert np.all(xn == 0.0)
    assert np.array_equal(out, L["x"])


def pin_block_uses_normalised_input(o):
    """The block routes on RMSNorm(x): scaling a row by 8 (exact in binary)
    leaves its routing unchanged when eps is negligible, and the MoE delta
    is the layer applied to the bf16-rounded normalised row."""
    L = _tiny_layer(73, T=20, scale=1.0)
    g = np.ones(12)
    a, _, ia, _, xa = o.block_forward(L["x"], g, 0.0, L["Wg"], L["W1"], L["W3"], L["W2"], 2)
    b, _, ib, _, xb = o.block_forward(8.0 * L["x"], g, 0.0, L["Wg"], L["W1"], L["W3"], L["W2"], 2)
    assert np.array_equal(ia, ib)
    assert np.allclose(a - L["x"], b - 8.0 * L["x"], rtol=1e-12, atol=1e-12)
    # every normalised value is a bf16 value
    assert np.array_equal(xa, torch.from_numpy(xa).to(torch.bfloat16).to(torch.float64).numpy())


# ------------------------------------------------------------------ shapes
def pin_parameter_counts_match_pages(o):
    """The 3-matrix bias-free SwiGLU experts at the pages' sizes reproduce the
    pages' ~46.7B total and ~12.9B active parameters."""
    with open(os.path.join(GOLDEN, "mixtral_8x7b_shapes.json")) as f:
        g = {k: v["value"] for k, v in json.load(f).items() if not k.startswith("_")}
    d, F, E, k, N = g["d_model"], g["d_ff"], g["num_experts"], g["top_k"], g["num_layers"]
    head = d // g["num_heads"]
    attn = 2 * d * d + 2 * d * (g["num_kv_heads"] * head)  # Wq, Wo; Wk, Wv
    norms = 2 * d
    emb = g["vocab_size"] * d * (1 if g["tie_embeddings"] else 2)
    total = N * (o.moe_layer_param_count(d, F, E) + attn + norms) + emb + d
    active = N * (o.moe_layer_active_param_count(d, F, E, k) + attn + norms) + emb + d
    assert round(total / 1e9, 1) == g["total_params_billion_1dp"], total
    assert round(active / 1e9, 1) == g["active_params_billion_1dp"], active
    assert o.moe_layer_param_count(d, F, E) == 1_409_318_912


# ------------------------------------------------------------------ int8 weight-only experts
# KerasFormers Mixtral docs, "Lower memory": weights alone quantised to int8.
# Reading: symmetric, one scale per output row, s = max|row| / 127, codes
# rounded half to even and clamped to [-127, 127].
def _bf16_rows(seed, rows, cols, scale=0.02):
    r = _rng(seed)
    w = torch.from_numpy(r.standard_normal((rows, cols)) * scale).to(torch.bfloat16)
    return w.to(torch.float64).numpy()


def pin_int8_hand_values(o):
    """Hand-worked rows (tests/golden/int8_rows_hand.json): ties to even, the
    127 divisor, a zero row."""
    with open(os.path.join(GOLDEN, "int8_rows_hand.json")) as f:
        rows = json.load(f)["rows"]
    for row in rows:
        q, s = o.quantize_int8_rows(np.array([row["w"]]))
        assert q.dtype == np.int8
        assert q[0].tolist() == row["q"], (row["w"], q[0].tolist())
        assert float(s[0]) == row["scale"], (row["w"], float(s[0]))


def pin_int8_exact_rational(o):
    """Every code is the integer nearest to w / s computed in exact rational
    arithmetic (ties to even), except where w / s lies within fp32 rounding of
    a midpoint; the scale is max|row| / 127 to fp32 rounding; the amax
    element gets +-127 with its sign."""
    from fractions import Fraction
    W = _bf16_rows(81, 24, 40)
    W[3] = 0.0
    q, s = o.quantize_int8_rows(W)
    assert q.shape == W.shape and s.shape == (24,)
    for i in range(W.shape[0]):
        amax = max(abs(Fraction(float(v))) for v in W[i])
        if amax == 0:
            assert s[i] == 0 and not q[i].any()
            continue
        si = Fraction(float(s[i]))
        assert abs(si - amax / 127) <= amax / 127 * Fraction(1, 1 << 23), i
        j = int(np.argmax(np.abs(W[i])))
        assert int(q[i, j]) == (127 if W[i, j] > 0 else -127), i
        for c in range(W.shape[1]):
            v = Fraction(float(W[i, c])) / si
            n = math.floor(v)
            frac = v - n
            if abs(frac - Fraction(1, 2)) <= abs(v) * Fraction(1, 1 << 22):
                assert int(q[i, c]) in (n, n + 1), (i, c)
                continue
            want = n + 1 if frac > Fraction(1, 2) else n
            want = max(-127, min(127, want))
            assert int(q[i, c]) == want, (i, c, float(v), int(q[i, c]))


def pin_int8_error_bound(o):
    """|w - s q| <= s / 2 (plus fp32 rounding of the quotient) for every
    element, |q| <= 127, on Mixtral-like rows of 4096."""
    W = _bf16_rows(83, 16, 4096)
    q, s = o.quantize_int8_rows(W)
    assert np.all(np.abs(q.astype(np.int64)) <= 127)
    err = np.abs(W - q.astype(np.float64) * s.astype(np.float64)[:, None])
    assert np.all(err <= s[:, None] * (0.5 + 127 * 2.0 ** -23))
    assert np.all(np.abs(o.dequantize_int8_rows(q, s) - W) <= s[:, None] * (0.5 + 127 * 2.0 ** -23))


def pin_int8_symmetry_scaling_rows(o):
    """Negating w negates q; scaling a row by 2^j scales s by 2^j and keeps q;
    each row is quantised on its own (per output channel, not per column)."""
    W = _bf16_rows(85, 12, 64)
    q, s = o.quantize_int8_rows(W)
    qn, sn = o.quantize_int8_rows(-W)
    assert np.array_equal(qn, -q) and np.array_equal(sn, s)
    for j in (-3, 5):
        qj, sj = o.quantize_int8_rows(W * 2.0 ** j)
        assert np.array_equal(qj, q) and np.array_equal(sj, (s * np.float32(2.0 ** j)).astype(np.float32))
    for i in range(12):
        qi, si = o.quantize_int8_rows(W[i:i + 1])
        assert np.array_equal(qi[0], q[i]) and si[0] == s[i]
    W3 = np.stack([W, 4.0 * W])
    q3, s3 = o.quantize_int8_rows(W3)
    assert np.array_equal(q3[0], q) and np.array_equal(q3[1], q) and np.array_equal(s3[1], 4 * s)


def pin_w8_layer_brute_force(o):
    """The int8-weight layer is the layer of the dequantised weights s * q,
    checked token by token with pure-Python loops; and it stays within the
    quantisation error of the unquantised layer."""
    L = _tiny_layer(87, T=8, d=12, F=10, E=4)
    q1, s1 = o.quantize_int8_rows(L["W1"])
    q3, s3 = o.quantize_int8_rows(L["W3"])
    q2, s2 = o.quantize_int8_rows(L["W2"])
    out, w, idx, _ = o.moe_forward_w8(L["x"], L["Wg"], q1, s1, q3, s3, q2, s2, 2)

    def deq(q, s, e):
        return [[float(s[e, r]) * int(q[e, r, c]) for c in range(q.shape[2])] for r in range(q.shape[1])]

    for t in range(8):
        logits = [_py_dot(L["x"][t], L["Wg"][e]) for e in range(4)]
        top = sorted(range(4), key=lambda e: -logits[e])[:2]
        z = [math.exp(logits[e] - logits[top[0]]) for e in top]
        want = [0.0] * 12
        for j, e in enumerate(top):
            y = _py_swiglu(L["x"][t], deq(q1, s1, e), deq(q3, s3, e), deq(q2, s2, e))
            want = [a + z[j] / sum(z) * b for a, b in zip(want, y)]
        assert np.allclose(out[t], want, rtol=1e-12, atol=1e-14), t
    ref, _, _, _ = o.moe_forward(L["x"], L["Wg"], L["W1"], L["W3"], L["W2"], 2)
    assert np.linalg.norm(out - ref) / np.linalg.norm(ref) < 0.03


# ------------------------------------------------------------------ backward
# Mixtral 8x7B model reference page, Training: experts and router are trained
# together.  The gradients are pinned to central finite differences of the
# oracle's own forward (a computation that shares no step with the backward's
# chain rule), to library autodiff for the dense special case, and to
# invariants.
def _loss_grad_fd(o, L, k, dout, name, eps=1e-6):
    args = {n: L[n] for n in ("x", "Wg", "W1", "W3", "W2")}
    base = args[name]
    fd = np.zeros_like(base)
    for i in np.ndindex(base.shape):
        for sgn in (1.0, -1.0):
            p = base.copy()
            p[i] += sgn * eps
            a = dict(args)
            a[name] = p
            out = o.moe_forward(a["x"], a["Wg"], a["W1"], a["W3"], a["W2"], k)[0]
            fd[i] += sgn * np.sum(out * dout)
    return fd / (2 * eps)


def pin_backward_finite_differences(o):
    """Every gradient equals central finite differences of the forward (the
    routing has clear gaps, so no top-k choice flips within +-eps)."""
    L = _tiny_layer(91, T=5, d=6, F=7, E=4)
    k = 2
    logits = L["x"] @ L["Wg"].T
    srt = -np.sort(-logits, axis=1)
    assert np.min(srt[:, 1] - srt[:, 2]) > 1e-3
    dout = _rng(92).standard_normal((5, 6))
    g = o.moe_backward(L["x"], L["Wg"], L["W1"], L["W3"], L["W2"], k, dout)
    for name in ("x", "Wg", "W1", "W3", "W2"):
        fd = _loss_grad_fd(o, L, k, dout, name)
        got = g["d" + name]
        assert got.shape == fd.shape, name
        assert np.max(np.abs(got - fd)) <= 1e-7 * max(1.0, np.max(np.abs(fd))), name


def pin_backward_silu_derivative(o):
    """silu'(a) against a 40-digit numerical derivative, and its closed values
    silu'(0) = 1/2 and silu'(a) -> 1 (a -> +inf), -> 0 (a -> -inf)."""
    pts = [-6.0, -1.3, -0.2, 0.0, 0.7, 2.5, 9.0]
    got = o.silu_grad(np.array(pts))
    for a, gv in zip(pts, got):
        want = mpmath.diff(lambda t: t / (1 + mpmath.exp(-t)), mpmath.mpf(a))
        assert abs(gv - float(want)) < 1e-14, a
    assert o.silu_grad(np.array([0.0]))[0] == 0.5
    assert abs(o.silu_grad(np.array([40.0]))[0] - 1.0) < 1e-12
    assert abs(o.silu_grad(np.array([-40.0]))[0]) < 1e-12


def pin_backward_scale_bounds_gradient(o):
    """The sum of absolute terms bounds each gradient element (triangle
    inequality) and is zero exactly where no term contributes."""
    L = _tiny_layer(97, T=10, d=8, F=6, E=4)
    g = o.moe_backward(L["x"], L["Wg"], L["W1"], L["W3"], L["W2"], 2, _rng(98).standard_normal((10, 8)),
                       with_scale=True)
    for n in ("dx", "dWg", "dW1", "dW3", "dW2"):
        assert np.all(np.abs(g[n]) <= g[n + "_scale"] * (1 + 1e-12) + 1e-300), n
        assert np.all(g[n][g[n + "_scale"] == 0] == 0), n


def pin_backward_linear_in_dout(o):
    """The gradients are linear in the output gradient."""
    L = _tiny_layer(93, T=12, d=8, F=6, E=4)
    r = _rng(94)
    d1, d2 = r.standard_normal((12, 8)), r.standard_normal((12, 8))
    g1 = o.moe_backward(L["x"], L["Wg"], L["W1"], L["W3"], L["W2"], 2, d1)
    g2 = o.moe_backward(L["x"], L["Wg"], L["W1"], L["W3"], L["W2"], 2, d2)
    g12 = o.moe_backward(L["x"], L["Wg"], L["W1"], L["W3"], L["W2"], 2, 2.0 * d1 - 3.0 * d2)
    for n in g1:
        assert np.allclose(g12[n], 2.0 * g1[n] - 3.0 * g2[n], rtol=1e-11, atol=1e-12), n


def pin_backward_identical_experts_no_router_gradient(o):
    """With identical experts every chosen expert gives the same output, the
    gate weights sum to 1, so the router receives no gradient."""
    r = _rng(95)
    T, d, F, E = 20, 8, 6, 5
    one = [r.standard_normal(s) / 3 for s in ((F, d), (F, d), (d, F))]
    W1, W3, W2 = (np.repeat(m[None], E, axis=0) for m in one)
    x = r.standard_normal((T, d))
    Wg = r.standard_normal((E, d))
    g = o.moe_backward(x, Wg, W1, W3, W2, 2, r.standard_normal((T, d)))
    assert np.max(np.abs(g["dWg"])) < 1e-12


def pin_backward_dense_reduction_autograd(o):
    """E=1, k=1: the layer is the dense SwiGLU FFN; its gradients match
    torch.autograd in fp64 and the gate gets none."""
    r = _rng(96)
    T, d, F = 9, 7, 5
    x = r.standard_normal((T, d))
    Wg = r.standard_normal((1, d))
    W1, W3 = r.standard_normal((1, F, d)) / 2, r.standard_normal((1, F, d)) / 2
    W2 = r.standard_normal((1, d, F)) / 2
    dout = r.standard_normal((T, d))
    g = o.moe_backward(x, Wg, W1, W3, W2, 1, dout)
    tx, t1, t3, t2 = (torch.tensor(v, dtype=torch.float64, requires_grad=True) for v in (x, W1[0], W3[0], W2[0]))
    out = (torch.nn.functional.silu(tx @ t1.T) * (tx @ t3.T)) @ t2.T
    out.backward(torch.tensor(dout, dtype=torch.float64))
    for name, tv in (("dx", tx), ("dW1", t1), ("dW3", t3), ("dW2", t2)):
        want = tv.grad.numpy()
        got = g[name] if name == "dx" else g[name][0]
        assert np.allclose(got, want, rtol=1e-12, atol=1e-12), name
    assert np.all(g["dWg"] == 0.0)


def pin_backward_symbolic(o):
    """Every gradient against exact symbolic differentiation (sympy) of the
    layer written out from the pages' definition on a hand-sized case: 2
    tokens, d=2, F=2, E=3, k=2, small rational inputs, the routing (clear
    logit gaps) held fixed, L = sum(out * dout).  Shares no step with the
    oracle's chain rule."""
    import sympy as sp
    T, d, F, E, k = 2, 2, 2, 3, 2
    vals = {
        "x": [[1, -2], [sp.Rational(1, 2), 3]],
        "Wg": [[1, 0], [0, 1], [-1, sp.Rational(1, 4)]],
        "W1": [[[1, -1], [sp.Rational(1, 2), 2]], [[-1, 1], [2, sp.Rational(-1, 3)]], [[0, 1], [1, 1]]],
        "W3": [[[2, 1], [-1, sp.Rational(1, 4)]], [[1, 1], [sp.Rational(1, 2), -2]], [[-1, 0], [1, -1]]],
        "W2": [[[1, 2], [-1, sp.Rational(1, 2)]], [[sp.Rational(-1, 2), 1], [1, 1]], [[2, -1], [0, 1]]],
    }
    dout = [[1, sp.Rational(-1, 2)], [2, 1]]
    sym = {n: np.array(sp.symbols(f"{n}_0:{np.array(v, dtype=object).size}"), dtype=object).reshape(
        np.array(v, dtype=object).shape) for n, v in vals.items()}
    subs = {sym[n].flat[i]: np.array(v, dtype=object).flat[i] for n, v in vals.items()
            for i in range(np.array(v, dtype=object).size)}
    silu = lambda a: a / (1 + sp.exp(-a))
    L = 0
    for t in range(T):
        logit = [sum(sym["Wg"][e, c] * sym["x"][t, c] for c in range(d)) for e in range(E)]
        num = [float(lv.xreplace(subs)) for lv in logit]
        top = sorted(range(E), key=lambda e: -num[e])[:k]
        assert num[top[-1]] - max(num[e] for e in range(E) if e not in top) > 0.1
        z = [sp.exp(logit[e]) for e in top]
        for j, e in enumerate(top):
            w = z[j] / sum(z)
            h = [silu(sum(sym["W1"][e, f, c] * sym["x"][t, c] for c in range(d)))
                 * sum(sym["W3"][e, f, c] * sym["x"][t, c] for c in range(d)) for f in range(F)]
            for c in range(d):
                L += dout[t][c] * w * sum(sym["W2"][e, c, f] * h[f] for f in range(F))
    num = {n: np.array(np.array(v, dtype=object), dtype=np.float64) for n, v in vals.items()}
    g = o.moe_backward(num["x"], num["Wg"], num["W1"], num["W3"], num["W2"], k,
                       np.array(np.array(dout, dtype=object), dtype=np.float64))
    for n in vals:
        want = np.array([float(sp.diff(L, s_).xreplace(subs).evalf(30)) for s_ in sym[n].flat]).reshape(num[n].shape)
        assert np.allclose(g["d" + n], want, rtol=1e-12, atol=1e-13), n


def pin_backward_hidden_unit_slice(o):
    """expert_grad_hidden_unit (one hidden unit's gradients, from that
    expert's rows) equals the corresponding rows of dW1, dW3 and columns of
    dW2 (and of their scales) of the full moe_backward."""
    L = _tiny_layer(99, T=16, d=8, F=6, E=4)
    k = 2
    dout = _rng(100).standard_normal((16, 8))
    g = o.moe_backward(L["x"], L["Wg"], L["W1"], L["W3"], L["W2"], k, dout, with_scale=True)
    w, idx, _ = o.router(L["x"], L["Wg"], k)
    for e in range(4):
        tok, slot = np.nonzero(idx == e)
        if tok.size == 0:
            continue
        for f in range(6):
            s = o.expert_grad_hidden_unit(L["x"][tok], dout[tok], w[tok, slot], L["W1"][e], L["W3"][e], L["W2"][e], f)
            for n, got, want in (("dW1", s["dW1"], g["dW1"][e, f]), ("dW3", s["dW3"], g["dW3"][e, f]),
                                 ("dW2", s["dW2"], g["dW2"][e, :, f])):
                assert np.allclose(got, want, rtol=1e-12, atol=1e-13), (n, e, f)
                assert np.allclose(s[n + "_scale"], g[n + "_scale"][e, f] if n != "dW2"
                                   else g[n + "_scale"][e, :, f], rtol=1e-12, atol=1e-13), (n, e, f)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
