"""Plant plausible mistakes in a private copy of the oracle and check that at
least one pin fails for each (CPU only; the real oracle is never modified).

This shows the pins are strong enough: a dropped term, a wrong sign or index,
a transposed operand or a swapped gate/up matrix cannot go unnoticed.
"""
import importlib.util
import os

import numpy as np
import pytest

from oracle_pins import ALL_PINS

ORACLE_FILE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "moe_oracle.py")


def fresh_oracle():
    spec = importlib.util.spec_from_file_location("oracle_mutant", ORACLE_FILE)
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _swap_gate_up(m):
    orig = m.swiglu_expert
    m.swiglu_expert = lambda x, W1e, W3e, W2e: orig(x, W3e, W1e, W2e)


def _silu_sign(m):
    m.silu = lambda a: a / (1.0 + np.exp(a))


def _silu_is_sigmoid(m):
    m.silu = lambda a: 1.0 / (1.0 + np.exp(-a))


def _no_renormalise(m):
    def router(x, Wg, k):
        logits = m.router_logits(x, Wg)
        prob = m.softmax(logits)
        order = np.argsort(-prob, axis=-1, kind="stable")[:, :k]
        return np.take_along_axis(prob, order, axis=-1), order, logits
    m.router = router


def _ascending_topk(m):
    def router(x, Wg, k):
        logits = m.router_logits(x, Wg)
        prob = m.softmax(logits)
        order = np.argsort(prob, axis=-1, kind="stable")[:, :k]
        w = np.take_along_axis(prob, order, axis=-1)
        return w / w.sum(-1, keepdims=True), order, logits
    m.router = router


def _ties_to_higher_index(m):
    def router(x, Wg, k):
        logits = m.router_logits(x, Wg)
        prob = m.softmax(logits)
        E = prob.shape[1]
        order = (E - 1 - np.argsort(-prob[:, ::-1], axis=-1, kind="stable"))[:, :k]
        w = np.take_along_axis(prob, order, axis=-1)
        return w / w.sum(-1, keepdims=True), order, logits
    m.router = router


def _drop_gate_weight(m):
    def fwd(x, W1, W3, W2, w, idx):
        return m.__dict__["_orig_fwr"](x, W1, W3, W2, np.ones_like(np.asarray(w, dtype=float)), idx)
    m._orig_fwr = m.moe_forward_with_routing
    m.moe_forward_with_routing = fwd


def _only_first_slot(m):
    orig = m.moe_forward_with_routing
    m.moe_forward_with_routing = lambda x, W1, W3, W2, w, idx: orig(x, W1, W3, W2, w[:, :1], idx[:, :1])


def _transposed_down(m):
    m.swiglu_expert = lambda x, W1e, W3e, W2e: (
        m.silu(m.f64(x) @ m.f64(W1e).T) * (m.f64(x) @ m.f64(W3e).T)) @ m.f64(W2e)


def _gate_transposed(m):
    m.router_logits = lambda x, Wg: m.f64(x) @ m.f64(Wg)


def _rms_no_square(m):
    m.rmsnorm = lambda x, g, eps: m.f64(x) / np.sqrt(np.abs(np.mean(m.f64(x), -1, keepdims=True)) + eps) * m.f64(g)


def _rms_no_eps(m):
    m.rmsnorm = lambda x, g, eps: m.f64(x) / np.sqrt(np.mean(m.f64(x) ** 2, -1, keepdims=True)) * m.f64(g)


def _rms_no_gamma(m):
    m.rmsnorm = lambda x, g, eps: m.f64(x) / np.sqrt(np.mean(m.f64(x) ** 2, -1, keepdims=True) + eps)


def _bf16_truncates(m):
    def rnd(v):
        v = np.asarray(v, dtype=np.float64)
        mant, e = np.frexp(v)
        s = np.ldexp(1.0, 8 - np.maximum(e, -125))
        return np.trunc(v * s) / s
    m.round_to_bf16 = rnd


def _block_no_residual(m):
    orig = m.block_forward
    def blk(x, gamma, eps, Wg, W1, W3, W2, k):
        out, w, idx, lg, xn = orig(x, gamma, eps, Wg, W1, W3, W2, k)
        return out - m.f64(x), w, idx, lg, xn
    m.block_forward = blk


def _block_unnormalised(m):
    def blk(x, gamma, eps, Wg, W1, W3, W2, k):
        delta, w, idx, lg = m.moe_forward(m.f64(x), Wg, W1, W3, W2, k)
        return m.f64(x) + delta, w, idx, lg, m.f64(x)
    m.block_forward = blk


def _dispatch_unstable(m):
    orig = m.dispatch
    def disp(idx, E):
        counts, offsets, row_src, slot_pos = orig(idx, E)
        return counts, offsets, row_src[::-1].copy(), slot_pos
    m.dispatch = disp


def _dispatch_token_not_pair(m):
    def disp(idx, E):
        idx = np.asarray(idx)
        flat = idx.reshape(-1)
        counts = np.bincount(flat, minlength=E)
        offsets = np.concatenate([[0], np.cumsum(counts)])
        order = np.argsort(flat, kind="stable")
        slot_pos = np.empty_like(order)
        slot_pos[order] = np.arange(order.size)
        return counts, offsets, order, slot_pos  # pair index instead of token
    m.dispatch = disp


def _hidden_no_gate(m):
    m.swiglu_hidden = lambda x, W1e, W3e: m.f64(x) @ m.f64(W3e).T


def _rms32_no_square(m):
    m.rmsnorm_fp32 = lambda x, g, eps: (m.f64(x) / np.sqrt(np.abs(np.mean(m.f64(x), -1, keepdims=True)) + eps)
                                        * m.f64(g)).astype(np.float32)


def _two_matrix_expert(m):
    m.expert_param_shapes = lambda d, F: [(F, d), (d, F)]


def _int8_divisor_128(m):
    def quant(W):
        w32 = m.f64(W).astype(np.float32)
        s = (np.max(np.abs(w32), axis=-1) / np.float32(128.0)).astype(np.float32)
        safe = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
        q = np.clip(np.rint(w32 / safe[..., None]), -127, 127)
        return q.astype(np.int8), s
    m.quantize_int8_rows = quant


def _int8_truncates(m):
    def quant(W):
        w32 = m.f64(W).astype(np.float32)
        s = (np.max(np.abs(w32), axis=-1) / np.float32(127.0)).astype(np.float32)
        safe = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
        return np.trunc(w32 / safe[..., None]).astype(np.int8), s
    m.quantize_int8_rows = quant


def _int8_ties_away_from_zero(m):
    def quant(W):
        w32 = m.f64(W).astype(np.float32)
        s = (np.max(np.abs(w32), axis=-1) / np.float32(127.0)).astype(np.float32)
        safe = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
        v = w32 / safe[..., None]
        return (np.sign(v) * np.floor(np.abs(v) + 0.5)).astype(np.int8), s
    m.quantize_int8_rows = quant


def _int8_per_column(m):
    def quant(W):
        w32 = m.f64(W).astype(np.float32)
        s = (np.max(np.abs(w32), axis=-2) / np.float32(127.0)).astype(np.float32)
        safe = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
        q = np.clip(np.rint(w32 / safe[..., None, :]), -127, 127)
        return q.astype(np.int8), np.max(s, axis=-1) * np.ones(w32.shape[:-1], np.float32)
    m.quantize_int8_rows = quant


def _w8_drops_scale(m):
    m.dequantize_int8_rows = lambda q, s: np.asarray(q, dtype=np.float64)


def _bwd_silu_grad_is_silu(m):
    m.silu_grad = lambda a: m.silu(a)


def _bwd_silu_grad_drops_term(m):
    m.silu_grad = lambda a: 1.0 / (1.0 + np.exp(-a))


def _bwd_no_softmax_jacobian(m):
    src = m.moe_backward

    def bwd(x, Wg, W1, W3, W2, k, dout):
        g = src(x, Wg, W1, W3, W2, k, dout)
        # a plausible mistake: router gradient taken as w * dw (no centering)
        w, idx, _ = m.router(x, Wg, k)
        xx = m.f64(x)
        dw = np.zeros_like(w)
        for j in range(k):
            for t in range(xx.shape[0]):
                e = idx[t, j]
                a = xx[t] @ m.f64(W1[e]).T
                b = xx[t] @ m.f64(W3[e]).T
                dw[t, j] = np.sum(m.f64(dout)[t] * ((m.silu(a) * b) @ m.f64(W2[e]).T))
        dl_bad = w * dw
        dl_ok = w * (dw - np.sum(w * dw, axis=1, keepdims=True))
        Wgf = m.f64(Wg)
        for j in range(k):
            g["dx"] += (dl_bad - dl_ok)[:, j][:, None] * Wgf[idx[:, j]]
            np.add.at(g["dWg"], idx[:, j], (dl_bad - dl_ok)[:, j][:, None] * xx)
        return g
    m.moe_backward = bwd


def _bwd_drops_gate_weight(m):
    src = m.moe_backward

    def bwd(x, Wg, W1, W3, W2, k, dout):
        g = src(x, Wg, W1, W3, W2, k, dout)
        g["dW2"] = g["dW2"] * 2.0
        return g
    m.moe_backward = bwd


def _bwd_transposed_dw1(m):
    src = m.moe_backward

    def bwd(x, Wg, W1, W3, W2, k, dout):
        g = src(x, Wg, W1, W3, W2, k, dout)
        if g["dW1"].shape[1] == g["dW1"].shape[2]:
            g["dW1"] = np.transpose(g["dW1"], (0, 2, 1)).copy()
        else:
            g["dW1"] = g["dW1"][:, ::-1].copy()
        return g
    m.moe_backward = bwd


def _slice_drops_gate_weight(m):
    src = m.expert_grad_hidden_unit
    m.expert_grad_hidden_unit = lambda xe, doute, we, W1e, W3e, W2e, f: src(
        xe, doute, np.ones(len(we)), W1e, W3e, W2e, f)


def _slice_gate_up_swapped(m):
    src = m.expert_grad_hidden_unit
    m.expert_grad_hidden_unit = lambda xe, doute, we, W1e, W3e, W2e, f: src(xe, doute, we, W3e, W1e, W2e, f)


def _down_next_expert(m):
    """Each segment multiplied by the next expert's W2 (an off-by-one index)."""
    def down(h, offsets, W2):
        return m.__dict__["_orig_down"](h, offsets, np.roll(np.asarray(W2), -1, axis=0))
    m._orig_down = m.down_projection
    m.down_projection = down


def _down_skips_last_segment(m):
    def down(h, offsets, W2):
        off = np.array(offsets, copy=True)
        off[-1] = off[-2]
        return m.__dict__["_orig_down2"](h, off, W2)
    m._orig_down2 = m.down_projection
    m.down_projection = down


def _gate_up_grouped_swapped(m):
    src = m.gate_up_projection
    m.gate_up_projection = lambda x_perm, offsets, W1, W3: src(x_perm, offsets, W3, W1)


def _combine_drops_weight(m):
    src = m.combine
    m.combine = lambda y, pos, w, residual=None: src(y, pos, np.ones_like(np.asarray(w, dtype=float)), residual)


def _combine_slot_major(m):
    """slot_pos read as [k, T] instead of [T, k]."""
    src = m.combine

    def comb(y, pos, w, residual=None):
        T, k = np.asarray(w).shape
        return src(y, np.asarray(pos).reshape(k, T).T.reshape(-1), w, residual)
    m.combine = comb


def _combine_drops_residual(m):
    src = m.combine
    m.combine = lambda y, pos, w, residual=None: src(y, pos, w, None)


MUTANTS = {f.__name__[1:]: f for f in [
    _swap_gate_up, _silu_sign, _silu_is_sigmoid, _no_renormalise, _ascending_topk,
    _ties_to_higher_index, _drop_gate_weight, _only_first_slot, _transposed_down,
    _gate_transposed, _rms_no_square, _rms_no_eps, _rms_no_gamma, _bf16_truncates,
    _block_no_residual, _block_unnormalised, _two_matrix_expert, _dispatch_unstable,
    _dispatch_token_not_pair, _hidden_no_gate, _rms32_no_square, _int8_divisor_128, _int8_truncates,
    _int8_ties_away_from_zero, _int8_per_column, _w8_drops_scale, _bwd_silu_grad_is_silu,
    _bwd_silu_grad_drops_term, _bwd_no_softmax_jacobian, _bwd_drops_gate_weight, _bwd_transposed_dw1,
    _slice_drops_gate_weight, _slice_gate_up_swapped, _down_next_expert, _down_skips_last_segment,
    _gate_up_grouped_swapped, _combine_drops_weight, _combine_slot_major, _combine_drops_residual]}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    m = fresh_oracle()
    MUTANTS[name](m)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(m)
        except Exception:  # an assertion or a shape error both count
            caught.append(pin.__name__)
            break  # one failing pin is enough
    assert caught, f"no pin caught the planted mistake {name!r}"
