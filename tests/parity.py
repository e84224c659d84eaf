"""Helpers for comparing the CUDA path with the fp64 oracle.

Routing rule: the expert sets must match exactly, in slot order, except on
near-tie tokens - those whose oracle gap between consecutive sorted logits,
among the top k+1, is below 1e-3.  There the GPU's choice must be one of the
tied candidates, and its output is scored against the oracle evaluated with
the GPU's routing.  Floating-point outputs are compared by relative L2 error
over all elements (5e-3 for bf16, 1e-5 for fp32) and by a per-element bound
that catches any single wrong row or tile.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle.moe_oracle as O

NEAR_TIE = 1e-3
W_TOL = 1e-6
REL_L2 = {"bf16": 5e-3, "f32": 1e-5}


def near_tie_mask(logits: np.ndarray, k: int, thr=NEAR_TIE) -> np.ndarray:
    """``thr`` may be a per-token array."""
    s = -np.sort(-logits, axis=1)
    m = min(k + 1, logits.shape[1])
    if m < 2:
        return np.zeros(logits.shape[0], dtype=bool)
    thr = np.asarray(thr, dtype=np.float64).reshape(-1, 1) if np.ndim(thr) else thr
    return np.any(s[:, : m - 1] - s[:, 1:m] < thr, axis=1)


def check_routing(gpu_idx, gpu_w, ora_idx, ora_w, logits, k, w_tol=W_TOL, extra_gap=0.0):
    """Assert the routing rule; returns (near_tie_tokens, of which GPU differs).

    ``w_tol`` and ``extra_gap`` may be per-token arrays (see
    block_input_tolerance): a token is near-tie when a gap is below
    NEAR_TIE + 2 * extra_gap."""
    gi = np.asarray(gpu_idx, dtype=np.int64)
    gw = np.asarray(gpu_w, dtype=np.float64)
    extra = np.broadcast_to(np.asarray(extra_gap, dtype=np.float64), (gi.shape[0],))
    nt = near_tie_mask(logits, k, NEAR_TIE + 2.0 * extra)
    differ = np.any(gi != ora_idx, axis=1)
    bad = np.nonzero(~nt & differ)[0]
    assert bad.size == 0, f"routing differs on {bad.size} clear tokens, e.g. {bad[:5]}: {gi[bad[:3]]} vs {ora_idx[bad[:3]]}"
    clear = ~nt
    tol = np.broadcast_to(np.asarray(w_tol, dtype=np.float64), (gi.shape[0],))
    if clear.any():
        err = np.max(np.abs(gw - ora_w), axis=1)
        worst = np.max(err[clear] / tol[clear])
        assert worst <= 1.0, f"gate weights differ by {worst:.2f}x the bound"
    for t in np.nonzero(nt)[0]:
        chosen = logits[t, gi[t]]
        assert len(set(gi[t].tolist())) == k, f"token {t}: repeated expert {gi[t]}"
        others = np.delete(logits[t], gi[t])
        slack = 2 * NEAR_TIE + 4.0 * extra[t]
        if others.size:
            assert chosen.min() >= others.max() - slack, f"token {t}: {gi[t]} is not a near-tie top-{k}"
        assert np.all(np.diff(chosen) <= slack), f"token {t}: slot order"
        err = np.max(np.abs(gw[t] - O.softmax(chosen)))
        assert err <= tol[t], f"token {t}: weights differ by {err}"
    return int(nt.sum()), int(np.sum(nt & differ))


def block_input_tolerance(xn_gpu, xn_ora, Wg):
    """Per-token (weight tolerance, extra near-tie gap) for the block form.

    The router's input there is RMSNorm(x) rounded once to bf16 from an fp32
    value on both sides, but the two sum mean(x^2) in different orders, so a
    rare element lands on the other side of a rounding midpoint.  Checks that
    such elements differ by one bf16 step and are rare, computes the exact
    logit change dl = (xn_gpu - xn_ora) Wg^T they cause, and returns per token
    W_TOL + max_e |dl| / 2 (a top-k softmax weight moves by at most half the
    change of a logit gap) and max_e |dl| (the gaps a token's routing may
    legitimately cross on that account).
    """
    xn_gpu = np.asarray(xn_gpu, dtype=np.float64)
    diff = xn_gpu - xn_ora
    ulp = np.ldexp(1.0, np.frexp(np.maximum(np.abs(xn_ora), 1e-30))[1] - 8)
    assert np.all(np.abs(diff) <= ulp * (1 + 1e-12)), "normalised input differs by more than one bf16 step"
    assert np.mean(diff != 0) < 1e-3, f"too many differing normalised elements: {np.mean(diff != 0):.2e}"
    dl = diff @ O.f64(Wg).T
    m = np.max(np.abs(dl), axis=1)
    assert np.max(m) < 1e-2, f"normalised-input logit change {np.max(m):.2e}"
    return W_TOL + 0.5 * m, m


def effective_routing(gpu_idx, ora_w, ora_idx, logits):
    """Routing to score outputs with: the oracle's, except on near-tie tokens
    where the GPU chose differently (weights: the oracle's softmax over the
    GPU-chosen fp64 logits)."""
    gi = np.asarray(gpu_idx, dtype=np.int64)
    w = ora_w.copy()
    idx = ora_idx.copy()
    for t in np.nonzero(np.any(gi != ora_idx, axis=1))[0]:
        idx[t] = gi[t]
        w[t] = O.softmax(logits[t, gi[t]])
    return w, idx


def rel_l2(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def check_close(got, ref, dtype: str, what: str):
    """Relative L2 within the dtype's bound, and every element within a bound
    scaled to its row (bf16: a few units in the last place of the larger of
    the element and the row's RMS)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    r = rel_l2(got, ref)
    assert r <= REL_L2[dtype], f"{what}: rel-L2 {r:.3e} > {REL_L2[dtype]}"
    if ref.size:
        rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True)) if ref.ndim > 1 else np.sqrt(np.mean(ref * ref))
        tol = (2.0 ** -6 if dtype == "bf16" else 1e-4) * np.maximum(np.abs(ref), rms) + 1e-30
        worst = np.max(np.abs(got - ref) / tol)
        assert worst <= 1.0, f"{what}: an element is off by {worst:.2f}x the per-element bound"
    return r


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy() if t.is_floating_point() else t.detach().cpu().numpy()


def check_backward_close(got, ref, scale, what, c=2.0 ** -7):
    """Gradient parity: relative L2 within the bf16 bound, and every element
    within c times its sum of absolute terms (``scale``, from the oracle).

    The first-order rounding-error bound of a sum of products whose factors
    were each rounded to bf16 (relative error u = 2^-9) and accumulated in
    fp32 over n terms is (2u + n 2^-24) times the sum of the absolute terms;
    c = 2^-7 covers two rounded factors per term and fp32 accumulation over
    up to ~16K terms (2^-8 + 2^-10)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    r = rel_l2(got, ref)
    assert r <= REL_L2["bf16"], f"{what}: rel-L2 {r:.3e} > {REL_L2['bf16']}"
    err = np.abs(got - ref)
    bound = c * np.asarray(scale, dtype=np.float64) + 1e-30
    worst = float(np.max(err / bound))
    assert worst <= 1.0, f"{what}: an element is off by {worst:.2f}x its rounding-error bound"
    return r, worst
