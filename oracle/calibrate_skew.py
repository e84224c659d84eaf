"""Calibrate the per-expert gate bias of the skewed-load workloads.

TEST INFRASTRUCTURE (a committed one-off script; run by hand, never imported
by the library).  The skewed workload wants the top-2 assignments split about
{40, 20, 12, 10, 8, 5, 3, 2}% over the 8 experts.  The layer has no router
bias ("The Evolving Transformer - 05 Mixtral", section 05: the gate is a
bias-free linear map), so the workload adds one constant input channel
x[:, 0] = 1 and puts the bias in that column of the gate, Wg[e, 0] = b_e.

b_e is found by the damped fixed-point iteration
b_e += 0.6 s log(target_e / share_e), with s the spread (standard deviation)
of the unbiased logits and the b_e kept centred, on a calibration draw of x
(seed 1) with the workload's own gate (seed 0), routing every token with the
oracle's router, with b_e rounded to bf16 as the gate stores it.  The result, with the shares it reached on the
calibration draw and the shares it gives on the seed-0 draw used by tests and
benchmarks, is written to moe_workloads/skew_bias.json.

    python -m oracle.calibrate_skew [workload ...]
"""
from __future__ import annotations

import json
import sys

import numpy as np

import moe_workloads as mw
from oracle.moe_oracle import router, router_logits


def shares_of(wl, bias, x_seed):
    t = mw.make_inputs(wl, seed=0, bias=bias, x_seed=x_seed, only=("x", "Wg"))
    _, idx, _ = router(t["x"], t["Wg"], wl.k)
    counts = np.bincount(idx.ravel(), minlength=wl.E)
    return counts / idx.size, [float(v) for v in t["Wg"][:, 0].float()]


def logit_spread(wl):
    t = mw.make_inputs(wl, seed=0, bias=[0.0] * wl.E, x_seed=1, only=("x", "Wg"))
    return float(np.std(router_logits(t["x"][:, 1:], t["Wg"][:, 1:])))


def calibrate(wl, iters=80, tol=0.002):
    target = np.array(mw.SKEW_TARGET_SHARES, dtype=np.float64)
    step = 0.6 * logit_spread(wl)
    b = np.zeros(wl.E)
    best = None
    for it in range(iters):
        share, b_stored = shares_of(wl, list(b), x_seed=1)
        err = float(np.max(np.abs(share - target)))
        if best is None or err < best[0]:
            best = (err, b_stored, share.copy())
        print(f"[{wl.name}] iter {it:2d} max|share-target| = {err:.4f}", flush=True)
        if err < tol:
            break
        b = b + step * np.log(target / np.maximum(share, 1e-4))
        b = b - np.mean(b)
    err, b_stored, share = best
    realised, _ = shares_of(wl, b_stored, x_seed=None)
    return {
        "bias": b_stored,
        "target_shares": list(target),
        "calibration_shares_seed1": [float(s) for s in share],
        "realised_shares_seed0": [float(s) for s in realised],
        "T": wl.T,
        "d": wl.d,
    }


def main(names):
    try:
        with open(mw.SKEW_BIAS_FILE) as f:
            table = json.load(f)
    except FileNotFoundError:
        table = {}
    for name in names:
        table[name] = calibrate(mw.get(name))
    with open(mw.SKEW_BIAS_FILE, "w") as f:
        json.dump(table, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main(sys.argv[1:] or ["small_skewed", "skewed"])
