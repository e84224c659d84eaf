"""Seeded workload generator: determinism, shapes and the realised skew (CPU only)."""
import json

import numpy as np
import pytest
import torch

import moe_workloads as mw
from oracle.moe_oracle import router


def test_deterministic_and_subset_stable():
    wl = mw.get("small_bf16")
    a = mw.make_inputs(wl)
    b = mw.make_inputs(wl)
    for k in a:
        assert torch.equal(a[k], b[k])
    sub = mw.make_inputs(wl, only=("W3",))
    assert list(sub) == ["W3"] and torch.equal(sub["W3"], a["W3"])


@pytest.mark.parametrize("name", sorted(mw.SMALL_WORKLOADS) + ["tiny_f32"])
def test_shapes_and_dtypes(name):
    wl = mw.get(name)
    t = mw.make_inputs(wl)
    assert t["x"].shape == (wl.T, wl.d)
    assert t["Wg"].shape == (wl.E, wl.d)
    assert t["W1"].shape == t["W3"].shape == (wl.E, wl.F, wl.d)
    assert t["W2"].shape == (wl.E, wl.d, wl.F)
    assert ("gamma" in t) == wl.block
    assert all(v.dtype == wl.torch_dtype and v.is_contiguous() for v in t.values())


def test_init_scales():
    t = mw.make_inputs(mw.get("tiny_f32"))
    assert abs(t["W1"].std().item() - 128 ** -0.5) < 0.01 * 128 ** -0.5 * 10
    assert abs(t["W2"].std().item() - 256 ** -0.5) < 0.1 * 256 ** -0.5
    t = mw.make_inputs(mw.get("small_bf16"))
    assert abs(t["W1"].float().std().item() - 0.02) < 0.001
    assert abs(t["x"].float().std().item() - 1.0) < 0.02


@pytest.mark.parametrize("name,tol", [("small_skewed", 0.02), ("skewed", 0.01)])
def test_skew_shares_realised(name, tol):
    wl = mw.get(name)
    t = mw.make_inputs(wl, only=("x", "Wg"))
    _, idx, _ = router(t["x"], t["Wg"], wl.k)
    share = np.bincount(idx.ravel(), minlength=wl.E) / idx.size
    with open(mw.SKEW_BIAS_FILE) as f:
        rec = json.load(f)[name]
    assert np.array_equal(share, np.array(rec["realised_shares_seed0"]))
    assert np.max(np.abs(share - np.array(mw.SKEW_TARGET_SHARES))) <= tol


@pytest.mark.parametrize("name", ["small_skewed_zero", "skewed_zero"])
def test_zero_token_expert(name):
    wl = mw.get(name)
    t = mw.make_inputs(wl, only=("x", "Wg"))
    _, idx, _ = router(t["x"], t["Wg"], wl.k)
    counts = np.bincount(idx.ravel(), minlength=wl.E)
    assert counts[mw.SKEW_ZERO_EXPERT] == 0
    assert np.all(np.delete(counts, mw.SKEW_ZERO_EXPERT) > 0)
