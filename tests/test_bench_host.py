"""bench.py's host-side arithmetic (CPU only): the algorithmic work it
divides by is the closed form of the layer at Mixtral shape (d=4096,
F=14336, E=8, k=2), and the committed ncu traffic is used only on the
kernel source it was taken on."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import moe_workloads as mw  # noqa: E402

D, F, E, K = 4096, 14336, 8, 2


def test_flops_per_token_closed_form():
    # k experts x (3 matrices x 2 d F) + the gate's 2 d E
    wl = mw.get("prefill")
    flops, _, gu_flops, _ = bench.algorithmic(wl, [1] * E)
    assert flops == wl.T * 704_708_608
    assert gu_flops == wl.T * K * 4 * D * F == 1_924_145_348_608


def test_decode_bytes_closed_form():
    wl = mw.get("decode")
    _, nbytes, _, gu_bytes = bench.algorithmic(wl, [4] * E)
    per_expert = 3 * D * F * 2
    assert per_expert == 352_321_536
    assert nbytes == 8 * per_expert + D * E * 2 + 2 * wl.T * D * 2
    assert gu_bytes == 8 * 2 * D * F * 2 == 1_879_048_192


def test_unused_experts_are_not_counted():
    wl = mw.get("skewed_zero")
    _, n8, _, g8 = bench.algorithmic(wl, [1] * E)
    _, n7, _, g7 = bench.algorithmic(wl, [1] * (E - 1) + [0])
    assert n8 - n7 == 3 * D * F * 2
    assert g8 - g7 == 2 * D * F * 2


def test_int8_bytes_are_codes_plus_scales():
    wl = mw.get("decode_w8")
    _, nbytes, _, gu_bytes = bench.algorithmic(wl, [4] * E)
    assert gu_bytes == 8 * (2 * D * F + 2 * F * 4)
    assert nbytes == 8 * (3 * D * F + (2 * F + D) * 4) + D * E * 2 + 2 * wl.T * D * 2


@pytest.mark.parametrize("name", ["decode", "prefill", "decode_w8"])
def test_ncu_traffic_only_on_matching_source(name, tmp_path, monkeypatch):
    got = bench.ncu_traffic(name)
    assert got is None or got > 0
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0000000000000000")
    assert bench.ncu_traffic(name) is None


class _FakeLayer:
    """A stand-in for bench.Layer whose routing and output are given."""

    def __init__(self, wl, idx, out):
        import torch
        self.wl = wl
        self.idx = torch.from_numpy(idx.astype("int32"))
        self.out = torch.from_numpy(out)


def test_accuracy_accounting_on_planted_results():
    """bench.accuracy counts near ties and clear-token routing differences and
    scores outputs: the oracle's own result scores 0; one clear token routed
    to other experts is counted."""
    import numpy as np
    import oracle.moe_oracle as O
    wl = mw.Workload("acc_probe", 40, 32, 48, 8, 2, "f32", "inv_sqrt")
    t = mw.make_inputs(wl)
    out, w, idx, logits = O.moe_forward(t["x"], t["Wg"], t["W1"], t["W3"], t["W2"], wl.k)
    top = -np.sort(-logits, axis=1)[:, :3]
    near = int(np.sum(np.any(top[:, :-1] - top[:, 1:] < 1e-3, axis=1)))
    a = bench.accuracy(_FakeLayer(wl, idx, out), t, sample=40)
    assert a["near_tie_tokens"] == near
    assert a["clear_tokens_routed_differently"] == 0 and a["near_tie_routed_differently"] == 0
    assert a["rel_l2"] < 1e-15 and a["scored_tokens"] == 40
    bad = idx.copy()
    clear = int(np.nonzero(~np.any(top[:, :-1] - top[:, 1:] < 1e-3, axis=1))[0][0])
    bad[clear] = [e for e in range(8) if e not in idx[clear]][:2]
    a = bench.accuracy(_FakeLayer(wl, bad, out), t, sample=40)
    assert a["clear_tokens_routed_differently"] == 1


def test_targets_of():
    res = {"decode": {"bound": "hbm", "layer_roofline_frac": 0.9}, "block": {"bound": "tensor",
                                                                           "layer_roofline_frac": 0.55}}
    t = bench.targets_of(res)
    assert t["decode"]["met"] and not t["block"]["met"] and "skewed" not in t


def test_fraction_of_nominal_peaks():
    """Fractions against the nominal B300 figures: GB/s over 8000 for an
    HBM-bound kernel, TFLOP/s over 2250 for a tensor-bound one."""
    assert bench.of_nominal("hbm", 6000.0) == 6000.0 / 8000.0
    assert bench.of_nominal("tensor", 1500.0) == 1500.0 / 2250.0
