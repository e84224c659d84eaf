"""Parity of the int8 weight-only path (KerasFormers Mixtral docs, "Lower
memory": weights alone quantised to int8) with the fp64 oracle, on GPU,
through the C ABI.

The quantiser is integer work decided in IEEE fp32 on both sides, so its
codes and scales must match the oracle's bit for bit.  The layer with int8
weights is compared with the oracle's layer of the dequantised weights
s * q, computed from the oracle's own quantisation: rel-L2 <= 5e-3 and the
per-element bound, as for bf16.  Routing is the bf16 router's and follows
the same near-tie rule.
"""
import json
import os

import numpy as np
import pytest
import torch

import moe_workloads as mw
import oracle.moe_oracle as O
from parity import check_close, check_routing, effective_routing, near_tie_mask, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from sparse_mixture_experts_50_b300 import binding
    binding.lib()
    binding.moe_get_device_status(reset=True)
    return binding


def dev(t):
    return t.to(DEV).contiguous()


def status_ok(B):
    s = B.moe_get_device_status(reset=True)
    assert s == 0, f"device status {s}"


def oracle_q(W):
    """The oracle's codes and scales as device tensors."""
    q, s = O.quantize_int8_rows(W)
    return dev(torch.from_numpy(q)), dev(torch.from_numpy(s))


def assert_same_quant(B, W):
    q, s = B.moe_quantize_int8(dev(W))
    status_ok(B)
    qo, so = O.quantize_int8_rows(W)
    assert np.array_equal(q.cpu().numpy(), qo), "int8 codes differ from the oracle's"
    assert np.array_equal(s.cpu().numpy().view(np.uint32), so.view(np.uint32)), "scales differ from the oracle's"


# ------------------------------------------------------------------ quantiser
def test_quantize_hand_rows(B):
    with open(os.path.join(GOLDEN, "int8_rows_hand.json")) as f:
        rows = json.load(f)["rows"]
    W = torch.tensor([r["w"] for r in rows], dtype=torch.bfloat16)
    q, s = B.moe_quantize_int8(dev(W))
    status_ok(B)
    assert q.cpu().tolist() == [r["q"] for r in rows]
    assert s.cpu().tolist() == [np.float32(r["scale"]).item() for r in rows]


@pytest.mark.parametrize("shape", [(300, 512), (8, 7, 4096), (3, 14336), (1, 8), (2, 5, 24)])
def test_quantize_bit_exact(B, shape):
    r = np.random.default_rng(sum(shape))
    W = torch.from_numpy(r.standard_normal(shape) * 0.02).to(torch.bfloat16)
    flat = W.view(-1, shape[-1])
    flat[0] = 0.0                                   # a zero row
    if flat.shape[0] > 2:
        # rows whose quotients sit exactly on midpoints: amax 127/128 makes
        # s = 1/128, and every other value is an integer or a half-integer
        # over 128 (all bf16 values)
        m = flat.shape[1]
        flat[1] = torch.tensor([((i % 253) - 126 + 0.5 * (i % 2)) / 128.0 for i in range(m)])
        flat[1, 0] = 127 / 128.0
        flat[2] = -flat[1]
    assert_same_quant(B, W)


# ------------------------------------------------------------------ experts
@pytest.mark.parametrize("counts", [
    [0, 128, 129, 1, 0, 255, 256, 300],  # wide tiles, empty experts
    [191, 192, 193, 0, 384, 385, 1, 0],   # wide tiles: uneven counts
    [223, 224, 225, 0, 448, 449, 1, 0],   # wide tiles: one short of, at and past 224-token edges
    [1000, 0, 0, 0, 0, 0, 0, 0],          # every row in one expert
    [0, 0, 0, 0, 0, 0, 0, 129],           # just past the small-batch limit, last expert only
    [3, 1, 4, 1, 5, 9, 2, 6],             # decode-like: a few rows each
    [40, 0, 33, 1, 32, 0, 22, 0],         # 128 rows: small-batch tiles of 32 tokens, ragged
    [0, 0, 0, 128, 0, 0, 0, 0],           # 128 rows in one expert: four 32-token tiles
])
def test_expert_w8_tiles(B, counts):
    """The int8 grouped GEMMs on hand-made segments: up to 128 rows the
    small-batch form, beyond it the wide form (224 tokens per tile); d is not
    a multiple of the 128-row weight blocks of the wide down GEMM, nor d_ff
    of the 256-column tiles."""
    r = np.random.default_rng(sum(counts) + 1)
    E, d, F = 8, 320, 448
    offsets = np.concatenate([[0], np.cumsum(counts)])
    Tk = int(offsets[-1])
    x = torch.from_numpy(r.standard_normal((Tk, d))).to(torch.bfloat16)
    W1 = torch.from_numpy(r.standard_normal((E, F, d)) * 0.05).to(torch.bfloat16)
    W3 = torch.from_numpy(r.standard_normal((E, F, d)) * 0.05).to(torch.bfloat16)
    W2 = torch.from_numpy(r.standard_normal((E, d, F)) * 0.05).to(torch.bfloat16)
    (q1, s1), (q3, s3), (q2, s2) = (O.quantize_int8_rows(W) for W in (W1, W3, W2))
    off = dev(torch.from_numpy(offsets).int())
    h = B.moe_expert_gate_up_w8(dev(x), off, *(dev(torch.from_numpy(v)) for v in (q1, s1, q3, s3)))
    y = B.moe_expert_down_w8(h, off, dev(torch.from_numpy(q2)), dev(torch.from_numpy(s2)))
    status_ok(B)
    D1, D3, D2 = O.dequantize_int8_rows(q1, s1), O.dequantize_int8_rows(q3, s3), O.dequantize_int8_rows(q2, s2)
    check_close(to_np(h), O.gate_up_projection(x, offsets, D1, D3), "bf16", "h (int8 weights)")
    check_close(to_np(y), O.down_projection(h.cpu(), offsets, D2), "bf16", "y (int8 weights)")


# ------------------------------------------------------------------ layer
@pytest.mark.parametrize("name", ["small_bf16", "small_ragged", "small_skewed_zero"])
@pytest.mark.parametrize("entry", ["ws", "alloc"])
def test_forward_w8_small(B, name, entry):
    wl = mw.get(name)
    t = mw.make_inputs(wl)
    qs = [O.quantize_int8_rows(t[n]) for n in ("W1", "W3", "W2")]
    args = [dev(torch.from_numpy(v)) for qv in qs for v in qv]
    x, Wg = dev(t["x"]), dev(t["Wg"])
    if entry == "ws":
        ws = B.workspace(wl.T, wl.d, wl.F, wl.E, wl.k, B.MOE_DTYPE_BF16)
        out = B.moe_forward_w8_ws(x, Wg, *args, wl.k, ws)
    else:
        out = B.moe_forward_w8(x, Wg, *args, wl.k)
    status_ok(B)
    ref, ora_w, ora_idx, logits = O.moe_forward_w8(t["x"], t["Wg"], *(v for qv in qs for v in qv), wl.k)
    idx, _ = B.moe_router_topk(x, Wg, wl.k)
    w_eff, idx_eff = effective_routing(to_np(idx), ora_w, ora_idx, logits)
    if not np.array_equal(idx_eff, ora_idx):
        D = [O.dequantize_int8_rows(*qv) for qv in qs]
        ref = O.moe_forward_with_routing(t["x"], *D, w_eff, idx_eff)
    check_close(to_np(out), ref, "bf16", f"{name} int8-weight layer")


def test_forward_w8_large_ragged(B):
    """Many rows per expert (the wide form), two experts with ragged tails,
    k=1: the layer against the oracle's layer of the dequantised weights."""
    wl = mw.Workload("w8_wide", 1100, 320, 448, 2, 1, "bf16", "std002")
    t = mw.make_inputs(wl)
    qs = [O.quantize_int8_rows(t[n]) for n in ("W1", "W3", "W2")]
    args = [dev(torch.from_numpy(v)) for qv in qs for v in qv]
    x, Wg = dev(t["x"]), dev(t["Wg"])
    ws = B.workspace(wl.T, wl.d, wl.F, wl.E, wl.k)
    out = B.moe_forward_w8_ws(x, Wg, *args, wl.k, ws)
    status_ok(B)
    ref, ora_w, ora_idx, logits = O.moe_forward_w8(t["x"], t["Wg"], *(v for qv in qs for v in qv), wl.k)
    idx, _ = B.moe_router_topk(x, Wg, wl.k)
    w_eff, idx_eff = effective_routing(to_np(idx), ora_w, ora_idx, logits)
    if not np.array_equal(idx_eff, ora_idx):
        D = [O.dequantize_int8_rows(*qv) for qv in qs]
        ref = O.moe_forward_with_routing(t["x"], *D, w_eff, idx_eff)
    check_close(to_np(out), ref, "bf16", "int8 layer, many rows per expert")


def test_forward_w8_matches_bf16_layer_within_quantisation(B):
    """The int8 layer is the same layer: its output stays within the
    quantisation error of the bf16 layer's (the oracle pins the same bound)."""
    wl = mw.get("small_bf16")
    t = {n: dev(v) for n, v in mw.make_inputs(wl).items()}
    q = [B.moe_quantize_int8(t[n]) for n in ("W1", "W3", "W2")]
    out8 = B.moe_forward_w8(t["x"], t["Wg"], *(v for qv in q for v in qv), wl.k)
    out16 = B.moe_forward(t["x"], t["Wg"], t["W1"], t["W3"], t["W2"], wl.k)
    status_ok(B)
    a, b = to_np(out8), to_np(out16)
    assert np.linalg.norm(a - b) / np.linalg.norm(b) < 0.03


# ------------------------------------------------------------------ full size
_SHARED = {}


@pytest.mark.parametrize("name", ["decode_w8", "prefill_w8"])
def test_full_size_w8_sampled(B, name):
    """Mixtral sizes, run exactly as bench.py runs a step (weights quantised
    on the GPU by moe_quantize_int8).  Every code and scale must equal the
    oracle's; routing is checked on every token, outputs on 128 seeded tokens
    + every near-tie token + the first and last."""
    import bench
    wl = mw.get(name)
    cpu = bench.make_tensors(wl, _SHARED)
    layer = bench.Layer(wl, cpu, DEV)
    out = layer.step()
    out = layer.step()
    status_ok(B)
    qs = []
    for n, (gq, gs) in (("W1", (layer.W1q, layer.W1s)), ("W3", (layer.W3q, layer.W3s)),
                        ("W2", (layer.W2q, layer.W2s))):
        qo, so = O.quantize_int8_rows(cpu[n])
        assert np.array_equal(gq.cpu().numpy(), qo), f"{n}: codes differ from the oracle's"
        assert np.array_equal(gs.cpu().numpy().view(np.uint32), so.view(np.uint32)), f"{n}: scales differ"
        qs.append((qo, so))
    xin = O.f64(cpu["x"])
    ora_w, ora_idx, logits = O.router(xin, cpu["Wg"], wl.k)
    n_tie, n_diff = check_routing(to_np(layer.idx), to_np(layer.w), ora_idx, ora_w, logits, wl.k)
    r = np.random.default_rng(2)
    sample = set(r.choice(wl.T, size=min(128, wl.T), replace=False).tolist())
    sample |= set(np.nonzero(near_tie_mask(logits, wl.k))[0].tolist()) | {0, wl.T - 1}
    s = np.array(sorted(sample))
    w_eff, idx_eff = effective_routing(to_np(layer.idx), ora_w, ora_idx, logits)
    D = [O.dequantize_int8_rows(*qv) for qv in qs]
    ref = O.moe_forward_with_routing(xin[s], *D, w_eff[s], idx_eff[s])
    check_close(to_np(out)[s], ref, "bf16", f"{name} out")
    print(f"{name}: near-tie tokens {n_tie}, routed differently {n_diff}")
