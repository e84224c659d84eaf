"""Parity of the CUDA path (through the C ABI) with the fp64 oracle, on GPU.

Each step is checked alone on the oracle's own inputs, then the whole layer
on every workload: the reduced sizes on all tokens, the full Mixtral sizes
(in the launch configuration bench.py times) on a seeded sample of tokens
plus every near-tie token.  Routing is bit-exact outside the near-tie set;
floating point is within rel-L2 5e-3 (bf16) / 1e-5 (fp32).
"""
import numpy as np
import pytest
import torch

import moe_workloads as mw
import oracle.moe_oracle as O
from parity import block_input_tolerance, check_close, check_routing, effective_routing, near_tie_mask, to_np

pytestmark = pytest.mark.gpu

SMALL = sorted(mw.SMALL_WORKLOADS) + ["tiny_f32"]
SMALL_BF16 = [n for n in SMALL if mw.get(n).dtype == "bf16"]
DEV = "cuda:0"


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from sparse_mixture_experts_50_b300 import binding
    binding.lib()
    assert binding.moe_get_device_status(reset=True) in (0, binding.MOE_EDEVICE, binding.MOE_ETIMEOUT)
    return binding


def dev(t):
    return t.to(DEV).contiguous()


def status_ok(B):
    s = B.moe_get_device_status(reset=True)
    assert s == 0, f"device status {s}"


_CACHE = {}


def inputs(name):
    if name not in _CACHE:
        _CACHE[name] = mw.make_inputs(mw.get(name))
    return _CACHE[name]


def router_input(name):
    wl, t = mw.get(name), inputs(name)
    if wl.block:
        return torch.from_numpy(O.block_normed_input(t["x"], t["gamma"], wl.eps)).to(wl.torch_dtype)
    return t["x"]


# ------------------------------------------------------------------ router
@pytest.mark.parametrize("name", SMALL)
def test_router(B, name):
    wl, t = mw.get(name), inputs(name)
    x = router_input(name)
    ora_w, ora_idx, logits = O.router(x, t["Wg"], wl.k)
    lg = torch.empty((wl.T, wl.E), dtype=torch.float32, device=DEV)
    idx, w = B.moe_router_topk(dev(x), dev(t["Wg"]), wl.k, logits=lg)
    status_ok(B)
    assert np.max(np.abs(to_np(lg) - logits)) < 2e-4
    check_routing(to_np(idx), to_np(w), ora_idx, ora_w, logits, wl.k)


def test_router_ties_and_k(B):
    """Equal logits keep the lower index first and split evenly; k up to 8,
    E up to 64."""
    T, d = 40, 64
    x = torch.ones((T, d), dtype=torch.float32)
    Wg = torch.zeros((64, d), dtype=torch.float32)
    Wg[[5, 9, 33, 60]] = 1.0 / d  # four equal, largest logits
    Wg[10] = -1.0
    idx, w = B.moe_router_topk(dev(x), dev(Wg), 4)
    status_ok(B)
    assert (to_np(idx) == np.array([5, 9, 33, 60])).all()
    assert np.all(to_np(w) == 0.25)
    r = np.random.default_rng(3)
    for E, k in ((64, 8), (33, 5), (2, 2), (8, 1), (1, 1)):
        x = torch.from_numpy(r.standard_normal((77, 96))).float()
        Wg = torch.from_numpy(r.standard_normal((E, 96)) / 10).float()
        ora_w, ora_idx, logits = O.router(x, Wg, k)
        idx, w = B.moe_router_topk(dev(x), dev(Wg), k)
        status_ok(B)
        check_routing(to_np(idx), to_np(w), ora_idx, ora_w, logits, k)


def test_router_logits_wide_e_large_batch(B):
    """E=64 at a batch large enough for one warp per token (32 threads per
    token, fewer than E): every logit is written and matches the oracle."""
    r = np.random.default_rng(29)
    T, d, E, k = 12000, 128, 64, 2
    x = torch.from_numpy(r.standard_normal((T, d))).to(torch.bfloat16)
    Wg = torch.from_numpy(r.standard_normal((E, d)) * 0.05).to(torch.bfloat16)
    lg = torch.full((T, E), float("nan"), dtype=torch.float32, device=DEV)
    idx, w = B.moe_router_topk(dev(x), dev(Wg), k, logits=lg)
    status_ok(B)
    ora_w, ora_idx, logits = O.router(x, Wg, k)
    got = to_np(lg)
    assert np.all(np.isfinite(got)), "logits left unwritten"
    assert np.max(np.abs(got - logits)) < 2e-4
    check_routing(to_np(idx), to_np(w), ora_idx, ora_w, logits, k)


def test_router_nan_logit_not_chosen(B):
    """A NaN logit (expert 0 here) is never picked while another expert is
    left; the routing among the others matches the oracle's over them."""
    r = np.random.default_rng(31)
    T, d, E, k = 50, 64, 8, 2
    x = torch.from_numpy(r.standard_normal((T, d))).float()
    Wg = torch.from_numpy(r.standard_normal((E, d)) * 0.1).float()
    Wg[0, 3] = float("nan")
    idx, w = B.moe_router_topk(dev(x), dev(Wg), k)
    status_ok(B)
    gi = to_np(idx)
    assert not np.any(gi == 0)
    ora_w, ora_idx, logits = O.router(x, Wg[1:], k)
    check_routing(gi - 1, to_np(w), ora_idx, ora_w, logits, k)


# ------------------------------------------------------------------ dispatch
@pytest.mark.parametrize("name", SMALL)
def test_permute(B, name):
    wl, t = mw.get(name), inputs(name)
    _, ora_idx, _ = O.router(t["x"], t["Wg"], wl.k)
    counts, offsets, row_src, slot_pos = O.dispatch(ora_idx, wl.E)
    g = B.moe_permute(dev(t["x"]), dev(torch.from_numpy(ora_idx).int()), wl.E)
    status_ok(B)
    gc, go, gr, gs, gx = (v.cpu() for v in g)
    assert np.array_equal(gc.numpy(), counts)
    assert np.array_equal(go.numpy(), offsets)
    assert np.array_equal(gr.numpy(), row_src)
    assert np.array_equal(gs.numpy(), slot_pos)
    assert torch.equal(gx, t["x"][torch.from_numpy(row_src)])


def test_permute_large_and_skewed(B):
    """Many chunks of the rank kernel, E=64, an expert with every token."""
    r = np.random.default_rng(11)
    for T, E, k in ((20000, 8, 2), (3000, 64, 8), (5000, 16, 1)):
        idx = np.stack([r.permutation(E)[:k] for _ in range(T)])
        if E == 16:
            idx[:] = 7
        x = torch.from_numpy(r.standard_normal((T, 64))).to(torch.bfloat16)
        counts, offsets, row_src, slot_pos = O.dispatch(idx, E)
        g = B.moe_permute(dev(x), dev(torch.from_numpy(idx).int()), E)
        status_ok(B)
        gc, go, gr, gs, gx = (v.cpu() for v in g)
        assert np.array_equal(gc.numpy(), counts) and np.array_equal(go.numpy(), offsets)
        assert np.array_equal(gr.numpy(), row_src) and np.array_equal(gs.numpy(), slot_pos)
        assert torch.equal(gx, x[torch.from_numpy(row_src)])


def test_permute_rejects_bad_index_on_device(B):
    """An expert index outside [0, E) is skipped by the kernel's bounds check
    and reported in the device status; the context stays usable."""
    x = torch.randn(64, 64).to(torch.bfloat16)
    idx = torch.zeros((64, 2), dtype=torch.int32)
    idx[:, 1] = 1
    idx[10, 1] = 99
    g = B.moe_permute(dev(x), dev(idx), 8)
    assert B.moe_get_device_status(reset=True) == B.MOE_EDEVICE
    assert g[0].cpu().tolist()[:2] == [64, 63]
    B.moe_permute(dev(x), dev(idx.clamp(max=7)), 8)
    status_ok(B)


# ------------------------------------------------------------------ experts
def segment_inputs(name):
    wl, t = mw.get(name), inputs(name)
    _, ora_idx, _ = O.router(t["x"], t["Wg"], wl.k)
    counts, offsets, row_src, _ = O.dispatch(ora_idx, wl.E)
    x_perm = t["x"][torch.from_numpy(row_src)]
    return wl, t, offsets, x_perm


@pytest.mark.parametrize("name", SMALL)
def test_expert_gate_up_and_down(B, name):
    wl, t, offsets, x_perm = segment_inputs(name)
    off = dev(torch.from_numpy(offsets).int())
    h = B.moe_expert_gate_up(dev(x_perm), off, dev(t["W1"]), dev(t["W3"]))
    status_ok(B)
    check_close(to_np(h), O.gate_up_projection(x_perm, offsets, t["W1"], t["W3"]), wl.dtype, f"{name} h")
    y = B.moe_expert_down(h, off, dev(t["W2"]))
    status_ok(B)
    check_close(to_np(y), O.down_projection(h.cpu(), offsets, t["W2"]), wl.dtype, f"{name} y")


@pytest.mark.parametrize("name", ["small_bf16", "small_ragged", "small_f32"])
def test_expert_ffn_entry_points(B, name):
    """moe_expert_ffn (pool scratch) and moe_expert_ffn_ws (caller scratch)
    against the oracle's grouped steps, and bit for bit against the two
    single-step calls."""
    wl, t, offsets, x_perm = segment_inputs(name)
    off = dev(torch.from_numpy(offsets).int())
    g = [dev(t[n]) for n in ("W1", "W3", "W2")]
    y = B.moe_expert_ffn(dev(x_perm), off, *g)
    h_ws, y_ws = B.moe_expert_ffn_ws(dev(x_perm), off, *g)
    h1 = B.moe_expert_gate_up(dev(x_perm), off, g[0], g[1])
    y1 = B.moe_expert_down(h1, off, g[2])
    status_ok(B)
    assert torch.equal(y, y1) and torch.equal(y_ws, y1) and torch.equal(h_ws, h1)
    ref = O.down_projection(O.gate_up_projection(x_perm, offsets, t["W1"], t["W3"]), offsets, t["W2"])
    check_close(to_np(y), ref, wl.dtype, f"{name} expert_ffn")


@pytest.mark.parametrize("counts", [
    [0, 128, 129, 1, 0, 255, 256, 300],  # tile boundaries, empty experts
    [1000, 0, 0, 0, 0, 0, 0, 0],          # every row in one expert
    [0, 0, 0, 0, 0, 0, 0, 7],             # only the last expert
    [3, 1, 4, 1, 5, 9, 2, 6],             # decode-like: a few rows each
    [40, 0, 33, 1, 32, 0, 22, 0],         # 128 rows: small-batch tiles of 32 tokens, ragged
    [0, 0, 0, 128, 0, 0, 0, 0],           # 128 rows in one expert: four 32-token tiles
])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_expert_tiles(B, counts, dtype):
    """The grouped GEMMs on hand-made segments: rows that cross tile edges,
    empty experts, one expert with everything; d and d_ff not multiples of
    the 256/128-wide output tiles."""
    r = np.random.default_rng(sum(counts))
    E, d, F = 8, 320, 448
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    offsets = np.concatenate([[0], np.cumsum(counts)])
    Tk = int(offsets[-1])
    x = torch.from_numpy(r.standard_normal((Tk, d))).to(tdt)
    W1 = torch.from_numpy(r.standard_normal((E, F, d)) * 0.05).to(tdt)
    W3 = torch.from_numpy(r.standard_normal((E, F, d)) * 0.05).to(tdt)
    W2 = torch.from_numpy(r.standard_normal((E, d, F)) * 0.05).to(tdt)
    off = dev(torch.from_numpy(offsets).int())
    h = B.moe_expert_gate_up(dev(x), off, dev(W1), dev(W3))
    y = B.moe_expert_down(h, off, dev(W2))
    status_ok(B)
    check_close(to_np(h), O.gate_up_projection(x, offsets, W1, W3), dtype, "h")
    check_close(to_np(y), O.down_projection(h.cpu(), offsets, W2), dtype, "y")


# ------------------------------------------------------------------ combine
@pytest.mark.parametrize("dtype,res", [("bf16", False), ("bf16", True), ("f32", False), ("f32", True)])
def test_combine(B, dtype, res):
    r = np.random.default_rng(5)
    T, d, k = 300, 256, 2
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    y = torch.from_numpy(r.standard_normal((T * k, d))).to(tdt)
    slot_pos = torch.from_numpy(r.permutation(T * k)).int()
    w = torch.from_numpy(r.uniform(0, 1, (T, k))).float()
    x = torch.from_numpy(r.standard_normal((T, d))).to(tdt)
    out = B.moe_combine(dev(y), dev(slot_pos), dev(w), T, residual=dev(x) if res else None)
    status_ok(B)
    ref = O.combine(y, slot_pos.numpy(), w.numpy(), x if res else None)
    check_close(to_np(out), ref, dtype, "combine")
    if dtype == "bf16":  # one rounding of the fp32 sum
        assert np.max(np.abs(to_np(out) - ref) / np.maximum(np.abs(ref), 1e-3)) <= 2.0 ** -8 + 1e-6


# ------------------------------------------------------------------ layer
def oracle_layer(name):
    wl, t = mw.get(name), inputs(name)
    if wl.block:
        out, w, idx, logits, xn = O.block_forward(t["x"], t["gamma"], wl.eps, t["Wg"], t["W1"], t["W3"], t["W2"], wl.k)
        return out, w, idx, logits, xn
    out, w, idx, logits = O.moe_forward(t["x"], t["Wg"], t["W1"], t["W3"], t["W2"], wl.k)
    return out, w, idx, logits, O.f64(t["x"])


@pytest.mark.parametrize("name", SMALL)
@pytest.mark.parametrize("entry", ["ws", "alloc"])
def test_forward_small(B, name, entry):
    wl, t = mw.get(name), inputs(name)
    g = {n: dev(v) for n, v in t.items()}
    if wl.block:
        if entry == "ws":
            ws = B.workspace(wl.T, wl.d, wl.F, wl.E, wl.k, 1 if wl.dtype == "bf16" else 0)
            out = B.moe_block_forward_ws(g["x"], g["gamma"], wl.eps, g["Wg"], g["W1"], g["W3"], g["W2"], wl.k, ws)
        else:
            out = B.moe_block_forward(g["x"], g["gamma"], wl.eps, g["Wg"], g["W1"], g["W3"], g["W2"], wl.k)
    elif entry == "ws":
        ws = B.workspace(wl.T, wl.d, wl.F, wl.E, wl.k, 1 if wl.dtype == "bf16" else 0)
        out = B.moe_forward_ws(g["x"], g["Wg"], g["W1"], g["W3"], g["W2"], wl.k, ws)
    elif wl.dtype == "bf16":
        out = B.moe_forward(g["x"], g["Wg"], g["W1"], g["W3"], g["W2"], wl.k)
    else:
        out = B.moe_forward_f32(g["x"], g["Wg"], g["W1"], g["W3"], g["W2"], wl.k)
    status_ok(B)
    ref, ora_w, ora_idx, logits, xin = oracle_layer(name)
    # The GPU's routing, for scoring near-tie tokens.
    idx, _ = B.moe_router_topk(dev(torch.from_numpy(xin).to(wl.torch_dtype)), g["Wg"], wl.k)
    w_eff, idx_eff = effective_routing(to_np(idx), ora_w, ora_idx, logits)
    if not np.array_equal(idx_eff, ora_idx):
        ref = O.moe_forward_with_routing(xin, t["W1"], t["W3"], t["W2"], w_eff, idx_eff)
        if wl.block:
            ref = ref + O.f64(t["x"])
    check_close(to_np(out), ref, wl.dtype, f"{name} out")


def block_delta_check(B, layer, xn_ref, cpu, rows, w_eff, idx_eff, what):
    """The block's MoE delta, gated on its own: the same step's expert outputs
    combined without the residual (out = x + delta is rounded to bf16 after
    the add, so out - x cannot resolve a delta much smaller than x)."""
    wl = layer.wl
    delta = B.moe_combine(layer.y, layer.slot_pos, layer.w, wl.T)
    status_ok(B)
    ref = O.moe_forward_with_routing(xn_ref[rows], cpu["W1"], cpu["W3"], cpu["W2"], w_eff[rows], idx_eff[rows])
    check_close(to_np(delta)[rows], ref, "bf16", f"{what} MoE delta")
    # The residual add rounds x + (fp32 delta) once; the bf16 delta above was
    # rounded once too, so the two differ by at most one bf16 unit in the
    # last place of the result plus the rounding of the delta.
    dl = to_np(delta)[rows]
    want = O.round_to_bf16(O.f64(cpu["x"][rows]) + dl)
    got = to_np(layer.out)[rows]
    assert np.all(np.abs(got - want) <= 2.0 ** -7 * (np.abs(want) + np.abs(dl)) + 1e-30)


def test_block_delta_small(B):
    import bench
    wl = mw.get("small_block")
    cpu = inputs("small_block")
    layer = bench.Layer(wl, cpu, DEV)
    layer.step()
    status_ok(B)
    xn = O.block_normed_input(cpu["x"], cpu["gamma"], wl.eps)
    ora_w, ora_idx, logits = O.router(xn, cpu["Wg"], wl.k)
    tol, extra = block_input_tolerance(to_np(layer.xn), xn, cpu["Wg"])
    check_routing(to_np(layer.idx), to_np(layer.w), ora_idx, ora_w, logits, wl.k, w_tol=tol, extra_gap=extra)
    w_eff, idx_eff = effective_routing(to_np(layer.idx), ora_w, ora_idx, logits)
    block_delta_check(B, layer, xn, cpu, np.arange(wl.T), w_eff, idx_eff, "small_block")


def test_forward_edge_cases(B):
    r = np.random.default_rng(17)

    def run(T, d, F, E, k, scale=0.05):
        x = torch.from_numpy(r.standard_normal((T, d))).to(torch.bfloat16)
        Wg = torch.from_numpy(r.standard_normal((E, d)) * scale).to(torch.bfloat16)
        W1 = torch.from_numpy(r.standard_normal((E, F, d)) * scale).to(torch.bfloat16)
        W3 = torch.from_numpy(r.standard_normal((E, F, d)) * scale).to(torch.bfloat16)
        W2 = torch.from_numpy(r.standard_normal((E, d, F)) * scale).to(torch.bfloat16)
        out = B.moe_forward(dev(x), dev(Wg), dev(W1), dev(W3), dev(W2), k)
        status_ok(B)
        ref, w, idx, logits = O.moe_forward(x, Wg, W1, W3, W2, k)
        gidx, _ = B.moe_router_topk(dev(x), dev(Wg), k)
        w2, i2 = effective_routing(to_np(gidx), w, idx, logits)
        if not np.array_equal(i2, idx):
            ref = O.moe_forward_with_routing(x, W1, W3, W2, w2, i2)
        check_close(to_np(out), ref, "bf16", f"T={T} d={d} F={F} E={E} k={k}")

    run(1, 64, 64, 8, 2)       # one token, smallest tile-legal sizes
    run(37, 128, 192, 1, 1)    # E=1, k=1: the dense SwiGLU FFN
    run(50, 128, 128, 4, 1)    # k=1
    run(130, 128, 128, 2, 2)   # E=2, k=2: every token uses both experts
    run(20, 256, 128, 64, 8)   # E=64, k=8
    x = torch.zeros((0, 64), dtype=torch.bfloat16, device=DEV)
    assert B.moe_forward(x, torch.zeros((8, 64), dtype=torch.bfloat16, device=DEV),
                         *(torch.zeros((8, 64, 64), dtype=torch.bfloat16, device=DEV) for _ in range(3)), 2).shape == (0, 64)


def test_forward_identical_experts(B):
    """All experts equal: the layer is one SwiGLU whatever the routing."""
    r = np.random.default_rng(23)
    T, d, F, E = 200, 256, 256, 8
    x = torch.from_numpy(r.standard_normal((T, d))).to(torch.bfloat16)
    Wg = torch.from_numpy(r.standard_normal((E, d)) * 0.05).to(torch.bfloat16)
    one = [torch.from_numpy(r.standard_normal(s) * 0.05).to(torch.bfloat16) for s in ((F, d), (F, d), (d, F))]
    W1, W3, W2 = (m.unsqueeze(0).repeat(E, 1, 1).contiguous() for m in one)
    out = B.moe_forward(dev(x), dev(Wg), dev(W1), dev(W3), dev(W2), 2)
    status_ok(B)
    check_close(to_np(out), O.swiglu_expert(x, *one), "bf16", "identical experts")


# ------------------------------------------------------------------ full size
_SHARED = {}
FULL = ["decode", "prefill", "skewed", "skewed_zero", "block"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(B, name):
    """Full Mixtral sizes, run exactly as bench.py runs a step; routing is
    checked on every token, outputs on 192 seeded tokens + every near-tie
    token + the first and last."""
    import bench
    wl = mw.get(name)
    cpu = bench.make_tensors(wl, _SHARED)
    layer = bench.Layer(wl, cpu, DEV)
    out = layer.step()
    out = layer.step()  # a second call on the same buffers must give the same answer
    status_ok(B)
    if wl.block:
        xin = O.block_normed_input(cpu["x"], cpu["gamma"], wl.eps)
    else:
        xin = O.f64(cpu["x"])
    ora_w, ora_idx, logits = O.router(xin, cpu["Wg"], wl.k)
    kw = {}
    if wl.block:
        tol, extra = block_input_tolerance(to_np(layer.xn), xin, cpu["Wg"])
        kw = {"w_tol": tol, "extra_gap": extra}
        print(f"{name}: normalised elements rounded differently: {int(np.sum(to_np(layer.xn) != xin))}")
    n_tie, n_diff = check_routing(to_np(layer.idx), to_np(layer.w), ora_idx, ora_w, logits, wl.k, **kw)
    counts = np.bincount(ora_idx.ravel(), minlength=wl.E)
    assert np.array_equal(to_np(layer.counts), counts)
    if name == "skewed_zero":
        assert counts[mw.SKEW_ZERO_EXPERT] == 0
    r = np.random.default_rng(1)
    sample = set(r.choice(wl.T, size=min(192, wl.T), replace=False).tolist())
    thr = near_tie_mask(logits, wl.k, 1e-3 + 2.0 * kw["extra_gap"]) if wl.block else near_tie_mask(logits, wl.k)
    sample |= set(np.nonzero(thr)[0].tolist()) | {0, wl.T - 1}
    s = np.array(sorted(sample))
    w_eff, idx_eff = effective_routing(to_np(layer.idx), ora_w, ora_idx, logits)
    ref = O.moe_forward_with_routing(xin[s], cpu["W1"], cpu["W3"], cpu["W2"], w_eff[s], idx_eff[s])
    got = to_np(out)[s]
    if wl.block:
        block_delta_check(B, layer, xin, cpu, s, w_eff, idx_eff, name)
        ref = ref + O.f64(cpu["x"][s])
    check_close(got, ref, "bf16", f"{name} out")
    print(f"{name}: near-tie tokens {n_tie}, routed differently {n_diff}, expert counts {counts.tolist()}")


@pytest.mark.parametrize("T,E,k,d", [(1, 8, 2, 256), (7, 8, 2, 4096), (16, 8, 2, 4096), (33, 8, 2, 512),
                                     (64, 8, 2, 1024), (16, 64, 8, 256), (100, 8, 1, 512)])
def test_layer_routing_tables_match_step_entry_points(B, T, E, k, d):
    """The layer call's routing, dispatch tables and permuted rows (read from
    its scratch) equal those of moe_router_topk + moe_permute bit for bit."""
    r = np.random.default_rng(T * 131 + E)
    F = 128
    x = torch.from_numpy(r.standard_normal((T, d))).to(torch.bfloat16)
    Wg = torch.from_numpy(r.standard_normal((E, d)) * 0.02).to(torch.bfloat16)
    W = [torch.from_numpy(r.standard_normal(s) * 0.05).to(torch.bfloat16) for s in ((E, F, d), (E, F, d), (E, d, F))]
    g = [dev(v) for v in (x, Wg, *W)]
    ws = B.workspace(T, d, F, E, k, B.MOE_DTYPE_BF16)
    B.moe_forward_ws(*g, k, ws)
    status_ok(B)
    v = B.workspace_views(ws, T, d, F, E, k)
    idx, w = B.moe_router_topk(g[0], g[1], k)
    counts, offsets, row_src, slot_pos, x_perm = B.moe_permute(g[0], idx, E)
    status_ok(B)
    assert torch.equal(v["idx"], idx) and torch.equal(v["w"], w)
    assert torch.equal(v["counts"], counts) and torch.equal(v["offsets"], offsets)
    assert torch.equal(v["row_src"], row_src) and torch.equal(v["slot_pos"], slot_pos)
    assert torch.equal(v["x_perm"], x_perm)
