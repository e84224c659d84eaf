"""Parity of the backward (Mixtral 8x7B model reference page, Training:
experts and router trained together) through the C ABI with the fp64 oracle's
gradients, on GPU.

The forward runs with caller scratch (moe_forward_ws); that scratch is the
backward's `saved` input.  dout is a seeded normal in bf16.  The oracle
differentiates with the GPU's routing wherever the forward's routing was a
near tie.  Gradients are compared by relative L2 (bf16 tolerance, 5e-3) and
a per-element bound; an expert with no tokens must get exactly zero weight
gradients.

Per-element bound (parity.check_backward_close): 2^-7 times the element's
sum of absolute terms through the chain, from the oracle - the first-order
bound of sums of products of bf16-rounded factors (the forward's h and y;
the backward's dy, da, db and permuted dx) accumulated in fp32.  The
gradients are sums in which terms can cancel, so neither the element nor its
row's RMS bounds their rounding error; a wrong row or tile breaks this bound
by orders of magnitude.
"""
import numpy as np
import pytest
import torch

import moe_workloads as mw
import oracle.moe_oracle as O
from parity import check_backward_close, check_routing, effective_routing, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from sparse_mixture_experts_50_b300 import binding
    binding.lib()
    binding.moe_get_device_status(reset=True)
    return binding


def status_ok(B):
    s = B.moe_get_device_status(reset=True)
    assert s == 0, f"device status {s}"


def seeded_dout(T, d, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn((T, d), generator=g).to(torch.bfloat16)


def run_gpu(B, t, k, dout, entry="alloc"):
    """entry: "alloc" / "ws" = moe_backward / moe_backward_ws after
    moe_forward_ws (a and b recomputed); "keep" / "ws_keep" the same after
    moe_forward_train_ws, with its kept a and b."""
    g = {n: v.to(DEV).contiguous() for n, v in t.items()}
    T, d = g["x"].shape
    E, F, _ = g["W1"].shape
    saved = B.workspace(T, d, F, E, k, B.MOE_DTYPE_BF16)
    keep = None
    if entry.endswith("keep"):
        _, keep = B.moe_forward_train_ws(g["x"], g["Wg"], g["W1"], g["W3"], g["W2"], k, saved)
    else:
        B.moe_forward_ws(g["x"], g["Wg"], g["W1"], g["W3"], g["W2"], k, saved)
    dd = dout.to(DEV)
    if entry.startswith("ws"):
        ws = torch.empty(B.moe_backward_workspace_bytes(T, d, F, E, k), dtype=torch.uint8, device=DEV)
        grads = B.moe_backward_ws(dd, g["x"], g["Wg"], g["W1"], g["W3"], g["W2"], k, saved, ws, keep=keep)
    else:
        grads = B.moe_backward(dd, g["x"], g["Wg"], g["W1"], g["W3"], g["W2"], k, saved, keep=keep)
    status_ok(B)
    v = B.workspace_views(saved, T, d, F, E, k)
    return grads, v["idx"].cpu().numpy(), v["w"].cpu().numpy()


def oracle_grads(t, k, dout, gidx, gw, experts=None):
    ora_w, ora_idx, logits = O.router(t["x"], t["Wg"], k)
    check_routing(gidx, gw, ora_idx, ora_w, logits, k)
    _, idx_eff = effective_routing(gidx, ora_w, ora_idx, logits)
    return O.moe_backward(t["x"], t["Wg"], t["W1"], t["W3"], t["W2"], k, dout, idx=idx_eff, experts=experts,
                          with_scale=True), idx_eff


@pytest.mark.parametrize("name", ["small_bf16", "small_ragged", "small_skewed_zero"])
@pytest.mark.parametrize("entry", ["alloc", "ws", "keep", "ws_keep"])
def test_backward_small(B, name, entry):
    wl = mw.get(name)
    t = mw.make_inputs(wl)
    dout = seeded_dout(wl.T, wl.d, 7)
    grads, gidx, gw = run_gpu(B, t, wl.k, dout, entry)
    ref, idx_eff = oracle_grads(t, wl.k, dout, gidx, gw)
    for n in ("dx", "dWg", "dW1", "dW3", "dW2"):
        check_backward_close(to_np(grads[n]), ref[n], ref[n + "_scale"], f"{name} {n}")
    used = set(np.unique(idx_eff).tolist())
    for e in range(wl.E):
        if e not in used:
            for n in ("dW1", "dW3", "dW2"):
                assert torch.count_nonzero(grads[n][e]).item() == 0, f"{name}: unused expert {e} has {n} != 0"


def test_backward_linear_in_dout(B):
    """Scaling dout by 2 scales every gradient by exactly 2 (every rounding
    step commutes with a power of two), so the GPU gradients are linear and
    deterministic."""
    wl = mw.get("small_bf16")
    t = mw.make_inputs(wl)
    dout = seeded_dout(wl.T, wl.d, 8)
    g1, _, _ = run_gpu(B, t, wl.k, dout)
    g2, _, _ = run_gpu(B, t, wl.k, dout * 2)
    for n in g1:
        assert torch.equal(g2[n], 2 * g1[n]), n


@pytest.mark.parametrize("entry", ["alloc", "keep"])
def test_backward_mixtral_shape(B, entry):
    """Mixtral sizes (d=4096, d_ff=14336, E=8, top-2) at 64 tokens: dx and dWg
    in full, the expert weight gradients of two experts."""
    wl = mw.get("decode").with_tokens(64)
    t = mw.make_inputs(wl)
    dout = seeded_dout(wl.T, wl.d, 9)
    grads, gidx, gw = run_gpu(B, t, wl.k, dout, entry)
    counts = np.bincount(gidx.ravel(), minlength=wl.E)
    pick = [int(np.argmax(counts)), int(np.argmin(np.where(counts > 0, counts, 1 << 30)))]
    ref, _ = oracle_grads(t, wl.k, dout, gidx, gw, experts=pick)
    for n in ("dx", "dWg"):
        check_backward_close(to_np(grads[n]), ref[n], ref[n + "_scale"], f"mixtral {n}")
    for e in pick:
        for n in ("dW1", "dW3", "dW2"):
            check_backward_close(to_np(grads[n][e]), ref[n][e], ref[n + "_scale"][e], f"mixtral {n}[{e}]")


@pytest.mark.parametrize("name", ["small_ragged", "decode"])
def test_forward_train_keeps_swiglu_derivatives(B, name):
    """moe_forward_train_ws: the same output and scratch as moe_forward_ws
    (bit for bit: the same kernels), plus the SwiGLU's local derivatives of
    every permuted row in bf16, p = b silu'(a) and q = silu(a) at
    a = x W1_e^T, b = x W3_e^T, checked against the oracle's fp64 values with
    the bf16 forward tolerance.  "decode" (T=1) runs the small-batch GEMM
    form, small_ragged the tiled one."""
    from parity import check_close
    wl = mw.get(name)
    t = mw.make_inputs(wl)
    g = {n: v.to(DEV).contiguous() for n, v in t.items()}
    T, d, F, E, k = wl.T, wl.d, wl.F, wl.E, wl.k
    ws1 = B.workspace(T, d, F, E, k)
    ws2 = B.workspace(T, d, F, E, k)
    ws1.zero_()
    ws2.zero_()
    out1 = B.moe_forward_ws(g["x"], g["Wg"], g["W1"], g["W3"], g["W2"], k, ws1)
    out2, keep = B.moe_forward_train_ws(g["x"], g["Wg"], g["W1"], g["W3"], g["W2"], k, ws2)
    status_ok(B)
    assert torch.equal(out1, out2)
    assert torch.equal(ws1, ws2)
    v = B.workspace_views(ws2, T, d, F, E, k)
    offs = v["offsets"].cpu().numpy()
    row_src = v["row_src"].cpu().numpy()
    p_got, q_got = to_np(keep[0]), to_np(keep[1])
    for e in range(E):
        lo, hi = int(offs[e]), int(offs[e + 1])
        if hi == lo:
            continue
        xs = to_np(t["x"])[row_src[lo:hi]]
        a, b = O.gate_up_preactivations(xs, to_np(t["W1"][e]), to_np(t["W3"][e]))
        check_close(p_got[lo:hi], b * O.silu_grad(a), "bf16", f"{name} p[{e}]")
        check_close(q_got[lo:hi], O.silu(a), "bf16", f"{name} q[{e}]")


def test_backward_full_size_sampled(B):
    """The backward at T=4096 with Mixtral shapes, in the configuration
    bench.py times (the training forward keeps p and q, then
    moe_backward_ws), checked on outputs the oracle computes one by one:
    dx of 12 sampled tokens (a token's dx depends on that token alone), and
    for 2 experts x 3 hidden units the row of dW1 and of dW3 and the column of
    dW2, over all of that expert's routed rows (expert_grad_hidden_unit)."""
    wl = mw.get("prefill_bwd")
    t = mw.make_inputs(wl)
    T, d, F, E, k = wl.T, wl.d, wl.F, wl.E, wl.k
    dout = t["dout"]
    g = {n: v.to(DEV).contiguous() for n, v in t.items()}
    saved = B.workspace(T, d, F, E, k)
    _, keep = B.moe_forward_train_ws(g["x"], g["Wg"], g["W1"], g["W3"], g["W2"], k, saved)
    ws = torch.empty(B.moe_backward_workspace_bytes(T, d, F, E, k), dtype=torch.uint8, device=DEV)
    grads = B.moe_backward_ws(g["dout"], g["x"], g["Wg"], g["W1"], g["W3"], g["W2"], k, saved, ws, keep=keep)
    status_ok(B)
    v = B.workspace_views(saved, T, d, F, E, k)
    gidx, gw = v["idx"].cpu().numpy(), v["w"].cpu().numpy()
    ora_w, ora_idx, logits = O.router(t["x"], t["Wg"], k)
    check_routing(gidx, gw, ora_idx, ora_w, logits, k)
    w_eff, idx_eff = effective_routing(gidx, ora_w, ora_idx, logits)
    rng = np.random.default_rng(11)
    S = np.sort(rng.choice(T, 12, replace=False))
    St = torch.from_numpy(S)
    ref = O.moe_backward(t["x"][St], t["Wg"], t["W1"], t["W3"], t["W2"], k, dout[St], idx=idx_eff[S],
                         with_scale=True, weight_grads=False)
    check_backward_close(to_np(grads["dx"][S.tolist()]), ref["dx"], ref["dx_scale"], "full-size dx (sampled tokens)")
    counts = np.bincount(idx_eff.ravel(), minlength=E)
    for e in (int(np.argmax(counts)), int(np.argmin(counts))):
        tok, slot = np.nonzero(idx_eff == e)
        tt = torch.from_numpy(tok)
        for f in rng.choice(F, 3, replace=False):
            f = int(f)
            r = O.expert_grad_hidden_unit(t["x"][tt], dout[tt], w_eff[tok, slot], t["W1"][e], t["W3"][e],
                                          t["W2"][e], f)
            check_backward_close(to_np(grads["dW1"][e, f]), r["dW1"], r["dW1_scale"], f"full-size dW1[{e},{f}]")
            check_backward_close(to_np(grads["dW3"][e, f]), r["dW3"], r["dW3_scale"], f"full-size dW3[{e},{f}]")
            check_backward_close(to_np(grads["dW2"][e, :, f]), r["dW2"], r["dW2_scale"], f"full-size dW2[{e},:,{f}]")
