"""Bounded device waits (GPU): a wait that runs out is reported, not hung.

The expert GEMM kernel bounds every spin on an mbarrier by a time limit set
with moe_set_wait_limit_ns.  With a 1 ns limit the first wait that has to
spin gives up: the kernel records MOE_ETIMEOUT, drains the copies and MMAs it
already issued (those drains keep a 2 s floor), frees its tensor memory and
returns.  The tests check the status and that the same context then computes
correct results with the default limit: for the large-batch form, and for
the small-batch forms (bf16, and int8 with its converter warps and two
MMA-issuing threads).
"""
import numpy as np
import pytest
import torch

import oracle.moe_oracle as O
from parity import check_close, to_np

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_survives():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from sparse_mixture_experts_50_b300 import binding as B
    r = np.random.default_rng(2)
    E, d, F = 8, 512, 1024
    counts = [300, 0, 129, 64, 1, 500, 7, 255]
    offsets = np.concatenate([[0], np.cumsum(counts)])
    Tk = int(offsets[-1])
    x = torch.from_numpy(r.standard_normal((Tk, d))).to(torch.bfloat16).cuda()
    W1, W3 = (torch.from_numpy(r.standard_normal((E, F, d)) * 0.05).to(torch.bfloat16).cuda() for _ in range(2))
    off = torch.from_numpy(offsets).int().cuda()
    B.moe_get_device_status(reset=True)
    try:
        B.moe_set_wait_limit_ns(1)
        B.moe_expert_gate_up(x, off, W1, W3)
        status = B.moe_get_device_status(reset=True)
    finally:
        B.moe_set_wait_limit_ns(0)  # back to the default limit
    assert status == B.MOE_ETIMEOUT
    h = B.moe_expert_gate_up(x, off, W1, W3)
    assert B.moe_get_device_status(reset=True) == 0
    xc, W1c, W3c = x.cpu(), W1.cpu(), W3.cpu()
    ref = np.zeros((Tk, F))
    for e in range(E):
        a, b = offsets[e], offsets[e + 1]
        if b > a:
            ref[a:b] = O.swiglu_hidden(xc[a:b], W1c[e], W3c[e])
    check_close(to_np(h), ref, "bf16", "h after a timed-out launch")


@pytest.mark.parametrize("w8", [False, True], ids=["bf16", "int8"])
def test_small_batch_wait_timeout(w8):
    """Decode-sized GEMMs (32 routed rows over 8 experts, one empty): a 1 ns
    limit ends both GEMMs with MOE_ETIMEOUT, and the next calls with the
    default limit give the same bits as the calls made before it.  K is
    long (d=4096, dff=2048: 32-64 weight stages per tile), so the epilogue's
    wait for its first accumulator outlasts any suspension of a barrier
    try-wait and has to spin; with K=512 a whole launch could finish inside
    the first try-waits and report no timeout."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from sparse_mixture_experts_50_b300 import binding as B
    E, d, F = 8, 4096, 2048
    counts = [5, 5, 6, 0, 2, 7, 3, 4]
    offsets = np.concatenate([[0], np.cumsum(counts)])
    Tk = int(offsets[-1])
    g = torch.Generator(device="cuda").manual_seed(3)
    x = torch.randn(Tk, d, device="cuda", generator=g).to(torch.bfloat16)
    W1, W3 = ((torch.randn(E, F, d, device="cuda", generator=g) * 0.02).to(torch.bfloat16) for _ in range(2))
    W2 = (torch.randn(E, d, F, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    off = torch.from_numpy(offsets).int().cuda()
    B.moe_get_device_status(reset=True)
    if w8:
        (q1, s1), (q3, s3), (q2, s2) = (B.moe_quantize_int8(W) for W in (W1, W3, W2))

        def run():
            h = B.moe_expert_gate_up_w8(x, off, q1, s1, q3, s3)
            return h, B.moe_expert_down_w8(h, off, q2, s2)
    else:
        def run():
            h = B.moe_expert_gate_up(x, off, W1, W3)
            return h, B.moe_expert_down(h, off, W2)
    h0, y0 = (t.clone() for t in run())
    assert B.moe_get_device_status(reset=True) == 0
    try:
        B.moe_set_wait_limit_ns(1)
        run()
        status = B.moe_get_device_status(reset=True)
    finally:
        B.moe_set_wait_limit_ns(0)
    assert status == B.MOE_ETIMEOUT
    h1, y1 = run()
    assert B.moe_get_device_status(reset=True) == 0
    assert torch.equal(h1, h0) and torch.equal(y1, y0)
