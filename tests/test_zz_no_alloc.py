"""moe_forward_noalloc: the bf16 layer for callers that must not allocate
device memory while they run (its scratch is a fixed 16 MiB array inside the
library), checked bit for bit against moe_forward on two calls in a row, and
a Mixtral-shape decode call against the oracle (GPU).

Both entry points run the same kernels on the same inputs, so their outputs
must be identical; a difference would mean scratch left by an earlier call
leaked into a later one.  The two calls of each pair use different inputs
and token counts, so the second runs on the scratch the first left behind.
The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import moe_workloads as mw
import oracle.moe_oracle as O
from parity import check_close, check_routing, effective_routing, to_np

pytestmark = pytest.mark.gpu

NOALLOC_SCRATCH_BYTES = 16 << 20


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from sparse_mixture_experts_50_b300 import binding
    binding.lib()
    binding.moe_get_device_status(reset=True)
    return binding


def call_noalloc(B, x, Wg, W1, W3, W2, k):
    """Straight through the C ABI."""
    T, d = x.shape
    E, dff, _ = W1.shape
    out = torch.empty_like(x)
    rc = B.lib().moe_forward_noalloc(x.data_ptr(), Wg.data_ptr(), W1.data_ptr(), W3.data_ptr(), W2.data_ptr(),
                                     out.data_ptr(), T, d, dff, E, k, torch.cuda.current_stream().cuda_stream)
    assert rc == 0, B.status_string(rc)
    return out


def test_noalloc_matches_moe_forward_twice(B):
    wl = mw.get("small_bf16")
    t = {n: v.cuda() for n, v in mw.make_inputs(wl).items()}
    r = np.random.default_rng(9)
    x2 = torch.from_numpy(r.standard_normal((123, wl.d))).to(torch.bfloat16).cuda()
    for x in (t["x"], x2):  # two calls in a row, different T
        got = call_noalloc(B, x, t["Wg"], t["W1"], t["W3"], t["W2"], wl.k)
        ref = B.moe_forward(x, t["Wg"], t["W1"], t["W3"], t["W2"], wl.k)
        assert B.moe_get_device_status(reset=True) == 0
        assert torch.equal(got, ref), f"noalloc differs from moe_forward, T={x.shape[0]}"


def test_noalloc_mixtral_decode_and_size_limit(B):
    wl = mw.get("decode")
    t = {n: v.cuda() for n, v in mw.make_inputs(wl).items()}
    outs = []
    for x in (t["x"], t["x"][:5].contiguous()):
        got = call_noalloc(B, x, t["Wg"], t["W1"], t["W3"], t["W2"], wl.k)
        ref = B.moe_forward(x, t["Wg"], t["W1"], t["W3"], t["W2"], wl.k)
        assert B.moe_get_device_status(reset=True) == 0
        assert torch.equal(got, ref), f"noalloc differs from moe_forward, decode T={x.shape[0]}"
        outs.append(got)
    # The first (all 16 decode tokens) against the fp64 oracle: routing exact
    # outside near ties, output within the bf16 bound.
    cpu = mw.make_inputs(wl)
    ora_out, ora_w, ora_idx, logits = O.moe_forward(cpu["x"], cpu["Wg"], cpu["W1"], cpu["W3"], cpu["W2"], wl.k)
    gidx, gw = B.moe_router_topk(t["x"], t["Wg"], wl.k)
    check_routing(to_np(gidx), to_np(gw), ora_idx, ora_w, logits, wl.k)
    w_eff, idx_eff = effective_routing(to_np(gidx), ora_w, ora_idx, logits)
    if not np.array_equal(idx_eff, ora_idx):
        ora_out = O.moe_forward_with_routing(cpu["x"], cpu["W1"], cpu["W3"], cpu["W2"], w_eff, idx_eff)
    check_close(to_np(outs[0]), ora_out, "bf16", "noalloc decode vs oracle")
    # The largest Mixtral-shape token count that fits, and the first that does not.
    need = B.lib().moe_workspace_bytes
    assert need(170, 4096, 14336, 8, 2, 1) <= NOALLOC_SCRATCH_BYTES < need(171, 4096, 14336, 8, 2, 1)
    big = torch.zeros((171, 4096), dtype=torch.bfloat16, device="cuda")
    rc = B.lib().moe_forward_noalloc(big.data_ptr(), t["Wg"].data_ptr(), t["W1"].data_ptr(), t["W3"].data_ptr(),
                                     t["W2"].data_ptr(), big.data_ptr(), 171, 4096, 14336, 8, 2,
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == B.MOE_ENOMEM
