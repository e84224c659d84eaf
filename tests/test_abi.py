"""The C-ABI library loads without a GPU, exports every symbol include/moe.h
declares, and rejects invalid arguments on the host before any CUDA call
(CPU only: none of these calls reaches the device)."""
import ctypes
import os
import re

import pytest

from sparse_mixture_experts_50_b300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(moe_[a-z0-9_]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    return B.lib()


def test_header_declares_the_layer_steps():
    names = declared_functions()
    for n in ["moe_router_topk", "moe_permute", "moe_expert_ffn", "moe_combine", "moe_forward",
              "moe_forward_f32", "moe_block_forward", "moe_rmsnorm", "moe_expert_gate_up", "moe_expert_down"]:
        assert n in names


# The layer's boundary calls, with each call's argument count
# (pointers, sizes, dtype and stream, in the header's order).
BOUNDARY_CALLS = {
    "moe_router_topk": 11,       # x, Wg, T, d, E, k, topk_idx, topk_w, logits_opt, dtype, stream
    "moe_permute": 13,           # x, topk_idx, T, d, E, k, counts, offsets, row_src, slot_pos, x_perm, dtype, stream
    "moe_expert_ffn": 12,        # x_perm, offsets, W1, W3, W2, y_perm, Tk, d, dff, E, dtype, stream
    "moe_combine": 10,           # y_perm, slot_pos, topk_w, residual_opt, out, T, d, k, dtype, stream
    "moe_forward": 12,           # x, Wg, W1, W3, W2, out, T, d, dff, E, k, stream
    "moe_forward_f32": 12,
    "moe_block_forward": 14,     # x, gamma, eps, then moe_forward's arguments
    "moe_workspace_bytes": 6,    # T, d, dff, E, k, dtype
}


def test_boundary_names_and_arities():
    names = declared_functions()
    for n, nargs in BOUNDARY_CALLS.items():
        assert n in names, f"include/moe.h does not declare {n}"
        assert len(B.SIGNATURES[n][1]) == nargs, (n, len(B.SIGNATURES[n][1]), nargs)
    assert B.SIGNATURES["moe_workspace_bytes"][0] is ctypes.c_size_t


def test_expert_ffn_validation(lib):
    """moe_expert_ffn checks its arguments before it allocates anything."""
    f = lib.moe_expert_ffn
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 10, 96, 128, 8, 1, NULL) == B.MOE_EUNSUPPORTED  # d % 64
    assert f(FAKE, NULL, FAKE, FAKE, FAKE, FAKE, 10, 128, 128, 8, 1, NULL) == B.MOE_EINVAL      # null offsets
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 8, 10, 128, 128, 8, 1, NULL) == B.MOE_EINVAL  # misaligned out
    assert f(NULL, NULL, NULL, NULL, NULL, NULL, 0, 128, 128, 8, 1, NULL) == B.MOE_OK           # Tk = 0
    g = lib.moe_expert_ffn_ws
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, NULL, FAKE, 10, 128, 128, 8, 1, NULL) == B.MOE_EINVAL  # null h_perm


def test_every_declared_symbol_is_exported_and_bound(lib):
    names = declared_functions()
    assert len(names) >= 19
    for n in names:
        assert hasattr(lib, n), f"libmoe.so does not export {n}"
        assert n in B.SIGNATURES, f"binding has no signature for {n}"
    assert sorted(B.SIGNATURES) == names


def test_version_and_status_strings(lib):
    assert lib.moe_version() == 100
    assert B.status_string(0) == "ok"
    for code in (-1, -2, -3, -4, -5, -6):
        assert B.status_string(code) not in ("ok", "unknown status")
    assert B.status_string(-99) == "unknown status"


NULL = None
FAKE = 0x7F0000000000  # never dereferenced: validation fails first


@pytest.mark.parametrize("args,want", [
    ((FAKE, FAKE, -1, 64, 8, 2, FAKE, FAKE, NULL, 1, NULL), B.MOE_EINVAL),    # T < 0
    ((FAKE, FAKE, 4, 64, 8, 9, FAKE, FAKE, NULL, 1, NULL), B.MOE_EINVAL),     # k > E
    ((FAKE, FAKE, 4, 64, 65, 2, FAKE, FAKE, NULL, 1, NULL), B.MOE_EUNSUPPORTED),  # E > 64
    ((FAKE, FAKE, 4, 64, 16, 9, FAKE, FAKE, NULL, 1, NULL), B.MOE_EUNSUPPORTED),  # k > 8
    ((FAKE, FAKE, 4, 60, 8, 2, FAKE, FAKE, NULL, 1, NULL), B.MOE_EUNSUPPORTED),   # bf16 d % 8
    ((FAKE, FAKE, 4, 64, 8, 2, FAKE, FAKE, NULL, 7, NULL), B.MOE_EINVAL),     # bad dtype
    ((NULL, FAKE, 4, 64, 8, 2, FAKE, FAKE, NULL, 1, NULL), B.MOE_EINVAL),     # null x
    ((FAKE + 2, FAKE, 4, 64, 8, 2, FAKE, FAKE, NULL, 1, NULL), B.MOE_EINVAL),  # misaligned x
    ((NULL, NULL, 0, 64, 8, 2, NULL, NULL, NULL, 1, NULL), B.MOE_OK),         # T = 0 no-op
])
def test_router_validation(lib, args, want):
    assert lib.moe_router_topk(*args) == want


def test_expert_ffn_shape_rules(lib):
    f = lib.moe_expert_gate_up
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 10, 96, 128, 8, 1, NULL) == B.MOE_EUNSUPPORTED  # d % 64
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 10, 128, 96, 8, 1, NULL) == B.MOE_EUNSUPPORTED  # dff % 64
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, -1, 128, 128, 8, 1, NULL) == B.MOE_EINVAL
    assert f(FAKE, NULL, FAKE, FAKE, FAKE, 10, 128, 128, 8, 1, NULL) == B.MOE_EINVAL  # null offsets
    assert f(NULL, NULL, NULL, NULL, NULL, 0, 128, 128, 8, 1, NULL) == B.MOE_OK  # Tk = 0
    g = lib.moe_expert_down
    assert g(FAKE, FAKE, FAKE, FAKE, 10, 4096, 14300, 8, 1, NULL) == B.MOE_EUNSUPPORTED
    assert g(NULL, NULL, NULL, NULL, 0, 4096, 14336, 8, 1, NULL) == B.MOE_OK


def test_forward_validation(lib):
    f = lib.moe_forward
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, 4096, 14300, 8, 2, NULL) == B.MOE_EUNSUPPORTED
    assert f(FAKE, FAKE, FAKE, FAKE, NULL, FAKE, 16, 4096, 14336, 8, 2, NULL) == B.MOE_EINVAL
    assert f(NULL, NULL, NULL, NULL, NULL, NULL, 0, 4096, 14336, 8, 2, NULL) == B.MOE_OK
    ws = lib.moe_forward_ws
    # workspace misaligned / missing
    assert ws(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, 4096, 14336, 8, 2, 1, NULL, 1 << 30, NULL) == B.MOE_EINVAL
    assert ws(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, 4096, 14336, 8, 2, 1, FAKE + 16, 1 << 30, NULL) == B.MOE_EINVAL
    blk = lib.moe_block_forward
    assert blk(FAKE, FAKE, ctypes.c_float(-1.0), FAKE, FAKE, FAKE, FAKE, FAKE, 4, 4096, 14336, 8, 2, NULL) == B.MOE_EINVAL
    assert blk(FAKE, NULL, ctypes.c_float(1e-5), FAKE, FAKE, FAKE, FAKE, FAKE, 4, 4096, 14336, 8, 2, NULL) == B.MOE_EINVAL


def test_workspace_bytes(lib):
    T, d, F, E, k = 8192, 4096, 14336, 8, 2
    n = lib.moe_workspace_bytes(T, d, F, E, k, 1)
    # x_perm + h + y + xn (bf16) plus index arrays
    act = T * k * d * 2 + T * k * F * 2 + T * k * d * 2 + T * d * 2
    assert act < n < act + 1 << 20
    assert lib.moe_workspace_bytes(-1, d, F, E, k, 1) == 0
    h = lib.moe_forward_host_workspace_bytes(T, d, F, E, k, 1)
    assert h == n + 2 * T * d * 2


def test_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        B.moe_router_topk(x, torch.zeros(8, 64, dtype=torch.bfloat16), 2)


def test_w8_workspace_bytes(lib):
    """The int8 layer needs the bf16 layer's scratch and nothing more: its
    weights are widened on the SM, never into a bf16 copy."""
    d, F, E, k = 4096, 14336, 8, 2
    for T in (1, 16, 2047, 2048, 4096, 8192):
        assert lib.moe_forward_w8_workspace_bytes(T, d, F, E, k) == \
            lib.moe_workspace_bytes(T, d, F, E, k, B.MOE_DTYPE_BF16)
    assert lib.moe_forward_w8_workspace_bytes(-1, d, F, E, k) == 0


def test_training_entry_validation(lib):
    """moe_forward_train_ws needs its keep buffer; moe_backward_ws checks
    keep's alignment and both scratch sizes before any device work."""
    T, d, F, E, k = 16, 4096, 14336, 8, 2
    fwd = lib.moe_forward_train_ws
    assert fwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, NULL, T, d, F, E, k, FAKE, 1 << 30, NULL) == B.MOE_EINVAL
    assert fwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 8, T, d, F, E, k, FAKE, 1 << 30, NULL) == B.MOE_EINVAL
    assert fwd(NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, d, F, E, k, NULL, 0, NULL) == B.MOE_OK
    bwd = lib.moe_backward_ws
    saved = lib.moe_workspace_bytes(T, d, F, E, k, B.MOE_DTYPE_BF16)
    need = lib.moe_backward_workspace_bytes(T, d, F, E, k)
    assert need > 0

    def call(keep=NULL, saved_bytes=saved, ws_bytes=need, T=T):
        return bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, saved_bytes, keep, FAKE, FAKE, FAKE, FAKE, FAKE,
                   T, d, F, E, k, FAKE, ws_bytes, NULL)
    assert call(keep=FAKE + 8) == B.MOE_EINVAL          # keep not 16-byte aligned
    assert call(saved_bytes=saved - 1) == B.MOE_ENOMEM  # saved scratch too small
    assert call(ws_bytes=need - 1) == B.MOE_ENOMEM      # backward scratch too small
    assert call(T=0) == B.MOE_OK


def test_gather_rows_validation(lib):
    f = lib.moe_gather_rows
    assert f(FAKE, 10, FAKE, 4, FAKE, 24, NULL) == B.MOE_EINVAL       # row bytes not a multiple of 16
    assert f(FAKE, 10, FAKE, 4, FAKE, 0, NULL) == B.MOE_EINVAL        # empty rows
    assert f(FAKE + 8, 10, FAKE, 4, FAKE, 32, NULL) == B.MOE_EINVAL   # misaligned src
    assert f(FAKE, 10, NULL, 4, FAKE, 32, NULL) == B.MOE_EINVAL       # null index
    assert f(FAKE, -1, FAKE, 4, FAKE, 32, NULL) == B.MOE_EINVAL
    assert f(NULL, 0, NULL, 0, NULL, 32, NULL) == B.MOE_OK            # nothing to copy
