"""Thin ctypes binding of libmoe (include/moe.h): argument marshalling only.

Every function here has the name of the C entry point it calls, takes CUDA
torch tensors, passes their device pointers, sizes and the current CUDA
stream, and raises ``MoEError`` on a non-zero status.  Output tensors the
caller does not pass are allocated with ``torch.empty`` on the input's device
(torch is used for device memory and streams only).  There is no CPU path:
a CPU tensor, or a missing ``libmoe.so``, raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe.so")

MOE_OK = 0
MOE_EINVAL = -1
MOE_EUNSUPPORTED = -2
MOE_ECUDA = -3
MOE_ETIMEOUT = -4
MOE_ENOMEM = -5
MOE_EDEVICE = -6
MOE_DTYPE_F32 = 0
MOE_DTYPE_BF16 = 1

_P, _I, _F, _SZ, _LL = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_longlong

# name -> (restype, argtypes), in the order of include/moe.h
SIGNATURES = {
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_version": (_I, []),
    "moe_router_topk": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _I, _P]),
    "moe_rmsnorm": (_I, [_P, _P, _F, _P, _I, _I, _I, _P]),
    "moe_permute": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _I, _P]),
    "moe_gather_rows": (_I, [_P, _I, _P, _I, _P, _SZ, _P]),
    "moe_expert_gate_up": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "moe_expert_down": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "moe_expert_ffn": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "moe_expert_ffn_ws": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "moe_combine": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "moe_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "moe_forward_w8_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "moe_forward_workspace_offsets": (_I, [_I, _I, _I, _I, _I, _I, ctypes.POINTER(_SZ)]),
    "moe_forward_ws": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _SZ, _P]),
    "moe_forward": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "moe_forward_f32": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "moe_block_forward_ws": (_I, [_P, _P, _F, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _SZ, _P]),
    "moe_block_forward": (_I, [_P, _P, _F, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "moe_forward_ex": (_I, [_P, _P, _F, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _SZ,
                            _P, _P]),
    "moe_forward_host_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "moe_forward_host": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _SZ, _P]),
    "moe_quantize_int8": (_I, [_P, _I, _I, _P, _P, _P]),
    "moe_expert_gate_up_w8": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "moe_expert_down_w8": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "moe_forward_w8_ws": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _SZ, _P]),
    "moe_forward_w8": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "moe_backward_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "moe_backward_ws": (_I, [_P, _P, _P, _P, _P, _P, _P, _SZ, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _SZ,
                             _P]),
    "moe_backward": (_I, [_P, _P, _P, _P, _P, _P, _P, _SZ, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "moe_forward_train_ws": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _SZ, _P]),
    "moe_forward_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "moe_get_device_status": (_I, [_P, ctypes.POINTER(_I), _I]),
    "moe_set_wait_limit_ns": (_I, [_LL]),
}


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status} ({status_string(status)})")


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libmoe.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m sparse_mixture_experts_50_b300.build`")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


def _check(name: str, rc: int) -> None:
    if rc != MOE_OK:
        raise MoEError(name, rc)


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return MOE_DTYPE_BF16
    if t.dtype == torch.float32:
        return MOE_DTYPE_F32
    raise TypeError(f"unsupported dtype {t.dtype}; libmoe takes bfloat16 or float32")


def _dev(*ts) -> None:
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("libmoe runs on the GPU only: got a CPU tensor")
        if not t.is_contiguous():
            raise ValueError("libmoe takes contiguous tensors")


def _p(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


# ------------------------------------------------------------------ steps
def moe_router_topk(x, Wg, k, topk_idx=None, topk_w=None, logits=None, stream=None):
    """Router (steps a1 + a2): returns (topk_idx[T,k] int32, topk_w[T,k] fp32)."""
    _dev(x, Wg, topk_idx, topk_w, logits)
    T, d = x.shape
    E = Wg.shape[0]
    if topk_idx is None:
        topk_idx = torch.empty((T, k), dtype=torch.int32, device=x.device)
    if topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=x.device)
    _check("moe_router_topk", lib().moe_router_topk(_p(x), _p(Wg), T, d, E, k, _p(topk_idx), _p(topk_w),
                                                    _p(logits), _dtype(x), _stream(stream)))
    return topk_idx, topk_w


def moe_rmsnorm(x, gamma, eps, xn=None, stream=None):
    """RMSNorm prologue (step a0): returns xn[T,d]."""
    _dev(x, gamma, xn)
    T, d = x.shape
    if xn is None:
        xn = torch.empty_like(x)
    _check("moe_rmsnorm", lib().moe_rmsnorm(_p(x), _p(gamma), eps, _p(xn), T, d, _dtype(x), _stream(stream)))
    return xn


def moe_permute(x, topk_idx, E, out=None, stream=None):
    """Dispatch (step a3): returns (counts, offsets, row_src, slot_pos, x_perm)."""
    _dev(x, topk_idx)
    T, d = x.shape
    k = topk_idx.shape[1]
    dev = x.device
    if out is None:
        out = (torch.empty(E, dtype=torch.int32, device=dev), torch.empty(E + 1, dtype=torch.int32, device=dev),
               torch.empty(T * k, dtype=torch.int32, device=dev), torch.empty(T * k, dtype=torch.int32, device=dev),
               torch.empty((T * k, d), dtype=x.dtype, device=dev))
    counts, offsets, row_src, slot_pos, x_perm = out
    _dev(*out)
    _check("moe_permute", lib().moe_permute(_p(x), _p(topk_idx), T, d, E, k, _p(counts), _p(offsets), _p(row_src),
                                            _p(slot_pos), _p(x_perm), _dtype(x), _stream(stream)))
    return counts, offsets, row_src, slot_pos, x_perm


def moe_gather_rows(src, row_idx, dst=None, stream=None):
    """dst[i] = src[row_idx[i]] (rows of any dtype, 16-byte multiples; row_idx int32)."""
    _dev(src, row_idx, dst)
    n = row_idx.shape[0]
    if dst is None:
        dst = src.new_empty((n,) + tuple(src.shape[1:]))
    row_bytes = src[0].numel() * src.element_size() if src.shape[0] else dst[0].numel() * dst.element_size()
    _check("moe_gather_rows", lib().moe_gather_rows(_p(src), src.shape[0], _p(row_idx), n, _p(dst), row_bytes,
                                                    _stream(stream)))
    return dst


def moe_expert_gate_up(x_perm, offsets, W1, W3, h_perm=None, stream=None):
    """Grouped gate/up GEMM + SwiGLU (step a4): returns h_perm[Tk,dff]."""
    _dev(x_perm, offsets, W1, W3, h_perm)
    Tk, d = x_perm.shape
    E, dff, _ = W1.shape
    if h_perm is None:
        h_perm = torch.empty((Tk, dff), dtype=x_perm.dtype, device=x_perm.device)
    _check("moe_expert_gate_up", lib().moe_expert_gate_up(_p(x_perm), _p(offsets), _p(W1), _p(W3), _p(h_perm), Tk,
                                                          d, dff, E, _dtype(x_perm), _stream(stream)))
    return h_perm


def moe_expert_down(h_perm, offsets, W2, y_perm=None, stream=None):
    """Grouped down-projection GEMM (step a5): returns y_perm[Tk,d]."""
    _dev(h_perm, offsets, W2, y_perm)
    Tk, dff = h_perm.shape
    E, d, _ = W2.shape
    if y_perm is None:
        y_perm = torch.empty((Tk, d), dtype=h_perm.dtype, device=h_perm.device)
    _check("moe_expert_down", lib().moe_expert_down(_p(h_perm), _p(offsets), _p(W2), _p(y_perm), Tk, d, dff, E,
                                                    _dtype(h_perm), _stream(stream)))
    return y_perm


def moe_expert_ffn(x_perm, offsets, W1, W3, W2, y_perm=None, stream=None):
    """Steps a4 + a5 (hidden activations in pool scratch): returns y_perm[Tk,d]."""
    _dev(x_perm, offsets, W1, W3, W2, y_perm)
    Tk, d = x_perm.shape
    E, dff, _ = W1.shape
    if y_perm is None:
        y_perm = torch.empty((Tk, d), dtype=x_perm.dtype, device=x_perm.device)
    _check("moe_expert_ffn", lib().moe_expert_ffn(_p(x_perm), _p(offsets), _p(W1), _p(W3), _p(W2), _p(y_perm), Tk,
                                                  d, dff, E, _dtype(x_perm), _stream(stream)))
    return y_perm


def moe_expert_ffn_ws(x_perm, offsets, W1, W3, W2, h_perm=None, y_perm=None, stream=None):
    """Steps a4 + a5 on caller scratch h_perm[Tk,dff]: returns (h_perm, y_perm)."""
    _dev(x_perm, offsets, W1, W3, W2, h_perm, y_perm)
    Tk, d = x_perm.shape
    E, dff, _ = W1.shape
    if h_perm is None:
        h_perm = torch.empty((Tk, dff), dtype=x_perm.dtype, device=x_perm.device)
    if y_perm is None:
        y_perm = torch.empty((Tk, d), dtype=x_perm.dtype, device=x_perm.device)
    _check("moe_expert_ffn_ws", lib().moe_expert_ffn_ws(_p(x_perm), _p(offsets), _p(W1), _p(W3), _p(W2),
                                                        _p(h_perm), _p(y_perm), Tk, d, dff, E, _dtype(x_perm),
                                                        _stream(stream)))
    return h_perm, y_perm


def moe_combine(y_perm, slot_pos, topk_w, T, residual=None, out=None, stream=None):
    """Combine + un-permute (step a6): returns out[T,d]."""
    _dev(y_perm, slot_pos, topk_w, residual, out)
    d = y_perm.shape[1]
    k = topk_w.shape[1]
    if out is None:
        out = torch.empty((T, d), dtype=y_perm.dtype, device=y_perm.device)
    _check("moe_combine", lib().moe_combine(_p(y_perm), _p(slot_pos), _p(topk_w), _p(residual), _p(out), T, d, k,
                                            _dtype(y_perm), _stream(stream)))
    return out


# ------------------------------------------------------------------ whole layer
def moe_workspace_bytes(T, d, dff, E, k, dtype=MOE_DTYPE_BF16) -> int:
    return int(lib().moe_workspace_bytes(T, d, dff, E, k, dtype))


def workspace_views(ws, T, d, dff, E, k, dtype=MOE_DTYPE_BF16):
    """Views of the layer's intermediates inside a forward scratch tensor:
    dict(idx, w, counts, offsets, row_src, slot_pos, x_perm, h, y, xn)."""
    o = (_SZ * 11)()
    _check("moe_forward_workspace_offsets", lib().moe_forward_workspace_offsets(T, d, dff, E, k, dtype, o))
    fdt = torch.bfloat16 if dtype == MOE_DTYPE_BF16 else torch.float32
    es = 2 if dtype == MOE_DTYPE_BF16 else 4

    def view(i, n, dt, shape):
        nbytes = n * (4 if dt in (torch.int32, torch.float32) else es)
        return ws[o[i]:o[i] + nbytes].view(dt).reshape(shape)

    Tk = T * k
    return {"idx": view(0, Tk, torch.int32, (T, k)), "w": view(1, Tk, torch.float32, (T, k)),
            "counts": view(2, E, torch.int32, (E,)), "offsets": view(3, E + 1, torch.int32, (E + 1,)),
            "row_src": view(4, Tk, torch.int32, (Tk,)), "slot_pos": view(5, Tk, torch.int32, (Tk,)),
            "x_perm": view(6, Tk * d, fdt, (Tk, d)), "h": view(7, Tk * dff, fdt, (Tk, dff)),
            "y": view(8, Tk * d, fdt, (Tk, d)), "xn": view(9, T * d, fdt, (T, d))}


def workspace(T, d, dff, E, k, dtype=MOE_DTYPE_BF16, device="cuda", host=False):
    """A uint8 device tensor big enough for moe_forward_ws (or moe_forward_host)."""
    fn = lib().moe_forward_host_workspace_bytes if host else lib().moe_workspace_bytes
    return torch.empty(max(int(fn(T, d, dff, E, k, dtype)), 256), dtype=torch.uint8, device=device)


def w8_workspace(T, d, dff, E, k, device="cuda"):
    """Scratch for the int8 layer (moe_forward_w8_ws, moe_forward_ex with int8
    weights): moe_forward_w8_workspace_bytes, the bf16 layer's size."""
    n = int(lib().moe_forward_w8_workspace_bytes(T, d, dff, E, k))
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def moe_forward_ws(x, Wg, W1, W3, W2, k, ws, out=None, stream=None):
    """The layer on caller scratch `ws` (uint8 tensor): returns out[T,d]."""
    _dev(x, Wg, W1, W3, W2, ws, out)
    T, d = x.shape
    E, dff, _ = W1.shape
    if out is None:
        out = torch.empty_like(x)
    _check("moe_forward_ws", lib().moe_forward_ws(_p(x), _p(Wg), _p(W1), _p(W3), _p(W2), _p(out), T, d, dff, E, k,
                                                  _dtype(x), _p(ws), ws.numel(), _stream(stream)))
    return out


def moe_forward(x, Wg, W1, W3, W2, k, out=None, stream=None):
    """The layer in bf16, one call (scratch from the stream-ordered pool)."""
    _dev(x, Wg, W1, W3, W2, out)
    if x.dtype != torch.bfloat16:
        raise TypeError("moe_forward is the bf16 entry point; use moe_forward_f32 for float32")
    T, d = x.shape
    E, dff, _ = W1.shape
    if out is None:
        out = torch.empty_like(x)
    _check("moe_forward", lib().moe_forward(_p(x), _p(Wg), _p(W1), _p(W3), _p(W2), _p(out), T, d, dff, E, k,
                                            _stream(stream)))
    return out


def moe_forward_f32(x, Wg, W1, W3, W2, k, out=None, stream=None):
    """The layer in fp32 (CUDA cores), one call."""
    _dev(x, Wg, W1, W3, W2, out)
    if x.dtype != torch.float32:
        raise TypeError("moe_forward_f32 takes float32 tensors")
    T, d = x.shape
    E, dff, _ = W1.shape
    if out is None:
        out = torch.empty_like(x)
    _check("moe_forward_f32", lib().moe_forward_f32(_p(x), _p(Wg), _p(W1), _p(W3), _p(W2), _p(out), T, d, dff, E,
                                                    k, _stream(stream)))
    return out


def moe_block_forward_ws(x, gamma, eps, Wg, W1, W3, W2, k, ws, out=None, stream=None):
    """Block form x + MoE(RMSNorm(x)) on caller scratch: returns out[T,d]."""
    _dev(x, gamma, Wg, W1, W3, W2, ws, out)
    T, d = x.shape
    E, dff, _ = W1.shape
    if out is None:
        out = torch.empty_like(x)
    _check("moe_block_forward_ws", lib().moe_block_forward_ws(_p(x), _p(gamma), eps, _p(Wg), _p(W1), _p(W3), _p(W2),
                                                              _p(out), T, d, dff, E, k, _dtype(x), _p(ws),
                                                              ws.numel(), _stream(stream)))
    return out


def moe_block_forward(x, gamma, eps, Wg, W1, W3, W2, k, out=None, stream=None):
    """Block form in bf16, one call."""
    _dev(x, gamma, Wg, W1, W3, W2, out)
    T, d = x.shape
    E, dff, _ = W1.shape
    if out is None:
        out = torch.empty_like(x)
    _check("moe_block_forward", lib().moe_block_forward(_p(x), _p(gamma), eps, _p(Wg), _p(W1), _p(W3), _p(W2),
                                                        _p(out), T, d, dff, E, k, _stream(stream)))
    return out


def moe_forward_ex(x, Wg, k, ws, W1=None, W3=None, W2=None, gamma=None, eps=0.0, w8=None, out=None, events=None,
                   stream=None):
    """The layer with every option on caller scratch `ws`: block form when
    `gamma` is given, int8 experts when `w8` = (W1q, W1s, W3q, W3s, W2q, W2s);
    `events` (5 torch.cuda.Event, already recorded once) are recorded at the
    step boundaries.  Returns out[T,d]."""
    _dev(x, Wg, W1, W3, W2, gamma, ws, out, *(w8 or ()))
    T, d = x.shape
    E = Wg.shape[0]
    dff = (w8[0] if w8 is not None else W1).shape[1]
    if out is None:
        out = torch.empty_like(x)
    ev = None
    if events is not None:
        for e in events:
            if not e.cuda_event:  # torch creates an event on its first record
                e.record()
        ev = (ctypes.c_void_p * 5)(*[e.cuda_event for e in events])
    q = [_p(v) for v in w8] if w8 is not None else [None] * 6
    _check("moe_forward_ex", lib().moe_forward_ex(_p(x), _p(gamma), eps, _p(Wg), _p(W1), _p(W3), _p(W2), *q, _p(out),
                                                  T, d, dff, E, k, _dtype(x), _p(ws), ws.numel(), ev,
                                                  _stream(stream)))
    return out


def moe_forward_host(x_host, Wg, W1, W3, W2, k, ws, out_host=None, stream=None):
    """End-to-end call with host activations (pinned CPU tensors); returns out_host."""
    _dev(Wg, W1, W3, W2, ws)
    if x_host.is_cuda:
        raise ValueError("moe_forward_host takes a host (CPU) x")
    T, d = x_host.shape
    E, dff, _ = W1.shape
    if out_host is None:
        out_host = torch.empty_like(x_host)
    _check("moe_forward_host", lib().moe_forward_host(_p(x_host), _p(Wg), _p(W1), _p(W3), _p(W2), _p(out_host), T, d,
                                                      dff, E, k, _dtype(x_host), _p(ws), ws.numel(),
                                                      _stream(stream)))
    return out_host


# ------------------------------------------------------------------ int8 weights
def moe_quantize_int8(W, q=None, scale=None, stream=None):
    """Per-row int8 quantisation of a bf16 matrix (any leading shape, rows =
    product of the leading dims): returns (q int8 like W, scale fp32 [rows])."""
    _dev(W, q, scale)
    if W.dtype != torch.bfloat16:
        raise TypeError("moe_quantize_int8 takes a bfloat16 matrix")
    cols = W.shape[-1]
    rows = W.numel() // cols
    if q is None:
        q = torch.empty(W.shape, dtype=torch.int8, device=W.device)
    if scale is None:
        scale = torch.empty(W.shape[:-1], dtype=torch.float32, device=W.device)
    _check("moe_quantize_int8", lib().moe_quantize_int8(_p(W), rows, cols, _p(q), _p(scale), _stream(stream)))
    return q, scale


def moe_expert_gate_up_w8(x_perm, offsets, W1q, W1s, W3q, W3s, h_perm=None, stream=None):
    """Step a4 with int8 weights: returns h_perm[Tk,dff] (bf16)."""
    _dev(x_perm, offsets, W1q, W1s, W3q, W3s, h_perm)
    Tk, d = x_perm.shape
    E, dff, _ = W1q.shape
    if h_perm is None:
        h_perm = torch.empty((Tk, dff), dtype=x_perm.dtype, device=x_perm.device)
    _check("moe_expert_gate_up_w8", lib().moe_expert_gate_up_w8(_p(x_perm), _p(offsets), _p(W1q), _p(W1s), _p(W3q),
                                                                _p(W3s), _p(h_perm), Tk, d, dff, E,
                                                                _stream(stream)))
    return h_perm


def moe_expert_down_w8(h_perm, offsets, W2q, W2s, y_perm=None, stream=None):
    """Step a5 with int8 weights: returns y_perm[Tk,d] (bf16)."""
    _dev(h_perm, offsets, W2q, W2s, y_perm)
    Tk, dff = h_perm.shape
    E, d, _ = W2q.shape
    if y_perm is None:
        y_perm = torch.empty((Tk, d), dtype=h_perm.dtype, device=h_perm.device)
    _check("moe_expert_down_w8", lib().moe_expert_down_w8(_p(h_perm), _p(offsets), _p(W2q), _p(W2s), _p(y_perm), Tk,
                                                          d, dff, E, _stream(stream)))
    return y_perm


def moe_forward_w8_ws(x, Wg, W1q, W1s, W3q, W3s, W2q, W2s, k, ws, out=None, stream=None):
    """The bf16 layer with int8 expert weights on caller scratch `ws`."""
    _dev(x, Wg, W1q, W1s, W3q, W3s, W2q, W2s, ws, out)
    T, d = x.shape
    E, dff, _ = W1q.shape
    if out is None:
        out = torch.empty_like(x)
    _check("moe_forward_w8_ws", lib().moe_forward_w8_ws(_p(x), _p(Wg), _p(W1q), _p(W1s), _p(W3q), _p(W3s), _p(W2q),
                                                        _p(W2s), _p(out), T, d, dff, E, k, _p(ws), ws.numel(),
                                                        _stream(stream)))
    return out


def moe_forward_w8(x, Wg, W1q, W1s, W3q, W3s, W2q, W2s, k, out=None, stream=None):
    """The bf16 layer with int8 expert weights, one call."""
    _dev(x, Wg, W1q, W1s, W3q, W3s, W2q, W2s, out)
    T, d = x.shape
    E, dff, _ = W1q.shape
    if out is None:
        out = torch.empty_like(x)
    _check("moe_forward_w8", lib().moe_forward_w8(_p(x), _p(Wg), _p(W1q), _p(W1s), _p(W3q), _p(W3s), _p(W2q),
                                                  _p(W2s), _p(out), T, d, dff, E, k, _stream(stream)))
    return out


# ------------------------------------------------------------------ backward
def moe_backward_workspace_bytes(T, d, dff, E, k) -> int:
    return int(lib().moe_backward_workspace_bytes(T, d, dff, E, k))


def _grads(x, Wg, W1, W3, W2, grads):
    if grads is not None:
        return grads
    dev = x.device
    return {"dx": torch.empty_like(x), "dWg": torch.empty(Wg.shape, dtype=torch.float32, device=dev),
            "dW1": torch.empty(W1.shape, dtype=torch.float32, device=dev),
            "dW3": torch.empty(W3.shape, dtype=torch.float32, device=dev),
            "dW2": torch.empty(W2.shape, dtype=torch.float32, device=dev)}


def keep_buffer(T, dff, k, device="cuda"):
    """The bf16 [2, T*k, dff] buffer moe_forward_train_ws fills with
    p = b silu'(a) (plane 0) and q = silu(a) (plane 1)."""
    return torch.empty((2, T * k, dff), dtype=torch.bfloat16, device=device)


def moe_forward_train_ws(x, Wg, W1, W3, W2, k, ws, keep=None, out=None, stream=None):
    """The bf16 layer on caller scratch `ws` that also keeps p and q for the
    backward: returns (out[T,d], keep[2,T*k,dff])."""
    _dev(x, Wg, W1, W3, W2, ws, out, keep)
    T, d = x.shape
    E, dff, _ = W1.shape
    if keep is None:
        keep = keep_buffer(T, dff, k, device=x.device)
    if out is None:
        out = torch.empty_like(x)
    _check("moe_forward_train_ws", lib().moe_forward_train_ws(_p(x), _p(Wg), _p(W1), _p(W3), _p(W2), _p(out),
                                                              _p(keep), T, d, dff, E, k, _p(ws), ws.numel(),
                                                              _stream(stream)))
    return out, keep


def moe_backward_ws(dout, x, Wg, W1, W3, W2, k, saved, ws, grads=None, stream=None, keep=None):
    """Backward of the bf16 layer.  `saved` is the uint8 scratch the forward
    (moe_forward_ws or moe_forward_train_ws) used on the same inputs; `keep`
    None or the p/q buffer of that moe_forward_train_ws call; `ws` the
    backward's scratch.  Returns dict(dx, dWg, dW1, dW3, dW2)."""
    _dev(dout, x, Wg, W1, W3, W2, saved, ws, keep)
    T, d = x.shape
    E, dff, _ = W1.shape
    g = _grads(x, Wg, W1, W3, W2, grads)
    _check("moe_backward_ws", lib().moe_backward_ws(_p(dout), _p(x), _p(Wg), _p(W1), _p(W3), _p(W2), _p(saved),
                                                    saved.numel(), _p(keep), _p(g["dx"]), _p(g["dWg"]),
                                                    _p(g["dW1"]), _p(g["dW3"]), _p(g["dW2"]), T, d, dff, E, k,
                                                    _p(ws), ws.numel(), _stream(stream)))
    return g


def moe_backward(dout, x, Wg, W1, W3, W2, k, saved, grads=None, stream=None, keep=None):
    """As moe_backward_ws with scratch from the stream-ordered pool."""
    _dev(dout, x, Wg, W1, W3, W2, saved, keep)
    T, d = x.shape
    E, dff, _ = W1.shape
    g = _grads(x, Wg, W1, W3, W2, grads)
    _check("moe_backward", lib().moe_backward(_p(dout), _p(x), _p(Wg), _p(W1), _p(W3), _p(W2), _p(saved),
                                              saved.numel(), _p(keep), _p(g["dx"]), _p(g["dWg"]),
                                              _p(g["dW1"]), _p(g["dW3"]), _p(g["dW2"]), T, d, dff, E, k,
                                              _stream(stream)))
    return g


def moe_forward_noalloc(x, Wg, W1, W3, W2, k, out=None, stream=None):
    """The bf16 layer with the library's built-in scratch (no device
    allocation by the library; see include/moe.h for its limit)."""
    _dev(x, Wg, W1, W3, W2, out)
    T, d = x.shape
    E, dff, _ = W1.shape
    if out is None:
        out = torch.empty_like(x)
    _check("moe_forward_noalloc", lib().moe_forward_noalloc(_p(x), _p(Wg), _p(W1), _p(W3), _p(W2), _p(out), T, d,
                                                            dff, E, k, _stream(stream)))
    return out


def moe_get_device_status(reset: bool = True, stream=None) -> int:
    """Synchronise the stream and return (and by default clear) the device status."""
    v = ctypes.c_int(0)
    _check("moe_get_device_status", lib().moe_get_device_status(_stream(stream), ctypes.byref(v), int(reset)))
    return v.value


def moe_set_wait_limit_ns(ns: int) -> None:
    _check("moe_set_wait_limit_ns", lib().moe_set_wait_limit_ns(int(ns)))
