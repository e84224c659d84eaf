"""Seeded synthetic inputs for the Mixtral sparse-MoE feed-forward layer.

This module is the one thing the CPU oracle and the CUDA path share: it draws
the layer's inputs (token activations and weights) from fixed seeds, and holds
none of the layer's arithmetic.  Every tensor is drawn on the CPU from its own
``torch.Generator`` so that its values do not depend on the sizes of the other
tensors, then rounded once (round-to-nearest-even) to the workload's dtype.

Shapes and scales follow the Mixtral 8x7B pages:
  * d_model=4096, d_ff=14336 per expert, 8 experts, top-2 routing, RMSNorm
    eps 1e-5 ("The Evolving Transformer - 05 Mixtral", section 00 Config;
    KerasFormers Mixtral docs, MixtralModel argument table).
  * Weight layouts follow the bias-free ``nn.Linear`` shapes of the tutorial's
    section 04 (SwiGLU) and 05 (MoERouter): Wg[E,d], W1/W3[E,F,d], W2[E,d,F].

Readings of the init notation (the workload descriptions leave them open):
  * ``N(0, 1/d)`` is read as variance 1/d (std d^-1/2).
  * ``N(0, 0.02)`` for bf16 weights is read as std 0.02.
  * RMSNorm gamma is ``1 + N(0, std 0.02)``.

The skewed workloads add one constant input channel: x[:, 0] = 1 and
Wg[e, 0] = b_e, a per-expert bias.  The b_e table was calibrated once, on a
separate draw (seed 1), by ``oracle/calibrate_skew.py`` and is stored in
``skew_bias.json`` beside this file; this module only reads it.
"""
from __future__ import annotations

import json
import os
from dataclasses import dataclass, replace

import torch

MIXTRAL_D = 4096
MIXTRAL_F = 14336
MIXTRAL_E = 8
MIXTRAL_K = 2
RMSNORM_EPS = 1e-5

# Target shares of the T*k expert assignments for the skewed-load workload.
SKEW_TARGET_SHARES = (0.40, 0.20, 0.12, 0.10, 0.08, 0.05, 0.03, 0.02)
# Bias that takes an expert out of every top-2 in the zero-token variant.
SKEW_ZERO_BIAS = -64.0
SKEW_ZERO_EXPERT = 7

_HERE = os.path.dirname(os.path.abspath(__file__))
SKEW_BIAS_FILE = os.path.join(_HERE, "skew_bias.json")

# One generator stream per tensor.
_STREAM = {"x": 1, "Wg": 2, "W1": 3, "W3": 4, "W2": 5, "gamma": 6, "dout": 7}


@dataclass(frozen=True)
class Workload:
    """Shape, dtype and init recipe of one synthetic MoE-layer workload."""

    name: str
    T: int
    d: int
    F: int
    E: int
    k: int
    dtype: str  # "f32" or "bf16"
    init: str  # "inv_sqrt" (std d^-1/2, W2 std F^-1/2) or "std002"
    skew: str | None = None  # None, "shares" or "zero"
    block: bool = False  # RMSNorm prologue + residual epilogue
    eps: float = RMSNORM_EPS
    bias_key: str | None = None  # skew_bias.json entry (default: name)
    w8: bool = False  # expert weights quantised to int8 (per-row scales) before use
    bwd: bool = False  # the backward of the layer (dout drawn from stream "dout")

    @property
    def Tk(self) -> int:
        return self.T * self.k

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def with_tokens(self, T: int) -> "Workload":
        return replace(self, T=T)


def _mixtral(name, T, **kw):
    return Workload(name, T, MIXTRAL_D, MIXTRAL_F, MIXTRAL_E, MIXTRAL_K, "bf16", "std002", **kw)


# The five Mixtral-shaped workloads (1 is the small fp32 case).
WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", 64, 128, 256, 8, 2, "f32", "inv_sqrt"),
    "decode": _mixtral("decode", 16),
    "prefill": _mixtral("prefill", 4096),
    "skewed": _mixtral("skewed", 8192, skew="shares"),
    "skewed_zero": _mixtral("skewed_zero", 8192, skew="zero", bias_key="skewed"),
    "block": _mixtral("block", 8192, block=True),
    # The same decode and prefill batches with int8 weight-only experts
    # (KerasFormers Mixtral docs, "Lower memory"); the bf16 weights drawn
    # here are quantised per row before the layer runs.
    "decode_w8": _mixtral("decode_w8", 16, w8=True),
    "prefill_w8": _mixtral("prefill_w8", 4096, w8=True),
    # The backward of the prefill batch (Mixtral 8x7B model reference page,
    # Training): dout ~ N(0, 1) in bf16.
    "prefill_bwd": _mixtral("prefill_bwd", 4096, bwd=True),
}

# Reduced sizes with the same structure, small enough for the oracle to finish
# in seconds while still spanning several 128-row tiles and a ragged tail.
SMALL_WORKLOADS = {
    "small_bf16": Workload("small_bf16", 300, 512, 384, 8, 2, "bf16", "std002"),
    "small_ragged": Workload("small_ragged", 389, 320, 448, 8, 2, "bf16", "std002"),
    "small_skewed": Workload("small_skewed", 700, 256, 256, 8, 2, "bf16", "std002", skew="shares"),
    "small_skewed_zero": Workload(
        "small_skewed_zero", 700, 256, 256, 8, 2, "bf16", "std002", skew="zero", bias_key="small_skewed"
    ),
    "small_block": Workload("small_block", 333, 256, 320, 8, 2, "bf16", "std002", block=True),
    "small_f32": Workload("small_f32", 257, 192, 320, 8, 2, "f32", "inv_sqrt"),
}

ALL_WORKLOADS = {**WORKLOADS, **SMALL_WORKLOADS}


def get(name: str) -> Workload:
    return ALL_WORKLOADS[name]


def _gen(seed: int, stream: str) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(1000 * seed + _STREAM[stream])
    return g


def _normal(shape, std, seed, stream) -> torch.Tensor:
    t = torch.randn(shape, generator=_gen(seed, stream), dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t


def load_skew_bias(key: str) -> list[float]:
    with open(SKEW_BIAS_FILE) as f:
        table = json.load(f)
    if key not in table:
        raise KeyError(f"no calibrated skew bias for {key!r} in {SKEW_BIAS_FILE}")
    return [float(b) for b in table[key]["bias"]]


def skew_bias(wl: Workload) -> list[float]:
    """Per-expert bias b_e placed in Wg[:, 0] for a skewed workload."""
    b = load_skew_bias(wl.bias_key or wl.name)
    if wl.skew == "zero":
        b = list(b)
        b[SKEW_ZERO_EXPERT] = SKEW_ZERO_BIAS
    return b


def make_inputs(wl: Workload, seed: int = 0, bias: list[float] | None = None,
                x_seed: int | None = None, only: tuple[str, ...] | None = None) -> dict[str, torch.Tensor]:
    """Draw the workload's tensors on the CPU.

    Returns x[T,d], Wg[E,d], W1[E,F,d], W3[E,F,d], W2[E,d,F] (and gamma[d] for
    a block workload), all contiguous, in the workload's dtype.  ``x_seed``
    redraws only x (the skew calibration uses it); ``bias`` overrides the
    stored skew table; ``only`` draws a subset of the tensors (each has its
    own stream, so the values do not change).
    """
    T, d, F, E = wl.T, wl.d, wl.F, wl.E
    xs = seed if x_seed is None else x_seed
    if wl.init == "inv_sqrt":
        s_in, s_down = d ** -0.5, F ** -0.5
    elif wl.init == "std002":
        s_in = s_down = 0.02
    else:
        raise ValueError(wl.init)
    recipe = {
        "x": lambda: _normal((T, d), 1.0, xs, "x"),
        "Wg": lambda: _normal((E, d), s_in, seed, "Wg"),
        "W1": lambda: _normal((E, F, d), s_in, seed, "W1"),
        "W3": lambda: _normal((E, F, d), s_in, seed, "W3"),
        "W2": lambda: _normal((E, d, F), s_down, seed, "W2"),
    }
    if wl.block:
        recipe["gamma"] = lambda: 1.0 + _normal((d,), 0.02, seed, "gamma")
    if wl.bwd:
        recipe["dout"] = lambda: _normal((T, d), 1.0, xs, "dout")
    names = list(recipe) if only is None else [n for n in recipe if n in only]
    out = {n: recipe[n]() for n in names}
    if wl.skew is not None:
        b = bias if bias is not None else skew_bias(wl)
        if "x" in out:
            out["x"][:, 0] = 1.0
        if "Wg" in out:
            out["Wg"][:, 0] = torch.tensor(b, dtype=torch.float32)
    dt = wl.torch_dtype
    return {k: v.to(dt).contiguous() for k, v in out.items()}
