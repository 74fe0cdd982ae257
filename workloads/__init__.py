"""Seeded synthetic inputs for fused RMSNorm forward and backward.

This module holds shapes, value distributions and seeds, nothing of the
normalisation itself, so that the oracle and the CUDA path can both draw
their inputs from it without sharing any arithmetic of the method.

Every tensor is drawn on the CPU with its own ``torch.Generator`` seeded
``seed + k`` (k = 0 for x, 1 for gamma, 2 for dy), in float32, scaled and
shifted, and then rounded once (round to nearest even) to the storage type.
Both sides therefore receive the same already-rounded values, which is the
comparison the precision page recommends ("Den dolda avrundningen i RMSNorm",
section "Ge testet samma precision som modellen").  A normal distribution
is written ``("normal", mean, variance)``: the second parameter is the
variance, so N(0, 64) has standard deviation 8.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional, Tuple

import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
ELEMENT_BYTES = {"f32": 4, "bf16": 2, "f16": 2}

Dist = Tuple[str, float, float]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    rows: int
    hidden: int
    dtype: str              # "f32" | "bf16" | "f16"
    eps: float
    offset: int             # 1: Gemma gain 1 + gamma
    cast_mode: str          # "round_once" | "round_twice"
    x_dist: Dist
    gamma_dist: Dist
    dy_dist: Dist
    seed: int = 0
    kind: str = "rms"                 # "rms", "ln" (LayerNorm), "softmax"
    beta_dist: Optional[Dist] = None  # LayerNorm bias; None: no bias
    out_fmt: Optional[str] = None     # "e4m3": FP8 forward output (RMSNorm)
    scale: float = 1.0                # per-tensor scale of the FP8 output
    channels: int = 0                 # GroupNorm: rows = samples, hidden = channels * spatial
    groups: int = 0

    @property
    def spatial(self) -> int:
        return self.hidden // self.channels if self.channels else 0

    @property
    def param_len(self) -> int:
        """Length of gamma / beta: one per channel for GroupNorm."""
        return self.channels if self.kind == "gn" else self.hidden

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def elem_bytes(self) -> int:
        return ELEMENT_BYTES[self.dtype]

    def fwd_bytes(self) -> int:
        """Bytes the forward must move: read x and gamma (and beta), write y
        and the fp32 row statistics (rstd; mean and rstd for LayerNorm)."""
        s, r, n = self.elem_bytes, self.rows, self.hidden
        if self.kind == "softmax":
            return 2 * r * n * s          # read x, write y
        if self.kind == "gn":
            nb = self.channels * s if self.beta_dist is not None else 0
            return 2 * r * n * s + 8 * r * self.groups + self.channels * s + nb
        if self.kind == "ln":
            nb = n * s if self.beta_dist is not None else 0
            return 2 * r * n * s + 8 * r + n * s + nb
        if self.out_fmt == "e4m3":
            # read x, write one byte per element, rstd, gamma, the scale
            return r * n * s + r * n + 4 * r + n * s + 4
        return 2 * r * n * s + 4 * r + n * s

    def bwd_bytes(self) -> int:
        """Bytes the backward must move: read dy, x, gamma and the statistics,
        write dx and the fp32 weight (and bias) gradients."""
        s, r, n = self.elem_bytes, self.rows, self.hidden
        if self.kind == "softmax":
            return 3 * r * n * s          # read y and dy, write dx
        if self.kind == "gn":
            return 3 * r * n * s + 8 * r * self.groups + self.channels * s + 8 * self.channels
        if self.kind == "ln":
            return 3 * r * n * s + 8 * r + n * s + 8 * n
        return 3 * r * n * s + 4 * r + n * s + 4 * n

    def step_bytes(self) -> int:
        return self.fwd_bytes() + self.bwd_bytes()


_N01: Dist = ("normal", 0.0, 1.0)
_U0911: Dist = ("uniform", 0.9, 1.1)

# Fixed fp32 case, small enough for the oracle to finish in well under a second.
FP32_256x1024 = Workload("fp32_256x1024", 256, 1024, "f32", 1e-6, 0, "round_once",
                         _N01, _U0911, _N01)
# Llama-shaped bf16 activation: 4 sequences of 1024 tokens, hidden 4096.
LLAMA_BF16_4096x4096 = Workload("llama_bf16_4096x4096", 4096, 4096, "bf16", 1e-5, 0,
                                "round_once", _N01, _U0911, _N01)
# Gemma-shaped bf16 activation with the 1 + gamma gain.
GEMMA_BF16_8192x3072 = Workload("gemma_bf16_8192x3072", 8192, 3072, "bf16", 1e-6, 1,
                                "round_once", ("normal", 0.0, 2.0),
                                ("normal", 0.0, 0.1), _N01)
# fp16 sweep over hidden sizes; x has variance 64 so that a sum of squares in
# fp16 would overflow.
FP16_SWEEP_HIDDEN = (1024, 2048, 4096, 8192, 16384, 32768)


def fp16_sweep(hidden: int, x_var: float = 64.0) -> Workload:
    tag = "" if x_var == 64.0 else f"_var{int(x_var)}"
    return Workload(f"fp16_4096x{hidden}{tag}", 4096, hidden, "f16", 1e-6, 0,
                    "round_once", ("normal", 0.0, x_var), _U0911, _N01)


def large_bf16(cast_mode: str) -> Workload:
    tag = "once" if cast_mode == "round_once" else "twice"
    return Workload(f"large_bf16_16384x8192_{tag}", 16384, 8192, "bf16", 1e-5, 0,
                    cast_mode, _N01, _U0911, _N01)


def all_workloads() -> Dict[str, Workload]:
    ws = [FP32_256x1024, LLAMA_BF16_4096x4096, GEMMA_BF16_8192x3072]
    ws += [fp16_sweep(n) for n in FP16_SWEEP_HIDDEN]
    ws += [large_bf16("round_once"), large_bf16("round_twice")]
    return {w.name: w for w in ws}


def fp8_workloads() -> Dict[str, Workload]:
    """The bf16 RMSNorm workloads with an FP8 E4M3 forward output, scale 32
    (|x_hat * gamma| stays below 448 / 32 for these draws except far in the
    tail, where the store saturates)."""
    ws = [LLAMA_BF16_4096x4096.with_(name="llama_bf16_4096x4096_fp8", out_fmt="e4m3", scale=32.0),
          large_bf16("round_once").with_(name="large_bf16_16384x8192_fp8", out_fmt="e4m3",
                                         scale=32.0)]
    return {w.name: w for w in ws}


# LayerNorm cases (the sibling op): x with a nonzero mean so that centring
# matters, gains near 1, a small bias.
_LN_X: Dist = ("normal", 0.5, 1.0)
_LN_BETA: Dist = ("normal", 0.0, 0.01)


def layer_norm_workloads() -> Dict[str, Workload]:
    ws = [
        Workload("ln_fp32_256x1024", 256, 1024, "f32", 1e-5, 0, "round_once", _LN_X, _U0911,
                 _N01, kind="ln", beta_dist=_LN_BETA),
        Workload("ln_bf16_4096x4096", 4096, 4096, "bf16", 1e-5, 0, "round_once", _LN_X, _U0911,
                 _N01, kind="ln", beta_dist=_LN_BETA),
        Workload("ln_fp16_4096x8192", 4096, 8192, "f16", 1e-5, 0, "round_once",
                 ("normal", 2.0, 64.0), _U0911, _N01, kind="ln", beta_dist=_LN_BETA),
        Workload("ln_bf16_16384x8192", 16384, 8192, "bf16", 1e-5, 0, "round_once", _LN_X,
                 _U0911, _N01, kind="ln", beta_dist=_LN_BETA),
    ]
    return {w.name: w for w in ws}


def _draw(shape, dist: Dist, seed: int) -> torch.Tensor:
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    kind, a, b = dist
    if kind == "normal":
        t = torch.randn(shape, generator=gen, dtype=torch.float32)
        return t * math.sqrt(b) + a
    if kind == "uniform":
        t = torch.rand(shape, generator=gen, dtype=torch.float32)
        return t * (b - a) + a
    if kind == "zeros":
        return torch.zeros(shape, dtype=torch.float32)
    if kind == "const":
        return torch.full(shape, float(a), dtype=torch.float32)
    raise ValueError(f"unknown distribution {kind!r}")


def make_inputs(w: Workload, rows: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """CPU tensors x [rows, hidden], gamma [hidden], dy [rows, hidden] in the
    workload's storage type.  ``rows`` overrides the row count (the first
    ``rows`` rows of the same draw are *not* guaranteed: a different count is
    a different draw)."""
    r = w.rows if rows is None else rows
    dt = DTYPES[w.dtype]
    x = _draw((r, w.hidden), w.x_dist, w.seed + 0).to(dt)
    gamma = _draw((w.param_len,), w.gamma_dist, w.seed + 1).to(dt)
    dy = _draw((r, w.hidden), w.dy_dist, w.seed + 2).to(dt)
    out = {"x": x, "gamma": gamma, "dy": dy}
    if w.beta_dist is not None:
        out["beta"] = _draw((w.param_len,), w.beta_dist, w.seed + 3).to(dt)
    if w.kind == "gn":
        for k in ("x", "dy"):
            out[k] = out[k].view(r, w.channels, w.spatial)
    return out


def as_float64(t: torch.Tensor):
    """The values of a CPU tensor as a float64 numpy array (exact widening)."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def softmax_workloads() -> Dict[str, Workload]:
    """Softmax over the last dimension: logits x ~ N(0, 4) (std 2, the
    spread of attention scores), dy ~ N(0, 1); the same shapes as the
    RMSNorm workloads plus many short rows.  eps, offset, cast mode and
    gamma are unused."""
    def sm(name, rows, cols, dtype):
        return Workload(name, rows, cols, dtype, 0.0, 0, "round_once", ("normal", 0.0, 4.0),
                        ("zeros", 0.0, 0.0), _N01, kind="softmax")
    ws = [sm("softmax_fp32_256x1024", 256, 1024, "f32"),
          sm("softmax_bf16_4096x4096", 4096, 4096, "bf16"),
          sm("softmax_bf16_16384x8192", 16384, 8192, "bf16"),
          sm("softmax_f16_65536x1024", 65536, 1024, "f16")]
    return {w.name: w for w in ws}


def group_norm(name, n, c, spatial, groups, dtype, x_dist=_N01, dy_dist=_N01,
               gamma_dist=_U0911, beta_dist=("normal", 0.0, 0.01), seed=0) -> Workload:
    """GroupNorm over x [n, c, spatial]: rows = n, hidden = c * spatial."""
    return Workload(name, n, c * spatial, dtype, 1e-5, 0, "round_once", x_dist, gamma_dist,
                    dy_dist, seed=seed, kind="gn", beta_dist=beta_dist, channels=c,
                    groups=groups)


def group_norm_workloads() -> Dict[str, Workload]:
    """The shapes Liger-Kernel PR #1608 times on B200 (x of (n, C, H, W) with
    H * W flattened, or (n, C, L)), in bf16, plus its fp16 case with an
    upstream gradient of ones and unit weights (where a channel sum in fp16
    overflows) and an input offset of 16."""
    ws = [group_norm("gn_bf16_16x32x256x256_g8", 16, 32, 256 * 256, 8, "bf16"),
          group_norm("gn_fp32_16x32x256x256_g8", 16, 32, 256 * 256, 8, "f32"),
          group_norm("gn_bf16_1x16x256x256_g4", 1, 16, 256 * 256, 4, "bf16"),
          group_norm("gn_bf16_16x512x64x64_g32", 16, 512, 64 * 64, 32, "bf16"),
          group_norm("gn_bf16_64x64x8192_g8", 64, 64, 8192, 8, "bf16"),
          group_norm("gn_f16_1x16x256x256_g4_ones", 1, 16, 256 * 256, 4, "f16",
                     dy_dist=("const", 1.0, 0.0), gamma_dist=("const", 1.0, 0.0),
                     beta_dist=("const", 0.0, 0.0)),
          group_norm("gn_bf16_2x64x32x32_g8_offset16", 2, 64, 32 * 32, 8, "bf16",
                     x_dist=("normal", 16.0, 1.0))]
    return {w.name: w for w in ws}
