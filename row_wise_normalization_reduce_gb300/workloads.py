"""Seeded synthetic inputs for the normalization workloads.

This module only draws random numbers; it holds none of the normalization
arithmetic.  Both the CUDA path and the CPU oracle are fed from it.

Every workload is drawn with a CPU ``torch.Generator`` seeded per workload, in
binary32, in the order listed, and then cast to the I/O type with
round-to-nearest-even (``Tensor.to``).  Both sides consume the cast values.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    name: str
    op: str                 # "ln" | "rms" | "add_rms" | "bn" | "bn_infer" | "bn_bwd" | "softmax"
    dtype: str              # "f32" | "f16" | "bf16"
    shape: tuple            # [rows, N] or [batch, C, H, W]
    seed: int
    eps: float
    momentum: float = 0.1
    note: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def torch_dtype(self):
        return DTYPES[self.dtype]


# The workloads, by operator, I/O type and shape.
LN_F32_64x1024 = Workload(
    "ln_f32_64x1024", "ln", "f32", (64, 1024), seed=0, eps=1e-5,
    note="x = 3 + 2*randn; gamma = 1 + 0.1*randn; beta = 0.1*randn")
RMS_F16_2048x4096 = Workload(
    "rms_f16_2048x4096", "rms", "f16", (2048, 4096), seed=1, eps=1e-6,
    note="x = randn with 1% of entries (rand < 0.01) scaled by 20; w = 1 + 0.05*randn")
ADD_RMS_BF16_4096x4096 = Workload(
    "add_rms_bf16_4096x4096", "add_rms", "bf16", (4096, 4096), seed=2, eps=1e-6,
    note="x = randn; residual = 2*randn (variance 4); w = 1 + 0.05*randn")
LN_BF16_1024x16384 = Workload(
    "ln_bf16_1024x16384", "ln", "bf16", (1024, 16384), seed=3, eps=1e-5,
    note="x = 1000 + randn (cancellation stress); gamma = 1 + 0.1*randn; beta = 0.1*randn")
BN_F32_32x64x56x56 = Workload(
    "bn_train_f32_32x64x56x56", "bn", "f32", (32, 64, 56, 56), seed=4, eps=1e-5,
    momentum=0.1,
    note="mean_c = U(-2,2); std_c = U(0.5,3); x = mean_c + std_c*randn; "
         "gamma = 1 + 0.1*randn; beta = 0.1*randn; running_mean = 0; running_var = 1")
LN_BF16_4096x4096 = Workload(
    "ln_bf16_4096x4096", "ln", "bf16", (4096, 4096), seed=5, eps=1e-5,
    note="x = randn; gamma = 1 + 0.1*randn; beta = 0.1*randn")

BN_INFER_F32_32x64x56x56 = Workload(
    "bn_infer_f32_32x64x56x56", "bn_infer", "f32", (32, 64, 56, 56), seed=6, eps=1e-5,
    note="x as bn_train_f32_32x64x56x56; gamma = 1 + 0.1*randn; beta = 0.1*randn; "
         "running_mean = U(-2,2); running_var = U(0.25,9)")
BN_BWD_F32_32x64x56x56 = Workload(
    "bn_bwd_f32_32x64x56x56", "bn_bwd", "f32", (32, 64, 56, 56), seed=7, eps=1e-5,
    note="x as bn_train_f32_32x64x56x56; dy = randn; gamma = 1 + 0.1*randn; "
         "save_mean = mean_c; save_rstd = 1/std_c (the draw's own parameters)")
# The BatchNorm page's own benchmark shape (its section 8: (64, 64, 112, 112)).
BN_F32_64x64x112x112 = Workload(
    "bn_train_f32_64x64x112x112", "bn", "f32", (64, 64, 112, 112), seed=8, eps=1e-5,
    momentum=0.1, note="as bn_train_f32_32x64x56x56")
BN_BWD_F32_64x64x112x112 = Workload(
    "bn_bwd_f32_64x64x112x112", "bn_bwd", "f32", (64, 64, 112, 112), seed=9, eps=1e-5,
    note="as bn_bwd_f32_32x64x56x56")

# 16-bit BatchNorm (the same draws as the binary32 workloads of each shape,
# cast to bfloat16).
BN_BF16_32x64x56x56 = Workload(
    "bn_train_bf16_32x64x56x56", "bn", "bf16", (32, 64, 56, 56), seed=4, eps=1e-5,
    momentum=0.1, note="as bn_train_f32_32x64x56x56, in bfloat16")
BN_BF16_64x64x112x112 = Workload(
    "bn_train_bf16_64x64x112x112", "bn", "bf16", (64, 64, 112, 112), seed=8, eps=1e-5,
    momentum=0.1, note="as bn_train_f32_64x64x112x112, in bfloat16")

# Softmax: the LLM-ops page's benchmark shape (section 1 table: Batch=128,
# Seq=4096, binary32), and the 4096 x 4096 bf16 shape of the norm headline
# for a working set larger than L2.  The page gives no input values; logits
# are drawn as 4*randn (a spread that exercises the max subtraction).
SOFTMAX_F32_128x4096 = Workload(
    "softmax_f32_128x4096", "softmax", "f32", (128, 4096), seed=10, eps=0.0,
    note="x = 4*randn")
SOFTMAX_BF16_4096x4096 = Workload(
    "softmax_bf16_4096x4096", "softmax", "bf16", (4096, 4096), seed=11, eps=0.0,
    note="x = 4*randn")

ALL = [LN_F32_64x1024, RMS_F16_2048x4096, ADD_RMS_BF16_4096x4096, LN_BF16_1024x16384,
       BN_F32_32x64x56x56, LN_BF16_4096x4096, BN_INFER_F32_32x64x56x56, BN_BWD_F32_32x64x56x56,
       BN_F32_64x64x112x112, BN_BWD_F32_64x64x112x112, SOFTMAX_F32_128x4096,
       SOFTMAX_BF16_4096x4096, BN_BF16_32x64x56x56, BN_BF16_64x64x112x112]
BY_NAME = {w.name: w for w in ALL}


def make_inputs(w: Workload, shape=None, dtype=None) -> dict:
    """Draw the inputs of workload ``w`` (optionally at another ``shape`` or I/O
    ``dtype`` -- "f32", "f16", "bf16" -- with the same distributions).  Returns
    CPU tensors in the I/O type; statistics inputs are binary32."""
    shape = tuple(shape) if shape is not None else w.shape
    g = torch.Generator().manual_seed(w.seed)
    dt = DTYPES[dtype] if dtype is not None else w.torch_dtype
    f32 = torch.float32

    def randn(*s):
        return torch.randn(*s, generator=g, dtype=f32)

    def rand(*s):
        return torch.rand(*s, generator=g, dtype=f32)

    if w.op == "ln":
        rows, n = shape
        if w.name == "ln_f32_64x1024":
            x = 3.0 + 2.0 * randn(rows, n)
        elif w.name == "ln_bf16_1024x16384":
            x = 1000.0 + randn(rows, n)
        else:
            x = randn(rows, n)
        gamma = 1.0 + 0.1 * randn(n)
        beta = 0.1 * randn(n)
        return {"x": x.to(dt), "gamma": gamma.to(dt), "beta": beta.to(dt)}
    if w.op == "rms":
        rows, n = shape
        x = randn(rows, n)
        mask = rand(rows, n) < 0.01
        x = torch.where(mask, x * 20.0, x)
        wgt = 1.0 + 0.05 * randn(n)
        return {"x": x.to(dt), "w": wgt.to(dt)}
    if w.op == "softmax":
        rows, n = shape
        return {"x": (4.0 * randn(rows, n)).to(dt)}
    if w.op == "add_rms":
        rows, n = shape
        x = randn(rows, n)
        res = 2.0 * randn(rows, n)
        wgt = 1.0 + 0.05 * randn(n)
        return {"x": x.to(dt), "residual": res.to(dt), "w": wgt.to(dt)}
    if w.op in ("bn", "bn_infer", "bn_bwd"):
        b, c = shape[0], shape[1]
        mean_c = -2.0 + 4.0 * rand(c)
        std_c = 0.5 + 2.5 * rand(c)
        view = (1, c) + (1,) * (len(shape) - 2)
        x = mean_c.view(view) + std_c.view(view) * randn(*shape)
        if w.op == "bn_bwd":
            dy = randn(*shape)
            gamma = 1.0 + 0.1 * randn(c)
            return {"x": x.to(dt), "dy": dy.to(dt), "gamma": gamma.to(dt),
                    "save_mean": mean_c.clone(), "save_rstd": 1.0 / std_c}
        gamma = 1.0 + 0.1 * randn(c)
        beta = 0.1 * randn(c)
        if w.op == "bn_infer":
            rm = -2.0 + 4.0 * rand(c)
            rv = 0.25 + 8.75 * rand(c)
            return {"x": x.to(dt), "gamma": gamma.to(dt), "beta": beta.to(dt),
                    "running_mean": rm, "running_var": rv}
        return {"x": x.to(dt), "gamma": gamma.to(dt), "beta": beta.to(dt),
                "running_mean": torch.zeros(c, dtype=f32),
                "running_var": torch.ones(c, dtype=f32)}
    raise ValueError(w.op)


def generic_rows(op: str, dtype: str, rows: int, n: int, seed: int, scale=1.0, shift=0.0):
    """Small seeded inputs of any shape for edge-case tests (normal draws)."""
    g = torch.Generator().manual_seed(seed)
    dt = DTYPES[dtype]
    x = (shift + scale * torch.randn(rows, n, generator=g)).to(dt)
    p1 = (1.0 + 0.1 * torch.randn(n, generator=g)).to(dt)
    p2 = (0.1 * torch.randn(n, generator=g)).to(dt)
    if op == "ln":
        return {"x": x, "gamma": p1, "beta": p2}
    if op == "rms":
        return {"x": x, "w": p1}
    if op == "add_rms":
        res = (scale * torch.randn(rows, n, generator=g)).to(dt)
        return {"x": x, "residual": res, "w": p1}
    if op == "softmax":
        return {"x": x}
    raise ValueError(op)
