"""Seeded synthetic inputs for the fused adaLN row operations.

This module only draws random numbers and lays them out; it holds none of
the method's arithmetic.  Both the CPU oracle and the CUDA path are fed from
it, so that the two read identical bits.  Every tensor is drawn in fp32 with
``torch.Generator('cpu').manual_seed(seed)`` in the listed order, scaled to
its distribution in fp32 and only then cast to bf16 (round to nearest even);
bf16 tensors are returned as ``numpy.uint16`` bit patterns, fp32 tensors as
``numpy.float32``.

The named workloads reproduce the shapes and value distributions of the
model sites the method is measured on (FLUX.1, ERNIE-Image, GLM-Image,
Wan 2.1 VAE).  No weights, prompts or datasets are involved.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _bits(t: torch.Tensor) -> np.ndarray:
    """fp32 tensor -> bf16 bit patterns (torch's round-to-nearest-even cast)."""
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def normal_bf16(g: torch.Generator, shape, std: float = 1.0, mean: float = 0.0) -> np.ndarray:
    t = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return _bits(t)


def normal_f32(g: torch.Generator, shape, std: float = 1.0, mean: float = 0.0) -> np.ndarray:
    t = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.numpy()


def bf16_from_float(values) -> np.ndarray:
    """Exact or rounded bf16 bit patterns of the given float values."""
    return _bits(torch.as_tensor(np.asarray(values, dtype=np.float32)))


# --------------------------------------------------------------------------
# generic builders (any shape)
# --------------------------------------------------------------------------

def ln_modulate_inputs(B: int, S: int, D: int, seed: int = 0, outlier_frac: float = 0.0,
                       per_batch_mod: bool = False, x_std: float = 1.0,
                       mod_std: float = 0.1) -> dict:
    """x [B, S, D] ~ N(0, x_std^2); a fraction of rows scaled x20 (outliers);
    scale, shift [B or 1, 1, D] ~ N(0, mod_std^2)."""
    g = _gen(seed)
    x = torch.randn(B, S, D, generator=g, dtype=torch.float32)
    if x_std != 1.0:
        x.mul_(x_std)
    n_out = int(B * S * outlier_frac)
    if n_out:
        idx = torch.randperm(B * S, generator=g)[:n_out]
        x.view(B * S, D)[idx] *= 20.0
    mb = B if per_batch_mod else 1
    scale = normal_bf16(g, (mb, 1, D), mod_std)
    shift = normal_bf16(g, (mb, 1, D), mod_std)
    return dict(x=_bits(x), scale=scale, shift=shift, B=B, S=S, D=D)


def rmsnorm_modulate_inputs(B: int, S: int, D: int, seed: int = 0, with_weight: bool = True,
                            per_batch_mod: bool = False) -> dict:
    """x [B, S, D] ~ N(0,1); weight [D] ~ 1 + N(0, 0.05^2); scale, shift ~ N(0, 0.1^2)."""
    g = _gen(seed)
    x = normal_bf16(g, (B, S, D))
    w = normal_bf16(g, (D,), 0.05, 1.0) if with_weight else None
    mb = B if per_batch_mod else 1
    scale = normal_bf16(g, (mb, 1, D), 0.1)
    shift = normal_bf16(g, (mb, 1, D), 0.1)
    return dict(x=x, weight=w, scale=scale, shift=shift, B=B, S=S, D=D)


def gated_inputs(B: int, S: int, D: int, seed: int = 0, with_weight: bool = True,
                 per_batch_mod: bool = False) -> dict:
    """residual, update [B, S, D] ~ N(0,1); gate [B or 1, 1, D] ~ N(0, 0.1^2);
    weight ~ 1 + N(0, 0.05^2); scale, shift ~ N(0, 0.1^2)."""
    g = _gen(seed)
    residual = normal_bf16(g, (B, S, D))
    update = normal_bf16(g, (B, S, D))
    mb = B if per_batch_mod else 1
    gate = normal_bf16(g, (mb, 1, D), 0.1)
    w = normal_bf16(g, (D,), 0.05, 1.0) if with_weight else None
    scale = normal_bf16(g, (mb, 1, D), 0.1)
    shift = normal_bf16(g, (mb, 1, D), 0.1)
    return dict(residual=residual, update=update, gate=gate, weight=w, scale=scale, shift=shift,
                B=B, S=S, D=D)


def qk_inputs(rows_q: int, rows_k: int, head_dim: int = 128, seed: int = 0,
              x_std: float = 2.0) -> dict:
    """q [rows_q, hd], k [rows_k, hd] ~ N(0, x_std^2); wq, wk ~ 1 + N(0, 0.05^2);
    bq, bk ~ N(0, 0.02^2)."""
    g = _gen(seed)
    q = normal_bf16(g, (rows_q, head_dim), x_std)
    k = normal_bf16(g, (rows_k, head_dim), x_std)
    wq = normal_bf16(g, (head_dim,), 0.05, 1.0)
    bq = normal_bf16(g, (head_dim,), 0.02)
    wk = normal_bf16(g, (head_dim,), 0.05, 1.0)
    bk = normal_bf16(g, (head_dim,), 0.02)
    return dict(q=q, k=k, wq=wq, bq=bq, wk=wk, bk=bk, rows_q=rows_q, rows_k=rows_k,
                head_dim=head_dim)


def wan_inputs(pixels: int, C: int, seed: int = 0, bias_fp32: bool = True) -> dict:
    """x [pixels, C] (a channels-last tensor viewed pixel-major) ~ N(0,1);
    bias [C] ~ N(0, 0.1^2) in fp32 (or bf16); gamma [C] ~ 1 + N(0, 0.05^2)."""
    g = _gen(seed)
    x = normal_bf16(g, (pixels, C))
    bias = normal_f32(g, (C,), 0.1) if bias_fp32 else normal_bf16(g, (C,), 0.1)
    gamma = normal_bf16(g, (C,), 0.05, 1.0)
    return dict(x=x, bias=bias, gamma=gamma, pixels=pixels, C=C)


# --------------------------------------------------------------------------
# the named workloads (model-site shapes)
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    name: str
    op: str
    description: str
    params: dict = field(default_factory=dict)

    def make(self, seed: int = 0) -> dict:
        p = dict(self.params)
        kind = p.pop("kind")
        return _BUILDERS[kind](seed=seed, **p)


_BUILDERS = {
    "ln": ln_modulate_inputs,
    "rms": rmsnorm_modulate_inputs,
    "gated": gated_inputs,
    "qk": qk_inputs,
    "wan": wan_inputs,
}

# Wan VAE activation [1, C, 4, 480, 832] in channels_last_3d order is
# 4 * 480 * 832 pixel rows of C contiguous channels.
WAN_PIXELS = 4 * 480 * 832

WORKLOADS = {
    w.name: w
    for w in [
        Workload("ln_modulate_1x256x1024", "ln_modulate",
                 "LayerNorm(no affine, eps 1e-6)+modulate, x [1,256,1024] ~N(0,1), "
                 "scale/shift [1,1024] ~N(0,0.1^2)",
                 dict(kind="ln", B=1, S=256, D=1024)),
        Workload("ln_modulate_flux_1x4608x3072", "ln_modulate",
                 "FLUX.1 adaLN: x [1,4608,3072] ~N(0,1) with 1% of rows x20, "
                 "scale/shift [1,3072] ~N(0,0.1^2)",
                 dict(kind="ln", B=1, S=4608, D=3072, outlier_frac=0.01)),
        Workload("ln_modulate_flux_cfg_2x4608x3072", "ln_modulate",
                 "FLUX.1 adaLN, CFG batch: x [2,4608,3072] with 1% outlier rows, "
                 "per-batch scale/shift [2,1,3072]",
                 dict(kind="ln", B=2, S=4608, D=3072, outlier_frac=0.01, per_batch_mod=True)),
        Workload("rmsnorm_modulate_ernie_1x4216x4096", "rmsnorm_modulate",
                 "ERNIE-Image adaLN: x [1,4216,4096] ~N(0,1), weight ~1+N(0,0.05^2), "
                 "scale/shift ~N(0,0.1^2), eps 1e-6",
                 dict(kind="rms", B=1, S=4216, D=4096)),
        Workload("gated_rmsnorm_modulate_ernie_1x4216x4096", "gated_rmsnorm_modulate",
                 "ERNIE-Image gated site: residual/update [1,4216,4096] ~N(0,1), "
                 "gate [1,4096] ~N(0,0.1^2), weight, scale, shift",
                 dict(kind="gated", B=1, S=4216, D=4096)),
        Workload("qk_layernorm_glm_1x4352x32x128", "qk_layernorm",
                 "GLM-Image qk-norm: q, k [1,4352,32,128] ~N(0,2^2), per-head LayerNorm(128) "
                 "with weight ~1+N(0,0.05^2), bias ~N(0,0.02^2), eps 1e-5",
                 dict(kind="qk", rows_q=4352 * 32, rows_k=4352 * 32, head_dim=128)),
        Workload("rmsnorm_silu_cl_wan_c96", "rmsnorm_silu_cl",
                 "Wan VAE: x [1,96,4,480,832] channels_last_3d ~N(0,1), fp32 conv bias "
                 "~N(0,0.1^2), gamma ~1+N(0,0.05^2)",
                 dict(kind="wan", pixels=WAN_PIXELS, C=96)),
        Workload("rmsnorm_silu_cl_wan_c192", "rmsnorm_silu_cl",
                 "Wan VAE: x [1,192,4,480,832] channels_last_3d",
                 dict(kind="wan", pixels=WAN_PIXELS, C=192)),
        Workload("rmsnorm_silu_cl_wan_c384", "rmsnorm_silu_cl",
                 "Wan VAE: x [1,384,4,480,832] channels_last_3d",
                 dict(kind="wan", pixels=WAN_PIXELS, C=384)),
    ]
}


# --------------------------------------------------------------------------
# structured edge rows
# --------------------------------------------------------------------------

def edge_rows(D: int, seed: int = 0) -> tuple[np.ndarray, list[str]]:
    """A [n, D] bf16 matrix of degenerate and extreme rows, with their labels."""
    g = _gen(seed)
    rows, labels = [], []

    def add(label, values):
        labels.append(label)
        rows.append(np.asarray(values, dtype=np.float32))

    base = torch.randn(D, generator=g, dtype=torch.float32).numpy()
    add("zeros", np.zeros(D))
    add("const_1.5", np.full(D, 1.5))
    add("const_-0.25", np.full(D, -0.25))
    add("const_96", np.full(D, 96.0))
    add("one_hot", np.eye(1, D, D // 3)[0] * 3.0)
    add("offset_mean_100", base + 100.0)
    add("tiny_1e-30", base * 1e-30)
    add("subnormal_bf16", base * 1e-39)
    add("huge_1e30", base.astype(np.float64) * 1e30)
    add("overflow_1e38", np.clip(base, -3.0, 3.0).astype(np.float64) * 1e38)
    add("wide_range", base * np.exp2(np.linspace(-40, 40, D)).astype(np.float32))
    add("alternating", np.where(np.arange(D) % 2 == 0, 1.0, -1.0))
    add("normal", base)
    add("normal_x20", base * 20.0)
    return _bits(torch.from_numpy(np.stack(rows))), labels


def special_rows(D: int, seed: int = 0) -> tuple[np.ndarray, list[str]]:
    """Rows holding Inf / NaN values (IEEE propagation cases)."""
    g = _gen(seed)
    base = torch.randn(D, generator=g, dtype=torch.float32).numpy()
    rows, labels = [], []
    for label, pos, val in [("pos_inf", D // 2, np.inf), ("neg_inf", 1, -np.inf),
                            ("nan", D - 1, np.nan)]:
        r = base.copy()
        r[pos] = val
        rows.append(r)
        labels.append(label)
    r = base.copy()
    r[0], r[-1] = np.inf, -np.inf
    rows.append(r)
    labels.append("both_inf")
    return _bits(torch.from_numpy(np.stack(rows).astype(np.float32))), labels
