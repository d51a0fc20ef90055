"""Pin: the oracle's elementwise chains equal the eager torch bf16 op chain.

The pages define each fused elementwise chain as the eager PyTorch chain
(one fp32 op then one bf16 rounding per op; sglang #34004 FLUX.1 page,
§Modifications commit 2), so eager torch on CPU is a library routine that
fixes the answer bit for bit.  Inputs include every bf16 bit pattern
(zeros, subnormals, Inf, NaN, the largest finite values).
"""
import numpy as np
import pytest
import torch

import workloads as W
from _util import is_nan_bf16


def T(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def N(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def same_bits(a, b):
    """Bit-identical, NaN payloads aside."""
    a = np.asarray(a).ravel()
    b = np.asarray(b).ravel()
    na, nb = is_nan_bf16(a), is_nan_bf16(b)
    assert np.array_equal(na, nb)
    assert np.array_equal(a[~na], b[~nb])


ALL = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)


def eager_modulate(y, scale, shift):
    return N(T(y) * (1 + T(scale)) + T(shift))


@pytest.mark.parametrize("seed", [0, 1])
def test_modulate_all_y_patterns(oracle_mod, seed):
    # y runs over all 65536 patterns in each row; scale/shift rows drawn at random
    g = torch.Generator().manual_seed(seed)
    D = 1 << 16
    y = np.tile(ALL, (4, 1)).reshape(1, 4, D)
    scale = W.normal_bf16(g, (1, 1, D), 0.5)
    shift = W.normal_bf16(g, (1, 1, D), 0.5)
    same_bits(oracle_mod.modulate(y, scale, shift), eager_modulate(y, scale, shift))


def test_modulate_all_scale_and_shift_patterns(oracle_mod):
    g = torch.Generator().manual_seed(3)
    D = 1 << 16
    y = W.normal_bf16(g, (1, 3, D))
    scale = np.random.default_rng(1).permutation(ALL).reshape(1, 1, D)
    shift = ALL.reshape(1, 1, D)
    same_bits(oracle_mod.modulate(y, scale, shift), eager_modulate(y, scale, shift))


def test_modulate_per_batch_rows(oracle_mod):
    g = torch.Generator().manual_seed(5)
    y = W.normal_bf16(g, (3, 7, 40))
    scale = W.normal_bf16(g, (3, 1, 40), 0.1)
    shift = W.normal_bf16(g, (3, 1, 40), 0.1)
    same_bits(oracle_mod.modulate(y, scale, shift), eager_modulate(y, scale, shift))


def test_modulate_identity_when_scale_and_shift_zero(oracle_mod):
    # R(1+0) = 1, R(y*1) = y, R(y+0) = y (with -0 + 0 = +0 under round to nearest)
    y = ALL.reshape(1, 1, -1)
    z = np.zeros((1, 1, y.shape[-1]), np.uint16)
    out = oracle_mod.modulate(y, z, z)
    want = np.where(y == 0x8000, 0, y)
    same_bits(out, want)


def test_residual_gate_add_all_patterns(oracle_mod):
    g = torch.Generator().manual_seed(7)
    D = 1 << 16
    residual = np.tile(ALL, (2, 1)).reshape(1, 2, D)
    update = W.normal_bf16(g, (1, 2, D), 2.0)
    gate = W.normal_bf16(g, (1, 1, D), 0.5)
    out = oracle_mod.residual_gate_add(residual, gate, update)
    same_bits(out, N(T(residual) + T(gate) * T(update)))
    # every gate and update pattern as well
    gate2 = ALL.reshape(1, 1, D)
    update2 = np.random.default_rng(2).permutation(ALL).reshape(1, 1, D)
    res2 = W.normal_bf16(g, (1, 1, D))
    same_bits(oracle_mod.residual_gate_add(res2, gate2, update2),
              N(T(res2) + T(gate2) * T(update2)))


def test_residual_gate_add_per_batch_gate(oracle_mod):
    g = torch.Generator().manual_seed(8)
    r = W.normal_bf16(g, (2, 5, 24))
    u = W.normal_bf16(g, (2, 5, 24))
    gate = W.normal_bf16(g, (2, 1, 24), 0.1)
    same_bits(oracle_mod.residual_gate_add(r, gate, u), N(T(r) + T(gate) * T(u)))


@pytest.mark.parametrize("bias_fp32", [True, False])
@pytest.mark.parametrize("with_residual", [False, True])
def test_conv_bias_epilogue_matches_aten_add(oracle_mod, bias_fp32, with_residual):
    g = torch.Generator().manual_seed(11)
    C = 96
    x = W.normal_bf16(g, (50, C), 3.0)
    bias = W.normal_f32(g, (C,), 0.1) if bias_fp32 else W.normal_bf16(g, (C,), 0.1)
    h = W.normal_bf16(g, (50, C)) if with_residual else None
    tb = torch.from_numpy(bias) if bias_fp32 else T(bias)
    want = T(x).clone().add_(tb.to(torch.bfloat16))
    if with_residual:
        want = want + T(h)
    same_bits(oracle_mod.conv_bias_epilogue(x, bias, h), N(want))


def test_conv_bias_epilogue_all_x_patterns(oracle_mod):
    g = torch.Generator().manual_seed(12)
    C = 128
    x = ALL.reshape(-1, C)
    bias = W.normal_f32(g, (C,), 1.0)
    want = T(x).clone().add_(torch.from_numpy(bias).to(torch.bfloat16))
    same_bits(oracle_mod.conv_bias_epilogue(x, bias), N(want))
