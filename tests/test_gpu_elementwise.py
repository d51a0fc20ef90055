"""The standalone elementwise chains (CUDA, through the C ABI): bit-exact
against the oracle and against eager torch on the GPU.

The fused kernels use hardware bf16x2 multiply and add where the eager chain
does an fp32 op followed by a bf16 rounding.  That substitution is checked
here over every one of the 2^32 (a, b) bf16 pairs, for the product and for
the sum, against eager torch bf16 arithmetic on the same GPU."""
import numpy as np
import pytest
import torch

import workloads as W
from _gpu import dev, host
from _util import is_nan_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rm():
    import rmsnorm_modulate_gb300 as rm

    yield rm
    assert rm.device_status(clear=True) == 0


def same_bits(a, b):
    a, b = np.asarray(a).ravel(), np.asarray(b).ravel()
    na, nb = is_nan_bf16(a), is_nan_bf16(b)
    assert np.array_equal(na, nb)
    assert np.array_equal(a[~na], b[~nb])


def dev_same_bits(a, b):
    """On the device: bit-identical except NaN payloads."""
    ai, bi = a.view(torch.int16), b.view(torch.int16)
    na, nb = torch.isnan(a), torch.isnan(b)
    assert torch.equal(na, nb)
    assert torch.equal(ai[~na], bi[~nb])


ALL = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16)


def test_every_bf16_product_and_sum(rm):
    """residual_gate_add(residual=0, gate=a, update=b) = R(0 + R(a * b)) and
    residual_gate_add(residual=a, gate=1, update=b) = R(a + b), compared with
    eager torch bf16 ops for all 2^16 x 2^16 operand pairs."""
    D = 1 << 16
    a = ALL.cuda().view(torch.bfloat16).view(1, 1, D)
    one = torch.ones(1, 1, D, dtype=torch.bfloat16, device="cuda")
    rows = 2048
    for start in range(0, 1 << 16, rows):
        b = (ALL[start:start + rows].cuda().view(torch.bfloat16).view(rows, 1)
             .expand(rows, D).contiguous().view(1, rows, D))
        zero = torch.zeros_like(b)
        prod = rm.residual_gate_add(zero, a, b)
        dev_same_bits(prod, zero + a * b)
        ssum = rm.residual_gate_add(b, one, a.expand(1, rows, D).contiguous())
        dev_same_bits(ssum, b + one * a)


@pytest.mark.parametrize("B,S,D,per_batch", [(1, 7, 8, False), (2, 33, 3072, True),
                                             (3, 5, 136, True)])
def test_modulate_scale_shift(rm, oracle_mod, B, S, D, per_batch):
    inp = W.ln_modulate_inputs(B, S, D, seed=D, per_batch_mod=per_batch, mod_std=2.0)
    out = rm.modulate_scale_shift(dev(inp["x"]), dev(inp["scale"]), dev(inp["shift"]))
    torch.cuda.synchronize()
    same_bits(host(out), oracle_mod.modulate(inp["x"], inp["scale"], inp["shift"]))


def test_modulate_every_y_pattern(rm, oracle_mod):
    D = 1 << 16
    y = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).reshape(1, 1, D)
    y = np.repeat(y, 3, axis=1)
    g = torch.Generator().manual_seed(1)
    scale = W.normal_bf16(g, (1, 1, D), 0.5)
    shift = W.normal_bf16(g, (1, 1, D), 0.5)
    out = rm.modulate_scale_shift(dev(y), dev(scale), dev(shift))
    torch.cuda.synchronize()
    same_bits(host(out), oracle_mod.modulate(y, scale, shift))


@pytest.mark.parametrize("per_batch", [False, True])
def test_residual_gate_add(rm, oracle_mod, per_batch):
    inp = W.gated_inputs(2, 45, 1024, seed=3, per_batch_mod=per_batch)
    out = rm.residual_gate_add(dev(inp["residual"]), dev(inp["gate"]), dev(inp["update"]))
    torch.cuda.synchronize()
    same_bits(host(out), oracle_mod.residual_gate_add(inp["residual"], inp["gate"],
                                                      inp["update"]))


@pytest.mark.parametrize("C", [8, 96, 384])
@pytest.mark.parametrize("bias_fp32", [True, False])
@pytest.mark.parametrize("with_h", [False, True])
def test_conv_bias_epilogue(rm, oracle_mod, C, bias_fp32, with_h):
    inp = W.wan_inputs(777, C, seed=C, bias_fp32=bias_fp32)
    h = W.normal_bf16(torch.Generator().manual_seed(2), (777, C)) if with_h else None
    out = rm.conv_bias_epilogue(dev(inp["x"]), dev(inp["bias"]), None if h is None else dev(h))
    torch.cuda.synchronize()
    same_bits(host(out), oracle_mod.conv_bias_epilogue(inp["x"], inp["bias"], h))


def test_epilogue_fed_oracle_normalised_values(rm, oracle_mod):
    """Spec invariant: given the oracle's normalised y, the GPU's
    modulate chain is bit-exact."""
    inp = W.ln_modulate_inputs(2, 300, 3072, seed=5, per_batch_mod=True)
    y, _, _ = oracle_mod.ln_normalize(inp["x"], 1e-6)
    out = rm.modulate_scale_shift(dev(y), dev(inp["scale"]), dev(inp["shift"]))
    torch.cuda.synchronize()
    want, _, _ = oracle_mod.ln_modulate(inp["x"], inp["scale"], inp["shift"])
    same_bits(host(out), want)
