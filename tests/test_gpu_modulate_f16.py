"""modulate_scale_shift on fp16 storage (CUDA, through the C ABI): bit-exact
against the oracle and against eager torch fp16 on the GPU.

The kernel uses hardware f16x2 add and multiply where the eager chain does an
fp32 op followed by an fp16 rounding; with scale = 0 the chain is
R16(y + shift), which is compared with eager torch over every one of the
2^32 (y, shift) fp16 pairs; products are covered by every y pattern against
random modulation rows."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rm():
    import rmsnorm_modulate_gb300 as rm

    yield rm
    assert rm.device_status(clear=True) == 0


def to_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.float16).cuda()


def to_host(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def is_nan_f16(bits):
    return ((bits & 0x7C00) == 0x7C00) & ((bits & 0x3FF) != 0)


def same_bits(a, b):
    a, b = np.asarray(a).ravel(), np.asarray(b).ravel()
    na, nb = is_nan_f16(a), is_nan_f16(b)
    assert np.array_equal(na, nb)
    assert np.array_equal(a[~na], b[~nb])


def dev_same_bits(a, b):
    na, nb = torch.isnan(a), torch.isnan(b)
    assert torch.equal(na, nb)
    assert torch.equal(a.view(torch.int16)[~na], b.view(torch.int16)[~nb])


def normal_f16(g, shape, std=1.0):
    return to_host((torch.randn(*shape, generator=g) * std).to(torch.float16))


ALL = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16)


def test_every_f16_sum(rm):
    # B = 2048 batches of one row each: batch b's shift row holds one value,
    # y runs over all 65536 patterns, scale = 0 so the chain is R16(y + shift)
    D, rows = 1 << 16, 2048
    y = ALL.cuda().view(torch.float16).view(1, 1, D).expand(rows, 1, D).contiguous()
    zero = torch.zeros(rows, 1, D, dtype=torch.float16, device="cuda")
    for start in range(0, 1 << 16, rows):
        sh = (ALL[start:start + rows].cuda().view(torch.float16).view(rows, 1, 1)
              .expand(rows, 1, D).contiguous())
        out = rm.modulate_scale_shift(y, zero, sh)
        dev_same_bits(out, y * (1 + zero) + sh)


@pytest.mark.parametrize("seed", [0, 1])
def test_every_y_pattern(rm, oracle_mod, seed):
    g = torch.Generator().manual_seed(seed)
    D = 1 << 16
    y = np.repeat(np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).reshape(1, 1, D), 3,
                  axis=1)
    scale = normal_f16(g, (1, 1, D), 0.5)
    shift = normal_f16(g, (1, 1, D), 0.5)
    out = rm.modulate_scale_shift(to_dev(y), to_dev(scale), to_dev(shift))
    torch.cuda.synchronize()
    same_bits(to_host(out), oracle_mod.modulate_f16(y, scale, shift))
    eager = to_dev(y) * (1 + to_dev(scale)) + to_dev(shift)
    dev_same_bits(out, eager)


@pytest.mark.parametrize("B,S,D,per_batch", [(1, 7, 8, False), (2, 33, 3072, True),
                                             (3, 5, 136, True)])
def test_shapes(rm, oracle_mod, B, S, D, per_batch):
    g = torch.Generator().manual_seed(D)
    y = normal_f16(g, (B, S, D))
    nb = B if per_batch else 1
    scale, shift = normal_f16(g, (nb, 1, D), 2.0), normal_f16(g, (nb, 1, D), 2.0)
    out = rm.modulate_scale_shift(to_dev(y), to_dev(scale), to_dev(shift))
    torch.cuda.synchronize()
    same_bits(to_host(out), oracle_mod.modulate_f16(y, scale, shift))


def test_dtype_mismatch_is_rejected(rm):
    y = torch.zeros(1, 4, 64, dtype=torch.float16, device="cuda")
    s = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(TypeError):
        rm.modulate_scale_shift(y, s, s)
