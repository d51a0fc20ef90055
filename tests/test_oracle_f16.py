"""Pins for the oracle's fp16 modulate chain (FLUX.1 page, §Accuracy Tests:
the modulate kernel is tested in bf16 and fp16).

* the fp32 -> fp16 rounding (the C _Float16 conversion) against torch's own
  float32 -> float16 cast over every one of the 2^32 fp32 patterns, and
  boundary cases that follow from ties-to-even (checked against numpy too);
* the chain against the eager torch fp16 op chain on CPU (each op one fp32
  operation followed by one fp16 rounding), with every fp16 pattern as y and
  as shift.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

ALL = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)


def is_nan_f16(bits):
    bits = np.asarray(bits)
    return ((bits & 0x7C00) == 0x7C00) & ((bits & 0x3FF) != 0)


def same_bits(a, b):
    a, b = np.asarray(a).ravel(), np.asarray(b).ravel()
    na, nb = is_nan_f16(a), is_nan_f16(b)
    assert np.array_equal(na, nb)
    assert np.array_equal(a[~na], b[~nb])


def _check_chunk(oracle_mod, start, chunk):
    ours = torch.from_numpy(oracle_mod.round_f16_sweep(start, chunk).view(np.int16))
    lo = start if start < (1 << 31) else start - (1 << 32)
    f = torch.arange(lo, lo + chunk, dtype=torch.int32).view(torch.float32)
    ref = f.to(torch.float16).view(torch.int16)
    nan = torch.isnan(f)
    ours_nan = ((ours & 0x7C00) == 0x7C00) & ((ours & 0x3FF) != 0)
    assert torch.equal(ours_nan, nan)
    return int(((ours != ref) & ~nan).sum())


def test_round_f16_exhaustive_against_torch_cast(oracle_mod):
    from concurrent.futures import ThreadPoolExecutor

    chunk = 1 << 24
    with ThreadPoolExecutor(max_workers=8) as ex:
        mism = sum(ex.map(lambda s: _check_chunk(oracle_mod, s, chunk),
                          range(0, 1 << 32, chunk)))
    assert mism == 0


@pytest.mark.parametrize("bits_in,bits_out", [
    (0x3F801000, 0x3C00),  # 1 + 2^-11 exactly halfway, kept mantissa even -> down
    (0x3F803000, 0x3C02),  # halfway, kept mantissa odd -> up to even
    (0x477FEFFF, 0x7BFF),  # just below 65520: the largest finite value
    (0x477FF000, 0x7C00),  # 65520, the tie with 65536: to even, i.e. +Inf
    (0x33000000, 0x0000),  # 2^-25, the tie between 0 and the smallest subnormal -> 0
    (0x33000001, 0x0001),  # just above -> the smallest subnormal 2^-24
    (0x33800000, 0x0001),  # 2^-24 exactly
    (0x387FC000, 0x03FF),  # largest subnormal
])
def test_round_f16_boundary_cases(oracle_mod, bits_in, bits_out):
    v = np.array([bits_in], dtype=np.uint32).view(np.float32)
    assert int(oracle_mod.round_f16_sweep(bits_in, 1)[0]) == bits_out
    assert int(v.astype(np.float16).view(np.uint16)[0]) == bits_out


def T(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.float16)


def N(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def eager(y, scale, shift):
    return N(T(y) * (1 + T(scale)) + T(shift))


def normal_f16(g, shape, std=1.0):
    return N((torch.randn(*shape, generator=g) * std).to(torch.float16))


@pytest.mark.parametrize("seed", [0, 1])
def test_modulate_f16_all_y_patterns(oracle_mod, seed):
    g = torch.Generator().manual_seed(seed)
    D = 1 << 16
    y = np.tile(ALL, (3, 1)).reshape(1, 3, D)
    scale = normal_f16(g, (1, 1, D), 0.5)
    shift = normal_f16(g, (1, 1, D), 0.5)
    same_bits(oracle_mod.modulate_f16(y, scale, shift), eager(y, scale, shift))


def test_modulate_f16_all_scale_and_shift_patterns(oracle_mod):
    g = torch.Generator().manual_seed(3)
    D = 1 << 16
    y = normal_f16(g, (1, 3, D))
    scale = np.random.default_rng(1).permutation(ALL).reshape(1, 1, D)
    shift = ALL.reshape(1, 1, D)
    same_bits(oracle_mod.modulate_f16(y, scale, shift), eager(y, scale, shift))


def test_modulate_f16_per_batch_rows(oracle_mod):
    g = torch.Generator().manual_seed(4)
    y = normal_f16(g, (3, 5, 64))
    scale, shift = normal_f16(g, (3, 1, 64), 0.5), normal_f16(g, (3, 1, 64), 0.5)
    same_bits(oracle_mod.modulate_f16(y, scale, shift), eager(y, scale, shift))
