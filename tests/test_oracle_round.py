"""Pin: the oracle's integer fp32->bf16 round-to-nearest-even helper.

Checked against torch's own fp32 -> bf16 cast (a library routine) over every
one of the 2^32 fp32 bit patterns, plus hand-picked boundary cases whose
rounding follows from the definition of ties-to-even.
"""
import numpy as np
import pytest
import torch

from _util import widen

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _check_chunk(oracle_mod, start, chunk):
    ours = torch.from_numpy(oracle_mod.round_bf16_sweep(start, chunk).view(np.int16))
    lo = start if start < (1 << 31) else start - (1 << 32)
    f = torch.arange(lo, lo + chunk, dtype=torch.int32).view(torch.float32)
    ref = f.to(torch.bfloat16).view(torch.int16)
    nan = torch.isnan(f)
    # NaN payloads differ between implementations; both must be NaN.
    ours_nan = ((ours & 0x7F80) == 0x7F80) & ((ours & 0x7F) != 0)
    assert torch.equal(ours_nan, nan)
    return int(((ours != ref) & ~nan).sum())


def test_exhaustive_against_torch_cast(oracle_mod):
    from concurrent.futures import ThreadPoolExecutor

    chunk = 1 << 24
    with ThreadPoolExecutor(max_workers=8) as ex:
        mism = sum(ex.map(lambda s: _check_chunk(oracle_mod, s, chunk),
                          range(0, 1 << 32, chunk)))
    assert mism == 0


@pytest.mark.parametrize("bits_in,bits_out", [
    (0x3F808000, 0x3F80),  # 1 + 2^-8 exactly halfway, kept mantissa even -> down
    (0x3F818000, 0x3F82),  # halfway, kept mantissa odd -> up to even
    (0x3F808001, 0x3F81),  # just above halfway -> up
    (0x3F807FFF, 0x3F80),  # just below halfway -> down
    (0x7F7FFFFF, 0x7F80),  # largest finite fp32 rounds to +Inf
    (0x7F7F7FFF, 0x7F7F),  # stays finite
    (0x00008000, 0x0000),  # subnormal tie, even -> down (no flush to zero elsewhere)
    (0x00018000, 0x0002),  # subnormal tie, odd -> up
    (0x80000001, 0x8000),  # tiny negative -> -0
    (0x7F800000, 0x7F80),  # +Inf
    (0xFF800000, 0xFF80),  # -Inf
])
def test_boundary_cases(oracle_mod, bits_in, bits_out):
    v = np.array([bits_in], dtype=np.uint32).view(np.float32)
    assert int(oracle_mod.round_bf16(v)[0]) == bits_out


def test_widen_roundtrip(oracle_mod):
    # every non-NaN bf16 pattern widens exactly and rounds back to itself
    pats = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = widen(pats)
    back = oracle_mod.round_bf16(f)
    keep = ~np.isnan(f)
    assert np.array_equal(back[keep], pats[keep])
