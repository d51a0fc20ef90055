"""Shared test helpers: bf16 bit views, ulp distances, exact rounding."""
from __future__ import annotations

from fractions import Fraction

import numpy as np


def widen(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float32 values."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def ordinal(bits: np.ndarray) -> np.ndarray:
    """Sign-magnitude bf16 patterns -> monotone integers (+0 and -0 both map to 0)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def is_nan_bf16(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    return ((b & 0x7F80) == 0x7F80) & ((b & 0x007F) != 0)


def ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """|ordinal(a) - ordinal(b)|; 0 where both are NaN, a huge value where only one is."""
    na, nb = is_nan_bf16(a), is_nan_bf16(b)
    d = np.abs(ordinal(a) - ordinal(b))
    d = np.where(na & nb, 0, d)
    d = np.where(na ^ nb, 1 << 20, d)
    return d


def assert_within_ulp(got, want, max_ulp=2, frac_1ulp=0.999, what="output"):
    """The end-to-end bar: <= 1 ulp on >= 99.9% of elements, <= max_ulp everywhere."""
    d = ulp_distance(np.asarray(got).ravel(), np.asarray(want).ravel())
    n = d.size
    if n == 0:
        return d
    worst = int(d.max())
    within1 = float((d <= 1).mean())
    assert worst <= max_ulp, (
        f"{what}: max ulp distance {worst} > {max_ulp} at flat index {int(d.argmax())} "
        f"(got {int(np.asarray(got).ravel()[d.argmax()]):#06x}, "
        f"want {int(np.asarray(want).ravel()[d.argmax()]):#06x})")
    assert within1 >= frac_1ulp, f"{what}: only {within1:.6f} of elements within 1 ulp"
    return d


def f32_rne_of_fraction(q: Fraction) -> np.float32:
    """The float32 nearest to the rational q (ties to even), by exact comparison."""
    if q == 0:
        return np.float32(0.0)
    c = np.float32(float(q))
    if not np.isfinite(c):
        return c
    best, best_err = None, None
    for cand in (np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))):
        if not np.isfinite(cand):
            continue
        err = abs(Fraction(float(cand)) - q)
        if best is None or err < best_err:
            best, best_err = cand, err
        elif err == best_err:
            if int(np.float32(cand).view(np.uint32)) & 1 == 0:
                best = cand
    return np.float32(best)


def rel_close(a, b, rtol):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    both_nan = np.isnan(a) & np.isnan(b)
    same = a == b
    close = np.abs(a - b) <= rtol * np.maximum(np.abs(a), np.abs(b))
    return both_nan | same | close


def assert_exact_where_stats_match(got, want, D, *stat_pairs, min_match=0.999):
    """Rows whose fp32 statistics equal the oracle's bit for bit go through
    the same elementwise fp32 / bf16 chain, so their outputs must be
    bit-identical (NaN payloads aside).  Also requires that almost every row's
    statistics match."""
    g = np.asarray(got).reshape(-1, D)
    w = np.asarray(want).reshape(-1, D)
    same = np.ones(g.shape[0], dtype=bool)
    for gs, ws in stat_pairs:
        gs = np.asarray(gs, np.float32)
        ws = np.asarray(ws, np.float32)
        same &= (gs.view(np.uint32) == ws.view(np.uint32)) | (np.isnan(gs) & np.isnan(ws))
    if g.shape[0]:
        assert same.mean() >= min_match, f"only {same.mean():.6f} of rows have equal statistics"
    d = ulp_distance(g[same], w[same])
    if d.size:
        bad = np.argwhere(d > 0)
        assert bad.size == 0, (f"{len(bad)} elements differ in rows with equal statistics, "
                               f"first at row {np.flatnonzero(same)[bad[0][0]]} col {bad[0][1]}")
    return same
