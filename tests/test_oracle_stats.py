"""Pin: the oracle's row statistics are the exact statistics rounded once to fp32.

Reference values come from exact rational arithmetic (``fractions``) on the
bf16 row values, rounded to the nearest fp32 by exact comparison.  Plus
closed forms (constant and zero rows) and order invariance.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import workloads as W
from _util import f32_rne_of_fraction, widen


def exact_stats(row_bits):
    vals = [Fraction(float(v)) for v in widen(row_bits)]
    n = len(vals)
    mu = sum(vals) / n
    var = sum((v - mu) ** 2 for v in vals) / n
    msq = sum(v * v for v in vals) / n
    return f32_rne_of_fraction(mu), f32_rne_of_fraction(var), f32_rne_of_fraction(msq)


def check_rows(oracle_mod, x):
    mean, var, msq = oracle_mod.row_stats(x)
    for r in range(x.shape[0]):
        em, ev, es = exact_stats(x[r])
        assert mean[r] == em, (r, mean[r], em)
        assert var[r] == ev, (r, var[r], ev)
        assert msq[r] == es, (r, msq[r], es)


@pytest.mark.parametrize("n", [8, 16, 24, 96, 128, 1000])
def test_random_rows_correctly_rounded(oracle_mod, n):
    g = torch.Generator().manual_seed(n)
    rows = 200 if n <= 128 else 20
    x = W.normal_bf16(g, (rows, n))
    check_rows(oracle_mod, x)


def test_outlier_and_offset_rows_correctly_rounded(oracle_mod):
    g = torch.Generator().manual_seed(99)
    a = W.normal_bf16(g, (30, 64), 20.0)
    b = W.normal_bf16(g, (30, 64), 1.0, 100.0)  # large common offset
    c = W.normal_bf16(g, (30, 64), 1e-3, 0.5)
    check_rows(oracle_mod, np.concatenate([a, b, c]))


def test_edge_rows_correctly_rounded(oracle_mod):
    x, labels = W.edge_rows(64)
    # skip rows whose exact statistics overflow fp32 (compared separately below)
    keep = [i for i, l in enumerate(labels) if l not in ("overflow_1e38",)]
    check_rows(oracle_mod, x[keep])


def test_overflowing_statistics_round_to_inf(oracle_mod):
    x, labels = W.edge_rows(64)
    i = labels.index("overflow_1e38")
    mean, var, msq = oracle_mod.row_stats(x[i:i + 1])
    assert np.isfinite(mean[0])
    assert np.isinf(var[0]) and np.isinf(msq[0])


@pytest.mark.parametrize("c", [1.5, -0.25, 3.0, 96.0, 2.0 ** -20])
def test_constant_row(oracle_mod, c):
    x = W.bf16_from_float(np.full((1, 3072), c))
    mean, var, msq = oracle_mod.row_stats(x)
    assert mean[0] == np.float32(c)
    assert var[0] == 0.0
    assert msq[0] == np.float32(c) * np.float32(c)


def test_order_invariance(oracle_mod):
    g = torch.Generator().manual_seed(5)
    x = W.normal_bf16(g, (50, 4096), 20.0)
    perm = np.random.default_rng(0).permutation(4096)
    a = oracle_mod.row_stats(x)
    b = oracle_mod.row_stats(np.ascontiguousarray(x[:, perm]))
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_special_values_propagate(oracle_mod):
    x, labels = W.special_rows(32)
    mean, var, msq = oracle_mod.row_stats(x)
    d = dict(zip(labels, range(len(labels))))
    assert mean[d["pos_inf"]] == np.inf and np.isnan(var[d["pos_inf"]])
    assert mean[d["neg_inf"]] == -np.inf and np.isnan(var[d["neg_inf"]])
    assert np.isnan(mean[d["nan"]]) and np.isnan(var[d["nan"]]) and np.isnan(msq[d["nan"]])
    assert np.isnan(mean[d["both_inf"]])
    assert msq[d["pos_inf"]] == np.inf and msq[d["both_inf"]] == np.inf
