"""Pins for the oracle's single-rounding LN + modulate tier
(FLUX.1 page, §Modifications commit 3: layer_norm(x, weight = R(1 + scale),
bias = shift) with one rounding).

* fp64 brute force: ((x - mu) / sigma) * R(1 + scale) + shift from the exact
  row statistics, rounded once to bf16, must equal the oracle's output except
  within the oracle's own fp32 error bound of a rounding midpoint (rare).
* library cross-check: torch.nn.functional.layer_norm in fp64 with the folded
  weight and bias.
* closed forms: scale = shift = 0 gives the plain LayerNorm output; scale = 1
  (weight exactly 2) doubles it; constant rows give the shift.
* relation to the lossless chain: the two tiers differ by at most the
  roundings the lossless chain adds (a few bf16 ulps), and share statistics.
"""
import numpy as np
import pytest
import torch

import workloads as W
from _util import widen
from test_oracle_ops import bf16_of_f64, exact_ln


@pytest.mark.parametrize("B,S,D,per_batch", [(1, 200, 128, False), (2, 64, 1024, True),
                                             (1, 48, 3072, False)])
def test_folded_brute_force_and_library(oracle_mod, B, S, D, per_batch):
    inp = W.ln_modulate_inputs(B, S, D, seed=D + B, per_batch_mod=per_batch)
    eps = 1e-6
    out, mean, rstd = oracle_mod.ln_modulate_folded(inp["x"], inp["scale"], inp["shift"], eps)
    xf = widen(inp["x"]).reshape(B, S, D).astype(np.float64)
    sc = widen(inp["scale"]).reshape(-1, 1, D).astype(np.float64)
    sh = widen(inp["shift"]).reshape(-1, 1, D).astype(np.float64)
    w = widen(oracle_mod.round_bf16((1.0 + sc).astype(np.float32))).astype(np.float64)
    mu, var = exact_ln(xf)
    rstd_e = 1.0 / np.sqrt(var + eps)
    z_e = (xf - mu) * rstd_e * w + sh
    r, dist = bf16_of_f64(z_e)
    m = mean.reshape(B, S, 1).astype(np.float64)
    bound = 8 * 2.0 ** -24 * (np.abs(z_e) + np.abs(sh)) + np.abs(m - mu) * rstd_e * np.abs(w) * 2
    near = dist <= bound
    assert np.array_equal(out[~near], r[~near])
    assert near.mean() < 1e-3
    for b in range(B):
        bb = b if per_batch else 0
        ref = torch.nn.functional.layer_norm(
            torch.from_numpy(xf[b]), (D,), torch.from_numpy(w[bb, 0]),
            torch.from_numpy(sh[bb, 0]), eps).numpy()
        assert np.all(np.abs(widen(out[b]) - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6)


def test_folded_zero_modulation_is_layer_norm(oracle_mod):
    inp = W.ln_modulate_inputs(1, 64, 1024, seed=5)
    zero = np.zeros(1024, np.uint16)
    out, mean, rstd = oracle_mod.ln_modulate_folded(inp["x"], zero, zero, 1e-6)
    y, mean_y, rstd_y = oracle_mod.ln_normalize(inp["x"], 1e-6)
    assert np.array_equal(out.reshape(-1), y.reshape(-1))
    assert np.array_equal(mean, mean_y) and np.array_equal(rstd, rstd_y)


def test_folded_weight_two_doubles_layer_norm(oracle_mod):
    # scale = 1 -> weight R(1 + 1) = 2 exactly; doubling commutes with RNE in
    # the normal range
    inp = W.ln_modulate_inputs(1, 64, 1024, seed=6)
    one = np.full(1024, 0x3F80, np.uint16)
    zero = np.zeros(1024, np.uint16)
    out, _, _ = oracle_mod.ln_modulate_folded(inp["x"], one, zero, 1e-6)
    y, _, _ = oracle_mod.ln_normalize(inp["x"], 1e-6)
    assert np.array_equal(widen(out.reshape(-1)), 2.0 * widen(y.reshape(-1)))


def test_folded_constant_rows_give_shift(oracle_mod):
    D = 256
    x = np.full((1, 4, D), W.bf16_from_float(np.array([1.5]))[0], np.uint16)
    inp = W.ln_modulate_inputs(1, 4, D, seed=7)
    out, mean, rstd = oracle_mod.ln_modulate_folded(x, inp["scale"], inp["shift"], 1e-6)
    assert np.all(mean == np.float32(1.5))
    # x - mean is +0 everywhere: out = R(0 * w + shift) = shift
    assert np.array_equal(out.reshape(4, D), np.broadcast_to(inp["shift"].reshape(1, D), (4, D)))


def test_folded_close_to_lossless_chain(oracle_mod):
    inp = W.ln_modulate_inputs(2, 128, 3072, seed=8, per_batch_mod=True)
    fo, fm, fr = oracle_mod.ln_modulate_folded(inp["x"], inp["scale"], inp["shift"], 1e-6)
    lo, lm, lr = oracle_mod.ln_modulate(inp["x"], inp["scale"], inp["shift"], 1e-6)
    assert np.array_equal(fm, lm) and np.array_equal(fr, lr)
    a, b = widen(fo).astype(np.float64), widen(lo).astype(np.float64)
    # each bf16 rounding moves a value v by at most 2^-8 |v|: the lossless
    # chain rounds y and y * w once more each, and both tiers end with a
    # rounding of their own output
    y, _, _ = oracle_mod.ln_normalize(inp["x"], 1e-6)
    sc = widen(inp["scale"]).reshape(2, 1, -1).astype(np.float64)
    yw = np.abs(widen(y).reshape(2, 128, -1) * (1 + sc))
    bound = 2.0 ** -8 * (2.01 * yw + np.abs(a) + np.abs(b)) + 1e-30
    assert np.all(np.abs(a - b) <= bound)
    assert (a != b).mean() > 0.01   # the tiers do differ (it is not a copy)
