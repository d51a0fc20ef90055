"""Pins for the oracle's normalisation and fused operations.

* fp64 brute force: y (and z, SiLU) computed in double from the exact row
  statistics, then rounded to bf16, must equal the oracle's except where the
  double value lies within the oracle's own fp32 error bound of a bf16
  rounding midpoint (counted, and required to be rare).
* hand-worked golden cases (tests/golden/hand_worked.txt).
* closed forms: constant and zero rows, scale = shift = 0.
* invariants: LayerNorm output mean ~0 / variance ~var/(var+eps), RMS ~1,
  row permutation equivariance, batch invariance, the conv-bias fold identity.
* library cross-check: torch.nn.functional.layer_norm in fp64.
"""
import numpy as np
import pytest
import torch

import workloads as W
from _util import widen
from golden.load import cases


def bf16_of_f64(v):
    """bf16 nearest to each float64 value (via an exact float32 step where safe)
    and the midpoint distance (relative) to the nearest rounding boundary."""
    import oracle

    v = np.asarray(v, dtype=np.float64)
    r = oracle.round_bf16(v.astype(np.float32))
    rf = widen(r).astype(np.float64)
    # neighbour on the other side of v
    step_up = widen(np.where(r & 0x8000, r - 1, r + 1).astype(np.uint16)).astype(np.float64)
    step_dn = widen(np.where(r & 0x8000, r + 1, r - 1).astype(np.uint16)).astype(np.float64)
    other = np.where(v >= rf, np.maximum(step_up, step_dn), np.minimum(step_up, step_dn))
    mid = 0.5 * (rf + other)
    return r, np.abs(v - mid)


def test_golden_hand_worked(oracle_mod):
    for c in cases():
        op, eps = c["op"], float(c["eps"][0])
        bits = lambda k: W.bf16_from_float(c[k])
        want = bits("out")
        if op == "ln_modulate":
            out, mean, rstd = oracle_mod.ln_modulate(bits("x").reshape(1, 1, -1), bits("scale"),
                                                     bits("shift"), eps)
            assert mean[0] == c["mean"][0]
        elif op == "rmsnorm_modulate":
            out, rstd = oracle_mod.rmsnorm_modulate(bits("x").reshape(1, 1, -1), bits("weight"),
                                                    bits("scale"), bits("shift"), eps)
        elif op == "qk_layernorm":
            x = bits("x").reshape(1, -1)
            out, _, mean, rstd = oracle_mod.qk_layernorm(x, x, bits("weight"), bits("bias"),
                                                         bits("weight"), bits("bias"), eps)
            assert mean[0] == c["mean"][0]
        elif op == "rmsnorm_silu_cl":
            out, rstd = oracle_mod.rmsnorm_silu_cl(bits("x").reshape(1, -1), c["bias_fp32"],
                                                   bits("gamma"), eps)
        else:
            raise AssertionError(op)
        assert rstd[0] == c["rstd"][0], (op, rstd[0])
        assert np.array_equal(out.ravel(), want), (op, widen(out.ravel()), c["out"])


def exact_ln(xf):
    x = xf.astype(np.float64)
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return mu, var


@pytest.mark.parametrize("D,std,outliers", [(8, 1.0, 0), (16, 1.0, 0), (128, 2.0, 0),
                                            (1024, 1.0, 0), (3072, 1.0, 0.05)])
def test_ln_normalize_brute_force(oracle_mod, D, std, outliers):
    inp = W.ln_modulate_inputs(1, 256, D, seed=D, outlier_frac=outliers, x_std=std)
    eps = 1e-6
    y, mean, rstd = oracle_mod.ln_normalize(inp["x"], eps)
    xf = widen(inp["x"]).reshape(-1, D)
    mu, var = exact_ln(xf)
    rstd_e = 1.0 / np.sqrt(var + eps)
    y_e = (xf - mu) * rstd_e
    r, dist = bf16_of_f64(y_e)
    # the oracle computes y in fp32 from fp32 mean and rstd: bound its error
    bound = 4 * 2.0 ** -24 * np.abs(y_e) + np.abs(mean[:, None] - mu) * rstd_e * 1.01
    near = dist <= bound
    assert np.array_equal(y.reshape(-1, D)[~near], r[~near])
    assert near.mean() < 1e-3
    # statistics: mean within 1e-6 relative of exact; rstd too
    assert np.all(np.abs(mean - mu[:, 0]) <= 2.0 ** -23 * np.abs(mu[:, 0]) + 1e-30)
    assert np.allclose(rstd, rstd_e[:, 0], rtol=2.0 ** -22, atol=0)


def test_ln_invariants(oracle_mod):
    inp = W.ln_modulate_inputs(1, 64, 4096, seed=4)
    y, _, _ = oracle_mod.ln_normalize(inp["x"], 1e-6)
    yf = widen(y).reshape(64, 4096).astype(np.float64)
    mu, var = exact_ln(widen(inp["x"]).reshape(64, 4096))
    # each bf16 rounding moves y by at most 2^-8 relative (rigorous bound);
    # rounding errors of equal x values are equal, so no sqrt(N) averaging
    bound = 2.0 ** -8 * np.abs(yf).mean(axis=1) + 1e-7
    assert np.all(np.abs(yf.mean(axis=1)) <= bound)
    assert np.allclose(yf.var(axis=1), (var / (var + 1e-6))[:, 0], rtol=2 * 2.0 ** -8)


def test_ln_library_cross_check(oracle_mod):
    inp = W.ln_modulate_inputs(1, 128, 1024, seed=9)
    y, _, _ = oracle_mod.ln_normalize(inp["x"], 1e-6)
    xf = torch.from_numpy(widen(inp["x"]).reshape(128, 1024).astype(np.float64))
    ref = torch.nn.functional.layer_norm(xf, (1024,), eps=1e-6).numpy()
    diff = np.abs(widen(y).reshape(128, 1024) - ref)
    assert np.all(diff <= 2.0 ** -8 * np.abs(ref) + 1e-12)


@pytest.mark.parametrize("D,with_w", [(8, True), (128, False), (4096, True)])
def test_rms_normalize_brute_force(oracle_mod, D, with_w):
    inp = W.rmsnorm_modulate_inputs(1, 200, D, seed=D, with_weight=with_w)
    eps = 1e-6
    y, rstd = oracle_mod.rms_normalize(inp["x"], inp["weight"], eps)
    xf = widen(inp["x"]).reshape(-1, D).astype(np.float64)
    ms = (xf ** 2).mean(axis=1, keepdims=True)
    rstd_e = 1.0 / np.sqrt(ms + eps)
    w = widen(inp["weight"]).astype(np.float64) if with_w else 1.0
    y_e = xf * rstd_e * w
    r, dist = bf16_of_f64(y_e)
    near = dist <= 4 * 2.0 ** -24 * np.abs(y_e)
    assert np.array_equal(y.reshape(-1, D)[~near], r[~near])
    assert near.mean() < 1e-3
    assert np.allclose(rstd, rstd_e[:, 0], rtol=2.0 ** -22, atol=0)
    if not with_w:
        rms_y = np.sqrt((widen(y).reshape(-1, D).astype(np.float64) ** 2).mean(axis=1))
        assert np.allclose(rms_y, np.sqrt(ms / (ms + eps))[:, 0], rtol=2.0 ** -8)


@pytest.mark.parametrize("hd", [128, 96, 64])
def test_qk_brute_force_and_library(oracle_mod, hd):
    inp = W.qk_inputs(300, 200, hd, seed=1)
    eps = 1e-5
    qo, ko, mean, rstd = oracle_mod.qk_layernorm(inp["q"], inp["k"], inp["wq"], inp["bq"],
                                                 inp["wk"], inp["bk"], eps)
    for x, w, b, o, off in ((inp["q"], inp["wq"], inp["bq"], qo, 0),
                            (inp["k"], inp["wk"], inp["bk"], ko, 300)):
        xf = widen(x).astype(np.float64)
        mu, var = exact_ln(xf)
        rstd_e = 1.0 / np.sqrt(var + eps)
        z_e = (xf - mu) * rstd_e * widen(w) + widen(b)
        r, dist = bf16_of_f64(z_e)
        m = mean[off:off + x.shape[0], None]
        bound = 8 * 2.0 ** -24 * (np.abs(z_e) + np.abs(widen(b))) + np.abs(m - mu) * rstd_e * 2
        near = dist <= bound
        assert np.array_equal(o[~near], r[~near])
        assert near.mean() < 1e-3
        ref = torch.nn.functional.layer_norm(torch.from_numpy(xf), (hd,),
                                             torch.from_numpy(widen(w).astype(np.float64)),
                                             torch.from_numpy(widen(b).astype(np.float64)),
                                             eps).numpy()
        assert np.all(np.abs(widen(o) - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6)


def test_qk_weights_are_per_tensor(oracle_mod):
    # the same rows through q and k must use their own (w, b)
    inp = W.qk_inputs(16, 16, 128, seed=2)
    qo, ko, _, _ = oracle_mod.qk_layernorm(inp["q"], inp["q"], inp["wq"], inp["bq"],
                                           inp["wk"], inp["bk"], 1e-5)
    assert not np.array_equal(qo, ko)
    qo2, ko2, _, _ = oracle_mod.qk_layernorm(inp["q"], inp["q"], inp["wq"], inp["bq"],
                                             inp["wq"], inp["bq"], 1e-5)
    assert np.array_equal(qo2, ko2) and np.array_equal(qo2, qo)


@pytest.mark.parametrize("C", [8, 96, 192])
def test_wan_brute_force(oracle_mod, C):
    inp = W.wan_inputs(500, C, seed=C)
    eps = 1e-6
    out, rstd = oracle_mod.rmsnorm_silu_cl(inp["x"], inp["bias"], inp["gamma"], eps)
    xb = widen(oracle_mod.conv_bias_epilogue(inp["x"], inp["bias"])).astype(np.float64)
    ms = (xb ** 2).mean(axis=1, keepdims=True)
    z = xb / np.sqrt(ms + eps) * widen(inp["gamma"])
    s = z / (1.0 + np.exp(-z))
    r, dist = bf16_of_f64(s)
    near = dist <= 8 * 2.0 ** -24 * np.abs(s) + 1e-30
    assert np.array_equal(out[~near], r[~near])
    assert near.mean() < 2e-3


def test_wan_bias_fold_identity(oracle_mod):
    for bias_fp32 in (True, False):
        inp = W.wan_inputs(300, 96, seed=5, bias_fp32=bias_fp32)
        a, ra = oracle_mod.rmsnorm_silu_cl(inp["x"], inp["bias"], inp["gamma"])
        pre = oracle_mod.conv_bias_epilogue(inp["x"], inp["bias"])
        b, rb = oracle_mod.rmsnorm_silu_cl(pre, None, inp["gamma"])
        assert np.array_equal(a, b) and np.array_equal(ra, rb)


@pytest.mark.parametrize("c", [1.5, -0.25, 96.0])
def test_constant_rows_give_shift(oracle_mod, c):
    D = 3072
    inp = W.ln_modulate_inputs(1, 4, D, seed=1)
    x = W.bf16_from_float(np.full((1, 4, D), c))
    out, mean, rstd = oracle_mod.ln_modulate(x, inp["scale"], inp["shift"], 1e-6)
    assert np.all(mean == np.float32(c))
    assert np.allclose(rstd, 1.0 / np.sqrt(1e-6), rtol=1e-6)
    assert np.array_equal(out, np.broadcast_to(inp["shift"].reshape(1, 1, D), out.shape))
    # gated variant: residual constant, update 0 -> res constant -> RMSNorm of constant
    g = W.gated_inputs(1, 4, D, seed=2)
    zero = np.zeros_like(g["update"])
    res, out2, rstd2 = oracle_mod.gated_rmsnorm_modulate(x, zero, g["gate"], None, g["scale"],
                                                         g["shift"], 1e-6)
    assert np.array_equal(res, x)
    y, _ = oracle_mod.rms_normalize(x, None, 1e-6)
    # (c * rstd) with rstd = 1/sqrt(c^2 + eps) is within 2^-20 of sign(c): rounds to +-1
    assert np.all(widen(y) == np.sign(c))


def test_zero_rows(oracle_mod):
    D = 1024
    inp = W.ln_modulate_inputs(1, 3, D, seed=3)
    x = np.zeros((1, 3, D), np.uint16)
    out, mean, rstd = oracle_mod.ln_modulate(x, inp["scale"], inp["shift"], 1e-6)
    assert np.all(mean == 0) and np.allclose(rstd, 1000.0, rtol=1e-6)
    sh = np.broadcast_to(inp["shift"].reshape(1, 1, D), out.shape)
    assert np.array_equal(np.where(out == 0x8000, 0, out), np.where(sh == 0x8000, 0, sh))
    out2, rstd2 = oracle_mod.rmsnorm_modulate(x, None, inp["scale"], inp["shift"], 1e-6)
    assert np.array_equal(np.where(out2 == 0x8000, 0, out2), np.where(sh == 0x8000, 0, sh))


def test_scale_shift_zero_gives_normalised_values(oracle_mod):
    inp = W.ln_modulate_inputs(1, 32, 3072, seed=6)
    z = np.zeros((1, 1, 3072), np.uint16)
    out, _, _ = oracle_mod.ln_modulate(inp["x"], z, z, 1e-6)
    y, _, _ = oracle_mod.ln_normalize(inp["x"], 1e-6)
    assert np.array_equal(out, np.where(y == 0x8000, 0, y))


def test_row_permutation_and_batch_invariance(oracle_mod):
    inp = W.ln_modulate_inputs(2, 50, 1024, seed=8, per_batch_mod=True)
    out, mean, rstd = oracle_mod.ln_modulate(inp["x"], inp["scale"], inp["shift"])
    perm = np.random.default_rng(1).permutation(50)
    out_p, _, _ = oracle_mod.ln_modulate(np.ascontiguousarray(inp["x"][:, perm]), inp["scale"],
                                         inp["shift"])
    assert np.array_equal(out_p, out[:, perm])
    # one row alone vs inside the batch
    one, m1, r1 = oracle_mod.ln_modulate(inp["x"][1:2, 7:8], inp["scale"][1:2], inp["shift"][1:2])
    assert np.array_equal(one[0, 0], out[1, 7]) and m1[0] == mean[57] and r1[0] == rstd[57]


def test_per_batch_modulation_rows_are_used(oracle_mod):
    inp = W.ln_modulate_inputs(2, 8, 256, seed=10, per_batch_mod=True)
    out, _, _ = oracle_mod.ln_modulate(inp["x"], inp["scale"], inp["shift"])
    y, _, _ = oracle_mod.ln_normalize(inp["x"], 1e-6)
    for b in range(2):
        assert np.array_equal(out[b:b + 1], oracle_mod.modulate(y[b:b + 1], inp["scale"][b],
                                                                inp["shift"][b]))


def test_gated_composition(oracle_mod):
    inp = W.gated_inputs(2, 20, 512, seed=3, per_batch_mod=True)
    res, out, rstd = oracle_mod.gated_rmsnorm_modulate(inp["residual"], inp["update"],
                                                       inp["gate"], inp["weight"], inp["scale"],
                                                       inp["shift"])
    assert np.array_equal(res, oracle_mod.residual_gate_add(inp["residual"], inp["gate"],
                                                            inp["update"]))
    out2, rstd2 = oracle_mod.rmsnorm_modulate(res, inp["weight"], inp["scale"], inp["shift"])
    assert np.array_equal(out, out2) and np.array_equal(rstd, rstd2)


def test_special_values(oracle_mod):
    D = 64
    x, labels = W.special_rows(D)
    inp = W.ln_modulate_inputs(1, 1, D, seed=1)
    out, mean, rstd = oracle_mod.ln_modulate(x.reshape(1, -1, D), inp["scale"], inp["shift"])
    assert np.all(np.isnan(widen(out)))
    out2, rstd2 = oracle_mod.rmsnorm_modulate(x.reshape(1, -1, D), None, inp["scale"],
                                              inp["shift"])
    d = dict(zip(labels, range(len(labels))))
    # an infinite element makes the mean square infinite, rstd 0: finite elements
    # normalise to +-0 and the infinite one to NaN
    assert rstd2[d["pos_inf"]] == 0.0 and np.isnan(rstd2[d["nan"]])
    row = widen(out2[0, d["pos_inf"]])
    assert np.isnan(row[D // 2]) and np.sum(np.isnan(row)) == 1
