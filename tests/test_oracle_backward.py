"""Pins for the oracle's backward of LayerNorm + modulate (Qwen-Image final
AdaLN page, §What: forward and backward; d_scale / d_shift are token sums
reduced by fixed 32-way balanced fp32 trees applied recursively until one
value remains).

* the token tree: exact on integer data at every length; hand-worked inputs
  where the tree order decides the fp32 result (a sequential sum and a
  strided pairing give other answers); independent of the batch and of the
  position in it.
* the row reductions c1 = sum(dyhat) / D and c2 = sum(dyhat * yhat) / D:
  equal to the exact rational sums rounded once to fp32.
* grad_x, grad_scale, grad_shift: against torch autograd of the unrounded
  forward in fp64, within the rounding the definition adds.
* the LayerNorm-backward projections: grad_x is orthogonal to 1 and to yhat
  up to its own bf16 rounding.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import workloads as W
from _util import f32_rne_of_fraction, widen


def f32(v):
    return np.asarray(v, dtype=np.float32)


@pytest.mark.parametrize("n", [1, 2, 3, 31, 32, 33, 64, 95, 1000, 1024, 1025, 4608, 40000])
def test_tree_exact_on_integers(oracle_mod, n):
    v = np.random.default_rng(n).integers(-1000, 1000, n).astype(np.float32)
    assert oracle_mod.token_tree_sum(v) == np.float32(int(v.astype(np.int64).sum()))


def test_tree_order_hand_worked(oracle_mod):
    e = np.float32(2.0 ** -24)
    # pairs (1 + 0) and (e + e): 1 + 2^-23, where a left-to-right sum stays at 1
    assert oracle_mod.token_tree_sum(f32([1, 0, e, e])) == np.float32(1 + 2.0 ** -23)
    # pairs (e + 1) and (e + 0): each 1 + 2^-24 ties to 1; a strided pairing
    # (e + e) + (1 + 0) would give 1 + 2^-23
    assert oracle_mod.token_tree_sum(f32([e, 1, e, 0])) == np.float32(1.0)
    # across the 32-value blocks: 32 copies of e sum exactly to 2^-19 in the
    # first block, then + 1 in the next level
    v = np.concatenate([np.full(32, e, np.float32), f32([1])])
    assert oracle_mod.token_tree_sum(v) == np.float32(1 + 2.0 ** -19)
    # the same values with the 1 first: in block 0 the leaf pair (1, e) ties
    # back to 1, the fifteen pairs (e, e) give 2^-23 each, and the upper
    # levels add those exactly: 1 + 15 * 2^-23; block 1 is e, and the last
    # add rounds 1 + 15.5 * 2^-23 to even (1 + 2^-19)
    v2 = np.concatenate([f32([1]), np.full(32, e, np.float32)])
    want = np.float32(np.float32(1 + 15 * 2.0 ** -23) + e)
    assert oracle_mod.token_tree_sum(v2) == want
    # a single value is returned as is (no +0 added: -0 stays -0)
    assert np.signbit(oracle_mod.token_tree_sum(f32([-0.0])))


def _backward_inputs(B, S, D, seed, per_batch=True):
    inp = W.ln_modulate_inputs(B, S, D, seed=seed, per_batch_mod=per_batch)
    g = torch.Generator().manual_seed(seed + 1)
    inp["g"] = W.normal_bf16(g, (B, S, D), 0.5)
    return inp


def test_tree_batch_invariance(oracle_mod):
    inp = _backward_inputs(3, 77, 64, seed=5)
    _, mean, rstd = oracle_mod.ln_modulate(inp["x"], inp["scale"], inp["shift"])
    gx, gsc, gsh, _, _ = oracle_mod.ln_modulate_backward(inp["x"], inp["scale"], inp["g"], mean,
                                                         rstd)
    sc = inp["scale"].reshape(3, 1, 64)
    for b in range(3):
        m, r = mean[b * 77:(b + 1) * 77], rstd[b * 77:(b + 1) * 77]
        gx1, gsc1, gsh1, _, _ = oracle_mod.ln_modulate_backward(
            inp["x"][b:b + 1], sc[b], inp["g"][b:b + 1], m, r)
        assert np.array_equal(gsc1[0], gsc[b]) and np.array_equal(gsh1[0], gsh[b])
        assert np.array_equal(gx1[0], gx[b])


def test_token_sums_compose_from_pinned_parts(oracle_mod):
    # grad_shift is the token tree of g; grad_scale the token tree of the
    # exact products g * y, with y the forward's rounded LayerNorm output
    B, S, D = 2, 45, 64
    inp = _backward_inputs(B, S, D, seed=10)
    _, mean, rstd = oracle_mod.ln_modulate(inp["x"], inp["scale"], inp["shift"])
    _, gsc, gsh, _, _ = oracle_mod.ln_modulate_backward(inp["x"], inp["scale"], inp["g"], mean,
                                                        rstd)
    y, _, _ = oracle_mod.ln_normalize(inp["x"], 1e-6)
    g = widen(inp["g"]).reshape(B, S, D)
    yw = widen(y).reshape(B, S, D)
    for b in range(B):
        for d in range(D):
            assert gsh[b, d] == oracle_mod.token_tree_sum(g[b, :, d])
            assert gsc[b, d] == oracle_mod.token_tree_sum(g[b, :, d] * yw[b, :, d])


def test_row_reductions_exact(oracle_mod):
    B, S, D = 1, 24, 96
    inp = _backward_inputs(B, S, D, seed=6, per_batch=False)
    _, mean, rstd = oracle_mod.ln_modulate(inp["x"], inp["scale"], inp["shift"])
    _, _, _, c1, c2 = oracle_mod.ln_modulate_backward(inp["x"], inp["scale"], inp["g"], mean,
                                                      rstd)
    s1 = widen(oracle_mod.round_bf16(f32(1.0) + widen(inp["scale"]).reshape(-1)))
    x = widen(inp["x"]).reshape(S, D)
    g = widen(inp["g"]).reshape(S, D)
    for r in range(S):
        yhat = (x[r] - mean[r]) * rstd[r]          # float32 ops, one rounding each
        dy = g[r] * s1                             # exact: two bf16 values
        q1 = sum(Fraction(float(a)) for a in dy) / D
        q2 = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(dy, yhat)) / D
        assert c1[r] == f32_rne_of_fraction(q1)
        assert c2[r] == f32_rne_of_fraction(q2)


@pytest.mark.parametrize("B,S,D", [(2, 40, 256), (1, 100, 3072), (1, 1, 64)])
def test_against_torch_autograd_fp64(oracle_mod, B, S, D):
    inp = _backward_inputs(B, S, D, seed=B * S + D)
    eps = 1e-6
    _, mean, rstd = oracle_mod.ln_modulate(inp["x"], inp["scale"], inp["shift"], eps)
    gx, gsc, gsh, c1, c2 = oracle_mod.ln_modulate_backward(inp["x"], inp["scale"], inp["g"],
                                                           mean, rstd)
    x = torch.from_numpy(widen(inp["x"]).reshape(B, S, D).astype(np.float64)).requires_grad_()
    s1v = widen(oracle_mod.round_bf16(f32(1.0) + widen(inp["scale"]))).reshape(B, 1, D)
    s1 = torch.from_numpy(s1v.astype(np.float64)).requires_grad_()
    sh = torch.from_numpy(widen(inp["shift"]).reshape(B, 1, D).astype(np.float64)) \
        .requires_grad_()
    g = torch.from_numpy(widen(inp["g"]).reshape(B, S, D).astype(np.float64))
    ln = torch.nn.functional.layer_norm(x, (D,), eps=eps)
    (ln * s1 + sh).backward(g)
    ref_gx = x.grad.numpy()
    ref_gsc = s1.grad.numpy().reshape(B, D)
    ref_gsh = sh.grad.numpy().reshape(B, D)
    gabs = np.abs(g.numpy())
    # shift: only the tree's fp32 rounding (depth <= 15 levels of adds)
    assert np.all(np.abs(gsh - ref_gsh) <= 16 * 2.0 ** -24 * gabs.sum(axis=1))
    # scale: the definition multiplies by y = R(yhat) (2^-8 relative) plus the tree
    lnv = np.abs(ln.detach().numpy())
    assert np.all(np.abs(gsc - ref_gsc) <= (gabs * lnv).sum(axis=1) * (2.0 ** -8 + 2.0 ** -19))
    # grad_x: its final bf16 rounding, plus fp32 statistics and operations
    yhat = ln.detach().numpy()
    r = rstd.reshape(B, S, 1).astype(np.float64)
    dy = g.numpy() * s1v
    slack = 2.0 ** -18 * r * (np.abs(dy) + np.abs(c1.reshape(B, S, 1)) +
                              np.abs(yhat * c2.reshape(B, S, 1)) + 1e-30)
    err = np.abs(widen(gx).reshape(B, S, D) - ref_gx)
    assert np.all(err <= 2.0 ** -8 * np.abs(ref_gx) + slack)


def test_projection_invariants(oracle_mod):
    B, S, D = 1, 64, 1024
    inp = _backward_inputs(B, S, D, seed=8, per_batch=False)
    _, mean, rstd = oracle_mod.ln_modulate(inp["x"], inp["scale"], inp["shift"])
    gx, _, _, _, _ = oracle_mod.ln_modulate_backward(inp["x"], inp["scale"], inp["g"], mean,
                                                     rstd)
    d = widen(gx).reshape(S, D).astype(np.float64)
    yhat = (widen(inp["x"]).reshape(S, D) - mean[:, None]) * rstd[:, None]
    bound = 2.0 ** -8 * np.abs(d).sum(axis=1) + 1e-6 * np.abs(d).sum(axis=1)
    assert np.all(np.abs(d.sum(axis=1)) <= bound)
    assert np.all(np.abs((d * yhat).sum(axis=1)) <= bound * np.abs(yhat).max(axis=1))


def test_zero_gradient(oracle_mod):
    inp = _backward_inputs(2, 9, 64, seed=9)
    _, mean, rstd = oracle_mod.ln_modulate(inp["x"], inp["scale"], inp["shift"])
    zero = np.zeros_like(inp["x"])
    gx, gsc, gsh, _, _ = oracle_mod.ln_modulate_backward(inp["x"], inp["scale"], zero, mean,
                                                         rstd)
    assert not widen(gx).any() and not gsc.any() and not gsh.any()
