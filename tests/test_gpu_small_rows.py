"""Parity of the few-rows launches (one CTA per row, for at most four rows per
SM at 1024 / 2048 / 3072 / 4096 values) with the oracle, their slow-path rows
(Inf / NaN, extreme magnitudes), aliasing, and bit-identity with the ring
kernels that take the same rows once there are more of them.

Bars as for the other row ops: statistics within 1e-5 relative (and here the
correctly rounded exact values on both sides), output within 1 bf16 ulp on
>= 99.9% and 2 ulp everywhere, bit-identical wherever the statistics agree,
the gated residual stream bit-exact.
"""
import numpy as np
import pytest
import torch

import workloads as W
from _gpu import dev, host, stat_report
from _util import assert_exact_where_stats_match, assert_within_ulp

pytestmark = pytest.mark.gpu

WIDTHS = (1024, 2048, 3072, 4096)


@pytest.fixture(scope="module")
def rm():
    import rmsnorm_modulate_gb300 as rm

    yield rm
    assert rm.device_status(clear=True) == 0


@pytest.fixture(scope="module")
def coop_rows():
    # the largest row count the few-rows launch takes on this GPU
    return 4 * torch.cuda.get_device_properties(0).multi_processor_count


def _ln(rm, oracle_mod, inp, folded=False, check_stats=True):
    B, S, D = inp["B"], inp["S"], inp["D"]
    mean = torch.empty(B * S, dtype=torch.float32, device="cuda")
    rstd = torch.empty_like(mean)
    f = rm.ln_modulate_folded if folded else rm.ln_modulate
    out = f(dev(inp["x"]), dev(inp["scale"]), dev(inp["shift"]), mean_out=mean, rstd_out=rstd)
    torch.cuda.synchronize()
    of = oracle_mod.ln_modulate_folded if folded else oracle_mod.ln_modulate
    o_out, o_mean, o_rstd = of(inp["x"], inp["scale"], inp["shift"])
    gm, gr = host(mean), host(rstd)
    if check_stats:
        assert np.array_equal(gm, o_mean) and np.array_equal(gr, o_rstd), (
            stat_report(gm, o_mean), stat_report(gr, o_rstd))
    assert_within_ulp(host(out), o_out)
    assert_exact_where_stats_match(host(out), o_out, D, (gm, o_mean), (gr, o_rstd),
                                   min_match=0.99 if check_stats else 0)
    return gm, gr, o_mean, o_rstd


def _rms(rm, oracle_mod, inp):
    B, S, D = inp["B"], inp["S"], inp["D"]
    rstd = torch.empty(B * S, dtype=torch.float32, device="cuda")
    w = None if inp["weight"] is None else dev(inp["weight"])
    out = rm.rmsnorm_modulate(dev(inp["x"]), w, dev(inp["scale"]), dev(inp["shift"]),
                              rstd_out=rstd)
    torch.cuda.synchronize()
    o_out, o_rstd = oracle_mod.rmsnorm_modulate(inp["x"], inp["weight"], inp["scale"],
                                                inp["shift"])
    assert np.array_equal(host(rstd), o_rstd), stat_report(host(rstd), o_rstd)
    assert_within_ulp(host(out), o_out)
    assert_exact_where_stats_match(host(out), o_out, D, (host(rstd), o_rstd))


def _gated(rm, oracle_mod, inp):
    B, S, D = inp["B"], inp["S"], inp["D"]
    rstd = torch.empty(B * S, dtype=torch.float32, device="cuda")
    w = None if inp["weight"] is None else dev(inp["weight"])
    res, out = rm.gated_rmsnorm_modulate(dev(inp["residual"]), dev(inp["update"]),
                                         dev(inp["gate"]), w, dev(inp["scale"]),
                                         dev(inp["shift"]), rstd_out=rstd)
    torch.cuda.synchronize()
    o_res, o_out, o_rstd = oracle_mod.gated_rmsnorm_modulate(
        inp["residual"], inp["update"], inp["gate"], inp["weight"], inp["scale"], inp["shift"])
    assert np.array_equal(host(res), o_res)
    assert np.array_equal(host(rstd), o_rstd), stat_report(host(rstd), o_rstd)
    assert_within_ulp(host(out), o_out)
    assert_exact_where_stats_match(host(out), o_out, D, (host(rstd), o_rstd))


@pytest.mark.parametrize("D", WIDTHS)
@pytest.mark.parametrize("B,S,per_batch", [(1, 1, False), (2, 37, True), (1, 0, False)])
def test_all_ops_match_oracle(rm, oracle_mod, coop_rows, D, B, S, per_batch):
    if S == 0:
        S = coop_rows  # the largest few-rows launch
    seed = B * 7919 + S + D
    _ln(rm, oracle_mod, W.ln_modulate_inputs(B, S, D, seed=seed, per_batch_mod=per_batch,
                                             outlier_frac=0.05))
    _ln(rm, oracle_mod, W.ln_modulate_inputs(B, S, D, seed=seed + 1, per_batch_mod=per_batch),
        folded=True)
    _rms(rm, oracle_mod, W.rmsnorm_modulate_inputs(B, S, D, seed=seed + 2,
                                                   per_batch_mod=per_batch))
    _rms(rm, oracle_mod, W.rmsnorm_modulate_inputs(B, S, D, seed=seed + 3, with_weight=False))
    _gated(rm, oracle_mod, W.gated_inputs(B, S, D, seed=seed + 4, per_batch_mod=per_batch))


@pytest.mark.parametrize("D", WIDTHS)
def test_edge_and_special_rows(rm, oracle_mod, D):
    # exact cancellations, tiny / huge magnitudes (the scaled slow path) and
    # Inf / NaN rows (plain IEEE sums), each a row of a few-rows launch
    rows, labels = W.edge_rows(D)
    inp = W.ln_modulate_inputs(1, len(labels), D, seed=5)
    inp["x"] = rows.reshape(1, len(labels), D)
    gm, gr, om, orr = _ln(rm, oracle_mod, inp, check_stats=False)
    for i, l in enumerate(labels):
        assert gm[i] == om[i] or (np.isnan(gm[i]) and np.isnan(om[i])), (D, l, gm[i], om[i])
        assert gr[i] == orr[i], (D, l, gr[i], orr[i])
    rows, labels = W.special_rows(D)
    inp = W.ln_modulate_inputs(1, len(labels), D, seed=6)
    inp["x"] = rows.reshape(1, len(labels), D)
    gm, gr, om, orr = _ln(rm, oracle_mod, inp, check_stats=False)
    for i in range(len(labels)):
        assert (gm[i] == om[i]) or (np.isnan(gm[i]) and np.isnan(om[i]))
        assert np.isnan(gr[i]) and np.isnan(orr[i])
    # the same rows through RMSNorm (sum of squares only) and through the
    # gated op (as the residual, with a zero update, so the residual stream
    # equals the rows exactly)
    for rows, labels in (W.edge_rows(D), W.special_rows(D)):
        S = len(labels)
        rinp = W.rmsnorm_modulate_inputs(1, S, D, seed=7)
        rinp["x"] = rows.reshape(1, S, D)
        rstd = torch.empty(S, dtype=torch.float32, device="cuda")
        out = rm.rmsnorm_modulate(dev(rinp["x"]), dev(rinp["weight"]), dev(rinp["scale"]),
                                  dev(rinp["shift"]), rstd_out=rstd)
        torch.cuda.synchronize()
        o_out, o_rstd = oracle_mod.rmsnorm_modulate(rinp["x"], rinp["weight"], rinp["scale"],
                                                    rinp["shift"])
        g = host(rstd)
        for i, l in enumerate(labels):
            assert g[i] == o_rstd[i] or (np.isnan(g[i]) and np.isnan(o_rstd[i])), (D, l)
        assert_within_ulp(host(out), o_out)
        ginp = W.gated_inputs(1, S, D, seed=8)
        ginp["residual"] = rows.reshape(1, S, D)
        ginp["update"] = np.zeros((1, S, D), np.uint16)
        rstd = torch.empty(S, dtype=torch.float32, device="cuda")
        res, out = rm.gated_rmsnorm_modulate(dev(ginp["residual"]), dev(ginp["update"]),
                                             dev(ginp["gate"]), dev(ginp["weight"]),
                                             dev(ginp["scale"]), dev(ginp["shift"]),
                                             rstd_out=rstd)
        torch.cuda.synchronize()
        o_res, o_out, o_rstd = oracle_mod.gated_rmsnorm_modulate(
            ginp["residual"], ginp["update"], ginp["gate"], ginp["weight"], ginp["scale"],
            ginp["shift"])
        assert_within_ulp(host(res), o_res, max_ulp=0, frac_1ulp=1.0, what="res")
        g = host(rstd)
        for i, l in enumerate(labels):
            assert g[i] == o_rstd[i] or (np.isnan(g[i]) and np.isnan(o_rstd[i])), (D, l)
        assert_within_ulp(host(out), o_out)


@pytest.mark.parametrize("D", WIDTHS)
def test_same_bits_as_the_ring(rm, coop_rows, D):
    # coop_rows rows take the few-rows launch, coop_rows + 1 the ring kernels:
    # the shared rows come out bit-identical (out, mean, rstd; gated res)
    n = coop_rows + 1
    inp = W.ln_modulate_inputs(1, n, D, seed=D, outlier_frac=0.05)
    x, sc, sh = dev(inp["x"]), dev(inp["scale"]), dev(inp["shift"])
    for f in (rm.ln_modulate, rm.ln_modulate_folded):
        outs = []
        for rows in (n, coop_rows):
            mean = torch.empty(rows, dtype=torch.float32, device="cuda")
            rstd = torch.empty_like(mean)
            o = f(x[:, :rows].contiguous(), sc, sh, mean_out=mean, rstd_out=rstd)
            outs.append((host(o)[:, :coop_rows], host(mean)[:coop_rows], host(rstd)[:coop_rows]))
        for a, b in zip(*outs):
            assert np.array_equal(a, b)
    g = W.gated_inputs(1, n, D, seed=D + 1)
    args = [dev(g[k]) for k in ("residual", "update", "gate", "weight", "scale", "shift")]
    outs = []
    for rows in (n, coop_rows):
        rstd = torch.empty(rows, dtype=torch.float32, device="cuda")
        res, o = rm.gated_rmsnorm_modulate(args[0][:, :rows].contiguous(),
                                           args[1][:, :rows].contiguous(), *args[2:],
                                           rstd_out=rstd)
        outs.append((host(res)[:, :coop_rows], host(o)[:, :coop_rows], host(rstd)[:coop_rows]))
    for a, b in zip(*outs):
        assert np.array_equal(a, b)


def test_in_place(rm, oracle_mod):
    # out aliases x; the gated residual stream written over the residual
    B, S, D = 2, 40, 3072
    inp = W.ln_modulate_inputs(B, S, D, seed=11, per_batch_mod=True)
    want, _, _ = oracle_mod.ln_modulate(inp["x"], inp["scale"], inp["shift"])
    x = dev(inp["x"])
    rm.ln_modulate(x, dev(inp["scale"]), dev(inp["shift"]), out=x)
    torch.cuda.synchronize()
    assert_within_ulp(host(x), want)
    g = W.gated_inputs(1, 33, 1024, seed=12)
    o_res, o_out, _ = oracle_mod.gated_rmsnorm_modulate(
        g["residual"], g["update"], g["gate"], g["weight"], g["scale"], g["shift"])
    r = dev(g["residual"])
    res, out = rm.gated_rmsnorm_modulate(r, dev(g["update"]), dev(g["gate"]), dev(g["weight"]),
                                         dev(g["scale"]), dev(g["shift"]), res_out=r)
    torch.cuda.synchronize()
    assert np.array_equal(host(r), o_res)
    assert_within_ulp(host(out), o_out)
