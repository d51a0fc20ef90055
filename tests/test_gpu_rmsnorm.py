"""Parity of rmsnorm_modulate and gated_rmsnorm_modulate (CUDA, through the C
ABI) with the oracle: rstd within 1e-5 relative, residual stream bit-exact,
output within 1 ulp on >= 99.9% and 2 ulp everywhere."""
import numpy as np
import pytest
import torch

import workloads as W
from _gpu import dev, host, stat_report
from _util import assert_exact_where_stats_match, assert_within_ulp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rm():
    import rmsnorm_modulate_gb300 as rm

    yield rm
    assert rm.device_status(clear=True) == 0


def run_rms(rm, oracle_mod, inp, eps=1e-6):
    B, S = inp["B"], inp["S"]
    rstd = torch.empty(B * S, dtype=torch.float32, device="cuda")
    w = None if inp["weight"] is None else dev(inp["weight"])
    out = rm.rmsnorm_modulate(dev(inp["x"]), w, dev(inp["scale"]), dev(inp["shift"]), eps,
                              rstd_out=rstd)
    torch.cuda.synchronize()
    o_out, o_rstd = oracle_mod.rmsnorm_modulate(inp["x"], inp["weight"], inp["scale"],
                                                inp["shift"], eps)
    frac, worst = stat_report(host(rstd), o_rstd)
    assert worst <= 1e-5
    d = assert_within_ulp(host(out), o_out)
    assert_exact_where_stats_match(host(out), o_out, inp["D"], (host(rstd), o_rstd))
    return d, host(rstd), o_rstd


def run_gated(rm, oracle_mod, inp, eps=1e-6):
    B, S = inp["B"], inp["S"]
    rstd = torch.empty(B * S, dtype=torch.float32, device="cuda")
    w = None if inp["weight"] is None else dev(inp["weight"])
    res, out = rm.gated_rmsnorm_modulate(dev(inp["residual"]), dev(inp["update"]),
                                         dev(inp["gate"]), w, dev(inp["scale"]),
                                         dev(inp["shift"]), eps, rstd_out=rstd)
    torch.cuda.synchronize()
    o_res, o_out, o_rstd = oracle_mod.gated_rmsnorm_modulate(
        inp["residual"], inp["update"], inp["gate"], inp["weight"], inp["scale"], inp["shift"],
        eps)
    assert np.array_equal(host(res), o_res)  # elementwise chain: bit-exact
    frac, worst = stat_report(host(rstd), o_rstd)
    assert worst <= 1e-5
    d = assert_within_ulp(host(out), o_out)
    assert_exact_where_stats_match(host(out), o_out, inp["D"], (host(rstd), o_rstd))
    return d, host(rstd), o_rstd


@pytest.mark.parametrize("B,S,D,with_w,per_batch", [
    (1, 64, 8, True, False),
    (2, 31, 40, False, True),
    (1, 100, 1024, True, False),
    (2, 50, 2048, True, True),
    (1, 40, 4096, True, False),
    (1, 40, 4096, False, False),
    (1, 6, 6144, True, False),
    (2, 5, 16384, True, True),
])
def test_rms_shapes(rm, oracle_mod, B, S, D, with_w, per_batch):
    inp = W.rmsnorm_modulate_inputs(B, S, D, seed=D + B, with_weight=with_w,
                                    per_batch_mod=per_batch)
    d, g, o = run_rms(rm, oracle_mod, inp)
    assert np.array_equal(g, o)


@pytest.mark.parametrize("B,S,D,with_w,per_batch", [
    (1, 64, 8, True, False),
    (2, 31, 40, True, True),
    (1, 70, 4096, True, False),
    # the 4096-value ring (4 + 12 warps, 12 two-row slots) wrapping many
    # times, per-batch gate and modulation rows
    (2, 600, 4096, True, True),
    (1, 2000, 4096, False, False),
    # rows of 3080..4088 values: the same ring with a bounds-checked tail
    (1, 300, 3584, True, False),
    (2, 257, 4088, True, True),
    (2, 9, 8192, False, True),
])
def test_gated_shapes(rm, oracle_mod, B, S, D, with_w, per_batch):
    inp = W.gated_inputs(B, S, D, seed=D + 7 * B, with_weight=with_w, per_batch_mod=per_batch)
    d, g, o = run_gated(rm, oracle_mod, inp)
    assert np.array_equal(g, o)


def test_ernie_full_size(rm, oracle_mod):
    inp = W.WORKLOADS["rmsnorm_modulate_ernie_1x4216x4096"].make()
    d, g, o = run_rms(rm, oracle_mod, inp)
    assert (g == o).mean() > 0.9999 and (d == 0).mean() > 0.9999


def test_ernie_gated_full_size(rm, oracle_mod):
    inp = W.WORKLOADS["gated_rmsnorm_modulate_ernie_1x4216x4096"].make()
    d, g, o = run_gated(rm, oracle_mod, inp)
    assert (g == o).mean() > 0.9999 and (d == 0).mean() > 0.9999


def test_rms_edge_and_special_rows(rm, oracle_mod):
    for D in (64, 4096, 8192):
        for rows, labels in (W.edge_rows(D), W.special_rows(D)):
            inp = W.rmsnorm_modulate_inputs(1, len(labels), D, seed=2)
            inp["x"] = rows.reshape(1, len(labels), D)
            B, S = 1, len(labels)
            rstd = torch.empty(S, dtype=torch.float32, device="cuda")
            out = rm.rmsnorm_modulate(dev(inp["x"]), dev(inp["weight"]), dev(inp["scale"]),
                                      dev(inp["shift"]), 1e-6, rstd_out=rstd)
            torch.cuda.synchronize()
            o_out, o_rstd = oracle_mod.rmsnorm_modulate(inp["x"], inp["weight"], inp["scale"],
                                                        inp["shift"], 1e-6)
            g = host(rstd)
            for i, l in enumerate(labels):
                assert g[i] == o_rstd[i] or (np.isnan(g[i]) and np.isnan(o_rstd[i])), (D, l)
            assert_within_ulp(host(out), o_out)
            assert_exact_where_stats_match(host(out), o_out, D, (g, o_rstd), min_match=0)


def test_gated_edge_and_special_rows(rm, oracle_mod):
    # outlier and non-finite rows through the gated kernels' slow statistics:
    # the rows are the residual, the update is zero, so the residual stream
    # equals the rows exactly
    for D in (64, 3584, 4096):
        for rows, labels in (W.edge_rows(D), W.special_rows(D)):
            S = len(labels)
            inp = W.gated_inputs(1, S, D, seed=3)
            inp["residual"] = rows.reshape(1, S, D)
            inp["update"] = np.zeros((1, S, D), np.uint16)
            rstd = torch.empty(S, dtype=torch.float32, device="cuda")
            res, out = rm.gated_rmsnorm_modulate(dev(inp["residual"]), dev(inp["update"]),
                                                 dev(inp["gate"]), dev(inp["weight"]),
                                                 dev(inp["scale"]), dev(inp["shift"]), 1e-6,
                                                 rstd_out=rstd)
            torch.cuda.synchronize()
            o_res, o_out, o_rstd = oracle_mod.gated_rmsnorm_modulate(
                inp["residual"], inp["update"], inp["gate"], inp["weight"], inp["scale"],
                inp["shift"], 1e-6)
            # bit-exact, NaN payloads aside
            assert_within_ulp(host(res), o_res, max_ulp=0, frac_1ulp=1.0, what="res")
            g = host(rstd)
            for i, l in enumerate(labels):
                assert g[i] == o_rstd[i] or (np.isnan(g[i]) and np.isnan(o_rstd[i])), (D, l)
            assert_within_ulp(host(out), o_out)
            assert_exact_where_stats_match(host(out), o_out, D, (g, o_rstd), min_match=0)


def test_gated_in_place_residual(rm, oracle_mod):
    inp = W.gated_inputs(1, 33, 3072, seed=5)
    o_res, o_out, _ = oracle_mod.gated_rmsnorm_modulate(inp["residual"], inp["update"],
                                                        inp["gate"], inp["weight"],
                                                        inp["scale"], inp["shift"])
    r = dev(inp["residual"])
    res, out = rm.gated_rmsnorm_modulate(r, dev(inp["update"]), dev(inp["gate"]),
                                         dev(inp["weight"]), dev(inp["scale"]),
                                         dev(inp["shift"]), res_out=r)
    torch.cuda.synchronize()
    assert np.array_equal(host(r), o_res)
    assert_within_ulp(host(out), o_out)
