"""Parity of qk_layernorm (CUDA, through the C ABI) with the oracle."""
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


def run_qk(rm, oracle_mod, inp, eps=1e-5):
    rq, rk = inp["rows_q"], inp["rows_k"]
    mean = torch.empty(rq + rk, dtype=torch.float32, device="cuda")
    rstd = torch.empty_like(mean)
    qo, ko = rm.qk_layernorm(dev(inp["q"]), dev(inp["k"]), dev(inp["wq"]), dev(inp["bq"]),
                             dev(inp["wk"]), dev(inp["bk"]), eps, mean_out=mean, rstd_out=rstd)
    torch.cuda.synchronize()
    oq, ok, om, orr = oracle_mod.qk_layernorm(inp["q"], inp["k"], inp["wq"], inp["bq"],
                                              inp["wk"], inp["bk"], eps)
    assert stat_report(host(mean), om)[1] <= 1e-5
    assert stat_report(host(rstd), orr)[1] <= 1e-5
    dq = assert_within_ulp(host(qo), oq, what="q")
    dk = assert_within_ulp(host(ko), ok, what="k")
    gm, gr = host(mean), host(rstd)
    assert_exact_where_stats_match(host(qo), oq, 128, (gm[:rq], om[:rq]), (gr[:rq], orr[:rq]))
    assert_exact_where_stats_match(host(ko), ok, 128, (gm[rq:], om[rq:]), (gr[rq:], orr[rq:]))
    return dq, dk, host(mean), host(rstd), om, orr


@pytest.mark.parametrize("rq,rk", [(1, 1), (7, 3), (64, 64), (1000, 333), (0, 50), (50, 0)])
def test_small(rm, oracle_mod, rq, rk):
    inp = W.qk_inputs(rq, rk, 128, seed=rq + 3 * rk)
    dq, dk, gm, gr, om, orr = run_qk(rm, oracle_mod, inp)
    assert np.array_equal(gm, om) and np.array_equal(gr, orr)


def test_glm_full_size(rm, oracle_mod):
    inp = W.WORKLOADS["qk_layernorm_glm_1x4352x32x128"].make()
    dq, dk, gm, gr, om, orr = run_qk(rm, oracle_mod, inp)
    assert (gr == orr).mean() > 0.9999 and (gm == om).mean() > 0.9999


def test_edge_and_special_rows(rm, oracle_mod):
    e, _ = W.edge_rows(128)
    sp, _ = W.special_rows(128)
    inp = W.qk_inputs(e.shape[0], sp.shape[0], 128, seed=1)
    inp["q"], inp["k"] = e, sp
    rq, rk = e.shape[0], sp.shape[0]
    mean = torch.empty(rq + rk, dtype=torch.float32, device="cuda")
    rstd = torch.empty_like(mean)
    qo, ko = rm.qk_layernorm(dev(e), dev(sp), dev(inp["wq"]), dev(inp["bq"]), dev(inp["wk"]),
                             dev(inp["bk"]), 1e-5, mean_out=mean, rstd_out=rstd)
    torch.cuda.synchronize()
    oq, ok, om, orr = oracle_mod.qk_layernorm(e, sp, inp["wq"], inp["bq"], inp["wk"], inp["bk"],
                                              1e-5)
    assert_within_ulp(host(qo), oq)
    assert_within_ulp(host(ko), ok)
    g = host(rstd)
    assert np.all((g == orr) | (np.isnan(g) & np.isnan(orr)))
    gm = host(mean)
    assert_exact_where_stats_match(host(qo), oq, 128, (gm[:rq], om[:rq]), (g[:rq], orr[:rq]))
    assert_exact_where_stats_match(host(ko), ok, 128, (gm[rq:], om[rq:]), (g[rq:], orr[rq:]),
                                   min_match=0)
