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


def run_qk(rm, oracle_mod, inp, eps=1e-5, hd=128):
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
    assert_exact_where_stats_match(host(qo), oq, hd, (gm[:rq], om[:rq]), (gr[:rq], orr[:rq]))
    assert_exact_where_stats_match(host(ko), ok, hd, (gm[rq:], om[rq:]), (gr[rq:], orr[rq:]))
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


@pytest.mark.parametrize("hd", [64, 96])
@pytest.mark.parametrize("rq,rk", [(1, 1), (33, 7), (1000, 333), (0, 50)])
def test_head_dims_below_128(rm, oracle_mod, hd, rq, rk):
    inp = W.qk_inputs(rq, rk, hd, seed=hd + rq + 3 * rk)
    dq, dk, gm, gr, om, orr = run_qk(rm, oracle_mod, inp, hd=hd)
    assert np.array_equal(gm, om) and np.array_equal(gr, orr)


@pytest.mark.parametrize("hd", [64, 96, 128])
def test_head_dim_edge_rows(rm, oracle_mod, hd):
    e, _ = W.edge_rows(hd)
    sp, _ = W.special_rows(hd)
    inp = W.qk_inputs(e.shape[0], sp.shape[0], hd, seed=2)
    inp["q"], inp["k"] = e, sp
    rq, rk = e.shape[0], sp.shape[0]
    mean = torch.empty(rq + rk, dtype=torch.float32, device="cuda")
    rstd = torch.empty_like(mean)
    qo, ko = rm.qk_layernorm(dev(inp["q"]), dev(inp["k"]), dev(inp["wq"]), dev(inp["bq"]),
                             dev(inp["wk"]), dev(inp["bk"]), 1e-5, mean_out=mean, rstd_out=rstd)
    torch.cuda.synchronize()
    oq, ok, om, orr = oracle_mod.qk_layernorm(inp["q"], inp["k"], inp["wq"], inp["bq"],
                                              inp["wk"], inp["bk"], 1e-5)
    # the same bar as at head_dim 128: <= 2 ulp everywhere, >= 99.9% within
    # 1 ulp (NaN exactly where the oracle has NaN), rstd bit-identical (NaN
    # where the oracle's is), rows exact where the statistics match
    assert_within_ulp(host(qo), oq, what="edge q")
    assert_within_ulp(host(ko), ok, what="special k")
    g, gm = host(rstd), host(mean)
    assert np.all((g == orr) | (np.isnan(g) & np.isnan(orr)))
    assert_exact_where_stats_match(host(qo), oq, hd, (gm[:rq], om[:rq]), (g[:rq], orr[:rq]))
    assert_exact_where_stats_match(host(ko), ok, hd, (gm[rq:], om[rq:]), (g[rq:], orr[rq:]),
                                   min_match=0)


def _qkv(T, H, hd, seed):
    """A fused QKV projection output [T, 3, H, hd] and the oracle inputs of
    its q and k slices (dense copies)."""
    inp_q = W.qk_inputs(T * H, T * H, hd, seed=seed)
    qkv = torch.empty(T, 3, H, hd, dtype=torch.bfloat16, device="cuda")
    qkv[:, 0] = dev(inp_q["q"]).view(T, H, hd)
    qkv[:, 1] = dev(inp_q["k"]).view(T, H, hd)
    qkv[:, 2] = 0
    return qkv, inp_q


@pytest.mark.parametrize("T,H,hd", [(37, 32, 128), (50, 24, 128), (40, 12, 96), (33, 40, 64),
                                    (1, 32, 128), (5, 3, 128)])
def test_strided_qkv_views(rm, oracle_mod, T, H, hd):
    qkv, inp = _qkv(T, H, hd, seed=T * H + hd)
    v_before = qkv[:, 2].clone()
    q, k = qkv[:, 0], qkv[:, 1]                       # token stride 3 * H * hd
    oq, ok, om, orr = oracle_mod.qk_layernorm(inp["q"], inp["k"], inp["wq"], inp["bq"],
                                              inp["wk"], inp["bk"], 1e-5)
    rows = T * H
    mean = torch.empty(2 * rows, dtype=torch.float32, device="cuda")
    rstd = torch.empty_like(mean)
    # separate dense outputs
    qo, ko = rm.qk_layernorm(q, k, dev(inp["wq"]), dev(inp["bq"]), dev(inp["wk"]),
                             dev(inp["bk"]), 1e-5, mean_out=mean, rstd_out=rstd)
    torch.cuda.synchronize()
    gm, gr = host(mean), host(rstd)
    assert_within_ulp(host(qo).reshape(-1), oq.reshape(-1), what="strided q")
    assert_within_ulp(host(ko).reshape(-1), ok.reshape(-1), what="strided k")
    assert_exact_where_stats_match(host(qo).reshape(-1), oq.reshape(-1), hd,
                                   (gm[:rows], om[:rows]), (gr[:rows], orr[:rows]))
    # in place inside the QKV buffer: v untouched
    rm.qk_layernorm(q, k, dev(inp["wq"]), dev(inp["bq"]), dev(inp["wk"]), dev(inp["bk"]), 1e-5,
                    q_out=q, k_out=k)
    torch.cuda.synchronize()
    assert torch.equal(qkv[:, 0].contiguous().view(-1), qo.view(-1))
    assert torch.equal(qkv[:, 1].contiguous().view(-1), ko.view(-1))
    assert torch.equal(qkv[:, 2], v_before)


def test_strided_overlap_is_refused(rm):
    qkv, inp = _qkv(8, 4, 128, seed=5)
    q, k = qkv[:, 0], qkv[:, 1]
    w, b = dev(inp["wq"]), dev(inp["bq"])
    # writing q's result over k's slice while k is an input: refused
    with pytest.raises(rm.RmsmodError):
        rm.qk_layernorm(q, k, w, b, w, b, 1e-5, q_out=k, k_out=q)
