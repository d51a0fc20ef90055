"""Parity of ln_modulate (CUDA, through the C ABI) with the oracle.

Bars: mean / rstd within 1e-5 relative (and reported bit-identical fraction);
output within 1 bf16 ulp on >= 99.9% of elements and 2 ulp everywhere
(ordinal ulp distance, +-0 equal, NaN only where the oracle has NaN).
"""
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


def run_ln(rm, oracle_mod, inp, eps=1e-6, check_stats=True):
    x, sc, sh = dev(inp["x"]), dev(inp["scale"]), dev(inp["shift"])
    B, S = inp["B"], inp["S"]
    mean = torch.empty(B * S, dtype=torch.float32, device="cuda")
    rstd = torch.empty_like(mean)
    out = rm.ln_modulate(x, sc, sh, eps, mean_out=mean, rstd_out=rstd)
    torch.cuda.synchronize()
    o_out, o_mean, o_rstd = oracle_mod.ln_modulate(inp["x"], inp["scale"], inp["shift"], eps)
    if check_stats:
        fm, wm = stat_report(host(mean), o_mean)
        fr, wr = stat_report(host(rstd), o_rstd)
        assert wm <= 1e-5 and wr <= 1e-5, (wm, wr)
    d = assert_within_ulp(host(out), o_out)
    assert_exact_where_stats_match(host(out), o_out, inp["D"], (host(mean), o_mean),
                                   (host(rstd), o_rstd), min_match=0.99 if check_stats else 0)
    return d, host(mean), host(rstd), o_mean, o_rstd


@pytest.mark.parametrize("B,S,D,per_batch", [
    (1, 256, 1024, False),     # the small config, full
    (2, 37, 8, True),          # one vector per row
    (3, 29, 24, True),         # ragged: 3 vectors
    (1, 33, 136, False),       # 17 vectors: ragged over one warp
    (2, 19, 1000, True),       # 125 vectors
    (1, 50, 3072, False),
    (1, 23, 4096, False),
    (1, 9, 5120, False),       # two warps per row
    (2, 5, 8192, True),
    (1, 7, 16384, False),      # four warps per row, the maximum D
    (1, 5, 12296, False),      # ragged over four warps
])
def test_shapes(rm, oracle_mod, B, S, D, per_batch):
    inp = W.ln_modulate_inputs(B, S, D, seed=B * 1000 + D, per_batch_mod=per_batch,
                               outlier_frac=0.1)
    d, gm, gr, om, orr = run_ln(rm, oracle_mod, inp)
    # the statistics are the correctly rounded exact values on both sides
    assert np.array_equal(gm, om) and np.array_equal(gr, orr)


def test_flux_full_size(rm, oracle_mod):
    inp = W.WORKLOADS["ln_modulate_flux_1x4608x3072"].make()
    d, gm, gr, om, orr = run_ln(rm, oracle_mod, inp)
    assert (gm == om).mean() > 0.9999 and (gr == orr).mean() > 0.9999
    assert (d == 0).mean() > 0.9999


def test_flux_cfg_full_size(rm, oracle_mod):
    inp = W.WORKLOADS["ln_modulate_flux_cfg_2x4608x3072"].make()
    d, gm, gr, om, orr = run_ln(rm, oracle_mod, inp)
    assert (d == 0).mean() > 0.9999


def test_edge_rows(rm, oracle_mod):
    for D in (64, 3072, 8192):
        rows, labels = W.edge_rows(D)
        inp = W.ln_modulate_inputs(1, len(labels), D, seed=3)
        inp["x"] = rows.reshape(1, len(labels), D)
        d, gm, gr, om, orr = run_ln(rm, oracle_mod, inp)
        for i, l in enumerate(labels):
            assert gm[i] == om[i] or (np.isnan(gm[i]) and np.isnan(om[i])), (D, l, gm[i], om[i])
            assert gr[i] == orr[i], (D, l, gr[i], orr[i])


def test_special_values(rm, oracle_mod):
    for D in (64, 3072, 8192):
        rows, labels = W.special_rows(D)
        inp = W.ln_modulate_inputs(1, len(labels), D, seed=4)
        inp["x"] = rows.reshape(1, len(labels), D)
        d, gm, gr, om, orr = run_ln(rm, oracle_mod, inp, check_stats=False)
        for i in range(len(labels)):
            assert (gm[i] == om[i]) or (np.isnan(gm[i]) and np.isnan(om[i]))
            assert np.isnan(gr[i]) and np.isnan(orr[i])


def test_in_place_and_chunk_views(rm, oracle_mod):
    B, S, D = 2, 40, 3072
    inp = W.ln_modulate_inputs(B, S, D, seed=7, per_batch_mod=True)
    want, _, _ = oracle_mod.ln_modulate(inp["x"], inp["scale"], inp["shift"])
    # scale/shift as chunk views of one [B, 2D] projection output (adaLN layout)
    proj = torch.cat([dev(inp["scale"]).view(B, D), dev(inp["shift"]).view(B, D)], dim=1)
    scale = proj[:, None, :D]
    shift = proj[:, None, D:]
    x = dev(inp["x"])
    rm.ln_modulate(x, scale, shift, out=x)  # out aliases x
    torch.cuda.synchronize()
    assert_within_ulp(host(x), want)


def test_empty_rows(rm):
    x = torch.empty(0, 5, 64, dtype=torch.bfloat16, device="cuda")
    s = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    out = rm.ln_modulate(x, s, s)
    assert out.shape == x.shape


def test_batch_invariance_and_determinism(rm):
    inp = W.ln_modulate_inputs(1, 3000, 3072, seed=9)
    x = dev(inp["x"])
    sc, sh = dev(inp["scale"]), dev(inp["shift"])
    full = host(rm.ln_modulate(x, sc, sh))
    again = host(rm.ln_modulate(x, sc, sh))
    assert np.array_equal(full, again)
    for start, n in ((0, 1), (1234, 1), (17, 257), (2999, 1)):
        part = host(rm.ln_modulate(x[:, start:start + n].contiguous(), sc, sh))
        assert np.array_equal(part, full[:, start:start + n])
