"""Parity of ln_modulate_folded (single-rounding tier, CUDA through the C ABI)
with the oracle.

Bars as ln_modulate: mean / rstd within 1e-5 relative; output within 1 bf16
ulp on >= 99.9% of elements and 2 ulp everywhere, bit-identical on every row
whose statistics match the oracle's.
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


def run_folded(rm, oracle_mod, inp, eps=1e-6, check_stats=True):
    x, sc, sh = dev(inp["x"]), dev(inp["scale"]), dev(inp["shift"])
    B, S = inp["B"], inp["S"]
    mean = torch.empty(B * S, dtype=torch.float32, device="cuda")
    rstd = torch.empty_like(mean)
    out = rm.ln_modulate_folded(x, sc, sh, eps, mean_out=mean, rstd_out=rstd)
    torch.cuda.synchronize()
    o_out, o_mean, o_rstd = oracle_mod.ln_modulate_folded(inp["x"], inp["scale"], inp["shift"],
                                                          eps)
    if check_stats:
        _, wm = stat_report(host(mean), o_mean)
        _, wr = stat_report(host(rstd), o_rstd)
        assert wm <= 1e-5 and wr <= 1e-5, (wm, wr)
    d = assert_within_ulp(host(out), o_out)
    assert_exact_where_stats_match(host(out), o_out, inp["D"], (host(mean), o_mean),
                                   (host(rstd), o_rstd), min_match=0.99 if check_stats else 0)
    return d, host(mean), host(rstd), o_mean, o_rstd


@pytest.mark.parametrize("B,S,D,per_batch", [
    (1, 256, 1024, False),
    (2, 37, 8, True),
    (3, 29, 24, True),
    (2, 19, 1000, True),
    (1, 50, 3072, False),
    (1, 9, 5120, False),
    (1, 5, 12296, False),
])
def test_shapes(rm, oracle_mod, B, S, D, per_batch):
    inp = W.ln_modulate_inputs(B, S, D, seed=B * 1000 + D + 1, per_batch_mod=per_batch,
                               outlier_frac=0.1)
    d, gm, gr, om, orr = run_folded(rm, oracle_mod, inp)
    assert np.array_equal(gm, om) and np.array_equal(gr, orr)


def test_flux_cfg_full_size(rm, oracle_mod):
    inp = W.WORKLOADS["ln_modulate_flux_cfg_2x4608x3072"].make()
    d, gm, gr, om, orr = run_folded(rm, oracle_mod, inp)
    assert (d == 0).mean() > 0.9999


def test_edge_and_special_rows(rm, oracle_mod):
    for D in (64, 3072):
        rows, labels = W.edge_rows(D)
        inp = W.ln_modulate_inputs(1, len(labels), D, seed=3)
        inp["x"] = rows.reshape(1, len(labels), D)
        d, gm, gr, om, orr = run_folded(rm, oracle_mod, inp)
        assert np.array_equal(gr, orr)
        rows, labels = W.special_rows(D)
        inp = W.ln_modulate_inputs(1, len(labels), D, seed=4)
        inp["x"] = rows.reshape(1, len(labels), D)
        run_folded(rm, oracle_mod, inp, check_stats=False)


def test_shares_statistics_with_lossless_tier(rm):
    inp = W.ln_modulate_inputs(2, 64, 3072, seed=11, per_batch_mod=True)
    x, sc, sh = dev(inp["x"]), dev(inp["scale"]), dev(inp["shift"])
    m1 = torch.empty(128, dtype=torch.float32, device="cuda")
    r1, m2, r2 = torch.empty_like(m1), torch.empty_like(m1), torch.empty_like(m1)
    a = rm.ln_modulate(x, sc, sh, mean_out=m1, rstd_out=r1)
    b = rm.ln_modulate_folded(x, sc, sh, mean_out=m2, rstd_out=r2)
    torch.cuda.synchronize()
    assert torch.equal(m1, m2) and torch.equal(r1, r2)
    assert not torch.equal(a, b)


def test_in_place(rm, oracle_mod):
    inp = W.ln_modulate_inputs(1, 40, 3072, seed=12)
    want, _, _ = oracle_mod.ln_modulate_folded(inp["x"], inp["scale"], inp["shift"])
    x = dev(inp["x"])
    rm.ln_modulate_folded(x, dev(inp["scale"]), dev(inp["shift"]), out=x)
    torch.cuda.synchronize()
    assert_within_ulp(host(x), want)
