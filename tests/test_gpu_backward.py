"""Parity of ln_modulate_backward (CUDA, through the C ABI) with the oracle.

Bars: grad_scale and grad_shift bit-identical (the fixed token trees are the
same fp32 operations in the same order on both sides; the products are
exact); grad_x within 1 bf16 ulp on >= 99.9% of elements and 2 ulp
everywhere, bit-identical on almost every row (the row reductions c1, c2 are
correctly rounded on both sides except near a rounding tie).  Both sides use
the oracle forward's mean / rstd.
"""
import numpy as np
import pytest
import torch

import workloads as W
from _gpu import dev, host
from _util import assert_within_ulp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rm():
    import rmsnorm_modulate_gb300 as rm

    yield rm
    assert rm.device_status(clear=True) == 0


def make(B, S, D, seed, per_batch=True, g_std=0.5):
    inp = W.ln_modulate_inputs(B, S, D, seed=seed, per_batch_mod=per_batch, outlier_frac=0.05)
    g = torch.Generator().manual_seed(seed + 1)
    inp["g"] = W.normal_bf16(g, (B, S, D), g_std)
    return inp


def run(rm, oracle_mod, inp, want_exact_rows=0.99):
    B, S, D = inp["B"], inp["S"], inp["D"]
    _, mean, rstd = oracle_mod.ln_modulate(inp["x"], inp["scale"], inp["shift"])
    gx_o, gsc_o, gsh_o, _, _ = oracle_mod.ln_modulate_backward(inp["x"], inp["scale"], inp["g"],
                                                               mean, rstd)
    x, sc, g = dev(inp["x"]), dev(inp["scale"]), dev(inp["g"])
    m, r = dev(mean), dev(rstd)
    gx, gsc, gsh = rm.ln_modulate_backward(x, sc, g, m, r)
    torch.cuda.synchronize()
    assert np.array_equal(host(gsh).view(np.uint32), gsh_o.view(np.uint32))
    assert np.array_equal(host(gsc).view(np.uint32), gsc_o.view(np.uint32))
    got = host(gx)
    d = assert_within_ulp(got, gx_o, what="grad_x")
    rows_exact = (got.reshape(B * S, D) == gx_o.reshape(B * S, D)).all(axis=1).mean()
    assert rows_exact >= want_exact_rows, rows_exact
    return d


@pytest.mark.parametrize("B,S,D,per_batch", [
    (1, 256, 1024, False),
    (2, 37, 64, True),      # a partial token block per batch
    (3, 33, 136, True),     # 33 tokens: two blocks, ragged row vectors
    (1, 32, 8, False),      # exactly one block, one vector per row
    (1, 1, 64, False),      # one token: the raw values, no tree
    (2, 1100, 256, True),   # 35 blocks: two tree levels above the first
    (1, 40, 3072, False),
    (1, 9, 16384, False),   # the largest D: one warp per CTA-share of shared memory
    # the one-pass kernel (D a multiple of 256 from 1024 to 3072, S >= 2)
    (3, 2, 1280, True),     # two-token sequences, five consumer warps
    (2, 100, 2048, True),   # a 4-token last block, eight warps
    (1, 40, 2560, False),   # ten warps
    (2, 1100, 1024, True),  # 35 blocks per batch, two CTAs per SM
    (3, 1700, 3072, True),  # more blocks than CTAs: each CTA loops over several
    (10, 40, 3072, True),   # more batches' s1 rows than shared memory holds
    # the trees above the first level
    (1, 32768, 8, False),   # 1024 blocks: 32 level-2 nodes, the widest lane groups
    (1, 33000, 8, False),   # 1032 blocks: past the lane groups, one thread per column
])
def test_shapes(rm, oracle_mod, B, S, D, per_batch):
    run(rm, oracle_mod, make(B, S, D, seed=B * 100 + S + D, per_batch=per_batch))


def test_flux_full_size(rm, oracle_mod):
    # every difference must come from a c1 / c2 rounding tie (rare); a fused
    # multiply-add anywhere in grad_x would leave ~1e-4 of all elements off
    inp = make(1, 4608, 3072, seed=21)
    d = run(rm, oracle_mod, inp, want_exact_rows=0.999)
    assert (d == 0).mean() > 0.99999


@pytest.mark.parametrize("need_x", [True, False])
def test_one_pass_and_token_only_paths_agree(rm, need_x):
    # the one-pass kernel (grad_x wanted) and the token-sum-only kernels give
    # the same bits; each equals the oracle's in test_shapes
    inp = make(2, 300, 2048, seed=25)
    x, sc, g = dev(inp["x"]), dev(inp["scale"]), dev(inp["g"])
    mean = torch.empty(600, dtype=torch.float32, device="cuda")
    rstd = torch.empty_like(mean)
    rm.ln_modulate(x, sc, dev(inp["shift"]), mean_out=mean, rstd_out=rstd)
    _, gsc0, gsh0 = rm.ln_modulate_backward(x, sc, g, mean, rstd, need_x=False)
    gx, gsc, gsh = rm.ln_modulate_backward(x, sc, g, mean, rstd, need_x=need_x)
    assert torch.equal(gsc, gsc0) and torch.equal(gsh, gsh0)
    if need_x:
        gx_only, _, _ = rm.ln_modulate_backward(x, sc, g, mean, rstd, need_mod=False)
        assert torch.equal(gx, gx_only)


@pytest.mark.parametrize("which", ["grad_scale", "grad_shift"])
def test_one_token_sum_requested(rm, which):
    # the C ABI with one modulation gradient left out: the other is unchanged
    B, S, D = 2, 300, 2048
    inp = make(B, S, D, seed=26)
    x, sc, g = dev(inp["x"]), dev(inp["scale"]), dev(inp["g"])
    mean = torch.empty(B * S, dtype=torch.float32, device="cuda")
    rstd = torch.empty_like(mean)
    rm.ln_modulate(x, sc, dev(inp["shift"]), mean_out=mean, rstd_out=rstd)
    gx, gsc, gsh = rm.ln_modulate_backward(x, sc, g, mean, rstd)
    want = gsc if which == "grad_scale" else gsh
    got = torch.full_like(want, float("nan"))
    gx1 = torch.empty_like(gx)
    ws = torch.empty(rm.backward_workspace_bytes(B, S, D), dtype=torch.uint8, device="cuda")
    P = __import__("ctypes").c_void_p
    ptr = lambda t: P(t.data_ptr())
    st = rm.library().ln_modulate_backward(
        ptr(x), ptr(sc), D, ptr(g), ptr(mean), ptr(rstd), B, S, D, ptr(gx1),
        ptr(got) if which == "grad_scale" else None, ptr(got) if which == "grad_shift" else None,
        ptr(ws), ws.numel(), P(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    assert torch.equal(got, want) and torch.equal(gx1, gx)


def test_token_sums_are_batch_invariant(rm):
    inp = make(3, 300, 256, seed=22)
    x, sc, g = dev(inp["x"]), dev(inp["scale"]), dev(inp["g"])
    mean = torch.empty(900, dtype=torch.float32, device="cuda")
    rstd = torch.empty_like(mean)
    rm.ln_modulate(x, sc, dev(inp["shift"]), mean_out=mean, rstd_out=rstd)
    _, gsc, gsh = rm.ln_modulate_backward(x, sc, g, mean, rstd, need_x=False)
    for b in range(3):
        _, gsc1, gsh1 = rm.ln_modulate_backward(
            x[b:b + 1].contiguous(), sc[b:b + 1].contiguous(), g[b:b + 1].contiguous(),
            mean[b * 300:(b + 1) * 300].contiguous(), rstd[b * 300:(b + 1) * 300].contiguous(),
            need_x=False)
        assert torch.equal(gsc1[0], gsc[b]) and torch.equal(gsh1[0], gsh[b])


def test_special_values(rm, oracle_mod):
    inp = make(1, 70, 64, seed=23, per_batch=False)
    g = inp["g"].reshape(70, 64).copy()
    g[3, 5] = 0x7F80    # +Inf
    g[40, 7] = 0xFF80   # -Inf
    g[41, 7] = 0x7F80   # +Inf in the same column: NaN in its token sum
    g[60, 9] = 0x7FC0   # NaN
    inp["g"] = g.reshape(1, 70, 64)
    B, S, D = 1, 70, 64
    _, mean, rstd = oracle_mod.ln_modulate(inp["x"], inp["scale"], inp["shift"])
    gx_o, gsc_o, gsh_o, _, _ = oracle_mod.ln_modulate_backward(inp["x"], inp["scale"], inp["g"],
                                                               mean, rstd)
    gx, gsc, gsh = rm.ln_modulate_backward(dev(inp["x"]), dev(inp["scale"]), dev(inp["g"]),
                                           dev(mean), dev(rstd))
    torch.cuda.synchronize()
    for got, want in ((host(gsh), gsh_o), (host(gsc), gsc_o)):
        assert np.array_equal(np.isnan(got), np.isnan(want))
        ok = ~np.isnan(want)
        assert np.array_equal(got[ok], want[ok])
    got = host(gx).reshape(S, D)
    want = gx_o.reshape(S, D)
    fin = lambda b: (b & 0x7F80) != 0x7F80
    # rows with a non-finite gradient are non-finite wherever the oracle's are
    for r in (3, 40, 41, 60):
        assert np.array_equal(fin(got[r]), fin(want[r]))
    clean = [r for r in range(S) if r not in (3, 40, 41, 60)]
    assert_within_ulp(got[clean], want[clean], what="grad_x (finite rows)")


def test_workspace_checks(rm):
    inp = make(1, 64, 64, seed=24)
    x, sc, g = dev(inp["x"]), dev(inp["scale"]), dev(inp["g"])
    mean = torch.zeros(64, dtype=torch.float32, device="cuda")
    rstd = torch.ones_like(mean)
    need = rm.backward_workspace_bytes(1, 64, 64)
    assert need == 2 * 2 * 64 * 4
    small = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):
        rm.ln_modulate_backward(x, sc, g, mean, rstd, workspace=small)
    lib = rm.library()
    P = __import__("ctypes").c_void_p
    gsc = torch.empty(1, 64, dtype=torch.float32, device="cuda")
    st = lib.ln_modulate_backward(P(x.data_ptr()), P(sc.data_ptr()), 0, P(g.data_ptr()),
                                  P(mean.data_ptr()), P(rstd.data_ptr()), 1, 64, 64, None,
                                  P(gsc.data_ptr()), None, P(small.data_ptr()), need - 16,
                                  P(torch.cuda.current_stream().cuda_stream))
    assert st == -2   # RMSMOD_ERR_SHAPE: workspace too small, nothing launched
