"""Batch invariance of LayerNorm + modulate, forward and backward, checked
bytewise at the scale of the Qwen-Image final AdaLN page (RL-Kernel #538,
§Prior art & reuse decision: a singleton against every row of large
batches, and B = 2 against B = 1 at long sequences).

For every batch position b of a batch of B different samples (per-sample
scale / shift rows, as the final AdaLN's projection gives them), the same
sample run alone (B = 1) must give byte-identical forward output, mean,
rstd, grad_x and per-batch token sums grad_scale[b], grad_shift[b].  The
token trees depend on S alone, and the statistics are the correctly rounded
exact values, so nothing may depend on B, on the position in the batch or
on the other samples.  S = 31 / 32 / 33 straddles the first 32-token tree
boundary; S = 6889 is the page's long sequence.  One singleton per shape is
also tied to the oracle (token sums bit-exact)."""
import numpy as np
import pytest
import torch

import workloads as W
from _gpu import dev, host

pytestmark = pytest.mark.gpu

D = 3072  # the Qwen-Image hidden size


@pytest.fixture(scope="module")
def rm():
    import rmsnorm_modulate_gb300 as rm

    yield rm
    assert rm.device_status(clear=True) == 0


def batch(B, S, seed):
    inp = W.ln_modulate_inputs(B, S, D, seed=seed, per_batch_mod=True, outlier_frac=0.02)
    g = torch.Generator().manual_seed(seed + 7)
    go = W.normal_bf16(g, (B, S, D), 0.5)
    return inp, go


def run(rm, x, sc, sh, go):
    B, S, _ = x.shape
    mean = torch.empty(B * S, dtype=torch.float32, device="cuda")
    rstd = torch.empty_like(mean)
    out = rm.ln_modulate(x, sc, sh, mean_out=mean, rstd_out=rstd)
    gx, gsc, gsh = rm.ln_modulate_backward(x, sc, go, mean, rstd)
    return out, mean, rstd, gx, gsc, gsh


def bits(t):
    return t.contiguous().view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32)


def assert_rows_invariant(rm, inp, go, singles):
    """Batch rows `singles` against the same samples run alone."""
    B, S = inp["B"], inp["S"]
    x, sc, sh, g = dev(inp["x"]), dev(inp["scale"]), dev(inp["shift"]), dev(go)
    out, mean, rstd, gx, gsc, gsh = run(rm, x, sc, sh, g)
    bad = []
    for b in singles:
        o1, m1, r1, gx1, gsc1, gsh1 = run(rm, x[b:b + 1].contiguous(), sc[b:b + 1].contiguous(),
                                          sh[b:b + 1].contiguous(), g[b:b + 1].contiguous())
        pairs = {"out": (out[b], o1[0]), "mean": (mean[b * S:(b + 1) * S], m1),
                 "rstd": (rstd[b * S:(b + 1) * S], r1), "grad_x": (gx[b], gx1[0]),
                 "grad_scale": (gsc[b], gsc1[0]), "grad_shift": (gsh[b], gsh1[0])}
        for name, (u, v) in pairs.items():
            if not torch.equal(bits(u), bits(v)):
                bad.append((b, name))
    torch.cuda.synchronize()
    assert not bad, f"batch rows differ from their singleton runs: {bad[:10]} ({len(bad)})"
    return host(mean), host(rstd), host(gsc), host(gsh)


def assert_token_sums_match_oracle(oracle_mod, inp, go, b, mean, rstd, gsc, gsh):
    """Batch row b's token sums against the oracle's backward of that sample,
    fed the same forward statistics."""
    S = inp["S"]
    sl = slice(b, b + 1)
    _, o_gsc, o_gsh, _, _ = oracle_mod.ln_modulate_backward(
        inp["x"][sl], inp["scale"][sl], go[sl], mean[b * S:(b + 1) * S],
        rstd[b * S:(b + 1) * S])
    assert np.array_equal(gsc[b], o_gsc.reshape(-1))
    assert np.array_equal(gsh[b], o_gsh.reshape(-1))


@pytest.mark.parametrize("S", [31, 32, 33])
@pytest.mark.parametrize("B", [64, 257])
def test_singleton_against_every_batch_row(rm, oracle_mod, B, S):
    inp, go = batch(B, S, seed=1000 * B + S)
    mean, rstd, gsc, gsh = assert_rows_invariant(rm, inp, go, range(B))
    # one batch row tied to the oracle: its token sums bit-exact
    assert_token_sums_match_oracle(oracle_mod, inp, go, B // 2, mean, rstd, gsc, gsh)


def test_singleton_against_a_large_batch_of_short_sequences(rm):
    # the page's B = 2048, S = 3 shape; every 8th row (256 singleton runs)
    inp, go = batch(2048, 3, seed=2048)
    assert_rows_invariant(rm, inp, go, range(0, 2048, 8))


@pytest.mark.parametrize("S", [4096, 6889])
def test_two_samples_against_one_at_long_sequences(rm, oracle_mod, S):
    inp, go = batch(2, S, seed=S)
    mean, rstd, gsc, gsh = assert_rows_invariant(rm, inp, go, (0, 1))
    assert_token_sums_match_oracle(oracle_mod, inp, go, 1, mean, rstd, gsc, gsh)
