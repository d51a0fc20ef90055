"""The pins are sharp enough: plant one plausible mistake at a time in a copy
of the oracle (compiled on the CPU, never used outside this test) and check
that the oracle pin-suite fails on every mutant.  The exhaustive rounding
sweep is skipped for speed; the boundary-case rounding pins stay in."""
import os
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "rmsmod_oracle.c")

# (label, original text, mutated text): dropped terms, wrong signs, wrong
# indices, transposed operands, wrong divisors, wrong rounding.
MUTATIONS = [
    ("one_minus_scale", "round_bf16(1.0f + widen(scale))", "round_bf16(1.0f - widen(scale))"),
    ("minus_shift", "round_bf16(widen(t) + widen(shift))", "round_bf16(widen(t) - widen(shift))"),
    ("no_one_plus", "round_bf16(1.0f + widen(scale))", "round_bf16(widen(scale))"),
    ("round_half_up", "u += 0x7FFFu + ((u >> 16) & 1u);", "u += 0x8000u;"),
    ("truncate", "u += 0x7FFFu + ((u >> 16) & 1u);", "u += 0u;"),
    ("unbiased_var", "*var_f = (float)(csum_value(&s2) / (double)n);",
     "*var_f = (float)(csum_value(&s2) / (double)(n - 1));"),
    ("dropped_eps", "float t = stat + eps;", "float t = stat;"),
    ("rsqrt_of_var_no_sqrt", "float r = sqrtf(t);", "float r = t;"),
    ("plus_mean", "float centred = widen(xr[d]) - mean;", "float centred = widen(xr[d]) + mean;"),
    ("dropped_rms_weight", "v = v * widen(w[d]);", "v = v;"),
    ("qk_k_uses_q_weights", "qk_rows(k, wk, bk, k_out", "qk_rows(k, wq, bq, k_out"),
    ("qk_dropped_bias", "round_bf16(scaled + widen(b[d]))", "round_bf16(scaled)"),
    ("gate_times_residual", "widen(gate) * widen(update)", "widen(gate) * widen(residual)"),
    ("residual_dropped", "round_bf16(widen(residual) + widen(g))", "round_bf16(widen(g))"),
    ("bias_not_rounded_first", "return round_bf16(((const float*)bias)[c]);",
     "return (bf16_t)(((const float*)bias)[c] != 0.0f);"),
    ("silu_wrong_sign", "zd / (1.0 + exp(-zd))", "zd / (1.0 + exp(zd))"),
    ("gamma_dropped", "(widen(orow[c]) * rstd) * widen(gamma[c])", "(widen(orow[c]) * rstd)"),
    ("scale_batch_ignored", "const bf16_t* sc = scale + b * mod_bstride;",
     "const bf16_t* sc = scale;"),
    ("gate_batch_ignored", "const bf16_t* g = gate + b * gate_bstride;",
     "const bf16_t* g = gate;"),
    ("mean_square_not_squared", "csum_add(&s, v * v);", "csum_add(&s, v * fabs(v));"),
    ("mean_off_by_one_row", "ln_stats(xr, D, &mean, &var);", "ln_stats(xr, D - 1, &mean, &var);"),
    ("folded_weight_not_rounded", "float w = widen(round_bf16(1.0f + widen(sc[d])));",
     "float w = 1.0f + widen(sc[d]);"),
    ("folded_one_minus_scale", "round_bf16(1.0f + widen(sc[d]))", "round_bf16(1.0f - widen(sc[d]))"),
    ("folded_shift_dropped", "out[r * D + d] = round_bf16(scaled + widen(sh[d]));",
     "out[r * D + d] = round_bf16(scaled);"),
    ("folded_normed_rounded", "float scaled = normed * w;",
     "float scaled = widen(round_bf16(normed)) * w;"),
    ("bwd_no_modulation_factor", "float dy = widen(gr[d]) * s1;\n                csum_add",
     "float dy = widen(gr[d]);\n                csum_add"),
    ("bwd_c2_sign", "float t = (dy - c1) - yhat * c2;", "float t = (dy - c1) + yhat * c2;"),
    ("bwd_c1_dropped", "float t = (dy - c1) - yhat * c2;", "float t = dy - yhat * c2;"),
    ("bwd_scale_unrounded_y", "float y = widen(round_bf16((widen(x[r * D + d]) - mean[r]) * rstd[r]));",
     "float y = (widen(x[r * D + d]) - mean[r]) * rstd[r];"),
    ("bwd_tree_strided_pairs", "level[i] = level[2 * i] + level[2 * i + 1];",
     "level[i] = level[i] + level[i + width / 2];"),
    ("bwd_tree_stops_at_one_block", "    while (n > 1) {\n        int64_t m",
     "    while (n > 32) {\n        int64_t m"),
]


def build_mutant(label, old, new, outdir):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation {label}: pattern not found"
    path = os.path.join(outdir, f"{label}.c")
    with open(path, "w") as fh:
        fh.write(src.replace(old, new, 1))
    lib = os.path.join(outdir, f"{label}.so")
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                           "-w", path, "-o", lib, "-lm"])
    return lib


def pins_fail(lib):
    env = dict(os.environ, RMSMOD_ORACLE_LIB=lib)
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
           "-m", "not gpu",
           os.path.join(ROOT, "tests", "test_oracle_round.py"),
           os.path.join(ROOT, "tests", "test_oracle_chains.py"),
           os.path.join(ROOT, "tests", "test_oracle_stats.py"),
           os.path.join(ROOT, "tests", "test_oracle_ops.py"),
           os.path.join(ROOT, "tests", "test_oracle_folded.py"),
           os.path.join(ROOT, "tests", "test_oracle_backward.py"),
           "-k", "not exhaustive"]
    res = subprocess.run(cmd, env=env, capture_output=True, text=True, cwd=ROOT)
    return res.returncode != 0


def test_every_planted_mistake_is_caught():
    with tempfile.TemporaryDirectory() as d:
        libs = [(label, build_mutant(label, old, new, d)) for label, old, new in MUTATIONS]
        with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
            caught = dict(zip([l for l, _ in libs], ex.map(lambda t: pins_fail(t[1]), libs)))
    missed = [l for l, c in caught.items() if not c]
    assert not missed, f"pins did not catch: {missed}"


def test_unmutated_copy_passes():
    with tempfile.TemporaryDirectory() as d:
        lib = build_mutant("identity", "#include <math.h>", "#include <math.h>", d)
        assert not pins_fail(lib)
