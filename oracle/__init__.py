"""rmsmod oracle -- TEST INFRASTRUCTURE ONLY.

A plain, slow CPU statement (``rmsmod_oracle.c``) of the fused adaLN row
operations, plus this ctypes wrapper that takes and returns numpy arrays.
Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never calls it,
and it shares no code with the CUDA path.

bf16 tensors are passed as ``numpy.uint16`` arrays holding the bf16 bit
patterns; fp32 inputs and outputs are ``numpy.float32``.

Parity status per function (what pins it; see ``tests/test_oracle_*.py``):

* ``round_bf16``: exhaustive over all 2^32 fp32 patterns against torch's
  fp32->bf16 cast.
* ``modulate``, ``residual_gate_add``, ``conv_bias_epilogue``: bit-identical
  to the eager torch bf16 op chain on CPU (the definition the pages give).
* ``round_f16`` (the C fp32 -> _Float16 conversion): exhaustive over all 2^32
  fp32 patterns against numpy's float32 -> float16 cast; ``modulate_f16``:
  bit-identical to the eager torch fp16 chain on CPU.
* row statistics: against exact rational arithmetic (``fractions``) rounded
  once to fp32, closed forms (constant and zero rows), invariants.
* ``ln_modulate``, ``rmsnorm_modulate``, ``gated_rmsnorm_modulate``,
  ``qk_layernorm``, ``rmsnorm_silu_cl``: fp64 brute force on small rows,
  closed forms, the bias-fold identity, permutation equivariance.
* ``token_tree_sum`` and ``ln_modulate_backward``: exact integer sums,
  hand-worked cases where the tree order decides the result, batch
  invariance; the row reductions c1, c2 against exact rational sums
  (``fractions``) rounded once; grad_x, grad_scale, grad_shift against torch
  autograd in fp64; the projection invariants of the LayerNorm backward.
* ``ln_modulate_folded``: fp64 brute force, torch layer_norm in fp64 with the
  folded weight and bias, closed forms (zero modulation = LayerNorm, weight 2
  doubles it, constant rows give the shift), the bound to the lossless chain.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rmsmod_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-fvisibility=hidden", "-Wall", "-Wextra"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no FMA contraction, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # A test may point this at a deliberately mutated build of the
            # oracle (tests/test_oracle_mutations.py); normally unset.
            override = os.environ.get("RMSMOD_ORACLE_LIB")
            if override:
                lib = ctypes.CDLL(override)
            else:
                build()
                lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int64
            F = ctypes.c_float
            lib.oracle_round_bf16.argtypes = [F]
            lib.oracle_round_bf16.restype = ctypes.c_uint16
            lib.oracle_round_bf16_array.argtypes = [P, P, I]
            lib.oracle_round_bf16_sweep.argtypes = [ctypes.c_uint32, I, P]
            lib.oracle_modulate.argtypes = [P, P, P, P, I, I, I, I]
            lib.oracle_round_f16.argtypes = [F]
            lib.oracle_round_f16.restype = ctypes.c_uint16
            lib.oracle_round_f16_sweep.argtypes = [ctypes.c_uint32, I, P]
            lib.oracle_modulate_f16.argtypes = [P, P, P, P, I, I, I, I]
            lib.oracle_residual_gate_add.argtypes = [P, P, P, P, I, I, I, I]
            lib.oracle_conv_bias_epilogue.argtypes = [P, P, ctypes.c_int, P, P, I, I]
            lib.oracle_row_stats.argtypes = [P, I, I, P, P, P]
            lib.oracle_ln_normalize.argtypes = [P, P, I, I, F, P, P]
            lib.oracle_rms_normalize.argtypes = [P, P, P, I, I, F, P]
            lib.oracle_ln_modulate.argtypes = [P, P, P, P, I, I, I, I, F, P, P]
            lib.oracle_ln_modulate_folded.argtypes = [P, P, P, P, I, I, I, I, F, P, P]
            lib.oracle_rmsnorm_modulate.argtypes = [P, P, P, P, P, I, I, I, I, F, P]
            lib.oracle_gated_rmsnorm_modulate.argtypes = [P, P, P, I, P, P, P, I, P, P, I, I,
                                                          I, F, P]
            lib.oracle_qk_layernorm.argtypes = [P, P, P, P, P, P, P, P, I, I, I, F, P, P]
            lib.oracle_rmsnorm_silu_cl.argtypes = [P, P, ctypes.c_int, P, P, I, I, F, P]
            lib.oracle_token_tree_sum.argtypes = [P, I, P]
            lib.oracle_token_tree_sum.restype = F
            lib.oracle_ln_modulate_backward.argtypes = [P, P, P, P, P, I, I, I, I, P, P, P, P,
                                                        P, P]
            for name in ("oracle_round_bf16_array", "oracle_round_bf16_sweep", "oracle_modulate",
                         "oracle_round_f16_sweep", "oracle_modulate_f16",
                         "oracle_residual_gate_add", "oracle_conv_bias_epilogue",
                         "oracle_row_stats", "oracle_ln_normalize", "oracle_rms_normalize",
                         "oracle_ln_modulate", "oracle_ln_modulate_folded",
                         "oracle_rmsnorm_modulate",
                         "oracle_gated_rmsnorm_modulate", "oracle_qk_layernorm",
                         "oracle_rmsnorm_silu_cl", "oracle_ln_modulate_backward"):
                getattr(lib, name).restype = None
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _u16(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected uint16 bf16 bit patterns, got {a.dtype}")
    return a


def _f32(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.float32:
        raise TypeError(f"expected float32, got {a.dtype}")
    return a


def _mod_rows(m, B, D):
    """scale/shift/gate given as [D], [1, D], [B, D] or [B, 1, D] -> ([rows, D], bstride)."""
    m = _u16(m).reshape(-1, D)
    if m.shape[0] == 1:
        return m, 0
    if m.shape[0] != B:
        raise ValueError(f"modulation rows {m.shape[0]} do not match batch {B}")
    return m, D


# --------------------------------------------------------------------------
# bf16 rounding
# --------------------------------------------------------------------------

def round_bf16(v: np.ndarray) -> np.ndarray:
    v = _f32(v)
    out = np.empty(v.shape, np.uint16)
    _load().oracle_round_bf16_array(_p(v), _p(out), v.size)
    return out


def round_bf16_sweep(start: int, count: int) -> np.ndarray:
    out = np.empty(count, np.uint16)
    _load().oracle_round_bf16_sweep(ctypes.c_uint32(start), count, _p(out))
    return out


def round_f16_sweep(start: int, count: int) -> np.ndarray:
    """fp16 bit patterns of the fp32 values with patterns start .. start+count-1."""
    out = np.empty(count, np.uint16)
    _load().oracle_round_f16_sweep(ctypes.c_uint32(start), count, _p(out))
    return out


# --------------------------------------------------------------------------
# elementwise chains
# --------------------------------------------------------------------------

def modulate(y, scale, shift):
    """y [B, S, D] -> R(R(y * R(1 + scale)) + shift)."""
    y = _u16(y)
    B, S, D = y.shape
    sc, bs = _mod_rows(scale, B, D)
    sh, bs2 = _mod_rows(shift, B, D)
    assert bs == bs2
    out = np.empty_like(y)
    _load().oracle_modulate(_p(y), _p(sc), _p(sh), _p(out), B, S, D, bs)
    return out


def modulate_f16(y, scale, shift):
    """fp16 bit patterns: y [B, S, D] -> R16(R16(y * R16(1 + scale)) + shift)."""
    y = _u16(y)
    B, S, D = y.shape
    sc, bs = _mod_rows(scale, B, D)
    sh, bs2 = _mod_rows(shift, B, D)
    assert bs == bs2
    out = np.empty_like(y)
    _load().oracle_modulate_f16(_p(y), _p(sc), _p(sh), _p(out), B, S, D, bs)
    return out


def residual_gate_add(residual, gate, update):
    """[B, S, D] -> R(residual + R(gate * update)), gate broadcast over S."""
    residual = _u16(residual)
    update = _u16(update)
    B, S, D = residual.shape
    g, gs = _mod_rows(gate, B, D)
    out = np.empty_like(residual)
    _load().oracle_residual_gate_add(_p(residual), _p(g), _p(update), _p(out), B, S, D, gs)
    return out


def conv_bias_epilogue(x, bias, h=None):
    """x [pixels, C] channels-last; bias fp32 or bf16 [C]; optional residual h."""
    x = _u16(x)
    C = x.shape[-1]
    x2 = x.reshape(-1, C)
    is32 = 1 if np.asarray(bias).dtype == np.float32 else 0
    bias = _f32(bias) if is32 else _u16(bias)
    h2 = None if h is None else _u16(h).reshape(-1, C)
    out = np.empty_like(x2)
    _load().oracle_conv_bias_epilogue(_p(x2), _p(bias), is32, _p(h2), _p(out), x2.shape[0], C)
    return out.reshape(x.shape)


# --------------------------------------------------------------------------
# statistics and normalisation
# --------------------------------------------------------------------------

def row_stats(x):
    """x [rows, n] -> (mean, var, meansq) fp32 per row."""
    x = _u16(x)
    rows, n = x.shape
    mean = np.empty(rows, np.float32)
    var = np.empty(rows, np.float32)
    msq = np.empty(rows, np.float32)
    _load().oracle_row_stats(_p(x), rows, n, _p(mean), _p(var), _p(msq))
    return mean, var, msq


def ln_normalize(x, eps):
    x = _u16(x)
    D = x.shape[-1]
    rows = x.size // D
    y = np.empty_like(x)
    mean = np.empty(rows, np.float32)
    rstd = np.empty(rows, np.float32)
    _load().oracle_ln_normalize(_p(x), _p(y), rows, D, eps, _p(mean), _p(rstd))
    return y, mean, rstd


def rms_normalize(x, weight, eps):
    x = _u16(x)
    D = x.shape[-1]
    rows = x.size // D
    w = None if weight is None else _u16(weight)
    y = np.empty_like(x)
    rstd = np.empty(rows, np.float32)
    _load().oracle_rms_normalize(_p(x), _p(w), _p(y), rows, D, eps, _p(rstd))
    return y, rstd


# --------------------------------------------------------------------------
# fused operations
# --------------------------------------------------------------------------

def ln_modulate(x, scale, shift, eps=1e-6):
    """x [B, S, D] -> (out, mean [B*S], rstd [B*S])."""
    x = _u16(x)
    B, S, D = x.shape
    sc, bs = _mod_rows(scale, B, D)
    sh, _ = _mod_rows(shift, B, D)
    out = np.empty_like(x)
    mean = np.empty(B * S, np.float32)
    rstd = np.empty(B * S, np.float32)
    _load().oracle_ln_modulate(_p(x), _p(sc), _p(sh), _p(out), B, S, D, bs, eps, _p(mean),
                               _p(rstd))
    return out, mean, rstd


def ln_modulate_folded(x, scale, shift, eps=1e-6):
    """Single-rounding tier: x [B, S, D] -> (out, mean [B*S], rstd [B*S])."""
    x = _u16(x)
    B, S, D = x.shape
    sc, bs = _mod_rows(scale, B, D)
    sh, _ = _mod_rows(shift, B, D)
    out = np.empty_like(x)
    mean = np.empty(B * S, np.float32)
    rstd = np.empty(B * S, np.float32)
    _load().oracle_ln_modulate_folded(_p(x), _p(sc), _p(sh), _p(out), B, S, D, bs, eps,
                                      _p(mean), _p(rstd))
    return out, mean, rstd


def rmsnorm_modulate(x, weight, scale, shift, eps=1e-6):
    """x [B, S, D], weight [D] or None -> (out, rstd [B*S])."""
    x = _u16(x)
    B, S, D = x.shape
    w = None if weight is None else _u16(weight)
    sc, bs = _mod_rows(scale, B, D)
    sh, _ = _mod_rows(shift, B, D)
    out = np.empty_like(x)
    rstd = np.empty(B * S, np.float32)
    _load().oracle_rmsnorm_modulate(_p(x), _p(w), _p(sc), _p(sh), _p(out), B, S, D, bs, eps,
                                    _p(rstd))
    return out, rstd


def gated_rmsnorm_modulate(residual, update, gate, weight, scale, shift, eps=1e-6):
    """-> (res, out, rstd)."""
    residual = _u16(residual)
    update = _u16(update)
    B, S, D = residual.shape
    g, gs = _mod_rows(gate, B, D)
    w = None if weight is None else _u16(weight)
    sc, bs = _mod_rows(scale, B, D)
    sh, _ = _mod_rows(shift, B, D)
    res = np.empty_like(residual)
    out = np.empty_like(residual)
    rstd = np.empty(B * S, np.float32)
    _load().oracle_gated_rmsnorm_modulate(_p(residual), _p(update), _p(g), gs, _p(w), _p(sc),
                                          _p(sh), bs, _p(res), _p(out), B, S, D, eps, _p(rstd))
    return res, out, rstd


def qk_layernorm(q, k, wq, bq, wk, bk, eps=1e-5):
    """q, k [..., head_dim] -> (q_out, k_out, mean [rq+rk], rstd [rq+rk])."""
    q = _u16(q)
    k = _u16(k)
    hd = q.shape[-1]
    rq = q.size // hd
    rk = k.size // hd
    qo = np.empty_like(q)
    ko = np.empty_like(k)
    mean = np.empty(rq + rk, np.float32)
    rstd = np.empty(rq + rk, np.float32)
    _load().oracle_qk_layernorm(_p(q), _p(k), _p(_u16(wq)), _p(_u16(bq)), _p(_u16(wk)),
                                _p(_u16(bk)), _p(qo), _p(ko), rq, rk, hd, eps, _p(mean),
                                _p(rstd))
    return qo, ko, mean, rstd


def rmsnorm_silu_cl(x, bias, gamma, eps=1e-6):
    """x [..., C] channels-last (pixels x C dense); bias fp32/bf16 [C] or None.
    -> (out, rstd [pixels])."""
    x = _u16(x)
    C = x.shape[-1]
    pixels = x.size // C
    if bias is None:
        b, is32 = None, 0
    else:
        is32 = 1 if np.asarray(bias).dtype == np.float32 else 0
        b = _f32(bias) if is32 else _u16(bias)
    out = np.empty_like(x)
    rstd = np.empty(pixels, np.float32)
    _load().oracle_rmsnorm_silu_cl(_p(x), _p(b), is32, _p(_u16(gamma)), _p(out), pixels, C, eps,
                                   _p(rstd))
    return out, rstd


# --------------------------------------------------------------------------
# backward of LayerNorm + modulate
# --------------------------------------------------------------------------

def token_tree_sum(v):
    """Fixed 32-way balanced-tree fp32 sum of a 1-D float32 array."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    scratch = np.empty(max(1, v.size), np.float32)
    return np.float32(_load().oracle_token_tree_sum(_p(v), v.size, _p(scratch)))


def ln_modulate_backward(x, scale, grad_out, mean, rstd):
    """x, grad_out [B, S, D] bf16 bits; scale [D] / [B, 1, D]; mean, rstd [B*S]
    (the forward's) -> (grad_x [B, S, D] bf16 bits, grad_scale [B, D] fp32,
    grad_shift [B, D] fp32, c1 [B*S], c2 [B*S])."""
    x = _u16(x)
    B, S, D = x.shape
    g = np.ascontiguousarray(_u16(grad_out).reshape(B, S, D))
    sc, bs = _mod_rows(scale, B, D)
    mean = np.ascontiguousarray(mean, dtype=np.float32).reshape(-1)
    rstd = np.ascontiguousarray(rstd, dtype=np.float32).reshape(-1)
    gx = np.empty_like(x)
    gsc = np.empty((B, D), np.float32)
    gsh = np.empty((B, D), np.float32)
    c1 = np.empty(B * S, np.float32)
    c2 = np.empty(B * S, np.float32)
    work = np.empty(3 * max(1, S), np.float32)
    _load().oracle_ln_modulate_backward(_p(x), _p(sc), _p(g), _p(mean), _p(rstd), B, S, D, bs,
                                        _p(gx), _p(gsc), _p(gsh), _p(c1), _p(c2), _p(work))
    return gx, gsc, gsh, c1, c2
