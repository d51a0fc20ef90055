"""rmsnorm_modulate_gb300 -- fused adaLN row normalisation + modulate for GB300.

Thin ctypes binding of ``librmsmod.so`` (C ABI in ``include/rmsmod.h``).
Each function here only checks tensor metadata, derives sizes and strides,
and passes device pointers plus the current CUDA stream to the library;
every step of the computation runs in the library's CUDA kernels.  There is
no CPU fallback: if the library is not built, or the tensors are not on a
CUDA device, the call raises.

Tensors are ``torch.bfloat16`` on a CUDA device with a contiguous innermost
dimension.  Modulation rows (``scale``, ``shift``, ``gate``) may be given
as ``[D]``, ``[1, D]``, ``[B, D]``, ``[1, 1, D]`` or ``[B, 1, D]``; per-batch
rows may be strided views (adaLN chunk views of one projection output).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "RmsmodError", "library", "library_path", "ln_modulate", "ln_modulate_folded",
    "ln_modulate_backward", "ln_modulate_backward_static", "backward_workspace_bytes",
    "rmsnorm_modulate",
    "gated_rmsnorm_modulate", "qk_layernorm", "rmsnorm_silu_cl", "modulate_scale_shift",
    "residual_gate_add", "conv_bias_epilogue", "supported", "status_string", "device_status",
    "selftest_wait_timeout",
    "OP_LN_MODULATE", "OP_RMSNORM_MODULATE", "OP_GATED_RMSNORM_MODULATE",
    "OP_QK_LAYERNORM", "OP_RMSNORM_SILU_CL", "OP_LN_MODULATE_FOLDED",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "librmsmod.so")

OP_LN_MODULATE = 1
OP_RMSNORM_MODULATE = 2
OP_GATED_RMSNORM_MODULATE = 3
OP_QK_LAYERNORM = 4
OP_RMSNORM_SILU_CL = 5
OP_LN_MODULATE_FOLDED = 6

_lock = threading.Lock()
_lib = None


class RmsmodError(RuntimeError):
    """A non-zero status returned by librmsmod."""

    def __init__(self, status: int, func: str):
        self.status = status
        super().__init__(f"{func}: status {status}: {status_string(status)}")


def library_path() -> str:
    return _LIB_PATH


def library() -> ctypes.CDLL:
    """The loaded librmsmod.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is not built: run `python -m rmsnorm_modulate_gb300._build` "
                "or __graft_entry__.build()")
        lib = ctypes.CDLL(_LIB_PATH)
        P, I, F, C = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int
        sig = {
            "ln_modulate": [P, P, P, P, I, I, I, I, F, P, P, P],
            "ln_modulate_folded": [P, P, P, P, I, I, I, I, F, P, P, P],
            "modulate_scale_shift_f16": [P, P, P, P, I, I, I, I, P],
            "ln_modulate_backward": [P, P, I, P, P, P, I, I, I, P, P, P, P, ctypes.c_size_t, P],
            "ln_modulate_backward_static": [P, P, I, P, P, P, I, I, I, P, P, P, P],
            "rmsnorm_modulate": [P, P, P, P, P, I, I, I, I, F, P, P],
            "gated_rmsnorm_modulate": [P, P, P, I, P, P, P, I, P, P, I, I, I, F, P, P],
            "qk_layernorm": [P, P, P, P, P, P, P, P, I, I, I, F, P, P, P],
            "qk_layernorm_strided": [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, F, P, P, P],
            "rmsnorm_silu_cl": [P, P, C, P, P, I, I, F, P, P],
            "modulate_scale_shift": [P, P, P, P, I, I, I, I, P],
            "residual_gate_add": [P, P, P, I, P, I, I, I, P],
            "conv_bias_epilogue": [P, P, C, P, P, I, I, P],
            "rmsmod_supported": [C, I, ctypes.POINTER(P), C],
            "rmsmod_status_string": [C],
            "rmsmod_version": [],
            "rmsmod_device_status": [ctypes.POINTER(ctypes.c_uint), C],
            "rmsmod_selftest_wait_timeout": [ctypes.c_uint64, P],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        lib.rmsmod_status_string.restype = ctypes.c_char_p
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return library().rmsmod_status_string(int(status)).decode()


def _call(name: str, *args) -> None:
    st = getattr(library(), name)(*args)
    if st != 0:
        raise RmsmodError(st, name)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _bf16(t, name, dtype=torch.bfloat16):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    return t


def _dense(t, name, dtype=torch.bfloat16):
    _bf16(t, name, dtype)
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _f32_out(t, n, name, device):
    if t is None:
        return None
    if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous() or t.numel() != n:
        raise ValueError(f"{name} must be a contiguous float32 CUDA tensor of {n} elements")
    return t


def _mod_rows(t, B, D, name, dtype=torch.bfloat16):
    """-> batch stride in elements (0 = one row shared by every batch)."""
    _bf16(t, name, dtype)
    if t.shape[-1] != D or t.stride(-1) != 1:
        raise ValueError(f"{name} must end in a unit-stride dimension of size {D}")
    lead = [s for s in t.shape[:-1]]
    rows = 1
    for s in lead:
        rows *= s
    if rows == 1:
        return 0
    if rows != B:
        raise ValueError(f"{name} has {rows} rows, expected 1 or B={B}")
    # the one non-trivial leading dimension carries the batch stride
    for size, stride in zip(t.shape[:-1], t.stride()[:-1]):
        if size == B:
            return stride
    raise ValueError(f"{name}: cannot find the batch dimension")


def _bsd(x, name="x", dtype=torch.bfloat16):
    _dense(x, name, dtype)
    if x.dim() == 2:
        return 1, x.shape[0], x.shape[1]
    if x.dim() != 3:
        raise ValueError(f"{name} must be [B, S, D] or [S, D]")
    return x.shape[0], x.shape[1], x.shape[2]


def _out_like(out, x, name="out"):
    if out is None:
        return torch.empty_like(x)
    _dense(out, name, x.dtype)
    if out.shape != x.shape:
        raise ValueError(f"{name} shape {tuple(out.shape)} != {tuple(x.shape)}")
    return out


def ln_modulate(x, scale, shift, eps: float = 1e-6, out=None, mean_out=None, rstd_out=None,
                stream=None):
    """LayerNorm (no affine) over the last dim, then R(R(y * R(1 + scale)) + shift)."""
    B, S, D = _bsd(x)
    bs = _mod_rows(scale, B, D, "scale")
    if _mod_rows(shift, B, D, "shift") != bs:
        raise ValueError("scale and shift must share one batch stride")
    out = _out_like(out, x)
    _f32_out(mean_out, B * S, "mean_out", x.device)
    _f32_out(rstd_out, B * S, "rstd_out", x.device)
    _call("ln_modulate", _ptr(x), _ptr(scale), _ptr(shift), _ptr(out), B, S, D, bs, eps,
          _ptr(mean_out), _ptr(rstd_out), _stream(stream))
    return out


def ln_modulate_folded(x, scale, shift, eps: float = 1e-6, out=None, mean_out=None,
                       rstd_out=None, stream=None):
    """Single-rounding tier: R(((x - mean) * rstd) * R(1 + scale) + shift) (not bit-exact
    with the eager chain; same arguments as ln_modulate)."""
    B, S, D = _bsd(x)
    bs = _mod_rows(scale, B, D, "scale")
    if _mod_rows(shift, B, D, "shift") != bs:
        raise ValueError("scale and shift must share one batch stride")
    out = _out_like(out, x)
    _f32_out(mean_out, B * S, "mean_out", x.device)
    _f32_out(rstd_out, B * S, "rstd_out", x.device)
    _call("ln_modulate_folded", _ptr(x), _ptr(scale), _ptr(shift), _ptr(out), B, S, D, bs, eps,
          _ptr(mean_out), _ptr(rstd_out), _stream(stream))
    return out


def backward_workspace_bytes(B: int, S: int, D: int) -> int:
    """Device workspace ln_modulate_backward needs for the token sums."""
    lib = library()
    f = lib.ln_modulate_backward_workspace_bytes
    f.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]
    f.restype = ctypes.c_size_t
    return int(f(B, S, D))


def ln_modulate_backward(x, scale, grad_out, mean, rstd, need_x=True, need_mod=True,
                         grad_x=None, grad_scale=None, grad_shift=None, workspace=None,
                         stream=None):
    """Gradients of ln_modulate (x, scale rows as in the forward; mean, rstd the
    forward's fp32 statistics).  -> (grad_x bf16 like x or None, grad_scale fp32
    [B, D] or None, grad_shift fp32 [B, D] or None).  grad_scale / grad_shift
    are batch-invariant token sums (fixed 32-way trees); the workspace they need
    is allocated here unless one is passed."""
    B, S, D = _bsd(x)
    bs = _mod_rows(scale, B, D, "scale")
    _dense(grad_out, "grad_out")
    if grad_out.shape != x.shape:
        raise ValueError("grad_out must match x")
    _f32_out(mean, B * S, "mean", x.device)
    _f32_out(rstd, B * S, "rstd", x.device)
    if mean is None or rstd is None:
        raise ValueError("mean and rstd (the forward's statistics) are required")
    if need_x:
        grad_x = _out_like(grad_x, x, "grad_x")
    else:
        grad_x = None
    if need_mod:
        if grad_scale is None:
            grad_scale = torch.empty(B, D, dtype=torch.float32, device=x.device)
        if grad_shift is None:
            grad_shift = torch.empty(B, D, dtype=torch.float32, device=x.device)
        _f32_out(grad_scale, B * D, "grad_scale", x.device)
        _f32_out(grad_shift, B * D, "grad_shift", x.device)
        need = backward_workspace_bytes(B, S, D)
        if workspace is None:
            workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=x.device)
        elif workspace.numel() * workspace.element_size() < need:
            raise ValueError(f"workspace holds fewer than the {need} bytes needed")
        wbytes = workspace.numel() * workspace.element_size()
    else:
        grad_scale = grad_shift = None
        workspace, wbytes = None, 0
    _call("ln_modulate_backward", _ptr(x), _ptr(scale), bs, _ptr(grad_out), _ptr(mean),
          _ptr(rstd), B, S, D, _ptr(grad_x), _ptr(grad_scale), _ptr(grad_shift),
          _ptr(workspace), wbytes, _stream(stream))
    return grad_x, grad_scale, grad_shift


def ln_modulate_backward_static(x, scale, grad_out, mean, rstd, grad_x, grad_scale,
                                grad_shift, stream=None):
    """ln_modulate_backward through the entry point that uses the library's
    fixed 8 MiB device scratch instead of a workspace (allocates nothing; every
    output is passed in, None to skip it).  Calls overlapping in time race."""
    B, S, D = _bsd(x)
    bs = _mod_rows(scale, B, D, "scale")
    _dense(grad_out, "grad_out")
    if grad_out.shape != x.shape:
        raise ValueError("grad_out must match x")
    if mean is None or rstd is None:
        raise ValueError("mean and rstd (the forward's statistics) are required")
    _f32_out(mean, B * S, "mean", x.device)
    _f32_out(rstd, B * S, "rstd", x.device)
    if grad_x is not None:
        _out_like(grad_x, x, "grad_x")
    _f32_out(grad_scale, B * D, "grad_scale", x.device)
    _f32_out(grad_shift, B * D, "grad_shift", x.device)
    _call("ln_modulate_backward_static", _ptr(x), _ptr(scale), bs, _ptr(grad_out), _ptr(mean),
          _ptr(rstd), B, S, D, _ptr(grad_x), _ptr(grad_scale), _ptr(grad_shift),
          _stream(stream))
    return grad_x, grad_scale, grad_shift


def rmsnorm_modulate(x, weight, scale, shift, eps: float = 1e-6, out=None, rstd_out=None,
                     stream=None):
    """RMSNorm (weight may be None) over the last dim, then the modulate chain."""
    B, S, D = _bsd(x)
    if weight is not None:
        _dense(weight, "weight")
        if weight.numel() != D:
            raise ValueError("weight must have D elements")
    bs = _mod_rows(scale, B, D, "scale")
    if _mod_rows(shift, B, D, "shift") != bs:
        raise ValueError("scale and shift must share one batch stride")
    out = _out_like(out, x)
    _f32_out(rstd_out, B * S, "rstd_out", x.device)
    _call("rmsnorm_modulate", _ptr(x), _ptr(weight), _ptr(scale), _ptr(shift), _ptr(out), B, S,
          D, bs, eps, _ptr(rstd_out), _stream(stream))
    return out


def gated_rmsnorm_modulate(residual, update, gate, weight, scale, shift, eps: float = 1e-6,
                           res_out=None, out=None, rstd_out=None, stream=None):
    """res = R(residual + R(gate * update)); out = rmsnorm_modulate(res).  -> (res, out)."""
    B, S, D = _bsd(residual, "residual")
    _dense(update, "update")
    if update.shape != residual.shape:
        raise ValueError("update must match residual")
    gs = _mod_rows(gate, B, D, "gate")
    if weight is not None:
        _dense(weight, "weight")
        if weight.numel() != D:
            raise ValueError("weight must have D elements")
    bs = _mod_rows(scale, B, D, "scale")
    if _mod_rows(shift, B, D, "shift") != bs:
        raise ValueError("scale and shift must share one batch stride")
    res_out = _out_like(res_out, residual, "res_out")
    out = _out_like(out, residual)
    _f32_out(rstd_out, B * S, "rstd_out", residual.device)
    _call("gated_rmsnorm_modulate", _ptr(residual), _ptr(update), _ptr(gate), gs, _ptr(weight),
          _ptr(scale), _ptr(shift), bs, _ptr(res_out), _ptr(out), B, S, D, eps, _ptr(rstd_out),
          _stream(stream))
    return res_out, out


def _token_view(t, name):
    """[..., heads, head_dim] view with dense heads and one uniform stride
    over the leading dims -> (tokens, heads, token_stride in elements)."""
    _bf16(t, name)
    if t.dim() < 2 or t.stride(-1) != 1 or (t.dim() >= 2 and t.shape[-2] > 1 and
                                             t.stride(-2) != t.shape[-1]):
        raise ValueError(f"{name}: heads must be dense [..., heads, head_dim]")
    heads, hd = (t.shape[-2], t.shape[-1]) if t.dim() >= 2 else (1, t.shape[-1])
    lead = list(zip(t.shape[:-2], t.stride()[:-2]))
    tokens, ts = 1, heads * hd
    for size, stride in reversed(lead):
        if size == 1:
            continue
        if tokens == 1:
            ts = stride
        elif stride != ts * tokens:
            raise ValueError(f"{name}: leading dims do not collapse to one token stride")
        tokens *= size
    return tokens, heads, ts


def qk_layernorm(q, k, wq, bq, wk, bk, eps: float = 1e-5, q_out=None, k_out=None,
                 mean_out=None, rstd_out=None, stream=None):
    """Per-head LayerNorm(head_dim) with affine on q and k in one launch. -> (q_out, k_out).
    q / k may be token-strided views (e.g. slices of a fused QKV projection)
    whose heads are dense; head_dim 64, 96 or 128."""
    hd = q.shape[-1]
    if k.shape[-1] != hd:
        raise ValueError("q and k must share head_dim")
    for t, n in ((wq, "wq"), (bq, "bq"), (wk, "wk"), (bk, "bk")):
        _dense(t, n)
        if t.numel() != hd:
            raise ValueError(f"{n} must have head_dim elements")
    dense = all(t.is_contiguous() for t in (q, k)) and all(
        t is None or t.is_contiguous() for t in (q_out, k_out))
    if dense:
        _dense(q, "q")
        _dense(k, "k")
        rq, rk = q.numel() // hd, k.numel() // hd
        q_out = _out_like(q_out, q, "q_out")
        k_out = _out_like(k_out, k, "k_out")
        _f32_out(mean_out, rq + rk, "mean_out", q.device)
        _f32_out(rstd_out, rq + rk, "rstd_out", q.device)
        _call("qk_layernorm", _ptr(q), _ptr(k), _ptr(wq), _ptr(bq), _ptr(wk), _ptr(bk),
              _ptr(q_out), _ptr(k_out), rq, rk, hd, eps, _ptr(mean_out), _ptr(rstd_out),
              _stream(stream))
        return q_out, k_out
    tq, hq, qts = _token_view(q, "q")
    tk, hk, kts = _token_view(k, "k")
    if tq != tk:
        raise ValueError("q and k must have the same number of tokens")
    if q_out is None:
        q_out = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    if k_out is None:
        k_out = torch.empty(k.shape, dtype=k.dtype, device=k.device)
    if q_out.shape != q.shape or k_out.shape != k.shape:
        raise ValueError("q_out / k_out must match q / k")
    to, _, qots = _token_view(q_out, "q_out")
    _, _, kots = _token_view(k_out, "k_out")
    rows = tq * (hq + hk)
    _f32_out(mean_out, rows, "mean_out", q.device)
    _f32_out(rstd_out, rows, "rstd_out", q.device)
    _call("qk_layernorm_strided", _ptr(q), _ptr(k), _ptr(wq), _ptr(bq), _ptr(wk), _ptr(bk),
          _ptr(q_out), _ptr(k_out), tq, hq, hk, hd, qts, kts, qots, kots, eps, _ptr(mean_out),
          _ptr(rstd_out), _stream(stream))
    return q_out, k_out


def _pixels_c(x):
    """Dense channels-last activation -> (pixels, C).  Accepts [..., C] contiguous
    tensors or channels_last(_3d) N C (T) H W tensors."""
    if x.dim() in (4, 5) and not x.is_contiguous():
        fmt = torch.channels_last if x.dim() == 4 else torch.channels_last_3d
        if not x.is_contiguous(memory_format=fmt):
            raise ValueError("x must be dense channels-last")
        return x.numel() // x.shape[1], x.shape[1]
    if not x.is_contiguous():
        raise ValueError("x must be dense channels-last")
    if x.dim() in (4, 5):
        raise ValueError("a 4-D/5-D x must be in channels_last(_3d) memory format")
    return x.numel() // x.shape[-1], x.shape[-1]


def rmsnorm_silu_cl(x, bias, gamma, eps: float = 1e-6, out=None, rstd_out=None, stream=None):
    """SiLU(RMSNorm_C(x + bias) * gamma) on a channels-last activation."""
    _bf16(x, "x")
    pixels, C = _pixels_c(x)
    if bias is not None:
        if bias.dtype not in (torch.float32, torch.bfloat16) or not bias.is_cuda or \
                bias.numel() != C or not bias.is_contiguous():
            raise ValueError("bias must be a contiguous fp32/bf16 CUDA tensor of C elements")
    _dense(gamma, "gamma")
    if gamma.numel() != C:
        raise ValueError("gamma must have C elements")
    if out is None:
        out = torch.empty_like(x)  # keeps the channels-last strides
    elif out.shape != x.shape or out.stride() != x.stride() or out.dtype != torch.bfloat16:
        raise ValueError("out must match x's shape, strides and dtype")
    _f32_out(rstd_out, pixels, "rstd_out", x.device)
    is32 = 1 if (bias is not None and bias.dtype == torch.float32) else 0
    _call("rmsnorm_silu_cl", _ptr(x), _ptr(bias), is32, _ptr(gamma), _ptr(out), pixels, C, eps,
          _ptr(rstd_out), _stream(stream))
    return out


def modulate_scale_shift(y, scale, shift, out=None, stream=None):
    """R(R(y * R(1 + scale)) + shift) over y [B, S, D], in y's storage type
    (bfloat16 or float16; scale and shift must match it)."""
    if isinstance(y, torch.Tensor) and y.dtype == torch.float16:
        dt, entry = torch.float16, "modulate_scale_shift_f16"
    else:
        dt, entry = torch.bfloat16, "modulate_scale_shift"
    B, S, D = _bsd(y, "y", dt)
    bs = _mod_rows(scale, B, D, "scale", dt)
    if _mod_rows(shift, B, D, "shift", dt) != bs:
        raise ValueError("scale and shift must share one batch stride")
    out = _out_like(out, y)
    _call(entry, _ptr(y), _ptr(scale), _ptr(shift), _ptr(out), B, S, D, bs, _stream(stream))
    return out


def residual_gate_add(residual, gate, update, out=None, stream=None):
    """R(residual + R(gate * update)) over [B, S, D]."""
    B, S, D = _bsd(residual, "residual")
    _dense(update, "update")
    if update.shape != residual.shape:
        raise ValueError("update must match residual")
    gs = _mod_rows(gate, B, D, "gate")
    out = _out_like(out, residual)
    _call("residual_gate_add", _ptr(residual), _ptr(gate), _ptr(update), gs, _ptr(out), B, S, D,
          _stream(stream))
    return out


def conv_bias_epilogue(x, bias, h=None, out=None, stream=None):
    """R(x + R(bias)) (and + h) on a channels-last activation."""
    _bf16(x, "x")
    pixels, C = _pixels_c(x)
    if bias.dtype not in (torch.float32, torch.bfloat16) or not bias.is_cuda or \
            bias.numel() != C or not bias.is_contiguous():
        raise ValueError("bias must be a contiguous fp32/bf16 CUDA tensor of C elements")
    if h is not None:
        _bf16(h, "h")
        if h.shape != x.shape or h.stride() != x.stride():
            raise ValueError("h must match x's shape and strides")
    if out is None:
        out = torch.empty_like(x)
    is32 = 1 if bias.dtype == torch.float32 else 0
    _call("conv_bias_epilogue", _ptr(x), _ptr(bias), is32, _ptr(h), _ptr(out), pixels, C,
          _stream(stream))
    return out


def device_status(clear: bool = False) -> int:
    """Error bits recorded by kernels on the current device (0 = none).
    Synchronous.  Bit 0: an asynchronous copy timed out (output invalid)."""
    bits = ctypes.c_uint(0)
    _call("rmsmod_device_status", ctypes.byref(bits), 1 if clear else 0)
    return int(bits.value)


def selftest_wait_timeout(limit_ns: int = 1_000_000, stream=None) -> None:
    """Launch the library's bounded-wait self-test: one warp waits `limit_ns`
    on a barrier nothing completes, then sets bit 0 of the device error word
    (read it with device_status after synchronising)."""
    _call("rmsmod_selftest_wait_timeout", int(limit_ns), _stream(stream))


def supported(op: int, d_or_c: int, *tensors) -> bool:
    """The library's predicate: never raises, never touches the GPU."""
    ptrs = (ctypes.c_void_p * max(1, len(tensors)))(
        *[t.data_ptr() if t is not None else None for t in tensors])
    return bool(library().rmsmod_supported(int(op), int(d_or_c), ptrs, len(tensors)))
