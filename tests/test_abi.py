"""The C ABI without a GPU: the library loads, exports every entry point the
public header declares, and rejects bad arguments on the host (status codes,
nothing launched).  No call here passes a complete set of valid arguments,
so nothing can reach a kernel launch."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rmsmod.h")

OK, ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_STRIDE, ERR_UNSUPPORTED, ERR_CUDA, ERR_DEVICE = \
    0, -1, -2, -3, -4, -5, -6, -7


@pytest.fixture(scope="module")
def lib():
    from rmsnorm_modulate_gb300 import _build

    _build.build()
    import rmsnorm_modulate_gb300 as rm

    return rm.library()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?(?:int|size_t|char\s*\*|const char\s*\*)\s*\*?\s*"
                                 r"([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = header_functions()
    for n in ("ln_modulate", "ln_modulate_folded", "ln_modulate_backward",
              "ln_modulate_backward_workspace_bytes", "modulate_scale_shift_f16", "rmsnorm_modulate", "gated_rmsnorm_modulate", "qk_layernorm",
              "rmsnorm_silu_cl", "modulate_scale_shift", "residual_gate_add",
              "conv_bias_epilogue", "rmsmod_supported", "rmsmod_status_string",
              "rmsmod_version"):
        assert n in names, n


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), f"librmsmod.so does not export {name}"


def test_exports_are_plain_c_symbols(lib):
    out = os.popen(f"nm -D --defined-only {lib._name}").read()
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    for name in header_functions():
        assert name in exported
    # nothing C++-mangled leaks into the dynamic symbol table
    assert not [s for s in exported if s.startswith("_Z")]


def test_status_strings(lib):
    for st in (OK, ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_STRIDE, ERR_UNSUPPORTED, ERR_CUDA,
               ERR_DEVICE, 12345):
        s = lib.rmsmod_status_string(st)
        assert isinstance(s, bytes) and s
    assert lib.rmsmod_version() == 10000


P = ctypes.c_void_p
A = 0x100000  # 16-byte aligned fake addresses, never dereferenced on the host
MIS = 0x100008


def p(v):
    return P(v)


def test_backward_validation_and_workspace_size(lib):
    ws = lib.ln_modulate_backward_workspace_bytes
    ws.argtypes = [ctypes.c_int64] * 3
    ws.restype = ctypes.c_size_t
    assert ws(1, 4608, 3072) == 1 * 144 * 2 * 3072 * 4
    assert ws(2, 33, 64) == 2 * 2 * 2 * 64 * 4
    assert ws(0, 4, 64) == 0 and ws(1, 0, 64) == 0
    f = lib.ln_modulate_backward
    f.argtypes = [P, P, ctypes.c_int64, P, P, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                  P, P, P, P, ctypes.c_size_t, P]
    s = P(0)
    X, SC, G, M, R = A, A + 4096, A + (1 << 24), A + (2 << 24), A + (3 << 24)
    GX, GS, GH, W = A + (4 << 24), A + (5 << 24), A + (6 << 24), A + (7 << 24)
    args = lambda **k: [p(k.get("x", X)), p(k.get("sc", SC)), k.get("bs", 0), p(k.get("g", G)),
                        p(k.get("m", M)), p(k.get("r", R)), k.get("B", 1), k.get("S", 64),
                        k.get("D", 64), p(k.get("gx", GX)), p(k.get("gs", GS)),
                        p(k.get("gh", GH)), p(k.get("w", W)), k.get("wb", 1 << 20), s]
    assert f(*args(D=12)) == ERR_SHAPE
    assert f(*args(bs=12)) == ERR_STRIDE
    assert f(*args(g=0)) == ERR_NULL
    assert f(*args(w=0)) == ERR_NULL                       # token sums need a workspace
    assert f(*args(x=MIS)) == ERR_ALIGN
    assert f(*args(w=A + (7 << 24) + 16)) == ERR_ALIGN     # workspace 256-byte aligned
    assert f(*args(wb=16)) == ERR_SHAPE                    # workspace too small
    assert f(*args(gx=X)) == ERR_UNSUPPORTED               # grad_x may not alias x
    assert f(*args(w=GX)) == ERR_UNSUPPORTED               # workspace overlaps grad_x
    assert f(*args(gx=0, gs=0, gh=0)) == OK                # nothing requested: no work
    # outputs written while other CTAs still read scale, mean and rstd: any
    # overlap with those inputs is refused, not raced on (the scale rows sit
    # apart from x here, so each case overlaps exactly one input)
    SC2 = A + (8 << 24)
    assert f(*args(sc=SC2, w=SC2)) == ERR_UNSUPPORTED      # workspace over the scale row
    assert f(*args(w=M)) == ERR_UNSUPPORTED                # workspace over mean
    assert f(*args(w=R - 256)) == ERR_UNSUPPORTED          # workspace reaching into rstd
    assert f(*args(sc=SC2, gs=SC2)) == ERR_UNSUPPORTED     # grad_scale over the scale row
    assert f(*args(sc=SC2, gh=SC2 + 64)) == ERR_UNSUPPORTED  # grad_shift inside the scale row
    assert f(*args(gh=M + 64)) == ERR_UNSUPPORTED          # grad_shift inside mean
    assert f(*args(gs=R)) == ERR_UNSUPPORTED               # grad_scale over rstd
    assert f(*args(gx=M)) == ERR_UNSUPPORTED               # grad_x over mean
    assert f(*args(gx=R - 16)) == ERR_UNSUPPORTED          # grad_x reaching into rstd
    # per-batch scale rows: the span reaches the last batch's row
    assert f(*args(B=2, bs=4096, sc=SC2, gs=SC2 + 2 * 4096)) == ERR_UNSUPPORTED


def test_ln_modulate_folded_validation(lib):
    f = lib.ln_modulate_folded
    f.argtypes = [P, P, P, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                  ctypes.c_float, P, P, P]
    s = P(0)
    assert f(p(A), p(A + 4096), p(A + 8192), p(A + (1 << 24)), 1, 4, 12, 0, 1e-6, None, None,
             s) == ERR_SHAPE                                # D % 8
    assert f(None, p(A + 4096), p(A + 8192), p(A + (1 << 24)), 1, 4, 16, 0, 1e-6, None, None,
             s) == ERR_NULL
    assert f(p(MIS), p(A + 4096), p(A + 8192), p(A + (1 << 24)), 1, 4, 16, 0, 1e-6, None,
             None, s) == ERR_ALIGN
    assert f(p(A), p(A + 4096), p(A + 8192), p(A + (1 << 24)), 1, 4, 16, 12, 1e-6, None, None,
             s) == ERR_STRIDE
    # a partially overlapping output
    assert f(p(A), p(A + 4096), p(A + 8192), p(A + 16), 1, 4, 16, 0, 1e-6, None, None,
             s) == ERR_UNSUPPORTED
    assert lib.rmsmod_supported(6, 3072, None, 0) == 1


def test_ln_modulate_validation(lib):
    f = lib.ln_modulate
    s = P(0)
    # sizes
    assert f(p(A), p(A + 4096), p(A + 8192), p(A + 1 << 24), 1, 4, 12, 0, 1e-6, None, None, s) \
        == ERR_SHAPE                                       # D % 8
    assert f(p(A), p(A), p(A), p(A), 1, 4, 0, 0, 1e-6, None, None, s) == ERR_SHAPE
    assert f(p(A), p(A), p(A), p(A), -1, 4, 8, 0, 1e-6, None, None, s) == ERR_SHAPE
    assert f(p(A), p(A), p(A), p(A), 1, 4, 16392, 0, 1e-6, None, None, s) == ERR_SHAPE
    assert f(p(A), p(A), p(A), p(A), 1 << 40, 1 << 40, 8, 0, 1e-6, None, None, s) == ERR_SHAPE
    # strides
    assert f(p(A), p(A), p(A), p(A), 2, 4, 8, 4, 1e-6, None, None, s) == ERR_STRIDE
    assert f(p(A), p(A), p(A), p(A), 2, 4, 8, -8, 1e-6, None, None, s) == ERR_STRIDE
    # zero rows: OK, nothing launched even with NULL pointers
    assert f(None, None, None, None, 0, 4, 8, 0, 1e-6, None, None, s) == OK
    assert f(None, None, None, None, 3, 0, 8, 0, 1e-6, None, None, s) == OK
    # NULLs
    assert f(None, p(A), p(A), p(A), 1, 4, 8, 0, 1e-6, None, None, s) == ERR_NULL
    assert f(p(A), None, p(A), p(A), 1, 4, 8, 0, 1e-6, None, None, s) == ERR_NULL
    assert f(p(A), p(A), p(A), None, 1, 4, 8, 0, 1e-6, None, None, s) == ERR_NULL
    # alignment
    assert f(p(MIS), p(A), p(A), p(A), 1, 4, 8, 0, 1e-6, None, None, s) == ERR_ALIGN
    assert f(p(A), p(A), p(MIS), p(A), 1, 4, 8, 0, 1e-6, None, None, s) == ERR_ALIGN
    assert f(p(A), p(A), p(A), p(A), 1, 4, 8, 0, 1e-6, p(A + 2), None, s) == ERR_ALIGN
    # partial overlap of out and x (exact aliasing is allowed)
    assert f(p(A), p(A + 1 << 20), p(A + 1 << 21), p(A + 16), 1, 4, 8, 0, 1e-6, None, None, s) \
        == ERR_UNSUPPORTED
    # out overlapping scale
    assert f(p(A), p(A + 4096 + 16), p(A + 1 << 21), p(A + 4096), 1, 4, 8, 0, 1e-6, None, None,
             s) == ERR_UNSUPPORTED


def test_rms_and_gated_validation(lib):
    s = P(0)
    r = lib.rmsnorm_modulate
    assert r(p(A), p(MIS), p(A), p(A), p(A), 1, 2, 8, 0, 1e-6, None, s) == ERR_ALIGN
    assert r(p(A), None, None, p(A), p(A), 1, 2, 8, 0, 1e-6, None, s) == ERR_NULL
    assert r(p(A), None, p(A), p(A), p(A), 1, 2, 7, 0, 1e-6, None, s) == ERR_SHAPE
    g = lib.gated_rmsnorm_modulate
    args = [p(A), p(A + 1 << 20), p(A + 1 << 21), 0, None, p(A + 1 << 22), p(A + 1 << 23), 0,
            p(A + 1 << 24), p(A + 1 << 25), 1, 2, 8, 1e-6, None, s]
    bad = list(args)
    bad[3] = 3
    assert g(*bad) == ERR_STRIDE
    bad = list(args)
    bad[2] = None
    assert g(*bad) == ERR_NULL
    bad = list(args)
    bad[9] = bad[0]  # out aliasing residual is not allowed (only res_out may)
    assert g(*bad) == ERR_UNSUPPORTED
    bad = list(args)
    bad[9] = bad[8]  # out == res_out
    assert g(*bad) == ERR_UNSUPPORTED


def test_qk_strided_validation(lib):
    f = lib.qk_layernorm_strided
    I = ctypes.c_int64
    f.argtypes = [P] * 8 + [I] * 8 + [ctypes.c_float, P, P, P]
    s = P(0)
    T, H, hd = 16, 4, 128
    qkv = A                     # [T, 3, H, hd] bf16: token stride 3 * H * hd
    ts = 3 * H * hd
    q, k = qkv, qkv + 2 * H * hd
    w = A + (1 << 26)
    args = lambda **kw: [p(kw.get("q", q)), p(kw.get("k", k)), p(w), p(w + 256), p(w + 512),
                         p(w + 768), p(kw.get("qo", A + (1 << 27))),
                         p(kw.get("ko", A + (1 << 28))), kw.get("T", T), kw.get("hq", H),
                         kw.get("hk", H), kw.get("hd", hd), kw.get("qts", ts), kw.get("kts", ts),
                         kw.get("qots", H * hd), kw.get("kots", H * hd), 1e-5, None, None, s]
    assert f(*args(hd=80)) == ERR_SHAPE
    assert f(*args(qts=H * hd - 8)) == ERR_STRIDE       # shorter than a token's heads
    assert f(*args(kts=ts + 4)) == ERR_STRIDE           # not a multiple of 8
    # q_out = the k slice of the same buffer while k is read: shared bytes
    assert f(*args(qo=k, qots=ts)) == ERR_UNSUPPORTED
    # a dense q_out that overlaps the strided q span partially
    assert f(*args(qo=q + 2 * hd, qots=H * hd)) == ERR_UNSUPPORTED
    assert f(*args(T=0)) == OK                           # nothing to do


def test_qk_validation(lib):
    s = P(0)
    f = lib.qk_layernorm
    base = [p(A), p(A + 1 << 20), p(A + 1 << 21), p(A + 1 << 22), p(A + 1 << 23), p(A + 1 << 24),
            p(A + 1 << 25), p(A + 1 << 26), 4, 4, 128, 1e-5, None, None, s]
    for hd in (32, 80, 100, 256):  # head_dim 64, 96, 128 only
        bad = list(base)
        bad[10] = hd
        assert f(*bad) == ERR_SHAPE
    bad = list(base)
    bad[8] = -1
    assert f(*bad) == ERR_SHAPE
    bad = list(base)
    bad[2] = None
    assert f(*bad) == ERR_NULL
    bad = list(base)
    bad[6] = p(A + 16)  # q_out partially overlapping q
    assert f(*bad) == ERR_UNSUPPORTED
    bad = list(base)
    bad[8], bad[9] = 0, 0
    assert f(*bad) == OK


def test_wan_and_elementwise_validation(lib):
    s = P(0)
    w = lib.rmsnorm_silu_cl
    assert w(p(A), None, 1, p(A + 1 << 20), p(A + 1 << 21), 10, 4, 1e-6, None, s) == ERR_SHAPE
    assert w(p(A), None, 1, p(A + 1 << 20), p(A + 1 << 21), 10, 1032, 1e-6, None, s) == ERR_SHAPE
    assert w(p(A), p(A + 8), 1, p(A + 1 << 20), p(A + 1 << 21), 10, 96, 1e-6, None, s) == ERR_ALIGN
    assert w(p(A), None, 1, None, p(A + 1 << 21), 10, 96, 1e-6, None, s) == ERR_NULL
    assert w(None, None, 1, None, None, 0, 96, 1e-6, None, s) == OK
    m = lib.modulate_scale_shift
    assert m(p(A), p(A), p(A), p(A), 1, 2, 10, 0, s) == ERR_SHAPE
    assert m(p(A), p(A), p(A), p(A), 2, 2, 8, 12, s) == ERR_STRIDE
    assert m(p(A), None, p(A), p(A), 2, 2, 8, 0, s) == ERR_NULL
    ga = lib.residual_gate_add
    assert ga(p(A), p(A), p(MIS), 0, p(A), 1, 2, 8, s) == ERR_ALIGN
    cb = lib.conv_bias_epilogue
    assert cb(p(A), None, 1, None, p(A), 4, 96, s) == ERR_NULL
    assert cb(p(A), p(A + 1 << 20), 1, p(MIS), p(A + 1 << 21), 4, 96, s) == ERR_ALIGN


def test_supported_predicate(lib):
    arr = (P * 3)(A, A + 32, None)
    assert lib.rmsmod_supported(1, 3072, arr, 3) == 1
    assert lib.rmsmod_supported(1, 3073, arr, 3) == 0
    assert lib.rmsmod_supported(1, 16392, arr, 3) == 0
    assert lib.rmsmod_supported(4, 128, arr, 3) == 1
    assert lib.rmsmod_supported(4, 64, arr, 3) == 1
    assert lib.rmsmod_supported(4, 96, arr, 3) == 1
    assert lib.rmsmod_supported(4, 80, arr, 3) == 0
    assert lib.rmsmod_supported(5, 96, arr, 3) == 1
    assert lib.rmsmod_supported(5, 2048, arr, 3) == 0
    assert lib.rmsmod_supported(99, 96, arr, 3) == 0
    mis = (P * 2)(A, MIS)
    assert lib.rmsmod_supported(2, 4096, mis, 2) == 0
    assert lib.rmsmod_supported(2, 4096, None, 0) == 1
    assert lib.rmsmod_supported(2, 4096, None, 2) == 0


def test_valid_call_without_gpu_reports_device_error(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: a valid call would launch")
    st = lib.ln_modulate(p(A), p(A + 1 << 20), p(A + 1 << 21), p(A + 1 << 22), 1, 4, 8, 0,
                         1e-6, None, None, P(0))
    assert st == ERR_DEVICE


def test_binding_has_no_cpu_fallback():
    torch = pytest.importorskip("torch")
    import rmsnorm_modulate_gb300 as rm

    x = torch.zeros(1, 4, 8, dtype=torch.bfloat16)
    s = torch.zeros(8, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        rm.ln_modulate(x, s, s)
