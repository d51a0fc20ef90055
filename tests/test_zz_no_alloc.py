"""ln_modulate_backward_static: the backward entry point for callers that
cannot give the library device memory (a framework whose allocator owns the
device, a hot path that must not call cudaMalloc), which uses the library's
fixed device scratch instead of a caller workspace.  Three calls in a row on
different inputs, largest first so that later calls meet stale scratch, must
each give bit-identical results to the workspace entry point; a call changes
neither torch's allocations nor the device's free memory; sizes beyond the
fixed scratch are refused.  Collected last on purpose, and independent of
what ran before it."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from _gpu import dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rm():
    import rmsnorm_modulate_gb300 as rm

    yield rm
    assert rm.device_status(clear=True) == 0


def inputs(rm, B, S, D, seed):
    inp = W.ln_modulate_inputs(B, S, D, seed=seed, per_batch_mod=True)
    g = torch.Generator().manual_seed(seed + 1)
    x, sc, sh = dev(inp["x"]), dev(inp["scale"]), dev(inp["shift"])
    go = dev(W.normal_bf16(g, (B, S, D), 0.5))
    mean = torch.empty(B * S, dtype=torch.float32, device="cuda")
    rstd = torch.empty_like(mean)
    rm.ln_modulate(x, sc, sh, mean_out=mean, rstd_out=rstd)
    return x, sc, go, mean, rstd


def outputs(B, S, D):
    return (torch.empty(B, S, D, dtype=torch.bfloat16, device="cuda"),
            torch.empty(B, D, dtype=torch.float32, device="cuda"),
            torch.empty(B, D, dtype=torch.float32, device="cuda"))


def test_two_calls_in_a_row_match_the_workspace_entry_point(rm):
    # the largest case first, so the later calls (other B, S not a multiple
    # of 32, other D; the one-pass kernel, then the separate token kernels at
    # D = 256) find stale values of the first in the scratch: nothing they
    # read may depend on them
    cases = [(2, 4608, 3072, 32), (3, 1100, 1024, 31), (1, 700, 256, 30)]
    data = [inputs(rm, B, S, D, seed) for B, S, D, seed in cases]
    outs = [outputs(B, S, D) for B, S, D, _ in cases]
    # back to back on one stream, the second reusing the scratch the first wrote
    for (x, sc, go, m, r), (gx, gsc, gsh) in zip(data, outs):
        rm.ln_modulate_backward_static(x, sc, go, m, r, gx, gsc, gsh)
    torch.cuda.synchronize()
    for (x, sc, go, m, r), (gx, gsc, gsh) in zip(data, outs):
        rx, rsc, rsh = rm.ln_modulate_backward(x, sc, go, m, r)
        torch.cuda.synchronize()
        assert torch.equal(gx.view(torch.int16), rx.view(torch.int16))
        assert torch.equal(gsc.view(torch.int32), rsc.view(torch.int32))
        assert torch.equal(gsh.view(torch.int32), rsh.view(torch.int32))


def test_a_call_allocates_no_device_memory(rm):
    B, S, D = 1, 333, 3072
    x, sc, go, m, r = inputs(rm, B, S, D, 7)
    gx, gsc, gsh = outputs(B, S, D)
    rm.ln_modulate_backward_static(x, sc, go, m, r, gx, gsc, gsh)   # set-up call
    torch.cuda.synchronize()
    torch_before = torch.cuda.memory_allocated()
    free_before, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        rm.ln_modulate_backward_static(x, sc, go, m, r, gx, gsc, gsh)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == torch_before
    assert free_after == free_before
    rx, rsc, rsh = rm.ln_modulate_backward(x, sc, go, m, r)
    torch.cuda.synchronize()
    assert torch.equal(gx.view(torch.int16), rx.view(torch.int16))
    assert torch.equal(gsc.view(torch.int32), rsc.view(torch.int32))


def test_sizes_beyond_the_fixed_scratch_are_refused(rm):
    lib = rm.library()
    need = rm.backward_workspace_bytes(4, 8192, 4096)
    assert need > (8 << 20)
    P = ctypes.c_void_p
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")   # never read: refused first
    f32 = torch.zeros(16, dtype=torch.float32, device="cuda")
    st = lib.ln_modulate_backward_static(P(x.data_ptr()), P(x.data_ptr()), 0, P(x.data_ptr()),
                                         P(f32.data_ptr()), P(f32.data_ptr()), 4, 8192, 4096,
                                         None, P(f32.data_ptr()), None,
                                         P(torch.cuda.current_stream().cuda_stream))
    assert st == -2   # RMSMOD_ERR_SHAPE, nothing launched
    # grad_x alone needs no scratch: only the token sums are limited
    B, S, D = 1, 40, 3072
    xx, sc, go, m, r = inputs(rm, B, S, D, 33)
    gx, _, _ = outputs(B, S, D)
    rm.ln_modulate_backward_static(xx, sc, go, m, r, gx, None, None)
    rx, _, _ = rm.ln_modulate_backward(xx, sc, go, m, r, need_mod=False)
    torch.cuda.synchronize()
    assert torch.equal(gx.view(torch.int16), rx.view(torch.int16))
