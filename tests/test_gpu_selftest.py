"""The bounded-wait error path, made to run out on purpose without a fault:
rmsmod_selftest_wait_timeout launches one warp that waits on an mbarrier
nothing completes, with a short limit, then records the timeout in the
device error word.  The host reads the bit, clears it, and the context is
still usable for a normal launch."""
import numpy as np
import pytest
import torch

import workloads as W
from _gpu import dev, host

pytestmark = pytest.mark.gpu


def test_wait_runs_out_and_is_reported(oracle_mod):
    import rmsnorm_modulate_gb300 as rm

    assert rm.device_status(clear=True) == 0
    rm.selftest_wait_timeout(2_000_000)  # 2 ms
    torch.cuda.synchronize()
    assert rm.device_status() == 1       # RMSMOD_DEVICE_ERR_COPY_TIMEOUT
    assert rm.device_status(clear=True) == 1
    assert rm.device_status() == 0

    # the context still runs kernels, and they are right
    inp = W.ln_modulate_inputs(1, 40, 1024, seed=31)
    out, _, _ = oracle_mod.ln_modulate(inp["x"], inp["scale"], inp["shift"])
    got = rm.ln_modulate(dev(inp["x"]), dev(inp["scale"]), dev(inp["shift"]))
    torch.cuda.synchronize()
    assert np.array_equal(host(got), out)
    assert rm.device_status(clear=True) == 0


def test_limit_out_of_range_launches_nothing():
    import rmsnorm_modulate_gb300 as rm

    lib = rm.library()
    s = __import__("ctypes").c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.rmsmod_selftest_wait_timeout(0, s) == -2
    assert lib.rmsmod_selftest_wait_timeout(100_000_001, s) == -2
    torch.cuda.synchronize()
    assert rm.device_status(clear=True) == 0
