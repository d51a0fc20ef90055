// The bounded-wait self-test (selftest.cu).
#pragma once

#include <cuda_runtime.h>

namespace rmsmod {

// One warp waiting `limit_ns` on an mbarrier nothing completes, then setting
// the timeout bit of this unit's device error word.
cudaError_t launch_selftest_wait(unsigned long long limit_ns, cudaStream_t stream);

// Reads the self-test unit's device error word, optionally clearing it;
// synchronous.
cudaError_t selftest_error(unsigned* bits, bool clear);

}  // namespace rmsmod
