// Standalone bit-exact elementwise chains on sm_103a: the fused kernels'
// modulate epilogue, gated-residual prologue and conv-bias fold, exported on
// their own.
//   modulate_scale_shift (bf16 and fp16): sglang #34004 FLUX.1, §Modifications
//                         commit 2 and §Accuracy Tests
//   residual_gate_add:    sglang #33854 ERNIE-Image residual variant; #34008 ff gate
//   conv_bias_epilogue:   sglang #38650 Wan VAE, §New kernel, lossless
//
// Flat grid-stride over 16-byte vectors, four vectors in flight per thread;
// row and batch indices come from multiply-shift division.
#include "device_common.cuh"
#include "launch.h"

namespace rmsmod {

namespace {

constexpr int kThreads = 256;
constexpr int kIlp = 4;

template <int OP>
__device__ __forceinline__ uint4 apply(const EwArgs& a, uint32_t i, const FastDiv& fd_row,
                                       const FastDiv& fd_batch, uint4 av)
{
    const uint32_t row = fd_row.div(i);
    const uint32_t c = i - row * fd_row.d;
    uint4 o;
    if (OP == kEwModulate) {
        const uint32_t b = fd_batch.div(row);
        const int64_t off = static_cast<int64_t>(b) * a.bstride + c;
        uint4 s = ld_cached(static_cast<const uint4*>(a.b) + off);
        uint4 h = ld_cached(static_cast<const uint4*>(a.c) + off);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            word(o, k) = bf2_add(bf2_mul(word(av, k), bf2_add(word(s, k), kBf2One)), word(h, k));
    } else if (OP == kEwModulateF16) {
        const uint32_t b = fd_batch.div(row);
        const int64_t off = static_cast<int64_t>(b) * a.bstride + c;
        uint4 s = ld_cached(static_cast<const uint4*>(a.b) + off);
        uint4 h = ld_cached(static_cast<const uint4*>(a.c) + off);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            word(o, k) = h2_add(h2_mul(word(av, k), h2_add(word(s, k), kH2One)), word(h, k));
    } else if (OP == kEwGateAdd) {
        const uint32_t b = fd_batch.div(row);
        uint4 g = ld_cached(static_cast<const uint4*>(a.b) + static_cast<int64_t>(b) * a.bstride + c);
        uint4 u = ld_stream(static_cast<const uint4*>(a.c) + i);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            word(o, k) = bf2_add(word(av, k), bf2_mul(word(g, k), word(u, k)));
    } else {
        uint4 bb;
        if (a.bias_is_fp32) {
            const float4* bf = static_cast<const float4*>(a.b) + 2 * c;
            const float4 lo = ld_cached_f4(bf), hi = ld_cached_f4(bf + 1);
            bb = make_uint4(pack_bf2(lo.x, lo.y), pack_bf2(lo.z, lo.w), pack_bf2(hi.x, hi.y),
                            pack_bf2(hi.z, hi.w));
        } else {
            bb = ld_cached(static_cast<const uint4*>(a.b) + c);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
            word(o, k) = bf2_add(word(av, k), word(bb, k));
        if (a.c) {
            uint4 h = ld_stream(static_cast<const uint4*>(a.c) + i);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                word(o, k) = bf2_add(word(o, k), word(h, k));
        }
    }
    return o;
}

template <int OP>
__global__ void __launch_bounds__(kThreads)
    ew_kernel(const EwArgs a, uint32_t total, FastDiv fd_row, FastDiv fd_batch)
{
    grid_dependency_sync();
    const uint4* __restrict__ src = static_cast<const uint4*>(a.a);
    uint4* __restrict__ dst = static_cast<uint4*>(a.out);
    const uint32_t stride = gridDim.x * kThreads;
    for (uint32_t i0 = blockIdx.x * kThreads + threadIdx.x; i0 < total; i0 += kIlp * stride) {
        uint4 v[kIlp];
#pragma unroll
        for (int k = 0; k < kIlp; ++k) {
            const uint32_t i = i0 + k * stride;
            if (i < total)
                v[k] = ld_stream(src + i);
        }
#pragma unroll
        for (int k = 0; k < kIlp; ++k) {
            const uint32_t i = i0 + k * stride;
            if (i < total)
                st_stream(dst + i, apply<OP>(a, i, fd_row, fd_batch, v[k]));
        }
    }
}

template <int OP>
cudaError_t launch(const EwArgs& a, const DeviceInfo& dev, cudaStream_t stream)
{
    static PerDeviceInt blocks_per_sm;
    int bps = 0;
    {
        const cudaError_t e0 = blocks_per_sm.get(dev.device, bps, [&](int& v) -> cudaError_t {
            int nb = 0;
            cudaError_t e =
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, ew_kernel<OP>, kThreads, 0);
            if (e != cudaSuccess)
                return e;
            v = nb > 0 ? nb : 1;
            return cudaSuccess;
        });
        if (e0 != cudaSuccess)
            return e0;
    }
    const uint32_t total = static_cast<uint32_t>(a.rows * a.Dv);
    const int64_t want = (static_cast<int64_t>(total) + kThreads * kIlp - 1) / (kThreads * kIlp);
    const int64_t cap = static_cast<int64_t>(dev.sms) * bps;
    const int grid = static_cast<int>(want < cap ? want : cap);
    const FastDiv fd_row = FastDiv::make(static_cast<uint32_t>(a.Dv));
    const FastDiv fd_batch = FastDiv::make(static_cast<uint32_t>(a.S > 0 ? a.S : 1));
    return launch_dependent(ew_kernel<OP>, grid, kThreads, 0, stream, a, total, fd_row, fd_batch);
}

}  // namespace

cudaError_t launch_elementwise(int op, const EwArgs& a, const DeviceInfo& dev,
                               cudaStream_t stream)
{
    switch (op) {
    case kEwModulate:
        return launch<kEwModulate>(a, dev, stream);
    case kEwModulateF16:
        return launch<kEwModulateF16>(a, dev, stream);
    case kEwGateAdd:
        return launch<kEwGateAdd>(a, dev, stream);
    default:
        return launch<kEwBias>(a, dev, stream);
    }
}

}  // namespace rmsmod
