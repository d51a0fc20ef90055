// rmsnorm_silu_cl on sm_103a: channels-last RMSNorm * gamma + SiLU with the
// deferred conv bias folded in (sglang #38650 Wan VAE, §Quality-gated and
// §Modifications).
//
// In a channels_last(_3d) activation each pixel's C channels are contiguous
// and consecutive pixels are adjacent, so a run of pixels is one contiguous
// byte range.  P lanes share a pixel (V 16-byte vectors each, P * V * 8 >= C)
// and a warp covers 32 / P consecutive pixels per step; that tile is one
// contiguous span of at most 32 * V vectors, brought into shared memory by a
// 1-D bulk copy (TMA) into a ring of kStages tiles per warp.  Gamma and the
// bias (rounded to bf16 once) are staged in shared memory per CTA, so a lane
// carries only its pixel's values in registers and V can be large enough to
// amortise the per-pixel reduction, rstd and bound checks over many values.
//
//   xb  = R(x + R(bias))              (aten add_ arithmetic, before the statistics)
//   z   = (xb * rstd) * gamma         (fp32, unrounded)
//   out = R(z * sigmoid(z))  (z / (1 + exp(-z)) with hardware exp2 / reciprocal
//                             approximations; an accurate form where |z| may
//                             exceed 64)
#include "device_common.cuh"
#include "launch.h"

namespace rmsmod {

namespace {

__device__ unsigned int g_error;

constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
// vectors per lane the lane split aims for (P = smallest power of two with
// P * kVecTarget >= C / 8)
constexpr int kVecTarget = 6;
constexpr int kMaxCv = 1024 / 8;  // C <= 1024

template <int N>
struct Log2Ceil {
    static constexpr int value = (N <= 1) ? 0 : 1 + Log2Ceil<(N + 1) / 2>::value;
};
template <>
struct Log2Ceil<1> {
    static constexpr int value = 0;
};

// Three CTAs (24 warps) per SM: the per-pixel reduction, rstd and SiLU are
// chains of dependent instructions, and more resident warps hide them
// better than deeper rings (the 80-register cap this implies costs no
// spills).  Tiles in flight per warp: 2 of up to 3 KB (V = 6), 4 below.
constexpr int kBlocksPerSm = 3;

template <int V>
struct WanShape {
    static constexpr int kTileVec = 32 * V;  // tile capacity in 16-byte vectors
    static constexpr int kStages = V >= 6 ? 2 : 4;
    static constexpr int kRingBytes = kWarps * kStages * kTileVec * 16;
};

// SiLU(z) = z * sigmoid(z) with sigmoid from e = exp(-|z|) in (0, 1], so
// nothing overflows: 1 / (1 + e) for z >= 0 and e / (1 + e) below zero.
// Accurate exp; used for pixels whose |z| may exceed kFastSiluLimit.
__device__ __forceinline__ float silu_wide(float z)
{
    const float e = expf(-fabsf(z));
    const float r = __fdividef(1.0f, __fadd_rn(1.0f, e));
    const float s = z >= 0.0f ? r : __fmul_rn(e, r);
    return __fmul_rn(z, s);
}

// Two SiLUs as z / (1 + 2^(-z * log2 e)) with the hardware exp2 and
// reciprocal approximations (relative error ~2^-21 for |z| <= 64, far below
// a bf16 rounding step).  For z > 87 the exponential underflows to 0 and
// the result is z; below about -88 it would overflow, which the caller
// excludes with a bound on |z|.
constexpr float kFastSiluLimit = 64.0f;

__device__ __forceinline__ u64 silu2_fast(u64 z)
{
    const u64 t = f2_mul(z, f2_splat(-1.4426950408889634f));
    float t0, t1;
    f2_unpack(t, t0, t1);
    float e0, e1;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e0) : "f"(t0));
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e1) : "f"(t1));
    float d0, d1;
    f2_unpack(f2_add(f2_pack(e0, e1), f2_splat(1.0f)), d0, d1);
    float r0, r1;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r0) : "f"(d0));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r1) : "f"(d1));
    return f2_mul(z, f2_pack(r0, r1));
}

// EXACT: C == 8 * P * V, so no channel vector needs a bounds check.
template <int P, int V, bool EXACT>
__global__ void __launch_bounds__(kThreads, kBlocksPerSm) wan_kernel(const WanArgs a)
{
    grid_dependency_sync();
    constexpr int kL = Log2Ceil<8 * V>::value;
    constexpr int kPix = 32 / P;  // pixels per warp step
    constexpr int kTileVec = WanShape<V>::kTileVec;
    constexpr int kStages = WanShape<V>::kStages;

    extern __shared__ __align__(128) uint4 ring[];
    __shared__ __align__(8) unsigned long long bars[kWarps][kStages];
    __shared__ uint32_t s_gmax;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int sub = lane % P;
    const int psub = lane / P;
    const int Cv = a.Cv;

    const uint4* __restrict__ x = static_cast<const uint4*>(a.x);
    uint4* __restrict__ out = static_cast<uint4*>(a.out);
    const bool has_bias = a.bias != nullptr;
    uint4* c_gamma = ring + WanShape<V>::kRingBytes / 16;
    uint4* c_bias = c_gamma + Cv;

    uint4* wbuf = ring + warp * kStages * kTileVec;
    const uint32_t bar0 = smem_addr(&bars[warp][0]);
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < kStages; ++s)
            mbar_init(bar0 + 8u * s, 1u);
        mbar_init_fence();
    }
    if (threadIdx.x == 0)
        s_gmax = 0u;
    __syncwarp();

    const int64_t first = static_cast<int64_t>(blockIdx.x) * kWarps + warp;  // tile index
    const int64_t step = static_cast<int64_t>(gridDim.x) * kWarps;
    auto issue = [&](int64_t k) {
        const int64_t pix0 = (first + k * step) * kPix;
        if (lane != 0 || pix0 >= a.pixels)
            return;
        const int64_t left = a.pixels - pix0;
        const uint32_t bytes =
            static_cast<uint32_t>((left < kPix ? left : kPix) * Cv) * 16u;
        const int st = static_cast<int>(k % kStages);
        const uint32_t bar = bar0 + 8u * st;
        fence_proxy_async();
        mbar_expect_tx(bar, bytes);
        bulk_g2s(smem_addr(wbuf + st * kTileVec), x + pix0 * Cv, bytes, bar);
    };
#pragma unroll
    for (int k = 0; k < kStages; ++k)
        issue(k);

    // gamma and R(bias) for every channel, and max |gamma| (the bound on |z|
    // below uses it), while the first tiles are in flight
    __syncthreads();
    {
        uint32_t gm = 0;
        for (int c = threadIdx.x; c < Cv; c += kThreads) {
            const uint4 g = ld_cached(static_cast<const uint4*>(a.gamma) + c);
            uint4 bb = make_uint4(0u, 0u, 0u, 0u);
            if (has_bias) {
                if (a.bias_is_fp32) {
                    const float4* bf = static_cast<const float4*>(a.bias) + 2 * c;
                    const float4 lo = ld_cached_f4(bf), hi = ld_cached_f4(bf + 1);
                    bb = make_uint4(pack_bf2(lo.x, lo.y), pack_bf2(lo.z, lo.w),
                                    pack_bf2(hi.x, hi.y), pack_bf2(hi.z, hi.w));
                } else {
                    bb = ld_cached(static_cast<const uint4*>(a.bias) + c);
                }
            }
            c_gamma[c] = g;
            c_bias[c] = bb;
            gm = bf2_absmax(bf2_absmax(gm, bf2_absmax(g.x, g.y)), bf2_absmax(g.z, g.w));
        }
        atomicMax(&s_gmax, absmax_bits(gm));
    }
    __syncthreads();
    const float gmax = __uint_as_float(s_gmax << 16);

    bool broken = false;
    for (int64_t k = 0; (first + k * step) * kPix < a.pixels; ++k) {
        const int64_t pix0 = (first + k * step) * kPix;
        const int st = static_cast<int>(k % kStages);
        if (!broken && !mbar_wait(bar0 + 8u * st, static_cast<uint32_t>((k / kStages) & 1),
                                  kWaitLimitNs)) {
            broken = true;
            if (lane == 0)
                atomicOr(&g_error, kErrCopyTimeout);
        }
        const int64_t pix = pix0 + psub;
        const bool valid = pix < a.pixels;
        const int64_t base = pix * Cv;

        const uint4* tile = wbuf + st * kTileVec + psub * Cv;
        uint4 xv[V];
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int c = sub + P * j;
            if (valid && (EXACT || c < Cv)) {
                uint4 v = tile[c];
                if (has_bias) {
                    const uint4 bb = c_bias[c];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        word(v, i) = bf2_add(word(v, i), word(bb, i));
                }
                xv[j] = v;
            } else {
                xv[j] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        __syncwarp();
        issue(k + kStages);

        const uint32_t mm = tree_absmax<V>(xv);
        const uint32_t E = offset_exponent(mm);

        ExactSums<false> acc;
        acc.init(offset_k1<kL>(E), offset_k2<kL>(E));
#pragma unroll
        for (int j = 0; j < V; ++j)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                acc.add(f2_from_bf2(word(xv[j], i)));
        float s1h, s1l, s2h, s2l;
        acc.lane_total(s1h, s1l, s2h, s2l);
        dd_allreduce<P>(s2h, s2l);
        uint32_t cls = allreduce_max<P>(static_cast<uint32_t>(magnitude_class(mm)));
        uint32_t emax = allreduce_max<P>(mm == 0 ? 0u : (mm >> 7));
        float stat = finalize_ms(s2h, s2l, a.n, a.inv_n);

        if (__any_sync(kFullMask, cls != kClassFast)) {
            // Rare (Inf/NaN or extreme magnitudes in some pixel of this warp):
            // every lane runs both slow variants; each pixel keeps its own.
            float p2 = 0.0f;
            RowScale rs;
            rs.set(emax);
            ExactSums<false> acc2;
            acc2.init(offset_k1<kL>(127u), offset_k2<kL>(127u));
#pragma unroll
            for (int j = 0; j < V; ++j)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const u64 xx = f2_from_bf2(word(xv[j], i));
                    float lo, hi;
                    f2_unpack(xx, lo, hi);
                    p2 = __fadd_rn(__fadd_rn(p2, __fmul_rn(lo, lo)), __fmul_rn(hi, hi));
                    acc2.add(rs.apply(xx));
                }
            p2 = allreduce_add<P>(p2);
            float t1h, t1l, t2h, t2l;
            acc2.lane_total(t1h, t1l, t2h, t2l);
            dd_allreduce<P>(t2h, t2l);
            if (cls == kClassNonFinite)
                stat = __fmul_rn(p2, a.inv_n);
            else if (cls == kClassScaled)
                stat = rs.unscale(finalize_ms(t2h, t2l, a.n, a.inv_n), 2);
        }
        const float rstd = rstd_from(stat, a.eps);
        if (valid && sub == 0 && a.rstd_out)
            a.rstd_out[pix] = rstd;

        const u64 rstd2 = f2_splat(rstd);
        // |z| <= max|xb| * rstd * max|gamma|: the fast SiLU is exact enough
        // below the limit; any pixel of the warp above it (or NaN) sends the
        // whole step through the accurate form
        const float zbound =
            __fmul_rn(__fmul_rn(__uint_as_float(mm << 16), rstd), gmax);
        const bool wide = __any_sync(kFullMask, !(zbound <= kFastSiluLimit));
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int c = sub + P * j;
            if (valid && (EXACT || c < Cv)) {
                const uint4 g = c_gamma[c];
                uint4 o;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const u64 z = f2_mul(f2_mul(f2_from_bf2(word(xv[j], i)), rstd2),
                                         f2_from_bf2(word(g, i)));
                    if (!wide) {
                        word(o, i) = bf2_from_f2(silu2_fast(z));
                    } else {
                        float z0, z1;
                        f2_unpack(z, z0, z1);
                        word(o, i) = pack_bf2(silu_wide(z0), silu_wide(z1));
                    }
                }
                st_stream(out + base + c, o);
            }
        }
    }
    if (broken)
        drain_pause();
}

template <int P, int V, bool EXACT>
cudaError_t launch_shape(const WanArgs& a, const DeviceInfo& dev, cudaStream_t stream)
{
    auto kern = wan_kernel<P, V, EXACT>;
    constexpr int kSmemMax = WanShape<V>::kRingBytes + 2 * kMaxCv * 16;
    static PerDeviceInt blocks_per_sm;
    int bps = 0;
    {
        const cudaError_t e0 = blocks_per_sm.get(dev.device, bps, [&](int& v) -> cudaError_t {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 kSmemMax);
            if (e != cudaSuccess)
                return e;
            int nb = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, kThreads,
                                                              WanShape<V>::kRingBytes + 2 * a.Cv * 16);
            if (e != cudaSuccess)
                return e;
            v = nb > 0 ? nb : 1;
            return cudaSuccess;
        });
        if (e0 != cudaSuccess)
            return e0;
    }
    constexpr int kPixPerBlock = (32 / P) * kWarps;
    const int64_t want = (a.pixels + kPixPerBlock - 1) / kPixPerBlock;
    const int64_t cap = static_cast<int64_t>(dev.sms) * bps;
    const int grid = static_cast<int>(want < cap ? want : cap);
    const int smem = WanShape<V>::kRingBytes + 2 * a.Cv * 16;
    return launch_dependent(kern, grid, kThreads, smem, stream, a);
}

template <int P, int V>
cudaError_t launch_cfg(const WanArgs& a, const DeviceInfo& dev, cudaStream_t stream)
{
    if (a.Cv == P * V)
        return launch_shape<P, V, true>(a, dev, stream);
    return launch_shape<P, V, false>(a, dev, stream);
}

template <int P>
cudaError_t launch_p(const WanArgs& a, const DeviceInfo& dev, cudaStream_t stream)
{
    const int V = (a.Cv + P - 1) / P;
    if (V <= 1)
        return launch_cfg<P, 1>(a, dev, stream);
    if (V <= 2)
        return launch_cfg<P, 2>(a, dev, stream);
    if (V <= 3)
        return launch_cfg<P, 3>(a, dev, stream);
    if (V <= 4)
        return launch_cfg<P, 4>(a, dev, stream);
    return launch_cfg<P, kVecTarget>(a, dev, stream);
}

}  // namespace

cudaError_t launch_wan_kernel(const WanArgs& a, const DeviceInfo& dev, cudaStream_t stream)
{
    const int need = (a.Cv + kVecTarget - 1) / kVecTarget;
    if (need <= 1)
        return launch_p<1>(a, dev, stream);
    if (need <= 2)
        return launch_p<2>(a, dev, stream);
    if (need <= 4)
        return launch_p<4>(a, dev, stream);
    if (need <= 8)
        return launch_p<8>(a, dev, stream);
    if (need <= 16)
        return launch_p<16>(a, dev, stream);
    return launch_p<32>(a, dev, stream);
}

cudaError_t wan_kernel_error(unsigned* bits, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(bits, g_error, sizeof(unsigned));
    if (e == cudaSuccess && clear && *bits) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_error, &zero, sizeof(unsigned));
    }
    return e;
}

}  // namespace rmsmod
