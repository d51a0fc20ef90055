// ln_modulate / rmsnorm_modulate / gated_rmsnorm_modulate on sm_103a.
//
// One warp (or a group of 2 / 4 warps for D > 4096) owns one row at a time
// and loops persistently over rows.  The row is loaded once with 16-byte
// streaming loads and stays in registers as packed bf16 while the exact
// statistics are formed; the normalise + modulate epilogue then runs on
// packed f32x2 / bf16x2 instructions and streams the result out.  HBM is
// touched exactly once per element in each direction; scale, shift, weight
// and gate rows are re-read from L1/L2.
//
// Arithmetic per element follows the eager chain of the pages:
//   LayerNorm (sglang #34008 GLM-Image, §What "rounding-faithful" means here):
//     y = R((x - mean) * rstd)
//   RMSNorm (sglang #33854 ERNIE-Image, same section):
//     y = R((x * rstd) * w)
//   gated residual (sglang #33854, residual variant):
//     res = R(residual + R(gate * update))
//   modulate chain (both pages; sglang #34004 FLUX.1 §Modifications commit 2):
//     out = R(R(y * R(1 + scale)) + shift)
#include "device_common.cuh"
#include "launch.h"

namespace rmsmod {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <int N>
struct Log2Ceil {
    static constexpr int value = (N <= 1) ? 0 : 1 + Log2Ceil<(N + 1) / 2>::value;
};
template <>
struct Log2Ceil<1> {
    static constexpr int value = 0;
};

// Per-group exchange slot used when several warps share a row.
struct Slot {
    float s1h, s1l, s2h, s2l;
    uint32_t cls, emax, pad0, pad1;
};

template <int WPR>
__device__ __forceinline__ void group_barrier(int group)
{
    if (WPR > 1)
        asm volatile("bar.sync %0, %1;" ::"r"(group + 1), "r"(WPR * 32) : "memory");
}

// Combines the per-warp double-float partials of one row (fixed order, so
// every lane of every warp of the group gets bit-identical totals).
template <int WPR>
__device__ __forceinline__ void group_combine(Slot* slots, int wig, int lane, int group,
                                              float& s1h, float& s1l, float& s2h, float& s2l,
                                              uint32_t& cls, uint32_t& emax)
{
    if (WPR == 1)
        return;
    if (lane == 0)
        slots[wig] = Slot{s1h, s1l, s2h, s2l, cls, emax, 0u, 0u};
    group_barrier<WPR>(group);
    Slot t = slots[0];
    s1h = t.s1h;
    s1l = t.s1l;
    s2h = t.s2h;
    s2l = t.s2l;
    cls = t.cls;
    emax = t.emax;
#pragma unroll
    for (int w = 1; w < WPR; ++w) {
        Slot o = slots[w];
        u64 H = f2_pack(s1h, s2h), Lo = f2_pack(s1l, s2l);
        dd2_add(H, Lo, f2_pack(o.s1h, o.s2h), f2_pack(o.s1l, o.s2l));
        f2_unpack(H, s1h, s2h);
        f2_unpack(Lo, s1l, s2l);
        cls = cls > o.cls ? cls : o.cls;
        emax = emax > o.emax ? emax : o.emax;
    }
}

// Plain IEEE fp32 sums of two values over the warps of a group (fixed order).
template <int WPR>
__device__ __forceinline__ void group_sum_plain(Slot* slots, int wig, int lane, int group,
                                                float& p1, float& p2)
{
    if (WPR == 1)
        return;
    if (lane == 0)
        slots[wig] = Slot{p1, 0.0f, p2, 0.0f, 0u, 0u, 0u, 0u};
    group_barrier<WPR>(group);
    p1 = slots[0].s1h;
    p2 = slots[0].s2h;
#pragma unroll
    for (int w = 1; w < WPR; ++w) {
        p1 = __fadd_rn(p1, slots[w].s1h);
        p2 = __fadd_rn(p2, slots[w].s2h);
    }
    group_barrier<WPR>(group);
}

template <int OP, int V, int WPR>
__global__ void __launch_bounds__(kThreads) row_kernel(const RowArgs a)
{
    constexpr int kGroups = kWarps / WPR;
    constexpr int kL = Log2Ceil<8 * V>::value;
    constexpr bool kNeedSum = (OP == kOpLN);
    // [parity][group][warp in group] for the common path, plus one slot row
    // per group for the rare slow path.
    __shared__ Slot slots[2][kGroups][WPR];
    __shared__ Slot slow_slots[kGroups][WPR];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int group = warp / WPR;
    const int wig = warp % WPR;
    const int Dv = a.Dv;

    const uint4* __restrict__ x = static_cast<const uint4*>(a.x);
    const uint4* __restrict__ residual = static_cast<const uint4*>(a.residual);
    const uint4* __restrict__ update = static_cast<const uint4*>(a.update);
    const uint4* __restrict__ gate = static_cast<const uint4*>(a.gate);
    const uint4* __restrict__ weight = static_cast<const uint4*>(a.weight);
    const uint4* __restrict__ scale = static_cast<const uint4*>(a.scale);
    const uint4* __restrict__ shift = static_cast<const uint4*>(a.shift);
    uint4* __restrict__ res_out = static_cast<uint4*>(a.res_out);
    uint4* __restrict__ out = static_cast<uint4*>(a.out);
    const bool has_w = (weight != nullptr);

    int parity = 0;
    for (int64_t row = static_cast<int64_t>(blockIdx.x) * kGroups + group; row < a.rows;
         row += static_cast<int64_t>(gridDim.x) * kGroups, parity ^= 1) {
        const int64_t b = row / a.S;
        const int64_t base = row * Dv;

        // ---- load (and for the gated op, form and store the residual stream)
        uint4 xv[V];
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int c = j * (32 * WPR) + wig * 32 + lane;
            if (c < Dv) {
                if (OP == kOpGated) {
                    uint4 r = ld_stream(residual + base + c);
                    uint4 u = ld_stream(update + base + c);
                    uint4 g = ld_cached(gate + b * a.gate_bstride + c);
                    uint4 s;
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        word(s, i) = bf2_add(word(r, i), bf2_mul(word(g, i), word(u, i)));
                    st_stream(res_out + base + c, s);
                    xv[j] = s;
                } else {
                    xv[j] = ld_stream(x + base + c);
                }
            } else {
                xv[j] = make_uint4(0u, 0u, 0u, 0u);
            }
        }

        // ---- magnitude class of this lane's values
        uint32_t m = 0;
#pragma unroll
        for (int j = 0; j < V; ++j)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                m = bf2_absmax(m, word(xv[j], i));
        const uint32_t mm = absmax_bits(m);
        const uint32_t E = offset_exponent(mm);

        // ---- exact sums (fast path; discarded if the row needs the slow path)
        ExactSums<kNeedSum> acc;
        acc.init(offset_k1<kL>(E), offset_k2<kL>(E));
#pragma unroll
        for (int j = 0; j < V; ++j)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                acc.add(f2_from_bf2(word(xv[j], i)));
        float s1h, s1l, s2h, s2l;
        acc.lane_total(s1h, s1l, s2h, s2l);
        if (kNeedSum)
            dd2_allreduce<32>(s1h, s1l, s2h, s2l);
        else
            dd_allreduce<32>(s2h, s2l);
        uint32_t cls = __reduce_max_sync(kFullMask, static_cast<uint32_t>(magnitude_class(mm)));
        uint32_t emax = __reduce_max_sync(kFullMask, mm == 0 ? 0u : (mm >> 7));
        group_combine<WPR>(&slots[parity][group][0], wig, lane, group, s1h, s1l, s2h, s2l,
                           cls, emax);

        float mean = 0.0f, stat;
        if (cls == kClassFast) {
            if (kNeedSum)
                finalize_ln(s1h, s1l, s2h, s2l, a.n, a.inv_n, mean, stat);
            else
                stat = finalize_ms(s2h, s2l, a.n, a.inv_n);
        } else if (cls == kClassNonFinite) {
            // Inf / NaN in the row: plain IEEE sums propagate them the way
            // the exact (double) sums do.
            float p1 = 0.0f, p2 = 0.0f;
#pragma unroll
            for (int j = 0; j < V; ++j)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float lo, hi;
                    f2_unpack(f2_from_bf2(word(xv[j], i)), lo, hi);
                    p1 = __fadd_rn(__fadd_rn(p1, lo), hi);
                    p2 = __fadd_rn(__fadd_rn(p2, __fmul_rn(lo, lo)), __fmul_rn(hi, hi));
                }
            p1 = allreduce_add<32>(p1);
            p2 = allreduce_add<32>(p2);
            group_sum_plain<WPR>(&slow_slots[group][0], wig, lane, group, p1, p2);
            mean = __fmul_rn(p1, a.inv_n);
            const float msq = __fmul_rn(p2, a.inv_n);
            stat = kNeedSum ? __fsub_rn(msq, __fmul_rn(mean, mean)) : msq;
        } else {
            // Extreme magnitudes: scale the row to unit size by a power of
            // two (exact), sum, and scale the statistics back.
            RowScale rs;
            rs.set(emax);
            ExactSums<kNeedSum> acc2;
            acc2.init(offset_k1<kL>(127u), offset_k2<kL>(127u));
#pragma unroll
            for (int j = 0; j < V; ++j)
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    acc2.add(rs.apply(f2_from_bf2(word(xv[j], i))));
            acc2.lane_total(s1h, s1l, s2h, s2l);
            if (kNeedSum)
                dd2_allreduce<32>(s1h, s1l, s2h, s2l);
            else
                dd_allreduce<32>(s2h, s2l);
            uint32_t c2 = cls, e2 = emax;
            group_combine<WPR>(&slow_slots[group][0], wig, lane, group, s1h, s1l, s2h, s2l, c2,
                               e2);
            group_barrier<WPR>(group);
            if (kNeedSum) {
                float ms, vs;
                finalize_ln(s1h, s1l, s2h, s2l, a.n, a.inv_n, ms, vs);
                mean = rs.unscale(ms, 1);
                stat = rs.unscale(vs, 2);
            } else {
                stat = rs.unscale(finalize_ms(s2h, s2l, a.n, a.inv_n), 2);
            }
        }
        const float rstd = rstd_from(stat, a.eps);
        if (lane == 0 && wig == 0) {
            if (a.mean_out)
                a.mean_out[row] = mean;
            if (a.rstd_out)
                a.rstd_out[row] = rstd;
        }

        // ---- normalise + modulate + store
        const u64 mean2 = f2_splat(mean);
        const u64 rstd2 = f2_splat(rstd);
        const uint4* sc = scale + b * a.mod_bstride;
        const uint4* sh = shift + b * a.mod_bstride;
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int c = j * (32 * WPR) + wig * 32 + lane;
            if (c < Dv) {
                const uint4 s = ld_cached(sc + c);
                const uint4 h = ld_cached(sh + c);
                uint4 w = make_uint4(0u, 0u, 0u, 0u);
                if (OP != kOpLN && has_w)
                    w = ld_cached(weight + c);
                uint4 o;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const u64 xx = f2_from_bf2(word(xv[j], i));
                    u64 y;
                    if (OP == kOpLN) {
                        y = f2_mul(f2_sub(xx, mean2), rstd2);
                    } else {
                        y = f2_mul(xx, rstd2);
                        if (has_w)
                            y = f2_mul(y, f2_from_bf2(word(w, i)));
                    }
                    const uint32_t yb = bf2_from_f2(y);
                    const uint32_t s1 = bf2_add(word(s, i), kBf2One);
                    word(o, i) = bf2_add(bf2_mul(yb, s1), word(h, i));
                }
                st_stream(out + base + c, o);
            }
        }
    }
}

template <int OP, int V, int WPR>
cudaError_t launch_cfg(const RowArgs& a, const DeviceInfo& dev, cudaStream_t stream)
{
    auto kern = row_kernel<OP, V, WPR>;
    static int blocks_per_sm[64] = {0};
    int d = dev.device & 63;
    if (blocks_per_sm[d] == 0) {
        int n = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, 0);
        if (e != cudaSuccess)
            return e;
        blocks_per_sm[d] = n > 0 ? n : 1;
    }
    constexpr int kGroups = kWarps / WPR;
    int64_t want = (a.rows + kGroups - 1) / kGroups;
    int64_t cap = static_cast<int64_t>(dev.sms) * blocks_per_sm[d];
    int grid = static_cast<int>(want < cap ? want : cap);
    kern<<<grid, kThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

template <int OP>
cudaError_t launch_op(const RowArgs& a, const DeviceInfo& dev, cudaStream_t stream)
{
    const int Dv = a.Dv;
    if (Dv <= 32)
        return launch_cfg<OP, 1, 1>(a, dev, stream);
    if (Dv <= 64)
        return launch_cfg<OP, 2, 1>(a, dev, stream);
    if (Dv <= 128)
        return launch_cfg<OP, 4, 1>(a, dev, stream);
    if (Dv <= 256)
        return launch_cfg<OP, 8, 1>(a, dev, stream);
    if (Dv <= 384)
        return launch_cfg<OP, 12, 1>(a, dev, stream);
    if (Dv <= 512)
        return launch_cfg<OP, 16, 1>(a, dev, stream);
    if (Dv <= 1024)
        return launch_cfg<OP, 16, 2>(a, dev, stream);
    return launch_cfg<OP, 16, 4>(a, dev, stream);
}

}  // namespace

cudaError_t launch_row_kernel(int op, const RowArgs& a, const DeviceInfo& dev,
                              cudaStream_t stream)
{
    switch (op) {
    case kOpLN:
        return launch_op<kOpLN>(a, dev, stream);
    case kOpRMS:
        return launch_op<kOpRMS>(a, dev, stream);
    default:
        return launch_op<kOpGated>(a, dev, stream);
    }
}

}  // namespace rmsmod
