// qk_layernorm on sm_103a: per-head LayerNorm(128) with affine, q rows and k
// rows in one launch (sglang #34008 GLM-Image, §Motivation qk-norm bullet and
// §What "rounding-faithful" means here, qk bullet).
//
// A 128-element head row is 256 bytes.  Four lanes own one row (32 values
// each, as four 16-byte vectors), so one warp covers eight rows per step and
// every lane is busy -- the eager kernel spends a 128-thread block per row
// with three of its four warps idle.  A warp-instruction's 32 loads cover
// eight 64-byte segments: full 32-byte sectors, no wasted DRAM bytes.
// Blocks are split between the q rows and the k rows in proportion, so a
// lane's weight and bias (32 columns, kept as fp32 pairs in registers) are
// loaded once per kernel.
//
//   z = R(((x - mean) * rstd) * w + b)   -- fp32, one final rounding
#include "device_common.cuh"
#include "launch.h"

namespace rmsmod {

namespace {

constexpr int kThreads = 256;
constexpr int kLanesPerRow = 4;
constexpr int kVecPerLane = 4;         // 4 x 8 = 32 values per lane
constexpr int kRowsPerWarp = 32 / kLanesPerRow;
constexpr int kRowsPerBlock = kRowsPerWarp * (kThreads / 32);
constexpr int kL = 5;                  // 32 values per lane = 2^5

__global__ void __launch_bounds__(kThreads) qk_kernel(const QkArgs a, int blocks_q)
{
    const bool is_q = static_cast<int>(blockIdx.x) < blocks_q;
    const int64_t rows = is_q ? a.rows_q : a.rows_k;
    const int blk = is_q ? blockIdx.x : blockIdx.x - blocks_q;
    const int nblk = is_q ? blocks_q : gridDim.x - blocks_q;
    const uint4* __restrict__ src = static_cast<const uint4*>(is_q ? a.q : a.k);
    uint4* __restrict__ dst = static_cast<uint4*>(is_q ? a.q_out : a.k_out);
    const uint4* __restrict__ wv = static_cast<const uint4*>(is_q ? a.wq : a.wk);
    const uint4* __restrict__ bv = static_cast<const uint4*>(is_q ? a.bq : a.bk);
    const int64_t stat_off = is_q ? 0 : a.rows_q;

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int sub = lane & (kLanesPerRow - 1);   // position inside the row
    const int rsub = lane / kLanesPerRow;        // row inside the warp's eight

    // this lane's columns: vectors sub, sub + 4, sub + 8, sub + 12
    u64 w2[kVecPerLane][4], b2[kVecPerLane][4];
#pragma unroll
    for (int j = 0; j < kVecPerLane; ++j) {
        uint4 w = ld_cached(wv + sub + kLanesPerRow * j);
        uint4 b = ld_cached(bv + sub + kLanesPerRow * j);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            w2[j][i] = f2_from_bf2(word(w, i));
            b2[j][i] = f2_from_bf2(word(b, i));
        }
    }

    const float n = 128.0f, inv_n = 1.0f / 128.0f;
    for (int64_t row0 = (static_cast<int64_t>(blk) * (kThreads / 32) + warp) * kRowsPerWarp;
         row0 < rows; row0 += static_cast<int64_t>(nblk) * kRowsPerBlock) {
        const int64_t row = row0 + rsub;
        const bool valid = row < rows;
        const int64_t base = row * 16;

        uint4 xv[kVecPerLane];
#pragma unroll
        for (int j = 0; j < kVecPerLane; ++j)
            xv[j] = valid ? ld_stream(src + base + sub + kLanesPerRow * j)
                          : make_uint4(0u, 0u, 0u, 0u);

        uint32_t m = 0;
#pragma unroll
        for (int j = 0; j < kVecPerLane; ++j)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                m = bf2_absmax(m, word(xv[j], i));
        const uint32_t mm = absmax_bits(m);

        ExactSums<true> acc;
        const uint32_t E = offset_exponent(mm);
        acc.init(offset_k1<kL>(E), offset_k2<kL>(E));
#pragma unroll
        for (int j = 0; j < kVecPerLane; ++j)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                acc.add(f2_from_bf2(word(xv[j], i)));
        float s1h, s1l, s2h, s2l;
        acc.lane_total(s1h, s1l, s2h, s2l);
        dd2_allreduce<kLanesPerRow>(s1h, s1l, s2h, s2l);

        // row class over its four lanes
        uint32_t cls = static_cast<uint32_t>(magnitude_class(mm));
        uint32_t emax = mm == 0 ? 0u : (mm >> 7);
        cls = allreduce_max<kLanesPerRow>(cls);
        emax = allreduce_max<kLanesPerRow>(emax);

        float mean, var;
        finalize_ln(s1h, s1l, s2h, s2l, n, inv_n, mean, var);
        if (__any_sync(kFullMask, cls != kClassFast)) {
            // Rare: some row of this warp holds Inf/NaN or extreme magnitudes.
            // Every lane runs both slow variants (warp-uniform control flow)
            // and each row keeps the one its class asks for.
            float p1 = 0.0f, p2 = 0.0f;
            RowScale rs;
            rs.set(emax);
            ExactSums<true> acc2;
            acc2.init(offset_k1<kL>(127u), offset_k2<kL>(127u));
#pragma unroll
            for (int j = 0; j < kVecPerLane; ++j)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const u64 xx = f2_from_bf2(word(xv[j], i));
                    float lo, hi;
                    f2_unpack(xx, lo, hi);
                    p1 = __fadd_rn(__fadd_rn(p1, lo), hi);
                    p2 = __fadd_rn(__fadd_rn(p2, __fmul_rn(lo, lo)), __fmul_rn(hi, hi));
                    acc2.add(rs.apply(xx));
                }
            p1 = allreduce_add<kLanesPerRow>(p1);
            p2 = allreduce_add<kLanesPerRow>(p2);
            float t1h, t1l, t2h, t2l;
            acc2.lane_total(t1h, t1l, t2h, t2l);
            dd2_allreduce<kLanesPerRow>(t1h, t1l, t2h, t2l);
            if (cls == kClassNonFinite) {
                mean = __fmul_rn(p1, inv_n);
                var = __fsub_rn(__fmul_rn(p2, inv_n), __fmul_rn(mean, mean));
            } else if (cls == kClassScaled) {
                float ms, vs;
                finalize_ln(t1h, t1l, t2h, t2l, n, inv_n, ms, vs);
                mean = rs.unscale(ms, 1);
                var = rs.unscale(vs, 2);
            }
        }
        const float rstd = rstd_from(var, a.eps);
        if (valid && sub == 0) {
            if (a.mean_out)
                a.mean_out[stat_off + row] = mean;
            if (a.rstd_out)
                a.rstd_out[stat_off + row] = rstd;
        }
        if (valid) {
            const u64 mean2 = f2_splat(mean), rstd2 = f2_splat(rstd);
#pragma unroll
            for (int j = 0; j < kVecPerLane; ++j) {
                uint4 o;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const u64 xx = f2_from_bf2(word(xv[j], i));
                    u64 z = f2_mul(f2_sub(xx, mean2), rstd2);
                    z = f2_add(f2_mul(z, w2[j][i]), b2[j][i]);
                    word(o, i) = bf2_from_f2(z);
                }
                st_stream(dst + base + sub + kLanesPerRow * j, o);
            }
        }
    }
}

}  // namespace

cudaError_t launch_qk_kernel(const QkArgs& a, const DeviceInfo& dev, cudaStream_t stream)
{
    static int blocks_per_sm[64] = {0};
    const int d = dev.device & 63;
    if (blocks_per_sm[d] == 0) {
        int nb = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, qk_kernel, kThreads, 0);
        if (e != cudaSuccess)
            return e;
        blocks_per_sm[d] = nb > 0 ? nb : 1;
    }
    const int64_t total = a.rows_q + a.rows_k;
    const int64_t cap = static_cast<int64_t>(dev.sms) * blocks_per_sm[d];
    const int64_t need_q = (a.rows_q + kRowsPerBlock - 1) / kRowsPerBlock;
    const int64_t need_k = (a.rows_k + kRowsPerBlock - 1) / kRowsPerBlock;
    int64_t bq, bk;
    if (need_q + need_k <= cap) {
        bq = need_q;
        bk = need_k;
    } else {
        bq = (cap * a.rows_q + total / 2) / total;
        if (a.rows_q > 0 && bq < 1)
            bq = 1;
        if (a.rows_k > 0 && cap - bq < 1)
            bq = cap - 1;
        bk = cap - bq;
    }
    const int grid = static_cast<int>(bq + bk);
    qk_kernel<<<grid, kThreads, 0, stream>>>(a, static_cast<int>(bq));
    return cudaGetLastError();
}

}  // namespace rmsmod
