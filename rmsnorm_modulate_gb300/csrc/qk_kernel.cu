// qk_layernorm on sm_103a: per-head LayerNorm(128) with affine, q rows and k
// rows in one launch (sglang #34008 GLM-Image, §Motivation qk-norm bullet and
// §What "rounding-faithful" means here, qk bullet).
//
// A 128-element head row is 256 bytes (16 vectors of eight bf16).  P lanes
// own one row (16 / P vectors each), so a warp covers a tile of 32 / P
// consecutive rows per step and every lane is busy -- the eager kernel
// spends a 128-thread block per row with three of its four warps idle.
// Tiles reach shared memory by 1-D bulk copies (TMA) into a ring per warp,
// so the next tiles are in flight while one is computed.  Blocks are split
// between the q rows and the k rows in proportion; a block stages its
// weight and bias once, widened to fp32, in shared memory.  A lane visits
// its vectors in an order rotated by its row inside the tile, which keeps
// the row reads (256-byte stride) and the weight reads free of bank
// conflicts.
//
//   z = R(((x - mean) * rstd) * w + b)   -- fp32, one final rounding
#include "device_common.cuh"
#include "launch.h"

namespace rmsmod {

namespace {

__device__ unsigned int g_error;

constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int kRowVec = 16;                       // 16-byte vectors per row
constexpr int kLanesPerRow = 2;                   // P
constexpr int kVecPerLane = kRowVec / kLanesPerRow;
constexpr int kTileRows = 32 / kLanesPerRow;      // rows per warp step
constexpr int kTileVec = kTileRows * kRowVec;     // 16-byte vectors per tile
constexpr int kStages = 3;
constexpr int kSmem = kWarps * kStages * kTileVec * 16;
constexpr int kL = 6;                             // 8 * kVecPerLane = 2^kL values per lane
static_assert((8 << kL) == 8 * 8 * kVecPerLane, "kL must be log2 of the values per lane");

__global__ void __launch_bounds__(kThreads, 2) qk_kernel(const QkArgs a, int blocks_q)
{
    grid_dependency_sync();
    extern __shared__ __align__(128) uint4 ring[];
    __shared__ __align__(8) unsigned long long bars[kWarps][kStages];
    // weight and bias of this block's tensor, fp32, as [vector][half] float4
    __shared__ __align__(16) float4 s_w[2][kRowVec], s_b[2][kRowVec];

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
    const int sub = lane % kLanesPerRow;   // position inside the row
    const int rsub = lane / kLanesPerRow;  // row inside the tile
    const int rot = rsub % kVecPerLane;

    uint4* wbuf = ring + warp * kStages * kTileVec;
    const uint32_t bar0 = smem_addr(&bars[warp][0]);
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < kStages; ++s)
            mbar_init(bar0 + 8u * s, 1u);
        mbar_init_fence();
    }
    __syncwarp();

    const int64_t first = static_cast<int64_t>(blk) * kWarps + warp;  // tile index
    const int64_t step = static_cast<int64_t>(nblk) * kWarps;
    auto issue = [&](int64_t k) {
        const int64_t row0 = (first + k * step) * kTileRows;
        if (lane != 0 || row0 >= rows)
            return;
        const int64_t left = rows - row0;
        const uint32_t bytes = static_cast<uint32_t>(left < kTileRows ? left : kTileRows) * 256u;
        const int st = static_cast<int>(k % kStages);
        const uint32_t bar = bar0 + 8u * st;
        fence_proxy_async();
        mbar_expect_tx(bar, bytes);
        bulk_g2s(smem_addr(wbuf + st * kTileVec), src + row0 * kRowVec, bytes, bar);
    };
#pragma unroll
    for (int k = 0; k < kStages; ++k)
        issue(k);

    if (threadIdx.x < 2 * kRowVec) {
        const int c = threadIdx.x >> 1, h = threadIdx.x & 1;
        const uint4 w = ld_cached(wv + c), b = ld_cached(bv + c);
        const uint32_t w0 = h ? w.z : w.x, w1 = h ? w.w : w.y;
        const uint32_t b0 = h ? b.z : b.x, b1 = h ? b.w : b.y;
        float l0, h0, l1, h1;
        f2_unpack(f2_from_bf2(w0), l0, h0);
        f2_unpack(f2_from_bf2(w1), l1, h1);
        s_w[h][c] = make_float4(l0, h0, l1, h1);
        f2_unpack(f2_from_bf2(b0), l0, h0);
        f2_unpack(f2_from_bf2(b1), l1, h1);
        s_b[h][c] = make_float4(l0, h0, l1, h1);
    }
    __syncthreads();

    const float n = 128.0f, inv_n = 1.0f / 128.0f;
    bool broken = false;
    for (int64_t k = 0; (first + k * step) * kTileRows < rows; ++k) {
        const int64_t row0 = (first + k * step) * kTileRows;
        const int st = static_cast<int>(k % kStages);
        if (!broken && !mbar_wait(bar0 + 8u * st, static_cast<uint32_t>((k / kStages) & 1),
                                  kWaitLimitNs)) {
            broken = true;
            if (lane == 0)
                atomicOr(&g_error, kErrCopyTimeout);
        }
        const int64_t row = row0 + rsub;
        const bool valid = row < rows;
        const int64_t base = row * kRowVec;

        // vector j of this lane is c(j) = sub + P * ((j + rot) mod V)
        const uint4* tile = wbuf + st * kTileVec + rsub * kRowVec;
        uint4 xv[kVecPerLane];
#pragma unroll
        for (int j = 0; j < kVecPerLane; ++j) {
            const int jj = (j + rot) % kVecPerLane;
            xv[j] = valid ? tile[sub + kLanesPerRow * jj] : make_uint4(0u, 0u, 0u, 0u);
        }
        __syncwarp();
        issue(k + kStages);

        const uint32_t mm = tree_absmax<kVecPerLane>(xv);
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

        // row class over its lanes
        uint32_t cls = allreduce_max<kLanesPerRow>(static_cast<uint32_t>(magnitude_class(mm)));
        uint32_t emax = allreduce_max<kLanesPerRow>(mm == 0 ? 0u : (mm >> 7));

        float mean, var;
        finalize_ln_pow2(s1h, s1l, s2h, s2l, n, inv_n, mean, var);
        if (__any_sync(kFullMask, cls != kClassFast)) {
            // Rare: some row of this tile holds Inf/NaN or extreme magnitudes.
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
                finalize_ln_pow2(t1h, t1l, t2h, t2l, n, inv_n, ms, vs);
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
                const int c = sub + kLanesPerRow * ((j + rot) % kVecPerLane);
                const float4 w_lo = s_w[0][c], w_hi = s_w[1][c];
                const float4 b_lo = s_b[0][c], b_hi = s_b[1][c];
                const u64 w2[4] = {f2_pack(w_lo.x, w_lo.y), f2_pack(w_lo.z, w_lo.w),
                                   f2_pack(w_hi.x, w_hi.y), f2_pack(w_hi.z, w_hi.w)};
                const u64 b2[4] = {f2_pack(b_lo.x, b_lo.y), f2_pack(b_lo.z, b_lo.w),
                                   f2_pack(b_hi.x, b_hi.y), f2_pack(b_hi.z, b_hi.w)};
                uint4 o;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const u64 xx = f2_from_bf2(word(xv[j], i));
                    const u64 z = f2_mul_then_add(f2_mul(f2_sub(xx, mean2), rstd2), w2[i], b2[i]);
                    word(o, i) = bf2_from_f2(z);
                }
                st_stream(dst + base + c, o);
            }
        }
    }
    if (broken)
        drain_pause();
}

}  // namespace

cudaError_t launch_qk_kernel(const QkArgs& a, const DeviceInfo& dev, cudaStream_t stream)
{
    static int blocks_per_sm[64] = {0};
    const int d = dev.device & 63;
    if (blocks_per_sm[d] == 0) {
        cudaError_t e =
            cudaFuncSetAttribute(qk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (e != cudaSuccess)
            return e;
        int nb = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, qk_kernel, kThreads, kSmem);
        if (e != cudaSuccess)
            return e;
        blocks_per_sm[d] = nb > 0 ? nb : 1;
    }
    constexpr int kRowsPerBlock = kTileRows * kWarps;
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
    return launch_dependent(qk_kernel, grid, kThreads, kSmem, stream, a, static_cast<int>(bq));
}

cudaError_t qk_kernel_error(unsigned* bits, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(bits, g_error, sizeof(unsigned));
    if (e == cudaSuccess && clear && *bits) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_error, &zero, sizeof(unsigned));
    }
    return e;
}

}  // namespace rmsmod
