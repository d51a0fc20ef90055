// qk_layernorm on sm_103a: per-head LayerNorm(head_dim) with affine, q rows
// and k rows in one launch (sglang #34008 GLM-Image, §Motivation qk-norm
// bullet and §What "rounding-faithful" means here, qk bullet; head_dim 64 /
// 96 and strided q/k views of a fused QKV projection at the other sites the
// page lists).
//
// A head row of head_dim = 8 * RV values is RV 16-byte vectors.  P lanes own
// one row (V = RV / P vectors each), so a warp covers a tile of 32 / P rows
// and every lane is busy -- the eager kernel spends a 128-thread block per
// row with three of its four warps idle.  The rows of a tile are consecutive
// heads of one token, so a tile is one contiguous span even when q and k are
// token-strided views; tiles reach shared memory by 1-D bulk copies (TMA)
// into a CTA ring shared by statistics warps (per-row mean / rstd) and output
// warps (the affine), so the reduction chains of some tiles overlap the
// epilogue of others.  Blocks are split between the q rows and the k rows in
// proportion; a block stages its weight and bias once, widened to fp32, in
// shared memory.  A lane visits its vectors in an order rotated by its row
// inside the tile, which keeps the row reads and the weight reads free of
// bank conflicts at 64 and 128 values per row (two-way at 96).
//
//   z = R(((x - mean) * rstd) * w + b)   -- fp32, one final rounding
#include "device_common.cuh"
#include "launch.h"

namespace rmsmod {

namespace {

__device__ unsigned int g_error;

constexpr int kMaxRowVec = 16;  // head_dim <= 128

template <int N>
struct Log2Ceil {
    static constexpr int value = (N <= 1) ? 0 : 1 + Log2Ceil<(N + 1) / 2>::value;
};
template <>
struct Log2Ceil<1> {
    static constexpr int value = 0;
};

template <int RV, int P>
struct QkShape {
    static constexpr int kVecPerLane = RV / P;
    static constexpr int kTileRows = 32 / P;
    static constexpr int kTileVec = kTileRows * RV;
    static constexpr int kL = Log2Ceil<8 * kVecPerLane>::value;
    static_assert(RV % P == 0, "a lane owns whole vectors");
};

// The rows of a tile whose class is not fast (Inf/NaN or extreme magnitudes):
// every lane runs both slow variants (warp-uniform control flow) and each row
// keeps the one its class asks for.
template <int RV, int P>
__device__ __noinline__ void qk_slow_stats(const uint4 (&xv)[QkShape<RV, P>::kVecPerLane],
                                           uint32_t cls, uint32_t emax, float& mean,
                                           float& var)
{
    using Shape = QkShape<RV, P>;
    constexpr int V = Shape::kVecPerLane;
    constexpr int kL = Shape::kL;
    constexpr float kN = 8.0f * RV;
    const float inv_n = 1.0f / kN;
    float p1 = 0.0f, p2 = 0.0f;
    RowScale rs;
    rs.set(emax);
    ExactSums<true> acc2;
    acc2.init(offset_k1<kL>(127u), offset_k2<kL>(127u));
#pragma unroll
    for (int j = 0; j < V; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const u64 xx = f2_from_bf2(word(xv[j], i));
            float lo, hi;
            f2_unpack(xx, lo, hi);
            p1 = __fadd_rn(__fadd_rn(p1, lo), hi);
            p2 = __fadd_rn(__fadd_rn(p2, __fmul_rn(lo, lo)), __fmul_rn(hi, hi));
            acc2.add(rs.apply(xx));
        }
    p1 = allreduce_add<P>(p1);
    p2 = allreduce_add<P>(p2);
    float t1h, t1l, t2h, t2l;
    acc2.lane_total(t1h, t1l, t2h, t2l);
    dd2_allreduce<P>(t1h, t1l, t2h, t2l);
    if (cls == kClassNonFinite) {
        mean = __fmul_rn(p1, inv_n);
        var = __fsub_rn(__fmul_rn(p2, inv_n), __fmul_rn(mean, mean));
    } else if (cls == kClassScaled) {
        float ms, vs;
        if ((RV & (RV - 1)) == 0)
            finalize_ln_pow2(t1h, t1l, t2h, t2l, kN, inv_n, ms, vs);
        else
            finalize_ln(t1h, t1l, t2h, t2l, kN, inv_n, ms, vs);
        mean = rs.unscale(ms, 1);
        var = rs.unscale(vs, 2);
    }
}

// mean and biased variance of each row of a tile (P lanes per row, V
// vectors per lane in registers; warp-uniform control flow).
template <int RV, int P>
__device__ __forceinline__ void qk_row_stats(const uint4 (&xv)[QkShape<RV, P>::kVecPerLane],
                                             float& mean, float& var)
{
    using Shape = QkShape<RV, P>;
    constexpr int V = Shape::kVecPerLane;
    constexpr int kL = Shape::kL;
    constexpr float kN = 8.0f * RV;
    const float inv_n = 1.0f / kN;
    const uint32_t mm = tree_absmax<V>(xv);
    ExactSums<true> acc;
    const uint32_t E = offset_exponent(mm);
    acc.init(offset_k1<kL>(E), offset_k2<kL>(E));
#pragma unroll
    for (int j = 0; j < V; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i)
            acc.add(f2_from_bf2(word(xv[j], i)));
    float s1h, s1l, s2h, s2l;
    acc.lane_total(s1h, s1l, s2h, s2l);
    dd2_allreduce<P>(s1h, s1l, s2h, s2l);

    // row class over its lanes
    uint32_t cls = allreduce_max<P>(static_cast<uint32_t>(magnitude_class(mm)));
    uint32_t emax = allreduce_max<P>(mm == 0 ? 0u : (mm >> 7));

    if ((RV & (RV - 1)) == 0)
        finalize_ln_pow2(s1h, s1l, s2h, s2l, kN, inv_n, mean, var);
    else
        finalize_ln(s1h, s1l, s2h, s2l, kN, inv_n, mean, var);
    if (__any_sync(kFullMask, cls != kClassFast))
        qk_slow_stats<RV, P>(xv, cls, emax, mean, var);
}

// ---------------------------------------------------------------------------
// Warp-specialised variant: statistics warps and output warps around a CTA
// ring of kSlots tiles fed by 1-D bulk copies (as the row kernels' ring).  A
// statistics warp forms the tile's per-row mean / rstd, leaves them beside
// the tile and arrives on the slot's "ready" barrier; an output warp applies
// the affine from the same slot and refills it with the tile kSlots ahead.
// kSlots is a multiple of both warp counts, so a slot always returns to the
// same two warps, which take their tiles in order.
// ---------------------------------------------------------------------------

constexpr int kWsStatWarps = 8;
constexpr int kWsOutWarps = 4;
constexpr int kWsThreads = 32 * (kWsStatWarps + kWsOutWarps);
constexpr int kWsSlots = 16;
static_assert(kWsSlots % kWsStatWarps == 0 && kWsSlots % kWsOutWarps == 0,
              "a slot must return to the same warps");

template <int RV, int P>
__global__ void __launch_bounds__(kWsThreads, 2)
    qk_kernel_ws(const QkArgs a, int blocks_q, FastDiv chunks_q, FastDiv chunks_k)
{
    using Shape = QkShape<RV, P>;
    constexpr int V = Shape::kVecPerLane;
    constexpr int kTileRows = Shape::kTileRows;
    constexpr int kTileVec = Shape::kTileVec;

    extern __shared__ __align__(128) uint4 ring[];
    __shared__ __align__(8) unsigned long long full_bar[kWsSlots], ready_bar[kWsSlots];
    __shared__ float2 tile_stats[kWsSlots][kTileRows];  // (mean, rstd) per row
    __shared__ __align__(16) float4 s_w[2][kMaxRowVec], s_b[2][kMaxRowVec];

    const bool is_q = static_cast<int>(blockIdx.x) < blocks_q;
    const QkTensor t = is_q ? a.t[0] : a.t[1];
    const int blk = is_q ? blockIdx.x : blockIdx.x - blocks_q;
    const int nblk = is_q ? blocks_q : gridDim.x - blocks_q;
    const uint4* __restrict__ src = static_cast<const uint4*>(t.in);
    uint4* __restrict__ dst = static_cast<uint4*>(t.out);
    const int64_t stat_off = is_q ? 0 : a.t[0].tokens * a.t[0].heads;
    const int64_t chunks = (t.heads + kTileRows - 1) / kTileRows;
    const int64_t tiles = t.tokens * chunks;
    const int64_t in_tv = t.in_ts / 8, out_tv = t.out_ts / 8;
    const bool one_token = t.tokens == 1;
    const bool small = tiles < (int64_t(1) << 32);
    // tile -> token: a multiply-shift division by the tiles per token (the
    // hardware has no integer divide; a plain division costs ~20 instructions
    // per tile, a sizeable share of a 16-row tile's statistics)
    const FastDiv cdiv = is_q ? chunks_q : chunks_k;
    auto token_of = [&](int64_t tile) -> int64_t {
        if (one_token)
            return 0;
        if (small)
            return cdiv.div(static_cast<uint32_t>(tile));
        return tile / chunks;
    };
    // this CTA's tiles: blk, blk + nblk, ...
    const int64_t n_local = blk < tiles ? (tiles - blk + nblk - 1) / nblk : 0;
    auto tile_of = [&](int64_t i) { return blk + i * nblk; };

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int sub = lane % P;
    const int rsub = lane / P;
    const int rot = rsub % V;

    if (threadIdx.x == 0) {
        for (int sl = 0; sl < kWsSlots; ++sl) {
            mbar_init(smem_addr(&full_bar[sl]), 1u);
            mbar_init(smem_addr(&ready_bar[sl]), 1u);
        }
        mbar_init_fence();
    }
    // only shared memory so far: the barriers are ready when the previous
    // grid's results become visible
    grid_dependency_sync();
    if (threadIdx.x < 2 * RV) {
        const uint4* __restrict__ wv = static_cast<const uint4*>(t.w);
        const uint4* __restrict__ bv = static_cast<const uint4*>(t.b);
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

    auto issue = [&](int64_t i) {  // one thread
        if (i >= n_local)
            return;
        const int64_t tile = tile_of(i);
        const int64_t tok = token_of(tile);
        const int64_t h0 = (tile - tok * chunks) * kTileRows;
        const int64_t left = t.heads - h0;
        const uint32_t bytes =
            static_cast<uint32_t>(left < kTileRows ? left : kTileRows) * (RV * 16u);
        const int sl = static_cast<int>(i % kWsSlots);
        const uint32_t bar = smem_addr(&full_bar[sl]);
        fence_proxy_async();
        mbar_expect_tx(bar, bytes);
        bulk_g2s(smem_addr(ring + sl * kTileVec), src + tok * in_tv + h0 * RV, bytes, bar);
    };
    bool broken = false;
    auto wait = [&](uint32_t bar, uint32_t parity) {
        if (!broken && !mbar_wait(bar, parity, kWaitLimitNs)) {
            broken = true;
            if (lane == 0)
                atomicOr(&g_error, kErrCopyTimeout);
        }
    };
    // half of the ring now, the other half as the first tiles land
    if (threadIdx.x == 0)
        for (int64_t i = 0; i < kWsStatWarps && i < n_local; ++i)
            issue(i);

    if (warp < kWsStatWarps) {
        for (int64_t i = warp; i < n_local; i += kWsStatWarps) {
            const int sl = static_cast<int>(i % kWsSlots);
            wait(smem_addr(&full_bar[sl]), static_cast<uint32_t>((i / kWsSlots) & 1));
            if (i + kWsStatWarps < kWsSlots && lane == 0)
                issue(i + kWsStatWarps);
            const int64_t tile = tile_of(i);
            const int64_t tok = token_of(tile);
            const int64_t h = (tile - tok * chunks) * kTileRows + rsub;
            const bool valid = h < t.heads;
            const uint4* tile_p = ring + sl * kTileVec + rsub * RV;
            uint4 xv[V];
#pragma unroll
            for (int j = 0; j < V; ++j) {
                const int jj = (j + rot) % V;
                xv[j] = valid ? tile_p[sub + P * jj] : make_uint4(0u, 0u, 0u, 0u);
            }
            float mean, var;
            qk_row_stats<RV, P>(xv, mean, var);
            const float rstd = rstd_from(var, a.eps);
            if (sub == 0) {
                tile_stats[sl][rsub] = make_float2(mean, rstd);
                if (valid) {
                    const int64_t row = tok * t.heads + h;
                    if (a.mean_out)
                        a.mean_out[stat_off + row] = mean;
                    if (a.rstd_out)
                        a.rstd_out[stat_off + row] = rstd;
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_addr(&ready_bar[sl]));
        }
    } else {
        const int ow = warp - kWsStatWarps;
        for (int64_t i = ow; i < n_local; i += kWsOutWarps) {
            const int sl = static_cast<int>(i % kWsSlots);
            wait(smem_addr(&ready_bar[sl]), static_cast<uint32_t>((i / kWsSlots) & 1));
            const int64_t tile = tile_of(i);
            const int64_t tok = token_of(tile);
            const int64_t h = (tile - tok * chunks) * kTileRows + rsub;
            if (h < t.heads) {
                const float2 st = tile_stats[sl][rsub];
                const u64 mean2 = f2_splat(st.x), rstd2 = f2_splat(st.y);
                const uint4* tile_p = ring + sl * kTileVec + rsub * RV;
                const int64_t base = tok * out_tv + h * RV;
#pragma unroll
                for (int j = 0; j < V; ++j) {
                    const int c = sub + P * ((j + rot) % V);
                    const uint4 xvj = tile_p[c];
                    const float4 w_lo = s_w[0][c], w_hi = s_w[1][c];
                    const float4 b_lo = s_b[0][c], b_hi = s_b[1][c];
                    const u64 w2[4] = {f2_pack(w_lo.x, w_lo.y), f2_pack(w_lo.z, w_lo.w),
                                       f2_pack(w_hi.x, w_hi.y), f2_pack(w_hi.z, w_hi.w)};
                    const u64 b2[4] = {f2_pack(b_lo.x, b_lo.y), f2_pack(b_lo.z, b_lo.w),
                                       f2_pack(b_hi.x, b_hi.y), f2_pack(b_hi.z, b_hi.w)};
                    uint4 o;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const u64 xx = f2_from_bf2(word(xvj, q));
                        const u64 z =
                            f2_mul_then_add(f2_mul(f2_sub(xx, mean2), rstd2), w2[q], b2[q]);
                        word(o, q) = bf2_from_f2(z);
                    }
                    st_stream(dst + base + c, o);
                }
            }
            // the tile is consumed: refill its slot with the tile kSlots ahead
            __syncwarp();
            if (lane == 0)
                issue(i + kWsSlots);
        }
    }
    if (broken)
        drain_pause();
}

template <int RV, int P>
cudaError_t launch_ws(const QkArgs& a, const DeviceInfo& dev, cudaStream_t stream)
{
    using Shape = QkShape<RV, P>;
    auto kern = qk_kernel_ws<RV, P>;
    constexpr int kSmem = kWsSlots * Shape::kTileVec * 16;
    static PerDeviceInt blocks_per_sm;
    int bps = 0;
    {
        const cudaError_t e0 = blocks_per_sm.get(dev.device, bps, [&](int& v) -> cudaError_t {
            cudaError_t e =
                cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
            if (e != cudaSuccess)
                return e;
            int nb = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, kWsThreads, kSmem);
            if (e != cudaSuccess)
                return e;
            v = nb > 0 ? nb : 1;
            return cudaSuccess;
        });
        if (e0 != cudaSuccess)
            return e0;
    }
    auto tiles_of = [](const QkTensor& t) {
        return t.tokens * ((t.heads + Shape::kTileRows - 1) / Shape::kTileRows);
    };
    const int64_t tq = tiles_of(a.t[0]), tk = tiles_of(a.t[1]);
    const int64_t total = tq + tk;
    const int64_t cap = static_cast<int64_t>(dev.sms) * bps;
    int64_t bq, bk;
    if (tq + tk <= cap) {
        bq = tq;
        bk = tk;
    } else {
        bq = (cap * tq + total / 2) / total;
        if (tq > 0 && bq < 1)
            bq = 1;
        if (tk > 0 && cap - bq < 1)
            bq = cap - 1;
        bk = cap - bq;
    }
    const int grid = static_cast<int>(bq + bk);
    // tiles per token of q and of k (at least 1; used only when it fits 32 bits)
    auto chunks_of = [](const QkTensor& t) {
        const int64_t c = (t.heads + Shape::kTileRows - 1) / Shape::kTileRows;
        return FastDiv::make(static_cast<uint32_t>(c > 0 && c < (int64_t(1) << 31) ? c : 1));
    };
    return launch_dependent(kern, grid, kWsThreads, kSmem, stream, a, static_cast<int>(bq),
                            chunks_of(a.t[0]), chunks_of(a.t[1]));
}

}  // namespace

// head_dim 64: one lane per row (8 vectors); 96 and 128: two lanes per row.
cudaError_t launch_qk_kernel(const QkArgs& a, const DeviceInfo& dev, cudaStream_t stream)
{
    switch (a.head_dim) {
    case 64:
        return launch_ws<8, 1>(a, dev, stream);
    case 96:
        return launch_ws<12, 2>(a, dev, stream);
    default:
        return launch_ws<16, 2>(a, dev, stream);
    }
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
