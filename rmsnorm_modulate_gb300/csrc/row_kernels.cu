// ln_modulate / rmsnorm_modulate / gated_rmsnorm_modulate on sm_103a.
//
// Two kernels, both fed by 1-D bulk copies (TMA, cp.async.bulk) into shared
// memory tracked by mbarriers, so HBM sees a continuous stream independent of
// how long the arithmetic takes:
//   row_kernel     (D <= 2048, D > 4096, and gated rows up to 3072) one warp (or a
//                  group of 2 / 4 warps for D > 4096, each owning a contiguous
//                  segment of the row) processes one row at a time from a
//                  two-stage ring of its own and loops persistently over rows.
//   row_kernel_ws  (2048 < D <= 4096) warp-specialised: statistics warps and
//                  output warps around one ring of row slots per CTA; a
//                  statistics warp forms a row's mean / rstd and hands the
//                  slot to the output warps, which normalise, modulate, store
//                  and refill it.
// The exact statistics are formed from packed bf16, the normalise + modulate
// epilogue runs on packed f32x2 / bf16x2 instructions and streams the result
// out.  HBM is touched once per element in each direction; scale, shift,
// weight and gate rows are staged once per work item in shared memory (rows
// of up to 4096 values) or re-read from L1/L2 (longer rows).
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

// This translation unit's error word (see kErr* in device_common.cuh).
__device__ unsigned int g_error;

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

// Statistics of a row that holds Inf/NaN (plain IEEE sums, which propagate
// them the way the exact double sums do) or extreme magnitudes (scaled to
// unit size by a power of two, exact sums, scaled back).  Group-uniform.
template <bool kNeedSum, int V, int WPR, int kL>
__device__ __noinline__ void slow_stats(const uint4 (&xv)[V], uint32_t cls, uint32_t emax,
                                        Slot* slots, int wig, int lane, int group, float n,
                                        float inv_n, float& mean, float& stat)
{
    if (cls == kClassNonFinite) {
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
        group_sum_plain<WPR>(slots, wig, lane, group, p1, p2);
        mean = __fmul_rn(p1, inv_n);
        const float msq = __fmul_rn(p2, inv_n);
        stat = kNeedSum ? __fsub_rn(msq, __fmul_rn(mean, mean)) : msq;
        return;
    }
    RowScale rs;
    rs.set(emax);
    ExactSums<kNeedSum> acc2;
    acc2.init(offset_k1<kL>(127u), offset_k2<kL>(127u));
#pragma unroll
    for (int j = 0; j < V; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i)
            acc2.add(rs.apply(f2_from_bf2(word(xv[j], i))));
    float s1h, s1l, s2h, s2l;
    acc2.lane_total(s1h, s1l, s2h, s2l);
    if (kNeedSum)
        dd2_allreduce<32>(s1h, s1l, s2h, s2l);
    else
        dd_allreduce<32>(s2h, s2l);
    uint32_t c2 = cls, e2 = emax;
    group_combine<WPR>(slots, wig, lane, group, s1h, s1l, s2h, s2l, c2, e2);
    group_barrier<WPR>(group);
    if (kNeedSum) {
        float ms, vs;
        finalize_ln(s1h, s1l, s2h, s2l, n, inv_n, ms, vs);
        mean = rs.unscale(ms, 1);
        stat = rs.unscale(vs, 2);
    } else {
        mean = 0.0f;
        stat = rs.unscale(finalize_ms(s2h, s2l, n, inv_n), 2);
    }
}

// Compile-time shape of one kernel instance.
template <int OP, int V, int WPR>
struct RowShape {
    static constexpr int kStages = V >= 8 ? 1 : 2;  // rows in flight per warp
    static constexpr int kNbuf = (OP == kOpGated) ? 2 : 1;   // residual + update
    static constexpr int kSegVec = 32 * V;                   // 16-byte vectors per buffer
    static constexpr int kWarpBytes = kStages * kNbuf * kSegVec * 16;
    // Rows of up to 4096 values keep the per-row re-read vectors in shared
    // memory: R(1 + scale) and shift, plus weight (RMS) and gate (gated).
    static constexpr bool kCached = 32 * V * WPR <= 512;
    static constexpr int kNmod = (OP == kOpLN || OP == kOpLNFold) ? 2 : (OP == kOpRMS ? 3 : 4);
    static constexpr int kCacheBytes = kCached ? kNmod * 32 * V * WPR * 16 : 0;
    // as many warps as ~108 KB per CTA allows, a multiple of WPR; at most 8,
    // or 6 for the larger per-lane rows so three CTAs per SM keep ~110
    // registers per thread
    // registers bound the resident rows: 8 warps x 2 CTAs (128 registers) up
    // to 12 vectors per lane, 6 warps x 2 CTAs (170) for 16
    static constexpr int kMaxWarps = V >= 16 ? 6 : 8;
    static constexpr int kFit = (108 * 1024 - kCacheBytes) / kWarpBytes;
    static constexpr int kWarps0 = kFit > kMaxWarps ? kMaxWarps : (kFit < 1 ? 1 : kFit);
    static constexpr int kWarps = (kWarps0 / WPR) * WPR < WPR ? WPR : (kWarps0 / WPR) * WPR;
    static constexpr int kThreads = 32 * kWarps;
    static constexpr int kRingBytes = kWarps * kWarpBytes;
    // CTAs per SM the shared memory allows (the register budget follows it)
    static constexpr int kSmemPerCta = kRingBytes + kCacheBytes + 2048;
    static constexpr int kBlocks0 = (224 * 1024) / kSmemPerCta;
    static constexpr int kBlockCap = V >= 8 ? 2 : 3;
    static constexpr int kBlocks = kBlocks0 > kBlockCap ? kBlockCap : (kBlocks0 < 1 ? 1 : kBlocks0);
};

// out = R(R(y * s1) + shift) for one 16-byte vector, y from x and the row's
// statistics: the normalise step and the modulate chain (or, for the folded
// tier, the single-rounding affine with weight s1 and bias shift).
template <int OP>
__device__ __forceinline__ uint4 normalise_modulate(const uint4& xv, u64 mean2, u64 rstd2,
                                                    const uint4& s1, const uint4& sh,
                                                    const uint4& w, bool has_w)
{
    uint4 o;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const u64 xx = f2_from_bf2(word(xv, i));
        u64 y;
        if (OP == kOpLNFold) {
            // one rounding: R(((x - mean) * rstd) * f(s1) + f(shift)), the
            // multiply and the add rounded separately
            const u64 yn = f2_mul(f2_sub(xx, mean2), rstd2);
            word(o, i) = bf2_from_f2(
                f2_mul_then_add(yn, f2_from_bf2(word(s1, i)), f2_from_bf2(word(sh, i))));
            continue;
        }
        if (OP == kOpLN) {
            y = f2_mul(f2_sub(xx, mean2), rstd2);
        } else {
            y = f2_mul(xx, rstd2);
            if (has_w)
                y = f2_mul(y, f2_from_bf2(word(w, i)));
        }
        word(o, i) = bf2_add(bf2_mul(bf2_from_f2(y), word(s1, i)), word(sh, i));
    }
    return o;
}

// Work is split into items: a contiguous range of rows of one batch, so an
// item needs one set of modulation rows.  A CTA takes items blockIdx.x,
// blockIdx.x + gridDim.x, ...; its row groups take the item's rows in turn.
struct Items {
    int64_t per_batch;  // items per batch
    int64_t chunk;      // rows per item (the last item of a batch may be shorter)
    int64_t count;
};

// EXACT: every warp segment is exactly 32 * V vectors (D = 256 * V * WPR),
// so no vector needs a bounds check.
template <int OP, int V, int WPR, bool EXACT>
__global__ void __launch_bounds__(RowShape<OP, V, WPR>::kThreads, RowShape<OP, V, WPR>::kBlocks)
    row_kernel(const RowArgs a, const Items items)
{
    grid_dependency_sync();
    using Shape = RowShape<OP, V, WPR>;
    constexpr int kWarps = Shape::kWarps;
    constexpr int kGroups = kWarps / WPR;
    constexpr int kStages = Shape::kStages;
    constexpr int kNbuf = Shape::kNbuf;
    constexpr int kSegVec = Shape::kSegVec;
    constexpr bool kCached = Shape::kCached;
    constexpr int kL = Log2Ceil<8 * V>::value;
    constexpr bool kNeedSum = (OP == kOpLN || OP == kOpLNFold);
    constexpr bool kWeighted = (OP == kOpRMS || OP == kOpGated);

    extern __shared__ __align__(128) uint4 ring[];
    __shared__ __align__(8) unsigned long long bars[kWarps][kStages];
    __shared__ Slot slots[2][kGroups][WPR];
    __shared__ Slot slow_slots[kGroups][WPR];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int group = warp / WPR;
    const int wig = warp % WPR;
    const int Dv = a.Dv;
    // this warp's contiguous segment of every row
    const int seg = (Dv + WPR - 1) / WPR;
    const int s0 = wig * seg;
    int seg_len = Dv - s0;
    seg_len = seg_len > seg ? seg : (seg_len < 0 ? 0 : seg_len);
    const uint32_t seg_bytes = static_cast<uint32_t>(seg_len) * 16u;

    const uint4* __restrict__ src0 =
        static_cast<const uint4*>(OP == kOpGated ? a.residual : a.x);
    const uint4* __restrict__ src1 = static_cast<const uint4*>(a.update);
    const uint4* __restrict__ gate = static_cast<const uint4*>(a.gate);
    const uint4* __restrict__ weight = static_cast<const uint4*>(a.weight);
    const uint4* __restrict__ scale = static_cast<const uint4*>(a.scale);
    const uint4* __restrict__ shift = static_cast<const uint4*>(a.shift);
    uint4* __restrict__ res_out = static_cast<uint4*>(a.res_out);
    uint4* __restrict__ out = static_cast<uint4*>(a.out);
    const bool has_w = (weight != nullptr);

    // modulation rows of the current item's batch (kCached only)
    uint4* cache = ring + Shape::kRingBytes / 16;
    uint4* c_s1 = cache;
    uint4* c_sh = cache + Dv;
    uint4* c_w = cache + 2 * Dv;
    uint4* c_g = cache + 3 * Dv;

    uint4* wbuf = ring + static_cast<size_t>(warp) * kStages * kNbuf * kSegVec;
    const uint32_t bar0 = smem_addr(&bars[warp][0]);
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < kStages; ++s)
            mbar_init(bar0 + 8u * s, 1u);
        mbar_init_fence();
    }
    __syncwarp();

    bool broken = false;  // a copy timed out: keep going (barriers stay matched), skip waits
    int parity = 0;
    int64_t uses = 0;     // rows this warp has run through its ring

    for (int64_t item = blockIdx.x; item < items.count; item += gridDim.x) {
        const int64_t b = item / items.per_batch;
        const int64_t r_begin = b * a.S + (item % items.per_batch) * items.chunk;
        const int64_t r_lim = (b + 1) * a.S;
        const int64_t r_end = r_begin + items.chunk < r_lim ? r_begin + items.chunk : r_lim;

        // lane 0 starts the copy of this group's k-th row of the item into
        // its ring (use counter uses + k)
        auto issue = [&](int64_t k) {
            const int64_t row = r_begin + group + k * kGroups;
            if (lane != 0 || row >= r_end)
                return;
            const int st = static_cast<int>((uses + k) % kStages);
            const uint32_t bar = bar0 + 8u * st;
            fence_proxy_async();
            mbar_expect_tx(bar, kNbuf * seg_bytes);
            if (seg_bytes) {
                const uint32_t dst = smem_addr(wbuf + st * kNbuf * kSegVec);
                bulk_g2s(dst, src0 + row * Dv + s0, seg_bytes, bar);
                if (kNbuf == 2)
                    bulk_g2s(dst + kSegVec * 16u, src1 + row * Dv + s0, seg_bytes, bar);
            }
        };
#pragma unroll
        for (int k = 0; k < kStages; ++k)
            issue(k);

        if (kCached) {
            __syncthreads();  // every group is done with the previous item's rows
            for (int c = threadIdx.x; c < Dv; c += blockDim.x) {
                c_s1[c] = bf2x4_add(ld_cached(scale + b * a.mod_bstride + c), kBf2One);
                c_sh[c] = ld_cached(shift + b * a.mod_bstride + c);
                if (kWeighted && has_w)
                    c_w[c] = ld_cached(weight + c);
                if (OP == kOpGated)
                    c_g[c] = ld_cached(gate + b * a.gate_bstride + c);
            }
            __syncthreads();
        }

        int64_t k = 0;
        for (int64_t row = r_begin + group; row < r_end; row += kGroups, ++k, parity ^= 1) {
            const int st = static_cast<int>((uses + k) % kStages);
            const uint32_t phase = static_cast<uint32_t>(((uses + k) / kStages) & 1);
            if (!broken && !mbar_wait(bar0 + 8u * st, phase, kWaitLimitNs)) {
                broken = true;
                if (lane == 0)
                    atomicOr(&g_error, kErrCopyTimeout);
            }
            const uint4* b0 = wbuf + st * kNbuf * kSegVec;
            const int64_t base = row * Dv + s0;

            // ---- shared -> registers (and for the gated op, form and store
            //      the residual stream)
            uint4 xv[V];
#pragma unroll
            for (int j = 0; j < V; ++j) {
                const int v = j * 32 + lane;
                if (EXACT || v < seg_len) {
                    if (OP == kOpGated) {
                        const uint4 r = b0[v];
                        const uint4 u = b0[kSegVec + v];
                        const uint4 g = kCached ? c_g[s0 + v]
                                                : ld_cached(gate + b * a.gate_bstride + s0 + v);
                        uint4 s;
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            word(s, i) = bf2_add(word(r, i), bf2_mul(word(g, i), word(u, i)));
                        st_stream(res_out + base + v, s);
                        xv[j] = s;
                    } else {
                        xv[j] = b0[v];
                    }
                } else {
                    xv[j] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            // the stage is consumed: refill it with the row kStages ahead
            __syncwarp();
            issue(k + kStages);

            // ---- magnitude class of this lane's values
            const uint32_t mm = tree_absmax<V>(xv);
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
            uint32_t cls =
                __reduce_max_sync(kFullMask, static_cast<uint32_t>(magnitude_class(mm)));
            uint32_t emax = __reduce_max_sync(kFullMask, mm == 0 ? 0u : (mm >> 7));
            group_combine<WPR>(&slots[parity][group][0], wig, lane, group, s1h, s1l, s2h, s2l,
                               cls, emax);

            float mean = 0.0f, stat;
            if (cls == kClassFast) {
                if (kNeedSum)
                    finalize_ln(s1h, s1l, s2h, s2l, a.n, a.inv_n, mean, stat);
                else
                    stat = finalize_ms(s2h, s2l, a.n, a.inv_n);
            } else {
                slow_stats<kNeedSum, V, WPR, kL>(xv, cls, emax, &slow_slots[group][0], wig, lane,
                                                 group, a.n, a.inv_n, mean, stat);
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
#pragma unroll
            for (int j = 0; j < V; ++j) {
                const int v = j * 32 + lane;
                if (EXACT || v < seg_len) {
                    uint4 s1, h, w = make_uint4(0u, 0u, 0u, 0u);
                    if (kCached) {
                        s1 = c_s1[s0 + v];
                        h = c_sh[s0 + v];
                        if (kWeighted && has_w)
                            w = c_w[s0 + v];
                    } else {
                        s1 = bf2x4_add(ld_cached(scale + b * a.mod_bstride + s0 + v), kBf2One);
                        h = ld_cached(shift + b * a.mod_bstride + s0 + v);
                        if (kWeighted && has_w)
                            w = ld_cached(weight + s0 + v);
                    }
                    st_stream(out + base + v,
                              normalise_modulate<OP>(xv[j], mean2, rstd2, s1, h, w, has_w));
                }
            }
        }
        uses += k;
    }
    // nothing is left in flight on the normal path (every issued row was
    // waited for); after a timeout, give outstanding copies a bounded time
    // to land before the CTA's shared memory is released
    if (broken)
        drain_pause();
}

// ---------------------------------------------------------------------------
// Warp-specialised variant for one warp per row (LN / RMS / folded LN,
// 2048 < D <= 4096).  The CTA owns a ring of kSlots row buffers fed by 1-D
// bulk copies.  Statistics warps take rows in turn, read a row from shared
// memory once into registers (its abs-max on the way), then run the exact
// sums, butterfly, finalisation and rstd from registers, leave mean / rstd
// beside the row and arrive on the slot's "ready" barrier;
// output warps wait for it, normalise + modulate the row from the same
// buffer, store it, and refill the slot with the row kSlots ahead.  The
// latency-bound reductions of some rows thus overlap the FMA-bound epilogue
// of others instead of running in lock-step phases.
// ---------------------------------------------------------------------------

// Rows up to 3072 values: 8 statistics + 4 output warps, two CTAs per SM;
// with SHORT work items (16 rows or fewer per CTA, where the output warps'
// last rows set the end of the launch) 4 + 8.  4096 values: 8 + 8 warps and
// one CTA per SM with a 176 KB ring (the epilogue's share of the work grows
// with the weight row of RMSNorm); gated, whose slots hold two rows and
// whose statistics warps also write the residual stream out, 4 + 8 warps
// around 8 slots (128 KB).  At 4096 values two output warps share each row
// (half of its vectors each; the later of the two refills the slot), which
// halves the epilogue latency of a CTA's last rows.
template <int OP, int V, bool SHORT = false>
struct WsShape {
    static constexpr bool kGatedWide = (V >= 16 && OP == kOpGated);
    static constexpr int kStatWarps = kGatedWide ? 4 : ((V < 16 && SHORT) ? 4 : 8);
    static constexpr int kOutWarps = kGatedWide ? 8 : ((V >= 16 || SHORT) ? 8 : 4);
    static constexpr int kBlocks = V >= 16 ? 1 : 2;
    static constexpr int kRingBudget = (kGatedWide ? 192 : (V >= 16 ? 176 : 100)) * 1024;
    static constexpr int kOutGroup = V >= 16 ? 2 : 1;  // output warps sharing one row
    static constexpr int kOutGroups = kOutWarps / kOutGroup;
    static_assert(kOutWarps % kOutGroup == 0 && V % kOutGroup == 0, "output groups");
    static constexpr int kWarps = kStatWarps + kOutWarps;
    static constexpr int kThreads = 32 * kWarps;
    static constexpr int kSegVec = 32 * V;
    static constexpr int kNbuf = (OP == kOpGated) ? 2 : 1;  // residual + update
    static constexpr int kSlotVec = kNbuf * kSegVec;
    static constexpr int kNmod = (OP == kOpLN || OP == kOpLNFold) ? 2 : (OP == kOpRMS ? 3 : 4);
    static constexpr int kCacheBytes = kNmod * 32 * V * 16;
    // Rows r and r + kSlots share a slot; with kSlots a multiple of both warp
    // counts they also share their statistics warp and their output warp,
    // which take their rows in order, so no barrier is ever waited on with
    // the parity of a phase two steps ahead (which would read as complete).
    static constexpr int kSlotsRaw = kRingBudget / (kSlotVec * 16);
    static constexpr int kSlotStep = kGatedWide ? 8 : kStatWarps;  // a multiple of both
    static constexpr int kSlots = kSlotsRaw / kSlotStep * kSlotStep;
    static constexpr int kRingBytes = kSlots * kSlotVec * 16;
    static_assert(kSlots >= kStatWarps && kSlots % kStatWarps == 0 && kSlots % kOutGroups == 0,
                  "a slot must return to the same statistics and output warps");
};

// Statistics of a non-fast row (see slow_stats) streamed from its buffer.
template <bool kNeedSum, int V, int kL, bool EXACT>
__device__ __noinline__ void slow_stats_smem(const uint4* buf, int Dv, uint32_t cls,
                                             uint32_t emax, int lane, float n, float inv_n,
                                             float& mean, float& stat)
{
    if (cls == kClassNonFinite) {
        float p1 = 0.0f, p2 = 0.0f;
        for (int j = 0; j < V; ++j) {
            const int v = j * 32 + lane;
            const uint4 xv = (EXACT || v < Dv) ? buf[v] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float lo, hi;
                f2_unpack(f2_from_bf2(word(xv, i)), lo, hi);
                p1 = __fadd_rn(__fadd_rn(p1, lo), hi);
                p2 = __fadd_rn(__fadd_rn(p2, __fmul_rn(lo, lo)), __fmul_rn(hi, hi));
            }
        }
        p1 = allreduce_add<32>(p1);
        p2 = allreduce_add<32>(p2);
        mean = __fmul_rn(p1, inv_n);
        const float msq = __fmul_rn(p2, inv_n);
        stat = kNeedSum ? __fsub_rn(msq, __fmul_rn(mean, mean)) : msq;
        return;
    }
    RowScale rs;
    rs.set(emax);
    ExactSums<kNeedSum> acc;
    acc.init(offset_k1<kL>(127u), offset_k2<kL>(127u));
    for (int j = 0; j < V; ++j) {
        const int v = j * 32 + lane;
        const uint4 xv = (EXACT || v < Dv) ? buf[v] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            acc.add(rs.apply(f2_from_bf2(word(xv, i))));
    }
    float s1h, s1l, s2h, s2l;
    acc.lane_total(s1h, s1l, s2h, s2l);
    if (kNeedSum) {
        dd2_allreduce<32>(s1h, s1l, s2h, s2l);
        float ms, vs;
        finalize_ln(s1h, s1l, s2h, s2l, n, inv_n, ms, vs);
        mean = rs.unscale(ms, 1);
        stat = rs.unscale(vs, 2);
    } else {
        dd_allreduce<32>(s2h, s2l);
        mean = 0.0f;
        stat = rs.unscale(finalize_ms(s2h, s2l, n, inv_n), 2);
    }
}

// One arrival on a shared-memory counter, ordered after this thread's
// earlier shared-memory reads (acquire-release at CTA scope); returns the
// count before it.
__device__ __forceinline__ uint32_t release_add_smem(uint32_t addr)
{
    uint32_t old;
    asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], 1;"
                 : "=r"(old)
                 : "r"(addr)
                 : "memory");
    return old;
}

template <int OP, int V, bool EXACT, bool SHORT>
__global__ void __launch_bounds__(WsShape<OP, V, SHORT>::kThreads, WsShape<OP, V, SHORT>::kBlocks)
    row_kernel_ws(const RowArgs a, const Items items)
{
    using Shape = WsShape<OP, V, SHORT>;
    constexpr int kSlots = Shape::kSlots;
    constexpr int kSegVec = Shape::kSegVec;
    constexpr int kSlotVec = Shape::kSlotVec;
    constexpr int kStatWarps = Shape::kStatWarps;
    constexpr int kL = Log2Ceil<8 * V>::value;
    constexpr bool kNeedSum = (OP == kOpLN || OP == kOpLNFold);
    constexpr bool kWeighted = (OP == kOpRMS || OP == kOpGated);

    extern __shared__ __align__(128) uint4 ring[];
    __shared__ __align__(8) unsigned long long full_bar[kSlots], ready_bar[kSlots];
    __shared__ float2 slot_stats[kSlots];  // (mean, rstd) of the row in each slot
    __shared__ uint32_t consumed[kSlots];  // output-warp releases of each slot, cumulative

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int Dv = a.Dv;
    const uint32_t row_bytes = static_cast<uint32_t>(Dv) * 16u;

    const uint4* __restrict__ src = static_cast<const uint4*>(OP == kOpGated ? a.residual : a.x);
    const uint4* __restrict__ src1 = static_cast<const uint4*>(a.update);
    const uint4* __restrict__ gate = static_cast<const uint4*>(a.gate);
    uint4* __restrict__ res_out = static_cast<uint4*>(a.res_out);
    const uint4* __restrict__ weight = static_cast<const uint4*>(a.weight);
    const uint4* __restrict__ scale = static_cast<const uint4*>(a.scale);
    const uint4* __restrict__ shift = static_cast<const uint4*>(a.shift);
    uint4* __restrict__ out = static_cast<uint4*>(a.out);
    const bool has_w = (weight != nullptr);

    uint4* cache = ring + Shape::kRingBytes / 16;
    uint4* c_s1 = cache;
    uint4* c_sh = cache + Dv;
    uint4* c_w = cache + 2 * Dv;
    uint4* c_g = cache + 3 * Dv;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(smem_addr(&full_bar[s]), 1u);
            mbar_init(smem_addr(&ready_bar[s]), 1u);
            consumed[s] = 0u;
        }
        mbar_init_fence();
    }
    __syncthreads();
    // only shared memory so far: the barriers are ready when the previous
    // grid's results become visible
    grid_dependency_sync();

    bool broken = false;
    int64_t uses = 0;  // rows the CTA has run through its ring

    for (int64_t item = blockIdx.x; item < items.count; item += gridDim.x) {
        const int64_t b = item / items.per_batch;
        const int64_t r_begin = b * a.S + (item % items.per_batch) * items.chunk;
        const int64_t r_lim = (b + 1) * a.S;
        const int64_t r_end = r_begin + items.chunk < r_lim ? r_begin + items.chunk : r_lim;
        const int64_t nrows = r_end > r_begin ? r_end - r_begin : 0;

        auto slot_of = [&](int64_t r) { return static_cast<int>((uses + r) % kSlots); };
        auto parity_of = [&](int64_t r) {
            return static_cast<uint32_t>(((uses + r) / kSlots) & 1);
        };
        auto issue = [&](int64_t r) {  // one thread
            if (r >= nrows)
                return;
            const int s = slot_of(r);
            const uint32_t bar = smem_addr(&full_bar[s]);
            fence_proxy_async();
            mbar_expect_tx(bar, Shape::kNbuf * row_bytes);
            bulk_g2s(smem_addr(ring + s * kSlotVec), src + (r_begin + r) * Dv, row_bytes, bar);
            if (OP == kOpGated)
                bulk_g2s(smem_addr(ring + s * kSlotVec + kSegVec), src1 + (r_begin + r) * Dv,
                         row_bytes, bar);
        };
        auto wait = [&](uint32_t bar, uint32_t parity) {
            if (!broken && !mbar_wait(bar, parity, kWaitLimitNs)) {
                broken = true;
                if (lane == 0)
                    atomicOr(&g_error, kErrCopyTimeout);
            }
        };

        // the first row of every statistics warp now; the rest of the ring
        // once those have landed, so the first rows arrive as early as they can
        if (threadIdx.x == 0)
            for (int64_t r = 0; r < kStatWarps && r < nrows; ++r)
                issue(r);
        for (int c = threadIdx.x; c < Dv; c += blockDim.x) {
            c_s1[c] = bf2x4_add(ld_cached(scale + b * a.mod_bstride + c), kBf2One);
            c_sh[c] = ld_cached(shift + b * a.mod_bstride + c);
            if (kWeighted && has_w)
                c_w[c] = ld_cached(weight + c);
            if (OP == kOpGated)
                c_g[c] = ld_cached(gate + b * a.gate_bstride + c);
        }
        __syncthreads();

        if (warp < kStatWarps) {
            // ---- statistics warps
            for (int64_t r = warp; r < nrows; r += kStatWarps) {
                const int s = slot_of(r);
                wait(smem_addr(&full_bar[s]), parity_of(r));
                if (r + kStatWarps < kSlots && lane == 0)
                    issue(r + kStatWarps);  // the ring's second half, once
                uint4* buf = ring + s * kSlotVec;
                uint32_t m = 0;
                uint4 xr[V];  // the lane's vectors, for the sums pass
#pragma unroll
                for (int j = 0; j < V; ++j) {
                    const int v = j * 32 + lane;
                    xr[j] = make_uint4(0u, 0u, 0u, 0u);
                    if (EXACT || v < Dv) {
                        uint4 xv = buf[v];
                        if (OP == kOpGated) {
                            // the residual stream res = R(residual + R(gate * update)):
                            // written out, and over the residual in the slot for
                            // the statistics and the output warp
                            const uint4 u = buf[kSegVec + v], g = c_g[v];
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                word(xv, i) = bf2_add(word(xv, i), bf2_mul(word(g, i), word(u, i)));
                            buf[v] = xv;
                            st_stream(res_out + (r_begin + r) * Dv + v, xv);
                        }
                        xr[j] = xv;
                        m = bf2_absmax(m, bf2_absmax(bf2_absmax(xv.x, xv.y),
                                                     bf2_absmax(xv.z, xv.w)));
                    }
                }
                if (OP == kOpGated)
                    fence_proxy_async();  // res written over the slot, which the
                                          // async proxy refills later
                const uint32_t mm = absmax_bits(m);
                const uint32_t E = offset_exponent(mm);
                ExactSums<kNeedSum> acc;
                acc.init(offset_k1<kL>(E), offset_k2<kL>(E));
#pragma unroll
                for (int j = 0; j < V; ++j) {
                    const int v = j * 32 + lane;
                    if (EXACT || v < Dv) {
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            acc.add(f2_from_bf2(word(xr[j], i)));
                    }
                }
                float s1h, s1l, s2h, s2l;
                acc.lane_total(s1h, s1l, s2h, s2l);
                if (kNeedSum)
                    dd2_allreduce<32>(s1h, s1l, s2h, s2l);
                else
                    dd_allreduce<32>(s2h, s2l);
                const uint32_t cls =
                    __reduce_max_sync(kFullMask, static_cast<uint32_t>(magnitude_class(mm)));
                const uint32_t emax = __reduce_max_sync(kFullMask, mm == 0 ? 0u : (mm >> 7));
                float mean = 0.0f, stat;
                if (cls == kClassFast) {
                    if (kNeedSum)
                        finalize_ln(s1h, s1l, s2h, s2l, a.n, a.inv_n, mean, stat);
                    else
                        stat = finalize_ms(s2h, s2l, a.n, a.inv_n);
                } else {
                    slow_stats_smem<kNeedSum, V, kL, EXACT>(buf, Dv, cls, emax, lane, a.n,
                                                            a.inv_n, mean, stat);
                }
                const float rstd = rstd_from(stat, a.eps);
                if (lane == 0) {
                    const int64_t row = r_begin + r;
                    if (a.mean_out)
                        a.mean_out[row] = mean;
                    if (a.rstd_out)
                        a.rstd_out[row] = rstd;
                    slot_stats[s] = make_float2(mean, rstd);
                    mbar_arrive(smem_addr(&ready_bar[s]));
                }
                __syncwarp();
            }
        } else {
            // ---- output warps
            const int ow = warp - kStatWarps;
            constexpr int kG = Shape::kOutGroup;
            constexpr int kVG = V / kG;
            const int grp = ow / kG, q = ow - grp * kG;
            for (int64_t r = grp; r < nrows; r += Shape::kOutGroups) {
                const int s = slot_of(r);
                wait(smem_addr(&ready_bar[s]), parity_of(r));
                const float2 st = slot_stats[s];
                const uint4* buf = ring + s * kSlotVec;
                const int64_t base = (r_begin + r) * Dv;
                const u64 mean2 = f2_splat(st.x), rstd2 = f2_splat(st.y);
#pragma unroll
                for (int j = q * kVG; j < (q + 1) * kVG; ++j) {
                    const int v = j * 32 + lane;
                    if (EXACT || v < Dv) {
                        const uint4 w =
                            (kWeighted && has_w) ? c_w[v] : make_uint4(0u, 0u, 0u, 0u);
                        st_stream(out + base + v, normalise_modulate<OP>(buf[v], mean2, rstd2,
                                                                         c_s1[v], c_sh[v], w,
                                                                         has_w));
                    }
                }
                // this warp's part of the slot is consumed (its statistics
                // warp finished reading before it arrived); the last warp of
                // the group to finish refills it with the row kSlots ahead
                __syncwarp();
                if (lane == 0) {
                    if constexpr (kG == 1) {
                        issue(r + kSlots);
                    } else {
                        const uint32_t old = release_add_smem(smem_addr(&consumed[s]));
                        const uint32_t round = static_cast<uint32_t>((uses + r) / kSlots);
                        if (old + 1u == static_cast<uint32_t>(kG) * (round + 1u))
                            issue(r + kSlots);
                    }
                }
            }
        }
        uses += nrows;
        __syncthreads();  // the ring and the cache are free for the next item
    }
    if (broken)
        drain_pause();
}

template <int OP, int V, bool EXACT, bool SHORT>
cudaError_t launch_ws(const RowArgs& a, const DeviceInfo& dev, cudaStream_t stream)
{
    using Shape = WsShape<OP, V, SHORT>;
    auto kern = row_kernel_ws<OP, V, EXACT, SHORT>;
    constexpr int kSmemMax = Shape::kRingBytes + Shape::kCacheBytes;
    static PerDeviceInt blocks_per_sm;
    int bps = 0;
    {
        const cudaError_t e0 = blocks_per_sm.get(dev.device, bps, [&](int& v) -> cudaError_t {
            cudaError_t e =
                cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
            if (e != cudaSuccess)
                return e;
            int n = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, Shape::kThreads, kSmemMax);
            if (e != cudaSuccess)
                return e;
            v = n > 0 ? n : 1;
            return cudaSuccess;
        });
        if (e0 != cudaSuccess)
            return e0;
    }
    const int64_t cap = static_cast<int64_t>(dev.sms) * bps;
    const int64_t B = a.rows / a.S;
    int64_t per_batch = cap / (B > 0 ? B : 1);
    const int64_t max_items = (a.S + Shape::kStatWarps - 1) / Shape::kStatWarps;
    if (per_batch > max_items)
        per_batch = max_items;
    if (per_batch < 1)
        per_batch = 1;
    Items items;
    items.per_batch = per_batch;
    items.chunk = (a.S + per_batch - 1) / per_batch;
    items.count = B * per_batch;
    const int grid = static_cast<int>(items.count < cap ? items.count : cap);
    const int smem = Shape::kRingBytes + Shape::kNmod * a.Dv * 16;
    return launch_dependent(kern, grid, Shape::kThreads, smem, stream, a, items);
}

template <int OP, int V, int WPR, bool EXACT>
cudaError_t launch_shape(const RowArgs& a, const DeviceInfo& dev, cudaStream_t stream)
{
    using Shape = RowShape<OP, V, WPR>;
    auto kern = row_kernel<OP, V, WPR, EXACT>;
    constexpr int kSmemMax = Shape::kRingBytes + Shape::kCacheBytes;
    static PerDeviceInt blocks_per_sm;
    int bps = 0;
    {
        const cudaError_t e0 = blocks_per_sm.get(dev.device, bps, [&](int& v) -> cudaError_t {
            cudaError_t e =
                cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
            if (e != cudaSuccess)
                return e;
            int n = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, Shape::kThreads, kSmemMax);
            if (e != cudaSuccess)
                return e;
            v = n > 0 ? n : 1;
            return cudaSuccess;
        });
        if (e0 != cudaSuccess)
            return e0;
    }
    constexpr int kGroups = Shape::kWarps / WPR;
    const int64_t cap = static_cast<int64_t>(dev.sms) * bps;
    const int64_t B = a.rows / a.S;
    // split each batch into enough items to fill the GPU, each item at least
    // one row per group when the rows allow it
    int64_t per_batch = cap / (B > 0 ? B : 1);
    const int64_t max_items = (a.S + kGroups - 1) / kGroups;
    if (per_batch > max_items)
        per_batch = max_items;
    if (per_batch < 1)
        per_batch = 1;
    Items items;
    items.per_batch = per_batch;
    items.chunk = (a.S + per_batch - 1) / per_batch;
    items.count = B * per_batch;
    const int grid = static_cast<int>(items.count < cap ? items.count : cap);
    const int smem = Shape::kRingBytes + (Shape::kCached ? Shape::kNmod * a.Dv * 16 : 0);
    return launch_dependent(kern, grid, Shape::kThreads, smem, stream, a, items);
}

// Rows up to 1024 values: one warp each.  Longer rows are split over two or
// four warps (contiguous segments), which keeps registers and shared memory
// per warp small enough for ~24 resident warps per SM.
template <int OP, int V, int WPR>
cudaError_t launch_cfg(const RowArgs& a, const DeviceInfo& dev, cudaStream_t stream)
{
    if constexpr (WPR == 1 && (V == 16 || (V == 12 && OP != kOpGated))) {
        if constexpr (V == 12) {
            // rows per work item at two CTAs per SM (as launch_ws splits them)
            const int64_t B = a.rows / a.S;
            int64_t per_batch = static_cast<int64_t>(dev.sms) * 2 / (B > 0 ? B : 1);
            const int64_t max_items = (a.S + 7) / 8;
            per_batch = per_batch > max_items ? max_items : (per_batch < 1 ? 1 : per_batch);
            if ((a.S + per_batch - 1) / per_batch <= 16) {
                if (a.Dv == 32 * V)
                    return launch_ws<OP, V, true, true>(a, dev, stream);
                return launch_ws<OP, V, false, true>(a, dev, stream);
            }
        }
        if (a.Dv == 32 * V)
            return launch_ws<OP, V, true, false>(a, dev, stream);
        return launch_ws<OP, V, false, false>(a, dev, stream);
    }
    if (a.Dv == 32 * V * WPR)
        return launch_shape<OP, V, WPR, true>(a, dev, stream);
    return launch_shape<OP, V, WPR, false>(a, dev, stream);
}

// ---------------------------------------------------------------------------
// Few rows (a latency-bound launch): one CTA of kCoopWarps warps per row, V
// 16-byte vectors per lane (D = 1024 V).  A row's statistics then take V
// vectors of exact sums per lane, a warp butterfly and a combine over the
// CTA's warps, and nothing waits on a ring; used for at most kCoopRowsPerSm
// rows per SM, when every row gets a resident CTA at once.  EARLY: the
// modulation vectors are loaded before the statistics (their latency hidden
// behind them) instead of after (fewer registers).  Each thread reads its own
// vectors before it writes them, so out may alias x (and res_out residual).
// ---------------------------------------------------------------------------
constexpr int kCoopWarps = 4;
constexpr int64_t kCoopRowsPerSm = 4;

template <int OP, int V, bool EARLY>
__global__ void __launch_bounds__(32 * kCoopWarps) row_kernel_coop(const RowArgs a)
{
    grid_dependency_sync();
    constexpr int WPR = kCoopWarps;
    constexpr bool kNeedSum = (OP == kOpLN || OP == kOpLNFold);
    constexpr int kL = Log2Ceil<8 * V>::value;
    __shared__ Slot slots[2][WPR];   // the fast path's exchange, by row parity
    __shared__ Slot slow_slots[WPR];  // the rare slow path's own exchange

    const int lane = threadIdx.x & 31;
    const int wig = threadIdx.x >> 5;
    const int Dv = a.Dv;
    const uint4* __restrict__ src = static_cast<const uint4*>(OP == kOpGated ? a.residual : a.x);
    const uint4* __restrict__ upd = static_cast<const uint4*>(a.update);
    const uint4* __restrict__ gate = static_cast<const uint4*>(a.gate);
    const uint4* __restrict__ weight = static_cast<const uint4*>(a.weight);
    const uint4* __restrict__ scale = static_cast<const uint4*>(a.scale);
    const uint4* __restrict__ shift = static_cast<const uint4*>(a.shift);
    uint4* __restrict__ res_out = static_cast<uint4*>(a.res_out);
    uint4* __restrict__ out = static_cast<uint4*>(a.out);
    const bool has_w = (weight != nullptr);
    int par = 0;
    for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x, par ^= 1) {
        const int64_t b = row / a.S;
        const int64_t base = row * Dv;
        uint4 xv[V];
#pragma unroll
        for (int j = 0; j < V; ++j)
            xv[j] = ld_stream(src + base + j * 32 * WPR + threadIdx.x);
        if (OP == kOpGated) {
#pragma unroll
            for (int j = 0; j < V; ++j) {
                const int v = j * 32 * WPR + threadIdx.x;
                const uint4 u = ld_stream(upd + base + v);
                const uint4 g = ld_cached(gate + b * a.gate_bstride + v);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    word(xv[j], i) = bf2_add(word(xv[j], i), bf2_mul(word(g, i), word(u, i)));
                st_stream(res_out + base + v, xv[j]);
            }
        }
        uint4 s1[V], h[V], w[V];
        auto load_mod = [&]() {
#pragma unroll
            for (int j = 0; j < V; ++j) {
                const int v = j * 32 * WPR + threadIdx.x;
                s1[j] = ld_cached(scale + b * a.mod_bstride + v);
                h[j] = ld_cached(shift + b * a.mod_bstride + v);
                w[j] = (OP == kOpRMS || OP == kOpGated) && has_w ? ld_cached(weight + v)
                                                                 : make_uint4(0u, 0u, 0u, 0u);
            }
        };
        if (EARLY)
            load_mod();
        const uint32_t mm = tree_absmax<V>(xv);
        const uint32_t E = offset_exponent(mm);
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
        group_combine<WPR>(&slots[par][0], wig, lane, 0, s1h, s1l, s2h, s2l, cls, emax);
        float mean = 0.0f, stat;
        if (cls == kClassFast) {
            if (kNeedSum)
                finalize_ln(s1h, s1l, s2h, s2l, a.n, a.inv_n, mean, stat);
            else
                stat = finalize_ms(s2h, s2l, a.n, a.inv_n);
        } else {
            slow_stats<kNeedSum, V, WPR, kL>(xv, cls, emax, slow_slots, wig, lane, 0, a.n, a.inv_n,
                                             mean, stat);
        }
        const float rstd = rstd_from(stat, a.eps);
        if (threadIdx.x == 0) {
            if (a.mean_out)
                a.mean_out[row] = mean;
            if (a.rstd_out)
                a.rstd_out[row] = rstd;
        }
        if (!EARLY)
            load_mod();
        const u64 mean2 = f2_splat(mean), rstd2 = f2_splat(rstd);
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const int v = j * 32 * WPR + threadIdx.x;
            st_stream(out + base + v, normalise_modulate<OP>(xv[j], mean2, rstd2,
                                                             bf2x4_add(s1[j], kBf2One), h[j],
                                                             w[j], has_w));
        }
    }
}

// Launches the cooperative kernel for at most kCoopRowsPerSm rows per SM when
// every row gets a resident CTA at once (one wave); otherwise returns false
// and leaves the launch to the ring.  Early modulation loads measured faster
// at 1024 and 4096 values, late ones at 3072 (where the early form needs ~127
// registers).
template <int OP, int V>
bool launch_coop(const RowArgs& a, const DeviceInfo& dev, cudaStream_t stream, cudaError_t& err)
{
    if (a.rows > kCoopRowsPerSm * dev.sms)
        return false;
    auto kern = row_kernel_coop<OP, V, V != 3>;
    static PerDeviceInt blocks_per_sm;
    int bps = 0;
    err = blocks_per_sm.get(dev.device, bps, [&](int& v) -> cudaError_t {
        int n = 0;
        const cudaError_t e =
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, 32 * kCoopWarps, 0);
        v = n;
        return e;
    });
    if (err != cudaSuccess)
        return true;
    if (a.rows > static_cast<int64_t>(bps) * dev.sms)
        return false;
    err = launch_dependent(kern, static_cast<int>(a.rows), 32 * kCoopWarps, 0, stream, a);
    return true;
}

// Rows of up to 4096 values: one warp each (V vectors per lane); longer rows
// are split over two or four warps (contiguous segments).
template <int OP>
cudaError_t launch_op(const RowArgs& a, const DeviceInfo& dev, cudaStream_t stream)
{
    const int Dv = a.Dv;
    {
        cudaError_t e = cudaSuccess;
        bool done = false;
        switch (Dv) {
        case 128:
            done = launch_coop<OP, 1>(a, dev, stream, e);
            break;
        case 256:
            done = launch_coop<OP, 2>(a, dev, stream, e);
            break;
        case 384:
            done = launch_coop<OP, 3>(a, dev, stream, e);
            break;
        case 512:
            done = launch_coop<OP, 4>(a, dev, stream, e);
            break;
        default:
            break;
        }
        if (done)
            return e;
    }
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
    case kOpLNFold:
        return launch_op<kOpLNFold>(a, dev, stream);
    default:
        return launch_op<kOpGated>(a, dev, stream);
    }
}

cudaError_t row_kernels_error(unsigned* bits, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(bits, g_error, sizeof(unsigned));
    if (e == cudaSuccess && clear && *bits) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_error, &zero, sizeof(unsigned));
    }
    return e;
}

}  // namespace rmsmod
