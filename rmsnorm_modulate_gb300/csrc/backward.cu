// Backward of LayerNorm (no affine) + modulate on sm_103a (Qwen-Image final
// AdaLN page, §What: forward and backward of LayerNorm(x) * (1 + scale) +
// shift; the modulation gradients are token sums reduced by fixed 32-way
// balanced fp32 trees, applied recursively until one value remains, so they
// depend only on the sequence length).
//
// With the forward's roundings passed straight through, per row r of batch b
// (mean, rstd: the forward's statistics; s1 = R(1 + scale_b)):
//   yhat   = (f(x) - mean) * rstd          dyhat = f(g) * f(s1)   (exact)
//   c1     = fp32(sum dyhat / D)           c2    = fp32(sum dyhat * yhat / D)
//   grad_x = R(rstd * ((dyhat - c1) - yhat * c2))
// and per column d of batch b
//   grad_shift = T_s(f(g))                 grad_scale = T_s(f(g) * f(R(yhat)))
// with T_s the token tree over the S rows of the batch.
//
// Kernels:
//   bwd_ws_kernel  grad_x and the first tree level (the value of every
//                  32-token block) in one pass over x and g: statistics warps
//                  (c1, c2 per row) and output warps (grad_x, the block
//                  trees) around a ring of rows fed by 1-D bulk copies.  Used
//                  when both are wanted, D is a multiple of 256 from 1024 to
//                  3072 and S >= 2.
//   dx_kernel      grad_x alone (or at other D): one warp per row, x and g
//                  rows in shared memory, pass 1 forms c1, c2, pass 2 writes
//                  grad_x.
//   tokens_l1      the block values alone (or at other D): four lanes per
//                  (batch, block, 4 columns), 8 token slots per lane in
//                  registers, two butterfly steps for the top levels.
//   tokens_top     the trees above the first level for 2..1024 blocks: one
//                  lane per level-2 node, lane groups per column.
//   tokens_up      the same for any number of blocks: one thread per
//                  (batch, column), completed to 32^L slots.
// c1 and c2 are double-float sums everywhere (TwoSum per value, TwoProd for
// dyhat * yhat): the exact sums up to the rounding of the low word.
#include <cstddef>
#include <mutex>

#include "device_common.cuh"
#include "launch.h"

namespace rmsmod {

namespace {

__device__ unsigned int g_error;

// As mbar_try_wait, but the thread may be suspended (up to `hint_ns`) until the
// phase completes instead of returning at once: waiters take no issue slots.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity,
                                                    uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// mbar_wait for waits that are usually long (a consumer behind its
// producer): suspended waits of up to 20 us each, same overall limit.
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity,
                                                unsigned long long limit_ns)
{
    if (mbar_try_wait_sleep(bar, parity, 20000u))
        return true;
    const unsigned long long t0 = global_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 20000u))
            return true;
        if (global_ns() - t0 > limit_ns)
            return false;
    }
}

// ---------------------------------------------------------------------------
// grad_x
// ---------------------------------------------------------------------------

constexpr int kDxMaxWarps = 8;
constexpr int kDxThreads = 32 * kDxMaxWarps;  // upper bound; long rows use fewer warps
constexpr int kDxSmemMax = 200 * 1024;         // shared memory of one dx_kernel CTA, at most

// (hi, lo) += v, exactly up to the rounding of lo (TwoSum).
__device__ __forceinline__ void dd_acc(u64& hi, u64& lo, u64 v)
{
    const u64 s = f2_add(hi, v);
    const u64 bb = f2_sub(s, hi);
    const u64 e = f2_add(f2_sub(hi, f2_sub(s, bb)), f2_sub(v, bb));
    lo = f2_add(lo, e);
    hi = s;
}

// Pass 1 of one row (one warp; x, g and s1 rows in shared memory):
//   c1 = fp32(sum dyhat / D), c2 = fp32(sum dyhat * yhat / D)
// with both sums carried as double-float values (TwoSum per value, TwoProd
// for dyhat * yhat), so each is the exact sum up to the rounding of its low
// word; all lanes return both.
// S1_GLOBAL: s1 is formed here from the scale row in global memory (s1buf
// points there) instead of read ready-made from shared memory.
template <bool S1_GLOBAL>
__device__ __forceinline__ void row_c1c2(const uint4* xbuf, const uint4* gbuf, const uint4* s1buf,
                                         int Dv, int lane, u64 mean2, u64 rstd2, float n,
                                         float inv_n, float& c1, float& c2)
{
    u64 h1 = 0, l1 = 0, h2 = 0, l2 = 0, e2 = 0;
#pragma unroll 2
    for (int v = lane; v < Dv; v += 32) {
        const uint4 xv = xbuf[v], gv = gbuf[v];
        const uint4 sv = S1_GLOBAL ? bf2x4_add(ld_cached(s1buf + v), kBf2One) : s1buf[v];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const u64 yhat = f2_mul(f2_sub(f2_from_bf2(word(xv, i)), mean2), rstd2);
            const u64 dy = f2_mul(f2_from_bf2(word(gv, i)), f2_from_bf2(word(sv, i)));
            dd_acc(h1, l1, dy);
            // p = RN(dyhat * yhat) as separately rounded products (a packed
            // product feeding the TwoSum could be contracted into it); e =
            // the exact product error (TwoProd)
            float d0, d1, y0, y1;
            f2_unpack(dy, d0, d1);
            f2_unpack(yhat, y0, y1);
            const u64 p = f2_pack(__fmul_rn(d0, y0), __fmul_rn(d1, y1));
            e2 = f2_add(e2, f2_fma(dy, yhat, f2_neg(p)));
            dd_acc(h2, l2, p);
        }
    }
    l2 = f2_add(l2, e2);
    // the two lanes of each pair, then the warp
    float s1h, s1l, s2h, s2l;
    {
        float a0, a1, b0, b1;
        f2_unpack(h1, a0, a1);
        f2_unpack(l1, b0, b1);
        s1h = a0;
        s1l = b0;
        dd_add(s1h, s1l, a1, b1);
        f2_unpack(h2, a0, a1);
        f2_unpack(l2, b0, b1);
        s2h = a0;
        s2l = b0;
        dd_add(s2h, s2l, a1, b1);
    }
    dd2_allreduce<32>(s1h, s1l, s2h, s2l);
    float q1, q2;
    dd_div_n(s1h, s1l, n, inv_n, q1, q2);
    c1 = __fadd_rn(q1, q2);
    dd_div_n(s2h, s2l, n, inv_n, q1, q2);
    c2 = __fadd_rn(q1, q2);
}

__global__ void __launch_bounds__(kDxThreads, 2) dx_kernel(const BwdArgs a)
{
    grid_dependency_sync();
    extern __shared__ __align__(128) uint4 smem[];
    __shared__ __align__(8) unsigned long long bars[kDxMaxWarps];

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int Dv = a.Dv;
    const uint32_t row_bytes = static_cast<uint32_t>(Dv) * 16u;

    const uint4* __restrict__ xg = static_cast<const uint4*>(a.x);
    const uint4* __restrict__ gg = static_cast<const uint4*>(a.grad_out);
    const uint4* __restrict__ scale = static_cast<const uint4*>(a.scale);
    uint4* __restrict__ gx = static_cast<uint4*>(a.grad_x);

    // s1 = R(1 + scale) of the current batch, then each warp's x and g rows
    uint4* c_s1 = smem;
    uint4* xbuf = smem + Dv + static_cast<size_t>(warp) * 2 * Dv;  // [warp][x, g][Dv]
    uint4* gbuf = xbuf + Dv;

    const uint32_t bar = smem_addr(&bars[warp]);
    if (lane == 0) {
        mbar_init(bar, 1u);
        mbar_init_fence();
    }
    __syncwarp();

    bool broken = false;
    uint32_t phase = 0;
    const float n = a.n, inv_n = a.inv_n;
    for (int64_t item = blockIdx.x; item < a.items; item += gridDim.x) {
        const int64_t b = item / a.items_per_batch;
        const int64_t r_begin = b * a.S + (item % a.items_per_batch) * a.chunk;
        const int64_t r_lim = (b + 1) * a.S;
        const int64_t r_end = r_begin + a.chunk < r_lim ? r_begin + a.chunk : r_lim;

        auto issue = [&](int64_t row) {
            if (lane != 0 || row >= r_end)
                return;
            fence_proxy_async();
            mbar_expect_tx(bar, 2u * row_bytes);
            bulk_g2s(smem_addr(xbuf), xg + row * Dv, row_bytes, bar);
            bulk_g2s(smem_addr(gbuf), gg + row * Dv, row_bytes, bar);
        };
        issue(r_begin + warp);

        __syncthreads();  // every warp is done with the previous item's s1
        for (int c = threadIdx.x; c < Dv; c += blockDim.x)
            c_s1[c] = bf2x4_add(ld_cached(scale + b * a.mod_bstride + c), kBf2One);
        __syncthreads();

        for (int64_t row = r_begin + warp; row < r_end; row += nwarps, phase ^= 1u) {
            if (!broken && !mbar_wait(bar, phase, kWaitLimitNs)) {
                broken = true;
                if (lane == 0)
                    atomicOr(&g_error, kErrCopyTimeout);
            }
            const float mean = a.mean[row], rstd = a.rstd[row];
            const u64 mean2 = f2_splat(mean), rstd2 = f2_splat(rstd);

            // ---- pass 1: c1 = sum dyhat, c2 = sum dyhat * yhat (double-float)
            float c1, c2;
            row_c1c2<false>(xbuf, gbuf, c_s1, Dv, lane, mean2, rstd2, n, inv_n, c1, c2);

            // ---- pass 2: grad_x = R(rstd * ((dyhat - c1) - yhat * c2))
            const int64_t base = row * Dv;
            for (int v = lane; v < Dv; v += 32) {
                const uint4 xv = xbuf[v], gv = gbuf[v], sv = c_s1[v];
                uint4 o;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const u64 yhat = f2_mul(f2_sub(f2_from_bf2(word(xv, i)), mean2), rstd2);
                    const u64 dy = f2_mul(f2_from_bf2(word(gv, i)), f2_from_bf2(word(sv, i)));
                    float y0, y1, d0, d1;
                    f2_unpack(yhat, y0, y1);
                    f2_unpack(dy, d0, d1);
                    // the product yhat * c2 is rounded before the subtraction
                    const float t0 = __fsub_rn(__fsub_rn(d0, c1), __fmul_rn(y0, c2));
                    const float t1 = __fsub_rn(__fsub_rn(d1, c1), __fmul_rn(y1, c2));
                    word(o, i) = pack_bf2(__fmul_rn(rstd, t0), __fmul_rn(rstd, t1));
                }
                st_stream(gx + base + v, o);
            }
            // both buffers are consumed: start this warp's next row
            __syncwarp();
            issue(row + nwarps);
        }
    }
    if (broken)
        drain_pause();
}

// ---------------------------------------------------------------------------
// token trees
// ---------------------------------------------------------------------------

constexpr int kTokThreads = 256;

// Binary counter over the slots of a complete binary tree: push the value of
// slot k (k = 0, 1, ...); stack[l] holds a finished subtree of 2^l slots
// while bit l of the count is set.  The left operand of every add is the
// earlier subtree.  Called with k a compile-time constant after unrolling,
// so the stack stays in registers.
template <int LEVELS>
struct TreeCounter {
    u64 stack[LEVELS];

    __device__ __forceinline__ void push(int k, u64 v)
    {
#pragma unroll
        for (int l = 0; l < LEVELS; ++l) {
            if (((k >> l) & 1) == 0) {
                stack[l] = v;
                return;
            }
            v = f2_add(stack[l], v);
        }
        stack[LEVELS - 1] = v;  // the last slot closes the whole tree
    }
};

__global__ void __launch_bounds__(kTokThreads) tokens_l1_kernel(const BwdArgs a)
{
    grid_dependency_sync();
    // four consecutive lanes share (batch b, block j of 32 tokens, columns
    // 4c .. 4c + 3): lane q sums tokens 8q .. 8q + 7 (the slots' three lowest
    // tree levels), two butterfly steps form the top two levels, so every
    // lane ends with the block's tree
    const int cols4 = a.Dv * 2;
    const int64_t per_batch = static_cast<int64_t>(a.nblk) * cols4;
    const int64_t total = a.B * per_batch;  // groups of four lanes
    const uint2* __restrict__ xg = static_cast<const uint2*>(a.x);
    const uint2* __restrict__ gg = static_cast<const uint2*>(a.grad_out);
    float4* __restrict__ ws = static_cast<float4*>(a.workspace);
    const int q = threadIdx.x & 3;
    const int64_t groups_per_cta = blockDim.x / 4;
    // every lane of a warp runs the same number of iterations (the shuffles)
    const int64_t rounds = (total + gridDim.x * groups_per_cta - 1) / (gridDim.x * groups_per_cta);
    for (int64_t it = 0; it < rounds; ++it) {
        const int64_t t = (it * gridDim.x + blockIdx.x) * groups_per_cta + (threadIdx.x >> 2);
        const bool active = t < total;
        const int64_t tt = active ? t : 0;
        const int64_t b = tt / per_batch;
        const int64_t rem = tt - b * per_batch;
        const int64_t j = rem / cols4;
        const int c = static_cast<int>(rem - j * cols4);
        const int64_t s0 = j * 32 + 8 * q;
        const int n = !active ? 0 : (a.S - s0 < 8 ? (a.S - s0 > 0 ? static_cast<int>(a.S - s0) : 0) : 8);
        const int64_t row0 = b * a.S + s0;

        TreeCounter<3> tg[2], tp[2];
        u64 raw_g[2] = {0, 0}, raw_p[2] = {0, 0};  // slot 0 (a one-token sequence)
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            u64 gv2[2], pv2[2];
            if (k < n) {
                const int64_t row = row0 + k;
                const uint2 xv = ld_stream2(xg + row * cols4 + c);
                const uint2 gv = ld_stream2(gg + row * cols4 + c);
                const u64 mean2 = f2_splat(a.mean[row]), rstd2 = f2_splat(a.rstd[row]);
                const uint32_t xw[2] = {xv.x, xv.y}, gw[2] = {gv.x, gv.y};
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const u64 yhat = f2_mul(f2_sub(f2_from_bf2(xw[i]), mean2), rstd2);
                    const u64 y = f2_from_bf2(bf2_from_f2(yhat));
                    gv2[i] = f2_from_bf2(gw[i]);
                    pv2[i] = f2_mul(gv2[i], y);  // exact: two bf16 values
                }
                if (k == 0) {
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        raw_g[i] = gv2[i];
                        raw_p[i] = pv2[i];
                    }
                }
            } else {
#pragma unroll
                for (int i = 0; i < 2; ++i)
                    gv2[i] = pv2[i] = 0;  // +0 past the end of the sequence
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                tg[i].push(k, gv2[i]);
                tp[i].push(k, pv2[i]);
            }
        }
        u64 vg[2], vp[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            if (a.S == 1) {
                // a sequence of one token: its value as is, no tree (lane 0 of
                // the group holds it and is the one that writes)
                vg[i] = raw_g[i];
                vp[i] = raw_p[i];
                continue;
            }
            vg[i] = tg[i].stack[2];
            vp[i] = tp[i].stack[2];
            // levels 3 and 4: (T0 + T1) + (T2 + T3), the left operand the
            // earlier tokens (the adds are commutative, so every lane agrees)
#pragma unroll
            for (int off = 1; off <= 2; off <<= 1) {
                const u64 og = __shfl_xor_sync(kFullMask, vg[i], off);
                const u64 op = __shfl_xor_sync(kFullMask, vp[i], off);
                const bool left = (q & off) == 0;
                vg[i] = left ? f2_add(vg[i], og) : f2_add(og, vg[i]);
                vp[i] = left ? f2_add(vp[i], op) : f2_add(op, vp[i]);
            }
        }
        if (active && q == 0) {
            float rg[4], rp[4];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                f2_unpack(vg[i], rg[2 * i], rg[2 * i + 1]);
                f2_unpack(vp[i], rp[2 * i], rp[2 * i + 1]);
            }
            // workspace [B][nblk][2][D] fp32: quantity 0 = grad_shift, 1 = grad_scale
            const int64_t o = ((b * a.nblk + j) * 2) * static_cast<int64_t>(cols4) + c;
            ws[o] = make_float4(rg[0], rg[1], rg[2], rg[3]);
            ws[o + cols4] = make_float4(rp[0], rp[1], rp[2], rp[3]);
        }
    }
}

// Above the first level: the block values of one column are the leaves of a
// complete binary tree over 32^L slots (32^L >= nblk, slots past nblk +0).
// Each run of 32 block values is one level-2 node: its 32 loads are issued
// together and combined by a register binary counter; the level-2 nodes then
// go through a small counter in local memory, completed with +0 subtrees.
template <int LEVELS>
struct ScalarTree {
    float stack[LEVELS];

    __device__ __forceinline__ void push(int k, float v)
    {
#pragma unroll
        for (int l = 0; l < LEVELS; ++l) {
            if (((k >> l) & 1) == 0) {
                stack[l] = v;
                return;
            }
            v = __fadd_rn(stack[l], v);
        }
        stack[LEVELS - 1] = v;
    }
};

__global__ void __launch_bounds__(kTokThreads) tokens_up_kernel(const BwdArgs a)
{
    grid_dependency_sync();
    const int D = a.Dv * 8;
    const int64_t total = a.B * static_cast<int64_t>(D);
    const float* __restrict__ ws = static_cast<const float*>(a.workspace);
    const int64_t nblk = a.nblk;
    const int64_t n2 = (nblk + 31) / 32;
    int K2 = 0;  // levels of the tree over the level-2 nodes: 2^K2 = 32^L2 >= n2
    for (int64_t cap = 1; cap < n2; cap *= 32)
        K2 += 5;
    const int64_t stride = 2 * static_cast<int64_t>(D);
    for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t < total;
         t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t b = t / D;
        const int d = static_cast<int>(t - b * D);
        const float* col0 = ws + (b * nblk * 2) * static_cast<int64_t>(D) + d;  // quantity 0
        const float* col1 = col0 + D;                                          // quantity 1
        float res0, res1;
        if (nblk == 1) {
            res0 = col0[0];
            res1 = col1[0];
        } else {
            float st0[32], st1[32];  // counter over the level-2 nodes (K2 <= 30)
            for (int64_t m = 0; m < n2; ++m) {
                ScalarTree<5> t0, t1;
                float v0[32], v1[32];
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    const int64_t idx = 32 * m + k;
                    v0[k] = idx < nblk ? col0[idx * stride] : 0.0f;
                    v1[k] = idx < nblk ? col1[idx * stride] : 0.0f;
                }
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    t0.push(k, v0[k]);
                    t1.push(k, v1[k]);
                }
                float u0 = t0.stack[4], u1 = t1.stack[4];
                int l = 0;
                for (; (m >> l) & 1; ++l) {
                    u0 = __fadd_rn(st0[l], u0);
                    u1 = __fadd_rn(st1[l], u1);
                }
                st0[l] = u0;
                st1[l] = u1;
            }
            if (K2 == 0) {
                res0 = st0[0];
                res1 = st1[0];
            } else {
                // complete the tree: level-2 slots n2 .. 2^K2 - 1 hold +0
                float c0 = 0.0f, c1 = 0.0f;
                for (int l = 0; l < K2; ++l) {
                    if ((n2 >> l) & 1) {
                        c0 = __fadd_rn(st0[l], c0);  // finished left subtree + the rest
                        c1 = __fadd_rn(st1[l], c1);
                    } else {
                        c0 = __fadd_rn(c0, 0.0f);    // the rest + an all-zero subtree
                        c1 = __fadd_rn(c1, 0.0f);
                    }
                }
                res0 = c0;
                res1 = c1;
            }
        }
        if (a.grad_shift)
            a.grad_shift[t] = res0;
        if (a.grad_scale)
            a.grad_scale[t] = res1;
    }
}


// ---------------------------------------------------------------------------
// grad_x and the first token-tree level in one pass over HBM
// ---------------------------------------------------------------------------
//
// Warp-specialised, one CTA per SM walking its blocks (batch b, block j of
// 32 tokens) in order; the rows of those blocks form the CTA's sequence, and
// row i of the sequence lands by bulk copy (x row, then g row) in slot
// i % nslots of a shared-memory ring.
//   output warps (Wout = Dv / 32; thread t owns the 8 columns of vector t)
//       take every row in sequence order: grad_x of their columns, and both
//       token trees of the block for them (binary counter over the 32 slots,
//       +0 past the end; levels 0-1 in registers, 2-4 in shared memory)
//   statistics warps (kBwdStatWarps) take rows i = w, w + 8, ...: c1, c2
//       into the slot's statistics, then the slot's ready barrier
// Each output warp releases a slot with one atomic add; the last of them
// refills it with the row nslots further on, after tagging the slot with that
// row's sequence number.  Were nslots not a multiple of the statistics warps,
// a statistics warp could reach a slot before the previous fill of it has
// landed (its rows would not be nslots apart), where the barrier's parity
// aliases; the launcher sizes the ring in such multiples, and the warp checks
// the tag before waiting all the same.  x and g are read from HBM once.

constexpr int kBwdStatWarps = 8;
constexpr int kBwdMaxOutWarps = 12;  // D <= 3072
constexpr int kBwdMinOutWarps = 4;   // D >= 1024
constexpr int kBwdMaxSlots = 32;

__device__ __forceinline__ void st_release_u32(uint32_t addr, uint32_t v)
{
    asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_u32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// Release of a slot by one output warp (lane 0, after __syncwarp): returns
// the count before this add (acquire-release, so the last releaser sees every
// warp's reads of the slot as done).
__device__ __forceinline__ uint32_t release_add(uint32_t addr)
{
    uint32_t old;
    asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], 1;"
                 : "=r"(old)
                 : "r"(addr)
                 : "memory");
    return old;
}

// One block of the sequence: batch b, block j of 32 tokens (item = b * nblk
// + j; item counts fit in 32 bits).
struct SeqBlock {
    int64_t r0;  // its first row
    int64_t b;
    int nrows;   // 0: past the end of the sequence
};

struct BwdSeq {
    uint32_t items, stride, nblk;
    int64_t S;

    __device__ __forceinline__ SeqBlock block(uint32_t item) const
    {
        if (item >= items)
            return SeqBlock{0, 0, 0};
        const uint32_t b = item / nblk, j = item - b * nblk;
        const int64_t left = S - 32 * static_cast<int64_t>(j);
        return SeqBlock{static_cast<int64_t>(b) * S + 32 * static_cast<int64_t>(j),
                        static_cast<int64_t>(b), static_cast<int>(left < 32 ? left : 32)};
    }
};

// A walk along the sequence (one division per block entered).
struct SeqCursor {
    uint32_t item;
    int r;
    SeqBlock blk;

    __device__ __forceinline__ void start(const BwdSeq& sq, uint32_t first)
    {
        item = first;
        r = 0;
        blk = sq.block(first);
    }

    __device__ __forceinline__ bool done() const { return blk.nrows == 0; }

    __device__ __forceinline__ int64_t row() const { return blk.r0 + r; }

    __device__ __forceinline__ void advance(const BwdSeq& sq, int by)
    {
        r += by;
        while (blk.nrows != 0 && r >= blk.nrows) {
            r -= blk.nrows;
            item += sq.stride;
            blk = sq.block(item);
        }
    }
};

// Ring slot and fill parity of a sequence position, advanced in step with it.
struct SlotPos {
    uint32_t slot, par, round;

    __device__ __forceinline__ void advance(uint32_t by, uint32_t ns)
    {
        slot += by;
        while (slot >= ns) {
            slot -= ns;
            par ^= 1u;
            ++round;
        }
    }
};

// The two token trees of one 32-token block for 8 columns (4 packed pairs)
// as a binary counter over the slots: level l holds a finished subtree of
// 2^l slots while bit l of the count is set, the left operand of every add is
// the earlier subtree.  Rows come in groups of four (slot k = 4 m + i, i known
// at compile time), so levels 0 and 1 are resolved in registers without
// tests; each finished 4-slot subtree enters a counter over m with levels
// 2-4 in this thread's columns of up[3][8][nthreads] in shared memory.
struct BlockTrees {
    u64 g0[4], p0[4], g1[4], p1[4];  // levels 0 and 1
    u64* up;                         // &up[0][0][t]
    int stride;                      // nthreads

    __device__ __forceinline__ u64& lvl(int l, int q, int i) const
    {
        return up[((l - 2) * 8 + q * 4 + i) * stride];
    }

    // slot 4 m + I, pair i
    template <int I>
    __device__ __forceinline__ void push(int m, int i, u64 vg, u64 vp)
    {
        if (I == 0 || I == 2) {
            g0[i] = vg;
            p0[i] = vp;
        } else if (I == 1) {
            g1[i] = f2_add(g0[i], vg);
            p1[i] = f2_add(p0[i], vp);
        } else {
            // the 4-slot subtree (s0 + s1) + (s2 + s3), then the counter over
            // m: the finished subtrees below the first clear bit of m join it,
            // and it takes that bit's level (slot group 7 closes the tree at
            // level 4)
            vg = f2_add(g1[i], f2_add(g0[i], vg));
            vp = f2_add(p1[i], f2_add(p0[i], vp));
            const int ones = __ffs(~m) - 1;
            for (int l = 2; l < 2 + ones && l < 5; ++l) {
                vg = f2_add(lvl(l, 0, i), vg);
                vp = f2_add(lvl(l, 1, i), vp);
            }
            const int dst = 2 + ones < 4 ? 2 + ones : 4;
            lvl(dst, 0, i) = vg;
            lvl(dst, 1, i) = vp;
        }
    }
};

__global__ void __launch_bounds__(32 * (kBwdMaxOutWarps + kBwdStatWarps), 1)
    bwd_ws_kernel(const BwdArgs a, const int nslots)
{
    extern __shared__ __align__(128) uint4 smem[];
    __shared__ __align__(8) unsigned long long full_bar[kBwdMaxSlots], ready_bar[kBwdMaxSlots];
    __shared__ float4 slot_stats[kBwdMaxSlots];  // (mean, rstd, c1, c2) of the row in each slot
    __shared__ uint32_t released[kBwdMaxSlots];  // output-warp releases, cumulative
    __shared__ uint32_t slot_seq[kBwdMaxSlots];  // sequence number of the slot's latest fill

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int Dv = a.Dv;
    const int Wout = Dv >> 5;
    const int nout = 32 * Wout;
    const uint32_t ns = static_cast<uint32_t>(nslots);
    const uint32_t row_bytes = static_cast<uint32_t>(Dv) * 16u;
    uint4* ring = smem;                                                   // [nslots][x, g][Dv]
    u64* up = reinterpret_cast<u64*>(ring + static_cast<size_t>(nslots) * 2 * Dv);  // [3][8][nout]

    const uint4* __restrict__ xg = static_cast<const uint4*>(a.x);
    const uint4* __restrict__ gg = static_cast<const uint4*>(a.grad_out);
    const BwdSeq sq{static_cast<uint32_t>(a.B * a.nblk), gridDim.x,
                    static_cast<uint32_t>(a.nblk), a.S};

    // the copy of `row` (sequence number q) into slot s (one thread)
    auto issue = [&](int64_t row, uint32_t s, uint32_t q) {
        const uint32_t bar = smem_addr(&full_bar[s]);
        uint4* dst = ring + static_cast<size_t>(s) * 2 * Dv;
        st_release_u32(smem_addr(&slot_seq[s]), q);
        fence_proxy_async();
        mbar_expect_tx(bar, 2u * row_bytes);
        bulk_g2s(smem_addr(dst), xg + row * Dv, row_bytes, bar);
        bulk_g2s(smem_addr(dst + Dv), gg + row * Dv, row_bytes, bar);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < nslots; ++s) {
            mbar_init(smem_addr(&full_bar[s]), 1u);
            mbar_init(smem_addr(&ready_bar[s]), 1u);
            released[s] = 0;
        }
        mbar_init_fence();
    }
    // only shared memory so far: the barriers are ready when the previous
    // grid's results become visible
    grid_dependency_sync();
    if (threadIdx.x == 0) {
        // the first nslots rows of the sequence
        SeqCursor c;
        c.start(sq, blockIdx.x);
        for (uint32_t s = 0; s < ns && !c.done(); ++s) {
            issue(c.row(), s, s);
            c.advance(sq, 1);
        }
    }
    __syncthreads();

    bool broken = false;
    auto wait = [&](uint32_t bar, uint32_t parity) {
        if (!broken && !mbar_wait_sleep(bar, parity, kWaitLimitNs)) {
            broken = true;
            atomicOr(&g_error, kErrCopyTimeout);
        }
    };

    if (warp >= Wout) {
        // ---- statistics warps: rows w, w + 8, ... of the sequence
        const int sw = warp - Wout;
        const uint4* __restrict__ scale = static_cast<const uint4*>(a.scale);
        const float n = a.n, inv_n = a.inv_n;
        SeqCursor c;
        c.start(sq, blockIdx.x);
        c.advance(sq, sw);
        SlotPos sp{0, 0, 0};
        sp.advance(static_cast<uint32_t>(sw), ns);
        uint32_t q = static_cast<uint32_t>(sw);  // sequence number of the row
        while (!c.done()) {
            const uint32_t s = sp.slot;
            const int64_t row = c.row();
            const int64_t b = c.blk.b;
            // the row's forward statistics load while its copy lands
            const float mean = a.mean[row], rstd = a.rstd[row];
            // the slot's fill for this row is issued (so the fill before it
            // has landed), then the fill itself
            const uint32_t tag = smem_addr(&slot_seq[s]);
            if (!broken && ld_acquire_u32(tag) != q) {
                const unsigned long long t0 = global_ns();
                while (ld_acquire_u32(tag) != q) {
                    __nanosleep(64);
                    if (global_ns() - t0 > kWaitLimitNs) {
                        broken = true;
                        atomicOr(&g_error, kErrCopyTimeout);
                        break;
                    }
                }
            }
            wait(smem_addr(&full_bar[s]), sp.par);
            const uint4* xbuf = ring + static_cast<size_t>(s) * 2 * Dv;
            float c1, c2;
            row_c1c2<true>(xbuf, xbuf + Dv, scale + b * a.mod_bstride, Dv, lane, f2_splat(mean),
                           f2_splat(rstd), n, inv_n, c1, c2);
            if (lane == 0) {
                slot_stats[s] = make_float4(mean, rstd, c1, c2);
                mbar_arrive(smem_addr(&ready_bar[s]));
            }
            __syncwarp();
            c.advance(sq, kBwdStatWarps);
            sp.advance(kBwdStatWarps, ns);
            q += kBwdStatWarps;
        }
        if (broken)
            drain_pause();
        return;
    }

    // ---- output warps
    const int t = threadIdx.x;  // this thread's vector of 8 columns
    const uint4* __restrict__ scale = static_cast<const uint4*>(a.scale);
    uint4* __restrict__ gx = static_cast<uint4*>(a.grad_x);
    float4* __restrict__ ws = static_cast<float4*>(a.workspace);
    SlotPos sp{0, 0, 0};
    uint32_t seq = 0;  // sequence number of the next row
    for (uint32_t item = blockIdx.x; item < sq.items; item += gridDim.x) {
        const SeqBlock blk = sq.block(item);
        const SeqBlock next = sq.block(item + gridDim.x);
        const int64_t b = blk.b, r0 = blk.r0;
        const int nrows = blk.nrows;
        const uint4 s1v = bf2x4_add(ld_cached(scale + b * a.mod_bstride + t), kBf2One);
        BlockTrees tr;
        tr.up = up + t;
        tr.stride = nout;
#pragma unroll 1
        for (int m = 0; m < 8; ++m) {
#pragma unroll
        for (int i4 = 0; i4 < 4; ++i4) {
            const int k = 4 * m + i4;
            if (k < nrows) {
                const uint32_t s = sp.slot;
                wait(smem_addr(&ready_bar[s]), sp.par);
                const uint4* xbuf = ring + static_cast<size_t>(s) * 2 * Dv;
                const uint4 xv = xbuf[t], gv = xbuf[Dv + t];
                const float4 st = slot_stats[s];
                __syncwarp();
                if (lane == 0) {
                    // the slot is consumed by this warp; the last of the
                    // output warps refills it with the row nslots further on
                    const uint32_t old = release_add(smem_addr(&released[s]));
                    if (old + 1u == static_cast<uint32_t>(Wout) * (sp.round + 1u)) {
                        const int q = k + nslots;
                        const uint32_t qseq = seq + ns;
                        if (q < nrows) {
                            issue(r0 + q, s, qseq);
                        } else if (q - nrows < next.nrows) {
                            issue(next.r0 + (q - nrows), s, qseq);
                        } else {  // short blocks: walk on
                            SeqCursor c;
                            c.start(sq, item);
                            c.advance(sq, q);
                            if (!c.done())
                                issue(c.row(), s, qseq);
                        }
                    }
                }
                sp.advance(1u, ns);
                ++seq;
                const u64 mean2 = f2_splat(st.x), rstd2 = f2_splat(st.y);
                const u64 c1c1 = f2_splat(st.z);
                uint4 o;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const u64 yhat = f2_mul(f2_sub(f2_from_bf2(word(xv, i)), mean2), rstd2);
                    const u64 gf = f2_from_bf2(word(gv, i));
                    // grad_x = R(rstd * ((dyhat - c1) - R32(yhat * c2))).  Packed:
                    // dyhat = g * s1 is exact (two bf16), so whether it is
                    // contracted into the subtraction or not, d = RN(dyhat -
                    // c1); the inexact yhat * c2 is two separately rounded
                    // products (never contracted)
                    const u64 d = f2_sub(f2_mul(gf, f2_from_bf2(word(s1v, i))), c1c1);
                    float y0, y1;
                    f2_unpack(yhat, y0, y1);
                    const u64 t = f2_sub(d, f2_pack(__fmul_rn(y0, st.w), __fmul_rn(y1, st.w)));
                    word(o, i) = bf2_from_f2(f2_mul(rstd2, t));
                    // token-tree values: g, and g * R(yhat) (exact: two bf16)
                    const u64 gp = f2_mul(gf, f2_from_bf2(bf2_from_f2(yhat)));
                    if (i4 == 0)
                        tr.push<0>(m, i, gf, gp);
                    else if (i4 == 1)
                        tr.push<1>(m, i, gf, gp);
                    else if (i4 == 2)
                        tr.push<2>(m, i, gf, gp);
                    else
                        tr.push<3>(m, i, gf, gp);
                }
                st_stream(gx + (r0 + k) * Dv + t, o);
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) {  // +0 past the end of the sequence
                    if (i4 == 0)
                        tr.push<0>(m, i, 0ull, 0ull);
                    else if (i4 == 1)
                        tr.push<1>(m, i, 0ull, 0ull);
                    else if (i4 == 2)
                        tr.push<2>(m, i, 0ull, 0ull);
                    else
                        tr.push<3>(m, i, 0ull, 0ull);
                }
            }
        }
        }

        // the block's values -> workspace [B][nblk][2][D]: quantity 0 =
        // grad_shift, 1 = grad_scale
        float rg[8], rp[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f2_unpack(tr.lvl(4, 0, i), rg[2 * i], rg[2 * i + 1]);
            f2_unpack(tr.lvl(4, 1, i), rp[2 * i], rp[2 * i + 1]);
        }
        const int64_t o = (static_cast<int64_t>(item) * 2) * (2 * Dv) + 2 * t;  // item = b nblk + j
        ws[o] = make_float4(rg[0], rg[1], rg[2], rg[3]);
        ws[o + 1] = make_float4(rg[4], rg[5], rg[6], rg[7]);
        ws[o + 2 * Dv] = make_float4(rp[0], rp[1], rp[2], rp[3]);
        ws[o + 2 * Dv + 1] = make_float4(rp[4], rp[5], rp[6], rp[7]);
    }
    if (broken)
        drain_pause();
}

// Above the first level when 2 <= nblk <= 1024 (one level-2 node per run of
// 32 block values, at most 32 of them): lane groups of P lanes (P = n2
// rounded up to a power of two) per column and quantity, lane m forming
// level-2 node m (its 32 loads issued together, +0 past nblk; lanes m >= n2
// hold +0); a butterfly over the group gives the tree over P slots, and
// adding +0 once per doubling up to 32 completes it to the 32-slot tree.  With
// n2 == 1 the level-2 node is the result.  Lanes of a warp: m = lane / C, C =
// 32 / P columns side by side, so every load instruction reads C adjacent
// columns of P block rows.
// 512 threads a CTA: fewer CTAs than the first level's 256, so more SMs are
// free for the next launch sooner (35.14 vs 35.42 us a call at the FLUX.1
// B=1 shape; 1024 measured 39.5).
constexpr int kTopThreads = 512;
__global__ void __launch_bounds__(kTopThreads) tokens_top_kernel(const BwdArgs a, const int P)
{
    grid_dependency_sync();
    const int D = a.Dv * 8;
    const int C = 32 / P;
    const int lane = threadIdx.x & 31;
    const int m = lane / C, c = lane - m * C;
    const int64_t nblk = a.nblk;
    const int n2 = static_cast<int>((nblk + 31) / 32);
    const int64_t warps_per_q = (D + C - 1) / C;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (warp >= a.B * 2 * warps_per_q)
        return;  // whole warps only
    const int64_t bq = warp / warps_per_q;
    const int64_t b = bq >> 1;
    const int q = static_cast<int>(bq & 1);  // 0: grad_shift, 1: grad_scale
    const int d = static_cast<int>((warp - bq * warps_per_q) * C + c);
    const bool active = d < D;
    const float* col = static_cast<const float*>(a.workspace) +
                       ((b * nblk) * 2 + q) * static_cast<int64_t>(D) + (active ? d : 0);
    const int64_t stride = 2 * static_cast<int64_t>(D);

    float v = 0.0f;
    if (active && m < n2) {
        float x[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            const int64_t idx = 32 * static_cast<int64_t>(m) + k;
            x[k] = idx < nblk ? col[idx * stride] : 0.0f;
        }
        ScalarTree<5> t;
#pragma unroll
        for (int k = 0; k < 32; ++k)
            t.push(k, x[k]);
        v = t.stack[4];
    }
    if (n2 > 1) {
        for (int off = C; off < 32; off <<= 1)
            v = __fadd_rn(v, __shfl_xor_sync(kFullMask, v, off));
        for (int w = P; w < 32; w <<= 1)
            v = __fadd_rn(v, 0.0f);  // the all-zero right subtree
    }
    if (active && m == 0) {
        float* out = q == 0 ? a.grad_shift : a.grad_scale;
        if (out)
            out[b * D + d] = v;
    }
}

}  // namespace

// Fixed device scratch for ln_modulate_backward_static: the token-sum
// workspace of calls whose need fits, in the module's own device memory, so
// that entry point allocates nothing.  One buffer per device shared by every
// call: calls whose work overlaps in time (another stream, another host
// thread) race on it.
static __device__ __align__(256) unsigned char g_backward_scratch[kBackwardScratchBytes];

cudaError_t backward_static_scratch(int device, void** ptr)
{
    static std::mutex mu;
    static void* addr[kMaxDevices] = {nullptr};
    if (device < 0 || device >= kMaxDevices)
        return cudaErrorInvalidDevice;
    const int d = device;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[d]) {
        // once per device (loads the module's device data if needed)
        cudaError_t e = cudaGetSymbolAddress(&addr[d], g_backward_scratch);
        if (e != cudaSuccess) {
            addr[d] = nullptr;
            return e;
        }
    }
    *ptr = addr[d];
    return cudaSuccess;
}

size_t backward_workspace_bytes(int64_t B, int64_t S, int64_t D)
{
    const int64_t nblk = (S + 31) / 32;
    return static_cast<size_t>(B) * static_cast<size_t>(nblk) * 2u * static_cast<size_t>(D) *
           sizeof(float);
}

// The token trees above the first level (block values in the workspace):
// lane groups per column where at most 32 level-2 nodes exist, else one
// thread per column.
static cudaError_t launch_upper(const BwdArgs& a, const DeviceInfo& dev, cudaStream_t stream)
{
    if (a.nblk >= 2 && a.nblk <= 32 * 32) {
        const int n2 = static_cast<int>((a.nblk + 31) / 32);
        int P = 1;
        while (P < n2)
            P <<= 1;
        const int64_t D = a.Dv * 8;
        const int64_t lanes = a.B * 2 * ((D + 32 / P - 1) / (32 / P)) * 32;
        const int64_t grid = (lanes + kTopThreads - 1) / kTopThreads;
        return launch_dependent(tokens_top_kernel, static_cast<int>(grid), kTopThreads, 0,
                                stream, a, P);
    }
    const int64_t up = a.B * a.Dv * 8;
    const int64_t g2 = (up + kTokThreads - 1) / kTokThreads;
    const int64_t cap = static_cast<int64_t>(dev.sms) * 4;
    return launch_dependent(tokens_up_kernel, static_cast<int>(g2 < cap ? g2 : cap), kTokThreads,
                            0, stream, a);
}

// grad_x and the token sums of one call through bwd_ws_kernel, then the
// upper tree levels; false (nothing launched) where its shape rules do not
// hold: S >= 2 (a one-token sequence takes no tree), D a multiple of 256
// from 1024 to 3072.
static bool launch_fused(const BwdArgs& a, const DeviceInfo& dev, cudaStream_t stream,
                         cudaError_t& e)
{
    if (!a.grad_x || !(a.grad_scale || a.grad_shift) || a.S < 2 || a.Dv % 32 != 0)
        return false;
    const int Wout = a.Dv / 32;
    if (Wout < kBwdMinOutWarps || Wout > kBwdMaxOutWarps)
        return false;
    // ring slots: about 96 KB of rows in multiples of the statistics warps
    // (8 slots at D = 3072; at that shape 8 measured faster than 6, 10, 12
    // or 14), within what ~220 KB holds beside the upper tree levels
    constexpr int kBudget = 220 * 1024;
    const int slot_bytes = 2 * a.Dv * 16;
    const int up_bytes = 3 * 8 * 32 * Wout * 8;
    int nslots = (96 * 1024 / slot_bytes) / kBwdStatWarps * kBwdStatWarps;
    nslots = nslots < kBwdStatWarps ? kBwdStatWarps : nslots;
    const int fit = (kBudget - up_bytes) / slot_bytes;
    nslots = nslots > fit ? fit : nslots;
    nslots = nslots > kBwdMaxSlots ? kBwdMaxSlots : nslots;
    const int smem = nslots * slot_bytes + up_bytes;
    const int threads = 32 * (Wout + kBwdStatWarps);
    static PerDeviceInt configured;
    int done = 0;
    e = configured.get(dev.device, done, [&](int& v) -> cudaError_t {
        v = 1;
        return cudaFuncSetAttribute(bwd_ws_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kBudget);
    });
    if (e != cudaSuccess)
        return true;
    const int64_t items = a.B * a.nblk;
    const int64_t cap = dev.sms;  // one CTA per SM
    e = launch_dependent(bwd_ws_kernel, static_cast<int>(items < cap ? items : cap), threads,
                         smem, stream, a, nslots);
    if (e != cudaSuccess)
        return true;
    e = launch_upper(a, dev, stream);
    return true;
}

cudaError_t launch_backward(BwdArgs a, const DeviceInfo& dev, cudaStream_t stream)
{
    cudaError_t e = cudaSuccess;
    if (launch_fused(a, dev, stream, e))
        return e;
    if (a.grad_x) {
        // warps per CTA: as many as ~200 KB of shared memory hold (x and g
        // rows per warp plus the s1 row), at most eight
        const int row_vec = a.Dv;
        int warps = (kDxSmemMax / 16 - row_vec) / (2 * row_vec);
        warps = warps > kDxMaxWarps ? kDxMaxWarps : (warps < 1 ? 1 : warps);
        const int smem = (row_vec + warps * 2 * row_vec) * 16;
        // the kernel's largest dynamic shared memory (~200 KB), set once per device
        static PerDeviceInt configured;
        int done = 0;
        e = configured.get(dev.device, done, [&](int& v) -> cudaError_t {
            v = 1;
            return cudaFuncSetAttribute(dx_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        kDxSmemMax);
        });
        if (e != cudaSuccess)
            return e;
        int nb = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, dx_kernel, 32 * warps, smem);
        if (e != cudaSuccess)
            return e;
        const int64_t cap = static_cast<int64_t>(dev.sms) * (nb > 0 ? nb : 1);
        int64_t per_batch = cap / (a.B > 0 ? a.B : 1);
        const int64_t max_items = (a.S + warps - 1) / warps;
        if (per_batch > max_items)
            per_batch = max_items;
        if (per_batch < 1)
            per_batch = 1;
        a.items_per_batch = per_batch;
        a.chunk = (a.S + per_batch - 1) / per_batch;
        a.items = a.B * per_batch;
        const int grid = static_cast<int>(a.items < cap ? a.items : cap);
        e = launch_dependent(dx_kernel, grid, 32 * warps, smem, stream, a);
        if (e != cudaSuccess)
            return e;
    }
    if (a.grad_scale || a.grad_shift) {
        const int64_t l1 = a.B * a.nblk * a.Dv * 2 * 4;  // four lanes per group
        int64_t g1 = (l1 + kTokThreads - 1) / kTokThreads;
        // a persistent grid (four CTAs per SM loop over the blocks)
        const int64_t cap = static_cast<int64_t>(dev.sms) * 4;
        e = launch_dependent(tokens_l1_kernel, static_cast<int>(g1 < cap ? g1 : cap),
                             kTokThreads, 0, stream, a);
        if (e != cudaSuccess)
            return e;
        e = launch_upper(a, dev, stream);
    }
    return e;
}

cudaError_t backward_error(unsigned* bits, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(bits, g_error, sizeof(unsigned));
    if (e == cudaSuccess && clear && *bits) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_error, &zero, sizeof(unsigned));
    }
    return e;
}

}  // namespace rmsmod
