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
// Three launches:
//   dx_kernel      one warp per row: x and g rows land in shared memory by
//                  1-D bulk copies; pass 1 forms c1, c2 as double-float sums
//                  (TwoSum per value, TwoProd for dyhat * yhat), pass 2
//                  writes grad_x.
//   tokens_l1      four lanes per (batch, 32-token block, 4 columns): each
//                  lane the tree of 8 token slots in registers (a binary
//                  counter, +0 for slots past the end), two butterfly steps
//                  for the top levels, both quantities; the block values go
//                  to the workspace.
//   tokens_up      one thread per (batch, column): the trees above the first
//                  level over the block values, completed to 32^L slots.
#include <cstddef>
#include <mutex>

#include "device_common.cuh"
#include "launch.h"

namespace rmsmod {

namespace {

__device__ unsigned int g_error;

// ---------------------------------------------------------------------------
// grad_x
// ---------------------------------------------------------------------------

constexpr int kDxMaxWarps = 8;
constexpr int kDxThreads = 32 * kDxMaxWarps;  // upper bound; long rows use fewer warps

// (hi, lo) += v, exactly up to the rounding of lo (TwoSum).
__device__ __forceinline__ void dd_acc(u64& hi, u64& lo, u64 v)
{
    const u64 s = f2_add(hi, v);
    const u64 bb = f2_sub(s, hi);
    const u64 e = f2_add(f2_sub(hi, f2_sub(s, bb)), f2_sub(v, bb));
    lo = f2_add(lo, e);
    hi = s;
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
            u64 h1 = 0, l1 = 0, h2 = 0, l2 = 0, e2 = 0;
#pragma unroll 2
            for (int v = lane; v < Dv; v += 32) {
                const uint4 xv = xbuf[v], gv = gbuf[v], sv = c_s1[v];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const u64 yhat = f2_mul(f2_sub(f2_from_bf2(word(xv, i)), mean2), rstd2);
                    const u64 dy = f2_mul(f2_from_bf2(word(gv, i)), f2_from_bf2(word(sv, i)));
                    dd_acc(h1, l1, dy);
                    // p = RN(dyhat * yhat) as separately rounded products (a
                    // packed product feeding the TwoSum could be contracted
                    // into it); e = the exact product error (TwoProd)
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
            const float c1 = __fadd_rn(q1, q2);
            dd_div_n(s2h, s2l, n, inv_n, q1, q2);
            const float c2 = __fadd_rn(q1, q2);

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
    static void* addr[64] = {nullptr};
    const int d = device & 63;
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

cudaError_t launch_backward(BwdArgs a, const DeviceInfo& dev, cudaStream_t stream)
{
    cudaError_t e = cudaSuccess;
    if (a.grad_x) {
        // warps per CTA: as many as ~200 KB of shared memory hold (x and g
        // rows per warp plus the s1 row), at most eight
        const int row_vec = a.Dv;
        int warps = (200 * 1024 / 16 - row_vec) / (2 * row_vec);
        warps = warps > kDxMaxWarps ? kDxMaxWarps : (warps < 1 ? 1 : warps);
        const int smem = (row_vec + warps * 2 * row_vec) * 16;
        static int configured[64] = {0};
        const int d = dev.device & 63;
        if (configured[d] < smem) {
            e = cudaFuncSetAttribute(dx_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     smem);
            if (e != cudaSuccess)
                return e;
            configured[d] = smem;
        }
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
        const int64_t up = a.B * a.Dv * 8;
        const int64_t g2 = (up + kTokThreads - 1) / kTokThreads;
        e = launch_dependent(tokens_up_kernel, static_cast<int>(g2 < cap ? g2 : cap),
                             kTokThreads, 0, stream, a);
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
