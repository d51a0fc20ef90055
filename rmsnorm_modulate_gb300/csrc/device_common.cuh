// Device building blocks shared by the rmsmod kernels (sm_103a).
//
//  * packed bf16x2 and f32x2 arithmetic as inline PTX (Blackwell issues one
//    f32x2 instruction for two fp32 lanes);
//  * the bf16 rounding boundaries of the eager op chain;
//  * an exact-statistics engine: per-lane sums of x and x^2 that are exact
//    (error-free transformations against a power-of-two offset), combined
//    across lanes in double-float arithmetic and rounded once to fp32, so
//    the fp32 mean / variance / mean square are the correctly rounded exact
//    statistics except when the exact value lies within ~2^-44 (relative) of
//    an fp32 rounding boundary.
//
// Every arithmetic step whose rounding matters is an explicit .rn PTX
// instruction or __f*_rn intrinsic, so no FMA contraction can cross a
// rounding boundary regardless of compiler flags.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace rmsmod {

typedef unsigned long long u64;

constexpr unsigned kFullMask = 0xFFFFFFFFu;

// ---------------------------------------------------------------------------
// loads / stores
// ---------------------------------------------------------------------------

// Streaming 16-byte load of data touched once (no L1 allocation).  The
// coherent path, not the read-only one: an output may alias its input.
// 8-byte read-only streaming load (input never written by the same kernel).
__device__ __forceinline__ uint2 ld_stream2(const uint2* p)
{
    uint2 v;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p)
{
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// 16-byte load of small tensors re-read by every row (scale, shift, weight):
// read-only path, cached.
__device__ __forceinline__ uint4 ld_cached(const uint4* p)
{
    uint4 v;
    asm("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

__device__ __forceinline__ float4 ld_cached_f4(const float4* p)
{
    float4 v;
    asm("ld.global.nc.v4.f32 {%0,%1,%2,%3}, [%4];"
        : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
        : "l"(p));
    return v;
}

// Streaming 16-byte store (evict-first).
__device__ __forceinline__ void st_stream(uint4* p, uint4 v)
{
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint32_t& word(uint4& v, int i)
{
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

__device__ __forceinline__ uint32_t word(const uint4& v, int i)
{
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// ---------------------------------------------------------------------------
// Asynchronous bulk copies (TMA, 1-D) into shared memory, tracked by mbarriers
// ---------------------------------------------------------------------------

// Longest a kernel waits for one bulk copy before it gives up, records an
// error in its error word and carries on without the data (1 s).
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

// Error-word bits.
constexpr unsigned kErrCopyTimeout = 1u;

__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// One plain arrival (release semantics: this thread's earlier shared-memory
// writes are visible to threads that observe the phase complete).
__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Makes barrier initialisation visible to the asynchronous (TMA) proxy.
__device__ __forceinline__ void mbar_init_fence()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// Orders this thread's earlier generic-proxy accesses to shared memory before
// later asynchronous-proxy writes (reuse of a buffer that was just read).
__device__ __forceinline__ void fence_proxy_async()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// global -> shared bulk copy of `bytes` (multiple of 16, both addresses
// 16-byte aligned); completion is signalled on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for the phase of `bar` with the given parity; false if it did not
// complete within `limit_ns`.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          unsigned long long limit_ns)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const unsigned long long t0 = global_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (global_ns() - t0 > limit_ns)
            return false;
    }
}

// After a copy timed out: a bounded pause (1 ms) so that copies still in
// flight land before the CTA exits and its shared memory is reused.
__device__ __forceinline__ void drain_pause()
{
    const unsigned long long t0 = global_ns();
    while (global_ns() - t0 < 1000000ull) {
    }
}

// ---------------------------------------------------------------------------
// bf16x2 (two bf16 in one 32-bit word: element 2i in the low half)
// ---------------------------------------------------------------------------

// R(f(a) + f(b)) per half.  For bf16 operands the fp32 sum followed by a
// bf16 rounding equals the single correctly rounded bf16 sum: either the
// fp32 sum is exact (exponents within 15) or the smaller operand is below a
// quarter ulp of the larger and both routes return the larger one.
__device__ __forceinline__ uint32_t bf2_add(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// R(f(a) * f(b)) per half: the product of two bf16 is exact in fp32 above
// the fp32 subnormal range, so one correctly rounded bf16 product is the
// same value (checked exhaustively on the GPU by the test-suite).
__device__ __forceinline__ uint32_t bf2_mul(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// max(|a|, |b|) per half (sign bits garbage: callers mask them); NaN wins.
__device__ __forceinline__ uint32_t bf2_absmax(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// R(lo), R(hi) packed: round-to-nearest-even, no flush of subnormals.
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi)
{
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

constexpr uint32_t kBf2One = 0x3F803F80u;  // (1.0, 1.0)

// Packed fp16 (IEEE binary16, subnormals kept): correctly rounded add and
// multiply, which for fp16 operands equal "fp32 op, then round to fp16" (the
// product is exact in fp32; for the sum fp32 carries more than 2 * 11 + 2
// bits, so the double rounding is innocuous).
__device__ __forceinline__ uint32_t h2_add(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t h2_mul(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

constexpr uint32_t kH2One = 0x3C003C00u;  // (1.0, 1.0) in fp16

// R(f(v) + f(c)) for the eight bf16 of a vector against a bf16x2 constant.
__device__ __forceinline__ uint4 bf2x4_add(uint4 v, uint32_t c)
{
    return make_uint4(bf2_add(v.x, c), bf2_add(v.y, c), bf2_add(v.z, c), bf2_add(v.w, c));
}

// ---------------------------------------------------------------------------
// f32x2 (two fp32 in one 64-bit register pair)
// ---------------------------------------------------------------------------

__device__ __forceinline__ u64 f2_pack(float lo, float hi)
{
    u64 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void f2_unpack(u64 v, float& lo, float& hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ u64 f2_splat(float v) { return f2_pack(v, v); }

// The two bf16 of a word widened exactly to an fp32 pair.
// First statement of every kernel (they are launched as programmatic
// dependents): waits until the previous grid in the stream has completed and
// its memory is visible, then lets the next grid's CTAs be scheduled as this
// grid's CTAs retire.  No global memory is touched before it.
__device__ __forceinline__ void grid_dependency_sync()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ u64 f2_from_bf2(uint32_t w)
{
    return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

__device__ __forceinline__ uint32_t bf2_from_f2(u64 v)
{
    float lo, hi;
    f2_unpack(v, lo, hi);
    return pack_bf2(lo, hi);
}

__device__ __forceinline__ u64 f2_add(u64 a, u64 b)
{
    u64 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ u64 f2_sub(u64 a, u64 b)
{
    u64 d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ u64 f2_mul(u64 a, u64 b)
{
    u64 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ u64 f2_fma(u64 a, u64 b, u64 c)
{
    u64 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ u64 f2_neg(u64 a) { return a ^ 0x8000000080000000ull; }

// a * b then + c as two separately rounded fp32 operations.  The packed
// f32x2 forms are not used here: a packed multiply feeding a packed add was
// observed to come out fused, while __fmul_rn / __fadd_rn are documented
// never to be merged into a multiply-add.
__device__ __forceinline__ u64 f2_mul_then_add(u64 a, u64 b, u64 c)
{
    float a0, a1, b0, b1, c0, c1;
    f2_unpack(a, a0, a1);
    f2_unpack(b, b0, b1);
    f2_unpack(c, c0, c1);
    return f2_pack(__fadd_rn(__fmul_rn(a0, b0), c0), __fadd_rn(__fmul_rn(a1, b1), c1));
}

// ---------------------------------------------------------------------------
// Double-float helpers (value = hi + lo, two fp32)
// ---------------------------------------------------------------------------

// (a.hi + b.hi, ...) both lanes: s + e == (ah + al) + (bh + bl) up to
// ~2^-47 |max operand|.  TwoSum on the high parts, low parts added, then a
// Fast2Sum renormalisation.  11 packed instructions.
__device__ __forceinline__ void dd2_add(u64& ah, u64& al, u64 bh, u64 bl)
{
    u64 s = f2_add(ah, bh);
    u64 v = f2_sub(s, ah);
    u64 e = f2_add(f2_sub(ah, f2_sub(s, v)), f2_sub(bh, v));
    e = f2_add(e, f2_add(al, bl));
    u64 h = f2_add(s, e);
    al = f2_sub(e, f2_sub(h, s));
    ah = h;
}

__device__ __forceinline__ void dd_add(float& ah, float& al, float bh, float bl)
{
    float s = __fadd_rn(ah, bh);
    float v = __fsub_rn(s, ah);
    float e = __fadd_rn(__fsub_rn(ah, __fsub_rn(s, v)), __fsub_rn(bh, v));
    e = __fadd_rn(e, __fadd_rn(al, bl));
    float h = __fadd_rn(s, e);
    al = __fsub_rn(e, __fsub_rn(h, s));
    ah = h;
}

// (hi, lo) / N as a double-float (q1, q2) with |q2| <= ~ulp(q1); n is the
// exact row length, inv_n = fp32(1/n).  The FMA remainder is exact or
// within 2^-24 of itself, which is far below what the result keeps.
__device__ __forceinline__ void dd_div_n(float hi, float lo, float n, float inv_n, float& q1,
                                         float& q2)
{
    q1 = __fmul_rn(hi, inv_n);
    float r = __fmaf_rn(-q1, n, hi);
    r = __fadd_rn(r, lo);
    q2 = __fmul_rn(r, inv_n);
}

// ---------------------------------------------------------------------------
// The exact-statistics engine
// ---------------------------------------------------------------------------
//
// A lane holding k = 2^L (or fewer) bf16 values whose magnitudes are all
// below 2^(e+1) accumulates
//     acc1 = K1 + sum x,   K1 = 2^(e+2+L)
//     acc2 = K2 + sum x^2, K2 = 2^(2e+3+L)
// Partial sums stay below K/2 in magnitude, so every accumulator stays in
// [K/2, 3K/2], and each step's rounding error is recovered exactly by
// Fast2Sum (|acc| >= |x|): s = acc + x; t = x - (s - acc).  The errors are
// summed in err1 / err2; those sums are exact unless the lane's values span
// more than ~2^30 (x) / ~2^11 (x^2) in magnitude, and even then their
// rounding is ~2^-48 relative.  acc - K is exact (Sterbenz).  The f32x2
// registers keep two independent accumulators (even / odd elements).
//
// The offsets follow a bound on the lane's (or the whole row's) largest
// magnitude; where that magnitude is outside [2^-40, 2^40) or non-finite the
// row takes a slow path (scaled to unit magnitude, or plain IEEE sums that
// propagate Inf / NaN like the oracle's double sums).  Any bound at or above
// the largest magnitude keeps the sums exact; a looser one moves more of each
// value into the error terms, whose own fp32 rounding then weighs more.

// The fast range keeps n * sum x^2 and (sum x)^2 (n <= 2^14) far from fp32
// overflow and every Fast2Sum error term far from the subnormal range.
constexpr uint32_t kMinFastExp = 127 - 40;  // biased exponent of 2^-40
constexpr uint32_t kMaxFastExp = 127 + 39;  // biased exponent of 2^39 (|x| < 2^40)

enum : int { kClassFast = 0, kClassScaled = 1, kClassNonFinite = 2 };

// Largest |x| bits (15-bit magnitude) of a running bf16x2 abs-max.
__device__ __forceinline__ uint32_t absmax_bits(uint32_t m)
{
    m &= 0x7FFF7FFFu;
    uint32_t lo = m & 0xFFFFu, hi = m >> 16;
    return lo > hi ? lo : hi;
}

__device__ __forceinline__ int magnitude_class(uint32_t mm)
{
    if (mm >= 0x7F80u)
        return kClassNonFinite;
    uint32_t E = mm >> 7;
    if (mm != 0 && (E < kMinFastExp || E > kMaxFastExp))
        return kClassScaled;
    return kClassFast;
}

// Biased exponent used to place the offsets (zero lanes use 2^0).
__device__ __forceinline__ uint32_t offset_exponent(uint32_t mm)
{
    return mm == 0 ? 127u : (mm >> 7);
}

template <int L>
__device__ __forceinline__ float offset_k1(uint32_t E)
{
    return __uint_as_float((E + 2u + L) << 23);
}

template <int L>
__device__ __forceinline__ float offset_k2(uint32_t E)
{
    return __uint_as_float((2u * E - 124u + L) << 23);
}

// Accumulator for sum x (optional) and sum x^2.  Each f32x2 register holds
// two independent accumulators (even / odd elements).
template <bool NEED_SUM>
struct ExactSums {
    u64 acc1, err1, acc2, err2, k1, k2;

    __device__ __forceinline__ void init(float K1, float K2)
    {
        k1 = f2_splat(K1);
        k2 = f2_splat(K2);
        acc1 = k1;
        acc2 = k2;
        err1 = 0ull;
        err2 = 0ull;
    }

    __device__ __forceinline__ void add(u64 xx)
    {
        if (NEED_SUM) {
            const u64 s = f2_add(acc1, xx);
            const u64 z = f2_sub(s, acc1);
            err1 = f2_add(err1, f2_sub(xx, z));
            acc1 = s;
        }
        // s2 = acc + x^2 rounded; acc - s2 is exact (Sterbenz), so the
        // rounding error x^2 - (s2 - acc) is one more FMA with no negation
        const u64 s2 = f2_fma(xx, xx, acc2);
        const u64 zn = f2_sub(acc2, s2);
        err2 = f2_add(err2, f2_fma(xx, xx, zn));
        acc2 = s2;
    }

    // Lane totals as double-floats: (s1h, s1l) = sum x, (s2h, s2l) = sum x^2.
    __device__ __forceinline__ void lane_total(float& s1h, float& s1l, float& s2h, float& s2l)
    {
        // halves: h = acc - K exact, l = err
        const u64 h1 = f2_sub(acc1, k1), h2 = f2_sub(acc2, k2);
        float a0, a1, b0, b1, c0, c1, d0, d1;
        f2_unpack(h1, a0, a1);
        f2_unpack(err1, b0, b1);
        f2_unpack(h2, c0, c1);
        f2_unpack(err2, d0, d1);
        // even + odd halves: (a0 + b0) + (a1 + b1), (c0 + d0) + (c1 + d1)
        u64 H = f2_pack(a0, c0), Lo = f2_pack(b0, d0);
        dd2_add(H, Lo, f2_pack(a1, c1), f2_pack(b1, d1));
        f2_unpack(H, s1h, s2h);
        f2_unpack(Lo, s1l, s2l);
    }
};

// Largest |x| bits over V vectors, as a balanced tree (short dependency chain).
template <int V>
__device__ __forceinline__ uint32_t tree_absmax(const uint4 (&xv)[V])
{
    uint32_t m[V];
#pragma unroll
    for (int j = 0; j < V; ++j)
        m[j] = bf2_absmax(bf2_absmax(xv[j].x, xv[j].y), bf2_absmax(xv[j].z, xv[j].w));
#pragma unroll
    for (int w = 1; w < V; w *= 2)
#pragma unroll
        for (int j = 0; j + w < V; j += 2 * w)
            m[j] = bf2_absmax(m[j], m[j + w]);
    return absmax_bits(m[0]);
}

// Butterfly over `width` lanes (power of two) of two double-floats at once;
// every participating lane ends with the total.
template <int WIDTH>
__device__ __forceinline__ void dd2_allreduce(float& s1h, float& s1l, float& s2h, float& s2l)
{
#pragma unroll
    for (int off = WIDTH / 2; off > 0; off >>= 1) {
        float o1h = __shfl_xor_sync(kFullMask, s1h, off);
        float o1l = __shfl_xor_sync(kFullMask, s1l, off);
        float o2h = __shfl_xor_sync(kFullMask, s2h, off);
        float o2l = __shfl_xor_sync(kFullMask, s2l, off);
        u64 H = f2_pack(s1h, s2h), Lo = f2_pack(s1l, s2l);
        dd2_add(H, Lo, f2_pack(o1h, o2h), f2_pack(o1l, o2l));
        f2_unpack(H, s1h, s2h);
        f2_unpack(Lo, s1l, s2l);
    }
}

template <int WIDTH>
__device__ __forceinline__ void dd_allreduce(float& sh, float& sl)
{
#pragma unroll
    for (int off = WIDTH / 2; off > 0; off >>= 1) {
        float oh = __shfl_xor_sync(kFullMask, sh, off);
        float ol = __shfl_xor_sync(kFullMask, sl, off);
        dd_add(sh, sl, oh, ol);
    }
}

template <int WIDTH>
__device__ __forceinline__ float allreduce_add(float v)
{
#pragma unroll
    for (int off = WIDTH / 2; off > 0; off >>= 1)
        v = __fadd_rn(v, __shfl_xor_sync(kFullMask, v, off));
    return v;
}

template <int WIDTH>
__device__ __forceinline__ uint32_t allreduce_max(uint32_t v)
{
#pragma unroll
    for (int off = WIDTH / 2; off > 0; off >>= 1) {
        uint32_t o = __shfl_xor_sync(kFullMask, v, off);
        v = v > o ? v : o;
    }
    return v;
}

// mean = fp32(S1 / n) and var = fp32((n * S2 - S1^2) / n^2) from
// double-float sums.  n * S2 and S1^2 are formed with error-free products,
// so rows whose sums are exact (constant rows, for instance) cancel to an
// exact zero; otherwise both results are the fp32 rounding of a
// double-float value within ~2^-44 (relative) of the exact statistic.
__device__ __forceinline__ void finalize_ln(float s1h, float s1l, float s2h, float s2l, float n,
                                            float inv_n, float& mean, float& var)
{
    float q1, q2;
    dd_div_n(s1h, s1l, n, inv_n, q1, q2);
    mean = __fadd_rn(q1, q2);

    const float p1 = __fmul_rn(n, s2h);
    const float e1 = __fmaf_rn(n, s2h, -p1);
    const float p2 = __fmul_rn(s1h, s1h);
    const float e2 = __fmaf_rn(s1h, s1h, -p2);
    // TwoSum(p1, -p2), then the small terms
    const float s = __fsub_rn(p1, p2);
    const float v = __fsub_rn(s, p1);
    float e = __fadd_rn(__fsub_rn(p1, __fsub_rn(s, v)), __fsub_rn(-p2, v));
    const float cross = __fmaf_rn(n, s2l, -__fmul_rn(__fmul_rn(2.0f, s1h), s1l));
    e = __fadd_rn(e, __fadd_rn(__fsub_rn(e1, e2), cross));
    float nh = __fadd_rn(s, e);
    float nl = __fsub_rn(e, __fsub_rn(nh, s));
    // divide by n twice
    dd_div_n(nh, nl, n, inv_n, q1, q2);
    nh = __fadd_rn(q1, q2);
    nl = __fsub_rn(q2, __fsub_rn(nh, q1));
    dd_div_n(nh, nl, n, inv_n, q1, q2);
    var = __fadd_rn(q1, q2);
    var = var > 0.0f ? var : 0.0f;
}

// finalize_ln for a power-of-two n (inv_n exact): the divisions become exact
// scalings, so only the two roundings to fp32 remain.
__device__ __forceinline__ void finalize_ln_pow2(float s1h, float s1l, float s2h, float s2l,
                                                 float n, float inv_n, float& mean, float& var)
{
    mean = __fmul_rn(__fadd_rn(s1h, s1l), inv_n);
    const float p1 = __fmul_rn(n, s2h);  // exact
    const float p2 = __fmul_rn(s1h, s1h);
    const float e2 = __fmaf_rn(s1h, s1h, -p2);
    const float s = __fsub_rn(p1, p2);
    const float v = __fsub_rn(s, p1);
    float e = __fadd_rn(__fsub_rn(p1, __fsub_rn(s, v)), __fsub_rn(-p2, v));
    const float cross = __fmaf_rn(n, s2l, -__fmul_rn(__fmul_rn(2.0f, s1h), s1l));
    e = __fadd_rn(e, __fsub_rn(cross, e2));
    var = __fmul_rn(__fmul_rn(__fadd_rn(s, e), inv_n), inv_n);
    var = var > 0.0f ? var : 0.0f;
}

__device__ __forceinline__ float finalize_ms(float s2h, float s2l, float n, float inv_n)
{
    float a1, a2;
    dd_div_n(s2h, s2l, n, inv_n, a1, a2);
    return __fadd_rn(a1, a2);
}

// rstd = 1 / sqrt(stat + eps): three correctly rounded fp32 operations.
__device__ __forceinline__ float rstd_from(float stat, float eps)
{
    return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(stat, eps)));
}

// 2^k for k in [-126, 127] as an fp32.
__device__ __forceinline__ float exp2i(int k)
{
    return __uint_as_float(static_cast<uint32_t>(k + 127) << 23);
}

// Scale factors that bring a row whose largest biased exponent is E to
// magnitudes below 2 (two exact power-of-two multiplies, each in range).
struct RowScale {
    float down_a, down_b;  // x * down_a * down_b  = x * 2^-e
    int e;

    __device__ __forceinline__ void set(uint32_t E)
    {
        e = (E == 0 ? -126 : static_cast<int>(E) - 127);
        int ha = -e / 2;
        down_a = exp2i(ha);
        down_b = exp2i(-e - ha);
    }

    __device__ __forceinline__ u64 apply(u64 xx) const
    {
        return f2_mul(f2_mul(xx, f2_splat(down_a)), f2_splat(down_b));
    }

    // v * 2^(mult * e), mult in {1, 2}: both factors 2^(k/2), 2^(k - k/2)
    // lie in [-126, 127].
    __device__ __forceinline__ float unscale(float v, int mult) const
    {
        int k = mult * e;
        int ha = k / 2;
        return __fmul_rn(__fmul_rn(v, exp2i(ha)), exp2i(k - ha));
    }
};

}  // namespace rmsmod
