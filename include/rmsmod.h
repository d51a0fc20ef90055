/*
 * rmsmod.h -- C ABI of librmsmod.so: fused adaLN row normalisation + modulate
 * for NVIDIA GB300 (sm_103a).
 *
 * Each entry point fuses what an eager diffusion-transformer adaLN site runs
 * as several bandwidth-bound kernels into one pass over HBM, and reproduces
 * the eager chain's bf16 rounding after every elementwise op:
 *   R(v) = round fp32 -> bf16, nearest-even;  f(h) = exact bf16 -> fp32.
 *
 * Conventions shared by every entry point
 *   - Tensors are device pointers.  bf16 tensors are passed as raw 16-bit
 *     patterns (any type the caller likes, e.g. torch.bfloat16 storage).
 *   - Row-major, innermost dimension contiguous (unit stride).  A "row" is
 *     the vector that is normalised (D, head_dim or C values).
 *   - Every bf16 pointer must be 16-byte aligned; D, head_dim and C must be
 *     multiples of 8 (one 16-byte vector = 8 bf16); batch strides are in
 *     elements and must be multiples of 8.  fp32 pointers must be 16-byte
 *     aligned too (per-channel fp32 bias) or 4-byte aligned (per-row outputs).
 *   - Row statistics are fp32: the exact mean / biased variance / mean square
 *     of the row, rounded once to fp32; rstd = 1 / sqrt(stat + eps) as
 *     three correctly rounded fp32 operations.
 *   - The caller owns every buffer.  The library allocates nothing, needs no
 *     workspace and keeps no global state other than cached device
 *     attributes.  Calls are asynchronous on `stream` (NULL = the legacy
 *     default stream); nothing synchronises the host.
 *   - Output buffers may alias their row input exactly (out == x,
 *     res_out == residual); any other overlap is rejected when detected and
 *     is otherwise undefined.
 *   - Errors: arguments are validated before anything is launched; on any
 *     failure the call returns a negative rmsmod_status and launches
 *     nothing.  A zero row count returns RMSMOD_OK and launches nothing.
 *     There is no fallback inside the library: a caller that wants one
 *     tests rmsmod_supported() or the returned status and runs its own.
 *
 * Sources (web pages describing the method):
 *   [GLM]   sglang PR #34008 "GLM-Image bit-exact fused aten LayerNorm+modulate / qk-LN"
 *   [ERNIE] sglang PR #33854 "ERNIE-Image bit-exact fused RMSNorm+scale/shift"
 *   [FLUX]  sglang PR #34004 "FLUX.1 fused adaLN modulate (bit-exact) + RoPE cache hoist"
 *   [QWEN]  RL-Kernel PR #538 "[Qwen-Image][CUDA] Final AdaLN output (final_adaln_out)"
 *   [WAN]   sglang PR #38650 "Fuse the Wan VAE conv bias epilogue and tile the RMSNorm+SiLU kernel"
 */
#ifndef RMSMOD_H
#define RMSMOD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* rmsmod_stream_t;

typedef enum {
    RMSMOD_OK = 0,
    RMSMOD_ERR_NULL = -1,        /* a required pointer is NULL */
    RMSMOD_ERR_SHAPE = -2,       /* negative size, D/C/head_dim not a multiple of 8,
                                    above the supported maximum, C == 1, ... */
    RMSMOD_ERR_ALIGN = -3,       /* a pointer is not aligned as required */
    RMSMOD_ERR_STRIDE = -4,      /* a batch stride is negative or not a multiple of 8 */
    RMSMOD_ERR_UNSUPPORTED = -5, /* partially overlapping buffers or another unsupported combination */
    RMSMOD_ERR_CUDA = -6,        /* the CUDA runtime reported an error at launch */
    RMSMOD_ERR_DEVICE = -7       /* no usable CUDA device is current */
} rmsmod_status;

/* Largest supported row length D (ln / rms / gated) and channel count C. */
#define RMSMOD_MAX_D 16384
#define RMSMOD_MAX_C 1024

/* ------------------------------------------------------------------------
 * ln_modulate -- LayerNorm without affine, then the adaLN modulate chain.
 *   [GLM] §Motivation (GlmImageAdaLayerNormZero) and §What "rounding-faithful"
 *   means here; [QWEN] §What (out = LayerNorm(x, eps, no affine) * (1 + scale) + shift);
 *   [FLUX] §Modifications commit 2 (per-op rounding of the modulate chain).
 *
 *   For each row r = (b, s) of x [B, S, D]:
 *     mean, var  = fp32 mean and biased variance of f(x[r, :])
 *     rstd       = 1 / sqrt(var + eps)
 *     y[d]       = R((f(x[r,d]) - mean) * rstd)                (no FMA)
 *     out[r, d]  = R(f(R(f(y[d]) * f(R(1 + f(scale_b[d]))))) + f(shift_b[d]))
 *   scale_b = scale + b * mod_bstride (elements; 0 = one row for every batch),
 *   same for shift_b: this covers per-batch CFG rows and adaLN chunk views.
 *
 *   x, out        bf16 [B*S*D], out may equal x
 *   scale, shift  bf16, each row D values at base + b * mod_bstride
 *   mean_out, rstd_out  nullable fp32 [B*S]
 * ---------------------------------------------------------------------- */
int ln_modulate(const void* x, const void* scale, const void* shift, void* out,
                int64_t B, int64_t S, int64_t D, int64_t mod_bstride, float eps,
                float* mean_out, float* rstd_out, rmsmod_stream_t stream);

/* ------------------------------------------------------------------------
 * ln_modulate_folded -- single-rounding tier of ln_modulate (not bit-exact
 * with the eager chain).
 *   [FLUX] §Modifications commit 3 (quality="high": the modulate folds into
 *   the LayerNorm's elementwise affine, layer_norm(x, weight = 1 + scale,
 *   bias = shift), with 1 + scale keeping the eager rounding of its row;
 *   max abs difference to the lossless chain at the bf16 rounding level).
 *
 *   Statistics, rstd, arguments, layout, aliasing and errors as ln_modulate;
 *   per element
 *     w          = R(1 + f(scale_b[d]))
 *     out[r, d]  = R(((f(x[r,d]) - mean) * rstd) * f(w) + f(shift_b[d]))
 *   in fp32 with each operation rounded separately (no FMA) and one final
 *   rounding to bf16.  Unlike the page's aten route it takes per-batch
 *   modulation rows (mod_bstride) for B > 1.
 * ---------------------------------------------------------------------- */
int ln_modulate_folded(const void* x, const void* scale, const void* shift, void* out,
                       int64_t B, int64_t S, int64_t D, int64_t mod_bstride, float eps,
                       float* mean_out, float* rstd_out, rmsmod_stream_t stream);

/* ------------------------------------------------------------------------
 * ln_modulate_backward -- gradients of ln_modulate.
 *   [QWEN] §What (forward and backward of out = LayerNorm(x, eps, no affine)
 *   * (1 + scale) + shift; d_scale and d_shift are token sums reduced by
 *   fixed 32-way balanced fp32 trees applied recursively until one value
 *   remains, so the result depends only on S, not on B or the batch
 *   position).
 *
 *   With the forward's roundings passed straight through, per row r of
 *   batch b (mean, rstd: the forward's statistics, as ln_modulate writes
 *   them to mean_out / rstd_out; s1 = R(1 + f(scale_b))):
 *     yhat[d]   = (f(x[r,d]) - mean) * rstd           (fp32, as the forward)
 *     dyhat[d]  = f(grad_out[r,d]) * f(s1[d])          (exact)
 *     c1, c2    = fp32(sum_d dyhat / D), fp32(sum_d dyhat * yhat / D)
 *                 (double-float sums, rounded once)
 *     grad_x    = R(rstd * ((dyhat - c1) - yhat * c2)) (fp32 ops, no FMA)
 *   and per column d of batch b, over the S rows of the batch:
 *     grad_shift[b, d] = T(f(grad_out[., d]))
 *     grad_scale[b, d] = T(f(grad_out[., d]) * f(R(yhat[., d])))
 *   T: the values are the leaves of a complete binary tree over 32^L slots
 *   (32^L the smallest power of 32 >= S; slots past S hold +0) summed in
 *   fp32 with adjacent pairing; S == 1 returns the single value.
 *
 *   x, grad_out  bf16 [B*S*D];  scale bf16 rows at base + b * mod_bstride
 *   mean, rstd   fp32 [B*S], the forward's
 *   grad_x       nullable bf16 [B*S*D]
 *   grad_scale, grad_shift  nullable fp32 [B, D] (one row per batch; with a
 *                shared modulation row the caller sums the rows over b)
 *   No output (grad_x, grad_scale, grad_shift, workspace) may overlap an
 *   input (x, grad_out, the scale rows, mean, rstd) or another output:
 *   RMSMOD_ERR_UNSUPPORTED, nothing launched.
 *   workspace    device memory of at least
 *                ln_modulate_backward_workspace_bytes(B, S, D) bytes,
 *                256-byte aligned; needed when grad_scale or grad_shift is
 *                given (NULL is fine otherwise); owned by the caller,
 *                overwritten, and in use until the call's work on `stream`
 *                is done.
 *   Errors as ln_modulate; RMSMOD_ERR_SHAPE also when workspace_bytes is
 *   too small.  One to three kernel launches on `stream` (two when grad_x
 *   and a modulation gradient are both wanted, D is a multiple of 256 from
 *   1024 to 3072 and S >= 2); nothing is allocated.
 * ---------------------------------------------------------------------- */
size_t ln_modulate_backward_workspace_bytes(int64_t B, int64_t S, int64_t D);

int ln_modulate_backward(const void* x, const void* scale, int64_t mod_bstride,
                         const void* grad_out, const float* mean, const float* rstd,
                         int64_t B, int64_t S, int64_t D, void* grad_x, float* grad_scale,
                         float* grad_shift, void* workspace, size_t workspace_bytes,
                         rmsmod_stream_t stream);

/* ------------------------------------------------------------------------
 * ln_modulate_backward_static -- ln_modulate_backward without a caller
 * workspace.  The pages have no counterpart: this is a library convenience.
 *
 *   For callers that cannot hand the library device memory: a host
 *   framework whose own allocator owns the device and exposes no buffer to
 *   plug-ins, or a latency-critical path that must not call cudaMalloc
 *   (which can synchronise the whole device) between steps.
 *   Same arguments, results and errors as ln_modulate_backward minus the
 *   workspace: the token-sum scratch is a fixed 8 MiB (8 << 20 bytes) array
 *   of the library's own device memory, so the call allocates nothing
 *   (every GPU that loads the library holds those 8 MiB until the process
 *   exits).
 *   Sizes whose ln_modulate_backward_workspace_bytes(B, S, D) exceeds
 *   8 MiB return RMSMOD_ERR_SHAPE and launch nothing (grad_x alone needs no
 *   scratch and has no such limit).  Nothing in the scratch needs clearing:
 *   every slot the upper tree levels read is written by the first level of
 *   the same call.
 *   Set-up: the first call on a device that asks for a token sum looks the
 *   array's address up once (it may load the module's device data); make
 *   that first call outside any stream capture.
 *   The scratch is one buffer per device: two calls whose work overlaps in
 *   time (different streams, or host threads issuing at once) race on it and
 *   give undefined token sums.  Calls on one stream are ordered and safe.
 * ---------------------------------------------------------------------- */
int ln_modulate_backward_static(const void* x, const void* scale, int64_t mod_bstride,
                                const void* grad_out, const float* mean, const float* rstd,
                                int64_t B, int64_t S, int64_t D, void* grad_x,
                                float* grad_scale, float* grad_shift, rmsmod_stream_t stream);

/* ------------------------------------------------------------------------
 * rmsnorm_modulate -- RMSNorm (optional weight), then the modulate chain.
 *   [ERNIE] §What "rounding-faithful" means here (rstd from sum_sq / H + eps;
 *   one final rounding of x * rstd * w; the aten modulate chain).
 *
 *     ms    = fp32 mean of f(x)^2 over the row;  rstd = 1 / sqrt(ms + eps)
 *     y[d]  = R((f(x[d]) * rstd) * f(w[d]))       (w = 1 when weight is NULL)
 *     out   = modulate chain of ln_modulate.
 *   weight nullable bf16 [D]; rstd_out nullable fp32 [B*S].
 * ---------------------------------------------------------------------- */
int rmsnorm_modulate(const void* x, const void* weight, const void* scale, const void* shift,
                     void* out, int64_t B, int64_t S, int64_t D, int64_t mod_bstride,
                     float eps, float* rstd_out, rmsmod_stream_t stream);

/* ------------------------------------------------------------------------
 * gated_rmsnorm_modulate -- gated residual add, then RMSNorm + modulate.
 *   [ERNIE] §What "rounding-faithful" means here (residual variant) and
 *   §Modifications (the second site returns the residual stream too).
 *
 *     res[r, d] = R(f(residual[r,d]) + f(R(f(gate_b[d]) * f(update[r,d]))))
 *     out       = rmsnorm_modulate(res)  (statistics over res)
 *   residual, update, res_out, out  bf16 [B*S*D]; res_out may equal residual.
 *   gate bf16 rows at gate + b * gate_bstride; weight nullable bf16 [D].
 * ---------------------------------------------------------------------- */
int gated_rmsnorm_modulate(const void* residual, const void* update, const void* gate,
                           int64_t gate_bstride, const void* weight, const void* scale,
                           const void* shift, int64_t mod_bstride, void* res_out, void* out,
                           int64_t B, int64_t S, int64_t D, float eps, float* rstd_out,
                           rmsmod_stream_t stream);

/* ------------------------------------------------------------------------
 * qk_layernorm -- per-head LayerNorm with affine over head_dim values, q rows
 * and k rows in one launch, each tensor with its own weight and bias.
 *   [GLM] §Motivation (qk-norm nn.LayerNorm(128) on (1, S, 32, 128)) and
 *   §What "rounding-faithful" means here (q and k in one launch; the same
 *   kernel for head_dim <= 128 rows).
 *
 *     z[d] = R(((f(x[d]) - mean) * rstd) * f(w[d]) + f(b[d]))
 *   q, q_out [rows_q * head_dim]; k, k_out [rows_k * head_dim] (bf16, dense);
 *   wq, bq, wk, bk bf16 [head_dim]; head_dim 64, 96 or 128.
 *   mean_out, rstd_out nullable fp32 [rows_q + rows_k], q rows first.
 *   q_out may equal q and k_out may equal k (in place).
 * ---------------------------------------------------------------------- */
int qk_layernorm(const void* q, const void* k, const void* wq, const void* bq, const void* wk,
                 const void* bk, void* q_out, void* k_out, int64_t rows_q, int64_t rows_k,
                 int64_t head_dim, float eps, float* mean_out, float* rstd_out,
                 rmsmod_stream_t stream);

/* qk_layernorm_strided -- the same on token-strided views, such as the q and
 * k slices of a fused QKV projection [tokens, 3, heads, head_dim].
 *   [GLM] §What "rounding-faithful" means here (qk bullet) and the sites it
 *   lists beyond (1, S, 32, 128).
 *
 *   Row (t, h) of q starts at q + t * q_token_stride + h * head_dim
 *   (elements): the heads_q rows of a token are contiguous, tokens are
 *   q_token_stride apart; likewise k (heads_k rows), q_out and k_out with
 *   their own token strides.  Strides are multiples of 8 and at least
 *   heads * head_dim (when tokens > 1).  Statistics rows are numbered
 *   t * heads + h, q rows first.  q_out may equal q with the same stride (in
 *   place, e.g. inside the QKV buffer); views that interleave in one buffer
 *   without sharing bytes are accepted; any other overlap is
 *   RMSMOD_ERR_UNSUPPORTED.  RMSMOD_ERR_STRIDE for a bad stride.
 * ---------------------------------------------------------------------- */
int qk_layernorm_strided(const void* q, const void* k, const void* wq, const void* bq,
                         const void* wk, const void* bk, void* q_out, void* k_out,
                         int64_t tokens, int64_t heads_q, int64_t heads_k, int64_t head_dim,
                         int64_t q_token_stride, int64_t k_token_stride,
                         int64_t q_out_token_stride, int64_t k_out_token_stride, float eps,
                         float* mean_out, float* rstd_out, rmsmod_stream_t stream);

/* ------------------------------------------------------------------------
 * rmsnorm_silu_cl -- channels-last RMSNorm * gamma, then SiLU, with the
 * deferred conv bias folded in first.
 *   [WAN] §Quality-gated (tiled [ROWS, C] RMSNorm+SiLU, optional conv_bias)
 *   and §New kernel, lossless (bias arithmetic of aten add_).
 *
 *   x is a dense channels-last activation viewed as `pixels` rows of C:
 *     xb[c]  = R(f(x[c]) + f(b16[c]))   b16 = R(bias[c]) for an fp32 bias;
 *                                       xb = x when bias is NULL
 *     rstd   = 1 / sqrt(fp32 mean of f(xb)^2 + eps)
 *     z[c]   = (f(xb[c]) * rstd) * f(gamma[c])        (fp32, unrounded)
 *     out[c] = R(z / (1 + exp(-z)))
 *   bias nullable ([C] fp32 when bias_is_fp32, else bf16); gamma bf16 [C];
 *   C a multiple of 8 in [8, RMSMOD_MAX_C]; rstd_out nullable fp32 [pixels].
 * ---------------------------------------------------------------------- */
int rmsnorm_silu_cl(const void* x, const void* bias, int bias_is_fp32, const void* gamma,
                    void* out, int64_t pixels, int64_t C, float eps, float* rstd_out,
                    rmsmod_stream_t stream);

/* ------------------------------------------------------------------------
 * Standalone elementwise chains (the fused kernels' epilogue / prologue,
 * exported on their own; bit-exact to the eager chain by construction).
 * ---------------------------------------------------------------------- */

/* modulate_scale_shift: out = R(f(R(f(y) * f(R(1 + f(scale_b))))) + f(shift_b)) over
 * y [B, S, D]; rows of scale/shift at base + b * mod_bstride.
 *   [FLUX] §Modifications commit 2 (modulate_scale_shift: round(round(x * round(1+scale)) + shift)). */
int modulate_scale_shift(const void* y, const void* scale, const void* shift, void* out,
                         int64_t B, int64_t S, int64_t D, int64_t mod_bstride,
                         rmsmod_stream_t stream);

/* modulate_scale_shift_f16: the same chain on fp16 storage, R16 = fp32 -> fp16
 * round-to-nearest-even (subnormals kept, overflow to Inf), every operand and
 * result an IEEE binary16 bit pattern; arguments, layout, aliasing and errors
 * as modulate_scale_shift.
 *   [FLUX] §Accuracy Tests (the modulate kernel covers bf16 and fp16). */
int modulate_scale_shift_f16(const void* y, const void* scale, const void* shift, void* out,
                             int64_t B, int64_t S, int64_t D, int64_t mod_bstride,
                             rmsmod_stream_t stream);

/* residual_gate_add: res = R(f(residual) + f(R(f(gate_b) * f(update)))) over [B, S, D].
 *   [GLM] §Motivation (ff gate) and [ERNIE] §What (residual variant). */
int residual_gate_add(const void* residual, const void* gate, const void* update,
                      int64_t gate_bstride, void* res_out, int64_t B, int64_t S, int64_t D,
                      rmsmod_stream_t stream);

/* conv_bias_epilogue: out = R(f(x) + f(b16)); with a residual h (nullable):
 * out = R(f(R(f(x) + f(b16))) + f(h)).  x, h, out: `pixels` channels-last rows of C.
 *   [WAN] §New kernel, lossless. */
int conv_bias_epilogue(const void* x, const void* bias, int bias_is_fp32, const void* h,
                       void* out, int64_t pixels, int64_t C, rmsmod_stream_t stream);

/* ------------------------------------------------------------------------
 * Predicates and diagnostics
 * ---------------------------------------------------------------------- */

enum {
    RMSMOD_OP_LN_MODULATE = 1,
    RMSMOD_OP_RMSNORM_MODULATE = 2,
    RMSMOD_OP_GATED_RMSNORM_MODULATE = 3,
    RMSMOD_OP_QK_LAYERNORM = 4,
    RMSMOD_OP_RMSNORM_SILU_CL = 5,
    RMSMOD_OP_LN_MODULATE_FOLDED = 6
};

/* 1 if `op` supports row length / channel count `D_or_C` and every non-NULL
 * pointer in ptrs[0..nptrs) is suitably aligned; 0 otherwise.  Never fails,
 * never touches the GPU.  ([WAN] §New kernel: the predicate never raises;
 * the kernel validates.) */
int rmsmod_supported(int op, int64_t D_or_C, const void* const* ptrs, int nptrs);

/* Device error word of the kernels launched so far on the current device:
 * bit 0 (RMSMOD_DEVICE_ERR_COPY_TIMEOUT) = an asynchronous bulk copy into
 * shared memory did not complete within the kernel's wait limit (1 s); the
 * kernel then finished without that data instead of hanging, so its output
 * is invalid.  Synchronous (it reads device memory); `clear` != 0 resets the
 * word.  Returns RMSMOD_OK or RMSMOD_ERR_CUDA / RMSMOD_ERR_NULL. */
#define RMSMOD_DEVICE_ERR_COPY_TIMEOUT 1u
int rmsmod_device_status(unsigned int* bits, int clear);

/* Self-test of that error path (the pages have no counterpart): launches
 * one warp on `stream` that waits `limit_ns` nanoseconds (1 .. 100,000,000)
 * on an mbarrier that nothing ever completes, the way every TMA-fed kernel
 * of this library bounds its waits, then sets RMSMOD_DEVICE_ERR_COPY_TIMEOUT
 * in the device error word and returns.  No fault, no hang: after the stream
 * is synchronised, rmsmod_device_status reports the bit and the context
 * stays usable.  Returns RMSMOD_OK, RMSMOD_ERR_SHAPE (limit out of range,
 * nothing launched) or RMSMOD_ERR_CUDA. */
int rmsmod_selftest_wait_timeout(uint64_t limit_ns, rmsmod_stream_t stream);

/* Static text for a status code (never NULL). */
const char* rmsmod_status_string(int status);

/* ABI version of this header: major * 10000 + minor * 100 + patch. */
int rmsmod_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RMSMOD_H */
