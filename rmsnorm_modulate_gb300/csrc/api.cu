// C ABI of librmsmod.so: argument validation, device-attribute cache and
// dispatch to the kernel translation units.  Every check runs on the host
// before any CUDA call, so a rejected call touches neither the device nor
// the CUDA runtime.
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/rmsmod.h"
#include "launch.h"
#include "selftest.h"

#define RMSMOD_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

using rmsmod::DeviceInfo;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// [p, p + bytes) and [q, q + bytes2) overlap
bool overlap(const void* p, int64_t bytes, const void* q, int64_t bytes2)
{
    if (!p || !q || bytes <= 0 || bytes2 <= 0)
        return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(p), b0 = reinterpret_cast<uintptr_t>(q);
    return a0 < b0 + static_cast<uintptr_t>(bytes2) && b0 < a0 + static_cast<uintptr_t>(bytes);
}

// An output may coincide exactly with its own input; any other overlap is an error.
bool bad_alias(const void* out, const void* in, int64_t bytes, bool exact_ok)
{
    if (out == in)
        return !exact_ok;
    return overlap(out, bytes, in, bytes);
}

// rows * D as bytes, or -1 on overflow
int64_t tensor_bytes(int64_t rows, int64_t D)
{
    if (rows < 0 || D < 0)
        return -1;
    if (D != 0 && rows > (INT64_MAX / 4) / D)
        return -1;
    return rows * D * 2;
}

std::mutex g_dev_mutex;
DeviceInfo g_dev[64];
bool g_dev_valid[64];

int device_info(DeviceInfo& info)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return RMSMOD_ERR_DEVICE;
    }
    if (dev < 0 || dev >= 64)
        return RMSMOD_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (!g_dev_valid[dev]) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            sms <= 0) {
            cudaGetLastError();
            return RMSMOD_ERR_DEVICE;
        }
        g_dev[dev] = DeviceInfo{dev, sms};
        g_dev_valid[dev] = true;
    }
    info = g_dev[dev];
    return RMSMOD_OK;
}

int launch_status(cudaError_t e)
{
    if (e == cudaSuccess)
        return RMSMOD_OK;
    return RMSMOD_ERR_CUDA;
}

// Shape checks shared by the [B, S, D] operations.
int check_bsd(int64_t B, int64_t S, int64_t D)
{
    if (B < 0 || S < 0 || D <= 0)
        return RMSMOD_ERR_SHAPE;
    if (D % 8 != 0 || D > RMSMOD_MAX_D)
        return RMSMOD_ERR_SHAPE;
    if (B != 0 && S > INT64_MAX / B)
        return RMSMOD_ERR_SHAPE;
    if (tensor_bytes(B * S, D) < 0)
        return RMSMOD_ERR_SHAPE;
    return RMSMOD_OK;
}

int check_bstride(int64_t s)
{
    if (s < 0 || s % 8 != 0)
        return RMSMOD_ERR_STRIDE;
    return RMSMOD_OK;
}

}  // namespace

RMSMOD_EXPORT int rmsmod_version(void) { return 10000; }

RMSMOD_EXPORT const char* rmsmod_status_string(int status)
{
    switch (status) {
    case RMSMOD_OK:
        return "ok";
    case RMSMOD_ERR_NULL:
        return "a required pointer is NULL";
    case RMSMOD_ERR_SHAPE:
        return "unsupported or inconsistent size";
    case RMSMOD_ERR_ALIGN:
        return "a pointer is not aligned as required (16 bytes for tensors)";
    case RMSMOD_ERR_STRIDE:
        return "a batch stride is negative or not a multiple of 8 elements";
    case RMSMOD_ERR_UNSUPPORTED:
        return "overlapping buffers or an unsupported combination of arguments";
    case RMSMOD_ERR_CUDA:
        return "the CUDA runtime reported an error at launch";
    case RMSMOD_ERR_DEVICE:
        return "no usable CUDA device is current";
    default:
        return "unknown status";
    }
}

RMSMOD_EXPORT int rmsmod_device_status(unsigned int* bits, int clear)
{
    if (!bits)
        return RMSMOD_ERR_NULL;
    unsigned a = 0, b = 0, c = 0, d = 0, e = 0;
    if (rmsmod::row_kernels_error(&a, clear != 0) != cudaSuccess ||
        rmsmod::qk_kernel_error(&b, clear != 0) != cudaSuccess ||
        rmsmod::wan_kernel_error(&c, clear != 0) != cudaSuccess ||
        rmsmod::backward_error(&d, clear != 0) != cudaSuccess ||
        rmsmod::selftest_error(&e, clear != 0) != cudaSuccess) {
        cudaGetLastError();
        return RMSMOD_ERR_CUDA;
    }
    *bits = a | b | c | d | e;
    return RMSMOD_OK;
}

RMSMOD_EXPORT int rmsmod_selftest_wait_timeout(uint64_t limit_ns, rmsmod_stream_t stream)
{
    if (limit_ns == 0 || limit_ns > 100000000ull)
        return RMSMOD_ERR_SHAPE;
    return launch_status(rmsmod::launch_selftest_wait(limit_ns, stream));
}

static bool qk_head_dim_ok(int64_t hd) { return hd == 64 || hd == 96 || hd == 128; }

RMSMOD_EXPORT int rmsmod_supported(int op, int64_t D_or_C, const void* const* ptrs, int nptrs)
{
    if (D_or_C <= 0 || D_or_C % 8 != 0)
        return 0;
    switch (op) {
    case RMSMOD_OP_LN_MODULATE:
    case RMSMOD_OP_LN_MODULATE_FOLDED:
    case RMSMOD_OP_RMSNORM_MODULATE:
    case RMSMOD_OP_GATED_RMSNORM_MODULATE:
        if (D_or_C > RMSMOD_MAX_D)
            return 0;
        break;
    case RMSMOD_OP_QK_LAYERNORM:
        if (!qk_head_dim_ok(D_or_C))
            return 0;
        break;
    case RMSMOD_OP_RMSNORM_SILU_CL:
        if (D_or_C > RMSMOD_MAX_C || D_or_C < 8)
            return 0;
        break;
    default:
        return 0;
    }
    if (nptrs < 0 || (nptrs > 0 && !ptrs))
        return 0;
    for (int i = 0; i < nptrs; ++i)
        if (ptrs[i] && !aligned(ptrs[i], 16))
            return 0;
    return 1;
}

static int ln_modulate_op(int op, const void* x, const void* scale, const void* shift, void* out,
                          int64_t B, int64_t S, int64_t D, int64_t mod_bstride, float eps,
                          float* mean_out, float* rstd_out, rmsmod_stream_t stream)
{
    int st = check_bsd(B, S, D);
    if (st != RMSMOD_OK)
        return st;
    if ((st = check_bstride(mod_bstride)) != RMSMOD_OK)
        return st;
    const int64_t rows = B * S;
    if (rows == 0)
        return RMSMOD_OK;
    if (!x || !scale || !shift || !out)
        return RMSMOD_ERR_NULL;
    if (!aligned(x, 16) || !aligned(scale, 16) || !aligned(shift, 16) || !aligned(out, 16) ||
        !aligned(mean_out, 4) || !aligned(rstd_out, 4))
        return RMSMOD_ERR_ALIGN;
    const int64_t bytes = tensor_bytes(rows, D);
    if (bad_alias(out, x, bytes, true) || overlap(out, bytes, scale, 2 * D) ||
        overlap(out, bytes, shift, 2 * D) || overlap(mean_out, 4 * rows, out, bytes) ||
        overlap(rstd_out, 4 * rows, out, bytes) || overlap(mean_out, 4 * rows, rstd_out, 4 * rows))
        return RMSMOD_ERR_UNSUPPORTED;
    DeviceInfo dev;
    if ((st = device_info(dev)) != RMSMOD_OK)
        return st;
    rmsmod::RowArgs a{};
    a.x = x;
    a.scale = scale;
    a.shift = shift;
    a.mod_bstride = mod_bstride / 8;
    a.out = out;
    a.mean_out = mean_out;
    a.rstd_out = rstd_out;
    a.rows = rows;
    a.S = S;
    a.Dv = static_cast<int>(D / 8);
    a.n = static_cast<float>(D);
    a.inv_n = 1.0f / static_cast<float>(D);
    a.eps = eps;
    return launch_status(rmsmod::launch_row_kernel(op, a, dev, stream));
}

RMSMOD_EXPORT int ln_modulate(const void* x, const void* scale, const void* shift, void* out,
                              int64_t B, int64_t S, int64_t D, int64_t mod_bstride, float eps,
                              float* mean_out, float* rstd_out, rmsmod_stream_t stream)
{
    return ln_modulate_op(rmsmod::kOpLN, x, scale, shift, out, B, S, D, mod_bstride, eps,
                          mean_out, rstd_out, stream);
}

RMSMOD_EXPORT int ln_modulate_folded(const void* x, const void* scale, const void* shift,
                                     void* out, int64_t B, int64_t S, int64_t D,
                                     int64_t mod_bstride, float eps, float* mean_out,
                                     float* rstd_out, rmsmod_stream_t stream)
{
    return ln_modulate_op(rmsmod::kOpLNFold, x, scale, shift, out, B, S, D, mod_bstride, eps,
                          mean_out, rstd_out, stream);
}

RMSMOD_EXPORT size_t ln_modulate_backward_workspace_bytes(int64_t B, int64_t S, int64_t D)
{
    if (B <= 0 || S <= 0 || D <= 0 || D > RMSMOD_MAX_D || B > INT64_MAX / S)
        return 0;
    return rmsmod::backward_workspace_bytes(B, S, D);
}

RMSMOD_EXPORT int ln_modulate_backward(const void* x, const void* scale, int64_t mod_bstride,
                                       const void* grad_out, const float* mean,
                                       const float* rstd, int64_t B, int64_t S, int64_t D,
                                       void* grad_x, float* grad_scale, float* grad_shift,
                                       void* workspace, size_t workspace_bytes,
                                       rmsmod_stream_t stream)
{
    int st = check_bsd(B, S, D);
    if (st != RMSMOD_OK)
        return st;
    if ((st = check_bstride(mod_bstride)) != RMSMOD_OK)
        return st;
    const int64_t rows = B * S;
    if (rows == 0 || (!grad_x && !grad_scale && !grad_shift))
        return RMSMOD_OK;
    if (!x || !scale || !grad_out || !mean || !rstd)
        return RMSMOD_ERR_NULL;
    const bool tokens = grad_scale || grad_shift;
    if (tokens && !workspace)
        return RMSMOD_ERR_NULL;
    if (!aligned(x, 16) || !aligned(scale, 16) || !aligned(grad_out, 16) || !aligned(mean, 4) ||
        !aligned(rstd, 4) || !aligned(grad_x, 16) || !aligned(grad_scale, 16) ||
        !aligned(grad_shift, 16) || !aligned(workspace, 256))
        return RMSMOD_ERR_ALIGN;
    const size_t need = rmsmod::backward_workspace_bytes(B, S, D);
    if (tokens && workspace_bytes < need)
        return RMSMOD_ERR_SHAPE;
    const int64_t bytes = tensor_bytes(rows, D);
    const int64_t col_bytes = B * D * 4;
    // the scale rows the kernels read: row b at scale + b * mod_bstride
    const int64_t scale_bytes = ((B - 1) * mod_bstride + D) * 2;
    // outputs overlap no input and no other output (grad_x may not alias x):
    // the kernels write grad_x, the workspace and the gradients while other
    // CTAs still read x, grad_out, scale, mean and rstd
    struct Span {
        const void* p;
        int64_t n;
    };
    const Span ins[] = {{x, bytes}, {grad_out, bytes}, {scale, scale_bytes},
                        {mean, 4 * rows}, {rstd, 4 * rows}};
    for (const Span& in : ins)
        if (overlap(grad_x, bytes, in.p, in.n) || overlap(grad_scale, col_bytes, in.p, in.n) ||
            overlap(grad_shift, col_bytes, in.p, in.n) ||
            (tokens && overlap(workspace, static_cast<int64_t>(need), in.p, in.n)))
            return RMSMOD_ERR_UNSUPPORTED;
    if (overlap(grad_x, bytes, grad_scale, col_bytes) ||
        overlap(grad_x, bytes, grad_shift, col_bytes) ||
        overlap(grad_scale, col_bytes, grad_shift, col_bytes) ||
        (tokens && (overlap(workspace, static_cast<int64_t>(need), grad_x, bytes) ||
                    overlap(workspace, static_cast<int64_t>(need), grad_scale, col_bytes) ||
                    overlap(workspace, static_cast<int64_t>(need), grad_shift, col_bytes))) ||
        overlap(grad_x, bytes, mean, 4 * rows) || overlap(grad_x, bytes, rstd, 4 * rows))
        return RMSMOD_ERR_UNSUPPORTED;
    DeviceInfo dev;
    if ((st = device_info(dev)) != RMSMOD_OK)
        return st;
    rmsmod::BwdArgs a{};
    a.x = x;
    a.scale = scale;
    a.mod_bstride = mod_bstride / 8;
    a.grad_out = grad_out;
    a.mean = mean;
    a.rstd = rstd;
    a.grad_x = grad_x;
    a.grad_scale = grad_scale;
    a.grad_shift = grad_shift;
    a.workspace = workspace;
    a.B = B;
    a.S = S;
    a.Dv = static_cast<int>(D / 8);
    a.n = static_cast<float>(D);
    a.inv_n = 1.0f / static_cast<float>(D);
    a.nblk = (S + 31) / 32;
    return launch_status(rmsmod::launch_backward(a, dev, stream));
}

RMSMOD_EXPORT int ln_modulate_backward_static(const void* x, const void* scale,
                                              int64_t mod_bstride, const void* grad_out,
                                              const float* mean, const float* rstd, int64_t B,
                                              int64_t S, int64_t D, void* grad_x,
                                              float* grad_scale, float* grad_shift,
                                              rmsmod_stream_t stream)
{
    const bool tokens = grad_scale || grad_shift;
    void* scratch = nullptr;
    if (tokens) {
        int st = check_bsd(B, S, D);
        if (st != RMSMOD_OK)
            return st;
        if (B * S > 0 && rmsmod::backward_workspace_bytes(B, S, D) > rmsmod::kBackwardScratchBytes)
            return RMSMOD_ERR_SHAPE;
        DeviceInfo dev;
        if ((st = device_info(dev)) != RMSMOD_OK)
            return st;
        if (rmsmod::backward_static_scratch(dev.device, &scratch) != cudaSuccess) {
            cudaGetLastError();
            return RMSMOD_ERR_CUDA;
        }
    }
    return ln_modulate_backward(x, scale, mod_bstride, grad_out, mean, rstd, B, S, D, grad_x,
                                grad_scale, grad_shift, scratch,
                                tokens ? rmsmod::kBackwardScratchBytes : 0, stream);
}

RMSMOD_EXPORT int rmsnorm_modulate(const void* x, const void* weight, const void* scale,
                                   const void* shift, void* out, int64_t B, int64_t S, int64_t D,
                                   int64_t mod_bstride, float eps, float* rstd_out,
                                   rmsmod_stream_t stream)
{
    int st = check_bsd(B, S, D);
    if (st != RMSMOD_OK)
        return st;
    if ((st = check_bstride(mod_bstride)) != RMSMOD_OK)
        return st;
    const int64_t rows = B * S;
    if (rows == 0)
        return RMSMOD_OK;
    if (!x || !scale || !shift || !out)
        return RMSMOD_ERR_NULL;
    if (!aligned(x, 16) || !aligned(weight, 16) || !aligned(scale, 16) || !aligned(shift, 16) ||
        !aligned(out, 16) || !aligned(rstd_out, 4))
        return RMSMOD_ERR_ALIGN;
    const int64_t bytes = tensor_bytes(rows, D);
    if (bad_alias(out, x, bytes, true) || overlap(out, bytes, weight, 2 * D) ||
        overlap(out, bytes, scale, 2 * D) || overlap(out, bytes, shift, 2 * D) ||
        overlap(rstd_out, 4 * rows, out, bytes))
        return RMSMOD_ERR_UNSUPPORTED;
    DeviceInfo dev;
    if ((st = device_info(dev)) != RMSMOD_OK)
        return st;
    rmsmod::RowArgs a{};
    a.x = x;
    a.weight = weight;
    a.scale = scale;
    a.shift = shift;
    a.mod_bstride = mod_bstride / 8;
    a.out = out;
    a.rstd_out = rstd_out;
    a.rows = rows;
    a.S = S;
    a.Dv = static_cast<int>(D / 8);
    a.n = static_cast<float>(D);
    a.inv_n = 1.0f / static_cast<float>(D);
    a.eps = eps;
    return launch_status(rmsmod::launch_row_kernel(rmsmod::kOpRMS, a, dev, stream));
}

RMSMOD_EXPORT int gated_rmsnorm_modulate(const void* residual, const void* update,
                                         const void* gate, int64_t gate_bstride,
                                         const void* weight, const void* scale,
                                         const void* shift, int64_t mod_bstride, void* res_out,
                                         void* out, int64_t B, int64_t S, int64_t D, float eps,
                                         float* rstd_out, rmsmod_stream_t stream)
{
    int st = check_bsd(B, S, D);
    if (st != RMSMOD_OK)
        return st;
    if ((st = check_bstride(mod_bstride)) != RMSMOD_OK ||
        (st = check_bstride(gate_bstride)) != RMSMOD_OK)
        return st;
    const int64_t rows = B * S;
    if (rows == 0)
        return RMSMOD_OK;
    if (!residual || !update || !gate || !scale || !shift || !res_out || !out)
        return RMSMOD_ERR_NULL;
    if (!aligned(residual, 16) || !aligned(update, 16) || !aligned(gate, 16) ||
        !aligned(weight, 16) || !aligned(scale, 16) || !aligned(shift, 16) ||
        !aligned(res_out, 16) || !aligned(out, 16) || !aligned(rstd_out, 4))
        return RMSMOD_ERR_ALIGN;
    const int64_t bytes = tensor_bytes(rows, D);
    if (bad_alias(res_out, residual, bytes, true) || bad_alias(res_out, update, bytes, false) ||
        bad_alias(out, residual, bytes, false) || bad_alias(out, update, bytes, false) ||
        bad_alias(out, res_out, bytes, false) || overlap(out, bytes, gate, 2 * D) ||
        overlap(res_out, bytes, gate, 2 * D) || overlap(out, bytes, weight, 2 * D) ||
        overlap(out, bytes, scale, 2 * D) || overlap(out, bytes, shift, 2 * D) ||
        overlap(rstd_out, 4 * rows, out, bytes) || overlap(rstd_out, 4 * rows, res_out, bytes))
        return RMSMOD_ERR_UNSUPPORTED;
    DeviceInfo dev;
    if ((st = device_info(dev)) != RMSMOD_OK)
        return st;
    rmsmod::RowArgs a{};
    a.residual = residual;
    a.update = update;
    a.gate = gate;
    a.gate_bstride = gate_bstride / 8;
    a.weight = weight;
    a.scale = scale;
    a.shift = shift;
    a.mod_bstride = mod_bstride / 8;
    a.res_out = res_out;
    a.out = out;
    a.rstd_out = rstd_out;
    a.rows = rows;
    a.S = S;
    a.Dv = static_cast<int>(D / 8);
    a.n = static_cast<float>(D);
    a.inv_n = 1.0f / static_cast<float>(D);
    a.eps = eps;
    return launch_status(rmsmod::launch_row_kernel(rmsmod::kOpGated, a, dev, stream));
}

// Do two token-strided tensors (tokens rows of `len` bytes, `ts` bytes apart)
// share a byte?  Same stride: compare the per-token windows modulo the
// stride (q and k views of one fused QKV buffer interleave without
// overlapping); otherwise compare the spans.
static bool strided_overlap(const void* a, int64_t a_ts, int64_t a_len, const void* b,
                            int64_t b_ts, int64_t b_len, int64_t tokens)
{
    if (!a || !b || tokens <= 0 || a_len <= 0 || b_len <= 0)
        return false;
    const int64_t a_span = (tokens - 1) * a_ts + a_len, b_span = (tokens - 1) * b_ts + b_len;
    if (!overlap(a, a_span, b, b_span))
        return false;
    if (a_ts != b_ts || tokens == 1)
        return true;
    const int64_t ts = a_ts;
    const int64_t diff = static_cast<int64_t>(reinterpret_cast<uintptr_t>(b) -
                                              reinterpret_cast<uintptr_t>(a));
    int64_t r = diff % ts;
    if (r < 0)
        r += ts;
    return r < a_len || r + b_len > ts;
}

static int qk_launch(const void* q, const void* k, const void* wq, const void* bq,
                     const void* wk, const void* bk, void* q_out, void* k_out, int64_t tokens,
                     int64_t heads_q, int64_t heads_k, int64_t head_dim, int64_t q_ts,
                     int64_t k_ts, int64_t qo_ts, int64_t ko_ts, float eps, float* mean_out,
                     float* rstd_out, rmsmod_stream_t stream)
{
    const int64_t rows_q = tokens * heads_q, rows_k = tokens * heads_k;
    if (rows_q + rows_k == 0)
        return RMSMOD_OK;
    if ((rows_q > 0 && (!q || !wq || !bq || !q_out)) ||
        (rows_k > 0 && (!k || !wk || !bk || !k_out)))
        return RMSMOD_ERR_NULL;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(wq, 16) || !aligned(bq, 16) ||
        !aligned(wk, 16) || !aligned(bk, 16) || !aligned(q_out, 16) || !aligned(k_out, 16) ||
        !aligned(mean_out, 4) || !aligned(rstd_out, 4))
        return RMSMOD_ERR_ALIGN;
    // byte geometry of the four views: tokens rows of heads * head_dim values
    const int64_t ql = 2 * heads_q * head_dim, kl = 2 * heads_k * head_dim;
    const int64_t qts = 2 * q_ts, kts = 2 * k_ts, qots = 2 * qo_ts, kots = 2 * ko_ts;
    const int64_t nst = 4 * (rows_q + rows_k);
    const int64_t qo_span = rows_q ? (tokens - 1) * qots + ql : 0;
    const int64_t ko_span = rows_k ? (tokens - 1) * kots + kl : 0;
    // an output may be its own input exactly (same base, same stride)
    const bool q_inplace = q_out == q && qo_ts == q_ts;
    const bool k_inplace = k_out == k && ko_ts == k_ts;
    if ((!q_inplace && strided_overlap(q_out, qots, ql, q, qts, ql, rows_q ? tokens : 0)) ||
        (!k_inplace && strided_overlap(k_out, kots, kl, k, kts, kl, rows_k ? tokens : 0)) ||
        strided_overlap(q_out, qots, ql, k, kts, kl, rows_q && rows_k ? tokens : 0) ||
        strided_overlap(k_out, kots, kl, q, qts, ql, rows_q && rows_k ? tokens : 0) ||
        strided_overlap(q_out, qots, ql, k_out, kots, kl, rows_q && rows_k ? tokens : 0) ||
        overlap(mean_out, nst, rstd_out, nst) || overlap(q_out, qo_span, mean_out, nst) ||
        overlap(k_out, ko_span, mean_out, nst) || overlap(q_out, qo_span, rstd_out, nst) ||
        overlap(k_out, ko_span, rstd_out, nst))
        return RMSMOD_ERR_UNSUPPORTED;
    DeviceInfo dev;
    int st;
    if ((st = device_info(dev)) != RMSMOD_OK)
        return st;
    rmsmod::QkArgs a{};
    a.t[0] = rmsmod::QkTensor{q, q_out, wq, bq, rows_q ? tokens : 0, heads_q, q_ts, qo_ts};
    a.t[1] = rmsmod::QkTensor{k, k_out, wk, bk, rows_k ? tokens : 0, heads_k, k_ts, ko_ts};
    a.mean_out = mean_out;
    a.rstd_out = rstd_out;
    a.head_dim = static_cast<int>(head_dim);
    a.eps = eps;
    return launch_status(rmsmod::launch_qk_kernel(a, dev, stream));
}

RMSMOD_EXPORT int qk_layernorm(const void* q, const void* k, const void* wq, const void* bq,
                               const void* wk, const void* bk, void* q_out, void* k_out,
                               int64_t rows_q, int64_t rows_k, int64_t head_dim, float eps,
                               float* mean_out, float* rstd_out, rmsmod_stream_t stream)
{
    if (rows_q < 0 || rows_k < 0 || !qk_head_dim_ok(head_dim))
        return RMSMOD_ERR_SHAPE;
    if (tensor_bytes(rows_q, head_dim) < 0 || tensor_bytes(rows_k, head_dim) < 0 ||
        rows_q > INT64_MAX / 2 - rows_k)
        return RMSMOD_ERR_SHAPE;
    // a dense tensor is one "token" of rows heads
    if (rows_q + rows_k == 0)
        return RMSMOD_OK;
    return qk_launch(q, k, wq, bq, wk, bk, q_out, k_out, 1, rows_q, rows_k, head_dim,
                     rows_q * head_dim, rows_k * head_dim, rows_q * head_dim,
                     rows_k * head_dim, eps, mean_out, rstd_out, stream);
}

RMSMOD_EXPORT int qk_layernorm_strided(const void* q, const void* k, const void* wq,
                                       const void* bq, const void* wk, const void* bk,
                                       void* q_out, void* k_out, int64_t tokens,
                                       int64_t heads_q, int64_t heads_k, int64_t head_dim,
                                       int64_t q_token_stride, int64_t k_token_stride,
                                       int64_t q_out_token_stride, int64_t k_out_token_stride,
                                       float eps, float* mean_out, float* rstd_out,
                                       rmsmod_stream_t stream)
{
    if (tokens < 0 || heads_q < 0 || heads_k < 0 || !qk_head_dim_ok(head_dim))
        return RMSMOD_ERR_SHAPE;
    if (tokens > 0 && (heads_q > INT64_MAX / head_dim / tokens / 2 ||
                       heads_k > INT64_MAX / head_dim / tokens / 2))
        return RMSMOD_ERR_SHAPE;
    const int64_t strides[4] = {q_token_stride, k_token_stride, q_out_token_stride,
                                k_out_token_stride};
    const int64_t need[4] = {heads_q * head_dim, heads_k * head_dim, heads_q * head_dim,
                             heads_k * head_dim};
    for (int i = 0; i < 4; ++i)
        if (need[i] > 0 && tokens > 1 &&
            (strides[i] < need[i] || strides[i] % 8 != 0 || strides[i] > INT64_MAX / 4 / tokens))
            return RMSMOD_ERR_STRIDE;
    return qk_launch(q, k, wq, bq, wk, bk, q_out, k_out, tokens, heads_q, heads_k, head_dim,
                     q_token_stride, k_token_stride, q_out_token_stride, k_out_token_stride, eps,
                     mean_out, rstd_out, stream);
}

RMSMOD_EXPORT int rmsnorm_silu_cl(const void* x, const void* bias, int bias_is_fp32,
                                  const void* gamma, void* out, int64_t pixels, int64_t C,
                                  float eps, float* rstd_out, rmsmod_stream_t stream)
{
    if (pixels < 0 || C < 8 || C % 8 != 0 || C > RMSMOD_MAX_C)
        return RMSMOD_ERR_SHAPE;
    if (tensor_bytes(pixels, C) < 0)
        return RMSMOD_ERR_SHAPE;
    if (pixels == 0)
        return RMSMOD_OK;
    if (!x || !gamma || !out)
        return RMSMOD_ERR_NULL;
    if (!aligned(x, 16) || !aligned(bias, 16) || !aligned(gamma, 16) || !aligned(out, 16) ||
        !aligned(rstd_out, 4))
        return RMSMOD_ERR_ALIGN;
    const int64_t bytes = tensor_bytes(pixels, C);
    const int64_t bias_bytes = bias_is_fp32 ? 4 * C : 2 * C;
    if (bad_alias(out, x, bytes, true) || overlap(out, bytes, bias, bias_bytes) ||
        overlap(out, bytes, gamma, 2 * C) || overlap(rstd_out, 4 * pixels, out, bytes))
        return RMSMOD_ERR_UNSUPPORTED;
    DeviceInfo dev;
    int st;
    if ((st = device_info(dev)) != RMSMOD_OK)
        return st;
    rmsmod::WanArgs a{};
    a.x = x;
    a.bias = bias;
    a.bias_is_fp32 = bias_is_fp32 ? 1 : 0;
    a.gamma = gamma;
    a.out = out;
    a.rstd_out = rstd_out;
    a.pixels = pixels;
    a.Cv = static_cast<int>(C / 8);
    a.n = static_cast<float>(C);
    a.inv_n = 1.0f / static_cast<float>(C);
    a.eps = eps;
    return launch_status(rmsmod::launch_wan_kernel(a, dev, stream));
}

// ---- standalone elementwise chains --------------------------------------

namespace {

// Elementwise kernels index 16-byte vectors with 32-bit integers.
constexpr int64_t kMaxEwVectors = (int64_t{1} << 31) - 1;

int check_ew_rows(int64_t rows, int64_t D)
{
    if (rows < 0 || D <= 0 || D % 8 != 0 || D > (int64_t{1} << 30))
        return RMSMOD_ERR_SHAPE;
    if (tensor_bytes(rows, D) < 0 || rows * (D / 8) > kMaxEwVectors)
        return RMSMOD_ERR_SHAPE;
    return RMSMOD_OK;
}

}  // namespace

static int modulate_op(int op, const void* y, const void* scale, const void* shift, void* out,
                       int64_t B, int64_t S, int64_t D, int64_t mod_bstride,
                       rmsmod_stream_t stream)
{
    if (B < 0 || S < 0 || (B != 0 && S > INT64_MAX / B))
        return RMSMOD_ERR_SHAPE;
    int st = check_ew_rows(B * S, D);
    if (st != RMSMOD_OK)
        return st;
    if (S > UINT32_MAX)
        return RMSMOD_ERR_SHAPE;
    if ((st = check_bstride(mod_bstride)) != RMSMOD_OK)
        return st;
    if (B * S == 0)
        return RMSMOD_OK;
    if (!y || !scale || !shift || !out)
        return RMSMOD_ERR_NULL;
    if (!aligned(y, 16) || !aligned(scale, 16) || !aligned(shift, 16) || !aligned(out, 16))
        return RMSMOD_ERR_ALIGN;
    const int64_t bytes = tensor_bytes(B * S, D);
    if (bad_alias(out, y, bytes, true) || overlap(out, bytes, scale, 2 * D) ||
        overlap(out, bytes, shift, 2 * D))
        return RMSMOD_ERR_UNSUPPORTED;
    DeviceInfo dev;
    if ((st = device_info(dev)) != RMSMOD_OK)
        return st;
    rmsmod::EwArgs a{};
    a.a = y;
    a.b = scale;
    a.c = shift;
    a.out = out;
    a.bstride = mod_bstride / 8;
    a.rows = B * S;
    a.S = S;
    a.Dv = static_cast<int>(D / 8);
    return launch_status(rmsmod::launch_elementwise(op, a, dev, stream));
}

RMSMOD_EXPORT int modulate_scale_shift(const void* y, const void* scale, const void* shift,
                                       void* out, int64_t B, int64_t S, int64_t D,
                                       int64_t mod_bstride, rmsmod_stream_t stream)
{
    return modulate_op(rmsmod::kEwModulate, y, scale, shift, out, B, S, D, mod_bstride, stream);
}

RMSMOD_EXPORT int modulate_scale_shift_f16(const void* y, const void* scale, const void* shift,
                                           void* out, int64_t B, int64_t S, int64_t D,
                                           int64_t mod_bstride, rmsmod_stream_t stream)
{
    return modulate_op(rmsmod::kEwModulateF16, y, scale, shift, out, B, S, D, mod_bstride,
                       stream);
}

RMSMOD_EXPORT int residual_gate_add(const void* residual, const void* gate, const void* update,
                                    int64_t gate_bstride, void* res_out, int64_t B, int64_t S,
                                    int64_t D, rmsmod_stream_t stream)
{
    if (B < 0 || S < 0 || (B != 0 && S > INT64_MAX / B))
        return RMSMOD_ERR_SHAPE;
    int st = check_ew_rows(B * S, D);
    if (st != RMSMOD_OK)
        return st;
    if (S > UINT32_MAX)
        return RMSMOD_ERR_SHAPE;
    if ((st = check_bstride(gate_bstride)) != RMSMOD_OK)
        return st;
    if (B * S == 0)
        return RMSMOD_OK;
    if (!residual || !gate || !update || !res_out)
        return RMSMOD_ERR_NULL;
    if (!aligned(residual, 16) || !aligned(gate, 16) || !aligned(update, 16) ||
        !aligned(res_out, 16))
        return RMSMOD_ERR_ALIGN;
    const int64_t bytes = tensor_bytes(B * S, D);
    if (bad_alias(res_out, residual, bytes, true) || bad_alias(res_out, update, bytes, true) ||
        overlap(res_out, bytes, gate, 2 * D))
        return RMSMOD_ERR_UNSUPPORTED;
    DeviceInfo dev;
    if ((st = device_info(dev)) != RMSMOD_OK)
        return st;
    rmsmod::EwArgs a{};
    a.a = residual;
    a.b = gate;
    a.c = update;
    a.out = res_out;
    a.bstride = gate_bstride / 8;
    a.rows = B * S;
    a.S = S;
    a.Dv = static_cast<int>(D / 8);
    return launch_status(rmsmod::launch_elementwise(rmsmod::kEwGateAdd, a, dev, stream));
}

RMSMOD_EXPORT int conv_bias_epilogue(const void* x, const void* bias, int bias_is_fp32,
                                     const void* h, void* out, int64_t pixels, int64_t C,
                                     rmsmod_stream_t stream)
{
    int st = check_ew_rows(pixels, C);
    if (st != RMSMOD_OK)
        return st;
    if (pixels == 0)
        return RMSMOD_OK;
    if (!x || !bias || !out)
        return RMSMOD_ERR_NULL;
    if (!aligned(x, 16) || !aligned(bias, 16) || !aligned(h, 16) || !aligned(out, 16))
        return RMSMOD_ERR_ALIGN;
    const int64_t bytes = tensor_bytes(pixels, C);
    const int64_t bias_bytes = bias_is_fp32 ? 4 * C : 2 * C;
    if (bad_alias(out, x, bytes, true) || bad_alias(out, h, bytes, true) ||
        overlap(out, bytes, bias, bias_bytes))
        return RMSMOD_ERR_UNSUPPORTED;
    DeviceInfo dev;
    if ((st = device_info(dev)) != RMSMOD_OK)
        return st;
    rmsmod::EwArgs a{};
    a.a = x;
    a.b = bias;
    a.c = h;
    a.out = out;
    a.bias_is_fp32 = bias_is_fp32 ? 1 : 0;
    a.rows = pixels;
    a.S = 1;
    a.Dv = static_cast<int>(C / 8);
    return launch_status(rmsmod::launch_elementwise(rmsmod::kEwBias, a, dev, stream));
}
