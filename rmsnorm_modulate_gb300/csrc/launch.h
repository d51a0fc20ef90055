// Host-side launch interface between the C ABI (api.cu) and the kernel
// translation units.  Internal to librmsmod.so.
#pragma once

#include <atomic>
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

namespace rmsmod {

// Devices the library serves: the C ABI refuses a current device ordinal
// outside [0, kMaxDevices) before anything is launched.
constexpr int kMaxDevices = 64;

struct DeviceInfo {
    int device;  // in [0, kMaxDevices)
    int sms;
};

// One int per device, worked out by the first call on that device (a kernel
// attribute set, an occupancy query) and read by every later call.  Host
// threads whose first calls coincide serialise on one mutex, so the set-up
// runs once per device and a reader never sees a half-written value.
class PerDeviceInt {
public:
    // value for `device`; `make(int& v)` computes it (non-zero) on first use
    template <typename F>
    cudaError_t get(int device, int& value, F make)
    {
        if (device < 0 || device >= kMaxDevices)
            return cudaErrorInvalidDevice;
        int v = v_[device].load(std::memory_order_acquire);
        if (v == 0) {
            std::lock_guard<std::mutex> lock(mu_);
            v = v_[device].load(std::memory_order_relaxed);
            if (v == 0) {
                const cudaError_t e = make(v);
                if (e != cudaSuccess)
                    return e;
                v = v != 0 ? v : 1;
                v_[device].store(v, std::memory_order_release);
            }
        }
        value = v;
        return cudaSuccess;
    }

private:
    std::atomic<int> v_[kMaxDevices] = {};
    std::mutex mu_;
};

// Integer division by a runtime constant: q = (umulhi(n, m) + n) >> s,
// exact for every 32-bit n (Granlund-Montgomery round-up multiplier).
struct FastDiv {
    uint32_t d, m, s;

    static FastDiv make(uint32_t d)
    {
        FastDiv f;
        f.d = d;
        uint32_t s = 0;
        while ((1ull << s) < d)
            ++s;
        f.s = s;
        f.m = static_cast<uint32_t>(((1ull << 32) * ((1ull << s) - d)) / d + 1);
        return f;
    }

#ifdef __CUDACC__
    __device__ __forceinline__ uint32_t div(uint32_t n) const
    {
        return static_cast<uint32_t>((static_cast<uint64_t>(__umulhi(n, m)) + n) >> s);
    }
#endif
};

// kOpLNFold: the single-rounding tier of LN + modulate (the modulate folded
// into the LayerNorm's fp32 affine).
enum RowOp : int { kOpLN = 0, kOpRMS = 1, kOpGated = 2, kOpLNFold = 3 };

// Every kernel is launched with programmatic stream serialisation: its CTAs
// may be scheduled while the previous grid in the stream is draining, and the
// kernel's first statement (griddepcontrol.wait) holds them until that grid
// has completed and its writes are visible, so ordering is unchanged and only
// the launch gap is hidden.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), int grid, int block, int smem,
                             cudaStream_t stream, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(block));
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

struct RowArgs {
    const void* x;         // LN / RMS input rows
    const void* residual;  // gated
    const void* update;
    const void* gate;
    int64_t gate_bstride;  // in 8-element vectors
    const void* weight;    // nullable
    const void* scale;
    const void* shift;
    int64_t mod_bstride;   // in 8-element vectors
    void* res_out;
    void* out;
    float* mean_out;
    float* rstd_out;
    int64_t rows;
    int64_t S;
    int Dv;                // D / 8
    float n;               // D
    float inv_n;           // fp32(1 / D)
    float eps;
};

cudaError_t launch_row_kernel(int op, const RowArgs& a, const DeviceInfo& dev,
                              cudaStream_t stream);

// One of the two tensors of a qk launch: rows = tokens * heads head rows of
// head_dim values; the heads of a token are contiguous, tokens are in_ts /
// out_ts elements apart (a strided view of a fused QKV projection, or
// tokens = 1 for a dense tensor).
struct QkTensor {
    const void* in;
    void* out;
    const void* w;
    const void* b;
    int64_t tokens;
    int64_t heads;
    int64_t in_ts;   // elements, a multiple of 8
    int64_t out_ts;
};

struct QkArgs {
    QkTensor t[2];     // q, k
    float* mean_out;   // nullable [rows_q + rows_k], q rows first
    float* rstd_out;
    int head_dim;      // 64, 96 or 128
    float eps;
};

cudaError_t launch_qk_kernel(const QkArgs& a, const DeviceInfo& dev, cudaStream_t stream);

struct WanArgs {
    const void* x;
    const void* bias;  // nullable
    int bias_is_fp32;
    const void* gamma;
    void* out;
    float* rstd_out;
    int64_t pixels;
    int Cv;            // C / 8
    float n;           // C
    float inv_n;
    float eps;
};

cudaError_t launch_wan_kernel(const WanArgs& a, const DeviceInfo& dev, cudaStream_t stream);

enum EwOp : int { kEwModulate = 0, kEwGateAdd = 1, kEwBias = 2, kEwModulateF16 = 3 };

struct EwArgs {
    const void* a;        // y / residual / x
    const void* b;        // scale / gate / bias
    const void* c;        // shift / update / h (nullable for bias)
    void* out;
    int64_t bstride;      // scale/shift or gate batch stride (vectors)
    int bias_is_fp32;
    int64_t rows;         // B*S or pixels
    int64_t S;            // rows per batch (1 for the bias epilogue)
    int Dv;               // row length in vectors
};

cudaError_t launch_elementwise(int op, const EwArgs& a, const DeviceInfo& dev,
                               cudaStream_t stream);

struct BwdArgs {
    const void* x;         // forward input [B*S*D] bf16
    const void* scale;     // rows at base + b * mod_bstride
    int64_t mod_bstride;   // in 8-element vectors
    const void* grad_out;  // [B*S*D] bf16
    const float* mean;     // forward statistics [B*S]
    const float* rstd;
    void* grad_x;          // nullable [B*S*D] bf16
    float* grad_scale;     // nullable [B*D]
    float* grad_shift;     // nullable [B*D]
    void* workspace;       // [B][nblk][2][D] fp32 when a token sum is wanted
    int64_t B;
    int64_t S;
    int Dv;                // D / 8
    float n;               // D
    float inv_n;           // fp32(1 / D)
    int64_t nblk;          // ceil(S / 32)
    int64_t items;         // set by the launcher (row kernel work split)
    int64_t items_per_batch;
    int64_t chunk;
};
size_t backward_workspace_bytes(int64_t B, int64_t S, int64_t D);
// Size of the fixed device scratch behind ln_modulate_backward_static.
constexpr size_t kBackwardScratchBytes = size_t(8) << 20;
// Its address on `device` (looked up once per device, then cached).
cudaError_t backward_static_scratch(int device, void** ptr);
cudaError_t launch_backward(BwdArgs a, const DeviceInfo& dev, cudaStream_t stream);

// Each kernel translation unit keeps a device error word (bit kErrCopyTimeout:
// an asynchronous copy did not complete in time).  Reads it, optionally
// clearing it; synchronous.
cudaError_t row_kernels_error(unsigned* bits, bool clear);
cudaError_t qk_kernel_error(unsigned* bits, bool clear);
cudaError_t wan_kernel_error(unsigned* bits, bool clear);
cudaError_t backward_error(unsigned* bits, bool clear);

}  // namespace rmsmod
