// noalloc.cu -- Fprop for callers that cannot allocate device memory.
//
// mxfp4_linear_fprop needs scratch for the quantised copies of X and W, and asks the
// caller for it.  Some callers have no way to provide it: a plugin running inside a
// host framework whose allocator owns all device memory and hands the plugin only
// its input and output pointers, or a latency-critical loop that must not call
// cudaMalloc/cudaFree (they can synchronise the whole device).  For them this file
// keeps a fixed scratch area in the library's own device memory and runs the same
// Fprop path on it.
#include <stdarg.h>
#include <stdio.h>

#include <mutex>

#include "internal.h"

namespace {

// The scratch area: kScratchBytes of device memory on every GPU where this library's
// kernels are loaded, held until the process exits.
constexpr size_t kScratchBytes = size_t(64) << 20;  // 64 MiB
static __device__ __align__(256) uint8_t g_fprop_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};  // device address of g_fprop_scratch, per device

// Host code cannot use g_fprop_scratch directly (its host-side name is only a
// stand-in), so the device address is looked up once per device, with that device
// current, and cached.
mxfp4_status scratch_for_current_device(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return mx::record_error(MXFP4_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return mx::record_error(MXFP4_ERR_UNSUPPORTED_DEVICE, "device index %d", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_fprop_scratch);
        if (e != cudaSuccess)
            return mx::record_error(MXFP4_ERR_CUDA, "cudaGetSymbolAddress(fprop scratch): %s", cudaGetErrorString(e));
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return MXFP4_OK;
}

}  // namespace

extern "C" size_t mxfp4_noalloc_scratch_bytes(void) { return kScratchBytes; }

extern "C" mxfp4_status mxfp4_linear_fprop_noalloc(const void* x, const void* w, int64_t M, int64_t N, int64_t K,
                                                   const mxfp4_config* cfg, void* y, mxfp4_tensor* save_xT,
                                                   mxfp4_tensor* save_wT, mxfp4_stream_t stream) {
    if (!cfg) return mx::record_error(MXFP4_ERR_INVALID_ARG, "cfg is NULL");
    if (M <= 0 || N <= 0 || K <= 0) return mx::record_error(MXFP4_ERR_UNSUPPORTED_SHAPE, "M, N, K must be positive");
    if (K % 32) return mx::record_error(MXFP4_ERR_UNSUPPORTED_SHAPE, "K %% 32 != 0");
    const size_t need = mxfp4_workspace_bytes(MXFP4_OP_FPROP, M, N, K, cfg);
    if (need > kScratchBytes)
        return mx::record_error(MXFP4_ERR_WORKSPACE,
                                "M=%lld N=%lld K=%lld needs %zu bytes of scratch, more than the %zu bytes of the "
                                "library's static scratch area; use mxfp4_linear_fprop with a caller workspace",
                                (long long)M, (long long)N, (long long)K, need, kScratchBytes);
    void* scratch = nullptr;
    mxfp4_status st = scratch_for_current_device(&scratch);
    if (st) return st;
    return mxfp4_linear_fprop(x, w, M, N, K, cfg, y, save_xT, save_wT, scratch, kScratchBytes, stream);
}
