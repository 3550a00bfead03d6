// mxfp4_api.cu -- host side of the C ABI (include/mxfp4.h): argument validation,
// tensor-map encoding, workspace carving and kernel dispatch.  Nothing here
// allocates memory; the only global state is one device status word per device.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include <initializer_list>

#include "internal.h"
#include "ptx.cuh"

namespace mx {

__device__ uint32_t g_status_word;

namespace {

constexpr int kMaxDevices = 64;
thread_local char t_last_error[512] = "";
thread_local uint64_t t_wait_ns = 0;
thread_local int t_inject_gemm_faults = 0;  // test hook: see mxfp4_test_inject_gemm_fault
constexpr uint64_t kDefaultWaitNs = 2000000000ull;

std::mutex g_mu;
uint32_t* g_status_ptr[kMaxDevices] = {};
int g_device_ok[kMaxDevices] = {};  // 0 unknown, 1 ok, -1 unsupported

mxfp4_status fail(mxfp4_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_last_error, sizeof t_last_error, fmt, ap);
    va_end(ap);
    return st;
}

mxfp4_status ok() {
    t_last_error[0] = 0;
    return MXFP4_OK;
}

mxfp4_status cuda_fail(cudaError_t e, const char* what) {
    return fail(MXFP4_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

uint64_t wait_limit() { return t_wait_ns ? t_wait_ns : kDefaultWaitNs; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

CtxGetCurrentFn ctx_get_current_fn() {
    static std::atomic<CtxGetCurrentFn> fn{nullptr};
    CtxGetCurrentFn f = fn.load();
    if (!f) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            f = reinterpret_cast<CtxGetCurrentFn>(p);
            fn.store(f);
        }
    }
    return f;
}

// Checks that the current device is a GB300 (compute capability 10.3) and looks up
// the device address of its status word once.  It also makes sure the calling thread
// has a current context: the runtime binds the device's primary context to a thread
// only at that thread's first call that needs one, and the tensor-map encoder (a
// driver call) runs before any launch -- a thread that has made no launch yet (for
// example an autograd worker thread) would otherwise encode without a context.
mxfp4_status check_device(int* dev_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    CtxGetCurrentFn get_ctx = ctx_get_current_fn();
    CUcontext ctx = nullptr;
    if (!get_ctx || get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) {
        e = cudaSetDevice(dev);  // binds (and if needed initialises) the primary context
        if (e != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
    }
    if (dev < 0 || dev >= kMaxDevices) return fail(MXFP4_ERR_UNSUPPORTED_DEVICE, "device index %d", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_device_ok[dev] == 0) {
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        g_device_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
        if (g_device_ok[dev] == 1) {
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_status_word);
            if (e != cudaSuccess) {
                g_device_ok[dev] = 0;
                return cuda_fail(e, "cudaGetSymbolAddress(status word)");
            }
            g_status_ptr[dev] = static_cast<uint32_t*>(p);
        }
    }
    if (g_device_ok[dev] != 1)
        return fail(MXFP4_ERR_UNSUPPORTED_DEVICE, "device %d is not compute capability 10.3 (GB300)", dev);
    *dev_out = dev;
    return MXFP4_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::atomic<EncodeTiledFn> fn{nullptr};
    EncodeTiledFn f = fn.load();
    if (!f) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            f = reinterpret_cast<EncodeTiledFn>(p);
            fn.store(f);
        }
    }
    return f;
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

thread_local int t_encode_result = 0;  // CUresult of this thread's last tensor-map encode
int last_encode_result() { return t_encode_result; }

bool valid_had(int h) { return h == 0 || h == 16 || h == 32; }
bool valid_mode(int m) { return m == 0 || m == 1; }

}  // namespace

mxfp4_status record_error(mxfp4_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_last_error, sizeof t_last_error, fmt, ap);
    va_end(ap);
    return st;
}

uint32_t* device_status_ptr() {
    int dev = 0;
    cudaGetDevice(&dev);
    return (dev >= 0 && dev < kMaxDevices) ? g_status_ptr[dev] : nullptr;
}

// 2D tensor map over packed codes [rows, cols/2] bytes: box = 128 bytes x box_rows,
// 128-byte swizzle (the K-major layout the MMA descriptors expect), zero fill.
bool encode_codes_map(CUtensorMap* map, const void* codes, int64_t rows, int64_t cols, uint32_t box_rows) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)(cols / 2), (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)(cols / 2)};
    const cuuint32_t box[2] = {128, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return (t_encode_result = f(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(codes), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE)) == CUDA_SUCCESS;
}

// 2D tensor map over the GEMM output C [rows, cols] (bf16 or fp32, leading dimension
// ldc elements): box = 64 bytes of a row x 32 rows, 64-byte swizzle.
bool encode_out_map(CUtensorMap* map, void* c, int64_t rows, int64_t cols, int64_t ldc, bool bf16) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    const int64_t esz = bf16 ? 2 : 4;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)(ldc * esz)};
    const cuuint32_t box[2] = {(cuuint32_t)(64 / esz), 32};
    const cuuint32_t estr[2] = {1, 1};
    return (t_encode_result = f(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, c, dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE)) == CUDA_SUCCESS;
}

// 2D tensor map over MMA-order scale factors of a [rows, cols] operand, viewed as
// [512-byte atoms x 4, 128] bytes: box = 128 bytes x 8 rows, i.e. the two atoms (128
// rows x 8 blocks) of one 256-element K stage; no swizzle, zero fill out of bounds.
bool encode_sf_map(CUtensorMap* map, const void* scales, int64_t rows, int64_t cols) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    const cuuint64_t dims[2] = {128, (cuuint64_t)(sf_rows_pad(rows) * sf_kb_pad(cols) / 128)};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {128, 8};
    const cuuint32_t estr[2] = {1, 1};
    return (t_encode_result = f(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(scales), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE)) == CUDA_SUCCESS;
}

}  // namespace mx

using namespace mx;

namespace {

// Validates a caller-provided quantised output descriptor.
mxfp4_status check_out(const mxfp4_tensor* t, const char* name, bool allow_mma) {
    if (!t) return fail(MXFP4_ERR_INVALID_ARG, "%s is NULL", name);
    if (!t->codes || !t->scales) return fail(MXFP4_ERR_INVALID_ARG, "%s: codes/scales NULL", name);
    if (!aligned16(t->codes) || !aligned16(t->scales))
        return fail(MXFP4_ERR_MISALIGNED, "%s: codes/scales not 16-byte aligned", name);
    if (t->sf_layout != MXFP4_SF_PLAIN && t->sf_layout != MXFP4_SF_MMA)
        return fail(MXFP4_ERR_INVALID_ARG, "%s: bad sf_layout %d", name, t->sf_layout);
    if (t->sf_layout == MXFP4_SF_MMA && !allow_mma)
        return fail(MXFP4_ERR_INVALID_ARG, "%s: the 2D layout has PLAIN scales only", name);
    return MXFP4_OK;
}

QuantOut to_out(const mxfp4_tensor* t) {
    QuantOut o{};
    if (t) {
        o.codes = static_cast<uint8_t*>(t->codes);
        o.scales = t->scales;
        o.sf_mma = t->sf_layout == MXFP4_SF_MMA;
        o.kb_pad = sf_kb_pad(t->cols);
    }
    return o;
}

bool needs_sf_padding(const mxfp4_tensor* t) {
    return t && t->sf_layout == MXFP4_SF_MMA && (t->rows % 128 != 0 || (t->cols / 32) % 8 != 0);
}

mxfp4_status check_gemm_operand(const mxfp4_tensor* t, const char* name) {
    if (!t) return fail(MXFP4_ERR_INVALID_ARG, "%s is NULL", name);
    if (!t->codes || !t->scales) return fail(MXFP4_ERR_INVALID_ARG, "%s: codes/scales NULL", name);
    if (!aligned16(t->codes) || !aligned16(t->scales))
        return fail(MXFP4_ERR_MISALIGNED, "%s: codes/scales not 16-byte aligned", name);
    if (t->sf_layout != MXFP4_SF_MMA) return fail(MXFP4_ERR_INVALID_ARG, "%s: GEMM operands need MMA scales", name);
    if (t->layout == MXFP4_LAYOUT_2D)
        return fail(MXFP4_ERR_INVALID_ARG, "%s: 2D-layout tensors cannot feed the GEMM", name);
    if (t->layout != MXFP4_LAYOUT_ROW && t->layout != MXFP4_LAYOUT_COLT)
        return fail(MXFP4_ERR_INVALID_ARG, "%s: bad layout %d", name, t->layout);
    if (!valid_had(t->had) || !valid_mode(t->mode))
        return fail(MXFP4_ERR_INVALID_ARG, "%s: bad had %d / mode %d", name, t->had, t->mode);
    if (t->rows <= 0 || t->cols <= 0) return fail(MXFP4_ERR_UNSUPPORTED_SHAPE, "%s: empty", name);
    if (t->cols % 32 != 0) return fail(MXFP4_ERR_UNSUPPORTED_SHAPE, "%s: cols %% 32 != 0", name);
    if (t->rows > (int64_t)INT32_MAX || t->cols / 2 > (int64_t)INT32_MAX)
        return fail(MXFP4_ERR_UNSUPPORTED_SHAPE, "%s: too large", name);
    return MXFP4_OK;
}

}  // namespace

extern "C" {

size_t mxfp4_codes_bytes(int64_t rows, int64_t cols) {
    if (rows < 0 || cols < 0 || cols % 2) return 0;
    return (size_t)rows * (size_t)(cols / 2);
}

size_t mxfp4_scales_bytes(int64_t rows, int64_t cols, int layout, int sf_layout) {
    if (rows < 0 || cols < 0 || cols % 32) return 0;
    if (layout == MXFP4_LAYOUT_2D) {
        if (sf_layout != MXFP4_SF_PLAIN || rows % 32) return 0;
        return (size_t)(rows / 32) * (size_t)(cols / 32);
    }
    if (layout != MXFP4_LAYOUT_ROW && layout != MXFP4_LAYOUT_COLT) return 0;
    if (sf_layout == MXFP4_SF_PLAIN) return (size_t)rows * (size_t)(cols / 32);
    if (sf_layout == MXFP4_SF_MMA) return (size_t)sf_rows_pad(rows) * (size_t)sf_kb_pad(cols);
    return 0;
}

size_t mxfp4_quantized_bytes(int64_t rows, int64_t cols, int layout, int sf_layout) {
    const size_t s = mxfp4_scales_bytes(rows, cols, layout, sf_layout);
    if (!s && rows * cols) return 0;
    return round_up(mxfp4_codes_bytes(rows, cols), 256) + round_up(s, 256);
}

const char* mxfp4_status_string(mxfp4_status s) {
    switch (s) {
        case MXFP4_OK: return "ok";
        case MXFP4_ERR_INVALID_ARG: return "invalid argument";
        case MXFP4_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case MXFP4_ERR_MISALIGNED: return "misaligned pointer or leading dimension";
        case MXFP4_ERR_WORKSPACE: return "workspace missing or too small";
        case MXFP4_ERR_CUDA: return "CUDA error";
        case MXFP4_ERR_TIMEOUT: return "device-side wait timed out";
        case MXFP4_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs sm_103 / GB300)";
    }
    return "unknown status";
}

const char* mxfp4_last_error(void) { return t_last_error; }

void mxfp4_set_wait_limit_ns(uint64_t ns) { t_wait_ns = ns; }

void mxfp4_test_inject_gemm_fault(int launches) { t_inject_gemm_faults = launches > 0 ? launches : 0; }

mxfp4_status mxfp4_device_status(mxfp4_stream_t stream) {
    int dev;
    mxfp4_status st = check_device(&dev);
    if (st) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    uint32_t word = 0;
    e = cudaMemcpyFromSymbol(&word, g_status_word, sizeof word);
    if (e != cudaSuccess) return cuda_fail(e, "read status word");
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof zero);
    if (e != cudaSuccess) return cuda_fail(e, "clear status word");
    if (word & kStatusTimeout) return fail(MXFP4_ERR_TIMEOUT, "a bounded device wait expired (status 0x%x)", word);
    if (word & kStatusSmemLayout)
        return fail(MXFP4_ERR_CUDA, "a kernel's shared memory was not 1024-byte aligned; it returned early (status 0x%x)",
                    word);
    return ok();
}

}  // extern "C"

namespace {

void fill_desc(mxfp4_tensor* t, int64_t r, int64_t c, int layout, int had, int mode) {
    t->rows = r;
    t->cols = c;
    t->layout = layout;
    t->had = had;
    t->mode = mode;
}

// Every check of a rotate+quantise call, with no CUDA call: nothing is touched or
// launched.  *empty: the problem has no elements (no pointer is used).
mxfp4_status rq_validate(const void* x, int64_t rows, int64_t cols, int64_t ld, int had, int mode, unsigned layouts,
                         const mxfp4_tensor* row_out, const mxfp4_tensor* colT_out, const mxfp4_tensor* twoD_out,
                         bool* empty) {
    *empty = false;
    if (rows < 0 || cols < 0) return fail(MXFP4_ERR_INVALID_ARG, "negative size");
    if (!valid_had(had)) return fail(MXFP4_ERR_INVALID_ARG, "hadamard must be 0, 16 or 32 (got %d)", had);
    if (!valid_mode(mode)) return fail(MXFP4_ERR_INVALID_ARG, "scale mode must be 0 or 1 (got %d)", mode);
    const bool want_row = layouts & MXFP4_LAYOUT_ROW, want_colT = layouts & MXFP4_LAYOUT_COLT,
               want_2d = layouts & MXFP4_LAYOUT_2D;
    if (!layouts || (layouts & ~7u)) return fail(MXFP4_ERR_INVALID_ARG, "bad layout mask 0x%x", layouts);
    if (want_2d && (want_row || want_colT))
        return fail(MXFP4_ERR_INVALID_ARG, "the 2D layout is produced on its own");
    if (cols % 32) return fail(MXFP4_ERR_UNSUPPORTED_SHAPE, "cols (%lld) %% 32 != 0", (long long)cols);
    if ((want_colT || want_2d) && rows % 32)
        return fail(MXFP4_ERR_UNSUPPORTED_SHAPE, "rows (%lld) %% 32 != 0 for the column / 2D layout",
                    (long long)rows);
    if ((want_row && !row_out) || (want_colT && !colT_out) || (want_2d && !twoD_out))
        return fail(MXFP4_ERR_INVALID_ARG, "a requested output descriptor is NULL");
    if (rows == 0 || cols == 0) {
        *empty = true;
        return MXFP4_OK;
    }
    if (!x) return fail(MXFP4_ERR_INVALID_ARG, "x is NULL");
    if (ld < cols || ld % 8)
        return fail(MXFP4_ERR_MISALIGNED, "ld (%lld) must be >= cols and a multiple of 8", (long long)ld);
    if (!aligned16(x)) return fail(MXFP4_ERR_MISALIGNED, "x not 16-byte aligned");
    if ((rows + 63) / 64 > 65535) return fail(MXFP4_ERR_UNSUPPORTED_SHAPE, "too many rows");
    mxfp4_status st;
    if (want_row && (st = check_out(row_out, "row_out", true))) return st;
    if (want_colT && (st = check_out(colT_out, "colT_out", true))) return st;
    if (want_2d && (st = check_out(twoD_out, "twoD_out", false))) return st;
    return MXFP4_OK;
}

// Fills the descriptors of a validated, non-empty rotate+quantise call on a checked
// device, clears MMA scale padding and launches the kernel.
mxfp4_status rq_launch(const void* x, int64_t rows, int64_t cols, int64_t ld, int had, int mode, unsigned layouts,
                       mxfp4_tensor* row_out, mxfp4_tensor* colT_out, mxfp4_tensor* twoD_out, cudaStream_t s) {
    const bool want_row = layouts & MXFP4_LAYOUT_ROW, want_colT = layouts & MXFP4_LAYOUT_COLT,
               want_2d = layouts & MXFP4_LAYOUT_2D;
    if (want_row) fill_desc(row_out, rows, cols, MXFP4_LAYOUT_ROW, had, mode);
    if (want_colT) fill_desc(colT_out, cols, rows, MXFP4_LAYOUT_COLT, had, mode);
    if (want_2d) fill_desc(twoD_out, rows, cols, MXFP4_LAYOUT_2D, had, mode);
    for (mxfp4_tensor* t : {want_row ? row_out : nullptr, want_colT ? colT_out : nullptr}) {
        if (needs_sf_padding(t)) {
            cudaError_t e =
                cudaMemsetAsync(t->scales, 0, mxfp4_scales_bytes(t->rows, t->cols, t->layout, t->sf_layout), s);
            if (e != cudaSuccess) return cuda_fail(e, "clear scale padding");
        }
    }
    QuantParams p{};
    p.x = static_cast<const uint16_t*>(x);
    p.R = rows;
    p.C = cols;
    p.ld = ld;
    p.mode = mode;
    p.row = to_out(want_row ? row_out : nullptr);
    p.colT = to_out(want_colT ? colT_out : nullptr);
    p.twoD = to_out(want_2d ? twoD_out : nullptr);
    cudaError_t e = launch_rotate_quantize(p, had, layouts, s);
    if (e != cudaSuccess) return cuda_fail(e, "rotate_quantize launch");
    return ok();
}

// Both matrices of a validated pair call (same cols, same layouts), on a checked device:
// descriptors filled, MMA scale padding cleared, one launch.
mxfp4_status rq_pair_launch(const void* a, int64_t a_rows, int64_t a_ld, const void* b, int64_t b_rows, int64_t b_ld,
                            int64_t cols, int had, int mode, unsigned layouts, mxfp4_tensor* a_row,
                            mxfp4_tensor* a_colT, mxfp4_tensor* b_row, mxfp4_tensor* b_colT, cudaStream_t s) {
    const bool want_row = layouts & MXFP4_LAYOUT_ROW, want_colT = layouts & MXFP4_LAYOUT_COLT;
    if (want_row) {
        fill_desc(a_row, a_rows, cols, MXFP4_LAYOUT_ROW, had, mode);
        fill_desc(b_row, b_rows, cols, MXFP4_LAYOUT_ROW, had, mode);
    }
    if (want_colT) {
        fill_desc(a_colT, cols, a_rows, MXFP4_LAYOUT_COLT, had, mode);
        fill_desc(b_colT, cols, b_rows, MXFP4_LAYOUT_COLT, had, mode);
    }
    for (mxfp4_tensor* t : {want_row ? a_row : nullptr, want_colT ? a_colT : nullptr, want_row ? b_row : nullptr,
                            want_colT ? b_colT : nullptr}) {
        if (needs_sf_padding(t)) {
            cudaError_t e =
                cudaMemsetAsync(t->scales, 0, mxfp4_scales_bytes(t->rows, t->cols, t->layout, t->sf_layout), s);
            if (e != cudaSuccess) return cuda_fail(e, "clear scale padding");
        }
    }
    QuantParams pa{}, pb{};
    pa.x = static_cast<const uint16_t*>(a);
    pa.R = a_rows;
    pa.C = cols;
    pa.ld = a_ld;
    pa.mode = mode;
    pa.row = to_out(want_row ? a_row : nullptr);
    pa.colT = to_out(want_colT ? a_colT : nullptr);
    pb = pa;
    pb.x = static_cast<const uint16_t*>(b);
    pb.R = b_rows;
    pb.ld = b_ld;
    pb.row = to_out(want_row ? b_row : nullptr);
    pb.colT = to_out(want_colT ? b_colT : nullptr);
    cudaError_t e = launch_rotate_quantize_pair(pa, pb, had, layouts, s);
    if (e != cudaSuccess) return cuda_fail(e, "rotate_quantize_pair launch");
    return ok();
}

}  // namespace

extern "C" {

mxfp4_status mxfp4_rotate_quantize_pair(const void* a, int64_t a_rows, int64_t a_ld, const void* b, int64_t b_rows,
                                        int64_t b_ld, int64_t cols, int had, int mode, unsigned layouts,
                                        mxfp4_tensor* a_row, mxfp4_tensor* a_colT, mxfp4_tensor* b_row,
                                        mxfp4_tensor* b_colT, mxfp4_stream_t stream) {
    if (layouts & MXFP4_LAYOUT_2D) return fail(MXFP4_ERR_INVALID_ARG, "the pair call makes row and column copies only");
    bool ea, eb;
    mxfp4_status st;
    if ((st = rq_validate(a, a_rows, cols, a_ld, had, mode, layouts, a_row, a_colT, nullptr, &ea))) return st;
    if ((st = rq_validate(b, b_rows, cols, b_ld, had, mode, layouts, b_row, b_colT, nullptr, &eb))) return st;
    if ((a_rows + 63) / 64 + (b_rows + 63) / 64 > 65535)
        return fail(MXFP4_ERR_UNSUPPORTED_SHAPE, "too many rows for one launch");
    int dev;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (ea || eb) {  // one side is empty: the other (if any) on its own
        if (ea) {
            if (layouts & MXFP4_LAYOUT_ROW) fill_desc(a_row, a_rows, cols, MXFP4_LAYOUT_ROW, had, mode);
            if (layouts & MXFP4_LAYOUT_COLT) fill_desc(a_colT, cols, a_rows, MXFP4_LAYOUT_COLT, had, mode);
        }
        if (eb) {
            if (layouts & MXFP4_LAYOUT_ROW) fill_desc(b_row, b_rows, cols, MXFP4_LAYOUT_ROW, had, mode);
            if (layouts & MXFP4_LAYOUT_COLT) fill_desc(b_colT, cols, b_rows, MXFP4_LAYOUT_COLT, had, mode);
        }
        if (ea && eb) return ok();
        if ((st = check_device(&dev))) return st;
        return ea ? rq_launch(b, b_rows, cols, b_ld, had, mode, layouts, b_row, b_colT, nullptr, s)
                  : rq_launch(a, a_rows, cols, a_ld, had, mode, layouts, a_row, a_colT, nullptr, s);
    }
    if ((st = check_device(&dev))) return st;
    return rq_pair_launch(a, a_rows, a_ld, b, b_rows, b_ld, cols, had, mode, layouts, a_row, a_colT, b_row, b_colT,
                          s);
}

mxfp4_status mxfp4_rotate_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld, int had, int mode,
                                   unsigned layouts, mxfp4_tensor* row_out, mxfp4_tensor* colT_out,
                                   mxfp4_tensor* twoD_out, mxfp4_stream_t stream) {
    bool empty;
    mxfp4_status st = rq_validate(x, rows, cols, ld, had, mode, layouts, row_out, colT_out, twoD_out, &empty);
    if (st) return st;
    if (empty) {  // nothing to read or write: no pointer is used
        if (layouts & MXFP4_LAYOUT_ROW) fill_desc(row_out, rows, cols, MXFP4_LAYOUT_ROW, had, mode);
        if (layouts & MXFP4_LAYOUT_COLT) fill_desc(colT_out, cols, rows, MXFP4_LAYOUT_COLT, had, mode);
        if (layouts & MXFP4_LAYOUT_2D) fill_desc(twoD_out, rows, cols, MXFP4_LAYOUT_2D, had, mode);
        return ok();
    }
    int dev;
    if ((st = check_device(&dev))) return st;
    return rq_launch(x, rows, cols, ld, had, mode, layouts, row_out, colT_out, twoD_out,
                     reinterpret_cast<cudaStream_t>(stream));
}

namespace {
// Shared checks of the row-layout quantiser fixes; fills the descriptors.  Returns
// MXFP4_OK with *empty set when there is nothing to compute.
mxfp4_status check_fix_args(const void* x, int64_t rows, int64_t cols, int64_t ld, int had, int mode,
                            int64_t col_multiple, std::initializer_list<mxfp4_tensor*> outs, bool* empty) {
    *empty = false;
    if (rows < 0 || cols < 0) return fail(MXFP4_ERR_INVALID_ARG, "negative size");
    if (!valid_had(had)) return fail(MXFP4_ERR_INVALID_ARG, "hadamard must be 0, 16 or 32 (got %d)", had);
    if (!valid_mode(mode)) return fail(MXFP4_ERR_INVALID_ARG, "scale mode must be 0 or 1 (got %d)", mode);
    if (cols % col_multiple)
        return fail(MXFP4_ERR_UNSUPPORTED_SHAPE, "cols (%lld) %% %lld != 0", (long long)cols, (long long)col_multiple);
    for (mxfp4_tensor* t : outs)
        if (!t) return fail(MXFP4_ERR_INVALID_ARG, "an output descriptor is NULL");
    for (mxfp4_tensor* t : outs) {
        t->rows = rows;
        t->cols = cols;
        t->layout = MXFP4_LAYOUT_ROW;
        t->had = had;
        t->mode = mode;
    }
    if (rows == 0 || cols == 0) {
        *empty = true;
        return MXFP4_OK;
    }
    if (!x) return fail(MXFP4_ERR_INVALID_ARG, "x is NULL");
    if (ld < cols || ld % 8)
        return fail(MXFP4_ERR_MISALIGNED, "ld (%lld) must be >= cols and a multiple of 8", (long long)ld);
    if (!aligned16(x)) return fail(MXFP4_ERR_MISALIGNED, "x not 16-byte aligned");
    if ((rows + 63) / 64 > 65535) return fail(MXFP4_ERR_UNSUPPORTED_SHAPE, "too many rows");
    mxfp4_status st;
    for (mxfp4_tensor* t : outs)
        if ((st = check_out(t, "output", true))) return st;
    return MXFP4_OK;
}

mxfp4_status clear_padding(std::initializer_list<mxfp4_tensor*> outs, cudaStream_t s) {
    for (mxfp4_tensor* t : outs)
        if (t && needs_sf_padding(t)) {
            cudaError_t e =
                cudaMemsetAsync(t->scales, 0, mxfp4_scales_bytes(t->rows, t->cols, t->layout, t->sf_layout), s);
            if (e != cudaSuccess) return cuda_fail(e, "clear scale padding");
        }
    return MXFP4_OK;
}
}  // namespace

mxfp4_status mxfp4_rotate_quantize_of(const void* x, int64_t rows, int64_t cols, int64_t ld, int had, int mode,
                                      int alpha_log2, mxfp4_tensor* q1, mxfp4_tensor* q2, mxfp4_stream_t stream) {
    if (alpha_log2 > 0 || alpha_log2 < -8)
        return fail(MXFP4_ERR_INVALID_ARG, "alpha_log2 must be in [-8, 0] (got %d)", alpha_log2);
    bool empty;
    mxfp4_status st = check_fix_args(x, rows, cols, ld, had, mode, 32, {q1, q2}, &empty);
    if (st || empty) return st ? st : ok();
    int dev;
    if ((st = check_device(&dev))) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if ((st = clear_padding({q1, q2}, s))) return st;
    QuantParams p{};
    p.x = static_cast<const uint16_t*>(x);
    p.R = rows;
    p.C = cols;
    p.ld = ld;
    p.mode = mode;
    p.row = to_out(q1);
    cudaError_t e = launch_rotate_quantize_of(p, to_out(q2), had, alpha_log2, s);
    if (e != cudaSuccess) return cuda_fail(e, "rotate_quantize_of launch");
    return ok();
}

mxfp4_status mxfp4_rotate_quantize_mbs(const void* x, int64_t rows, int64_t cols, int64_t ld, int had, int mode,
                                       mxfp4_tensor* q, uint8_t* mbs, mxfp4_stream_t stream) {
    bool empty;
    mxfp4_status st = check_fix_args(x, rows, cols, ld, had, mode, 128, {q}, &empty);
    if (st || empty) return st ? st : ok();
    if (!mbs) return fail(MXFP4_ERR_INVALID_ARG, "mbs is NULL");
    int dev;
    if ((st = check_device(&dev))) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if ((st = clear_padding({q}, s))) return st;
    QuantParams p{};
    p.x = static_cast<const uint16_t*>(x);
    p.R = rows;
    p.C = cols;
    p.ld = ld;
    p.mode = mode;
    p.row = to_out(q);
    cudaError_t e = launch_rotate_quantize_mbs(p, mbs, had, s);
    if (e != cudaSuccess) return cuda_fail(e, "rotate_quantize_mbs launch");
    return ok();
}

mxfp4_status mxfp4_rotate_quantize_ex(const void* x, int64_t rows, int64_t cols, int64_t ld, int had, int mode,
                                      unsigned layouts, const mxfp4_quant_opts* opts, mxfp4_tensor* row_out,
                                      mxfp4_tensor* colT_out, mxfp4_tensor* twoD_out, mxfp4_stream_t stream) {
    const bool any = opts && (opts->col_signs || opts->row_signs || opts->sr_row || opts->sr_colT);
    if (!any) return mxfp4_rotate_quantize(x, rows, cols, ld, had, mode, layouts, row_out, colT_out, twoD_out, stream);
    if (layouts & MXFP4_LAYOUT_2D)
        return fail(MXFP4_ERR_UNSUPPORTED_SHAPE, "random signs / stochastic rounding: row and column layouts only");
    const bool want_row = layouts & MXFP4_LAYOUT_ROW, want_colT = layouts & MXFP4_LAYOUT_COLT;
    const bool sr = (want_row && opts->sr_row) || (want_colT && opts->sr_colT);
    if (sr && ((want_row && !opts->sr_row) || (want_colT && !opts->sr_colT)))
        return fail(MXFP4_ERR_INVALID_ARG, "stochastic rounding needs random integers for every requested layout");
    for (const void* q : {(const void*)opts->col_signs, (const void*)opts->row_signs, (const void*)opts->sr_row,
                          (const void*)opts->sr_colT})
        if (q && !aligned16(q)) return fail(MXFP4_ERR_MISALIGNED, "option arrays must be 16-byte aligned");
    // Validation of shapes, descriptors and x exactly as the plain entry point; an empty
    // problem touches nothing.
    if (rows < 0 || cols < 0) return fail(MXFP4_ERR_INVALID_ARG, "negative size");
    if (!valid_had(had)) return fail(MXFP4_ERR_INVALID_ARG, "hadamard must be 0, 16 or 32 (got %d)", had);
    if (!valid_mode(mode)) return fail(MXFP4_ERR_INVALID_ARG, "scale mode must be 0 or 1 (got %d)", mode);
    if (!layouts || (layouts & ~3u)) return fail(MXFP4_ERR_INVALID_ARG, "bad layout mask 0x%x", layouts);
    if (cols % 32) return fail(MXFP4_ERR_UNSUPPORTED_SHAPE, "cols (%lld) %% 32 != 0", (long long)cols);
    if (want_colT && rows % 32)
        return fail(MXFP4_ERR_UNSUPPORTED_SHAPE, "rows (%lld) %% 32 != 0 for the column layout", (long long)rows);
    if ((want_row && !row_out) || (want_colT && !colT_out))
        return fail(MXFP4_ERR_INVALID_ARG, "a requested output descriptor is NULL");
    auto fill = [&](mxfp4_tensor* t, int64_t r, int64_t c, int layout) {
        t->rows = r;
        t->cols = c;
        t->layout = layout;
        t->had = had;
        t->mode = mode;
    };
    if (want_row) fill(row_out, rows, cols, MXFP4_LAYOUT_ROW);
    if (want_colT) fill(colT_out, cols, rows, MXFP4_LAYOUT_COLT);
    if (rows == 0 || cols == 0) return ok();
    if (!x) return fail(MXFP4_ERR_INVALID_ARG, "x is NULL");
    if (ld < cols || ld % 8)
        return fail(MXFP4_ERR_MISALIGNED, "ld (%lld) must be >= cols and a multiple of 8", (long long)ld);
    if (!aligned16(x)) return fail(MXFP4_ERR_MISALIGNED, "x not 16-byte aligned");
    if ((rows + 63) / 64 > 65535) return fail(MXFP4_ERR_UNSUPPORTED_SHAPE, "too many rows");
    mxfp4_status st;
    if (want_row && (st = check_out(row_out, "row_out", true))) return st;
    if (want_colT && (st = check_out(colT_out, "colT_out", true))) return st;
    int dev;
    if ((st = check_device(&dev))) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if ((st = clear_padding({want_row ? row_out : nullptr, want_colT ? colT_out : nullptr}, s))) return st;
    QuantParams p{};
    p.x = static_cast<const uint16_t*>(x);
    p.R = rows;
    p.C = cols;
    p.ld = ld;
    p.mode = mode;
    p.row = to_out(want_row ? row_out : nullptr);
    p.colT = to_out(want_colT ? colT_out : nullptr);
    RandOpts o{opts->col_signs, opts->row_signs, opts->sr_row, opts->sr_colT};
    cudaError_t e = launch_rotate_quantize_rand(p, o, had, layouts, s);
    if (e != cudaSuccess) return cuda_fail(e, "rotate_quantize_ex launch");
    return ok();
}

}  // extern "C"

namespace {

// Every check of a GEMM call C = A . B^T, with no CUDA call.  Beyond shapes and
// pointers: both operands must come from the same rotation and scale rule (the
// rotations cancel only when both sides of the contraction carry the same H,
// "Pretraining ... Native FP4 Hardware" C.1-C.3), and a transposed copy on the A side
// needs one on the B side too: the linear layer's GEMMs pair (row, row) in Fprop,
// (row, transposed) in Dgrad and (transposed, transposed) in Wgrad.
mxfp4_status gemm_validate(const mxfp4_tensor* A, const mxfp4_tensor* B, const void* C, int64_t ldc, int out_dtype,
                           int accumulate) {
    mxfp4_status st;
    if ((st = check_gemm_operand(A, "A")) || (st = check_gemm_operand(B, "B"))) return st;
    if (A->cols != B->cols)
        return fail(MXFP4_ERR_UNSUPPORTED_SHAPE, "contraction mismatch: A cols %lld, B cols %lld", (long long)A->cols,
                    (long long)B->cols);
    if (A->had != B->had || A->mode != B->mode)
        return fail(MXFP4_ERR_INVALID_ARG,
                    "A (had %d, mode %d) and B (had %d, mode %d) were quantised differently: the rotations cancel "
                    "only under the same Hadamard and scale rule",
                    A->had, A->mode, B->had, B->mode);
    if (A->layout == MXFP4_LAYOUT_COLT && B->layout != MXFP4_LAYOUT_COLT)
        return fail(MXFP4_ERR_INVALID_ARG, "A is a transposed copy but B is not (Wgrad takes two transposed copies)");
    if (!C) return fail(MXFP4_ERR_INVALID_ARG, "C is NULL");
    if (out_dtype != MXFP4_OUT_F32 && out_dtype != MXFP4_OUT_BF16)
        return fail(MXFP4_ERR_INVALID_ARG, "bad out_dtype %d", out_dtype);
    if (accumulate && out_dtype != MXFP4_OUT_F32) return fail(MXFP4_ERR_INVALID_ARG, "accumulate needs fp32 output");
    if (ldc < B->rows || ldc % 8)
        return fail(MXFP4_ERR_MISALIGNED, "ldc (%lld) must be >= N and a multiple of 8", (long long)ldc);
    if (!aligned16(C)) return fail(MXFP4_ERR_MISALIGNED, "C not 16-byte aligned");
    return MXFP4_OK;
}

// Encodes the tensor maps and fills the kernel parameters of a validated GEMM (a
// driver call, no launch).
mxfp4_status gemm_prepare(const mxfp4_tensor* A, const mxfp4_tensor* B, void* C, int64_t ldc, int out_dtype,
                          int accumulate, GemmParams* p) {
    if (reinterpret_cast<uintptr_t>(p) & 63u)
        return fail(MXFP4_ERR_CUDA, "internal: GEMM parameter block not 64-byte aligned");
    *p = GemmParams{};
    const char* which = !encode_codes_map(&p->map_a, A->codes, A->rows, A->cols, 128) ? "A codes"
                        : !encode_codes_map(&p->map_b, B->codes, B->rows, B->cols, 128) ? "B codes"
                        : !encode_out_map(&p->map_c, C, A->rows, B->rows, ldc, out_dtype == MXFP4_OUT_BF16) ? "C"
                        : !encode_sf_map(&p->map_sfa, A->scales, A->rows, A->cols) ? "A scales"
                        : !encode_sf_map(&p->map_sfb, B->scales, B->rows, B->cols) ? "B scales"
                                                                                      : nullptr;
    if (which) return fail(MXFP4_ERR_CUDA, "cuTensorMapEncodeTiled failed for %s (CUresult %d)", which, last_encode_result());
    p->sfa = A->scales;
    p->sfb = B->scales;
    p->M = A->rows;
    p->N = B->rows;
    p->K = A->cols;
    p->kb_pad = sf_kb_pad(A->cols);
    p->C = C;
    p->ldc = ldc;
    p->out_bf16 = out_dtype == MXFP4_OUT_BF16;
    p->accumulate = accumulate ? 1 : 0;
    return MXFP4_OK;
}

// The GEMM's parameter block, placed by hand on a 64-byte boundary: the driver's
// tensor-map encoder requires it, and a host stack (for example an autograd worker
// thread's) need not honour the alignas(64) of a local CUtensorMap.
struct GemmParamsBox {
    unsigned char raw[sizeof(GemmParams) + 64];
    GemmParams* get() { return reinterpret_cast<GemmParams*>((reinterpret_cast<uintptr_t>(raw) + 63) & ~uintptr_t(63)); }
};

mxfp4_status gemm_launch(GemmParams& p, cudaStream_t s) {
    p.status = device_status_ptr();
    p.wait_ns = wait_limit();
    if (t_inject_gemm_faults > 0) {
        --t_inject_gemm_faults;
        p.test_drop_first_stage = 1;
    }
    cudaError_t e = launch_gemm(p, s);
    if (e != cudaSuccess) return cuda_fail(e, "gemm launch");
    return ok();
}

}  // namespace

extern "C" {

mxfp4_status mxfp4_rotate_quantize_philox(const void* x, int64_t rows, int64_t cols, int64_t ld, int had, int mode,
                                          unsigned layouts, const mxfp4_philox_opts* opts, mxfp4_tensor* row_out,
                                          mxfp4_tensor* colT_out, mxfp4_stream_t stream) {
    if (!opts) return fail(MXFP4_ERR_INVALID_ARG, "opts is NULL");
    if (opts->reserved != 0) return fail(MXFP4_ERR_INVALID_ARG, "opts.reserved must be 0");
    if ((layouts & MXFP4_LAYOUT_2D) || !layouts || (layouts & ~3u))
        return fail(MXFP4_ERR_INVALID_ARG, "random signs / stochastic rounding: row and column layouts only");
    bool empty;
    mxfp4_status st = rq_validate(x, rows, cols, ld, had, mode, layouts, row_out, colT_out, nullptr, &empty);
    if (st) return st;
    const bool want_row = layouts & MXFP4_LAYOUT_ROW, want_colT = layouts & MXFP4_LAYOUT_COLT;
    if (want_row) fill_desc(row_out, rows, cols, MXFP4_LAYOUT_ROW, had, mode);
    if (want_colT) fill_desc(colT_out, cols, rows, MXFP4_LAYOUT_COLT, had, mode);
    if (empty) return ok();
    int dev;
    if ((st = check_device(&dev))) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if ((st = clear_padding({want_row ? row_out : nullptr, want_colT ? colT_out : nullptr}, s))) return st;
    QuantParams p{};
    p.x = static_cast<const uint16_t*>(x);
    p.R = rows;
    p.C = cols;
    p.ld = ld;
    p.mode = mode;
    p.row = to_out(want_row ? row_out : nullptr);
    p.colT = to_out(want_colT ? colT_out : nullptr);
    RandOpts o{};
    o.gen = 1;
    o.col_sign_on = opts->col_signs != 0;
    o.row_sign_on = opts->row_signs != 0;
    o.sr_on = opts->stochastic_rounding != 0;
    o.col_sign_seed = opts->col_sign_seed;
    o.row_sign_seed = opts->row_sign_seed;
    o.sr_seed = opts->sr_seed;
    cudaError_t e = launch_rotate_quantize_rand(p, o, had, layouts, s);
    if (e != cudaSuccess) return cuda_fail(e, "rotate_quantize_philox launch");
    return ok();
}

mxfp4_status mxfp4_gemm(const mxfp4_tensor* A, const mxfp4_tensor* B, void* C, int64_t ldc, int out_dtype,
                        int accumulate, void* ws, size_t ws_bytes, mxfp4_stream_t stream) {
    (void)ws;
    (void)ws_bytes;
    mxfp4_status st;
    if ((st = gemm_validate(A, B, C, ldc, out_dtype, accumulate))) return st;
    int dev;
    if ((st = check_device(&dev))) return st;
    GemmParamsBox box;
    GemmParams* p = box.get();
    if ((st = gemm_prepare(A, B, C, ldc, out_dtype, accumulate, p))) return st;
    return gemm_launch(*p, reinterpret_cast<cudaStream_t>(stream));
}

mxfp4_status mxfp4_gemm_group(const mxfp4_gemm_desc* descs, int count, mxfp4_stream_t stream) {
    if (!descs || count < 1 || count > kMaxGemmGroup)
        return fail(MXFP4_ERR_INVALID_ARG, "count must be 1 to %d with descs non-NULL (got %d)", kMaxGemmGroup, count);
    mxfp4_status st;
    for (int i = 0; i < count; ++i) {
        const mxfp4_gemm_desc& d = descs[i];
        if ((st = gemm_validate(d.A, d.B, d.C, d.ldc, d.out_dtype, d.accumulate))) {
            char msg[512];
            snprintf(msg, sizeof msg, "%s", t_last_error);
            return fail(st, "problem %d: %s", i, msg);
        }
    }
    // No two outputs may share a byte: the problems run concurrently.
    for (int i = 0; i < count; ++i)
        for (int j = i + 1; j < count; ++j) {
            auto span = [](const mxfp4_gemm_desc& d, uintptr_t* lo, uintptr_t* hi) {
                const uintptr_t esz = d.out_dtype == MXFP4_OUT_BF16 ? 2 : 4;
                *lo = reinterpret_cast<uintptr_t>(d.C);
                *hi = *lo + ((uintptr_t)(d.A->rows - 1) * (uintptr_t)d.ldc + (uintptr_t)d.B->rows) * esz;
            };
            uintptr_t a0, a1, b0, b1;
            span(descs[i], &a0, &a1);
            span(descs[j], &b0, &b1);
            if (a0 < b1 && b0 < a1) return fail(MXFP4_ERR_INVALID_ARG, "outputs of problems %d and %d overlap", i, j);
        }
    int dev;
    if ((st = check_device(&dev))) return st;
    struct Box {
        unsigned char raw[kMaxGemmGroup * sizeof(GemmParams) + 64];
    } box;
    GemmParams* ps = reinterpret_cast<GemmParams*>((reinterpret_cast<uintptr_t>(box.raw) + 63) & ~uintptr_t(63));
    for (int i = 0; i < count; ++i) {
        const mxfp4_gemm_desc& d = descs[i];
        if ((st = gemm_prepare(d.A, d.B, d.C, d.ldc, d.out_dtype, d.accumulate, ps + i))) return st;
        ps[i].status = device_status_ptr();
        ps[i].wait_ns = wait_limit();
    }
    if (t_inject_gemm_faults > 0) {
        --t_inject_gemm_faults;
        ps[0].test_drop_first_stage = 1;
    }
    cudaError_t e = launch_gemm_group(ps, count, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "gemm group launch");
    return ok();
}

mxfp4_status mxfp4_gemm_mbs(const mxfp4_tensor* A, const uint8_t* mbs_a, const mxfp4_tensor* B, const uint8_t* mbs_b,
                            void* C, int64_t ldc, int out_dtype, int accumulate, mxfp4_stream_t stream) {
    mxfp4_status st;
    if ((st = gemm_validate(A, B, C, ldc, out_dtype, accumulate))) return st;
    if (A->cols % 128) return fail(MXFP4_ERR_UNSUPPORTED_SHAPE, "K (%lld) %% 128 != 0 (macro blocks)", (long long)A->cols);
    if (A->cols / 128 > kMbsMaxMacroBlocks)
        return fail(MXFP4_ERR_UNSUPPORTED_SHAPE, "K (%lld) above %d", (long long)A->cols, 128 * kMbsMaxMacroBlocks);
    int dev;
    if ((st = check_device(&dev))) return st;
    struct Box {
        unsigned char raw[sizeof(MbsParams) + 64];
    } box;
    MbsParams* mp = reinterpret_cast<MbsParams*>((reinterpret_cast<uintptr_t>(box.raw) + 63) & ~uintptr_t(63));
    if ((st = gemm_prepare(A, B, C, ldc, out_dtype, accumulate, &mp->g))) return st;
    mp->g.status = device_status_ptr();
    mp->g.wait_ns = wait_limit();
    if (t_inject_gemm_faults > 0) {
        --t_inject_gemm_faults;
        mp->g.test_drop_first_stage = 1;
    }
    mp->mbs_a = mbs_a;
    mp->mbs_b = mbs_b;
    cudaError_t e = launch_gemm_mbs(*mp, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "gemm_mbs launch");
    return ok();
}

mxfp4_status mxfp4_error_decomposition(const void* x, int64_t rows, int64_t cols, int64_t ld, int had, int mode,
                                       double* out, mxfp4_stream_t stream) {
    if (rows < 0 || cols < 0) return fail(MXFP4_ERR_INVALID_ARG, "negative size");
    if (!valid_had(had)) return fail(MXFP4_ERR_INVALID_ARG, "hadamard must be 0, 16 or 32 (got %d)", had);
    if (!valid_mode(mode)) return fail(MXFP4_ERR_INVALID_ARG, "scale mode must be 0 or 1 (got %d)", mode);
    if (cols % 32) return fail(MXFP4_ERR_UNSUPPORTED_SHAPE, "cols (%lld) %% 32 != 0", (long long)cols);
    if (!out) return fail(MXFP4_ERR_INVALID_ARG, "out is NULL");
    if (reinterpret_cast<uintptr_t>(out) & 7u) return fail(MXFP4_ERR_MISALIGNED, "out not 8-byte aligned");
    if (rows && cols) {
        if (!x) return fail(MXFP4_ERR_INVALID_ARG, "x is NULL");
        if (ld < cols || ld % 8)
            return fail(MXFP4_ERR_MISALIGNED, "ld (%lld) must be >= cols and a multiple of 8", (long long)ld);
        if (!aligned16(x)) return fail(MXFP4_ERR_MISALIGNED, "x not 16-byte aligned");
    }
    int dev;
    mxfp4_status st;
    if ((st = check_device(&dev))) return st;
    cudaError_t e = launch_error_decomposition(static_cast<const uint16_t*>(x), rows, cols, ld, had, mode, out,
                                               reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "error decomposition launch");
    return ok();
}

mxfp4_status mxfp4_mma_peak_probe(int kind, int64_t iters, double* tflops) {
    if (kind < 0 || kind > 4) return fail(MXFP4_ERR_INVALID_ARG, "kind must be 0 to 4");
    if (iters <= 0 || !tflops) return fail(MXFP4_ERR_INVALID_ARG, "iters must be positive and tflops non-NULL");
    int dev, ctas = 0;
    mxfp4_status st;
    if ((st = check_device(&dev))) return st;
    float ms = 0.0f;
    cudaError_t e = run_mma_peak_probe(kind, iters, &ms, &ctas, device_status_ptr(), wait_limit());
    if (e != cudaSuccess) return cuda_fail(e, "mma peak probe");
    const double k = kind == 2 ? 16.0 : 64.0;  // K per instruction
    *tflops = (double)ctas * (double)iters * 2.0 * 128.0 * 256.0 * k / (ms * 1e-3) / 1e12;
    return ok();
}

size_t mxfp4_workspace_bytes(int op, int64_t M, int64_t N, int64_t K, const mxfp4_config* cfg) {
    (void)cfg;
    switch (op) {
        case MXFP4_OP_FPROP:
            return mxfp4_quantized_bytes(M, K, MXFP4_LAYOUT_ROW, MXFP4_SF_MMA) +
                   mxfp4_quantized_bytes(N, K, MXFP4_LAYOUT_ROW, MXFP4_SF_MMA);
        case MXFP4_OP_DGRAD:
            return mxfp4_quantized_bytes(M, N, MXFP4_LAYOUT_ROW, MXFP4_SF_MMA);
        case MXFP4_OP_WGRAD:
            return 0;
        case MXFP4_OP_BACKWARD:
            return mxfp4_quantized_bytes(M, N, MXFP4_LAYOUT_ROW, MXFP4_SF_MMA) +
                   mxfp4_quantized_bytes(N, M, MXFP4_LAYOUT_COLT, MXFP4_SF_MMA);
    }
    return 0;
}

}  // extern "C"

namespace {

// Carves one quantised tensor (codes, then scales at a 256-byte boundary) from ws.
mxfp4_tensor carve(uint8_t*& ws, int64_t rows, int64_t cols) {
    mxfp4_tensor t{};
    t.codes = ws;
    t.scales = ws + round_up(mxfp4_codes_bytes(rows, cols), 256);
    t.sf_layout = MXFP4_SF_MMA;
    ws += mxfp4_quantized_bytes(rows, cols, MXFP4_LAYOUT_ROW, MXFP4_SF_MMA);
    return t;
}

mxfp4_status check_cfg(const mxfp4_config* cfg) {
    if (!cfg) return fail(MXFP4_ERR_INVALID_ARG, "cfg is NULL");
    if (!valid_had(cfg->had)) return fail(MXFP4_ERR_INVALID_ARG, "cfg.had must be 0, 16 or 32");
    if (!valid_mode(cfg->mode)) return fail(MXFP4_ERR_INVALID_ARG, "cfg.mode must be 0 or 1");
    if (cfg->out_dtype != MXFP4_OUT_F32 && cfg->out_dtype != MXFP4_OUT_BF16)
        return fail(MXFP4_ERR_INVALID_ARG, "cfg.out_dtype invalid");
    return MXFP4_OK;
}

mxfp4_status check_ws(void* ws, size_t ws_bytes, size_t need) {
    if (need && (!ws || ws_bytes < need))
        return fail(MXFP4_ERR_WORKSPACE, "workspace needs %zu bytes (got %zu at %p)", need, ws_bytes, ws);
    if (need && (reinterpret_cast<uintptr_t>(ws) & 255u))
        return fail(MXFP4_ERR_MISALIGNED, "workspace must be 256-byte aligned");
    return MXFP4_OK;
}

}  // namespace

extern "C" {

mxfp4_status mxfp4_linear_fprop(const void* x, const void* w, int64_t M, int64_t N, int64_t K,
                                const mxfp4_config* cfg, void* y, mxfp4_tensor* save_xT, mxfp4_tensor* save_wT,
                                void* ws, size_t ws_bytes, mxfp4_stream_t stream) {
    // Every argument is checked (and the GEMM's tensor maps encoded) before the first
    // launch, so a rejected call leaves the workspace, the saved copies and y untouched.
    mxfp4_status st;
    if ((st = check_cfg(cfg))) return st;
    if (!x || !w || !y) return fail(MXFP4_ERR_INVALID_ARG, "x, w and y must be non-NULL");
    if (M <= 0 || N <= 0 || K <= 0) return fail(MXFP4_ERR_UNSUPPORTED_SHAPE, "M, N, K must be positive");
    if (K % 32) return fail(MXFP4_ERR_UNSUPPORTED_SHAPE, "K %% 32 != 0");
    if (save_xT && save_xT->sf_layout != MXFP4_SF_MMA) return fail(MXFP4_ERR_INVALID_ARG, "save_xT needs MMA scales");
    if (save_wT && save_wT->sf_layout != MXFP4_SF_MMA) return fail(MXFP4_ERR_INVALID_ARG, "save_wT needs MMA scales");
    if ((st = check_ws(ws, ws_bytes, mxfp4_workspace_bytes(MXFP4_OP_FPROP, M, N, K, cfg)))) return st;
    uint8_t* cur = static_cast<uint8_t*>(ws);
    mxfp4_tensor xq = carve(cur, M, K), wq = carve(cur, N, K);
    const unsigned lx = MXFP4_LAYOUT_ROW | (save_xT ? MXFP4_LAYOUT_COLT : 0);
    const unsigned lw = MXFP4_LAYOUT_ROW | (save_wT ? MXFP4_LAYOUT_COLT : 0);
    bool empty;
    if ((st = rq_validate(x, M, K, K, cfg->had, cfg->mode, lx, &xq, save_xT, nullptr, &empty))) return st;
    if ((st = rq_validate(w, N, K, K, cfg->had, cfg->mode, lw, &wq, save_wT, nullptr, &empty))) return st;
    // the GEMM operands as the two passes will describe them
    fill_desc(&xq, M, K, MXFP4_LAYOUT_ROW, cfg->had, cfg->mode);
    fill_desc(&wq, N, K, MXFP4_LAYOUT_ROW, cfg->had, cfg->mode);
    if ((st = gemm_validate(&xq, &wq, y, N, cfg->out_dtype, cfg->accumulate))) return st;
    int dev;
    if ((st = check_device(&dev))) return st;
    GemmParamsBox box;
    GemmParams* gp = box.get();
    if ((st = gemm_prepare(&xq, &wq, y, N, cfg->out_dtype, cfg->accumulate, gp))) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (lx == lw && (M + 63) / 64 + (N + 63) / 64 <= 65535) {
        // X and W in one launch: they share the contraction K
        if ((st = rq_pair_launch(x, M, K, w, N, K, K, cfg->had, cfg->mode, lx, &xq, save_xT, &wq, save_wT, s)))
            return st;
    } else {
        if ((st = rq_launch(x, M, K, K, cfg->had, cfg->mode, lx, &xq, save_xT, nullptr, s))) return st;
        if ((st = rq_launch(w, N, K, K, cfg->had, cfg->mode, lw, &wq, save_wT, nullptr, s))) return st;
    }
    return gemm_launch(*gp, s);
}

mxfp4_status mxfp4_linear_dgrad(const void* dy, const mxfp4_tensor* wT, int64_t M, int64_t N, int64_t K,
                                const mxfp4_config* cfg, void* dx, mxfp4_tensor* save_dyT, void* ws,
                                size_t ws_bytes, mxfp4_stream_t stream) {
    mxfp4_status st;
    if ((st = check_cfg(cfg))) return st;
    if (!dy || !wT || !dx) return fail(MXFP4_ERR_INVALID_ARG, "dy, wT and dx must be non-NULL");
    if (M <= 0 || N <= 0 || K <= 0) return fail(MXFP4_ERR_UNSUPPORTED_SHAPE, "M, N, K must be positive");
    if (N % 32) return fail(MXFP4_ERR_UNSUPPORTED_SHAPE, "N %% 32 != 0");
    if (wT->rows != K || wT->cols != N)
        return fail(MXFP4_ERR_UNSUPPORTED_SHAPE, "wT must be [K, N] = [%lld, %lld]", (long long)K, (long long)N);
    if (wT->layout != MXFP4_LAYOUT_COLT)
        return fail(MXFP4_ERR_INVALID_ARG, "wT must be the transposed copy of W (quantised along N)");
    if (wT->had != cfg->had || wT->mode != cfg->mode)
        return fail(MXFP4_ERR_INVALID_ARG, "wT was quantised with had %d / mode %d, the layer uses had %d / mode %d",
                    wT->had, wT->mode, cfg->had, cfg->mode);
    if (save_dyT && save_dyT->sf_layout != MXFP4_SF_MMA)
        return fail(MXFP4_ERR_INVALID_ARG, "save_dyT needs MMA scales");
    if ((st = check_ws(ws, ws_bytes, mxfp4_workspace_bytes(MXFP4_OP_DGRAD, M, N, K, cfg)))) return st;
    uint8_t* cur = static_cast<uint8_t*>(ws);
    mxfp4_tensor dyq = carve(cur, M, N);
    const unsigned ld_ = MXFP4_LAYOUT_ROW | (save_dyT ? MXFP4_LAYOUT_COLT : 0);
    bool empty;
    if ((st = rq_validate(dy, M, N, N, cfg->had, cfg->mode, ld_, &dyq, save_dyT, nullptr, &empty))) return st;
    fill_desc(&dyq, M, N, MXFP4_LAYOUT_ROW, cfg->had, cfg->mode);
    if ((st = gemm_validate(&dyq, wT, dx, K, cfg->out_dtype, cfg->accumulate))) return st;
    int dev;
    if ((st = check_device(&dev))) return st;
    GemmParamsBox box;
    GemmParams* gp = box.get();
    if ((st = gemm_prepare(&dyq, wT, dx, K, cfg->out_dtype, cfg->accumulate, gp))) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if ((st = rq_launch(dy, M, N, N, cfg->had, cfg->mode, ld_, &dyq, save_dyT, nullptr, s))) return st;
    return gemm_launch(*gp, s);
}

mxfp4_status mxfp4_linear_backward(const void* dy, const mxfp4_tensor* wT, const mxfp4_tensor* xT, int64_t M,
                                   int64_t N, int64_t K, const mxfp4_config* cfg, void* dx, void* dw, void* ws,
                                   size_t ws_bytes, mxfp4_stream_t stream) {
    mxfp4_status st;
    if ((st = check_cfg(cfg))) return st;
    if (!dy || !wT || !xT || !dx || !dw) return fail(MXFP4_ERR_INVALID_ARG, "dy, wT, xT, dx and dw must be non-NULL");
    if (M <= 0 || N <= 0 || K <= 0) return fail(MXFP4_ERR_UNSUPPORTED_SHAPE, "M, N, K must be positive");
    if (N % 32 || M % 32) return fail(MXFP4_ERR_UNSUPPORTED_SHAPE, "N and M must be multiples of 32");
    if (wT->rows != K || wT->cols != N)
        return fail(MXFP4_ERR_UNSUPPORTED_SHAPE, "wT must be [K, N] = [%lld, %lld]", (long long)K, (long long)N);
    if (xT->rows != K || xT->cols != M)
        return fail(MXFP4_ERR_UNSUPPORTED_SHAPE, "xT must be [K, M] = [%lld, %lld]", (long long)K, (long long)M);
    if (wT->layout != MXFP4_LAYOUT_COLT || xT->layout != MXFP4_LAYOUT_COLT)
        return fail(MXFP4_ERR_INVALID_ARG, "wT and xT must be transposed copies");
    if (wT->had != cfg->had || wT->mode != cfg->mode || xT->had != cfg->had || xT->mode != cfg->mode)
        return fail(MXFP4_ERR_INVALID_ARG, "wT and xT must be quantised with the layer's had %d / mode %d", cfg->had,
                    cfg->mode);
    if ((st = check_ws(ws, ws_bytes, mxfp4_workspace_bytes(MXFP4_OP_BACKWARD, M, N, K, cfg)))) return st;
    uint8_t* cur = static_cast<uint8_t*>(ws);
    mxfp4_tensor dyq = carve(cur, M, N);
    mxfp4_tensor dyT{};
    dyT.codes = cur;
    dyT.scales = cur + round_up(mxfp4_codes_bytes(N, M), 256);
    dyT.sf_layout = MXFP4_SF_MMA;
    const unsigned lay = MXFP4_LAYOUT_ROW | MXFP4_LAYOUT_COLT;
    bool empty;
    if ((st = rq_validate(dy, M, N, N, cfg->had, cfg->mode, lay, &dyq, &dyT, nullptr, &empty))) return st;
    fill_desc(&dyq, M, N, MXFP4_LAYOUT_ROW, cfg->had, cfg->mode);
    fill_desc(&dyT, N, M, MXFP4_LAYOUT_COLT, cfg->had, cfg->mode);
    // dX = dY W in cfg->out_dtype (no accumulation); dW = dY^T X in fp32, added to dw
    // when cfg->accumulate (gradient accumulation over micro-batches).
    if ((st = gemm_validate(&dyq, wT, dx, K, cfg->out_dtype, 0))) return st;
    if ((st = gemm_validate(&dyT, xT, dw, K, MXFP4_OUT_F32, cfg->accumulate))) return st;
    int dev;
    if ((st = check_device(&dev))) return st;
    struct Box {
        unsigned char raw[2 * sizeof(GemmParams) + 64];
    } box;
    GemmParams* gp = reinterpret_cast<GemmParams*>((reinterpret_cast<uintptr_t>(box.raw) + 63) & ~uintptr_t(63));
    if ((st = gemm_prepare(&dyq, wT, dx, K, cfg->out_dtype, 0, gp))) return st;
    if ((st = gemm_prepare(&dyT, xT, dw, K, MXFP4_OUT_F32, cfg->accumulate, gp + 1))) return st;
    for (int i = 0; i < 2; ++i) {
        gp[i].status = device_status_ptr();
        gp[i].wait_ns = wait_limit();
    }
    if (t_inject_gemm_faults > 0) {
        --t_inject_gemm_faults;
        gp[0].test_drop_first_stage = 1;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if ((st = rq_launch(dy, M, N, N, cfg->had, cfg->mode, lay, &dyq, &dyT, nullptr, s))) return st;
    cudaError_t e = launch_gemm_group(gp, 2, s);
    if (e != cudaSuccess) return cuda_fail(e, "backward gemm launch");
    return ok();
}

mxfp4_status mxfp4_linear_wgrad(const mxfp4_tensor* dyT, const mxfp4_tensor* xT, const mxfp4_config* cfg,
                                void* dw, void* ws, size_t ws_bytes, mxfp4_stream_t stream) {
    mxfp4_status st;
    if ((st = check_cfg(cfg))) return st;
    if (!dyT || !xT || !dw) return fail(MXFP4_ERR_INVALID_ARG, "dyT, xT and dw must be non-NULL");
    if (dyT->cols != xT->cols) return fail(MXFP4_ERR_UNSUPPORTED_SHAPE, "dyT and xT must share the token dim");
    if (dyT->layout != MXFP4_LAYOUT_COLT || xT->layout != MXFP4_LAYOUT_COLT)
        return fail(MXFP4_ERR_INVALID_ARG, "dyT and xT must be transposed copies (quantised along the tokens)");
    if (dyT->had != cfg->had || dyT->mode != cfg->mode || xT->had != cfg->had || xT->mode != cfg->mode)
        return fail(MXFP4_ERR_INVALID_ARG,
                    "dyT (had %d, mode %d) and xT (had %d, mode %d) must both match the layer's had %d / mode %d",
                    dyT->had, dyT->mode, xT->had, xT->mode, cfg->had, cfg->mode);
    return mxfp4_gemm(dyT, xT, dw, xT->rows, cfg->out_dtype, cfg->accumulate, ws, ws_bytes, stream);
}

}  // extern "C"
