// internal.h -- declarations shared by the library's translation units (not part
// of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/mxfp4.h"

namespace mx {

// Scale-factor MMA tile order: 128 rows x 4 blocks per 512-byte atom.
__host__ __device__ inline int64_t sf_kb_pad(int64_t cols) { return ((cols / 32 + 7) / 8) * 8; }
__host__ __device__ inline int64_t sf_rows_pad(int64_t rows) { return ((rows + 127) / 128) * 128; }
__host__ __device__ inline int64_t sf_mma_offset(int64_t r, int64_t k, int64_t kb_pad) {
    return ((r >> 7) * (kb_pad >> 2) + (k >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (k & 3);
}

struct QuantOut {
    uint8_t* codes;   // packed nibbles
    uint8_t* scales;  // E8M0 bytes
    int32_t sf_mma;   // 1: MMA tile order
    int64_t kb_pad;   // padded blocks per row (MMA order)
};

struct QuantParams {
    const uint16_t* x;  // bf16 [R, C]
    int64_t R, C, ld;
    int32_t mode;
    QuantOut row, colT, twoD;
};


// Launches the fused rotate+quantise kernel for the requested layouts.
cudaError_t launch_rotate_quantize(const QuantParams& p, int had, unsigned layouts, cudaStream_t s);
// The same for two matrices with the same number of columns (C) in one launch (row and
// transposed layouts; both get the same layouts, rotation and scale rule).
cudaError_t launch_rotate_quantize_pair(const QuantParams& a, const QuantParams& b, int had, unsigned layouts,
                                        cudaStream_t s);
// Quantiser fixes (row layout): OF writes Q(v) to p.row and Q(v - dq(Q(v))) to q2;
// MBS writes Q((1 + k/256) v) to p.row and the bytes k to mbs [R, C/128].
cudaError_t launch_rotate_quantize_of(const QuantParams& p, const QuantOut& q2, int had, int alpha_log2,
                                      cudaStream_t s);
cudaError_t launch_rotate_quantize_mbs(const QuantParams& p, uint8_t* mbs, int had, cudaStream_t s);

// Randomised baselines (row / transposed layouts): sign bitmasks and 16-bit random
// integers supplied by the caller (NULL: not used).
struct RandOpts {
    const uint8_t* col_signs;  // over C, for the row copy
    const uint8_t* row_signs;  // over R, for the transposed copy
    const uint16_t* sr_row;    // [R, C]
    const uint16_t* sr_colT;   // [C, R]
    // Generated instead (gen = 1): Philox4x32-10 sign vectors and stochastic-rounding
    // integers, keyed by these seeds (the arrays above are then unused).
    int32_t gen;
    int32_t col_sign_on, row_sign_on, sr_on;
    uint64_t col_sign_seed, row_sign_seed, sr_seed;
};
cudaError_t launch_rotate_quantize_rand(const QuantParams& p, const RandOpts& o, int had, unsigned layouts,
                                        cudaStream_t s);

struct GemmParams {
    CUtensorMap map_a;   // codes of A [M, K/2] bytes, box 128 rows x 128 B, 128B swizzle
    CUtensorMap map_b;   // codes of B [N, K/2] bytes
    CUtensorMap map_c;   // output C [M, N]: box 64 bytes x 32 rows, 64-byte swizzle
    CUtensorMap map_sfa;  // MMA-order scales of A as [atoms * 4, 128] bytes, box 128 B x 8 rows
    CUtensorMap map_sfb;  // same for B
    const uint8_t* sfa;  // MMA-order scales of A
    const uint8_t* sfb;  // MMA-order scales of B
    int64_t M, N, K, kb_pad;
    void* C;
    int64_t ldc;
    int32_t out_bf16;
    int32_t accumulate;
    uint32_t* status;
    uint64_t wait_ns;
    int32_t test_drop_first_stage;  // fault injection (tests only): stage 0 is never loaded
};

cudaError_t launch_gemm(const GemmParams& p, cudaStream_t s);

// Up to kMaxGemmGroup GEMMs in one persistent launch: one static tile schedule over
// the problems' 256 x 256 tiles (problem after problem, tile_start[i] = the first global
// tile of problem i, tile_start[count] = all tiles).
constexpr int kMaxGemmGroup = 8;
struct GemmGroup {
    GemmParams prob[kMaxGemmGroup];
    int64_t tile_start[kMaxGemmGroup + 1];
    int32_t count;
    uint32_t* status;
    uint64_t wait_ns;
    int32_t test_drop_first_stage;
};
cudaError_t launch_gemm_group(const GemmParams* probs, int n, cudaStream_t s);

// GEMM over macro-block-scaled operands: the plain GEMM's parameters plus the MBS bytes
// of A [M, K/128] and B [N, K/128] (NULL: that operand has no macro-block factor).
constexpr int kMbsMaxMacroBlocks = 128;  // K <= 16384
struct MbsParams {
    GemmParams g;
    const uint8_t* mbs_a;
    const uint8_t* mbs_b;
};
cudaError_t launch_gemm_mbs(const MbsParams& mp, cudaStream_t s);

cudaError_t run_mma_peak_probe(int kind, int64_t iters, float* ms, int* ctas, uint32_t* status, uint64_t wait_ns);

cudaError_t launch_error_decomposition(const uint16_t* x, int64_t R, int64_t C, int64_t ld, int had, int mode,
                                       double* out, cudaStream_t s);

// A launch setting computed once per device (a kernel's shared-memory opt-in, its grid
// limit).  Thread-safe: concurrent first calls may both run compute(dev, &value); the
// value is the same for both and is published with release / acquire ordering.  Values
// must be >= 0; a slot holds value + 1, so 0 means "not computed yet".
constexpr int kMaxCachedDevices = 64;
using DeviceSlots = std::atomic<int>[kMaxCachedDevices];
template <class F>
cudaError_t per_device_setting(DeviceSlots& slots, int* value, F&& compute) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxCachedDevices) return cudaErrorInvalidDevice;
    int v = slots[dev].load(std::memory_order_acquire);
    if (v == 0) {
        int r = 0;
        e = compute(dev, &r);
        if (e != cudaSuccess) return e;
        if (r < 0) return cudaErrorInvalidValue;
        v = r + 1;
        slots[dev].store(v, std::memory_order_release);
    }
    *value = v - 1;
    return cudaSuccess;
}

// Programmatic dependent launch (compile-time knobs).  MXF_PDL_GEMM: GEMM kernels are
// launched with programmatic stream serialization, so a GEMM's set-up (TMEM allocation,
// barriers, cluster sync) overlaps the previous kernel's drain; they wait
// (griddepcontrol.wait) before touching global memory.  MXF_PDL_QUANT: the same for the
// rotate+quantise kernel; MXF_QUANT_TRIGGER: that kernel lets a dependent launch start
// early.  Measured on the Llama-3.1-8B linear step (12 GEMMs + 12 dual quantisations):
// none 1.575 ms, GEMMs only 1.546, GEMMs + quantiser trigger 1.548, everything 1.652 --
// a wait in each of the quantiser's many short CTAs costs more than the overlap gives.
#ifndef MXF_PDL_GEMM
#define MXF_PDL_GEMM 1
#endif
#ifndef MXF_PDL_QUANT
#define MXF_PDL_QUANT 0
#endif
#ifndef MXF_QUANT_TRIGGER
#define MXF_QUANT_TRIGGER 0
#endif

// Launches kern<<<grid, block, smem, s>>>(args...) as a cluster of cluster_x CTAs (1:
// no cluster attribute), allowing programmatic dependent launch when `overlap` is set.
template <class Kern, class... Args>
cudaError_t launch_overlapped(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t s, unsigned cluster_x,
                              bool overlap, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (overlap) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Host helpers implemented in mxfp4_api.cu.
uint32_t* device_status_ptr();  // for the current device
// Records the thread-local message returned by mxfp4_last_error() and returns st.
mxfp4_status record_error(mxfp4_status st, const char* fmt, ...);
bool encode_codes_map(CUtensorMap* map, const void* codes, int64_t rows, int64_t cols, uint32_t box_rows);
bool encode_out_map(CUtensorMap* map, void* c, int64_t rows, int64_t cols, int64_t ldc, bool bf16);
bool encode_sf_map(CUtensorMap* map, const void* scales, int64_t rows, int64_t cols);

}  // namespace mx
