// gemm_mbs.cu -- block-scaled MXFP4 GEMM over macro-block-scaled (MBS) operands on the
// sm_103a tcgen05 tensor cores.
//
// "Decomposing MXFP4 quantization error for LLM reinforcement learning", MBS: one 8-bit
// mantissa correction m per macro block of 128 consecutive elements along the quantised
// dimension, x_hat = Q((1 + m) x) / (1 + m).  The quantised dimension is the GEMM's
// contraction, so the postscale changes every 128 elements of K and cannot follow the
// whole tensor-core sum as one epilogue factor:
//   C[m][n] = sum over macro blocks kb of  f_A[m][kb] f_B[n][kb] P_kb[m][n],
//   P_kb = the block-scaled MXFP4 product over the 128 K of macro block kb,
//   f = 256 / (256 + byte) (1 for an operand given without MBS bytes).
// Each P_kb is formed on the tensor cores in one of three TMEM buffers; the epilogue warps
// read it, scale it and add it into an fp32 register accumulator while the tensor cores
// fill the next ones.  At the tile's end the accumulator is stored like the plain
// GEMM's (TMA, bf16 or fp32, optional add-reduce).
//
// Structure (persistent, one CTA of 320 threads per SM walks 128 x 128 tiles):
//   warp 0     TMA producer: A and B codes (128 rows x 256 elements per stage, 128-byte
//              swizzle) and their 1 KB scale atoms, into a 4-stage ring;
//   warp 1     TMEM allocation; one thread copies each stage's scales to TMEM and issues
//              two MMAs (K = 64 each) per macro block into the macro block's buffer;
//   warps 2-9  epilogue: warp w reads TMEM lanes 32 (w % 4) .. +31 (its rows) and half
//              of the 128 columns.  Factors come from a 256-entry table in shared memory
//              (one per MBS byte); the tile's column factors are looked up once per tile
//              (K <= 16384), and each row's byte for the next macro block is loaded one
//              macro block ahead.
// Bounds: the rescale costs one packed multiply and one packed FMA per two outputs per
// macro block on the CUDA cores, and a 128 x 128 tile moves twice the operand bytes per
// FLOP of the CTA-pair kernel's 256 x 256 tile (three 128-column partial buffers leave no
// room for wider tiles in TMEM).  All waits are bounded.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace mx {
namespace {

constexpr int MB_STAGES = 4;
constexpr int MB_BUFS = 3;  // TMEM partial buffers of 128 columns
constexpr int MB_EPI_WARPS = 8;
constexpr int MB_THREADS = 64 + 32 * MB_EPI_WARPS;
constexpr int MB_STG_BYTES = 32 * 64;  // one warp's 32-row x 64-byte staging box

struct MbsCfg {
    static constexpr int A_STAGE = 128 * 128;  // 128 rows x 128 bytes (256 E2M1 elements)
    static constexpr int B_STAGE = 128 * 128;
    static constexpr int SF_STAGE = 1024;      // 128 rows x 8 scale bytes
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + MB_STAGES * A_STAGE;
    static constexpr int OFF_SFA = OFF_B + MB_STAGES * B_STAGE;
    static constexpr int OFF_SFB = OFF_SFA + MB_STAGES * SF_STAGE;
    static constexpr int OFF_FB = OFF_SFB + MB_STAGES * SF_STAGE;  // column factors [kb][128] fp32
    static constexpr int OFF_LUT = OFF_FB + kMbsMaxMacroBlocks * 128 * 4;  // 256 / (256 + byte), 256 floats
    static constexpr int OFF_BAR = OFF_LUT + 256 * 4;
    // full[S], empty[S], p_full[B], p_empty[B], mma_done
    static constexpr int OFF_TMEM = OFF_BAR + (2 * MB_STAGES + 2 * MB_BUFS + 1) * 8;
    static constexpr int OFF_STG = (OFF_TMEM + 16 + 1023) / 1024 * 1024;
    static constexpr int SMEM = OFF_STG + MB_EPI_WARPS * MB_STG_BYTES + 1024;  // + base alignment slack
    static constexpr uint32_t TX = A_STAGE + B_STAGE + 2 * SF_STAGE;
    static constexpr int SF_COLS = 16;  // TMEM columns of scales per stage: 8 for A, 8 for B
    static constexpr int TMEM_COLS = 512;
    static_assert(MB_BUFS * 128 + MB_STAGES * SF_COLS <= TMEM_COLS, "TMEM budget");
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
    static_assert(OFF_B % 1024 == 0 && OFF_BAR % 8 == 0 && OFF_FB % 16 == 0 && OFF_STG % 1024 == 0, "alignment");
};

__device__ __forceinline__ void epi_bar_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(32 * MB_EPI_WARPS) : "memory");
}

// 256 / (256 + byte): the MBS postscale 1 / (1 + byte/256), correctly rounded.
__device__ __forceinline__ float mbs_factor(uint32_t byte) { return __fdiv_rn(256.0f, 256.0f + (float)byte); }

// The warp's 32 rows x 32 consecutive fp32 values of C (from `v`, one row per lane) to
// global memory through the warp's staging box, as bf16 (one 32 x 64-byte box) or fp32
// (two boxes); the box is reused once the previous store has read it.
__device__ __forceinline__ void mbs_store_box(const GemmParams& p, uint8_t* stg, int lane, int64_t row_base,
                                              int64_t col0, const uint32_t* w) {
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint4*>(stg + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) =
            make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
        if (row_base < p.M && col0 < p.N) {
            if (p.accumulate)
                tma_reduce_add_2d(&p.map_c, stg, (int32_t)col0, (int32_t)row_base);
            else
                tma_store_2d(&p.map_c, stg, (int32_t)col0, (int32_t)row_base);
        }
        bulk_commit();
    }
}

__device__ __forceinline__ void mbs_store_chunk(const GemmParams& p, uint8_t* stg, int lane, int64_t row_base,
                                                int64_t col0, const float* acc) {
    if (p.out_bf16) {
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * j], acc[2 * j + 1]);
            w[j] = *reinterpret_cast<const uint32_t*>(&h);
        }
        mbs_store_box(p, stg, lane, row_base, col0, w);
    } else {
        uint32_t w[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) w[j] = __float_as_uint(acc[j]);
        mbs_store_box(p, stg, lane, row_base, col0, w);
        mbs_store_box(p, stg, lane, row_base, col0 + 16, w + 16);
    }
}

__global__ void __launch_bounds__(MB_THREADS, 1) mxf4_gemm_mbs_kernel(const __grid_constant__ MbsParams mp) {
    using Cfg = MbsCfg;
    const GemmParams& p = mp.g;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem + Cfg::OFF_A;
    uint8_t* sB = smem + Cfg::OFF_B;
    uint8_t* sSFA = smem + Cfg::OFF_SFA;
    uint8_t* sSFB = smem + Cfg::OFF_SFB;
    float* fB = reinterpret_cast<float*>(smem + Cfg::OFF_FB);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
    uint64_t* empty = full + MB_STAGES;
    float* lut = reinterpret_cast<float*>(smem + Cfg::OFF_LUT);
    uint64_t* p_full = empty + MB_STAGES;   // [B] MMA -> epilogue: a macro block's partial is ready
    uint64_t* p_empty = p_full + MB_BUFS;   // [B] epilogue -> MMA: the partial has been read
    uint64_t* mma_done = p_empty + MB_BUFS;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_TMEM);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nkb = (int)(p.K / 128);        // macro blocks
    const int num_k = (nkb + 1) / 2;         // 256-element stages (the last may hold one macro block)
    const int64_t num_n = (p.N + 127) / 128;
    const int64_t num_tiles = ((p.M + 127) / 128) * num_n;
    const int64_t atoms_per_row_block = p.kb_pad / 4;

    if (threadIdx.x == 0) {
        for (int s = 0; s < MB_STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < MB_BUFS; ++b) {
            mbar_init(&p_full[b], 1);
            mbar_init(&p_empty[b], MB_EPI_WARPS);
        }
        mbar_init(mma_done, 1);
        fence_mbar_init();
        prefetch_tmap(&p.map_a);
        prefetch_tmap(&p.map_b);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, Cfg::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
#if MXF_PDL_GEMM
    grid_dependency_wait();
    allow_dependent_launch();
#endif

    if (warp == 0) {
        // ---------------- TMA producer
        if (elect_one()) {
            uint32_t armed[MB_STAGES];
#pragma unroll
            for (int s = 0; s < MB_STAGES; ++s) armed[s] = 0;
            uint32_t it = 0;
            bool ok = true;
            for (int64_t tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                const int64_t m0 = (tile / num_n) * 128, n0 = (tile % num_n) * 128;
                for (int kt = 0; kt < num_k; ++kt, ++it) {
                    const int s = (int)(it % MB_STAGES);
                    const uint32_t ph = (it / MB_STAGES) & 1u;
                    if (it >= MB_STAGES && !wait_bounded(&empty[s], ph ^ 1u, p.wait_ns, p.status)) {
                        ok = false;
                        break;
                    }
                    if (it == 0 && p.test_drop_first_stage) continue;  // fault injection: never arrives
                    mbar_arrive_expect_tx(&full[s], Cfg::TX);
                    tma_load_2d(sA + s * Cfg::A_STAGE, &p.map_a, &full[s], kt * 128, (int32_t)m0);
                    tma_load_2d(sB + s * Cfg::B_STAGE, &p.map_b, &full[s], kt * 128, (int32_t)n0);
                    bulk_load(sSFA + s * Cfg::SF_STAGE, p.sfa + ((m0 / 128) * atoms_per_row_block + 2 * kt) * 512,
                              Cfg::SF_STAGE, &full[s]);
                    bulk_load(sSFB + s * Cfg::SF_STAGE, p.sfb + ((n0 / 128) * atoms_per_row_block + 2 * kt) * 512,
                              Cfg::SF_STAGE, &full[s]);
                    armed[s] = it / MB_STAGES + 1u;
                }
            }
#pragma unroll
            for (int s = 0; s < MB_STAGES; ++s)
                if (armed[s]) wait_bounded(&full[s], (armed[s] - 1u) & 1u, p.wait_ns, p.status);
        }
    } else if (warp == 1) {
        // ---------------- tensor-core issuer: two MMAs per macro block into buffer j % 3
        if (elect_one()) {
            constexpr uint32_t idesc = idesc_mxf4(128, 128);
            uint32_t it = 0, j = 0;
            bool ok = true;
            for (int64_t tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                for (int kt = 0; ok && kt < num_k; ++kt, ++it) {
                    const int s = (int)(it % MB_STAGES);
                    const uint32_t ph = (it / MB_STAGES) & 1u;
                    if (!wait_bounded(&full[s], ph, p.wait_ns, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sfa_t = tmem_base + MB_BUFS * 128 + s * Cfg::SF_COLS;
                    const uint32_t sfb_t = sfa_t + 8;
#pragma unroll
                    for (int a = 0; a < 2; ++a) {
                        tc_cp_32x128b_warpx4(sfa_t + a * 4,
                                             smem_desc(smem_u32(sSFA + s * Cfg::SF_STAGE + a * 512), 0, 128, kSwizzleNone));
                        tc_cp_32x128b_warpx4(sfb_t + a * 4,
                                             smem_desc(smem_u32(sSFB + s * Cfg::SF_STAGE + a * 512), 0, 128, kSwizzleNone));
                    }
                    const uint32_t a_base = smem_u32(sA + s * Cfg::A_STAGE);
                    const uint32_t b_base = smem_u32(sB + s * Cfg::B_STAGE);
                    for (int half = 0; half < 2 && 2 * kt + half < nkb; ++half, ++j) {
                        const uint32_t b = j % MB_BUFS;
                        if (j >= MB_BUFS) {
                            if (!wait_bounded(&p_empty[b], (j / MB_BUFS - 1u) & 1u, p.wait_ns, p.status)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                        }
#pragma unroll
                        for (int k = 0; k < 2; ++k) {
                            const int kk = 2 * half + k;  // 64-element step within the stage
                            const uint32_t sf_id = (uint32_t)(kk & 1) * 2u;
                            tc_mma_mxf4(tmem_base + b * 128, smem_desc(a_base + kk * 32, 16, 1024, kSwizzle128B),
                                        smem_desc(b_base + kk * 32, 16, 1024, kSwizzle128B),
                                        idesc_with_sf_ids(idesc, sf_id, sf_id), sfa_t + (kk >> 1) * 4,
                                        sfb_t + (kk >> 1) * 4, k);
                        }
                        tc_commit(&p_full[b]);
                    }
                    tc_commit(&empty[s]);
                }
            }
            tc_commit(mma_done);
            wait_bounded(mma_done, 0, p.wait_ns, p.status);
        }
    } else {
        // ---------------- epilogue: rows 32 q .. +31 of the tile, columns 64 h .. +63
        const int q = warp & 3;
        const int h = (warp - 2) >> 2;
        const int et = threadIdx.x - 64;  // 0 .. 255
        uint8_t* stg = smem + Cfg::OFF_STG + (warp - 2) * MB_STG_BYTES;
        uint32_t j = 0;
        bool ok = true;
        lut[et] = mbs_factor((uint32_t)et);  // 256 epilogue threads, one entry each
        for (int64_t tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            const int64_t m0 = (tile / num_n) * 128, n0 = (tile % num_n) * 128;
            // the tile's column factors, once every warp is done with the previous tile's
            // (the first barrier also publishes the table)
            epi_bar_sync();
            for (int idx = et; idx < nkb * 128; idx += 32 * MB_EPI_WARPS) {
                const int kb = idx >> 7, c = idx & 127;
                const int64_t n = n0 + c;
                fB[idx] = (mp.mbs_b && n < p.N) ? lut[mp.mbs_b[n * nkb + kb]] : 1.0f;
            }
            epi_bar_sync();
            const int64_t row = m0 + q * 32 + lane;
            const uint8_t* mrow = (mp.mbs_a && row < p.M) ? mp.mbs_a + row * nkb : nullptr;
            uint32_t next_byte = mrow ? mrow[0] : 0u;  // this row's byte, one macro block ahead
            float2 acc[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] = make_float2(0.0f, 0.0f);
            for (int kb = 0; kb < nkb; ++kb, ++j) {
                // After an expired wait the loops keep their shape (no more waits, loads or
                // stores), so every epilogue warp still reaches the tile's two barriers.
                if (!ok) continue;
                const float fa = mrow ? lut[next_byte] : 1.0f;
                if (mrow && kb + 1 < nkb) next_byte = mrow[kb + 1];
                const uint32_t b = j % MB_BUFS;
                if (!wait_bounded(&p_full[b], (j / MB_BUFS) & 1u, p.wait_ns, p.status)) {
                    ok = false;
                    continue;
                }
                tc_fence_after();
                uint32_t v0[32], v1[32];
                const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + b * 128 + (uint32_t)(h * 64);
                tmem_ld_32x32b_x32(taddr, v0);
                tmem_ld_32x32b_x32(taddr + 32, v1);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_empty[b]);
                const float4* f4 = reinterpret_cast<const float4*>(fB + kb * 128 + h * 64);
                const float2 fa2 = make_float2(fa, fa);
#pragma unroll
                for (int c4 = 0; c4 < 16; ++c4) {
                    const float4 f = f4[c4];
                    const uint32_t* src = c4 < 8 ? v0 + 4 * c4 : v1 + 4 * (c4 - 8);
                    const float2 g0 = f2_mul(fa2, make_float2(f.x, f.y));
                    const float2 g1 = f2_mul(fa2, make_float2(f.z, f.w));
                    acc[2 * c4] = f2_fma(make_float2(__uint_as_float(src[0]), __uint_as_float(src[1])), g0,
                                         acc[2 * c4]);
                    acc[2 * c4 + 1] = f2_fma(make_float2(__uint_as_float(src[2]), __uint_as_float(src[3])), g1,
                                             acc[2 * c4 + 1]);
                }
            }
            if (!ok) continue;
            const int64_t row_base = m0 + q * 32;
#pragma unroll
            for (int c = 0; c < 2; ++c)
                mbs_store_chunk(p, stg, lane, row_base, n0 + h * 64 + c * 32, reinterpret_cast<const float*>(acc) + 32 * c);
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

}  // namespace

cudaError_t launch_gemm_mbs(const MbsParams& mp, cudaStream_t s) {
    using Cfg = MbsCfg;
    static DeviceSlots sm_slots;
    int sm_count = 0;
    cudaError_t e = per_device_setting(sm_slots, &sm_count, [&](int dev, int* n) {
        cudaError_t r = cudaFuncSetAttribute(mxf4_gemm_mbs_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
        return r != cudaSuccess ? r : cudaDeviceGetAttribute(n, cudaDevAttrMultiProcessorCount, dev);
    });
    if (e != cudaSuccess) return e;
    const int64_t tiles = ((mp.g.M + 127) / 128) * ((mp.g.N + 127) / 128);
    const unsigned grid = (unsigned)(tiles < sm_count ? tiles : sm_count);
    return launch_overlapped(mxf4_gemm_mbs_kernel, dim3(grid), dim3(MB_THREADS), Cfg::SMEM, s, 1, MXF_PDL_GEMM != 0, mp);
}

}  // namespace mx
