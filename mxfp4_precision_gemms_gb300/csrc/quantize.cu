// quantize.cu -- fused rotate + MXFP4 quantise kernel (sm_103a).
//
// "Pretraining Large Language Models with MXFP4 on Native FP4 Hardware":
//   A.1 (x_B ~ 2^E * Q_FP4(x_B / 2^E), 32-element blocks), A.2 (deterministic tiled
//   Hadamard before quantisation), D (1x32 row, 32x1 column-transposed, 32x32 2D).
// "Decomposing MXFP4 quantization error ...": E8M0 scales, E2M1 grid, ceiling scale.
//
// One CTA of 128 threads (4 warps) owns a 64 x 128 tile of the bf16 input and reads it
// from HBM once.
//  - Row work: each thread owns two 32-element row segments (rows r and r + 32) in
//    registers and processes them in lockstep with packed f32x2 instructions:
//    rotation butterfly, block amax, E8M0 byte, 2 x 32 codes -> two 16-byte stores.
//  - Column work (transposed copy): the load also leaves the raw bf16 tile in shared
//    memory, swizzled so that the row-wise writes and the column-wise reads are
//    bank-conflict free.  Each thread then owns two adjacent columns of one 32-row block
//    (one 32-bit shared load per row gives both columns' values); a warp holds both row
//    blocks of its 16 column pairs, so each output row's two 16-byte halves meet in one
//    warp and leave, after one shuffle exchange, as one 32-byte store.
//  - 2D work: row segments as above, the per-segment amax is combined over the 32
//    rows of the block through shared memory.
// Per element the kernel moves 2 B in and 0.53 B (single) or 1.06 B (row + column)
// out; the dual pass is bound by instruction issue as much as by HBM.
#include "internal.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace mx {
namespace {

constexpr int TR = 64;        // tile rows
constexpr int TC = 128;       // tile cols
constexpr int QTHREADS = 2 * TR;
// Launch bound: CTAs per SM the register allocation must allow.  Six (80 registers, no
// spills) beat four (122 registers) by 7-9% on the dual pass.  The dual pass takes seven
// (72 registers; under H16 a 12-byte spill): measured 2% faster than six on 8192 x 14336
// and on the Llama-3.1-8B step's quantisations, outputs byte-identical.  Eight spill
// hundreds of bytes.  Single-copy passes keep six.
constexpr int QBLOCKS_PER_SM = 6;
constexpr int QBLOCKS_DUAL = 7;
constexpr int TILE_BYTES = TR * TC * 2;  // the raw bf16 tile

// One launch over up to two matrices with the same number of columns (a GEMM's two
// operands share their contraction): row tiles 0 .. split-1 belong to g.p[0], the rest
// to g.p[1].  A single matrix has split = its row-tile count.
struct QuantGroup {
    QuantParams p[2];
    int32_t split;
};

// PAIR: two matrices (the parameters are then read through the CTA's matrix index);
// one matrix keeps every parameter at a constant offset.  Measured: a single-matrix
// launch that indexed its parameters like a pair ran 4-6% slower.
template <int HAD, bool ROW, bool COLT, bool TWOD, bool PAIR>
__global__ void __launch_bounds__(QTHREADS, TWOD ? 4 : (ROW && COLT) ? QBLOCKS_DUAL : QBLOCKS_PER_SM) rq_kernel(const __grid_constant__ QuantGroup g) {
    extern __shared__ __align__(16) uint8_t q_smem[];
    uint32_t* tile_w = reinterpret_cast<uint32_t*>(q_smem);
    float* seg_amax = reinterpret_cast<float*>(q_smem + (COLT ? TILE_BYTES : 0));

    const int t = threadIdx.x;
    const int which = PAIR ? (int)blockIdx.y >= g.split : 0;
    // A copy selected field by field (two constant-offset loads and a select each) rather
    // than an indexed reference: measured 0.3-0.8% faster on the step's quantisations.
    const QuantParams p = which ? g.p[1] : g.p[0];
    const int64_t row0 = (int64_t)((int)blockIdx.y - (which ? g.split : 0)) * TR;
    const int64_t col0 = (int64_t)blockIdx.x * TC;
#if MXF_PDL_QUANT
    grid_dependency_wait();  // x may come from the previous kernel in the stream
#endif
#if MXF_QUANT_TRIGGER
    allow_dependent_launch();
#endif

    // ---- two row segments owned by this thread: rows pr and pr + TR/2, columns 32*s ..
    const int s = t & 3, pr = t >> 2;
    const int rx = pr, ry = pr + TR / 2;
    const int64_t gc = col0 + 32 * s;
    const int64_t grx = row0 + rx, gry = row0 + ry;
    const bool vx = grx < p.R && gc < p.C, vy = gry < p.R && gc < p.C;
    float2 v[32];
    {
        uint4 raw_x[4], raw_y[4];
        // 32-byte loads (whole sectors per instruction) when the rows allow them.
        // Measured on 8192 x {4096, 14336}: row + transposed 5-20% faster, transposed only
        // 2-14%, 2D unchanged; the row-only pass was 13% slower with them and keeps
        // 16-byte loads.
        load_row_pair(p, grx, gry, gc, vx, vy, (COLT || TWOD) && rows_32B_aligned(p), raw_x, raw_y);
        if constexpr (COLT) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                *reinterpret_cast<uint4*>(&tile_w[tile_chunk(rx, 4 * s + j)]) = raw_x[j];
                *reinterpret_cast<uint4*>(&tile_w[tile_chunk(ry, 4 * s + j)]) = raw_y[j];
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t a[4] = {raw_x[j].x, raw_x[j].y, raw_x[j].z, raw_x[j].w};
            const uint32_t b[4] = {raw_y[j].x, raw_y[j].y, raw_y[j].z, raw_y[j].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if constexpr (HAD > 1 && (ROW || TWOD)) {
                    // the row copy's stride-1 butterfly straight from each bf16 pair
                    // (measured +5-7% on the 8192 x 4096 dual pass, +1% row-only; the
                    // transposed copy keeps the plain unpack, where it measured slower)
                    bfly_lo(a[i], __uint_as_float(a[i] & 0xFFFF0000u), v[8 * j + 2 * i].x, v[8 * j + 2 * i + 1].x);
                    bfly_lo(b[i], __uint_as_float(b[i] & 0xFFFF0000u), v[8 * j + 2 * i].y, v[8 * j + 2 * i + 1].y);
                    continue;
                }
                v[8 * j + 2 * i] = make_float2(__uint_as_float(a[i] << 16), __uint_as_float(b[i] << 16));
                v[8 * j + 2 * i + 1] =
                    make_float2(__uint_as_float(a[i] & 0xFFFF0000u), __uint_as_float(b[i] & 0xFFFF0000u));
            }
        }
    }
    if constexpr (ROW || TWOD) {
        rotate32x2_from2<HAD>(v);
        float ax, ay;
        amax32x2<HAD>(v, ax, ay);
        if constexpr (TWOD) {
            seg_amax[rx * 4 + s] = ax;
            seg_amax[ry * 4 + s] = ay;
            __syncthreads();
            float tx = 0.0f, ty = 0.0f;
            const int bx = rx & ~31, by = ry & ~31;
#pragma unroll 8
            for (int i = 0; i < 32; ++i) {
                tx = fmaxf(tx, seg_amax[(bx + i) * 4 + s]);
                ty = fmaxf(ty, seg_amax[(by + i) * 4 + s]);
            }
            const uint32_t bytex = scale_byte(tx, p.mode), bytey = scale_byte(ty, p.mode);
            uint4 qx, qy;
            quant32x2<HAD>(v, bytex, bytey, qx, qy);
            if (vx) {
                *reinterpret_cast<uint4*>(p.twoD.codes + grx * (p.C / 2) + gc / 2) = qx;
                if ((rx & 31) == 0) p.twoD.scales[(grx / 32) * (p.C / 32) + gc / 32] = (uint8_t)bytex;
            }
            if (vy) {
                *reinterpret_cast<uint4*>(p.twoD.codes + gry * (p.C / 2) + gc / 2) = qy;
                if ((ry & 31) == 0) p.twoD.scales[(gry / 32) * (p.C / 32) + gc / 32] = (uint8_t)bytey;
            }
        } else {
            const uint32_t bytex = scale_byte(ax, p.mode), bytey = scale_byte(ay, p.mode);
            uint4 qx, qy;
            quant32x2<HAD>(v, bytex, bytey, qx, qy);
            if (vx) *reinterpret_cast<uint4*>(p.row.codes + grx * (p.C / 2) + gc / 2) = qx;
            if (vy) *reinterpret_cast<uint4*>(p.row.codes + gry * (p.C / 2) + gc / 2) = qy;
            store_row_scales(p.row, p, col0, s, grx, gry, vx, vy, bytex, bytey);
        }
    }

    if constexpr (COLT) {
        __syncthreads();
        // Two adjacent columns (2 cp, 2 cp + 1) x one 32-row block per thread.  A warp
        // holds both row blocks of 16 column pairs (lanes l and l ^ 16 share cp), so the
        // two 16-byte halves of each output row meet in one warp: one shuffle exchange,
        // then every lane writes one output row's 32 bytes and two scale bytes.
        const int lane = t & 31;
        const int rb = lane >> 4, cp = 16 * (t >> 5) + (lane & 15);
        const int q = cp >> 2, wi = cp & 3;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const uint32_t w = tile_w[tile_chunk(32 * rb + i, q) + wi];
            v[i] = make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
        }
        rotate32x2<HAD>(v);
        float ax, ay;
        amax32x2<HAD>(v, ax, ay);
        const uint32_t bytex = scale_byte(ax, p.mode), bytey = scale_byte(ay, p.mode);
        uint4 qx, qy;
        quant32x2<HAD>(v, bytex, bytey, qx, qy);
        store_colT_pair(p.colT, p, row0, col0, cp, rb, qx, qy, bytex, bytey);
    }
}

template <int HAD, bool ROW, bool COLT, bool TWOD, bool PAIR>
cudaError_t launch_one(const QuantParams& p, const QuantParams* p2, cudaStream_t s) {
    constexpr int smem = (COLT ? TILE_BYTES : 0) + (TWOD ? TR * 4 * 4 : 0);
    auto kern = rq_kernel<HAD, ROW, COLT, TWOD, PAIR>;
    if constexpr (smem > 48 * 1024) {
        static DeviceSlots opted_in;
        int unused = 0;
        const cudaError_t e = per_device_setting(opted_in, &unused, [&](int, int*) {
            return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        });
        if (e != cudaSuccess) return e;
    }
    QuantGroup g{};
    g.p[0] = p;
    g.p[1] = p2 ? *p2 : p;
    g.split = (int32_t)((p.R + TR - 1) / TR);
    const int64_t tiles_y = g.split + (p2 ? (p2->R + TR - 1) / TR : 0);
    const dim3 grid((unsigned)((p.C + TC - 1) / TC), (unsigned)tiles_y);
    return launch_overlapped(kern, grid, dim3(QTHREADS), smem, s, 1, MXF_PDL_QUANT != 0, g);
}

template <int HAD>
cudaError_t launch_had(const QuantParams& p, const QuantParams* p2, unsigned layouts, cudaStream_t s) {
    if (p2) {
        switch (layouts) {
            case MXFP4_LAYOUT_ROW:
                return launch_one<HAD, true, false, false, true>(p, p2, s);
            case MXFP4_LAYOUT_COLT:
                return launch_one<HAD, false, true, false, true>(p, p2, s);
            case MXFP4_LAYOUT_ROW | MXFP4_LAYOUT_COLT:
                return launch_one<HAD, true, true, false, true>(p, p2, s);
            default:
                return cudaErrorInvalidValue;
        }
    }
    switch (layouts) {
        case MXFP4_LAYOUT_ROW:
            return launch_one<HAD, true, false, false, false>(p, nullptr, s);
        case MXFP4_LAYOUT_COLT:
            return launch_one<HAD, false, true, false, false>(p, nullptr, s);
        case MXFP4_LAYOUT_ROW | MXFP4_LAYOUT_COLT:
            return launch_one<HAD, true, true, false, false>(p, nullptr, s);
        case MXFP4_LAYOUT_2D:
            return launch_one<HAD, false, false, true, false>(p, nullptr, s);
        default:
            return cudaErrorInvalidValue;
    }
}

cudaError_t launch_any(const QuantParams& p, const QuantParams* p2, int had, unsigned layouts, cudaStream_t s) {
    switch (had) {
        case 0:
            return launch_had<1>(p, p2, layouts, s);
        case 16:
            return launch_had<16>(p, p2, layouts, s);
        case 32:
            return launch_had<32>(p, p2, layouts, s);
        default:
            return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_rotate_quantize(const QuantParams& p, int had, unsigned layouts, cudaStream_t s) {
    return launch_any(p, nullptr, had, layouts, s);
}

cudaError_t launch_rotate_quantize_pair(const QuantParams& a, const QuantParams& b, int had, unsigned layouts,
                                        cudaStream_t s) {
    if (a.C != b.C || (layouts & MXFP4_LAYOUT_2D)) return cudaErrorInvalidValue;
    return launch_any(a, &b, had, layouts, s);
}

}  // namespace mx
