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
// spills) beat four (122 registers) by 7-9% on the dual pass; seven and eight spill.
constexpr int QBLOCKS_PER_SM = 6;
constexpr int TILE_BYTES = TR * TC * 2;  // the raw bf16 tile

// Staged tile: 32-bit word index of 16-byte chunk q (0..15) of row r.  The XOR on the
// chunk index (by q bits 2-3, row bit 0 and row bit 5) keeps the row-wise 16-byte writes
// (8 rows x 4 segments per warp) and the column-wise 32-bit reads (rows i and 32 + i,
// 16 column pairs each, per warp) bank-conflict free.
__device__ __forceinline__ int bf16_chunk(int r, int q) {
    return r * (TC / 2) + ((q ^ ((q >> 2) & 3) ^ (((r ^ (r >> 5)) & 1) << 2)) << 2);
}

// One 32-byte global store (the address must be 32-byte aligned).
__device__ __forceinline__ void st_global_32B(void* dst, uint4 a, uint4 b) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(a.x), "r"(a.y),
                 "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
                 : "memory");
}

// One 32-byte streaming global load (the address must be 32-byte aligned).
__device__ __forceinline__ void ld_global_cs_32B(const void* src, uint4& a, uint4& b) {
    asm volatile("ld.global.cs.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
                 : "l"(src));
}

template <int HAD, bool ROW, bool COLT, bool TWOD>
__global__ void __launch_bounds__(QTHREADS, TWOD ? 4 : QBLOCKS_PER_SM) rq_kernel(const QuantParams p) {
    extern __shared__ __align__(16) uint8_t q_smem[];
    uint32_t* tile_w = reinterpret_cast<uint32_t*>(q_smem);
    float* seg_amax = reinterpret_cast<float*>(q_smem + (COLT ? TILE_BYTES : 0));

    const int t = threadIdx.x;
    const int64_t row0 = (int64_t)blockIdx.y * TR;
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
#pragma unroll
        for (int j = 0; j < 4; ++j) raw_x[j] = raw_y[j] = make_uint4(0, 0, 0, 0);
        // 32-byte loads when every row segment starts on a 32-byte boundary, so that each
        // load instruction uses whole 32-byte sectors.  Measured on 8192 x {4096, 14336}:
        // row + transposed 5-20% faster, transposed only 2-14%, 2D unchanged; the
        // row-only pass was 13% slower with them and keeps 16-byte loads.
        const bool a32 = (COLT || TWOD) && ((reinterpret_cast<uintptr_t>(p.x) | (uintptr_t)(p.ld * 2)) & 31u) == 0;
        if (vx) {
            const uint4* src = reinterpret_cast<const uint4*>(p.x + grx * p.ld + gc);
            if (a32) {
                ld_global_cs_32B(src, raw_x[0], raw_x[1]);
                ld_global_cs_32B(src + 2, raw_x[2], raw_x[3]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) raw_x[j] = __ldcs(src + j);
            }
        }
        if (vy) {
            const uint4* src = reinterpret_cast<const uint4*>(p.x + gry * p.ld + gc);
            if (a32) {
                ld_global_cs_32B(src, raw_y[0], raw_y[1]);
                ld_global_cs_32B(src + 2, raw_y[2], raw_y[3]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) raw_y[j] = __ldcs(src + j);
            }
        }
        if constexpr (COLT) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                *reinterpret_cast<uint4*>(&tile_w[bf16_chunk(rx, 4 * s + j)]) = raw_x[j];
                *reinterpret_cast<uint4*>(&tile_w[bf16_chunk(ry, 4 * s + j)]) = raw_y[j];
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t a[4] = {raw_x[j].x, raw_x[j].y, raw_x[j].z, raw_x[j].w};
            const uint32_t b[4] = {raw_y[j].x, raw_y[j].y, raw_y[j].z, raw_y[j].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[8 * j + 2 * i] = make_float2(__uint_as_float(a[i] << 16), __uint_as_float(b[i] << 16));
                v[8 * j + 2 * i + 1] =
                    make_float2(__uint_as_float(a[i] & 0xFFFF0000u), __uint_as_float(b[i] & 0xFFFF0000u));
            }
        }
    }
    if constexpr (ROW || TWOD) {
        rotate32x2<HAD>(v);
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
            // The four segments of a row are lanes 4 pr .. 4 pr + 3 and their four bytes are
            // consecutive (k = col0/32 + s, col0/32 a multiple of 4) in both scale orders.
            // MMA order: one 32-bit store, rows past R and columns past C carrying byte 0
            // into the zeroed padding.  Plain order: one 32-bit store when the row exists,
            // all four blocks exist and the offset is 4-byte aligned, else byte stores.
            uint32_t wx = bytex << (8 * s), wy = bytey << (8 * s);
#pragma unroll
            for (int o = 1; o <= 2; o <<= 1) {
                wx |= __shfl_xor_sync(0xffffffffu, wx, o);
                wy |= __shfl_xor_sync(0xffffffffu, wy, o);
            }
            const int64_t k0 = col0 / 32, kb = p.C / 32;
            if (p.row.sf_mma) {
                if (s == 0) {
                    *reinterpret_cast<uint32_t*>(p.row.scales + sf_mma_offset(grx, k0, p.row.kb_pad)) = wx;
                    *reinterpret_cast<uint32_t*>(p.row.scales + sf_mma_offset(gry, k0, p.row.kb_pad)) = wy;
                }
            } else if (k0 + 4 <= kb && (kb & 3) == 0) {
                if (s == 0 && grx < p.R) *reinterpret_cast<uint32_t*>(p.row.scales + grx * kb + k0) = wx;
                if (s == 0 && gry < p.R) *reinterpret_cast<uint32_t*>(p.row.scales + gry * kb + k0) = wy;
            } else {
                if (vx) store_scale(p.row, grx, gc / 32, p.C / 32, bytex);
                if (vy) store_scale(p.row, gry, gc / 32, p.C / 32, bytey);
            }
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
            const uint32_t w = tile_w[bf16_chunk(32 * rb + i, q) + wi];
            v[i] = make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
        }
        rotate32x2<HAD>(v);
        float ax, ay;
        amax32x2<HAD>(v, ax, ay);
        const uint32_t bytex = scale_byte(ax, p.mode), bytey = scale_byte(ay, p.mode);
        uint4 qx, qy;
        quant32x2<HAD>(v, bytex, bytey, qx, qy);
        // row block 0 keeps output row 2 cp (its qx) and takes block 1's qx; row block 1
        // keeps output row 2 cp + 1 (its qy) and takes block 0's qy
        const uint4 send = rb == 0 ? qy : qx;
        uint4 recv;
        recv.x = __shfl_xor_sync(0xffffffffu, send.x, 16);
        recv.y = __shfl_xor_sync(0xffffffffu, send.y, 16);
        recv.z = __shfl_xor_sync(0xffffffffu, send.z, 16);
        recv.w = __shfl_xor_sync(0xffffffffu, send.w, 16);
        const uint32_t recv_b = __shfl_xor_sync(0xffffffffu, rb == 0 ? bytey : bytex, 16);
        const uint4 lo = rb == 0 ? qx : recv, hi = rb == 0 ? recv : qy;
        const uint32_t b0 = rb == 0 ? bytex : recv_b, b1 = rb == 0 ? recv_b : bytey;
        const int64_t orow = col0 + 2 * cp + rb;
        const int64_t left = (p.R - row0) / 32;
        const int nrb = left >= 2 ? 2 : (int)left;  // valid 32-row blocks of the tile
        if (orow < p.C && nrb > 0) {
            uint8_t* dst = p.colT.codes + orow * (p.R / 2) + row0 / 2;
            if (nrb == 2) {
                if ((reinterpret_cast<uintptr_t>(dst) & 31u) == 0) {
                    st_global_32B(dst, lo, hi);
                } else {
                    reinterpret_cast<uint4*>(dst)[0] = lo;
                    reinterpret_cast<uint4*>(dst)[1] = hi;
                }
            } else {
                *reinterpret_cast<uint4*>(dst) = lo;
            }
            // k = row0/32 (even) and k + 1 are adjacent bytes in both scale orders
            const int64_t off = p.colT.sf_mma ? sf_mma_offset(orow, row0 / 32, p.colT.kb_pad)
                                              : orow * (p.R / 32) + row0 / 32;
            if (nrb == 2 && (off & 1) == 0) {
                *reinterpret_cast<uint16_t*>(p.colT.scales + off) = (uint16_t)(b0 | (b1 << 8));
            } else {
                store_scale(p.colT, orow, row0 / 32, p.R / 32, b0);
                if (nrb == 2) store_scale(p.colT, orow, row0 / 32 + 1, p.R / 32, b1);
            }
        }
    }
}

template <int HAD, bool ROW, bool COLT, bool TWOD>
cudaError_t launch_one(const QuantParams& p, cudaStream_t s) {
    constexpr int smem = (COLT ? TILE_BYTES : 0) + (TWOD ? TR * 4 * 4 : 0);
    auto kern = rq_kernel<HAD, ROW, COLT, TWOD>;
    if constexpr (smem > 48 * 1024) {
        static DeviceSlots opted_in;
        int unused = 0;
        const cudaError_t e = per_device_setting(opted_in, &unused, [&](int, int*) {
            return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        });
        if (e != cudaSuccess) return e;
    }
    const dim3 grid((unsigned)((p.C + TC - 1) / TC), (unsigned)((p.R + TR - 1) / TR));
    return launch_overlapped(kern, grid, dim3(QTHREADS), smem, s, 1, MXF_PDL_QUANT != 0, p);
}

template <int HAD>
cudaError_t launch_had(const QuantParams& p, unsigned layouts, cudaStream_t s) {
    switch (layouts) {
        case MXFP4_LAYOUT_ROW:
            return launch_one<HAD, true, false, false>(p, s);
        case MXFP4_LAYOUT_COLT:
            return launch_one<HAD, false, true, false>(p, s);
        case MXFP4_LAYOUT_ROW | MXFP4_LAYOUT_COLT:
            return launch_one<HAD, true, true, false>(p, s);
        case MXFP4_LAYOUT_2D:
            return launch_one<HAD, false, false, true>(p, s);
        default:
            return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_rotate_quantize(const QuantParams& p, int had, unsigned layouts, cudaStream_t s) {
    switch (had) {
        case 0:
            return launch_had<1>(p, layouts, s);
        case 16:
            return launch_had<16>(p, layouts, s);
        case 32:
            return launch_had<32>(p, layouts, s);
        default:
            return cudaErrorInvalidValue;
    }
}

}  // namespace mx
