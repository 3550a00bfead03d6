// quantize.cu -- fused rotate + MXFP4 quantise kernel (sm_103a).
//
// "Pretraining Large Language Models with MXFP4 on Native FP4 Hardware":
//   A.1 (x_B ~ 2^E * Q_FP4(x_B / 2^E), 32-element blocks), A.2 (deterministic tiled
//   Hadamard before quantisation), D (1x32 row, 32x1 column-transposed, 32x32 2D).
// "Decomposing MXFP4 quantization error ...": E8M0 scales, E2M1 grid, ceiling scale.
//
// One CTA owns a 64 x 128 tile of the bf16 input and reads it from HBM once.
//  - Row work: each thread owns one 32-element segment of a row in registers:
//    rotation butterfly, block amax, E8M0 byte, 32 codes -> one 16-byte store.
//  - Column work (transposed copy): the tile is staged in shared memory (16-byte
//    chunks XOR-swizzled so that both the row-wise writes and the column-wise reads
//    are bank-conflict free); each thread then owns one 32-row segment of a column.
//  - 2D work: row segments as above, the per-segment amax is combined over the 32
//    rows of the tile through shared memory.
// The kernel is HBM-bound: 2 B read and 0.53 B (single) or 1.06 B (row + column)
// written per element.
#include "internal.h"
#include "ptx.cuh"

namespace mx {
namespace {

constexpr int TR = 64;   // tile rows
constexpr int TC = 128;  // tile cols
constexpr int QTHREADS = 256;

// fp32 rotation of a 32-element register vector by block-diagonal H_n (n = 1, 16, 32):
// stages of strides 1, 2, 4, 8 (, 16), each (a, b) -> (a + b, a - b) rounded to fp32,
// then one multiply by fl32(1/sqrt(n)).
template <int HAD>
__device__ __forceinline__ void rotate32(float (&v)[32]) {
    if constexpr (HAD > 1) {
#pragma unroll
        for (int s = 1; s < HAD; s <<= 1) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                if ((i & s) == 0) {
                    const float a = v[i], b = v[i + s];
                    v[i] = __fadd_rn(a, b);
                    v[i + s] = __fsub_rn(a, b);
                }
            }
        }
        const float c = (HAD == 16) ? 0.25f : 0.17677669529663687f;
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __fmul_rn(v[i], c);
    }
}

__device__ __forceinline__ float amax32(const float (&v)[32]) {
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) m = fmaxf(m, fabsf(v[i]));
    return m;
}

// E8M0 byte from the block amax (exponent bits of a non-negative fp32):
//   floor mode: biased_exp(amax) - 2
//   ceil mode:  biased_exp(amax) - 2, plus one when the mantissa exceeds 1.5
// clamped below at 0 (amax == 0 or tiny).  Never above 253 for finite input.
__device__ __forceinline__ uint32_t scale_byte(float amax, int mode) {
    const uint32_t b = __float_as_uint(amax);
    const int eb = (int)(b >> 23);
    const int adj = (mode == 1 && (b & 0x7FFFFFu) > 0x400000u) ? 1 : 2;
    return (uint32_t)max(eb - adj, 0);
}

// Codes of 32 values for E8M0 byte `byte`: u = v * 2^-(byte-127) (exact power-of-two
// scaling), then round-to-nearest-even E2M1 with saturation.
__device__ __forceinline__ uint4 quant32(const float (&v)[32], uint32_t byte) {
    const float inv = __uint_as_float((254u - byte) << 23);
    float u[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) u[i] = __fmul_rn(v[i], inv);
    uint4 q;
    q.x = cvt_e2m1x8(u + 0);
    q.y = cvt_e2m1x8(u + 8);
    q.z = cvt_e2m1x8(u + 16);
    q.w = cvt_e2m1x8(u + 24);
    return q;
}

__device__ __forceinline__ void unpack_bf16x8(const uint4& w, float* v) {
    const uint32_t a[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(a[i] << 16);
        v[2 * i + 1] = __uint_as_float(a[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ void store_scale(const QuantOut& o, int64_t r, int64_t kb, int64_t kb_per_row,
                                            uint32_t byte) {
    const int64_t off = o.sf_mma ? sf_mma_offset(r, kb, o.kb_pad) : r * kb_per_row + kb;
    o.scales[off] = (uint8_t)byte;
}

// Swizzled position (in 32-bit words) of 16-byte chunk q of tile row r.
__device__ __forceinline__ int tile_chunk(int r, int q) { return (q ^ ((q >> 2) & 3) ^ ((r & 1) << 2)) * 4; }

template <int HAD, bool ROW, bool COLT, bool TWOD>
__global__ void __launch_bounds__(QTHREADS) rq_kernel(const QuantParams p) {
    __shared__ __align__(16) uint32_t tile[COLT ? TR * (TC / 2) : 4];
    __shared__ float seg_amax[TWOD ? TR * 4 : 1];

    const int t = threadIdx.x;
    const int64_t row0 = (int64_t)blockIdx.y * TR;
    const int64_t col0 = (int64_t)blockIdx.x * TC;

    // ---- row segment owned by this thread
    const int r = t >> 2, s = t & 3;
    const int64_t gr = row0 + r, gc = col0 + 32 * s;
    const bool valid = gr < p.R && gc < p.C;
    uint4 raw[4];
    if (valid) {
        const uint4* src = reinterpret_cast<const uint4*>(p.x + gr * p.ld + gc);
#pragma unroll
        for (int j = 0; j < 4; ++j) raw[j] = __ldcs(src + j);
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) raw[j] = make_uint4(0, 0, 0, 0);
    }
    if constexpr (COLT) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4*>(&tile[r * (TC / 2) + tile_chunk(r, 4 * s + j)]) = raw[j];
    }

    if constexpr (ROW || TWOD) {
        float v[32];
#pragma unroll
        for (int j = 0; j < 4; ++j) unpack_bf16x8(raw[j], v + 8 * j);
        rotate32<HAD>(v);
        const float am = amax32(v);
        if constexpr (TWOD) {
            seg_amax[r * 4 + s] = am;
            __syncthreads();
            float tm = 0.0f;
            const int rb = r & ~31;
#pragma unroll 8
            for (int i = 0; i < 32; ++i) tm = fmaxf(tm, seg_amax[(rb + i) * 4 + s]);
            const uint32_t byte = scale_byte(tm, p.mode);
            if (valid) {
                *reinterpret_cast<uint4*>(p.twoD.codes + gr * (p.C / 2) + gc / 2) = quant32(v, byte);
                if ((r & 31) == 0) p.twoD.scales[(gr / 32) * (p.C / 32) + gc / 32] = (uint8_t)byte;
            }
        } else {
            const uint32_t byte = scale_byte(am, p.mode);
            if (valid) {
                *reinterpret_cast<uint4*>(p.row.codes + gr * (p.C / 2) + gc / 2) = quant32(v, byte);
                store_scale(p.row, gr, gc / 32, p.C / 32, byte);
            }
        }
    }

    if constexpr (COLT) {
        __syncthreads();
        const int c = t & (TC - 1), rb = t >> 7;
        const int64_t gcol = col0 + c, grow = row0 + 32 * rb;
        if (gcol < p.C && grow < p.R) {
            float v[32];
            const int word = c >> 1, q = word >> 2, wi = word & 3;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int rr = 32 * rb + i;
                const uint32_t w = tile[rr * (TC / 2) + tile_chunk(rr, q) + wi];
                v[i] = __uint_as_float((c & 1) ? (w & 0xFFFF0000u) : (w << 16));
            }
            rotate32<HAD>(v);
            const uint32_t byte = scale_byte(amax32(v), p.mode);
            *reinterpret_cast<uint4*>(p.colT.codes + gcol * (p.R / 2) + grow / 2) = quant32(v, byte);
            store_scale(p.colT, gcol, grow / 32, p.R / 32, byte);
        }
    }
}

template <int HAD>
cudaError_t launch_had(const QuantParams& p, unsigned layouts, cudaStream_t s) {
    const dim3 grid((unsigned)((p.C + TC - 1) / TC), (unsigned)((p.R + TR - 1) / TR));
    switch (layouts) {
        case MXFP4_LAYOUT_ROW:
            rq_kernel<HAD, true, false, false><<<grid, QTHREADS, 0, s>>>(p);
            break;
        case MXFP4_LAYOUT_COLT:
            rq_kernel<HAD, false, true, false><<<grid, QTHREADS, 0, s>>>(p);
            break;
        case MXFP4_LAYOUT_ROW | MXFP4_LAYOUT_COLT:
            rq_kernel<HAD, true, true, false><<<grid, QTHREADS, 0, s>>>(p);
            break;
        case MXFP4_LAYOUT_2D:
            rq_kernel<HAD, false, false, true><<<grid, QTHREADS, 0, s>>>(p);
            break;
        default:
            return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
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
