// quantize.cu -- fused rotate + MXFP4 quantise kernel (sm_103a).
//
// "Pretraining Large Language Models with MXFP4 on Native FP4 Hardware":
//   A.1 (x_B ~ 2^E * Q_FP4(x_B / 2^E), 32-element blocks), A.2 (deterministic tiled
//   Hadamard before quantisation), D (1x32 row, 32x1 column-transposed, 32x32 2D).
// "Decomposing MXFP4 quantization error ...": E8M0 scales, E2M1 grid, ceiling scale.
//
// One CTA owns a 128 x 128 tile of the bf16 input and reads it from HBM once.
//  - Row work: each thread owns two 32-element row segments (rows r and r + 64) in
//    registers and processes them in lockstep with packed f32x2 instructions:
//    rotation butterfly, block amax, E8M0 byte, 2 x 32 codes -> two 16-byte stores.
//  - Column work (transposed copy): the tile is staged in shared memory (16-byte
//    chunks XOR-swizzled so that both the row-wise writes and the column-wise reads
//    are bank-conflict free); each thread then owns two adjacent columns of one
//    32-row block (one 32-bit shared load gives both columns' values).
//  - 2D work: row segments as above, the per-segment amax is combined over the 32
//    rows of the tile through shared memory.
// The kernel is HBM-bound: 2 B read and 0.53 B (single) or 1.06 B (row + column)
// written per element.
#include "internal.h"
#include "ptx.cuh"

// 1: TMA-fed producer/consumer kernel (rq_tma_kernel); 0: one tile per CTA (rq_kernel).
#ifndef MXQ_TMA
#define MXQ_TMA 0
#endif

namespace mx {
namespace {

constexpr int TR = 128;  // tile rows
constexpr int TC = 128;  // tile cols
constexpr int QTHREADS = 256;

// Packed fp32 pairs: one instruction performs two independent IEEE fp32 operations
// (round to nearest even, subnormals kept), so results equal the scalar ones.
__device__ __forceinline__ float2 f2_add(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 f2_sub(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 f2_mul(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// Rotation of two independent 32-element vectors held as pairs (v[i] = element i of
// vector x and of vector y) by block-diagonal H_n (n = 1, 16, 32): stages of strides
// 1, 2, 4, 8 (, 16), each (a, b) -> (a + b, a - b) rounded to fp32.  H32 then
// multiplies by fl32(1/sqrt(32)).  For H16 the normalising x0.25 is left to the
// scaling step: with bf16 inputs every butterfly output is a multiple of 2^-133 (or
// rounded at a magnitude >= 2^-109), so s * 0.25 is exact and
// (s * 0.25) * 2^-e == s * 2^(-2-e) bit for bit.
template <int HAD>
__device__ __forceinline__ void rotate32x2(float2 (&v)[32]) {
    if constexpr (HAD > 1) {
#pragma unroll
        for (int s = 1; s < HAD; s <<= 1) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                if ((i & s) == 0) {
                    const float2 a = v[i], b = v[i + s];
                    v[i] = f2_add(a, b);
                    v[i + s] = f2_sub(a, b);
                }
            }
        }
        if constexpr (HAD == 32) {
            const float2 c = make_float2(0.17677669529663687f, 0.17677669529663687f);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = f2_mul(v[i], c);
        }
    }
}

// Block amax of the rotated values (x and y vectors).  For H16 the butterfly output
// still carries the factor 4, removed exactly here.
template <int HAD>
__device__ __forceinline__ void amax32x2(const float2 (&v)[32], float& ax, float& ay) {
    float mx = 0.0f, my = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        mx = fmaxf(mx, fabsf(v[i].x));
        my = fmaxf(my, fabsf(v[i].y));
    }
    if constexpr (HAD == 16) {
        mx *= 0.25f;
        my *= 0.25f;
    }
    ax = mx;
    ay = my;
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

// The factor that maps a rotated value to E2M1 units: 2^-e (e = byte - 127), times the
// deferred 0.25 for H16.  Both are powers of two (2^-128 .. 2^127, exact in fp32).
template <int HAD>
__device__ __forceinline__ float unit_factor(uint32_t byte) {
    if constexpr (HAD == 16) return __uint_as_float(byte <= 251u ? (252u - byte) << 23 : 0x00400000u >> (byte - 252u));
    return __uint_as_float((254u - byte) << 23);
}

__device__ __forceinline__ uint32_t cvt_e2m1x8v(float a0, float a1, float a2, float a3, float a4, float a5, float a6,
                                                float a7) {
    const float t[8] = {a0, a1, a2, a3, a4, a5, a6, a7};
    return cvt_e2m1x8(t);
}

// Codes of both vectors: u = v * factor (exact power-of-two scaling), then
// round-to-nearest-even E2M1 with saturation, 32 codes -> 16 bytes per vector.
template <int HAD>
__device__ __forceinline__ void quant32x2(const float2 (&v)[32], uint32_t bx, uint32_t by, uint4& qx, uint4& qy) {
    const float2 f = make_float2(unit_factor<HAD>(bx), unit_factor<HAD>(by));
    float2 u[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) u[i] = f2_mul(v[i], f);
    uint32_t wx[4], wy[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int b = 8 * j;
        wx[j] = cvt_e2m1x8v(u[b].x, u[b + 1].x, u[b + 2].x, u[b + 3].x, u[b + 4].x, u[b + 5].x, u[b + 6].x, u[b + 7].x);
        wy[j] = cvt_e2m1x8v(u[b].y, u[b + 1].y, u[b + 2].y, u[b + 3].y, u[b + 4].y, u[b + 5].y, u[b + 6].y, u[b + 7].y);
    }
    qx = make_uint4(wx[0], wx[1], wx[2], wx[3]);
    qy = make_uint4(wy[0], wy[1], wy[2], wy[3]);
}

__device__ __forceinline__ void store_scale(const QuantOut& o, int64_t r, int64_t kb, int64_t kb_per_row,
                                            uint32_t byte) {
    const int64_t off = o.sf_mma ? sf_mma_offset(r, kb, o.kb_pad) : r * kb_per_row + kb;
    o.scales[off] = (uint8_t)byte;
}

// Swizzled position (in 32-bit words) of 16-byte chunk q of tile row r: the row-wise
// writes (4 threads per row) and the column-wise reads (32 consecutive words of one
// row per warp) both hit 32 distinct banks.
[[maybe_unused]] __device__ __forceinline__ int tile_chunk(int r, int q) { return (q ^ ((q >> 2) & 3) ^ ((r & 1) << 2)) * 4; }

template <int HAD, bool ROW, bool COLT, bool TWOD>
__global__ void __launch_bounds__(QTHREADS, 2) rq_kernel(const QuantParams p) {
    __shared__ __align__(16) uint32_t tile[COLT ? TR * (TC / 2) : 4];
    __shared__ float seg_amax[TWOD ? TR * 4 : 1];

    const int t = threadIdx.x;
    const int64_t row0 = (int64_t)blockIdx.y * TR;
    const int64_t col0 = (int64_t)blockIdx.x * TC;

    // ---- two row segments owned by this thread: rows pr and pr + 64, columns 32*s ..
    const int s = t & 3, pr = t >> 2;
    const int rx = pr, ry = pr + 64;
    const int64_t gc = col0 + 32 * s;
    const int64_t grx = row0 + rx, gry = row0 + ry;
    const bool vx = grx < p.R && gc < p.C, vy = gry < p.R && gc < p.C;
    uint4 raw_x[4], raw_y[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) raw_x[j] = raw_y[j] = make_uint4(0, 0, 0, 0);
    if (vx) {
        const uint4* src = reinterpret_cast<const uint4*>(p.x + grx * p.ld + gc);
#pragma unroll
        for (int j = 0; j < 4; ++j) raw_x[j] = __ldcs(src + j);
    }
    if (vy) {
        const uint4* src = reinterpret_cast<const uint4*>(p.x + gry * p.ld + gc);
#pragma unroll
        for (int j = 0; j < 4; ++j) raw_y[j] = __ldcs(src + j);
    }
    if constexpr (COLT) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            *reinterpret_cast<uint4*>(&tile[rx * (TC / 2) + tile_chunk(rx, 4 * s + j)]) = raw_x[j];
            *reinterpret_cast<uint4*>(&tile[ry * (TC / 2) + tile_chunk(ry, 4 * s + j)]) = raw_y[j];
        }
    }

    if constexpr (ROW || TWOD) {
        float2 v[32];
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
            if (vx) {
                *reinterpret_cast<uint4*>(p.row.codes + grx * (p.C / 2) + gc / 2) = qx;
                store_scale(p.row, grx, gc / 32, p.C / 32, bytex);
            }
            if (vy) {
                *reinterpret_cast<uint4*>(p.row.codes + gry * (p.C / 2) + gc / 2) = qy;
                store_scale(p.row, gry, gc / 32, p.C / 32, bytey);
            }
        }
    }

    if constexpr (COLT) {
        __syncthreads();
        // two adjacent columns (2*cp, 2*cp + 1) x one 32-row block per thread
        const int cp = t & 63, rb = t >> 6;
        const int64_t gcol = col0 + 2 * cp, grow = row0 + 32 * rb;
        if (gcol < p.C && grow < p.R) {
            float2 v[32];
            const int q = cp >> 2, wi = cp & 3;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int rr = 32 * rb + i;
                const uint32_t w = tile[rr * (TC / 2) + tile_chunk(rr, q) + wi];
                v[i] = make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
            }
            rotate32x2<HAD>(v);
            float ax, ay;
            amax32x2<HAD>(v, ax, ay);
            const uint32_t bytex = scale_byte(ax, p.mode), bytey = scale_byte(ay, p.mode);
            uint4 qx, qy;
            quant32x2<HAD>(v, bytex, bytey, qx, qy);
            *reinterpret_cast<uint4*>(p.colT.codes + gcol * (p.R / 2) + grow / 2) = qx;
            *reinterpret_cast<uint4*>(p.colT.codes + (gcol + 1) * (p.R / 2) + grow / 2) = qy;
            store_scale(p.colT, gcol, grow / 32, p.R / 32, bytex);
            store_scale(p.colT, gcol + 1, grow / 32, p.R / 32, bytey);
        }
    }
}

// ---------------------------------------------------------------------------------
// TMA-fed variant: persistent CTAs (two per SM) walk 128 x 128 tiles; thread 0 keeps
// the next Q_STAGES - 1 tiles of its CTA in flight (two 64-column boxes per tile,
// 128-byte swizzle) while all 256 threads process the current one.  The arithmetic
// is the same as rq_kernel's.
constexpr int Q_STAGES = 3;
constexpr int Q_TILE_BYTES = TR * TC * 2;  // 32 KB
constexpr int Q_BOX_BYTES = Q_TILE_BYTES / 2;
constexpr int Q_OFF_BAR = Q_STAGES * Q_TILE_BYTES;
constexpr int Q_OFF_AMAX = Q_OFF_BAR + Q_STAGES * 8;
constexpr int Q_TMA_SMEM = Q_OFF_AMAX + TR * 4 * 4 + 1024;

// Word offset (32-bit units) of 16-byte chunk `chunk` (0..15) of tile row r in the
// swizzled stage: columns 0-63 are box 0, 64-127 box 1; within a box a row is 128 B
// with chunk c stored at c ^ (r % 8).
__device__ __forceinline__ int sw_word(int r, int chunk) {
    return ((chunk >> 3) * Q_BOX_BYTES + r * 128 + (((chunk & 7) ^ (r & 7)) << 4)) >> 2;
}

template <int HAD, bool ROW, bool COLT, bool TWOD>
__global__ void __launch_bounds__(QTHREADS, 2) rq_tma_kernel(const __grid_constant__ QuantTmaParams P) {
    const QuantParams& p = P.p;
    extern __shared__ uint8_t q_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(q_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Q_OFF_BAR);
    float* seg_amax = reinterpret_cast<float*>(smem + Q_OFF_AMAX);
    const int t = threadIdx.x;

    auto issue = [&](uint32_t j) {  // tile j of this CTA's sequence -> stage j % Q_STAGES
        const int64_t tile = blockIdx.x + (int64_t)j * gridDim.x;
        if (tile >= P.tiles) return;
        const int st = (int)(j % Q_STAGES);
        const int32_t row0 = (int32_t)((tile / P.tiles_c) * TR), col0 = (int32_t)((tile % P.tiles_c) * TC);
        mbar_arrive_expect_tx(&full[st], Q_TILE_BYTES);
        uint8_t* dst = smem + st * Q_TILE_BYTES;
        tma_load_2d(dst, &P.map_x, &full[st], col0, row0);
        tma_load_2d(dst + Q_BOX_BYTES, &P.map_x, &full[st], col0 + 64, row0);
    };

    if (t == 0) {
        for (int st = 0; st < Q_STAGES; ++st) mbar_init(&full[st], 1);
        fence_mbar_init();
        prefetch_tmap(&P.map_x);
        for (uint32_t j = 0; j + 1 < Q_STAGES; ++j) issue(j);
    }
    __syncthreads();

    uint32_t i = 0;
    for (int64_t tile = blockIdx.x; tile < P.tiles; tile += gridDim.x, ++i) {
        // the stage refilled here was released by the __syncthreads ending iteration i - 1
        if (t == 0) issue(i + Q_STAGES - 1);
        const int st = (int)(i % Q_STAGES);
        const bool landed = wait_bounded(&full[st], (i / Q_STAGES) & 1u, P.wait_ns, P.status);
        const uint32_t* buf = reinterpret_cast<const uint32_t*>(smem + st * Q_TILE_BYTES);
        const int64_t row0 = (tile / P.tiles_c) * TR, col0 = (tile % P.tiles_c) * TC;

        if constexpr (ROW || TWOD) {
            const int s = t & 3, pr = t >> 2;
            const int rx = pr, ry = pr + 64;
            const int64_t gc = col0 + 32 * s;
            const int64_t grx = row0 + rx, gry = row0 + ry;
            const bool vx = landed && grx < p.R && gc < p.C, vy = landed && gry < p.R && gc < p.C;
            float2 v[32];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint4 a4 = *reinterpret_cast<const uint4*>(&buf[sw_word(rx, 4 * s + j)]);
                const uint4 b4 = *reinterpret_cast<const uint4*>(&buf[sw_word(ry, 4 * s + j)]);
                const uint32_t a[4] = {a4.x, a4.y, a4.z, a4.w};
                const uint32_t b[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    v[8 * j + 2 * k] = make_float2(__uint_as_float(a[k] << 16), __uint_as_float(b[k] << 16));
                    v[8 * j + 2 * k + 1] =
                        make_float2(__uint_as_float(a[k] & 0xFFFF0000u), __uint_as_float(b[k] & 0xFFFF0000u));
                }
            }
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
                for (int k = 0; k < 32; ++k) {
                    tx = fmaxf(tx, seg_amax[(bx + k) * 4 + s]);
                    ty = fmaxf(ty, seg_amax[(by + k) * 4 + s]);
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
                if (vx) {
                    *reinterpret_cast<uint4*>(p.row.codes + grx * (p.C / 2) + gc / 2) = qx;
                    store_scale(p.row, grx, gc / 32, p.C / 32, bytex);
                }
                if (vy) {
                    *reinterpret_cast<uint4*>(p.row.codes + gry * (p.C / 2) + gc / 2) = qy;
                    store_scale(p.row, gry, gc / 32, p.C / 32, bytey);
                }
            }
        }

        if constexpr (COLT) {
            const int cp = t & 63, rb = t >> 6;
            const int64_t gcol = col0 + 2 * cp, grow = row0 + 32 * rb;
            if (landed && gcol < p.C && grow < p.R) {
                float2 v[32];
                const int chunk = cp >> 2, wi = cp & 3;  // 16-byte chunk of the row holding columns 2cp, 2cp+1
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    const int rr = 32 * rb + k;
                    const uint32_t w = buf[sw_word(rr, chunk) + wi];
                    v[k] = make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
                }
                rotate32x2<HAD>(v);
                float ax, ay;
                amax32x2<HAD>(v, ax, ay);
                const uint32_t bytex = scale_byte(ax, p.mode), bytey = scale_byte(ay, p.mode);
                uint4 qx, qy;
                quant32x2<HAD>(v, bytex, bytey, qx, qy);
                *reinterpret_cast<uint4*>(p.colT.codes + gcol * (p.R / 2) + grow / 2) = qx;
                *reinterpret_cast<uint4*>(p.colT.codes + (gcol + 1) * (p.R / 2) + grow / 2) = qy;
                store_scale(p.colT, gcol, grow / 32, p.R / 32, bytex);
                store_scale(p.colT, gcol + 1, grow / 32, p.R / 32, bytey);
            }
        }
        __syncthreads();  // every thread is done with this stage (and with seg_amax)
    }
    // every copy this CTA issued has been waited for by the loop above (issue only
    // targets tiles the loop visits), so nothing is in flight at exit.
}

template <int HAD, bool ROW, bool COLT, bool TWOD>
cudaError_t launch_tma(const QuantTmaParams& P, cudaStream_t st) {
    auto kern = rq_tma_kernel<HAD, ROW, COLT, TWOD>;
    static bool configured[64] = {};
    static int sms[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Q_TMA_SMEM);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    const int64_t max_grid = 2 * (int64_t)sms[dev];
    const unsigned grid = (unsigned)(P.tiles < max_grid ? P.tiles : max_grid);
    kern<<<grid, QTHREADS, Q_TMA_SMEM, st>>>(P);
    return cudaGetLastError();
}

template <int HAD>
cudaError_t launch_had_tma(const QuantTmaParams& P, unsigned layouts, cudaStream_t s) {
    switch (layouts) {
        case MXFP4_LAYOUT_ROW:
            return launch_tma<HAD, true, false, false>(P, s);
        case MXFP4_LAYOUT_COLT:
            return launch_tma<HAD, false, true, false>(P, s);
        case MXFP4_LAYOUT_ROW | MXFP4_LAYOUT_COLT:
            return launch_tma<HAD, true, true, false>(P, s);
        case MXFP4_LAYOUT_2D:
            return launch_tma<HAD, false, false, true>(P, s);
        default:
            return cudaErrorInvalidValue;
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
#if MXQ_TMA
    QuantTmaParams P{};
    P.p = p;
    if (!encode_bf16_map(&P.map_x, p.x, p.R, p.C, p.ld)) return cudaErrorInvalidValue;
    P.tiles_c = (p.C + TC - 1) / TC;
    P.tiles = P.tiles_c * ((p.R + TR - 1) / TR);
    P.status = device_status_ptr();
    P.wait_ns = quant_wait_ns();
    switch (had) {
        case 0:
            return launch_had_tma<1>(P, layouts, s);
        case 16:
            return launch_had_tma<16>(P, layouts, s);
        case 32:
            return launch_had_tma<32>(P, layouts, s);
        default:
            return cudaErrorInvalidValue;
    }
#else
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
#endif
}

}  // namespace mx
