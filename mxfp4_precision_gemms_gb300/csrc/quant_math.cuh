// quant_math.cuh -- per-thread arithmetic shared by the quantiser kernels: packed
// fp32 pairs, the block-diagonal Hadamard butterfly, block amax, E8M0 scale byte and
// E2M1 conversion ("Pretraining Large Language Models with MXFP4 on Native FP4
// Hardware", A.1-A.2; "Decomposing MXFP4 quantization error ...", E2M1 grid and E8M0
// scale).  Each thread works on two independent 32-element vectors at once (x and y
// halves of float2 values).
#pragma once

#include "internal.h"
#include "ptx.cuh"

namespace mx {

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

// d = a * b + c on each half, one rounding (IEEE fma).
__device__ __forceinline__ float2 f2_fma(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
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

// Stride-1 butterfly straight from a bf16 pair: w holds elements 2i (low half) and 2i + 1
// (high half); c is element 2i + 1 widened to fp32.  The mixed-precision add / sub widen
// the low half exactly and round once, so (s, d) equal fl32(x_2i + x_2i+1) and
// fl32(x_2i - x_2i+1) of the unpacked values.
__device__ __forceinline__ void bfly_lo(uint32_t w, float c, float& s, float& d) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tadd.rn.f32.bf16 %0, l, %3;\n\tsub.rn.f32.bf16 %1, l, %3;\n\t}"
        : "=f"(s), "=f"(d)
        : "r"(w), "f"(c));
}

// rotate32x2 without its stride-1 stage (done by bfly_lo while unpacking).
template <int HAD>
__device__ __forceinline__ void rotate32x2_from2(float2 (&v)[32]) {
    if constexpr (HAD > 1) {
#pragma unroll
        for (int s = 2; s < HAD; s <<= 1) {
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

// Three-input fp32 maximum (one instruction on sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Block amax of the rotated values (x and y vectors).  For H16 the butterfly output
// still carries the factor 4, removed exactly here.
template <int HAD>
__device__ __forceinline__ void amax32x2(const float2 (&v)[32], float& ax, float& ay) {
    float mx = 0.0f, my = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        mx = fmax3(mx, fabsf(v[i].x), fabsf(v[i + 1].x));
        my = fmax3(my, fabsf(v[i].y), fabsf(v[i + 1].y));
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

// ---- shared by the tiled quantiser kernels (64 x 128 bf16 tiles, 128 threads) ----

// Staged tile of 64 rows x 128 bf16: 32-bit word index of 16-byte chunk q (0..15) of row
// r.  The XOR on the chunk index (by q bits 2-3, row bit 0 and row bit 5) keeps the
// row-wise 16-byte writes (8 rows x 4 segments per warp) and the column-wise 32-bit reads
// (rows i and 32 + i, 16 column pairs each, per warp) bank-conflict free.
__device__ __forceinline__ int tile_chunk(int r, int q) {
    return r * 64 + ((q ^ ((q >> 2) & 3) ^ (((r ^ (r >> 5)) & 1) << 2)) << 2);
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

// The thread's two 64-byte row segments of bf16 (rows gx and gy of x, columns gc ..
// gc + 31; zeros where not valid).  32-byte loads when `wide` (every row segment starts
// on a 32-byte boundary), so that each load instruction uses whole 32-byte sectors.
__device__ __forceinline__ void load_row_pair(const QuantParams& p, int64_t gx, int64_t gy, int64_t gc, bool vx,
                                              bool vy, bool wide, uint4 (&rx)[4], uint4 (&ry)[4]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) rx[j] = ry[j] = make_uint4(0, 0, 0, 0);
    if (vx) {
        const uint4* src = reinterpret_cast<const uint4*>(p.x + gx * p.ld + gc);
        if (wide) {
            ld_global_cs_32B(src, rx[0], rx[1]);
            ld_global_cs_32B(src + 2, rx[2], rx[3]);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) rx[j] = __ldcs(src + j);
        }
    }
    if (vy) {
        const uint4* src = reinterpret_cast<const uint4*>(p.x + gy * p.ld + gc);
        if (wide) {
            ld_global_cs_32B(src, ry[0], ry[1]);
            ld_global_cs_32B(src + 2, ry[2], ry[3]);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) ry[j] = __ldcs(src + j);
        }
    }
}

// Whether every row segment of x starts on a 32-byte boundary.
__device__ __forceinline__ bool rows_32B_aligned(const QuantParams& p) {
    return ((reinterpret_cast<uintptr_t>(p.x) | (uintptr_t)(p.ld * 2)) & 31u) == 0;
}

// Row-copy scale bytes of one tile row: the four segments of the row are lanes
// 4 pr .. 4 pr + 3 (s = lane & 3) and their bytes are consecutive (k = col0/32 + s,
// col0/32 a multiple of 4) in both scale orders.  MMA order: one 32-bit store, rows past
// R and columns past C carrying byte 0 into the zeroed padding.  Plain order: one 32-bit
// store when the row exists, all four blocks exist and the offset is 4-byte aligned,
// else byte stores.  Every lane of the warp must call this.
__device__ __forceinline__ void store_row_scales(const QuantOut& o, const QuantParams& p, int64_t col0, int s,
                                                 int64_t gx, int64_t gy, bool vx, bool vy, uint32_t bx,
                                                 uint32_t by) {
    uint32_t wx = bx << (8 * s), wy = by << (8 * s);
#pragma unroll
    for (int d = 1; d <= 2; d <<= 1) {
        wx |= __shfl_xor_sync(0xffffffffu, wx, d);
        wy |= __shfl_xor_sync(0xffffffffu, wy, d);
    }
    const int64_t k0 = col0 / 32, kb = p.C / 32;
    if (o.sf_mma) {
        if (s == 0) {
            *reinterpret_cast<uint32_t*>(o.scales + sf_mma_offset(gx, k0, o.kb_pad)) = wx;
            *reinterpret_cast<uint32_t*>(o.scales + sf_mma_offset(gy, k0, o.kb_pad)) = wy;
        }
    } else if (k0 + 4 <= kb && (kb & 3) == 0) {
        if (s == 0 && gx < p.R) *reinterpret_cast<uint32_t*>(o.scales + gx * kb + k0) = wx;
        if (s == 0 && gy < p.R) *reinterpret_cast<uint32_t*>(o.scales + gy * kb + k0) = wy;
    } else {
        const int64_t gc = col0 + 32 * s;
        if (vx) store_scale(o, gx, gc / 32, kb, bx);
        if (vy) store_scale(o, gy, gc / 32, kb, by);
    }
}

// Transposed copy of one warp's 16 column pairs: lanes l and l ^ 16 hold row blocks 0
// and 1 of columns (2 cp, 2 cp + 1) as codes qx (column 2 cp), qy (column 2 cp + 1) and
// bytes bx, by.  One shuffle exchange gives every lane one whole output row (2 cp + rb):
// its two 16-byte halves leave as one 32-byte store and its two scale bytes as one 16-bit
// store.  Every lane of the warp must call this.
__device__ __forceinline__ void store_colT_pair(const QuantOut& o, const QuantParams& p, int64_t row0, int64_t col0,
                                                int cp, int rb, uint4 qx, uint4 qy, uint32_t bx, uint32_t by) {
    const uint4 send = rb == 0 ? qy : qx;
    uint4 recv;
    recv.x = __shfl_xor_sync(0xffffffffu, send.x, 16);
    recv.y = __shfl_xor_sync(0xffffffffu, send.y, 16);
    recv.z = __shfl_xor_sync(0xffffffffu, send.z, 16);
    recv.w = __shfl_xor_sync(0xffffffffu, send.w, 16);
    const uint32_t recv_b = __shfl_xor_sync(0xffffffffu, rb == 0 ? by : bx, 16);
    const uint4 lo = rb == 0 ? qx : recv, hi = rb == 0 ? recv : qy;
    const uint32_t b0 = rb == 0 ? bx : recv_b, b1 = rb == 0 ? recv_b : by;
    const int64_t orow = col0 + 2 * cp + rb;
    const int64_t left = (p.R - row0) / 32;
    const int nrb = left >= 2 ? 2 : (int)left;  // valid 32-row blocks of the tile
    if (orow >= p.C || nrb <= 0) return;
    uint8_t* dst = o.codes + orow * (p.R / 2) + row0 / 2;
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
    const int64_t off = o.sf_mma ? sf_mma_offset(orow, row0 / 32, o.kb_pad) : orow * (p.R / 32) + row0 / 32;
    if (nrb == 2 && (off & 1) == 0) {
        *reinterpret_cast<uint16_t*>(o.scales + off) = (uint16_t)(b0 | (b1 << 8));
    } else {
        store_scale(o, orow, row0 / 32, p.R / 32, b0);
        if (nrb == 2) store_scale(o, orow, row0 / 32 + 1, p.R / 32, b1);
    }
}

}  // namespace mx
