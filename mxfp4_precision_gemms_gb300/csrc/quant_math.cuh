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

}  // namespace mx
