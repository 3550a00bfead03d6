// quant_fixes.cu -- the quantiser fixes of "Decomposing MXFP4 quantization error for
// LLM reinforcement learning" (MBS -- macro block scaling, OF -- outlier fallback),
// row layout, on the rotated values of "Pretraining Large Language Models with MXFP4
// on Native FP4 Hardware" (A.1-A.2).
//
// Same tiling as the row work of rq_kernel: one CTA of 128 threads per 64 x 128 tile,
// each thread two 32-element row segments (rows r and r + 32) processed as f32x2
// pairs; the four threads of a tile row hold the row's 128 columns.
//  OF:  q1 = Q(v), r = v - dq(q1) (exact in fp32), q2 = Q(r); the second pass's E8M0
//       bytes carry alpha = 2^alpha_log2: stored byte = max(byte + alpha_log2, 0), so
//       that x_OF = dq(q1) + dq(q2).
//  MBS: per 128 values (one tile row) one byte k, the largest value with
//       (1 + k/256) f <= T for the macro amax A = f 2^E (T = 1.5 if f <= 1.5, else 3);
//       v' = fl32((1 + k/256) v), q = Q(v'); reconstruction dq(q) / (1 + k/256).
#include <cuda_fp16.h>

#include "quant_math.cuh"

namespace mx {
namespace {

constexpr int FX_TR = 64, FX_TC = 128, FX_THREADS = 128;

// Loads the thread's two bf16 row segments (zeros outside the matrix) as f32x2 pairs.
__device__ __forceinline__ void load_pairs(const QuantParams& p, int64_t grx, int64_t gry, int64_t gc, bool vx,
                                           bool vy, float2 (&v)[32]) {
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
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t a[4] = {raw_x[j].x, raw_x[j].y, raw_x[j].z, raw_x[j].w};
        const uint32_t b[4] = {raw_y[j].x, raw_y[j].y, raw_y[j].z, raw_y[j].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[8 * j + 2 * i] = make_float2(__uint_as_float(a[i] << 16), __uint_as_float(b[i] << 16));
            v[8 * j + 2 * i + 1] = make_float2(__uint_as_float(a[i] & 0xFFFF0000u), __uint_as_float(b[i] & 0xFFFF0000u));
        }
    }
}

// Rotated values in their normalised form (H16's x0.25 applied; exact).
template <int HAD>
__device__ __forceinline__ void rotate_normalised(float2 (&v)[32]) {
    rotate32x2<HAD>(v);
    if constexpr (HAD == 16) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = f2_mul(v[i], make_float2(0.25f, 0.25f));
    }
}

// Values of E2M1 codes 2B and 2B + 1 of a packed word (code i in nibble i): the hardware
// conversion of byte B to an f16 pair {nibble 2B, nibble 2B + 1}, widened to fp32.  Exact:
// every E2M1 value (0, 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives, -0 included) is an f16.
template <int B>
__device__ __forceinline__ float2 e2m1x2_value(uint32_t w) {
    uint32_t h;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b%2;\n\t}"
        : "=r"(h)
        : "r"(w), "n"(B));
    return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// Packed fused multiply-add of two independent fp32 pairs: a * b + c, one rounding each.
__device__ __forceinline__ float2 f2_fma(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

// Elements 2B, 2B + 1 of both vectors: v - dq(q1) = v + d * (-2^e).
template <int B>
__device__ __forceinline__ void residual_pair(uint32_t wx, uint32_t wy, float2 npx, float2& v0, float2& v1) {
    const float2 dx = e2m1x2_value<B>(wx), dy = e2m1x2_value<B>(wy);
    v0 = f2_fma(make_float2(dx.x, dy.x), npx, v0);
    v1 = f2_fma(make_float2(dx.y, dy.y), npx, v1);
}

// 2^e for e = byte - 127 in [-127, 127] (2^-127 is subnormal; exact).
__device__ __forceinline__ float pow2_of_byte(uint32_t byte) {
    return __uint_as_float(byte >= 1u ? byte << 23 : 0x00400000u);
}

// The thread's two 16-byte code pieces (rows gx and gy, columns gc .. gc + 31) and the
// tile rows' scale bytes (gathered into one 32-bit store per row).  Every lane calls it.
__device__ __forceinline__ void store_rows(const QuantOut& o, const QuantParams& p, int64_t col0, int s, int64_t gx,
                                           int64_t gy, int64_t gc, bool vx, bool vy, uint4 qx, uint4 qy,
                                           uint32_t bx, uint32_t by) {
    if (vx) *reinterpret_cast<uint4*>(o.codes + gx * (p.C / 2) + gc / 2) = qx;
    if (vy) *reinterpret_cast<uint4*>(o.codes + gy * (p.C / 2) + gc / 2) = qy;
    store_row_scales(o, p, col0, s, gx, gy, vx, vy, bx, by);
}

template <int HAD>
__global__ void __launch_bounds__(FX_THREADS, 5) rq_of_kernel(const QuantParams p, const QuantOut q2, int alpha_log2) {
    const int t = threadIdx.x;
    const int s = t & 3, pr = t >> 2;
    const int64_t row0 = (int64_t)blockIdx.y * FX_TR, col0 = (int64_t)blockIdx.x * FX_TC;
    const int64_t gc = col0 + 32 * s, grx = row0 + pr, gry = row0 + pr + 32;
    const bool vx = grx < p.R && gc < p.C, vy = gry < p.R && gc < p.C;
    float2 v[32];
    load_pairs(p, grx, gry, gc, vx, vy, v);
    rotate_normalised<HAD>(v);

    // first pass
    float ax, ay;
    amax32x2<1>(v, ax, ay);
    const uint32_t b1x = scale_byte(ax, p.mode), b1y = scale_byte(ay, p.mode);
    uint4 qx, qy;
    quant32x2<1>(v, b1x, b1y, qx, qy);
    store_rows(p.row, p, col0, s, grx, gry, gc, vx, vy, qx, qy, b1x, b1y);

    // residual v - dq(q1), exact in fp32: the product d * 2^e is exact (a power-of-two
    // scaling of an E2M1 value, at worst a subnormal well above 2^-149), so the fused
    // v + d * (-2^e) rounds once, to the exact difference
    const float2 npx = make_float2(-pow2_of_byte(b1x), -pow2_of_byte(b1y));
    const uint32_t wx[4] = {qx.x, qx.y, qx.z, qx.w}, wy[4] = {qy.x, qy.y, qy.z, qy.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        residual_pair<0>(wx[j], wy[j], npx, v[8 * j], v[8 * j + 1]);
        residual_pair<1>(wx[j], wy[j], npx, v[8 * j + 2], v[8 * j + 3]);
        residual_pair<2>(wx[j], wy[j], npx, v[8 * j + 4], v[8 * j + 5]);
        residual_pair<3>(wx[j], wy[j], npx, v[8 * j + 6], v[8 * j + 7]);
    }

    // second pass; alpha carried by the scale byte
    amax32x2<1>(v, ax, ay);
    const uint32_t b2x = scale_byte(ax, p.mode), b2y = scale_byte(ay, p.mode);
    quant32x2<1>(v, b2x, b2y, qx, qy);
    store_rows(q2, p, col0, s, grx, gry, gc, vx, vy, qx, qy, (uint32_t)max((int)b2x + alpha_log2, 0),
               (uint32_t)max((int)b2y + alpha_log2, 0));
}

// MBS byte from the macro-block amax A (fp32 bits): k = floor(256 (T - f) / f) with
// f = 1 + mant / 2^23; A zero or subnormal gives 0.
__device__ __forceinline__ uint32_t mbs_byte(float A) {
    const uint32_t bits = __float_as_uint(A);
    if (bits < 0x00800000u) return 0u;
    const uint64_t mant = bits & 0x7FFFFFu;
    const uint64_t num = mant <= 0x400000u ? 256ull * (0x400000u - mant) : 256ull * (0x1000000u - mant);
    return (uint32_t)(num / (0x800000u + mant));
}

template <int HAD>
__global__ void __launch_bounds__(FX_THREADS, 5) rq_mbs_kernel(const QuantParams p, uint8_t* mbs) {
    const int t = threadIdx.x;
    const int s = t & 3, pr = t >> 2;
    const int64_t row0 = (int64_t)blockIdx.y * FX_TR, col0 = (int64_t)blockIdx.x * FX_TC;
    const int64_t gc = col0 + 32 * s, grx = row0 + pr, gry = row0 + pr + 32;
    const bool vx = grx < p.R && gc < p.C, vy = gry < p.R && gc < p.C;
    float2 v[32];
    load_pairs(p, grx, gry, gc, vx, vy, v);
    rotate_normalised<HAD>(v);

    // macro-block amax: the four threads of a tile row are lanes 4*pr .. 4*pr + 3
    float ax, ay;
    amax32x2<1>(v, ax, ay);
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
        ax = fmaxf(ax, __shfl_xor_sync(0xffffffffu, ax, o));
        ay = fmaxf(ay, __shfl_xor_sync(0xffffffffu, ay, o));
    }
    const uint32_t kx = mbs_byte(ax), ky = mbs_byte(ay);
    const float2 mul = make_float2(1.0f + (float)kx * (1.0f / 256.0f), 1.0f + (float)ky * (1.0f / 256.0f));
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = f2_mul(v[i], mul);

    amax32x2<1>(v, ax, ay);
    const uint32_t bx = scale_byte(ax, p.mode), by = scale_byte(ay, p.mode);
    uint4 qx, qy;
    quant32x2<1>(v, bx, by, qx, qy);
    store_rows(p.row, p, col0, s, grx, gry, gc, vx, vy, qx, qy, bx, by);
    if (s == 0) {
        if (vx) mbs[grx * (p.C / 128) + col0 / 128] = (uint8_t)kx;
        if (vy) mbs[gry * (p.C / 128) + col0 / 128] = (uint8_t)ky;
    }
}

}  // namespace

cudaError_t launch_rotate_quantize_of(const QuantParams& p, const QuantOut& q2, int had, int alpha_log2,
                                      cudaStream_t s) {
    const dim3 grid((unsigned)((p.C + FX_TC - 1) / FX_TC), (unsigned)((p.R + FX_TR - 1) / FX_TR));
    switch (had) {
        case 0:
            rq_of_kernel<1><<<grid, FX_THREADS, 0, s>>>(p, q2, alpha_log2);
            break;
        case 16:
            rq_of_kernel<16><<<grid, FX_THREADS, 0, s>>>(p, q2, alpha_log2);
            break;
        case 32:
            rq_of_kernel<32><<<grid, FX_THREADS, 0, s>>>(p, q2, alpha_log2);
            break;
        default:
            return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_rotate_quantize_mbs(const QuantParams& p, uint8_t* mbs, int had, cudaStream_t s) {
    const dim3 grid((unsigned)((p.C + FX_TC - 1) / FX_TC), (unsigned)((p.R + FX_TR - 1) / FX_TR));
    switch (had) {
        case 0:
            rq_mbs_kernel<1><<<grid, FX_THREADS, 0, s>>>(p, mbs);
            break;
        case 16:
            rq_mbs_kernel<16><<<grid, FX_THREADS, 0, s>>>(p, mbs);
            break;
        case 32:
            rq_mbs_kernel<32><<<grid, FX_THREADS, 0, s>>>(p, mbs);
            break;
        default:
            return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace mx
