// quant_random.cu -- the randomised quantiser baselines of "Pretraining Large Language
// Models with MXFP4 on Native FP4 Hardware" (A.2: random sign flips before the
// Hadamard; the stochastic-rounding ablation of table 1), row and transposed layouts.
// The random numbers are inputs:
//   col_signs / row_signs: bitmasks over the rotated dimension (bit i set: element i
//     negated before the rotation, H D x); flipping a bf16 sign is exact;
//   sr_row [R, C] / sr_colT [C, R]: one uniform 16-bit integer per output element; a
//     magnitude a in [lo, lo + step) rounds up iff r < ((a - lo) / step) * 65536, every
//     term exact in fp32; a >= 6 saturates; the sign is kept.
// Same tiling as rq_kernel (64 x 128 tiles, 128 threads, bf16 tile staged in shared
// memory for the column work, transposed rows exchanged within a warp).
//
// Or the kernel draws them itself (GEN) from Philox4x32-10 (Salmon, Moraes, Dror and
// Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC'11), a counter-based
// generator, with a fixed counter layout (so any element's numbers can be recomputed):
//   sign bit j of a dimension's vector: bit j % 32 of output word (j % 128) / 32 of
//     Philox(counter (j / 128, 0, 0, 0), key = the dimension's 64-bit seed);
//   stochastic-rounding integer of (line l, position i) of copy c (0 row, 1 transposed):
//     16-bit half i % 8 (word (i % 8) / 2, low half first) of
//     Philox(counter (i / 8, l, c, 0), key = the SR seed).
// A GEMM's two operands share their contraction's sign vector by sharing its seed.
#include "quant_math.cuh"

namespace mx {
namespace {

constexpr int RQ_TR = 64, RQ_TC = 128, RQ_THREADS = 128;

// Philox4x32-10: ten rounds of (c0, c1, c2, c3) -> (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2),
// hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)) with M0 = 0xD2511F53, M1 = 0xCD9E8D57, the key
// bumped by (0x9E3779B9, 0xBB67AE85) between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint32_t h0 = __umulhi(0xD2511F53u, c.x), l0 = 0xD2511F53u * c.x;
        const uint32_t h1 = __umulhi(0xCD9E8D57u, c.z), l1 = 0xCD9E8D57u * c.z;
        c = make_uint4(h1 ^ c.y ^ k0, l1, h0 ^ c.w ^ k1, l0);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

// 32 sign bits of a dimension's vector starting at index j0 (a multiple of 32).
__device__ __forceinline__ uint32_t philox_sign_word(uint64_t seed, int64_t j0) {
    const uint4 o = philox4x32_10(make_uint4((uint32_t)(j0 >> 7), 0u, 0u, 0u), (uint32_t)seed, (uint32_t)(seed >> 32));
    const int w = (int)((j0 >> 5) & 3);
    return w == 0 ? o.x : w == 1 ? o.y : w == 2 ? o.z : o.w;
}

// The 32 stochastic-rounding integers of positions i0 .. i0 + 31 (i0 a multiple of 8) of
// line `line` of copy `copy`, two per word, in the layout load_r produces.
__device__ __forceinline__ void philox_sr32(uint64_t seed, int64_t i0, int64_t line, uint32_t copy,
                                            uint32_t (&w)[16]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint4 o = philox4x32_10(make_uint4((uint32_t)((i0 >> 3) + j), (uint32_t)line, copy, 0u),
                                      (uint32_t)seed, (uint32_t)(seed >> 32));
        w[4 * j] = o.x;
        w[4 * j + 1] = o.y;
        w[4 * j + 2] = o.z;
        w[4 * j + 3] = o.w;
    }
}

// Stochastically rounded grid value of u with the 16-bit integer r.
__device__ __forceinline__ float sr_grid(float u, uint32_t r) {
    const float a = fabsf(u);
    float mag = 6.0f;
    if (a < 6.0f) {
        const float step = a < 2.0f ? 0.5f : (a < 4.0f ? 1.0f : 2.0f);
        const float inv = a < 2.0f ? 2.0f : (a < 4.0f ? 1.0f : 0.5f);
        const float lo = floorf(a * inv) * step;
        const float pf = (a - lo) * inv * 65536.0f;  // p * 65536, exact
        mag = (float)r < pf ? lo + step : lo;
    }
    return copysignf(mag, u);
}

// Codes of both vectors with stochastic rounding: u = v * 2^-e exactly as in quant32x2,
// then the grid value from the random integer (rx: 16 words, two integers each, for the
// x vector; ry for y), converted exactly by cvt (grid values are their own codes).
template <int HAD>
__device__ __forceinline__ void quant32x2_sr(const float2 (&v)[32], uint32_t bx, uint32_t by,
                                             const uint32_t (&rx)[16], const uint32_t (&ry)[16], uint4& qx,
                                             uint4& qy) {
    const float2 f = make_float2(unit_factor<HAD>(bx), unit_factor<HAD>(by));
    float gx[32], gy[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const float2 u = f2_mul(v[i], f);
        const uint32_t shift = 16u * (uint32_t)(i & 1);
        gx[i] = sr_grid(u.x, (rx[i >> 1] >> shift) & 0xFFFFu);
        gy[i] = sr_grid(u.y, (ry[i >> 1] >> shift) & 0xFFFFu);
    }
    uint32_t wx[4], wy[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        wx[j] = cvt_e2m1x8(gx + 8 * j);
        wy[j] = cvt_e2m1x8(gy + 8 * j);
    }
    qx = make_uint4(wx[0], wx[1], wx[2], wx[3]);
    qy = make_uint4(wy[0], wy[1], wy[2], wy[3]);
}

// 32 random integers (64 bytes) as 16 words; zeros when not valid.
__device__ __forceinline__ void load_r(const uint16_t* src, bool valid, uint32_t (&w)[16]) {
#pragma unroll
    for (int j = 0; j < 16; ++j) w[j] = 0;
    if (!valid) return;
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint4 q = __ldcs(s4 + j);
        w[4 * j] = q.x;
        w[4 * j + 1] = q.y;
        w[4 * j + 2] = q.z;
        w[4 * j + 3] = q.w;
    }
}

template <int HAD, bool ROW, bool COLT, bool SR, bool GEN>
__global__ void __launch_bounds__(RQ_THREADS, SR ? 4 : 6) rq_rand_kernel(const QuantParams p, const RandOpts o) {
    __shared__ __align__(16) uint32_t tile[COLT ? RQ_TR * RQ_TC / 2 : 4];
    const int t = threadIdx.x;
    const int64_t row0 = (int64_t)blockIdx.y * RQ_TR, col0 = (int64_t)blockIdx.x * RQ_TC;

    const int s = t & 3, pr = t >> 2;
    const int rx = pr, ry = pr + 32;
    const int64_t gc = col0 + 32 * s, grx = row0 + rx, gry = row0 + ry;
    const bool vx = grx < p.R && gc < p.C, vy = gry < p.R && gc < p.C;
    uint4 raw_x[4], raw_y[4];
    load_row_pair(p, grx, gry, gc, vx, vy, COLT && rows_32B_aligned(p), raw_x, raw_y);
    if constexpr (COLT) {  // the unflipped tile, for the column work
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            *reinterpret_cast<uint4*>(&tile[tile_chunk(rx, 4 * s + j)]) = raw_x[j];
            *reinterpret_cast<uint4*>(&tile[tile_chunk(ry, 4 * s + j)]) = raw_y[j];
        }
    }

    if constexpr (ROW) {
        uint32_t bits;
        if constexpr (GEN)
            bits = o.col_sign_on ? philox_sign_word(o.col_sign_seed, gc) : 0u;
        else
            bits = (o.col_signs && gc < p.C) ? *reinterpret_cast<const uint32_t*>(o.col_signs + gc / 8) : 0u;
        float2 v[32];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t a[4] = {raw_x[j].x, raw_x[j].y, raw_x[j].z, raw_x[j].w};
            const uint32_t b[4] = {raw_y[j].x, raw_y[j].y, raw_y[j].z, raw_y[j].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int e = 8 * j + 2 * i;  // element index of the word's low half
                const uint32_t m = (((bits >> e) & 1u) << 15) | (((bits >> (e + 1)) & 1u) << 31);
                const uint32_t aw = a[i] ^ m, bw = b[i] ^ m;
                v[e] = make_float2(__uint_as_float(aw << 16), __uint_as_float(bw << 16));
                v[e + 1] = make_float2(__uint_as_float(aw & 0xFFFF0000u), __uint_as_float(bw & 0xFFFF0000u));
            }
        }
        rotate32x2<HAD>(v);
        float ax, ay;
        amax32x2<HAD>(v, ax, ay);
        const uint32_t bytex = scale_byte(ax, p.mode), bytey = scale_byte(ay, p.mode);
        uint4 qx, qy;
        if constexpr (SR) {
            uint32_t r_x[16], r_y[16];
            if constexpr (GEN) {
                philox_sr32(o.sr_seed, gc, grx, 0u, r_x);
                philox_sr32(o.sr_seed, gc, gry, 0u, r_y);
            } else {
                load_r(o.sr_row + grx * p.C + gc, vx, r_x);
                load_r(o.sr_row + gry * p.C + gc, vy, r_y);
            }
            quant32x2_sr<HAD>(v, bytex, bytey, r_x, r_y, qx, qy);
        } else {
            quant32x2<HAD>(v, bytex, bytey, qx, qy);
        }
        if (vx) *reinterpret_cast<uint4*>(p.row.codes + grx * (p.C / 2) + gc / 2) = qx;
        if (vy) *reinterpret_cast<uint4*>(p.row.codes + gry * (p.C / 2) + gc / 2) = qy;
        store_row_scales(p.row, p, col0, s, grx, gry, vx, vy, bytex, bytey);
    }

    if constexpr (COLT) {
        __syncthreads();
        // Two adjacent columns x one 32-row block per thread; a warp holds both row blocks
        // of its 16 column pairs (lanes l and l ^ 16), as in rq_kernel.  Lanes past the
        // matrix compute on the tile's zeros and store nothing.
        const int lane = t & 31;
        const int rb = lane >> 4, cp = 16 * (t >> 5) + (lane & 15);
        const int64_t gcol = col0 + 2 * cp, grow = row0 + 32 * rb;
        const bool valid = gcol < p.C && grow < p.R;
        uint32_t bits;
        if constexpr (GEN)
            bits = o.row_sign_on ? philox_sign_word(o.row_sign_seed, grow) : 0u;
        else
            bits = (o.row_signs && valid) ? *reinterpret_cast<const uint32_t*>(o.row_signs + grow / 8) : 0u;
        float2 v[32];
        const int q = cp >> 2, wi = cp & 3;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const uint32_t m = ((bits >> i) & 1u) * 0x80008000u;  // the row's sign, both columns
            const uint32_t w = tile[tile_chunk(32 * rb + i, q) + wi] ^ m;
            v[i] = make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
        }
        rotate32x2<HAD>(v);
        float ax, ay;
        amax32x2<HAD>(v, ax, ay);
        const uint32_t bytex = scale_byte(ax, p.mode), bytey = scale_byte(ay, p.mode);
        uint4 qx, qy;
        if constexpr (SR) {
            uint32_t r_x[16], r_y[16];
            if constexpr (GEN) {
                philox_sr32(o.sr_seed, grow, gcol, 1u, r_x);
                philox_sr32(o.sr_seed, grow, gcol + 1, 1u, r_y);
            } else {
                load_r(o.sr_colT + gcol * p.R + grow, valid, r_x);
                load_r(o.sr_colT + (gcol + 1) * p.R + grow, valid, r_y);
            }
            quant32x2_sr<HAD>(v, bytex, bytey, r_x, r_y, qx, qy);
        } else {
            quant32x2<HAD>(v, bytex, bytey, qx, qy);
        }
        store_colT_pair(p.colT, p, row0, col0, cp, rb, qx, qy, bytex, bytey);
    }
}

template <int HAD, bool SR, bool GEN>
cudaError_t launch_layouts(const QuantParams& p, const RandOpts& o, unsigned layouts, cudaStream_t s) {
    const dim3 grid((unsigned)((p.C + RQ_TC - 1) / RQ_TC), (unsigned)((p.R + RQ_TR - 1) / RQ_TR));
    switch (layouts) {
        case MXFP4_LAYOUT_ROW:
            rq_rand_kernel<HAD, true, false, SR, GEN><<<grid, RQ_THREADS, 0, s>>>(p, o);
            break;
        case MXFP4_LAYOUT_COLT:
            rq_rand_kernel<HAD, false, true, SR, GEN><<<grid, RQ_THREADS, 0, s>>>(p, o);
            break;
        case MXFP4_LAYOUT_ROW | MXFP4_LAYOUT_COLT:
            rq_rand_kernel<HAD, true, true, SR, GEN><<<grid, RQ_THREADS, 0, s>>>(p, o);
            break;
        default:
            return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

template <int HAD>
cudaError_t launch_sr(const QuantParams& p, const RandOpts& o, unsigned layouts, cudaStream_t s) {
    if (o.gen)
        return o.sr_on ? launch_layouts<HAD, true, true>(p, o, layouts, s)
                       : launch_layouts<HAD, false, true>(p, o, layouts, s);
    const bool sr = (layouts & MXFP4_LAYOUT_ROW && o.sr_row) || (layouts & MXFP4_LAYOUT_COLT && o.sr_colT);
    return sr ? launch_layouts<HAD, true, false>(p, o, layouts, s) : launch_layouts<HAD, false, false>(p, o, layouts, s);
}

}  // namespace

cudaError_t launch_rotate_quantize_rand(const QuantParams& p, const RandOpts& o, int had, unsigned layouts,
                                        cudaStream_t s) {
    switch (had) {
        case 0:
            return launch_sr<1>(p, o, layouts, s);
        case 16:
            return launch_sr<16>(p, o, layouts, s);
        case 32:
            return launch_sr<32>(p, o, layouts, s);
        default:
            return cudaErrorInvalidValue;
    }
}

}  // namespace mx
