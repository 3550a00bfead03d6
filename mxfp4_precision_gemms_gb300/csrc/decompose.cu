// decompose.cu -- measurement kernel: the three components of the MXFP4 error of a
// row-quantised tensor ("Decomposing MXFP4 quantization error for LLM reinforcement
// learning", core insight and property 1).
//
// For every 32-element block of the rotated rows (same fp32 rotation and E8M0 scale
// as the quantiser), with s_b the E8M0 scale and s* = amax / 6 the ideal scale:
//   Q(x)  = s_b * grid(x / s_b),   Q*(x) = s* * grid(x / s*)
//   e_scale = Q - Q*;  e_DZ = Q* - x on the deadzone |x| < amax/24;  e_grid = Q* - x off it.
// The kernel accumulates sum e^2, sum e_scale^2, sum e_DZ^2, sum e_grid^2,
// sum e_scale * e_grid, the deadzone count and the element count in fp64.
// Diagnostic, not on the training path: each thread owns one block, fp64 atomics.
#include "internal.h"
#include "ptx.cuh"

namespace mx {
namespace {

// Nearest E2M1 grid value of a real u (fp64), ties to the even code, saturating at 6.
__device__ __forceinline__ double grid_round_f64(double u) {
    const double a = fabs(u);
    double m;
    if (a <= 0.25) m = 0.0;
    else if (a < 0.75) m = 0.5;
    else if (a <= 1.25) m = 1.0;
    else if (a < 1.75) m = 1.5;
    else if (a <= 2.5) m = 2.0;
    else if (a < 3.5) m = 3.0;
    else if (a <= 5.0) m = 4.0;
    else m = 6.0;
    return copysign(m, u);
}

template <int HAD>
__device__ __forceinline__ void rotate_block(float (&v)[32]) {
    if constexpr (HAD > 1) {
#pragma unroll
        for (int s = 1; s < HAD; s <<= 1)
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if ((i & s) == 0) {
                    const float a = v[i], b = v[i + s];
                    v[i] = __fadd_rn(a, b);
                    v[i + s] = __fsub_rn(a, b);
                }
        const float c = (HAD == 16) ? 0.25f : 0.17677669529663687f;
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __fmul_rn(v[i], c);
    }
}

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <int HAD>
__global__ void __launch_bounds__(256) decompose_kernel(const uint16_t* x, int64_t R, int64_t C, int64_t ld, int mode,
                                                       double* out) {
    const int64_t nblk = R * (C / 32);
    double acc[7] = {0, 0, 0, 0, 0, 0, 0};
    for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < nblk; b += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = b / (C / 32), c0 = (b % (C / 32)) * 32;
        float v[32];
        const uint4* src = reinterpret_cast<const uint4*>(x + r * ld + c0);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 w = src[j];
            const uint32_t a[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[8 * j + 2 * i] = __uint_as_float(a[i] << 16);
                v[8 * j + 2 * i + 1] = __uint_as_float(a[i] & 0xFFFF0000u);
            }
        }
        rotate_block<HAD>(v);
        float amax_f = 0.0f;
#pragma unroll
        for (int i = 0; i < 32; ++i) amax_f = fmaxf(amax_f, fabsf(v[i]));
        const uint32_t bits = __float_as_uint(amax_f);
        const int eb = (int)(bits >> 23);
        const int adj = (mode == 1 && (bits & 0x7FFFFFu) > 0x400000u) ? 1 : 2;
        const int e = max(eb - adj, 0) - 127;
        const double amax = (double)amax_f;
        const double sstar = amax / 6.0;
        const double dz_lim = amax / 24.0;
#pragma unroll 4
        for (int i = 0; i < 32; ++i) {
            const double xv = (double)v[i];
            const double q = ldexp(grid_round_f64(ldexp(xv, -e)), e);
            const double qs = sstar > 0.0 ? sstar * grid_round_f64(xv / sstar) : 0.0;
            const bool dz = fabs(xv) < dz_lim;
            const double es = q - qs, ed = dz ? qs - xv : 0.0, eg = dz ? 0.0 : qs - xv, et = q - xv;
            acc[0] += et * et;
            acc[1] += es * es;
            acc[2] += ed * ed;
            acc[3] += eg * eg;
            acc[4] += es * eg;
            acc[5] += dz ? 1.0 : 0.0;
            acc[6] += 1.0;
        }
    }
#pragma unroll
    for (int k = 0; k < 7; ++k) {
        const double s = warp_sum(acc[k]);
        if ((threadIdx.x & 31) == 0) atomicAdd(out + k, s);
    }
}

}  // namespace

cudaError_t launch_error_decomposition(const uint16_t* x, int64_t R, int64_t C, int64_t ld, int had, int mode,
                                       double* out, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(out, 0, 7 * sizeof(double), s);
    if (e != cudaSuccess) return e;
    if (R == 0 || C == 0) return cudaSuccess;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t nblk = R * (C / 32);
    const int64_t want = (nblk + 255) / 256;
    const unsigned grid = (unsigned)(want < 8 * sms ? want : 8 * sms);
    switch (had) {
        case 0:
            decompose_kernel<1><<<grid, 256, 0, s>>>(x, R, C, ld, mode, out);
            break;
        case 16:
            decompose_kernel<16><<<grid, 256, 0, s>>>(x, R, C, ld, mode, out);
            break;
        case 32:
            decompose_kernel<32><<<grid, 256, 0, s>>>(x, R, C, ld, mode, out);
            break;
        default:
            return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace mx
