// peak.cu -- tensor-core peak probe: each CTA (one per SM) issues back-to-back
// tcgen05.mma instructions on operands resident in shared memory, with nothing else
// in the loop, and the host converts the kernel time into TFLOP/s.  This measures the
// dense MMA rate that the GEMM's roofline refers to, for:
//   kind 0: kind::mxf4.block_scale.scale_vec::2X   (E2M1 x E2M1, UE8M0 per 32)
//   kind 1: kind::mxf4nvf4.block_scale.scale_vec::2X (same operands and scales)
//   kind 2: kind::f16 with bf16 operands (calibration against the bf16 peak)
// M = 128, N = 256, fp32 accumulation in TMEM.  The operand values are zeros; the
// rate does not depend on them.
#include "internal.h"
#include "ptx.cuh"

namespace mx {
namespace {

constexpr int P_N = 256;
constexpr int P_SMEM = 16384 + 32768 + 2048 + 1024 + 64;  // A, B, scales, alignment, barrier

__device__ __forceinline__ void mma_nvf4_2x(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                            uint32_t sfb, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
            d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb)
        : "memory");
}

__device__ __forceinline__ void mma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

template <int KIND>
__global__ void __launch_bounds__(128, 1) peak_kernel(int64_t iters, uint32_t* status, uint64_t wait_ns) {
    extern __shared__ uint8_t raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + 16384;
    uint8_t* sSF = smem + 16384 + 32768;
    uint64_t* done = reinterpret_cast<uint64_t*>(sSF + 2048);
    __shared__ uint32_t tmem_holder;
    const int warp = threadIdx.x >> 5;

    for (int i = threadIdx.x; i < (16384 + 32768) / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
    for (int i = threadIdx.x; i < 2048 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(sSF)[i] = 0x7F7F7F7Fu;
    if (threadIdx.x == 0) {
        mbar_init(done, 1);
        fence_mbar_init();
    }
    fence_async_smem();
    if (warp == 0) {
        tmem_alloc(&tmem_holder, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_holder;

    if (threadIdx.x == 0) {
        const uint32_t sfa_t = tmem + 256, sfb_t = tmem + 264;
        if (KIND != 2) {
            tc_cp_32x128b_warpx4(sfa_t, smem_desc(smem_u32(sSF), 0, 128, kSwizzleNone));
            tc_cp_32x128b_warpx4(sfb_t, smem_desc(smem_u32(sSF + 512), 0, 128, kSwizzleNone));
            tc_cp_32x128b_warpx4(sfb_t + 4, smem_desc(smem_u32(sSF + 1024), 0, 128, kSwizzleNone));
        }
        const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB);
        constexpr uint32_t id_fp4 = idesc_mxf4(128, P_N);
        constexpr uint32_t id_bf16 = (1u << 4) | (1u << 7) | (1u << 10) | ((P_N >> 3) << 17) | ((128u >> 4) << 24);
        for (int64_t it = 0; it < iters; ++it) {
            const int k = (int)(it & 3);
            const uint64_t ad = smem_desc(a_base + k * 32, 16, 1024, kSwizzle128B);
            const uint64_t bd = smem_desc(b_base + k * 32, 16, 1024, kSwizzle128B);
            if (KIND == 0)
                tc_mma_mxf4(tmem, ad, bd, id_fp4, sfa_t, sfb_t, it != 0);
            else if (KIND == 1)
                mma_nvf4_2x(tmem, ad, bd, id_fp4, sfa_t, sfb_t, it != 0);
            else
                mma_bf16(tmem, ad, bd, id_bf16, it != 0);
        }
        tc_commit(done);
        wait_bounded(done, 0, wait_ns, status);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int KIND>
cudaError_t run_peak(int64_t iters, int sms, float* ms, uint32_t* status, uint64_t wait_ns) {
    auto kern = peak_kernel<KIND>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM);
    if (e != cudaSuccess) return e;
    cudaEvent_t a, b;
    cudaEventCreate(&a);
    cudaEventCreate(&b);
    kern<<<sms, 128, P_SMEM>>>(8, status, wait_ns);  // warm-up
    cudaEventRecord(a);
    kern<<<sms, 128, P_SMEM>>>(iters, status, wait_ns);
    cudaEventRecord(b);
    e = cudaEventSynchronize(b);
    if (e == cudaSuccess) e = cudaGetLastError();
    cudaEventElapsedTime(ms, a, b);
    cudaEventDestroy(a);
    cudaEventDestroy(b);
    return e;
}

}  // namespace

// Returns the kernel time in ms for `iters` MMAs on every SM (synchronous).
cudaError_t run_mma_peak_probe(int kind, int64_t iters, float* ms, uint32_t* status, uint64_t wait_ns) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    switch (kind) {
        case 0:
            return run_peak<0>(iters, sms, ms, status, wait_ns);
        case 1:
            return run_peak<1>(iters, sms, ms, status, wait_ns);
        case 2:
            return run_peak<2>(iters, sms, ms, status, wait_ns);
    }
    return cudaErrorInvalidValue;
}

}  // namespace mx
