// peak.cu -- tensor-core peak probe: each CTA (one per SM) issues back-to-back
// tcgen05.mma instructions on operands resident in shared memory, with nothing else
// in the loop, and the host converts the kernel time into TFLOP/s.  This measures the
// dense MMA rate that the GEMM's roofline refers to, for:
//   kind 0: kind::mxf4.block_scale.scale_vec::2X   (E2M1 x E2M1, UE8M0 per 32)
//   kind 1: kind::mxf4nvf4.block_scale.scale_vec::2X (same operands and scales)
//   kind 2: kind::f16 with bf16 operands (calibration against the bf16 peak)
//   kind 3: kind::mxf4nvf4.block_scale.scale_vec::4X with UE4M3 scales per 16 (NVFP4;
//           informational: UE4M3 cannot hold the E8M0 scale range, so the GEMM does
//           not use it)
//   kind 4: kind::mxf4 2X issued for a CTA pair (.cta_group::2, M = 256): each CTA
//           holds 128 rows of A and 128 of the 256 rows of B
// M = 128, N = 256, fp32 accumulation in TMEM.  The operand values are zeros; the
// rate does not depend on them.
#include "internal.h"
#include "ptx.cuh"

namespace mx {
namespace {

constexpr int P_N = 256;
constexpr int P_SMEM = 16384 + 32768 + 2048 + 1024 + 64;  // A, B, scales, alignment, barrier
// The pair kernel reserves more than half an SM's shared memory so that no SM ever holds
// two CTAs of it: two pairs that each held TMEM on one SM of the other's pair could wait
// on each other in the collective allocation.
constexpr int P_SMEM_PAIR = 120 * 1024;
static_assert(2 * P_SMEM_PAIR > 228 * 1024, "one pair CTA per SM");

__device__ __forceinline__ void mma_nvf4_2x(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                            uint32_t sfb, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
            d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb)
        : "memory");
}

__device__ __forceinline__ void mma_nvf4_4x(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                            uint32_t sfb, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
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
    // Unit scales: 0x7F is 2^0 in UE8M0, 0x38 is 1.0 in UE4M3.
    const uint32_t one = KIND == 3 ? 0x38383838u : 0x7F7F7F7Fu;
    for (int i = threadIdx.x; i < 2048 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(sSF)[i] = one;
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
        // Bit 23 selects the scale type: 1 = UE8M0, 0 = UE4M3.
        constexpr uint32_t id_fp4 = KIND == 3 ? (idesc_mxf4(128, P_N) & ~(1u << 23)) : idesc_mxf4(128, P_N);
        constexpr uint32_t id_bf16 = (1u << 4) | (1u << 7) | (1u << 10) | ((P_N >> 3) << 17) | ((128u >> 4) << 24);
        for (int64_t it = 0; it < iters; ++it) {
            const int k = (int)(it & 3);
            const uint64_t ad = smem_desc(a_base + k * 32, 16, 1024, kSwizzle128B);
            const uint64_t bd = smem_desc(b_base + k * 32, 16, 1024, kSwizzle128B);
            if (KIND == 0)
                tc_mma_mxf4(tmem, ad, bd, id_fp4, sfa_t, sfb_t, it != 0);
            else if (KIND == 1)
                mma_nvf4_2x(tmem, ad, bd, id_fp4, sfa_t, sfb_t, it != 0);
            else if (KIND == 3)
                mma_nvf4_4x(tmem, ad, bd, id_fp4, sfa_t, sfb_t, it != 0);
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

// CTA-pair version of kind 0: clusters of two CTAs, the even CTA issues M = 256 MMAs.
__global__ void __launch_bounds__(128, 1) peak_pair_kernel(int64_t iters, uint32_t* status, uint64_t wait_ns) {
    extern __shared__ uint8_t raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + 16384;
    uint8_t* sSF = smem + 16384 + 32768;
    uint64_t* done = reinterpret_cast<uint64_t*>(sSF + 2048);
    __shared__ uint32_t tmem_holder;
    const int warp = threadIdx.x >> 5;
    const uint32_t rank = cluster_ctarank();

    for (int i = threadIdx.x; i < (16384 + 32768) / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
    for (int i = threadIdx.x; i < 2048 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(sSF)[i] = 0x7F7F7F7Fu;
    if (threadIdx.x == 0) {
        mbar_init(done, 1);
        fence_mbar_init();
    }
    fence_async_smem();
    if (warp == 0) {
        tmem_alloc_pair(&tmem_holder, 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' operands and barriers are ready before the leader issues
    tc_fence_after();
    const uint32_t tmem = tmem_holder;

    if (rank == 0 && threadIdx.x == 0) {
        const uint32_t sfa_t = tmem + 256, sfb_t = tmem + 264;
        tc_cp_32x128b_warpx4_pair(sfa_t, smem_desc(smem_u32(sSF), 0, 128, kSwizzleNone));
        tc_cp_32x128b_warpx4_pair(sfb_t, smem_desc(smem_u32(sSF + 512), 0, 128, kSwizzleNone));
        tc_cp_32x128b_warpx4_pair(sfb_t + 4, smem_desc(smem_u32(sSF + 1024), 0, 128, kSwizzleNone));
        const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB);
        constexpr uint32_t id = idesc_mxf4(256, P_N);
        for (int64_t it = 0; it < iters; ++it) {
            const int k = (int)(it & 3);
            tc_mma_mxf4_pair(tmem, smem_desc(a_base + k * 32, 16, 1024, kSwizzle128B),
                             smem_desc(b_base + k * 32, 16, 1024, kSwizzle128B), id, sfa_t, sfb_t, it != 0);
        }
        tc_commit_pair(done, 0x3);
    }
    if (threadIdx.x == 0) wait_bounded(done, 0, wait_ns, status);
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // neither CTA frees TMEM while the pair's MMAs may still run
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, 512);
    }
}

cudaError_t run_peak_pair(int64_t iters, int sms, float* ms, uint32_t* status, uint64_t wait_ns) {
    cudaError_t e = cudaFuncSetAttribute(peak_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM_PAIR);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(sms & ~1));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = P_SMEM_PAIR;
    cfg.stream = 0;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaEvent_t a, b;
    cudaEventCreate(&a);
    cudaEventCreate(&b);
    e = cudaLaunchKernelEx(&cfg, peak_pair_kernel, (int64_t)8, status, wait_ns);  // warm-up
    if (e == cudaSuccess) {
        cudaEventRecord(a);
        e = cudaLaunchKernelEx(&cfg, peak_pair_kernel, iters, status, wait_ns);
        cudaEventRecord(b);
    }
    if (e == cudaSuccess) e = cudaEventSynchronize(b);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e == cudaSuccess) cudaEventElapsedTime(ms, a, b);
    cudaEventDestroy(a);
    cudaEventDestroy(b);
    return e;
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

// Returns the kernel time in ms for `iters` M=128-equivalent MMAs on each of *ctas
// CTAs, one per SM (synchronous).
cudaError_t run_mma_peak_probe(int kind, int64_t iters, float* ms, int* ctas, uint32_t* status, uint64_t wait_ns) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    *ctas = kind == 4 ? (sms & ~1) : sms;
    switch (kind) {
        case 4:
            return run_peak_pair(iters, sms, ms, status, wait_ns);
        case 0:
            return run_peak<0>(iters, sms, ms, status, wait_ns);
        case 1:
            return run_peak<1>(iters, sms, ms, status, wait_ns);
        case 2:
            return run_peak<2>(iters, sms, ms, status, wait_ns);
        case 3:
            return run_peak<3>(iters, sms, ms, status, wait_ns);
    }
    return cudaErrorInvalidValue;
}

}  // namespace mx
