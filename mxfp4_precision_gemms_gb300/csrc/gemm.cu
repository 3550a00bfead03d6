// gemm.cu -- block-scaled MXFP4 GEMM C = A . B^T on the sm_103a tcgen05 tensor cores.
//
// QDQ numerics ("Decomposing MXFP4 quantization error ...", experiments): E2M1
// elements, one E8M0 scale per 32 elements of K on both operands, FP32 accumulation.
// The operands are the quantised copies of "Pretraining Large Language Models with
// MXFP4 on Native FP4 Hardware" (C.1-C.3), already rotated along K.
//
// Two kernels.  The CTA-pair kernel (below the single-CTA one) runs whenever both M
// and N exceed 128; the single-CTA kernel covers narrow problems.
//
// Single-CTA structure (persistent: one CTA per SM walks 128 x BN tiles, 320 threads):
//   warp 0  TMA producer: 128x128-byte code tiles of A and B (128B swizzle) and the
//           matching 1 KB scale-factor atoms, into a STAGES-deep shared-memory ring.
//   warp 1  allocates TMEM; one elected thread copies each stage's scale factors
//           SMEM->TMEM (tcgen05.cp) and issues 4 tcgen05.mma.kind::mxf4 (K = 64
//           each) per 256-element stage into an fp32 TMEM accumulator.
//   warps 2-9 epilogue: TMEM -> registers (tcgen05.ld) -> fp32/bf16 global stores;
//           the accumulator is handed back to the MMA warp as soon as it has been
//           read, so the next tile's MMAs overlap the stores.
// All waits are bounded; on expiry the status word records a timeout and the CTA
// drains what it issued and exits.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace mx {
namespace {

// 1: problems with M > 128 and N > 128 use the CTA-pair kernel (256 x 256 tiles).
#ifndef MXG_PAIR
#define MXG_PAIR 1
#endif
#ifndef MXG_PAIR_STAGES
#define MXG_PAIR_STAGES 6
#endif

// Tuning knob (compile-time): pipeline depth of the 256-wide tiles.
#ifndef MXG_STAGES_256
#define MXG_STAGES_256 4
#endif

constexpr int BM = 128;
constexpr int BK_BYTES = 128;  // 256 E2M1 elements per stage
constexpr int EPI_WARPS = 8;  // two per TMEM lane quadrant, each owning half the columns
constexpr int GEMM_THREADS = 64 + 32 * EPI_WARPS;
constexpr int STG_PITCH = 64;                      // 32 rows x 64 B, 64-byte swizzle (TMA store box)
constexpr int STG_ALIGN = 1024;
constexpr int STG_WARP_BYTES = 32 * STG_PITCH;     // one warp's staging: 32 rows x 64 B

template <int BN, int STAGES, int ACC>
struct GemmCfg {
    static constexpr int A_STAGE = BM * BK_BYTES;
    static constexpr int B_STAGE = BN * BK_BYTES;
    static constexpr int SFA_STAGE = 1024;  // 128 rows x 8 blocks
    static constexpr int SFB_STAGE = (BN / 128) * 1024;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_STAGE;
    static constexpr int OFF_SFA = OFF_B + STAGES * B_STAGE;
    static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_STAGE;
    static constexpr int OFF_BAR = OFF_SFB + STAGES * SFB_STAGE;
    static constexpr int OFF_TMEM = OFF_BAR + (2 * STAGES + 2 * ACC + 1) * 8;
    static constexpr int OFF_STG = (OFF_TMEM + 16 + STG_ALIGN - 1) / STG_ALIGN * STG_ALIGN;  // epilogue staging
    static constexpr int SMEM = OFF_STG + EPI_WARPS * STG_WARP_BYTES + 1024;  // + alignment slack
    static constexpr int TX_BYTES = A_STAGE + B_STAGE + SFA_STAGE + SFB_STAGE;
    static constexpr int SF_COLS = 8 + 8 * (BN / 128);  // TMEM columns of scales per stage
    static constexpr int ACC_COLS = ACC * BN;               // fp32 accumulators (one per buffered tile)
    static constexpr int TMEM_USED = ACC_COLS + STAGES * SF_COLS;
    static constexpr int TMEM_COLS = TMEM_USED <= 32 ? 32 : TMEM_USED <= 64 ? 64 : TMEM_USED <= 128 ? 128
                                   : TMEM_USED <= 256 ? 256 : 512;
    static_assert(TMEM_USED <= 512, "TMEM budget");
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
    static_assert(OFF_STG % 16 == 0 && STG_PITCH % 16 == 0, "staging rows are accessed as 16-byte vectors");
    static_assert(OFF_BAR % 8 == 0 && OFF_A % 1024 == 0 && OFF_B % 1024 == 0, "barrier / swizzle-atom alignment");
};

// Lane i writes its row's 64 bytes into a 32-row x 64-byte staging box (64-byte
// swizzle: 16-byte chunk j of row r at j ^ ((r >> 1) & 3), conflict-free).
__device__ __forceinline__ void stage_box(uint8_t* box, int lane, const uint32_t* w) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint4*>(box + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) =
            make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
}

// One staged box to C with TMA (add-reduce for accumulate), skipped outside C.
__device__ __forceinline__ void issue_box(const GemmParams& p, const uint8_t* box, int64_t row_base, int64_t col0) {
    if (row_base < p.M && col0 < p.N) {
        if (p.accumulate)
            tma_reduce_add_2d(&p.map_c, box, (int32_t)col0, (int32_t)row_base);
        else
            tma_store_2d(&p.map_c, box, (int32_t)col0, (int32_t)row_base);
    }
}

// TMA-store epilogue through the warp's one staging box, which is reused only after
// the previous store has read it.
__device__ __forceinline__ void tma_store_block(const GemmParams& p, uint8_t* stg, int lane, int64_t row_base,
                                               int64_t col0, const uint32_t* w) {
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
    stage_box(stg, lane, w);
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
        issue_box(p, stg, row_base, col0);
        bulk_commit();
    }
}

// The warp's whole 32-row slice of its last tile (four 32-column chunks) staged at once
// in `area` (8 KB bf16, 16 KB fp32; boxes 2 KB apart), then stored with back-to-back TMA
// stores: the tile that ends the kernel does not wait on one box at a time.
__device__ __forceinline__ void store_slice_at_once(const GemmParams& p, uint8_t* area, int lane, int64_t row_base,
                                                   int64_t c0, const uint32_t (&v)[4][32]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        if (p.out_bf16) {
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const __nv_bfloat162 h =
                    __floats2bfloat162_rn(__uint_as_float(v[c][2 * j]), __uint_as_float(v[c][2 * j + 1]));
                w[j] = *reinterpret_cast<const uint32_t*>(&h);
            }
            stage_box(area + c * STG_WARP_BYTES, lane, w);
        } else {
            stage_box(area + (2 * c) * STG_WARP_BYTES, lane, v[c]);
            stage_box(area + (2 * c + 1) * STG_WARP_BYTES, lane, v[c] + 16);
        }
    }
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            if (p.out_bf16) {
                issue_box(p, area + c * STG_WARP_BYTES, row_base, c0 + c * 32);
            } else {
                issue_box(p, area + (2 * c) * STG_WARP_BYTES, row_base, c0 + c * 32);
                issue_box(p, area + (2 * c + 1) * STG_WARP_BYTES, row_base, c0 + c * 32 + 16);
            }
        }
        bulk_commit();
    }
}

__device__ __forceinline__ void store_chunk_tma(const GemmParams& p, uint8_t* stg, int lane, int64_t row_base,
                                               int64_t col0, const uint32_t (&v)[32]) {
    if (p.out_bf16) {
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
            w[j] = *reinterpret_cast<const uint32_t*>(&h);
        }
        tma_store_block(p, stg, lane, row_base, col0, w);
    } else {
        tma_store_block(p, stg, lane, row_base, col0, v);
        tma_store_block(p, stg, lane, row_base, col0 + 16, v + 16);
    }
}

template <int BN, int STAGES, int ACC>
__global__ void __launch_bounds__(GEMM_THREADS, 1) mxf4_gemm_kernel(const __grid_constant__ GemmParams p) {
    using Cfg = GemmCfg<BN, STAGES, ACC>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem + Cfg::OFF_A;
    uint8_t* sB = smem + Cfg::OFF_B;
    uint8_t* sSFA = smem + Cfg::OFF_SFA;
    uint8_t* sSFB = smem + Cfg::OFF_SFB;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
    uint64_t* empty = full + STAGES;
    uint64_t* acc_full = empty + STAGES;   // [ACC] MMA -> epilogue: accumulator holds a finished tile
    uint64_t* acc_empty = acc_full + ACC;  // [ACC] epilogue -> MMA: accumulator has been read out
    uint64_t* mma_done = acc_empty + ACC;  // every MMA issued by this CTA has completed
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_TMEM);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int num_k = (int)((p.K + 255) / 256);
    const int64_t num_n = (p.N + BN - 1) / BN;
    const int64_t num_tiles = ((p.M + BM - 1) / BM) * num_n;
    const int64_t atoms_per_row_block = p.kb_pad / 4;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < ACC; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], EPI_WARPS);  // one arrive per epilogue warp
        }
        mbar_init(mma_done, 1);
        fence_mbar_init();
        prefetch_tmap(&p.map_a);
        prefetch_tmap(&p.map_b);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, Cfg::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
#if MXF_PDL_GEMM
    // The set-up above touches no global memory, so it overlaps the previous kernel.
    grid_dependency_wait();
    allow_dependent_launch();
#endif

    if (warp == 0) {
        // ---------------- TMA producer
        if (elect_one()) {
            uint32_t armed[STAGES];  // number of phases armed per stage
#pragma unroll
            for (int s = 0; s < STAGES; ++s) armed[s] = 0;
            uint32_t it = 0;
            bool ok = true;
            for (int64_t tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                const int64_t m0 = (tile / num_n) * BM, n0 = (tile % num_n) * BN;
                for (int kt = 0; kt < num_k; ++kt, ++it) {
                    const int s = (int)(it % STAGES);
                    const uint32_t ph = (it / STAGES) & 1u;
                    if (it >= STAGES && !wait_bounded(&empty[s], ph ^ 1u, p.wait_ns, p.status)) {
                        ok = false;
                        break;
                    }
                    if (it == 0 && p.test_drop_first_stage) continue;  // fault injection: never arrives
                    mbar_arrive_expect_tx(&full[s], Cfg::TX_BYTES);
                    tma_load_2d(sA + s * Cfg::A_STAGE, &p.map_a, &full[s], kt * BK_BYTES, (int32_t)m0);
#pragma unroll
                    for (int j = 0; j < BN / 128; ++j)  // the tensor map's box is 128 rows
                        tma_load_2d(sB + s * Cfg::B_STAGE + j * (128 * BK_BYTES), &p.map_b, &full[s], kt * BK_BYTES,
                                    (int32_t)(n0 + j * 128));
                    bulk_load(sSFA + s * Cfg::SFA_STAGE, p.sfa + ((m0 / 128) * atoms_per_row_block + 2 * kt) * 512,
                              1024, &full[s]);
#pragma unroll
                    for (int j = 0; j < BN / 128; ++j)
                        bulk_load(sSFB + s * Cfg::SFB_STAGE + j * 1024,
                                  p.sfb + ((n0 / 128 + j) * atoms_per_row_block + 2 * kt) * 512, 1024, &full[s]);
                    armed[s] = it / STAGES + 1u;
                }
            }
            // Drain: the last armed phase of every stage has landed before the CTA exits.
#pragma unroll
            for (int s = 0; s < STAGES; ++s)
                if (armed[s]) wait_bounded(&full[s], (armed[s] - 1u) & 1u, p.wait_ns, p.status);
        }
    } else if (warp == 1) {
        // ---------------- tensor-core issuer
        if (elect_one()) {
            constexpr uint32_t idesc = idesc_mxf4(BM, BN);
            constexpr uint32_t SFB_KSTRIDE = 4 * (BN / 128);  // TMEM columns per 4-block group of B scales
            uint32_t it = 0, tcount = 0;
            bool ok = true;
            for (int64_t tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x, ++tcount) {
                const uint32_t ab = tcount % ACC;                 // accumulator buffer of this tile
                const uint32_t acc_t = tmem_base + ab * BN;
                if (tcount >= ACC) {
                    if (!wait_bounded(&acc_empty[ab], (tcount / ACC - 1u) & 1u, p.wait_ns, p.status)) break;
                    tc_fence_after();
                }
                for (int kt = 0; kt < num_k; ++kt, ++it) {
                    const int s = (int)(it % STAGES);
                    const uint32_t ph = (it / STAGES) & 1u;
                    if (!wait_bounded(&full[s], ph, p.wait_ns, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sfa_t = tmem_base + Cfg::ACC_COLS + s * Cfg::SF_COLS;
                    const uint32_t sfb_t = sfa_t + 8;
#pragma unroll
                    for (int a = 0; a < 2; ++a)
                        tc_cp_32x128b_warpx4(
                            sfa_t + a * 4,
                            smem_desc(smem_u32(sSFA + s * Cfg::SFA_STAGE + a * 512), 0, 128, kSwizzleNone));
#pragma unroll
                    for (int j = 0; j < BN / 128; ++j)
#pragma unroll
                        for (int a = 0; a < 2; ++a)
                            tc_cp_32x128b_warpx4(sfb_t + a * SFB_KSTRIDE + j * 4,
                                                 smem_desc(smem_u32(sSFB + s * Cfg::SFB_STAGE + j * 1024 + a * 512),
                                                           0, 128, kSwizzleNone));
                    const uint32_t a_base = smem_u32(sA + s * Cfg::A_STAGE);
                    const uint32_t b_base = smem_u32(sB + s * Cfg::B_STAGE);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint64_t adesc = smem_desc(a_base + k * 32, 16, 1024, kSwizzle128B);
                        const uint64_t bdesc = smem_desc(b_base + k * 32, 16, 1024, kSwizzle128B);
                        const uint32_t sf_id = (uint32_t)(k & 1) * 2u;
                        tc_mma_mxf4(acc_t, adesc, bdesc, idesc_with_sf_ids(idesc, sf_id, sf_id),
                                    sfa_t + (k >> 1) * 4, sfb_t + (k >> 1) * SFB_KSTRIDE, (kt | k) != 0);
                    }
                    tc_commit(&empty[s]);
                }
                if (ok) tc_commit(&acc_full[ab]);
            }
            // Every MMA issued here has completed before TMEM is released.
            tc_commit(mma_done);
            wait_bounded(mma_done, 0, p.wait_ns, p.status);
        }
    } else {
        // ---------------- epilogue: warp w may only read TMEM lanes 32*(w%4) .. +31; the
        // two warps of each lane quadrant split the columns in halves.  Each thread
        // pulls its whole slice out of TMEM (one wait), hands the accumulator back to
        // the MMA warp, and only then stores, so the stores overlap the next tile.
        const int q = warp & 3;
        const int h = (warp - 2) >> 2;
        uint8_t* stg = smem + Cfg::OFF_STG + (warp - 2) * STG_WARP_BYTES;
        constexpr int CH = BN / 2 / 32;  // 32-column chunks per thread
        uint32_t tcount = 0;
        for (int64_t tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++tcount) {
            const uint32_t ab = tcount % ACC;
            if (!wait_bounded(&acc_full[ab], (tcount / ACC) & 1u, p.wait_ns, p.status)) break;
            tc_fence_after();
            const int64_t row_base = (tile / num_n) * BM + q * 32;
            const int64_t c0 = (tile % num_n) * BN + h * (BN / 2);
            uint32_t v[CH][32];
#pragma unroll
            for (int c = 0; c < CH; ++c)
                tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(q * 32) << 16) + ab * BN + (uint32_t)(h * (BN / 2) + c * 32),
                                   v[c]);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[ab]);
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                store_chunk_tma(p, stg, lane, row_base, c0 + c * 32, v[c]);
            }
        }
        if (lane == 0) bulk_wait_all();  // every TMA store of this warp has completed
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}


// ---------------------------------------------------------------------------------
// CTA-pair kernel.  A cluster of two CTAs (on two SMs) computes 256 x 256 output tiles
// with M = 256 tcgen05.mma.cta_group::2 instructions.  CTA r (r = 0, 1) stages rows
// m0 + 128r .. +127 of A and rows n0 + 128r .. +127 of B, and its TMEM receives its
// 128 rows of the tile.  Each CTA thus loads 256 operand rows per K stage for a
// 128 x 256 share of the output, where a single-CTA 128 x 256 tile loads 384: a third
// less L2 -> SMEM traffic and shared-memory bandwidth per FLOP.
//   warp 0 (both CTAs)  TMA producer for the CTA's halves, plus the scale factors
//           its tensor core needs (its 128 rows of A, all 256 rows of B).  Completion
//           is counted on the leader's (CTA 0's) full barrier, which the leader arms
//           with the pair's bytes.
//   warp 1  allocates the pair's TMEM together with the other CTA; in the leader one
//           thread copies scale factors (tcgen05.cp.cta_group::2, each CTA's shared
//           memory -> its own TMEM) and issues the pair's MMAs; its commits arrive on
//           the barriers of both CTAs (stage free, accumulator full, all done).
//   warps 2-9 (both CTAs)  epilogue of the CTA's 128 rows; each warp reports the
//           accumulator read out to the leader's acc_empty barrier.
// One CTA per SM (shared memory > half the SM's): two pairs never compete for the
// TMEM of one SM, so the collective TMEM allocation cannot wait on another pair.
template <int STAGES>
struct PairCfg {
    static constexpr int A_STAGE = 128 * BK_BYTES;
    static constexpr int B_STAGE = 128 * BK_BYTES;
    static constexpr int SFA_STAGE = 1024;  // this CTA's 128 rows x 8 blocks
    static constexpr int SFB_STAGE = 2048;  // all 256 B rows x 8 blocks
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_STAGE;
    static constexpr int OFF_SFA = OFF_B + STAGES * B_STAGE;
    static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_STAGE;
    static constexpr int OFF_BAR = OFF_SFB + STAGES * SFB_STAGE;
    static constexpr int OFF_TMEM = OFF_BAR + (2 * STAGES + 3) * 8;
    // The 64-byte-swizzled staging tiles repeat every 512 bytes.  No alignment slack:
    // the kernel checks that dynamic shared memory starts on a 1024-byte boundary.
    static constexpr int PAIR_STG_ALIGN = 512;
    static constexpr int OFF_STG = (OFF_TMEM + 16 + PAIR_STG_ALIGN - 1) / PAIR_STG_ALIGN * PAIR_STG_ALIGN;
    static constexpr int SMEM = OFF_STG + EPI_WARPS * STG_WARP_BYTES;
    static constexpr uint32_t TX_PAIR = 2 * (A_STAGE + B_STAGE + SFA_STAGE + SFB_STAGE);
    static constexpr int SF_COLS = 24;  // TMEM columns of scales per stage: 8 for A, 16 for B
    static constexpr int TMEM_USED = 256 + STAGES * SF_COLS;
    static constexpr int TMEM_COLS = 512;
    static_assert(TMEM_USED <= TMEM_COLS, "TMEM budget");
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
    static_assert(2 * SMEM > 228 * 1024, "one CTA per SM");
    static_assert(OFF_BAR % 8 == 0 && OFF_B % 1024 == 0 && OFF_SFA % 1024 == 0 && OFF_STG % 16 == 0, "alignment");
    static_assert(EPI_WARPS * 8 * STG_WARP_BYTES <= OFF_SFA, "the last tile's slices fit in the A and B stages");
};

// The problem that global tile `tile` of a group belongs to, and the tile's index within
// that problem (tiles are numbered problem after problem; pair_tile_origin places them).
__device__ __forceinline__ int group_problem(const GemmGroup& g, int64_t tile, int64_t& local) {
    int pi = 0;
#pragma unroll
    for (int i = 1; i < kMaxGemmGroup; ++i)
        if (i < g.count && tile >= g.tile_start[i]) pi = i;
    local = tile - g.tile_start[pi];
    return pi;
}

// Origin (m0, n0) of tile lt of problem p's 256 x 256 tiling.  Consecutive tiles --
// which run at the same time on neighbouring clusters -- walk the dimension with fewer
// tiles fastest: the operand along it is then read by every wave and stays in L2, while
// the other operand streams through once.  (Measured on the down-projection Wgrad,
// 4096 x 14336 x 8192 with fp32 output: walking N fastest re-read the 62 MB B operand
// from DRAM in every wave, the fp32 output evicting it from L2; walking M fastest ran
// 8% faster.  The other Llama-shaped GEMMs were unchanged.)
__device__ __forceinline__ void pair_tile_origin(const GemmParams& p, int64_t lt, int64_t& m0, int64_t& n0) {
    const int64_t num_m = (p.M + 255) / 256, num_n = (p.N + 255) / 256;
    if (num_n > num_m) {
        m0 = (lt % num_m) * 256;
        n0 = (lt / num_m) * 256;
    } else {
        m0 = (lt / num_n) * 256;
        n0 = (lt % num_n) * 256;
    }
}

template <int STAGES>
__global__ void __launch_bounds__(GEMM_THREADS, 1) mxf4_gemm_pair_kernel(const __grid_constant__ GemmGroup g) {
    using Cfg = PairCfg<STAGES>;
    extern __shared__ uint8_t smem_raw[];
    // The layout has no slack for aligning the 128-byte-swizzled operand tiles.  Both
    // CTAs see the same base, so both return here, before any cluster barrier.
    if (smem_u32(smem_raw) & 1023u) {
        if (threadIdx.x == 0) atomicOr(g.status, kStatusSmemLayout);
        return;
    }
    uint8_t* smem = smem_raw;
    uint8_t* sA = smem + Cfg::OFF_A;
    uint8_t* sB = smem + Cfg::OFF_B;
    uint8_t* sSFA = smem + Cfg::OFF_SFA;
    uint8_t* sSFB = smem + Cfg::OFF_SFB;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);  // used in the leader
    uint64_t* empty = full + STAGES;
    uint64_t* acc_full = empty + STAGES;
    uint64_t* acc_empty = acc_full + 1;  // used in the leader: both CTAs' epilogues arrive
    uint64_t* mma_done = acc_empty + 1;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_TMEM);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int64_t num_tiles = g.tile_start[g.count];
    const int64_t cluster = blockIdx.x >> 1, num_clusters = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 2 * EPI_WARPS);
        mbar_init(mma_done, 1);
        fence_mbar_init();
        for (int i = 0; i < g.count; ++i) {
            prefetch_tmap(&g.prob[i].map_a);
            prefetch_tmap(&g.prob[i].map_b);
            prefetch_tmap(&g.prob[i].map_sfa);
            prefetch_tmap(&g.prob[i].map_sfb);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_holder, Cfg::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers exist before either signals the other's
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
#if MXF_PDL_GEMM
    // The set-up above touches no global memory, so it overlaps the previous kernel.
    grid_dependency_wait();
    allow_dependent_launch();
#endif

    if (warp == 0) {
        // ---------------- TMA producer (both CTAs)
        if (elect_one()) {
            const uint32_t full_leader = mapa_shared(smem_u32(full), 0);
            uint32_t armed[STAGES];  // phases issued per stage
#pragma unroll
            for (int s = 0; s < STAGES; ++s) armed[s] = 0;
            uint32_t it = 0;
            bool ok = true;
            for (int64_t tile = cluster; ok && tile < num_tiles; tile += num_clusters) {
                int64_t lt;
                const GemmParams& p = g.prob[group_problem(g, tile, lt)];
                const int num_k = (int)((p.K + 255) / 256);
                const int64_t atoms_per_row_block = p.kb_pad / 4;
                int64_t m0, n0;
                pair_tile_origin(p, lt, m0, n0);
                const int32_t ya = (int32_t)(m0 + rank * 128), yb = (int32_t)(n0 + rank * 128);
                const int32_t sfa_y = (int32_t)((m0 / 128 + rank) * atoms_per_row_block * 4);
                const int32_t sfb_y0 = (int32_t)((n0 / 128) * atoms_per_row_block * 4);
                const int32_t sfb_y1 = (int32_t)((n0 / 128 + 1) * atoms_per_row_block * 4);
                for (int kt = 0; kt < num_k; ++kt, ++it) {
                    const int s = (int)(it % STAGES);
                    const uint32_t ph = (it / STAGES) & 1u;
                    if (it >= STAGES && !wait_bounded(&empty[s], ph ^ 1u, g.wait_ns, g.status)) {
                        ok = false;
                        break;
                    }
                    if (it == 0 && g.test_drop_first_stage && rank == 0) continue;  // fault injection
                    if (rank == 0) mbar_arrive_expect_tx(&full[s], Cfg::TX_PAIR);
                    const uint32_t bar = full_leader + (uint32_t)s * 8u;
                    tma_load_2d_pair(sA + s * Cfg::A_STAGE, &p.map_a, bar, kt * BK_BYTES, ya);
                    tma_load_2d_pair(sB + s * Cfg::B_STAGE, &p.map_b, bar, kt * BK_BYTES, yb);
                    tma_load_2d_pair(sSFA + s * Cfg::SFA_STAGE, &p.map_sfa, bar, 0, sfa_y + kt * 8);
                    tma_load_2d_pair(sSFB + s * Cfg::SFB_STAGE, &p.map_sfb, bar, 0, sfb_y0 + kt * 8);
                    tma_load_2d_pair(sSFB + s * Cfg::SFB_STAGE + 1024, &p.map_sfb, bar, 0, sfb_y1 + kt * 8);
                    armed[s] = it / STAGES + 1u;
                }
            }
            // Drain.  The leader waits until the last armed phase of every stage has
            // landed (its full barriers count both CTAs' bytes); both CTAs wait until
            // the MMAs have released every stage they were given, so no commit is
            // still on its way to this CTA's barriers when it exits.
#pragma unroll
            for (int s = 0; s < STAGES; ++s) {
                if (!armed[s]) continue;
                if (rank == 0) wait_bounded(&full[s], (armed[s] - 1u) & 1u, g.wait_ns, g.status);
                wait_bounded(&empty[s], (armed[s] - 1u) & 1u, g.wait_ns, g.status);
            }
        }
    } else if (warp == 1) {
        // ---------------- tensor-core issuer (leader CTA)
        if (elect_one()) {
            if (rank == 0) {
                constexpr uint32_t idesc = idesc_mxf4(256, 256);
                uint32_t it = 0, tcount = 0;
                bool ok = true;
                for (int64_t tile = cluster; ok && tile < num_tiles; tile += num_clusters, ++tcount) {
                    int64_t lt;
                    const int num_k = (int)((g.prob[group_problem(g, tile, lt)].K + 255) / 256);
                    for (int kt = 0; kt < num_k; ++kt, ++it) {
                        const int s = (int)(it % STAGES);
                        const uint32_t ph = (it / STAGES) & 1u;
                        if (!wait_bounded(&full[s], ph, g.wait_ns, g.status)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sfa_t = tmem_base + 256 + s * Cfg::SF_COLS;
                        const uint32_t sfb_t = sfa_t + 8;
#pragma unroll
                        for (int a = 0; a < 2; ++a)
                            tc_cp_32x128b_warpx4_pair(
                                sfa_t + a * 4,
                                smem_desc(smem_u32(sSFA + s * Cfg::SFA_STAGE + a * 512), 0, 128, kSwizzleNone));
#pragma unroll
                        for (int j = 0; j < 2; ++j)
#pragma unroll
                            for (int a = 0; a < 2; ++a)
                                tc_cp_32x128b_warpx4_pair(
                                    sfb_t + a * 8 + j * 4,
                                    smem_desc(smem_u32(sSFB + s * Cfg::SFB_STAGE + j * 1024 + a * 512), 0, 128,
                                              kSwizzleNone));
                        // The scale copies above go to their own TMEM columns, so the
                        // accumulator is waited for only now: the copies of a tile's first
                        // stage overlap the epilogue's read-out of the previous tile.
                        if (kt == 0 && tcount > 0) {
                            if (!wait_bounded(acc_empty, (tcount - 1u) & 1u, g.wait_ns, g.status)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                        }
                        const uint32_t a_base = smem_u32(sA + s * Cfg::A_STAGE);
                        const uint32_t b_base = smem_u32(sB + s * Cfg::B_STAGE);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint32_t sf_id = (uint32_t)(k & 1) * 2u;
                            tc_mma_mxf4_pair(tmem_base, smem_desc(a_base + k * 32, 16, 1024, kSwizzle128B),
                                             smem_desc(b_base + k * 32, 16, 1024, kSwizzle128B),
                                             idesc_with_sf_ids(idesc, sf_id, sf_id), sfa_t + (k >> 1) * 4,
                                             sfb_t + (k >> 1) * 8, (kt | k) != 0);
                        }
                        tc_commit_pair(&empty[s], 0x3);
                    }
                    if (ok) tc_commit_pair(acc_full, 0x3);
                }
                tc_commit_pair(mma_done, 0x3);
            }
            // Both CTAs: every MMA of the pair has completed (and this CTA's mma_done
            // arrival has landed) before TMEM is released.
            wait_bounded(mma_done, 0, g.wait_ns, g.status);
        }
    } else {
        // ---------------- epilogue (both CTAs): the CTA's 128 rows of the tile
        const int q = warp & 3;
        const int h = (warp - 2) >> 2;
        uint8_t* stg = smem + Cfg::OFF_STG + (warp - 2) * STG_WARP_BYTES;
        const uint32_t acc_empty_leader = mapa_shared(smem_u32(acc_empty), 0);
        uint32_t tcount = 0;
        for (int64_t tile = cluster; tile < num_tiles; tile += num_clusters, ++tcount) {
            if (!wait_bounded(acc_full, tcount & 1u, g.wait_ns, g.status)) break;
            tc_fence_after();
            int64_t lt;
            const GemmParams& p = g.prob[group_problem(g, tile, lt)];
            int64_t m0, n0;
            pair_tile_origin(p, lt, m0, n0);
            const int64_t row_base = m0 + rank * 128 + q * 32;
            const int64_t c0 = n0 + h * 128;
            uint32_t v[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(h * 128 + c * 32), v[c]);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            // The TMEM reads above have completed (wait::ld); the arrive only reports it.
            if (lane == 0) mbar_arrive_cluster_relaxed(acc_empty_leader);
            if (tile + num_clusters >= num_tiles) {
                // This pair's last tile.  Its accumulator is full, so every MMA has
                // completed, and with it every read of the operand ring and every TMA load
                // into it: the ring is idle and takes the whole slice at once (16 KB per
                // warp, 128 KB for the eight warps, inside the ring's A and B stages).
                store_slice_at_once(p, smem + Cfg::OFF_A + (warp - 2) * 8 * STG_WARP_BYTES, lane, row_base, c0, v);
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    store_chunk_tma(p, stg, lane, row_base, c0 + c * 32, v[c]);
                }
            }
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // neither CTA frees TMEM or exits while the pair may still use it
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
    }
}

template <int BN, int STAGES, int ACC>
cudaError_t launch_cfg(const GemmParams& p, cudaStream_t s) {
    using Cfg = GemmCfg<BN, STAGES, ACC>;
    auto kern = mxf4_gemm_kernel<BN, STAGES, ACC>;
    static DeviceSlots sm_slots;
    int sm_count = 0;
    cudaError_t e = per_device_setting(sm_slots, &sm_count, [&](int dev, int* n) {
        cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
        return r != cudaSuccess ? r : cudaDeviceGetAttribute(n, cudaDevAttrMultiProcessorCount, dev);
    });
    if (e != cudaSuccess) return e;
    const int64_t tiles = ((p.M + BM - 1) / BM) * ((p.N + BN - 1) / BN);
    const unsigned grid = (unsigned)(tiles < sm_count ? tiles : sm_count);
    return launch_overlapped(kern, dim3(grid), dim3(GEMM_THREADS), Cfg::SMEM, s, 1, MXF_PDL_GEMM != 0, p);
}


// Returns cudaErrorNotSupported (nothing launched) when no cluster of two CTAs can be
// resident on this device, so the caller can fall back to the single-CTA kernel.
template <int STAGES>
cudaError_t launch_pair(const GemmGroup& g, cudaStream_t s) {
    using Cfg = PairCfg<STAGES>;
    auto kern = mxf4_gemm_pair_kernel<STAGES>;
    static DeviceSlots cluster_slots;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(GEMM_THREADS);
    cfg.dynamicSmemBytes = Cfg::SMEM;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int max_clusters = 0;
    cudaError_t e = per_device_setting(cluster_slots, &max_clusters, [&](int dev, int* n) {
        cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
        if (r != cudaSuccess) return r;
        int sms = 0;
        r = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (r != cudaSuccess) return r;
        cudaLaunchConfig_t probe = cfg;
        probe.gridDim = dim3((unsigned)(sms & ~1));
        return cudaOccupancyMaxActiveClusters(n, kern, &probe);
    });
    if (e != cudaSuccess) return e;
    if (max_clusters < 1) return cudaErrorNotSupported;
    const int64_t tiles = g.tile_start[g.count];
    const int64_t clusters = tiles < max_clusters ? tiles : max_clusters;
    return launch_overlapped(kern, dim3((unsigned)(2 * clusters)), dim3(GEMM_THREADS), Cfg::SMEM, s, 2,
                             MXF_PDL_GEMM != 0, g);
}

// A group of one, or several problems ordered by contraction length (longest first:
// the static round-robin schedule then ends on the shortest tiles).
GemmGroup make_group(const GemmParams* probs, int n) {
    GemmGroup g{};
    int order[kMaxGemmGroup];
    for (int i = 0; i < n; ++i) order[i] = i;
    for (int i = 1; i < n; ++i)  // stable insertion sort by K, descending
        for (int j = i; j > 0 && probs[order[j]].K > probs[order[j - 1]].K; --j) {
            const int t = order[j];
            order[j] = order[j - 1];
            order[j - 1] = t;
        }
    g.count = n;
    g.tile_start[0] = 0;
    for (int i = 0; i < n; ++i) {
        const GemmParams& p = probs[order[i]];
        g.prob[i] = p;
        g.tile_start[i + 1] = g.tile_start[i] + ((p.M + 255) / 256) * ((p.N + 255) / 256);
    }
    g.status = probs[0].status;
    g.wait_ns = probs[0].wait_ns;
    g.test_drop_first_stage = probs[0].test_drop_first_stage;
    return g;
}

}  // namespace

// Persistent launches.  M > 128 and N > 128: clusters of two CTAs walk 256 x 256
// tiles (as many clusters as fit at once).  Otherwise one CTA per SM walks 128 x BN
// tiles, BN = 256 unless the whole N fits in 128 columns.
cudaError_t launch_gemm(const GemmParams& p, cudaStream_t s) {
#if MXG_PAIR
    if (p.M > 128 && p.N > 128) {
        const cudaError_t e = launch_pair<MXG_PAIR_STAGES>(make_group(&p, 1), s);
        if (e != cudaErrorNotSupported) return e;
    }
#endif
    if (p.N <= 128) return launch_cfg<128, 6, 2>(p, s);
#ifdef MXG_FORCE_BN128
    return launch_cfg<128, 6, 2>(p, s);
#else
    return launch_cfg<256, MXG_STAGES_256, 1>(p, s);
#endif
}

// Several GEMMs in one persistent launch of the CTA-pair kernel (1 <= n <=
// kMaxGemmGroup); a group of one takes launch_gemm's kernel choice.
cudaError_t launch_gemm_group(const GemmParams* probs, int n, cudaStream_t s) {
    if (n < 1 || n > kMaxGemmGroup) return cudaErrorInvalidValue;
    if (n == 1) return launch_gemm(probs[0], s);
    const cudaError_t e = launch_pair<MXG_PAIR_STAGES>(make_group(probs, n), s);
    if (e != cudaErrorNotSupported) return e;
    for (int i = 0; i < n; ++i) {  // no pair cluster fits: one launch per problem
        const cudaError_t ei = launch_gemm(probs[i], s);
        if (ei != cudaSuccess) return ei;
    }
    return cudaSuccess;
}

}  // namespace mx
