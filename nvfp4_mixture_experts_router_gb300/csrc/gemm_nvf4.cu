// Grouped NVFP4 x NVFP4 GEMMs of the MoE layer on the 5th-generation tensor
// cores (tcgen05.mma kind::mxf4nvf4, block-scaled with UE4M3 scales per 16
// elements), with the FC1 and FC2 epilogues fused in.
//
//   D[row, n] = sum_k A[row, k] * B_e[n, k]       (rows of expert e only)
//
// A (activations) are the permuted route rows, B the expert's prepared
// weights; each expert segment of A is padded to whole 128-row tiles
// [FlashInfer PR #4366, "Tests": padding and partial tiles], so every M tile
// belongs to exactly one expert (tile_expert).
//
// Kernel design (one persistent CTA per SM, 224 threads):
//   warp 0      TMA producer: per pipeline stage one 128x128-byte A tile and
//               one 128x128-byte B tile (cp.async.bulk.tensor, 128-byte
//               swizzle) plus the matching 2 KB of scale atoms of each
//               operand (cp.async.bulk), all completing on one mbarrier.
//   warp 6      scale mover: once a stage has landed, tcgen05.cp of its 8
//               scale atoms into the stage's tensor-memory slot, then
//               tcgen05.commit to the stage's sf_ready barrier.
//   warp 1      allocates 512 tensor-memory columns; lane 0 issues, per
//               stage, four 128x128x64 block-scaled MMAs into an FP32
//               accumulator in tensor memory, then tcgen05.commit frees the
//               stage.  (The tcgen05 issue slot of a single thread is the
//               scarce resource at these tile sizes, so the scale copies are
//               issued from another warp.)
//   warps 2-5   epilogue: tcgen05.ld of the accumulator (warp w reads lanes
//               32*(w%4)..+31, one output row per thread), fused activation /
//               scaling / requantization / scatter, then release the buffer.
// Two accumulator buffers let the epilogue of tile i overlap the main loop
// of tile i+1.  Tiles are walked n-fastest so that concurrently running CTAs
// share the A tile and one expert's weights stay hot in L2.
// Every wait is bounded (1 s); a timeout sets a status bit and all roles
// drain and exit instead of hanging.
#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kBKBytes = 128;                 // 256 E2M1 elements per stage row
constexpr int kStages = 6;
constexpr int kTileBytesA = kBM * kBKBytes;   // 16 KB
constexpr int kTileBytesB = kBN * kBKBytes;   // 16 KB
constexpr int kSfBytes = 4 * 512;             // 4 scale atoms (128 rows x 64 elems each)
constexpr int kNumThreads = 224;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = 128;
constexpr uint32_t kSfColBase = 256;          // columns 256.. hold the per-stage scales
constexpr uint32_t kSfColsPerStage = 32;      // 16 (A) + 16 (B)
constexpr int kSmemBytes = kStages * (kTileBytesA + kTileBytesB + 2 * kSfBytes) + 1024 + 256;

static_assert(kSfColBase + kStages * kSfColsPerStage <= kTmemCols, "tensor memory budget");
static_assert(2 * kAccCols <= kSfColBase, "accumulators overlap scales");

struct Smem {
    uint8_t* a;
    uint8_t* b;
    uint8_t* sfa;
    uint8_t* sfb;
    uint64_t* full;
    uint64_t* empty;
    uint64_t* acc_full;
    uint64_t* acc_empty;
    uint64_t* drain;
    uint64_t* sf_ready;
    uint32_t* tmem_holder;
    volatile int* abort;
};

__device__ __forceinline__ Smem carve(uint8_t* raw) {
    Smem s;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    s.a = base;
    s.b = s.a + kStages * kTileBytesA;
    s.sfa = s.b + kStages * kTileBytesB;
    s.sfb = s.sfa + kStages * kSfBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(s.sfb + kStages * kSfBytes);
    s.full = bars;
    s.empty = bars + kStages;
    s.acc_full = bars + 2 * kStages;
    s.acc_empty = s.acc_full + 2;
    s.drain = s.acc_empty + 2;
    s.sf_ready = s.drain + 1;
    s.tmem_holder = reinterpret_cast<uint32_t*>(s.sf_ready + kStages);
    s.abort = reinterpret_cast<volatile int*>(s.tmem_holder + 1);
    return s;
}

}  // namespace

template <int EPI>
__global__ void __launch_bounds__(kNumThreads, 1)
    gemm_nvf4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    const Smem s = carve(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int no_abort = 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.acc_full[i], 1);
            mbar_init(&s.acc_empty[i], 4 * 32);
        }
        mbar_init(s.drain, 2);   // the MMA thread and the scale mover both retire their ops into it
        for (int i = 0; i < kStages; ++i) mbar_init(&s.sf_ready[i], 1);
        *s.abort = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(s.tmem_holder, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *s.tmem_holder;

    pdl_wait();  // A operand, tile map and tile count come from earlier kernels

    const int num_m_tiles = p.meta[1];
    const int n_tiles = p.n / kBN;
    const int total = num_m_tiles * n_tiles;
    const int kblocks = p.kdim / 64;          // 64-element MMA steps
    const int kstages = (kblocks + 3) / 4;    // 4 MMA steps per stage

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_normal();
            int stage = 0;
            uint32_t phase = 0;
            for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
                const int m_tile = tile / n_tiles, n_tile = tile % n_tiles;
                const int e = p.tile_expert[m_tile];
                if (e < 0 || e >= p.num_experts) {
                    atomicOr(p.status, kStatusBadExpert);
                    *s.abort = 1;
                    break;
                }
                const int a_row = m_tile * kBM;
                const int b_row = e * p.n + n_tile * kBN;
                const uint8_t* sfa_src = p.sfa + (size_t)m_tile * kblocks * 512;
                const uint8_t* sfb_src = p.sfb + ((size_t)e * n_tiles + n_tile) * kblocks * 512;
                for (int ks = 0; ks < kstages; ++ks) {
                    if (!mbar_wait(&s.empty[stage], phase ^ 1u, s.abort, p.status, kStatusTimeoutProducer)) goto done;
                    const int nkb = min(4, kblocks - 4 * ks);
                    const uint32_t sf_bytes = (uint32_t)nkb * 512u;
                    mbar_arrive_expect_tx(&s.full[stage], kTileBytesA + kTileBytesB + 2 * sf_bytes);
                    tma_load_2d(s.a + stage * kTileBytesA, &tmA, &s.full[stage], ks * kBKBytes, a_row, pol);
                    tma_load_2d(s.b + stage * kTileBytesB, &tmB, &s.full[stage], ks * kBKBytes, b_row, pol);
                    bulk_load(s.sfa + stage * kSfBytes, sfa_src + (size_t)ks * 4 * 512, sf_bytes, &s.full[stage], pol);
                    bulk_load(s.sfb + stage * kSfBytes, sfb_src + (size_t)ks * 4 * 512, sf_bytes, &s.full[stage], pol);
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_nvf4(kBM, kBN);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
                if (!mbar_wait(&s.acc_empty[acc], acc_phase ^ 1u, s.abort, p.status, kStatusTimeoutMma)) goto done;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)acc * kAccCols;
                for (int ks = 0; ks < kstages; ++ks) {
                    if (!mbar_wait(&s.full[stage], phase, s.abort, p.status, kStatusTimeoutMma)) goto done;
                    tc_fence_after();
                    const int nkb = min(4, kblocks - 4 * ks);
                    const uint32_t sfa_t = tmem_base + kSfColBase + (uint32_t)stage * kSfColsPerStage;
                    const uint32_t sfb_t = sfa_t + 16;
                    // the scale mover's copies for this stage have completed
                    if (!mbar_wait(&s.sf_ready[stage], phase, s.abort, p.status, kStatusTimeoutMma)) goto done;
                    tc_fence_after();
                    const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(s.a + stage * kTileBytesA));
                    const uint64_t bdesc = sdesc_kmajor_sw128(smem_u32(s.b + stage * kTileBytesB));
                    for (int j = 0; j < nkb; ++j) {
                        // advance 32 bytes (64 E2M1) along K inside the swizzled 128-byte rows
                        tc_mma_nvf4(d_tmem, adesc + 2u * j, bdesc + 2u * j, idesc, sfa_t + 4 * j, sfb_t + 4 * j,
                                    (ks | j) != 0);
                    }
                    tc_commit(&s.empty[stage]);
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
                tc_commit(&s.acc_full[acc]);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
        }
    } else if (warp == 6) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
                for (int ks = 0; ks < kstages; ++ks) {
                    if (!mbar_wait(&s.full[stage], phase, s.abort, p.status, kStatusTimeoutMma)) goto done;
                    tc_fence_after();
                    const int nkb = min(4, kblocks - 4 * ks);
                    const uint32_t sfa_t = tmem_base + kSfColBase + (uint32_t)stage * kSfColsPerStage;
                    const uint32_t sfb_t = sfa_t + 16;
                    for (int j = 0; j < nkb; ++j) {
                        tc_cp_sf_atom(sfa_t + 4 * j, sdesc_sf_atom(smem_u32(s.sfa + stage * kSfBytes + j * 512)));
                        tc_cp_sf_atom(sfb_t + 4 * j, sdesc_sf_atom(smem_u32(s.sfb + stage * kSfBytes + j * 512)));
                    }
                    tc_commit(&s.sf_ready[stage]);
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
            }
        }
    } else {
        const int q = warp & 3;  // tensor-memory lane quadrant of this warp
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            const int m_tile = tile / n_tiles, n_tile = tile % n_tiles;
            const int e = p.tile_expert[m_tile];
            if (e < 0 || e >= p.num_experts) break;
            if (!mbar_wait(&s.acc_full[acc], acc_phase, s.abort, p.status, kStatusTimeoutEpilogue)) break;
            tc_fence_after();
            const int row = m_tile * kBM + q * 32 + lane;
            const int route = p.route_of_row[row];
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)acc * kAccCols;
            if (EPI == kEpiFc1Quant || EPI == kEpiFc1F32) epilogue_fc1<EPI>(p, taddr, row, route, e, n_tile);
            else epilogue_fc2<EPI>(p, taddr, row, route, e, n_tile);
            tc_fence_before();
            mbar_arrive(&s.acc_empty[acc]);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }
done:
    if (*s.abort) {
        // Something timed out: let in-flight copies land and retire every
        // issued MMA before the tensor memory and shared memory go away.
        if ((warp == 1 || warp == 6) && lane == 0) {
            tc_commit(s.drain);
            mbar_wait(s.drain, 0, &no_abort, p.status, kStatusTimeoutMma);
        }
        for (int i = 0; i < 100; ++i) __nanosleep(10000);
    }
    tc_fence_before();
    __syncthreads();
    pdl_launch_dependents();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

cudaError_t setup_gemm_kernels() {
    cudaError_t e;
    e = cudaFuncSetAttribute(gemm_nvf4_kernel<kEpiFc1Quant>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gemm_nvf4_kernel<kEpiFc1F32>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gemm_nvf4_kernel<kEpiFc2Store>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(gemm_nvf4_kernel<kEpiFc2Scatter>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmemBytes);
}

cudaError_t launch_gemm_nvf4(const LaunchCtx& c, int epilogue, const CUtensorMap& tmA, const CUtensorMap& tmB,
                             const GemmParams& p, int num_sms) {
    const dim3 grid(num_sms), block(kNumThreads);
    switch (epilogue) {
        case kEpiFc1Quant: return c.launch(gemm_nvf4_kernel<kEpiFc1Quant>, grid, block, kSmemBytes, tmA, tmB, p);
        case kEpiFc1F32: return c.launch(gemm_nvf4_kernel<kEpiFc1F32>, grid, block, kSmemBytes, tmA, tmB, p);
        case kEpiFc2Store: return c.launch(gemm_nvf4_kernel<kEpiFc2Store>, grid, block, kSmemBytes, tmA, tmB, p);
        case kEpiFc2Scatter: return c.launch(gemm_nvf4_kernel<kEpiFc2Scatter>, grid, block, kSmemBytes, tmA, tmB, p);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace moe
