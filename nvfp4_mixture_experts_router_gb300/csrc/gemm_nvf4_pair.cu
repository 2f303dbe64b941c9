// Grouped NVFP4 x NVFP4 GEMMs on CTA pairs: the same products and fused
// epilogues as gemm_nvf4.cu, computed by tcgen05.mma.cta_group::2 with a
// 256 x 256 tile per pair of SMs.
//
// Why pairs: with the M = 256 pair MMA each SM keeps only its own 128 A rows
// and half of the 256 B rows in shared memory, so the operand bytes each SM
// loads per FLOP fall by a third against a single-CTA 128 x 256 tile.  The
// cost is a cross-CTA handshake per pipeline stage and a single 256-column
// accumulator (no room for two next to the scale slots), whose epilogue is
// not overlapped with the next tile; measured, that cost outweighs the saved
// bytes, so the library uses this kernel only on request
// (MOE_GEMM_PAIRS_ALWAYS).
//
// Pair tile: two consecutive 128-row M tiles of ONE expert (the scan kernel
// lists them in tile_pair: (first << 1) | has_second) x 256 weight rows.  The
// even CTA holds the first M tile, B rows 0..127 of the tile and the
// accumulator rows 0..127; the odd CTA the second M tile (when the expert
// has an odd number of M tiles it loads the first one again and discards its
// rows), B rows 128..255 and accumulator rows 128..255.  Both CTAs hold the
// B scales of all 256 rows in tensor memory, as the pair MMA requires.
//
// Roles per CTA (448 threads):
//   warp 0      producer: scale atoms (own 128 A rows, all 256 B rows) on
//               sf_full, then the A tile and this CTA's half of the B tile
//               (cp.async.bulk.tensor, 128-byte swizzle) on full.
//   warps 2-5   scale writers (one per tensor-memory lane quadrant), as in
//               the single-CTA kernel.
//   warp 1      allocates 512 tensor-memory columns in both CTAs together.
//               Even CTA, lane 0: waits for its own stage (data + scales)
//               and for the odd CTA's report, issues four 256x256x64 pair
//               MMAs and commits the stage to the empty barriers of both
//               CTAs (multicast).  Odd CTA, lane 0: waits for its own stage
//               and reports it to the even CTA's peer_ready barrier.
//   warps 6-13  epilogue over this CTA's 128 rows, 128 columns per warp
//               group; the accumulator (256 columns, one buffer) is released
//               to the even CTA's acc_empty barrier by every epilogue warp of
//               both CTAs.
// Every wait is bounded (1 s); a timeout sets a status bit, marks both CTAs
// aborted, and all roles drain and reach the final pair barrier.
#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kPStages = 5;
constexpr int kPRows = 128;                      // A rows per CTA (256 per pair)
constexpr int kPN = 256;                         // weight rows per pair tile (128 per CTA)
constexpr int kPKBytes = 128;                    // 256 E2M1 elements per stage row
constexpr int kPTileA = kPRows * kPKBytes;       // 16 KB
constexpr int kPTileB = (kPN / 2) * kPKBytes;    // 16 KB
constexpr int kPSfA = 4 * 512;                   // own 128 rows, 4 k-blocks of 64
constexpr int kPSfB = 2 * 4 * 512;               // all 256 B rows, 4 k-blocks
constexpr int kPStageBytes = kPTileA + kPTileB + kPSfA + kPSfB;
constexpr int kPSfWarps = 4;
constexpr int kPEpiWarp0 = 2 + kPSfWarps;
constexpr int kPEpiWarps = 8;
constexpr int kPThreads = (kPEpiWarp0 + kPEpiWarps) * 32;
constexpr uint32_t kPTmemCols = 512;
constexpr uint32_t kPSfCol0 = kPN;               // accumulator: columns 0..255
constexpr uint32_t kPSfColsStage = 16 + 32;      // A scales 4 x 4, B scales 4 x 8 columns
constexpr int kPSmemBytes = kPStages * kPStageBytes + 1024 + 512;
static_assert(kPSfCol0 + kPStages * kPSfColsStage <= kPTmemCols, "tensor memory budget");

struct PairSmem {
    uint8_t* a;
    uint8_t* b;
    uint8_t* sfa;
    uint8_t* sfb;
    uint64_t* full;
    uint64_t* sf_full;
    uint64_t* empty;
    uint64_t* sf_ready;
    uint64_t* peer_ready;   // even CTA: the odd CTA's stage is ready
    uint64_t* acc_full;
    uint64_t* acc_empty;    // even CTA: both CTAs' epilogues released the accumulator
    uint64_t* drain;
    uint32_t* tmem_holder;
    volatile int* abort;
};

__device__ __forceinline__ PairSmem carve_pair(uint8_t* raw) {
    PairSmem s;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    s.a = base;
    s.b = s.a + kPStages * kPTileA;
    s.sfa = s.b + kPStages * kPTileB;
    s.sfb = s.sfa + kPStages * kPSfA;
    uint64_t* bars = reinterpret_cast<uint64_t*>(s.sfb + kPStages * kPSfB);
    s.full = bars;
    s.sf_full = bars + kPStages;
    s.empty = bars + 2 * kPStages;
    s.sf_ready = bars + 3 * kPStages;
    s.peer_ready = bars + 4 * kPStages;
    s.acc_full = bars + 5 * kPStages;
    s.acc_empty = s.acc_full + 1;
    s.drain = s.acc_empty + 1;
    s.tmem_holder = reinterpret_cast<uint32_t*>(s.drain + 1);
    s.abort = reinterpret_cast<volatile int*>(s.tmem_holder + 1);
    return s;
}

}  // namespace

template <int EPI>
__global__ void __launch_bounds__(kPThreads, 1)
    gemm_nvf4_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                          const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    const PairSmem s = carve_pair(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_cta_rank();          // 0: issues the pair MMAs
    const int pair_slot = blockIdx.x >> 1, pair_slots = gridDim.x >> 1;
    volatile int no_abort = 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kPStages; ++i) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.sf_full[i], 1);
            mbar_init(&s.empty[i], 1);
            mbar_init(&s.sf_ready[i], kPSfWarps * 32);
            mbar_init(&s.peer_ready[i], 1);
        }
        mbar_init(s.acc_full, 1);
        mbar_init(s.acc_empty, 2 * kPEpiWarps);
        mbar_init(s.drain, 1);
        *s.abort = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc_pair(s.tmem_holder, kPTmemCols);
        tmem_relinquish_pair();
    }
    // both CTAs' barriers initialized and tensor memory allocated before any
    // cross-CTA arrival or pair MMA
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = *s.tmem_holder;

    pdl_wait();  // A operand, tile maps and counts come from earlier kernels

    const int num_pairs = p.meta[2];
    const int num_m_tiles = p.meta[1];
    const int n_tiles = p.n / kPN;
    const int total = num_pairs * n_tiles;
    const int kblocks = p.kdim / 64;
    const int kstages = (kblocks + 3) / 4;
    const int rb_per_expert = p.n / 128;

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_normal();
            int stage = 0;
            uint32_t phase = 0;
            for (int tile = pair_slot; tile < total; tile += pair_slots) {
                const int pr = tile / n_tiles, n_tile = tile % n_tiles;
                const int v = p.tile_pair[pr];
                const int m0 = v >> 1;
                const int m_tile = (rank == 1 && (v & 1)) ? m0 + 1 : m0;
                const int e = (m0 >= 0 && m0 < num_m_tiles) ? p.tile_expert[m0] : -1;
                if (e < 0 || e >= p.num_experts || m_tile >= num_m_tiles) {
                    atomicOr(p.status, kStatusBadExpert);
                    *s.abort = 1;
                    break;
                }
                const int a_row = m_tile * kPRows;
                const int b_row = e * p.n + n_tile * kPN + (int)rank * (kPN / 2);
                const uint8_t* sfa_src = p.sfa + (size_t)m_tile * kblocks * 512;
                const uint8_t* sfb_src = p.sfb + ((size_t)e * rb_per_expert + (size_t)n_tile * 2) * kblocks * 512;
                for (int ks = 0; ks < kstages; ++ks) {
                    if (!mbar_wait(&s.empty[stage], phase ^ 1u, s.abort, p.status, kStatusTimeoutProducer)) goto done;
                    const int nkb = min(4, kblocks - 4 * ks);
                    const uint32_t sf_bytes = (uint32_t)nkb * 512u;
                    mbar_arrive_expect_tx(&s.sf_full[stage], 3u * sf_bytes);
                    bulk_load(s.sfa + stage * kPSfA, sfa_src + (size_t)ks * 4 * 512, sf_bytes, &s.sf_full[stage], pol);
                    for (int rb = 0; rb < 2; ++rb)
                        bulk_load(s.sfb + stage * kPSfB + rb * kPSfA,
                                  sfb_src + ((size_t)rb * kblocks + (size_t)ks * 4) * 512, sf_bytes,
                                  &s.sf_full[stage], pol);
                    mbar_arrive_expect_tx(&s.full[stage], kPTileA + kPTileB);
                    tma_load_2d(s.a + stage * kPTileA, &tmA, &s.full[stage], ks * kPKBytes, a_row, pol);
                    tma_load_2d(s.b + stage * kPTileB, &tmB, &s.full[stage], ks * kPKBytes, b_row, pol);
                    if (++stage == kPStages) { stage = 0; phase ^= 1u; }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            const uint32_t idesc = idesc_nvf4(2 * kPRows, kPN);
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            for (int tile = pair_slot; tile < total; tile += pair_slots) {
                if (!mbar_wait(s.acc_empty, acc_phase ^ 1u, s.abort, p.status, kStatusTimeoutMma)) goto done;
                tc_fence_after();
                for (int ks = 0; ks < kstages; ++ks) {
                    if (!mbar_wait(&s.full[stage], phase, s.abort, p.status, kStatusTimeoutMma)) goto done;
                    if (!mbar_wait(&s.sf_ready[stage], phase, s.abort, p.status, kStatusTimeoutMma)) goto done;
                    if (!mbar_wait(&s.peer_ready[stage], phase, s.abort, p.status, kStatusTimeoutMma)) goto done;
                    tc_fence_after();
                    const int nkb = min(4, kblocks - 4 * ks);
                    const uint32_t sfa_t = tmem_base + kPSfCol0 + (uint32_t)stage * kPSfColsStage;
                    const uint32_t sfb_t = sfa_t + 16;
                    const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(s.a + stage * kPTileA));
                    const uint64_t bdesc = sdesc_kmajor_sw128(smem_u32(s.b + stage * kPTileB));
                    for (int j = 0; j < nkb; ++j)
                        tc_mma_nvf4_pair(tmem_base, adesc + 2u * j, bdesc + 2u * j, idesc, sfa_t + 4 * j,
                                         sfb_t + 8 * j, (ks | j) != 0);
                    tc_commit_pair_mc(&s.empty[stage], 0x3);
                    if (++stage == kPStages) { stage = 0; phase ^= 1u; }
                }
                tc_commit_pair_mc(s.acc_full, 0x3);
                acc_phase ^= 1u;
            }
        } else if (lane == 0) {
            // odd CTA: report each landed and scale-written stage to the even CTA
            const uint32_t ready0 = cluster_map(s.peer_ready, 0);
            int stage = 0;
            uint32_t phase = 0;
            for (int tile = pair_slot; tile < total; tile += pair_slots) {
                for (int ks = 0; ks < kstages; ++ks) {
                    if (!mbar_wait(&s.full[stage], phase, s.abort, p.status, kStatusTimeoutMma)) goto done;
                    if (!mbar_wait(&s.sf_ready[stage], phase, s.abort, p.status, kStatusTimeoutMma)) goto done;
                    mbar_arrive_cluster(ready0 + (uint32_t)stage * 8u);
                    if (++stage == kPStages) { stage = 0; phase ^= 1u; }
                }
            }
        }
    } else if (warp < kPEpiWarp0) {
        // scale writer for lane quadrant warp % 4 (same layout as the
        // single-CTA kernel with 256-wide tiles)
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        int stage = 0;
        uint32_t phase = 0;
        for (int tile = pair_slot; tile < total; tile += pair_slots) {
            for (int ks = 0; ks < kstages; ++ks) {
                // warp-uniform outcome: tcgen05.st below is a warp-collective instruction
                if (!__all_sync(0xffffffffu,
                                mbar_wait(&s.sf_full[stage], phase, s.abort, p.status, kStatusTimeoutMma)))
                    goto done;
                const uint32_t sfa_t = tmem_base + kPSfCol0 + (uint32_t)stage * kPSfColsStage;
                const uint32_t sfb_t = sfa_t + 16;
                uint32_t ra[16];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 v = *reinterpret_cast<const uint4*>(s.sfa + stage * kPSfA + j * 512 + lane * 16);
                    ra[4 * j] = v.x; ra[4 * j + 1] = v.y; ra[4 * j + 2] = v.z; ra[4 * j + 3] = v.w;
                }
                tmem_st16(sfa_t + lane_off, ra);
                uint32_t rb_[32];
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int rb = 0; rb < 2; ++rb) {
                        const uint4 v =
                            *reinterpret_cast<const uint4*>(s.sfb + stage * kPSfB + rb * kPSfA + j * 512 + lane * 16);
                        rb_[8 * j + 4 * rb] = v.x; rb_[8 * j + 4 * rb + 1] = v.y;
                        rb_[8 * j + 4 * rb + 2] = v.z; rb_[8 * j + 4 * rb + 3] = v.w;
                    }
                tmem_st32(sfb_t + lane_off, rb_);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&s.sf_ready[stage]);
                if (++stage == kPStages) { stage = 0; phase ^= 1u; }
            }
        }
    } else {
        const int q = warp & 3;                            // tensor-memory lane quadrant of this warp
        const int half = (warp - kPEpiWarp0) >> 2;         // accumulator columns 0..127 or 128..255
        const uint32_t release = cluster_map(s.acc_empty, 0);
        uint32_t acc_phase = 0;
        for (int tile = pair_slot; tile < total; tile += pair_slots) {
            const int pr = tile / n_tiles, n_tile = tile % n_tiles;
            const int v = p.tile_pair[pr];
            const int m0 = v >> 1;
            const int m_tile = rank == 0 ? m0 : ((v & 1) ? m0 + 1 : -1);
            const int e = (m0 >= 0 && m0 < num_m_tiles) ? p.tile_expert[m0] : -1;
            if (e < 0 || e >= p.num_experts || m_tile >= num_m_tiles) break;
            // warp-uniform outcome: tcgen05.ld below is a warp-collective instruction
            if (!__all_sync(0xffffffffu,
                            mbar_wait(s.acc_full, acc_phase, s.abort, p.status, kStatusTimeoutEpilogue)))
                break;
            tc_fence_after();
            if (m_tile >= 0) {
                const int row = m_tile * kPRows + q * 32 + lane;
                const int route = p.route_of_row[row];
                const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(half * 128);
                const int vtile = n_tile * 2 + half;        // index of this 128-column slice
                if (EPI == kEpiFc1Quant || EPI == kEpiFc1F32) epilogue_fc1<EPI>(p, taddr, row, route, e, vtile);
                else epilogue_fc2<EPI>(p, taddr, row, route, e, vtile);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(release);
            acc_phase ^= 1u;
        }
    }
done:
    if (*s.abort) {
        // Something timed out or a tile map entry was bad: tell the other CTA,
        // let in-flight copies land and retire every issued MMA and store
        // before the memories go away.
        st_cluster_u32(cluster_map((const void*)s.abort, rank ^ 1u), 1u);
        if (warp == 1 && lane == 0 && rank == 0) {
            tc_commit_pair(s.drain);
            mbar_wait(s.drain, 0, &no_abort, p.status, kStatusTimeoutMma);
        }
        if (warp >= 2 && warp < kPEpiWarp0) tmem_st_wait();
        for (int i = 0; i < 100; ++i) __nanosleep(10000);
    }
    tc_fence_before();
    __syncthreads();
    // neither CTA frees tensor memory or leaves (its shared memory is an
    // operand of the other CTA's MMAs) before both are done
    cluster_sync_all();
    pdl_launch_dependents();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kPTmemCols);
    }
}

namespace {
int g_pair_grid[64] = {};
}

cudaError_t setup_gemm_pair_kernels(int device, int num_sms) {
    cudaError_t e;
    const int b = kPSmemBytes;
    if ((e = cudaFuncSetAttribute(gemm_nvf4_pair_kernel<kEpiFc1Quant>, cudaFuncAttributeMaxDynamicSharedMemorySize, b)))
        return e;
    if ((e = cudaFuncSetAttribute(gemm_nvf4_pair_kernel<kEpiFc1F32>, cudaFuncAttributeMaxDynamicSharedMemorySize, b)))
        return e;
    if ((e = cudaFuncSetAttribute(gemm_nvf4_pair_kernel<kEpiFc2Store>, cudaFuncAttributeMaxDynamicSharedMemorySize, b)))
        return e;
    if ((e = cudaFuncSetAttribute(gemm_nvf4_pair_kernel<kEpiFc2Scatter>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  b)))
        return e;
    // persistent grid: as many CTA pairs as can be resident at once
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(num_sms / 2 * 2));
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = kPSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if ((e = cudaOccupancyMaxActiveClusters(&clusters, gemm_nvf4_pair_kernel<kEpiFc1Quant>, &cfg))) return e;
    if (clusters < 1) return cudaErrorInvalidConfiguration;
    if (device >= 0 && device < 64) g_pair_grid[device] = 2 * min(clusters, num_sms / 2);
    return cudaSuccess;
}

cudaError_t launch_gemm_nvf4_pair(const LaunchCtx& c, int epilogue, const CUtensorMap& tmA, const CUtensorMap& tmB,
                                  const GemmParams& p, int device) {
    if (device < 0 || device >= 64 || g_pair_grid[device] < 2) return cudaErrorInvalidValue;
    LaunchCtx cc = c;
    cc.cluster = 2;
    const dim3 grid((unsigned)g_pair_grid[device]), block(kPThreads);
    const size_t smem = kPSmemBytes;
    switch (epilogue) {
        case kEpiFc1Quant: return cc.launch(gemm_nvf4_pair_kernel<kEpiFc1Quant>, grid, block, smem, tmA, tmB, p);
        case kEpiFc1F32: return cc.launch(gemm_nvf4_pair_kernel<kEpiFc1F32>, grid, block, smem, tmA, tmB, p);
        case kEpiFc2Store: return cc.launch(gemm_nvf4_pair_kernel<kEpiFc2Store>, grid, block, smem, tmA, tmB, p);
        case kEpiFc2Scatter: return cc.launch(gemm_nvf4_pair_kernel<kEpiFc2Scatter>, grid, block, smem, tmA, tmB, p);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace moe
