// Grouped W4A16 GEMMs: BF16 activations x NVFP4 weights, FP32 accumulation
// on the tcgen05 tensor cores (kind::f16 with BF16 operands) [newruntime
// post on FlashInfer PR #5319, "Retrieval answer": W4A16 with BF16
// activations; W4A4 and W4A16 consume the same prepared NVFP4 weights].
//
// The tensor core has no mixed BF16 x E2M1 mode, so the weights are widened
// on chip: each stage brings the weight tile in as E2M1 codes plus its E4M3
// scale atom (a quarter of the bytes of BF16), and converter warps write
// q * s -- exact in BF16 (at most 6 significant bits, |q*s| in
// [2^-10, 2688]) -- into shared memory in the 128-byte-swizzled K-major
// layout the MMA reads.  The per-expert FP32 scale Gw is applied in the
// epilogue.
//
// One persistent CTA per SM, 320 threads:
//   warp 0      TMA producer: per stage a 128x64 BF16 activation tile
//               (128-byte swizzle), the 128x64 E2M1 weight tile (32 B rows)
//               and its 512-byte scale atom, one mbarrier per stage.
//   warps 6-9   converters: one weight row per thread, E2M1 x E4M3 -> BF16
//               into the swizzled tile, fence.proxy.async, arrive.
//   warp 1      allocates 256 tensor-memory columns; lane 0 issues four
//               128x128x16 BF16 MMAs per stage, commits the stage.
//   warps 2-5   epilogue (shared with the NVFP4 GEMM, epilogue.cuh).
// Waits are bounded as in gemm_nvf4.cu.
//
// CTA-pair variant (gemm_w4a16_pair_kernel, for experts averaging >= 256
// routes): a 256 x 256 tile per pair of SMs -- two consecutive 128-row M
// tiles of one expert x 256 weight rows -- with
// tcgen05.mma.cta_group::2.kind::f16.  Each CTA loads its own 128 activation
// rows and converts its own 128 of the 256 weight rows, so per FLOP it moves
// and converts half the weight bytes of a 128 x 256 single-CTA tile and a
// quarter of those of the 128 x 128 one.  Without block scales in tensor
// memory, two 256-column accumulators fit (all 512 columns): the epilogue of
// one tile overlaps the main loop of the next.
#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"
#include "pair_tiles.cuh"
#include "w4a16_convert.cuh"

namespace moe {

namespace {

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kStages = 6;
constexpr int kTileBytesA = kBM * 128;   // 64 BF16 per row
constexpr int kTileBytesB = kBN * 128;   // converted weights, 64 BF16 per row
constexpr int kTileBytesQ = kBN * 32;    // 64 E2M1 per row
constexpr int kSfBytes = 512;            // one scale atom: 128 rows x 4 scales
constexpr int kConvWarps = 4;
constexpr int kNumThreads = (6 + kConvWarps) * 32;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kAccCols = 128;
constexpr int kStgCols = 8;                           // FC2 epilogue staging, words per row
constexpr int kStgBytes = 4 * 32 * kStgCols * 4;      // one block per epilogue warp
constexpr int kSmemBytes = kStages * (kTileBytesA + kTileBytesB + kTileBytesQ + kSfBytes) + kStgBytes + 1024 + 256;
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Smem {
    uint8_t* a;
    uint8_t* b;
    uint8_t* q;
    uint8_t* sf;
    uint32_t* stg;
    uint64_t* full;
    uint64_t* conv;
    uint64_t* empty;
    uint64_t* acc_full;
    uint64_t* acc_empty;
    uint64_t* drain;
    uint32_t* tmem_holder;
    volatile int* abort;
};

__device__ __forceinline__ Smem carve(uint8_t* raw) {
    Smem s;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    s.a = base;
    s.b = s.a + kStages * kTileBytesA;
    s.q = s.b + kStages * kTileBytesB;
    s.sf = s.q + kStages * kTileBytesQ;
    s.stg = reinterpret_cast<uint32_t*>(s.sf + kStages * kSfBytes);
    uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(s.stg) + kStgBytes);
    s.full = bars;
    s.conv = bars + kStages;
    s.empty = bars + 2 * kStages;
    s.acc_full = bars + 3 * kStages;
    s.acc_empty = s.acc_full + 2;
    s.drain = s.acc_empty + 2;
    s.tmem_holder = reinterpret_cast<uint32_t*>(s.drain + 1);
    s.abort = reinterpret_cast<volatile int*>(s.tmem_holder + 1);
    return s;
}

}  // namespace

template <int EPI>
__global__ void __launch_bounds__(kNumThreads, 1)
    gemm_w4a16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmBq,
                      const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    const Smem s = carve(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int no_abort = 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.conv[i], kConvWarps);
            mbar_init(&s.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.acc_full[i], 1);
            mbar_init(&s.acc_empty[i], 4 * 32);
        }
        mbar_init(s.drain, 1);
        *s.abort = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmBq);
    }
    if (warp == 1) {
        tmem_alloc(s.tmem_holder, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *s.tmem_holder;

    pdl_wait();

    const int num_m_tiles = p.meta[1];
    const int n_tiles = p.n / kBN;
    const int total = num_m_tiles * n_tiles;
    const int kblocks = p.kdim / 64;   // one 64-element block per stage

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
                const uint8_t* sf_src = p.sfb + ((size_t)e * n_tiles + n_tile) * kblocks * 512;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait(&s.empty[stage], phase ^ 1u, s.abort, p.status, kStatusTimeoutProducer)) goto done;
                    mbar_arrive_expect_tx(&s.full[stage], kTileBytesA + kTileBytesQ + kSfBytes);
                    tma_load_2d(s.a + stage * kTileBytesA, &tmA, &s.full[stage], kb * 128, a_row, pol);
                    tma_load_2d(s.q + stage * kTileBytesQ, &tmBq, &s.full[stage], kb * 32, b_row, pol);
                    bulk_load(s.sf + stage * kSfBytes, sf_src + (size_t)kb * 512, kSfBytes, &s.full[stage], pol);
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(kBM, kBN);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
                if (!mbar_wait(&s.acc_empty[acc], acc_phase ^ 1u, s.abort, p.status, kStatusTimeoutMma)) goto done;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)acc * kAccCols;
                for (int kb = 0; kb < kblocks; ++kb) {
                    // converted weights ready (the converters waited for the whole stage to land)
                    if (!mbar_wait(&s.conv[stage], phase, s.abort, p.status, kStatusTimeoutMma)) goto done;
                    tc_fence_after();
                    const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(s.a + stage * kTileBytesA));
                    const uint64_t bdesc = sdesc_kmajor_sw128(smem_u32(s.b + stage * kTileBytesB));
#pragma unroll
                    for (int j = 0; j < 4; ++j)   // 16 BF16 = 32 bytes along K per MMA
                        tc_mma_bf16(d_tmem, adesc + 2u * j, bdesc + 2u * j, idesc, (kb | j) != 0);
                    tc_commit(&s.empty[stage]);
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
                tc_commit(&s.acc_full[acc]);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
        }
    } else if (warp >= 6) {
        // converter: thread r owns weight row r of every stage
        const int r = (warp - 6) * 32 + lane;
        const uint32_t sf_off = (uint32_t)(r & 31) * 16u + (uint32_t)(r >> 5) * 4u;
        int stage = 0;
        uint32_t phase = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            for (int kb = 0; kb < kblocks; ++kb) {
                if (!__all_sync(0xffffffffu,
                                mbar_wait(&s.full[stage], phase, s.abort, p.status, kStatusTimeoutProducer)))
                    goto done;
                const uint4 c0 = *reinterpret_cast<const uint4*>(s.q + stage * kTileBytesQ + r * 32);
                const uint4 c1 = *reinterpret_cast<const uint4*>(s.q + stage * kTileBytesQ + r * 32 + 16);
                const uint32_t sfw = *reinterpret_cast<const uint32_t*>(s.sf + stage * kSfBytes + sf_off);
                const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                uint8_t* brow = s.b + stage * kTileBytesB + r * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) {          // 16-byte chunk c = elements 8c .. 8c+7
                    const __half2 sc = __float2half2_rn(e4m3_to_f32((sfw >> (8 * (c >> 1))) & 0xFFu));
                    *reinterpret_cast<uint4*>(brow + ((c ^ (r & 7)) << 4)) = dequant8(words[c], sc);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s.conv[stage]);
                if (++stage == kStages) { stage = 0; phase ^= 1u; }
            }
        }
    } else {
        const int q = warp & 3;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            const int m_tile = tile / n_tiles, n_tile = tile % n_tiles;
            const int e = p.tile_expert[m_tile];
            if (e < 0 || e >= p.num_experts) break;
            // the row's epilogue scalars, loaded while the main loop runs
            const int row = m_tile * kBM + q * 32 + lane;
            const EpiRow meta = epi_row<EPI>(p, row, e);
            // warp-uniform outcome: tcgen05.ld below is a warp-collective instruction
            if (!__all_sync(0xffffffffu, mbar_wait(&s.acc_full[acc], acc_phase, s.abort, p.status,
                                                   kStatusTimeoutEpilogue)))
                break;
            tc_fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)acc * kAccCols;
            if (EPI == kEpiFc1Bf16)
                epilogue_fc1<EPI, kStgCols>(p, taddr, row, meta, n_tile, s.stg + q * 32 * kStgCols);
            else epilogue_fc2<EPI, kStgCols>(p, taddr, row, meta, n_tile, s.stg + q * 32 * kStgCols);
            tc_fence_before();
            mbar_arrive(&s.acc_empty[acc]);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }
done:
    if (*s.abort) {
        if (warp == 1 && lane == 0) {
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

cudaError_t setup_gemm_w4a16_kernels() {
    cudaError_t e;
    e = cudaFuncSetAttribute(gemm_w4a16_kernel<kEpiFc1Bf16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gemm_w4a16_kernel<kEpiFc2Store>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(gemm_w4a16_kernel<kEpiFc2Scatter>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmemBytes);
}

cudaError_t launch_gemm_w4a16(const LaunchCtx& c, int epilogue, const CUtensorMap& tmA, const CUtensorMap& tmBq,
                              const GemmParams& p, int num_sms) {
    const dim3 grid(num_sms), block(kNumThreads);
    switch (epilogue) {
        case kEpiFc1Bf16: return c.launch(gemm_w4a16_kernel<kEpiFc1Bf16>, grid, block, kSmemBytes, tmA, tmBq, p);
        case kEpiFc2Store: return c.launch(gemm_w4a16_kernel<kEpiFc2Store>, grid, block, kSmemBytes, tmA, tmBq, p);
        case kEpiFc2Scatter:
            return c.launch(gemm_w4a16_kernel<kEpiFc2Scatter>, grid, block, kSmemBytes, tmA, tmBq, p);
        default: return cudaErrorInvalidValue;
    }
}

// ---------------------------------------------------------------------------
// CTA-pair kernel
// ---------------------------------------------------------------------------
namespace {

constexpr int kQRows = 128;                       // A rows and converted B rows per CTA
constexpr int kQN = 256;                          // weight rows per pair tile
constexpr int kQStages = 5;
constexpr int kQConvWarps = 8;                 // two per lane quadrant: half a row's K block each
constexpr int kQEpiWarp0 = 2 + kQConvWarps;
constexpr int kQEpiWarps = 8;
constexpr int kQThreads = (kQEpiWarp0 + kQEpiWarps) * 32;
constexpr uint32_t kQTmemCols = 512;              // two 256-column accumulators
constexpr int kQTileA = kQRows * 128;
constexpr int kQTileB = kQRows * 128;
constexpr int kQTileQ = kQRows * 32;
constexpr int kQStgBytes = kQEpiWarps * 32 * kStgCols * 4;
constexpr int kQSmemBytes = kQStages * (kQTileA + kQTileB + kQTileQ + kSfBytes) + kQStgBytes + 1024 + 512;
static_assert(kQSmemBytes <= 232448, "shared memory budget");

struct PairSmemW {
    uint8_t* a;
    uint8_t* b;
    uint8_t* q;
    uint8_t* sf;
    uint32_t* stg;
    uint64_t* afull;      // [kQStages] rank 0: both CTAs' activation tiles landed
    uint64_t* qfull;      // [kQStages] this CTA's weight codes + scale atom landed
    uint64_t* conv;       // [kQStages] rank 0: both CTAs' converters wrote their weight rows
    uint64_t* empty;      // [kQStages] both CTAs: the stage's MMAs are done
    uint64_t* acc_full;   // [2]
    uint64_t* acc_empty;  // [2] rank 0: both CTAs' epilogues released the accumulator
    uint64_t* drain;
    uint32_t* tmem_holder;
    volatile int* abort;
};

__device__ __forceinline__ PairSmemW carve_pair_w(uint8_t* raw) {
    PairSmemW s;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    s.a = base;
    s.b = s.a + kQStages * kQTileA;
    s.q = s.b + kQStages * kQTileB;
    s.sf = s.q + kQStages * kQTileQ;
    s.stg = reinterpret_cast<uint32_t*>(s.sf + kQStages * kSfBytes);
    uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(s.stg) + kQStgBytes);
    s.afull = bars;
    s.qfull = bars + kQStages;
    s.conv = bars + 2 * kQStages;
    s.empty = bars + 3 * kQStages;
    s.acc_full = bars + 4 * kQStages;
    s.acc_empty = s.acc_full + 2;
    s.drain = s.acc_empty + 2;
    s.tmem_holder = reinterpret_cast<uint32_t*>(s.drain + 1);
    s.abort = reinterpret_cast<volatile int*>(s.tmem_holder + 1);
    return s;
}

}  // namespace

// Roles per CTA (576 threads): warp 0 producer (its A rows counted on rank
// 0's afull barrier, its weight codes and scales on its own qfull), warp 1
// tensor-memory allocation and, in rank 0, the MMA issuer; warps 2-9
// converters (this CTA's 128 weight rows, two threads per row, arriving on
// rank 0's conv barrier); warps 10-17 epilogue over this CTA's 128 rows (two
// groups of four warps, 128 accumulator columns each).  Every wait is bounded (1 s); a timeout
// marks both CTAs aborted and all roles drain to the final pair barrier.
template <int EPI>
__global__ void __launch_bounds__(kQThreads, 1)
    gemm_w4a16_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmBq,
                           const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    const PairSmemW s = carve_pair_w(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_cta_rank();
    const int pair_slot = blockIdx.x >> 1, pair_slots = gridDim.x >> 1;
    volatile int no_abort = 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kQStages; ++i) {
            mbar_init(&s.afull[i], 1);
            mbar_init(&s.qfull[i], 1);
            mbar_init(&s.conv[i], 2 * kQConvWarps);
            mbar_init(&s.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.acc_full[i], 1);
            mbar_init(&s.acc_empty[i], 2 * kQEpiWarps);
        }
        mbar_init(s.drain, 1);
        *s.abort = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmBq);
    }
    if (warp == 1) {
        tmem_alloc_pair(s.tmem_holder, kQTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = *s.tmem_holder;

    pdl_wait();

    const int num_pairs = p.meta[2];
    const int num_m_tiles = p.meta[1];
    const int n_tiles = p.n / kQN;
    const int total = num_pairs * n_tiles;
    const int kblocks = p.kdim / 64;                 // one 64-element block per stage
    const int rb_per_expert = p.n / 128;

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_normal();
            const uint32_t afull0 = cluster_map(s.afull, 0);
            int stage = 0;
            uint32_t phase = 0;
            for (int tile = pair_slot; tile < total; tile += pair_slots) {
                int m_tile, m0, n_tile;
                decode_pair(p, tile, n_tiles, num_pairs, rank, m_tile, m0, n_tile);
                const int ld_m = m_tile >= 0 ? m_tile : m0;     // rank 1 without a second tile reloads the first
                const int e = (m0 >= 0 && m0 < num_m_tiles) ? p.tile_expert[m0] : -1;
                if (e < 0 || e >= p.num_experts || ld_m >= num_m_tiles) {
                    atomicOr(p.status, kStatusBadExpert);
                    *s.abort = 1;
                    break;
                }
                const int a_row = ld_m * kQRows;
                const int rb = n_tile * 2 + (int)rank;            // this CTA's 128-row weight block
                const int b_row = e * p.n + rb * 128;
                const uint8_t* sf_src = p.sfb + ((size_t)e * rb_per_expert + rb) * kblocks * 512;
                for (int kb = 0; kb < kblocks; ++kb) {
                    // completed by rank 0's commit: acquire at cluster scope
                    if (!mbar_wait<true>(&s.empty[stage], phase ^ 1u, s.abort, p.status, kStatusTimeoutProducer))
                        goto done;
                    if (rank == 0) mbar_arrive_expect_tx(&s.afull[stage], 2u * kQTileA);
                    tma_load_2d_pair(s.a + stage * kQTileA, &tmA, afull0 + (uint32_t)stage * 8u, kb * 128, a_row, pol);
                    mbar_arrive_expect_tx(&s.qfull[stage], kQTileQ + kSfBytes);
                    tma_load_2d(s.q + stage * kQTileQ, &tmBq, &s.qfull[stage], kb * 32, b_row, pol);
                    bulk_load(s.sf + stage * kSfBytes, sf_src + (size_t)kb * 512, kSfBytes, &s.qfull[stage], pol);
                    if (++stage == kQStages) { stage = 0; phase ^= 1u; }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            const uint32_t idesc = idesc_bf16(2 * kQRows, kQN);
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            for (int tile = pair_slot; tile < total; tile += pair_slots) {
                if (!mbar_wait<true>(&s.acc_empty[acc], acc_phase ^ 1u, s.abort, p.status, kStatusTimeoutMma))
                    goto done;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)acc * kQN;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait<true>(&s.afull[stage], phase, s.abort, p.status, kStatusTimeoutMma)) goto done;
                    if (!mbar_wait<true>(&s.conv[stage], phase, s.abort, p.status, kStatusTimeoutMma)) goto done;
                    tc_fence_after();
                    const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(s.a + stage * kQTileA));
                    const uint64_t bdesc = sdesc_kmajor_sw128(smem_u32(s.b + stage * kQTileB));
#pragma unroll
                    for (int j = 0; j < 4; ++j)   // 16 BF16 = 32 bytes along K per MMA
                        tc_mma_bf16_pair(d_tmem, adesc + 2u * j, bdesc + 2u * j, idesc, (kb | j) != 0);
                    tc_commit_pair_mc(&s.empty[stage], 0x3);
                    if (++stage == kQStages) { stage = 0; phase ^= 1u; }
                }
                tc_commit_pair_mc(&s.acc_full[acc], 0x3);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
        }
    } else if (warp < kQEpiWarp0) {
        // converter: thread (r, hk) owns elements 32 hk .. 32 hk + 31 of weight
        // row r of this CTA's half of every stage
        const int r = ((warp - 2) & 3) * 32 + lane, hk = (warp - 2) >> 2;
        const uint32_t sf_off = (uint32_t)(r & 31) * 16u + (uint32_t)(r >> 5) * 4u;
        const uint32_t conv0 = cluster_map(s.conv, 0);
        int stage = 0;
        uint32_t phase = 0;
        for (int tile = pair_slot; tile < total; tile += pair_slots) {
            for (int kb = 0; kb < kblocks; ++kb) {
                // qfull lands only after the producer saw the stage empty, so
                // the converted-row slot is free as well
                if (!__all_sync(0xffffffffu,
                                mbar_wait(&s.qfull[stage], phase, s.abort, p.status, kStatusTimeoutProducer)))
                    goto done;
                const uint4 cw = *reinterpret_cast<const uint4*>(s.q + stage * kQTileQ + r * 32 + hk * 16);
                const uint32_t sfw = *reinterpret_cast<const uint32_t*>(s.sf + stage * kSfBytes + sf_off);
                const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
                uint8_t* brow = s.b + stage * kQTileB + r * 128;
#pragma unroll
                for (int j = 0; j < 4; ++j) {          // 16-byte chunk c = elements 8c .. 8c+7
                    const int c = 4 * hk + j;
                    const __half2 sc = __float2half2_rn(e4m3_to_f32((sfw >> (8 * (c >> 1))) & 0xFFu));
                    *reinterpret_cast<uint4*>(brow + ((c ^ (r & 7)) << 4)) = dequant8(words[j], sc);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (rank == 0) mbar_arrive(&s.conv[stage]);
                    else mbar_arrive_remote_cta_release(conv0 + (uint32_t)stage * 8u);
                }
                if (++stage == kQStages) { stage = 0; phase ^= 1u; }
            }
        }
    } else {
        const int q = warp & 3;                               // tensor-memory lane quadrant
        const int half = (warp - kQEpiWarp0) >> 2;            // accumulator columns 0..127 or 128..255
        const uint32_t release0 = cluster_map(s.acc_empty, 0);
        uint32_t* stg = s.stg + (warp - kQEpiWarp0) * 32 * kStgCols;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = pair_slot; tile < total; tile += pair_slots) {
            int m_tile, m0, n_tile;
            decode_pair(p, tile, n_tiles, num_pairs, rank, m_tile, m0, n_tile);
            const int e = (m0 >= 0 && m0 < num_m_tiles) ? p.tile_expert[m0] : -1;
            if (e < 0 || e >= p.num_experts || m_tile >= num_m_tiles) break;
            const int row = m_tile >= 0 ? m_tile * kQRows + q * 32 + lane : -1;
            const EpiRow meta = epi_row<EPI>(p, row, e);
            // warp-uniform outcome: tcgen05.ld below is a warp-collective instruction
            if (!__all_sync(0xffffffffu, mbar_wait<true>(&s.acc_full[acc], acc_phase, s.abort, p.status,
                                                         kStatusTimeoutEpilogue)))
                break;
            tc_fence_after();
            const uint32_t taddr =
                tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)acc * kQN + (uint32_t)(half * 128);
            const int vtile = n_tile * 2 + half;              // index of this 128-column slice
            if (m_tile >= 0) {
                if (EPI == kEpiFc1Bf16) epilogue_fc1<EPI, kStgCols>(p, taddr, row, meta, vtile, stg);
                else epilogue_fc2<EPI, kStgCols>(p, taddr, row, meta, vtile, stg);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (rank == 0) mbar_arrive(&s.acc_empty[acc]);
                else mbar_arrive_cluster(release0 + (uint32_t)acc * 8u);
            }
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }
done:
    if (*s.abort) {
        st_cluster_u32(cluster_map((const void*)s.abort, rank ^ 1u), 1u);
        if (warp == 1 && lane == 0 && rank == 0) {
            tc_commit_pair(s.drain);
            mbar_wait(s.drain, 0, &no_abort, p.status, kStatusTimeoutMma);
        }
        for (int i = 0; i < 100; ++i) __nanosleep(10000);
    }
    tc_fence_before();
    __syncthreads();
    // neither CTA frees tensor memory or leaves before both are done
    cluster_sync_all();
    pdl_launch_dependents();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kQTmemCols);
    }
}

namespace {
int g_w16_pair_grid[64] = {};
}

cudaError_t setup_gemm_w4a16_pair_kernels(int device, int num_sms) {
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(gemm_w4a16_pair_kernel<kEpiFc1Bf16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kQSmemBytes)))
        return e;
    if ((e = cudaFuncSetAttribute(gemm_w4a16_pair_kernel<kEpiFc2Store>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmemBytes)))
        return e;
    if ((e = cudaFuncSetAttribute(gemm_w4a16_pair_kernel<kEpiFc2Scatter>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmemBytes)))
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(num_sms / 2 * 2));
    cfg.blockDim = dim3(kQThreads);
    cfg.dynamicSmemBytes = kQSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if ((e = cudaOccupancyMaxActiveClusters(&clusters, gemm_w4a16_pair_kernel<kEpiFc1Bf16>, &cfg))) return e;
    if (clusters < 1) return cudaErrorInvalidConfiguration;
    if (device >= 0 && device < 64) g_w16_pair_grid[device] = 2 * min(clusters, num_sms / 2);
    return cudaSuccess;
}

cudaError_t launch_gemm_w4a16_pair(const LaunchCtx& c, int epilogue, const CUtensorMap& tmA,
                                   const CUtensorMap& tmBq, const GemmParams& p, int device) {
    if (device < 0 || device >= 64 || g_w16_pair_grid[device] < 2) return cudaErrorInvalidValue;
    LaunchCtx cc = c;
    cc.cluster = 2;
    const dim3 grid((unsigned)g_w16_pair_grid[device]), block(kQThreads);
    switch (epilogue) {
        case kEpiFc1Bf16:
            return cc.launch(gemm_w4a16_pair_kernel<kEpiFc1Bf16>, grid, block, (size_t)kQSmemBytes, tmA, tmBq, p);
        case kEpiFc2Store:
            return cc.launch(gemm_w4a16_pair_kernel<kEpiFc2Store>, grid, block, (size_t)kQSmemBytes, tmA, tmBq, p);
        case kEpiFc2Scatter:
            return cc.launch(gemm_w4a16_pair_kernel<kEpiFc2Scatter>, grid, block, (size_t)kQSmemBytes, tmA, tmBq,
                             p);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace moe
