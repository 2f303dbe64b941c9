// Grouped NVFP4 x NVFP4 GEMMs on CTA pairs: the same products and fused
// epilogues as gemm_nvf4.cu, computed by tcgen05.mma.cta_group::2 with a
// 256 x 256 tile per pair of SMs.
//
// Why pairs: the L2 -> SM copy rate of one SM's TMA ring is the limit of the
// single-CTA kernel at compute-bound shapes (measured on GB300: about 148
// GB/s per SM with all SMs loading, while a 128 x 256 tile needs about 218
// GB/s to keep the block-scaled MMA busy).  With the M = 256 pair MMA each SM
// holds its own 128 A rows and half of the 256 B rows, so it loads a third
// fewer operand bytes per FLOP (about 153 GB/s at the full MMA rate).
//
// Pair tile: two consecutive 128-row M tiles of ONE expert (the scan lists
// them in tile_pair: (first << 1) | has_second) x 256 weight rows.  CTA rank 0
// (even) holds the first M tile, B rows 0..127 of the tile and accumulator
// rows 0..127; rank 1 the second M tile, B rows 128..255 and accumulator rows
// 128..255 (an expert with an odd number of M tiles leaves rank 1 of its
// last pair loading the first tile again and discarding its rows).  Both
// CTAs hold the B scales of all 256 rows in tensor memory, as the pair MMA
// requires.
//
// Hand-off between the two CTAs, without a relay thread:
//   * operands: each CTA's producer copies its own A rows and B half with
//     cp.async.bulk.tensor.cta_group::2 whose completion is counted on the
//     stage barrier of rank 0 (rank 0 announces the bytes of both CTAs);
//   * scales: each CTA's four scale writers store their own tensor memory
//     (tcgen05.st) and arrive, one lane per warp, on rank 0's sf_ready
//     barrier (eight arrivals per stage);
//   * rank 0's MMA thread issues the pair MMAs and commits each stage to the
//     empty barriers of both CTAs (multicast), the finished accumulator to
//     both acc_full barriers;
//   * every epilogue warp of both CTAs releases the accumulator on rank 0's
//     acc_empty (sixteen arrivals) as soon as it has copied its 32 rows x 128
//     columns into registers; the activation, quantization and stores of
//     that tile then run while the MMAs of the next tile fill the
//     accumulator again.  (A second 256-column accumulator does not fit
//     beside the scale slots in the 512 tensor-memory columns; with a
//     single one that is drained in place, the MMA thread spent 26 % of the
//     K = 7168 FC1 and half of the scatter FC2 waiting for the epilogue.)
// Operand stages hold CH = 2 128-byte K chunks of every operand row (one
// 32 KB copy per operand and CTA: the copy rate of an SM's TMA ring grows
// with the bytes per stage, ~100 GB/s at 16-32 KB, ~148 GB/s at 64 KB), three
// of them; the scale atoms of a stage go through a separate two-deep ring
// (shared memory and tensor-memory slots), refilled as soon as the writers
// have read a slot and the MMAs two stages back have finished.
//
// Roles per CTA (512 threads, four warpgroups): warpgroup 0 = warp 0
// producer of the operand copies, warp 1 tensor-memory allocation (both
// CTAs together) and, in rank 0, the MMA issuer, warp 2 producer of the
// scale-atom copies, warp 3 idle; warpgroup 1 = the four scale
// writers; warpgroups 2-3 = the epilogue over this CTA's 128 rows (two groups
// of four warps, 128 accumulator columns each).  The launch gives every
// thread 128 registers; warpgroups 0 and 1 hand theirs down to 48 and 80 so
// that the epilogue warps can hold a 128-column slice (192 each; the split
// is the same on each of the four SM sub-partitions, which hold one warp of
// every warpgroup).
// Every wait is bounded (1 s); a timeout sets a status bit, marks both CTAs
// aborted, and all roles drain and reach the final pair barrier.
#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"
#include "pair_tiles.cuh"

namespace moe {

namespace {

constexpr int kPRows = 128;                      // A rows per CTA (256 per pair)
constexpr int kPN = 256;                         // weight rows per pair tile (128 per CTA)
constexpr int kPSfWarps = 4;
constexpr int kPSfWarp0 = 4;                     // warpgroup 1
constexpr int kPEpiWarp0 = kPSfWarp0 + kPSfWarps;
constexpr int kPEpiWarps = 8;                    // warpgroups 2 and 3
constexpr int kPThreads = (kPEpiWarp0 + kPEpiWarps) * 32;
// Register split (setmaxnreg, per warpgroup) within the launch's pool of
// kPThreads x kPRegsLaunch; the host refuses to launch if the compiled
// kernel's count differs from kPRegsLaunch.
constexpr uint32_t kPRegsLaunch = 65536 / kPThreads;
constexpr uint32_t kPRegsCtl = 48;
constexpr uint32_t kPRegsSf = 80;
constexpr uint32_t kPRegsEpi = 192;
static_assert(kPThreads == 512, "four warpgroups");
static_assert(128 * (kPRegsCtl + kPRegsSf) + 256 * kPRegsEpi <= kPThreads * kPRegsLaunch, "register split");
constexpr uint32_t kPTmemCols = 512;
constexpr uint32_t kPSfCol0 = kPN;               // accumulator: columns 0..255
// Two rings: operand stages (CH = 2 128-byte K chunks of every operand row)
// and scale stages (the same K range), the latter two deep in both shared and
// tensor memory, which is what bounds them.  The FC2 epilogues stage their
// row segments through shared memory (64-byte segments: 16 words per row and
// warp); they get two operand stages, the FC1 epilogues (no staging) three.
template <int EPI>
struct PCfg {
    static constexpr bool kFc2 = EPI == kEpiFc2Store || EPI == kEpiFc2Scatter;
    static constexpr int kCh = 2;                            // 128-byte K chunks per operand stage
    static constexpr int kKb = 4 * kCh;                      // 64-element MMA steps per stage
    static constexpr int kTileA = kPRows * 128 * kCh;        // own 128 A rows
    static constexpr int kTileB = (kPN / 2) * 128 * kCh;     // own half of the B rows
    static constexpr int kSfA = kKb * 512;                   // own A rows' scale atoms
    static constexpr int kSfB = 2 * kKb * 512;               // all 256 B rows' scale atoms
    static constexpr int kSfStages = 2;
    static constexpr int kStages = kFc2 ? 2 : 3;             // operand stages
    // epilogue staging, words per row: FC2 16; the FC1 FP32 store 8 (what
    // fits beside its three stages); the FC1 requantization none (staging
    // its 16-byte code rows was measured slower)
    static constexpr int kStgCols = kFc2 ? 16 : (EPI == kEpiFc1F32 ? 8 : 0);
    static constexpr int kStgBytes = kPEpiWarps * 32 * kStgCols * 4;
    static constexpr uint32_t kSfColsA = 4 * kKb;
    static constexpr uint32_t kSfColsB = 8 * kKb;
    static constexpr uint32_t kSfColsStage = kSfColsA + kSfColsB;
    static constexpr int kSmemBytes =
        kStages * (kTileA + kTileB) + kSfStages * (kSfA + kSfB) + kStgBytes + 1024 + 512;
    static_assert(kPSfCol0 + kSfStages * kSfColsStage <= kPTmemCols, "tensor memory budget");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct PairSmem {
    uint8_t* a;
    uint8_t* b;
    uint8_t* sfa;
    uint8_t* sfb;
    uint32_t* stg;
    uint64_t* full;        // [kStages] rank 0: both CTAs' operand bytes of a stage
    uint64_t* empty;       // [kStages] both CTAs: the stage's MMAs are done
    uint64_t* sf_full;     // [kSfStages] this CTA's scale atoms of a stage landed
    uint64_t* sf_free;     // [kSfStages] this CTA's scale writers have read them
    uint64_t* sf_ready;    // [kSfStages] rank 0: both CTAs' scale writers are done
    uint64_t* acc_full;
    uint64_t* acc_empty;   // rank 0: both CTAs' epilogues released the accumulator
    uint64_t* drain;
    uint32_t* tmem_holder;
    volatile int* abort;
};

template <int EPI>
__device__ __forceinline__ PairSmem carve_pair(uint8_t* raw) {
    using PC = PCfg<EPI>;
    PairSmem s;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    s.a = base;
    s.b = s.a + PC::kStages * PC::kTileA;
    s.sfa = s.b + PC::kStages * PC::kTileB;
    s.sfb = s.sfa + PC::kSfStages * PC::kSfA;
    s.stg = reinterpret_cast<uint32_t*>(s.sfb + PC::kSfStages * PC::kSfB);
    uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(s.stg) + PC::kStgBytes);
    s.full = bars;
    s.empty = bars + PC::kStages;
    s.sf_full = bars + 2 * PC::kStages;
    s.sf_free = s.sf_full + PC::kSfStages;
    s.sf_ready = s.sf_free + PC::kSfStages;
    s.acc_full = s.sf_ready + PC::kSfStages;
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
    using PC = PCfg<EPI>;
    extern __shared__ uint8_t smem_raw[];
    const PairSmem s = carve_pair<EPI>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_cta_rank();          // 0: issues the pair MMAs
    const int pair_slot = blockIdx.x >> 1, pair_slots = gridDim.x >> 1;
    volatile int no_abort = 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < PC::kStages; ++i) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.empty[i], 1);
        }
        for (int i = 0; i < PC::kSfStages; ++i) {
            mbar_init(&s.sf_full[i], 1);
            mbar_init(&s.sf_free[i], kPSfWarps);
            mbar_init(&s.sf_ready[i], 2 * kPSfWarps);
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
    // cross-CTA copy, arrival or pair MMA
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = *s.tmem_holder;

    pdl_wait();  // A operand, tile maps and counts come from earlier kernels

    const int num_pairs = p.meta[2];
    const int num_m_tiles = p.meta[1];
    const int n_tiles = p.n / kPN;
    const int total = num_pairs * n_tiles;
    const int kblocks = p.kdim / 64;                           // 64-element MMA steps = scale atoms per 128 rows
    const int kstages = (kblocks + PC::kKb - 1) / PC::kKb;
    const int row_chunks = (p.kdim / 2 + 127) / 128;           // 128-byte chunks per row
    const int rb_per_expert = p.n / 128;

    if (warp < kPSfWarp0) {
        regs_release<kPRegsCtl>();
        if (warp == 0 || warp == 2) {
            // warp 0: operand copies; warp 2: scale-atom copies, on their own
            // ring, so that neither waits behind the other's free slots
            if (lane == 0) {
                const bool sf_role = warp == 2;
                const uint64_t pol = policy_evict_normal();
                // slabs: the activation rows are re-read once per slab; evict them
                // first so that the slab of the accumulator stays in L2
                const uint64_t pol_a = p.n_slab > 0 ? policy_evict_first() : pol;
                const uint32_t full0 = cluster_map(s.full, 0);      // rank 0's stage barriers
                int stage = 0, sfs = 0;
                uint32_t phase = 0, sfp = 0;
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
                    const int a_row = ld_m * kPRows;
                    const int b_row = e * p.n + n_tile * kPN + (int)rank * (kPN / 2);
                    const uint8_t* sfa_src = p.sfa + (size_t)ld_m * kblocks * 512;
                    const uint8_t* sfb_src = p.sfb + ((size_t)e * rb_per_expert + (size_t)n_tile * 2) * kblocks * 512;
                    for (int ks = 0; ks < kstages; ++ks) {
                        if (sf_role) {
                            const int nkb = min(PC::kKb, kblocks - PC::kKb * ks);
                            const uint32_t sf_bytes = (uint32_t)nkb * 512u;
                            // this CTA's scale atoms (its own A rows, all 256 B
                            // rows) into the scale ring once the writers have
                            // read that slot
                            if (!mbar_wait(&s.sf_free[sfs], sfp ^ 1u, s.abort, p.status, kStatusTimeoutProducer))
                                goto done;
                            mbar_arrive_expect_tx(&s.sf_full[sfs], 3u * sf_bytes);
                            bulk_load(s.sfa + sfs * PC::kSfA, sfa_src + (size_t)ks * PC::kKb * 512, sf_bytes,
                                      &s.sf_full[sfs], pol);
                            for (int rb = 0; rb < 2; ++rb)
                                bulk_load(s.sfb + sfs * PC::kSfB + rb * PC::kSfA,
                                          sfb_src + ((size_t)rb * kblocks + (size_t)ks * PC::kKb) * 512, sf_bytes,
                                          &s.sf_full[sfs], pol);
                            if (++sfs == PC::kSfStages) { sfs = 0; sfp ^= 1u; }
                            continue;
                        }
                        // completed by rank 0's commit: acquire at cluster scope
                        if (!mbar_wait<true>(&s.empty[stage], phase ^ 1u, s.abort, p.status, kStatusTimeoutProducer))
                            goto done;
                        // operands: counted on rank 0's barrier, which rank 0
                        // announces for both CTAs
                        uint8_t* a_dst = s.a + stage * PC::kTileA;
                        uint8_t* b_dst = s.b + stage * PC::kTileB;
                        const int c0 = PC::kCh * ks;
                        const uint32_t bar = full0 + (uint32_t)stage * 8u;
                        if (p.chunk_maps) {
                            if (rank == 0) mbar_arrive_expect_tx(&s.full[stage], 2u * (PC::kTileA + PC::kTileB));
                            tma_load_3d_pair(a_dst, &tmA, bar, 0, a_row, c0, pol_a);
                            tma_load_3d_pair(b_dst, &tmB, bar, 0, b_row, c0, pol);
                        } else {
                            const int nch = min(PC::kCh, row_chunks - c0);
                            if (rank == 0)
                                mbar_arrive_expect_tx(&s.full[stage], 2u * (uint32_t)nch * (kPRows * 128 + (kPN / 2) * 128));
                            for (int c = 0; c < nch; ++c) {
                                tma_load_2d_pair(a_dst + c * kPRows * 128, &tmA, bar, (c0 + c) * 128, a_row, pol_a);
                                tma_load_2d_pair(b_dst + c * (kPN / 2) * 128, &tmB, bar, (c0 + c) * 128, b_row, pol);
                            }
                        }
                        if (++stage == PC::kStages) { stage = 0; phase ^= 1u; }
                    }
                }
            }
        } else if (warp == 1) {
            if (lane == 0 && rank == 0) {
                const uint32_t idesc = idesc_nvf4(2 * kPRows, kPN);
                int stage = 0, sfs = 0;
                uint32_t phase = 0, sfp = 0, acc_phase = 0;
                for (int tile = pair_slot; tile < total; tile += pair_slots) {
                    if (!mbar_wait<true>(s.acc_empty, acc_phase ^ 1u, s.abort, p.status, kStatusTimeoutMma)) goto done;
                    tc_fence_after();
                    for (int ks = 0; ks < kstages; ++ks) {
                        if (!mbar_wait<true>(&s.full[stage], phase, s.abort, p.status, kStatusTimeoutMma)) goto done;
                        if (!mbar_wait<true>(&s.sf_ready[sfs], sfp, s.abort, p.status, kStatusTimeoutMma)) goto done;
                        tc_fence_after();
                        const int nkb = min(PC::kKb, kblocks - PC::kKb * ks);
                        const uint32_t sfa_t = tmem_base + kPSfCol0 + (uint32_t)sfs * PC::kSfColsStage;
                        const uint32_t sfb_t = sfa_t + PC::kSfColsA;
                        const uint64_t adesc = sdesc_kmajor_sw128(smem_u32(s.a + stage * PC::kTileA));
                        const uint64_t bdesc = sdesc_kmajor_sw128(smem_u32(s.b + stage * PC::kTileB));
                        // descriptor start addresses count 16-byte units: a chunk of
                        // 128 rows x 128 bytes is 1024 of them, a 32-byte K step 2
                        constexpr uint64_t kChunkA = kPRows * 128 / 16, kChunkB = (kPN / 2) * 128 / 16;
                        if (nkb == PC::kKb) {
                            // a full stage, unrolled: every operand of the eight MMAs
                            // is a constant offset of the stage's descriptors, so the
                            // issuing thread spends a few instructions per MMA
    #pragma unroll
                            for (int j = 0; j < PC::kKb; ++j)
                                tc_mma_nvf4_pair(tmem_base, adesc + (uint64_t)(j >> 2) * kChunkA + 2u * (j & 3),
                                                 bdesc + (uint64_t)(j >> 2) * kChunkB + 2u * (j & 3), idesc,
                                                 sfa_t + 4 * j, sfb_t + 8 * j, (ks | j) != 0);
                        } else {
                            for (int j = 0; j < nkb; ++j)
                                tc_mma_nvf4_pair(tmem_base, adesc + (uint64_t)(j >> 2) * kChunkA + 2u * (j & 3),
                                                 bdesc + (uint64_t)(j >> 2) * kChunkB + 2u * (j & 3), idesc,
                                                 sfa_t + 4 * j, sfb_t + 8 * j, (ks | j) != 0);
                        }
                        tc_commit_pair_mc(&s.empty[stage], 0x3);
                        if (++stage == PC::kStages) { stage = 0; phase ^= 1u; }
                        if (++sfs == PC::kSfStages) { sfs = 0; sfp ^= 1u; }
                    }
                    tc_commit_pair_mc(s.acc_full, 0x3);
                    acc_phase ^= 1u;
                }
            }
        }  // warp 3: no role
    } else if (warp < kPEpiWarp0) {
        regs_release<kPRegsSf>();
        // scale writer for lane quadrant warp % 4: the stage's A atoms into
        // columns 4j..4j+3 of its slot, the B atoms of MMA step j (row block
        // rb) into columns 8j + 4rb .. +3 of the B part
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t ready0 = cluster_map(s.sf_ready, 0);
        int sfs = 0, es = 0;                  // scale slot; operand stage of the MMAs two stages back
        uint32_t sfp = 0, ep = 0;
        long long n = 0;                      // stages written so far
        for (int tile = pair_slot; tile < total; tile += pair_slots) {
            for (int ks = 0; ks < kstages; ++ks, ++n) {
                // the tensor-memory scale slot is free once the MMAs of the
                // stage that used it (two stages back) are done: their
                // operand stage's empty barrier (completed by rank 0's
                // commit, hence cluster scope; it cannot run two phases ahead
                // of this writer, whose next stage those MMAs would need)
                bool ok = mbar_wait(&s.sf_full[sfs], sfp, s.abort, p.status, kStatusTimeoutMma);
                if (ok && n >= PC::kSfStages) {
                    ok = mbar_wait<true>(&s.empty[es], ep, s.abort, p.status, kStatusTimeoutMma);
                    if (++es == PC::kStages) { es = 0; ep ^= 1u; }
                }
                // warp-uniform outcome: tcgen05.st below is a warp-collective instruction
                if (!__all_sync(0xffffffffu, ok)) goto done;
                const uint32_t sfa_t = tmem_base + kPSfCol0 + (uint32_t)sfs * PC::kSfColsStage;
                const uint32_t sfb_t = sfa_t + PC::kSfColsA;
#pragma unroll
                for (int g = 0; g < PC::kKb / 4; ++g) {
                    uint32_t ra[16];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint4 v =
                            *reinterpret_cast<const uint4*>(s.sfa + sfs * PC::kSfA + (4 * g + j) * 512 + lane * 16);
                        ra[4 * j] = v.x; ra[4 * j + 1] = v.y; ra[4 * j + 2] = v.z; ra[4 * j + 3] = v.w;
                    }
                    tmem_st16(sfa_t + 16 * g + lane_off, ra);
                    uint32_t rb_[32];
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int rb = 0; rb < 2; ++rb) {
                            const uint4 v = *reinterpret_cast<const uint4*>(s.sfb + sfs * PC::kSfB + rb * PC::kSfA +
                                                                            (4 * g + j) * 512 + lane * 16);
                            rb_[8 * j + 4 * rb] = v.x; rb_[8 * j + 4 * rb + 1] = v.y;
                            rb_[8 * j + 4 * rb + 2] = v.z; rb_[8 * j + 4 * rb + 3] = v.w;
                        }
                    tmem_st32(sfb_t + 32 * g + lane_off, rb_);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&s.sf_free[sfs]);
                    if (rank == 0) mbar_arrive(&s.sf_ready[sfs]);
                    else mbar_arrive_cluster(ready0 + (uint32_t)sfs * 8u);
                }
                if (++sfs == PC::kSfStages) { sfs = 0; sfp ^= 1u; }
            }
        }
    } else {
        regs_claim<kPRegsEpi>();
        const int q = warp & 3;                            // tensor-memory lane quadrant of this warp
        const int half = (warp - kPEpiWarp0) >> 2;         // accumulator columns 0..127 or 128..255
        const uint32_t release = cluster_map(s.acc_empty, 0);
        uint32_t* stg = s.stg + (warp - kPEpiWarp0) * 32 * PC::kStgCols;
        uint32_t acc_phase = 0;
        for (int tile = pair_slot; tile < total; tile += pair_slots) {
            int m_tile, m0, n_tile;
            decode_pair(p, tile, n_tiles, num_pairs, rank, m_tile, m0, n_tile);
            const int e = (m0 >= 0 && m0 < num_m_tiles) ? p.tile_expert[m0] : -1;
            if (e < 0 || e >= p.num_experts || m_tile >= num_m_tiles) break;
            // the row's epilogue scalars, loaded while the main loop runs
            const int row = m_tile >= 0 ? m_tile * kPRows + q * 32 + lane : -1;
            const EpiRow meta = epi_row<EPI>(p, row, e);
            // warp-uniform outcome: tcgen05.ld below is a warp-collective instruction
            if (!__all_sync(0xffffffffu,
                            mbar_wait<true>(s.acc_full, acc_phase, s.abort, p.status, kStatusTimeoutEpilogue)))
                break;
            tc_fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(half * 128);
            const int vtile = n_tile * 2 + half;           // index of this 128-column slice
            // copy the slice out and hand the accumulator back at once
            float acc[128];
            if (m_tile >= 0) {
                float a0[32], a1[32], a2[32], a3[32];
                tmem_ld32(taddr, a0);
                tmem_ld32(taddr + 32, a1);
                tmem_ld32(taddr + 64, a2);
                tmem_ld32(taddr + 96, a3);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    acc[i] = a0[i];
                    acc[32 + i] = a1[i];
                    acc[64 + i] = a2[i];
                    acc[96 + i] = a3[i];
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (rank == 0) mbar_arrive(s.acc_empty);
                else mbar_arrive_cluster(release);
            }
            acc_phase ^= 1u;
            if (m_tile >= 0) {
                if (EPI == kEpiFc1Quant || EPI == kEpiFc1F32)
                    epilogue_fc1_held<EPI, PC::kStgCols>(p, acc, row, meta, vtile, stg);
                else epilogue_fc2_held<EPI, PC::kStgCols>(p, acc, row, meta, vtile, stg);
            }
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
        if (warp >= kPSfWarp0 && warp < kPEpiWarp0) tmem_st_wait();
        for (int i = 0; i < 100; ++i) __nanosleep(10000);
    }
    tc_fence_before();
    __syncthreads();
    // neither CTA frees tensor memory or leaves (its shared memory is an
    // operand of the other CTA's MMAs and copies complete on its barriers)
    // before both are done
    cluster_sync_all();
    pdl_launch_dependents();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kPTmemCols);
    }
}

namespace {
int g_pair_grid[64] = {};

template <int EPI>
cudaError_t set_pair_smem() {
    // the register split assumes the launch's pool of 128 registers a
    // thread; with fewer, the epilogue's increase would never be granted
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, gemm_nvf4_pair_kernel<EPI>);
    if (e != cudaSuccess) return e;
    if ((uint32_t)((fa.numRegs + 7) / 8 * 8) != kPRegsLaunch) return cudaErrorInvalidKernelImage;
    return cudaFuncSetAttribute(gemm_nvf4_pair_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                PCfg<EPI>::kSmemBytes);
}
}  // namespace

int gemm_pair_chunks() { return PCfg<kEpiFc1Quant>::kCh; }

cudaError_t setup_gemm_pair_kernels(int device, int num_sms) {
    cudaError_t e;
    if ((e = set_pair_smem<kEpiFc1Quant>())) return e;
    if ((e = set_pair_smem<kEpiFc1F32>())) return e;
    if ((e = set_pair_smem<kEpiFc2Store>())) return e;
    if ((e = set_pair_smem<kEpiFc2Scatter>())) return e;
    // persistent grid: as many CTA pairs as can be resident at once
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(num_sms / 2 * 2));
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = PCfg<kEpiFc1Quant>::kSmemBytes;
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

int gemm_pair_grid(int device) { return (device >= 0 && device < 64) ? g_pair_grid[device] : 0; }

cudaError_t launch_gemm_nvf4_pair(const LaunchCtx& c, int epilogue, const CUtensorMap& tmA, const CUtensorMap& tmB,
                                  const GemmParams& p, int device) {
    if (device < 0 || device >= 64 || g_pair_grid[device] < 2) return cudaErrorInvalidValue;
    LaunchCtx cc = c;
    cc.cluster = 2;
    const dim3 grid((unsigned)g_pair_grid[device]), block(kPThreads);
#define MOE_PAIR_LAUNCH(E) \
    cc.launch(gemm_nvf4_pair_kernel<E>, grid, block, (size_t)PCfg<E>::kSmemBytes, tmA, tmB, p)
    switch (epilogue) {
        case kEpiFc1Quant: return MOE_PAIR_LAUNCH(kEpiFc1Quant);
        case kEpiFc1F32: return MOE_PAIR_LAUNCH(kEpiFc1F32);
        case kEpiFc2Store: return MOE_PAIR_LAUNCH(kEpiFc2Store);
        case kEpiFc2Scatter: return MOE_PAIR_LAUNCH(kEpiFc2Scatter);
        default: return cudaErrorInvalidValue;
    }
#undef MOE_PAIR_LAUNCH
}

}  // namespace moe
