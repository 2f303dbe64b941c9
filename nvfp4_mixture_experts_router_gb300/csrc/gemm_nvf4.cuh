// The grouped NVFP4 / MXFP8 GEMM engine as device-side building blocks:
// the pipeline configuration, the shared-memory carve-up, the one-time
// setup, the persistent tile loop of all roles (gemm_tiles) and the
// teardown.  gemm_nvf4.cu wraps them into one kernel per GEMM; the fused
// layer kernel (fused_layer.cu) runs the tile loop twice, FC1 then FC2, on
// the same pipeline.
// Grouped NVFP4 x NVFP4 GEMMs of the MoE layer on the 5th-generation tensor
// cores (tcgen05.mma kind::mxf4nvf4, block-scaled with UE4M3 scales per 16
// elements), with the FC1 and FC2 epilogues fused in.  The same engine runs
// the MXFP8 mode (KIND = 1: kind::mxf8f6f4, E4M3 elements, UE8M0 scales per
// 32): a 128-byte chunk of a row holds 256 E2M1 or 128 E4M3 elements, four
// 32-byte MMA steps either way; NVFP4 needs one 512-byte scale atom per MMA
// step and 128 rows, MXFP8 one per chunk (its four MMAs pick bytes 0-3 of
// each scale word through the scale-factor ids).
//
//   D[row, n] = sum_k A[row, k] * B_e[n, k]       (rows of expert e only)
//
// A (activations) are the permuted route rows, B the expert's prepared
// weights; each expert segment of A is padded to whole 128-row tiles
// [FlashInfer PR #4366, "Tests": padding and partial tiles], so every M tile
// belongs to exactly one expert (tile_expert).
//
// Kernel design (one persistent CTA per SM), tile 128 routes x BN weight
// rows, BN = 128 or 256, pipeline stage = 512 elements of K (two 128-byte
// chunks of every operand row):
//   warp 0      TMA producer: per stage ONE tensor copy of the A tile
//               (128 rows x 2 chunks, 32 KB) and ONE of the B tile (BN rows x
//               2 chunks), through 3-D tensor maps whose third dimension
//               walks the 128-byte chunks of a row (128-byte swizzle; each
//               chunk lands as its own swizzled [rows][128 B] tile), plus the
//               matching scale atoms of each operand (cp.async.bulk).  The
//               TMA unit costs about the same per copy instruction up to
//               32 KB (measured: 16 KB boxes ~66 GB/s per SM from L2, 32 KB
//               boxes ~131 GB/s), so two-chunk copies double the operand
//               bytes an SM can pull in.  Rows whose length is not a
//               multiple of 128 bytes use 2-D maps and one copy per chunk.
//   warps 2-5   scale writers, one per tensor-memory lane quadrant: once a
//               stage's scale atoms have landed (their own barrier, loaded
//               ahead of the operand tiles), every lane reads its 16-byte
//               atom row per k-block from shared memory and writes them with
//               tcgen05.st into the stage's tensor-memory slot; the four
//               quadrants together form the replicated layout the
//               block-scaled MMA reads (the same image tcgen05.cp .warpx4
//               would produce).  tcgen05.cp was measured at ~100 cycles of
//               copy-engine time per 512-byte atom, which capped a stage of
//               eight atoms at ~800 cycles whatever the memory traffic.
//   warp 1      allocates 512 tensor-memory columns; lane 0 issues, per
//               stage, eight 128xBNx64 block-scaled MMAs into an FP32
//               accumulator in tensor memory, then tcgen05.commit frees the
//               stage.
//   warps 6..   epilogue: tcgen05.ld of the accumulator (warp w reads lanes
//               32*(w%4)..+31, one output row per thread; with BN = 256 a
//               second group of four warps takes columns 128..255), fused
//               activation / scaling / requantization / scatter, then
//               release the accumulator.
// BN = 128 double-buffers the accumulator (epilogue of tile i overlaps the
// main loop of tile i+1); BN = 256 needs all 256 spare tensor-memory
// columns for one accumulator next to the scale slots and drains it with
// twice the epilogue warps instead.  A weight segment whose length is an odd
// multiple of 128 ends in a 128-wide tile (N = 128 MMAs).  Tiles are walked
// n-fastest so that concurrently running CTAs share the A tile and one
// expert's weights stay hot in L2.
// Every wait is bounded (1 s); a timeout sets a status bit and all roles
// drain and exit instead of hanging.
#pragma once
#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"

namespace moe {
namespace grouped {

constexpr int kBM = 128;
constexpr int kChunkBytes = 128;              // one 128-byte chunk = 256 E2M1 elements of a row
constexpr int kChunkBytesA = kBM * kChunkBytes;               // 16 KB
constexpr uint32_t kTmemCols = 512;

// BN = 128: stages of two chunks (3-stage ring); BN = 256: stages of one
// chunk (4-stage ring; its 256-row B box is already a 32 KB copy).  The ring
// turnaround (scale copies, scale writers, MMA commit) is a fixed latency per
// slot, so the deeper ring wins where the copies are large anyway (measured
// at K = 7168: 1087 us with four one-chunk stages, 1169 us with two
// two-chunk stages).
template <int BN, int KIND>
struct Cfg {
    static constexpr int kChunks = BN == 128 ? 2 : 1;            // chunks per pipeline stage
    static constexpr int kKbPerStage = 4 * kChunks;              // 32-byte MMA steps per stage
    static constexpr int kAtoms = KIND == 0 ? kKbPerStage : kChunks;   // scale atoms per 128 rows and stage
    static constexpr int kTileBytesA = kChunks * kChunkBytesA;
    static constexpr int kSfBytesA = kAtoms * 512;
    static constexpr int kStages = BN == 128 ? 3 : 4;
    static constexpr int kAccBufs = BN == 128 ? 2 : 1;
    static constexpr int kEpiWarps = BN == 128 ? 4 : 8;
    static constexpr int kSfWarps = 4;                           // scale writers, one per lane quadrant
    static constexpr int kEpiWarp0 = 2 + kSfWarps;
    static constexpr int kNumThreads = (kEpiWarp0 + kEpiWarps) * 32;
    static constexpr int kRowBlocks = BN / 128;                  // 128-row scale blocks of B
    static constexpr int kChunkBytesB = BN * kChunkBytes;
    static constexpr int kTileBytesB = kChunks * kChunkBytesB;
    static constexpr int kSfBytesB = kRowBlocks * kSfBytesA;
    static constexpr uint32_t kSfColBase = kAccBufs * BN;        // 256 either way
    static constexpr uint32_t kSfColsA = 4 * kAtoms;
    static constexpr uint32_t kSfColsB = 4 * kRowBlocks;         // per atom slot
    static constexpr uint32_t kSfColsPerStage = kSfColsA + kAtoms * kSfColsB;
    // FC2 epilogue staging (one block of 32 rows x kStgCols words per
    // epilogue warp; 8 KB either way)
    static constexpr int kStgCols = 64 / kEpiWarps;
    static constexpr int kStgBytes = kEpiWarps * 32 * kStgCols * 4;
    static constexpr int kSmemBytes =
        kStages * (kTileBytesA + kTileBytesB + kSfBytesA + kSfBytesB) + kStgBytes + 1024 + 256;
    static_assert(kSfColBase + kStages * kSfColsPerStage <= kTmemCols, "tensor memory budget");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct Smem {
    uint8_t* a;
    uint8_t* b;
    uint8_t* sfa;
    uint8_t* sfb;
    uint32_t* stg;
    uint64_t* full;
    uint64_t* sf_full;
    uint64_t* empty;
    uint64_t* sf_ready;
    uint64_t* acc_full;
    uint64_t* acc_empty;
    uint64_t* drain;
    uint32_t* tmem_holder;
    volatile int* abort;
};

template <int BN, int KIND>
__device__ __forceinline__ Smem carve(uint8_t* raw) {
    using C = Cfg<BN, KIND>;
    Smem s;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    s.a = base;
    s.b = s.a + C::kStages * C::kTileBytesA;
    s.sfa = s.b + C::kStages * C::kTileBytesB;
    s.sfb = s.sfa + C::kStages * C::kSfBytesA;
    s.stg = reinterpret_cast<uint32_t*>(s.sfb + C::kStages * C::kSfBytesB);
    uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(s.stg) + C::kStgBytes);
    s.full = bars;
    s.sf_full = bars + C::kStages;
    s.empty = bars + 2 * C::kStages;
    s.sf_ready = bars + 3 * C::kStages;
    s.acc_full = bars + 4 * C::kStages;
    s.acc_empty = s.acc_full + 2;
    s.drain = s.acc_empty + 2;
    s.tmem_holder = reinterpret_cast<uint32_t*>(s.drain + 1);
    s.abort = reinterpret_cast<volatile int*>(s.tmem_holder + 1);
    return s;
}


// Pipeline position of one role thread; carried from one gemm_tiles call to
// the next when a kernel runs several GEMMs on one pipeline.
// Tile index -> (M tile, N tile).  Default: N tiles fastest over the whole
// output width.  With slabs of n_slab N tiles (p.n_slab > 0), the width is
// walked slab by slab and every M tile runs within a slab before the next:
// the fused-finalize scatter then keeps adding into one slab of the output
// accumulator, which stays in L2 when the accumulator as a whole does not.
__device__ __forceinline__ void decode_tile(const GemmParams& p, int tile, int n_tiles, int num_m_tiles, int& m_tile,
                                            int& n_tile) {
    if (p.n_slab <= 0) {
        m_tile = tile / n_tiles;
        n_tile = tile % n_tiles;
        return;
    }
    const int per_slab = num_m_tiles * p.n_slab;
    const int slab = tile / per_slab, rem = tile % per_slab;
    const int width = min(p.n_slab, n_tiles - slab * p.n_slab);   // the last slab may be narrower
    m_tile = rem / width;
    n_tile = slab * p.n_slab + rem % width;
}

struct RingState {
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
};

// Barriers (thread 0) and tensor memory (warp 1); all threads then meet at
// a __syncthreads and read the tensor-memory base.
template <int BN, int KIND>
__device__ __forceinline__ uint32_t gemm_init(const Smem& s) {
    using C = Cfg<BN, KIND>;
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.sf_full[i], 1);
            mbar_init(&s.empty[i], 1);
            mbar_init(&s.sf_ready[i], C::kSfWarps * 32);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.acc_full[i], 1);
            mbar_init(&s.acc_empty[i], C::kEpiWarps * 32);
        }
        mbar_init(s.drain, 1);   // the MMA thread retires its MMAs into it
        *s.abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(s.tmem_holder, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    return *s.tmem_holder;
}

// One grouped GEMM over all M tiles (meta[1]) x N tiles, tiles walked
// n-fastest from blockIdx.x in steps of gridDim.x, every role of the CTA in
// its own branch.  Returns false when a wait gave up or a tile map entry was
// bad (the CTA's abort flag is then set).
template <int EPI, int BN, int KIND>
__device__ __forceinline__ bool gemm_tiles(const Smem& s, uint32_t tmem_base, const CUtensorMap* tmA,
                                           const CUtensorMap* tmB, const GemmParams& p, RingState& rs) {
    using C = Cfg<BN, KIND>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int num_m_tiles = p.meta[1];
    const int n_tiles = (p.n + BN - 1) / BN;
    const int total = num_m_tiles * n_tiles;
    const int row_bytes = KIND == 0 ? p.kdim / 2 : p.kdim;
    const int kblocks = row_bytes / 32;                       // 32-byte MMA steps
    constexpr int kKbPerStage = C::kKbPerStage, kChunks = C::kChunks, kAtoms = C::kAtoms;
    const int kstages = (kblocks + kKbPerStage - 1) / kKbPerStage;
    const int rb_per_expert = p.n / 128;
    const int row_chunks = (row_bytes + kChunkBytes - 1) / kChunkBytes;   // 128-byte chunks per row
    const int atoms = KIND == 0 ? kblocks : row_chunks;      // scale atoms per 128 rows over all of K

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_normal();
            // slabs: the activation rows are re-read once per slab; evict them
            // first so that the slab of the accumulator stays in L2
            const uint64_t pol_a = p.n_slab > 0 ? policy_evict_first() : pol;
            int stage = rs.stage;
            uint32_t phase = rs.phase;
            for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
                int m_tile, n_tile;
                decode_tile(p, tile, n_tiles, num_m_tiles, m_tile, n_tile);
                const int e = p.tile_expert[m_tile];
                if (e < 0 || e >= p.num_experts) {
                    atomicOr(p.status, kStatusBadExpert);
                    *s.abort = 1;
                    break;
                }
                const int nrb = min(C::kRowBlocks, rb_per_expert - n_tile * C::kRowBlocks);
                const int a_row = m_tile * kBM;
                const int b_row = e * p.n + n_tile * BN;
                const uint8_t* sfa_src = p.sfa + (size_t)m_tile * atoms * 512;
                const uint8_t* sfb_src =
                    p.sfb + ((size_t)e * rb_per_expert + (size_t)n_tile * C::kRowBlocks) * atoms * 512;
                for (int ks = 0; ks < kstages; ++ks) {
                    if (!mbar_wait(&s.empty[stage], phase ^ 1u, s.abort, p.status, kStatusTimeoutProducer)) return false;
                    if (p.debug_skip_first_stage && blockIdx.x == 0 && tile == (int)blockIdx.x && ks == 0) {
                        // test hook: nothing issued, nothing arrives on this
                        // stage's barriers; the consumers' bounded waits give up
                        if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
                        continue;
                    }
                    const int n_at = min(kAtoms, atoms - kAtoms * ks);
                    const uint32_t sf_bytes = (uint32_t)n_at * 512u;
                    // the small scale atoms first, on their own barrier, so the
                    // scale writers can start while the operand tiles are in flight
                    mbar_arrive_expect_tx(&s.sf_full[stage], (uint32_t)(1 + nrb) * sf_bytes);
                    bulk_load(s.sfa + stage * C::kSfBytesA, sfa_src + (size_t)ks * kAtoms * 512, sf_bytes,
                              &s.sf_full[stage], pol);
                    for (int rb = 0; rb < nrb; ++rb)
                        bulk_load(s.sfb + stage * C::kSfBytesB + rb * C::kSfBytesA,
                                  sfb_src + ((size_t)rb * atoms + (size_t)ks * kAtoms) * 512, sf_bytes,
                                  &s.sf_full[stage], pol);
                    uint8_t* a_dst = s.a + stage * C::kTileBytesA;
                    uint8_t* b_dst = s.b + stage * C::kTileBytesB;
                    const int c0 = kChunks * ks;
                    if (p.chunk_maps) {
                        // one copy per operand; a chunk past the row end is filled
                        // with zeros and skipped by the MMAs
                        mbar_arrive_expect_tx(&s.full[stage], C::kTileBytesA + C::kTileBytesB);
                        tma_load_3d(a_dst, tmA, &s.full[stage], 0, a_row, c0, pol_a);
                        tma_load_3d(b_dst, tmB, &s.full[stage], 0, b_row, c0, pol);
                    } else {
                        // rows of 64 + 128 j bytes: one 2-D copy per chunk that
                        // starts inside the row
                        const int nch = min(kChunks, row_chunks - c0);
                        mbar_arrive_expect_tx(&s.full[stage], (uint32_t)nch * (kChunkBytesA + C::kChunkBytesB));
                        for (int c = 0; c < nch; ++c) {
                            tma_load_2d(a_dst + c * kChunkBytesA, tmA, &s.full[stage], (c0 + c) * kChunkBytes, a_row,
                                        pol_a);
                            tma_load_2d(b_dst + c * C::kChunkBytesB, tmB, &s.full[stage], (c0 + c) * kChunkBytes,
                                        b_row, pol);
                        }
                    }
                    if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
                }
            }
            rs.stage = stage;
            rs.phase = phase;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = rs.stage;
            uint32_t phase = rs.phase;
            int acc = rs.acc;
            uint32_t acc_phase = rs.acc_phase;
            for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
                int m_tile, n_tile;
                decode_tile(p, tile, n_tiles, num_m_tiles, m_tile, n_tile);
                const int width = min(BN, p.n - n_tile * BN);
                const uint32_t idesc = idesc_nvf4(kBM, width);   // NVFP4 (MXFP8 builds its own per MMA)
                if (!mbar_wait(&s.acc_empty[acc], acc_phase ^ 1u, s.abort, p.status, kStatusTimeoutMma)) return false;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int ks = 0; ks < kstages; ++ks) {
                    if (!mbar_wait(&s.full[stage], phase, s.abort, p.status, kStatusTimeoutMma)) return false;
                    const int nkb = min(kKbPerStage, kblocks - kKbPerStage * ks);
                    const uint32_t sfa_t = tmem_base + C::kSfColBase + (uint32_t)stage * C::kSfColsPerStage;
                    const uint32_t sfb_t = sfa_t + C::kSfColsA;
                    // the scale writers' stores for this stage are done
                    if (!mbar_wait(&s.sf_ready[stage], phase, s.abort, p.status, kStatusTimeoutMma)) return false;
                    tc_fence_after();
                    // chunk j / 4, then 32 bytes (64 E2M1 / 32 E4M3) along K inside
                    // its swizzled 128-byte rows; descriptor start addresses
                    // count 16-byte units
                    const uint64_t adesc0 = sdesc_kmajor_sw128(smem_u32(s.a + stage * C::kTileBytesA));
                    const uint64_t bdesc0 = sdesc_kmajor_sw128(smem_u32(s.b + stage * C::kTileBytesB));
                    auto issue = [&](int j) {
                        const int c = j >> 2, jj = j & 3;
                        const uint64_t adesc = adesc0 + (uint64_t)c * (kChunkBytesA / 16) + 2u * jj;
                        const uint64_t bdesc = bdesc0 + (uint64_t)c * (C::kChunkBytesB / 16) + 2u * jj;
                        if (KIND == 0)
                            tc_mma_nvf4(d_tmem, adesc, bdesc, idesc, sfa_t + 4 * j, sfb_t + C::kSfColsB * j,
                                        (ks | j) != 0);
                        else
                            tc_mma_mxf8(d_tmem, adesc, bdesc, idesc_mxf8(kBM, width, jj), sfa_t + 4 * c,
                                        sfb_t + C::kSfColsB * c, (ks | j) != 0);
                    };
                    if (nkb == kKbPerStage) {
                        // a full stage, unrolled: constant offsets of the stage's
                        // descriptors, a few instructions per MMA
#pragma unroll
                        for (int j = 0; j < kKbPerStage; ++j) issue(j);
                    } else {
                        for (int j = 0; j < nkb; ++j) issue(j);
                    }
                    tc_commit(&s.empty[stage]);
                    if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
                }
                tc_commit(&s.acc_full[acc]);
                if (++acc == C::kAccBufs) { acc = 0; acc_phase ^= 1u; }
            }
            rs.stage = stage;
            rs.phase = phase;
            rs.acc = acc;
            rs.acc_phase = acc_phase;
        }
    } else if (warp < C::kEpiWarp0) {
        // scale writer for lane quadrant warp % 4: lane l holds row l of each
        // 512-byte atom (4 words = the 4 column slots of rows l, l+32, l+64, l+96)
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        int stage = rs.stage;
        uint32_t phase = rs.phase;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            for (int ks = 0; ks < kstages; ++ks) {
                // warp-uniform outcome: tcgen05.st below is a warp-collective instruction
                if (!__all_sync(0xffffffffu,
                                mbar_wait(&s.sf_full[stage], phase, s.abort, p.status, kStatusTimeoutMma)))
                    return false;
                const uint32_t sfa_t = tmem_base + C::kSfColBase + (uint32_t)stage * C::kSfColsPerStage;
                const uint32_t sfb_t = sfa_t + C::kSfColsA;
                // A scales: atom a -> columns 4a..4a+3; B scales: atom a, row
                // block rb -> columns 4 (a * kRowBlocks + rb) .. +3
                {
                    uint32_t ra[4 * kAtoms];
#pragma unroll
                    for (int a = 0; a < kAtoms; ++a) {
                        const uint4 v = *reinterpret_cast<const uint4*>(s.sfa + stage * C::kSfBytesA + a * 512 +
                                                                        lane * 16);
                        ra[4 * a] = v.x; ra[4 * a + 1] = v.y; ra[4 * a + 2] = v.z; ra[4 * a + 3] = v.w;
                    }
                    tmem_st_n<4 * kAtoms>(sfa_t + lane_off, ra);
                    uint32_t rb_[4 * kAtoms * C::kRowBlocks];
#pragma unroll
                    for (int a = 0; a < kAtoms; ++a)
#pragma unroll
                        for (int rb = 0; rb < C::kRowBlocks; ++rb) {
                            const uint4 v = *reinterpret_cast<const uint4*>(
                                s.sfb + stage * C::kSfBytesB + rb * C::kSfBytesA + a * 512 + lane * 16);
                            const int o = 4 * (a * C::kRowBlocks + rb);
                            rb_[o] = v.x; rb_[o + 1] = v.y; rb_[o + 2] = v.z; rb_[o + 3] = v.w;
                        }
                    tmem_st_n<4 * kAtoms * C::kRowBlocks>(sfb_t + lane_off, rb_);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&s.sf_ready[stage]);
                if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
            }
        }
        rs.stage = stage;
        rs.phase = phase;
    } else {
        const int q = warp & 3;                    // tensor-memory lane quadrant of this warp
        const int half = (warp - C::kEpiWarp0) >> 2;   // which 128 accumulator columns (BN = 256)
        int acc = rs.acc;
        uint32_t acc_phase = rs.acc_phase;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            int m_tile, n_tile;
            decode_tile(p, tile, n_tiles, num_m_tiles, m_tile, n_tile);
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
            const int width = min(BN, p.n - n_tile * BN);
            if (half * 128 < width) {
                const uint32_t taddr =
                    tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN + half * 128);
                const int vtile = n_tile * C::kRowBlocks + half;   // index of this 128-column slice
                if (EPI == kEpiFc1Quant || EPI == kEpiFc1F32 || EPI == kEpiFc1Mx)
                    epilogue_fc1<EPI>(p, taddr, row, meta, vtile);
                else
                    epilogue_fc2<EPI, C::kStgCols>(p, taddr, row, meta, vtile,
                                                   s.stg + (warp - C::kEpiWarp0) * 32 * C::kStgCols);
            }
            tc_fence_before();
            mbar_arrive(&s.acc_empty[acc]);
            if (++acc == C::kAccBufs) { acc = 0; acc_phase ^= 1u; }
        }
        rs.acc = acc;
        rs.acc_phase = acc_phase;
    }
    return *s.abort == 0;
}

// After an abort, let in-flight copies land and retire every issued MMA and
// tensor-memory store; then (every thread) free the tensor memory.
template <int BN, int KIND>
__device__ __forceinline__ void gemm_drain(const Smem& s, unsigned int* status) {
    using C = Cfg<BN, KIND>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile int no_abort = 0;
    if (*s.abort) {
        if (warp == 1 && lane == 0) {
            tc_commit(s.drain);
            mbar_wait(s.drain, 0, &no_abort, status, kStatusTimeoutMma);
        }
        if (warp >= 2 && warp < C::kEpiWarp0) tmem_st_wait();   // scale writers' stores in flight
        for (int i = 0; i < 100; ++i) __nanosleep(10000);
    }
}

__device__ __forceinline__ void gemm_free_tmem(uint32_t tmem_base) {
    if ((threadIdx.x >> 5) == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace grouped
}  // namespace moe
