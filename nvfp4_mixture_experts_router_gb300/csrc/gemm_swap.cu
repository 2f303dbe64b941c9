// Grouped NVFP4 GEMMs of the MoE layer with the operands swapped: the
// expert's weights are the MMA's M side (128 rows per operand) and the
// expert's routes its N side (64 rows per tile), for experts that hold few
// routes.
//
//   D^T[w, r] = sum_k W_e[w, k] * X[r, k]         (r: routes of expert e)
//
// Why: the standard orientation loads a 128-row activation tile per stage
// whatever the expert's route count (each expert segment is padded to whole
// 128-row tiles), so at a few dozen routes per expert half of every
// pipeline slot carries padding, and the GEMM, bound by how many weight
// bytes its slots keep in flight, streams weights well below the HBM rate.
// Here a slot holds 32 KB of weights and 8 KB of route rows (one 128-byte K
// chunk each), four slots keep 128 KB of weights in flight per SM (96 KB in
// the standard ring), and only the 64-route halves that hold routes are
// tiled (the permutation scan lists them).
//
// Tile = two weight operands of 128 rows x one 64-route half of an M tile.
// The operands come from one 3-D tensor map over the prepared weights viewed
// as [128-row blocks][128 rows][K bytes] with a box of 64 rows x 2 blocks:
// operand 0 = rows 0-63 of blocks 2t and 2t+1, operand 1 = rows 64-127.
// With the SwiGLU interleave of the prepared FC1 weights (64 gate rows then
// 64 up rows per block) operand 0 is 128 gate rows and operand 1 the 128 up
// rows of the same outputs, so gate and up land in the same tensor-memory
// lane of two accumulators.  Without a gate the two operands are 256
// consecutive output columns (lane r of operand o = column
// 128 (r / 64) + 64 o + r % 64 of the tile).
//
// Roles (448 threads, one persistent CTA per SM): warp 0 TMA producer (per
// stage one 16 KB copy per operand, one 8 KB copy of the route rows, and the
// scale atoms of the two weight blocks and of the routes' M tile), warp 1
// MMA issuer (per 32-byte K step one 128x64x64 block-scaled MMA per
// operand), warps 2-5 scale writers (compose each operand's scale image from
// the two source atoms and store it into tensor memory), warps 6-13 epilogue
// (thread = weight row, one column per route: coalesced across the warp; two
// warps per lane quadrant, 32 route columns each).
// Accumulators double-buffered: 2 x 2 operands x 64 columns.
//
// Epilogues: the same arithmetic as the standard orientation's
// (epilogue.cuh), element for element; the FC1 requantization takes an
// NVFP4 block as 16 consecutive lanes (block max by shuffles, each lane
// converts its own value, nibbles packed by shuffles), which gives the codes
// quant_block16 gives.  The fused-finalize scatter issues one coalesced
// scalar reduction per lane and route.
// Every wait is bounded (1 s); a timeout sets a status bit and all roles
// drain and exit.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace swapab {

constexpr int kNW = 128;                         // weight rows per operand (MMA M)
constexpr int kNR = 64;                          // route rows per tile (MMA N)
constexpr int kOps = 2;                          // weight operands per tile
constexpr int kStages = 4;
constexpr int kChunk = 128;                      // K bytes per stage (256 E2M1)
constexpr int kWBytes = kNW * kChunk;            // 16 KB per operand
constexpr int kXBytes = kNR * kChunk;            // 8 KB
constexpr int kAtom = 512;                       // scale atom: 128 rows x 4 scales
constexpr int kSfBlock = 4 * kAtom;              // a chunk's 4 atoms of one 128-row block
constexpr int kSlotW = kOps * kWBytes;
constexpr int kSlotSf = 3 * kSfBlock;            // weight blocks 2t, 2t+1 and the routes' M tile
constexpr int kSfWarps = 4;
constexpr int kEpiWarp0 = 2 + kSfWarps;
constexpr int kEpiWarps = 8;                     // two per lane quadrant: 32 route columns each
constexpr int kNumThreads = (kEpiWarp0 + kEpiWarps) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = kOps * kNR;        // one accumulator buffer
constexpr uint32_t kSfColBase = 2 * kAccCols;    // 256
constexpr uint32_t kSfColsPerStage = (kOps + 1) * 16;
constexpr int kSmemBytes = kStages * (kSlotW + kXBytes + kSlotSf) + 1024 + 256;
static_assert(kSfColBase + kStages * kSfColsPerStage <= kTmemCols, "tensor memory budget");
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Smem {
    uint8_t* w;
    uint8_t* x;
    uint8_t* sf;
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

__device__ __forceinline__ Smem carve(uint8_t* raw) {
    Smem s;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    s.w = base;
    s.x = s.w + kStages * kSlotW;
    s.sf = s.x + kStages * kXBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(s.sf + kStages * kSlotSf);
    s.full = bars;
    s.sf_full = bars + kStages;
    s.empty = bars + 2 * kStages;
    s.sf_ready = bars + 3 * kStages;
    s.acc_full = bars + 4 * kStages;
    s.acc_empty = s.acc_full + 2;
    s.drain = s.acc_empty + 2;
    s.tmem_holder = reinterpret_cast<uint32_t*>(s.drain + 1);
    s.abort = reinterpret_cast<volatile int*>(s.tmem_holder + 1);
    return s;
}

// Tile decomposition shared by every role: tile -> (occupied 64-route half
// of an M tile, from the scan's list, and weight tile), weight tiles
// fastest so that CTAs running at the same time share the route rows and
// walk one expert's weights.  Only halves holding routes are listed, so the
// persistent grid's tiles are all real work.
struct TileMap {
    int n_wt;          // weight tiles (of 256 rows) per expert
    __device__ __forceinline__ void decode(const GemmParams& p, int tile, int& m, int& h, int& wt) const {
        const int entry = p.tile_half[tile / n_wt];
        m = entry >> 1;
        h = entry & 1;
        wt = tile % n_wt;
    }
};

// Scale image of one 128-row MMA operand for tensor-memory lane l (one row
// of a 512-byte atom = 4 words, word q = scales of operand row l + 32 q):
// weight operand o takes rows 64 o .. 64 o + 63 of blocks 2t (operand rows
// 0-63) and 2t+1 (rows 64-127), i.e. words 2o, 2o+1 of each; the route
// operand (N = 64) takes rows 64 h .. 64 h + 63 of its M tile's atom.
__device__ __forceinline__ void compose_sf(const uint4& b0, const uint4& b1, const uint4& xa, int h,
                                           uint32_t (&w)[3][4]) {
    w[0][0] = b0.x; w[0][1] = b0.y; w[0][2] = b1.x; w[0][3] = b1.y;
    w[1][0] = b0.z; w[1][1] = b0.w; w[1][2] = b1.z; w[1][3] = b1.w;
    w[2][0] = h ? xa.z : xa.x;
    w[2][1] = h ? xa.w : xa.y;
    w[2][2] = 0u;
    w[2][3] = 0u;
}

// Per-lane NVFP4 requantization of an FC2-input value h for route row `row`
// and column i, the 16 lanes i & ~15 .. +15 of the warp forming one block:
// the arithmetic of quant_block16, with the block max taken by shuffles.
// Every lane of the warp must call it (the same row for the whole warp).
__device__ __forceinline__ void requant_lane(const GemmParams& p, float h, float g2, int row, int i, bool store) {
    const int lane = threadIdx.x & 31;
    float amax = fabsf(h);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const uint32_t s = f32_to_e4m3(__fdiv_rn(__fdiv_rn(amax, g2), 6.0f));
    const float sv = e4m3_to_f32(s);
    const float inv = (sv == 0.0f) ? 0.0f : __fdiv_rn(1.0f, __fmul_rn(sv, g2));
    uint32_t v = f32x2_to_e2m1x2(__fmul_rn(h, inv), 0.0f) & 0xFu;
    v |= __shfl_down_sync(0xffffffffu, v, 1) << 4;     // byte: elements l, l+1 (even lanes)
    v |= __shfl_down_sync(0xffffffffu, v, 2) << 8;     // lanes % 4 == 0: 4 elements
    v |= __shfl_down_sync(0xffffffffu, v, 4) << 16;    // lanes % 8 == 0: 8 elements
    if (!store) return;
    if ((lane & 7) == 0) *reinterpret_cast<uint32_t*>(p.out_codes + (size_t)row * (p.out_cols / 2) + i / 2) = v;
    if ((lane & 15) == 0) p.out_sf[sf_offset(row, i / 16, p.out_cols)] = (uint8_t)s;
}

__device__ __forceinline__ void red_add_f32(float* addr, float v) {
    asm volatile("red.relaxed.gpu.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

template <int EPI, bool GATED>
__global__ void __launch_bounds__(kNumThreads, 1)
    gemm_swap_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                     const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    const Smem s = carve(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        prefetch_tensormap(&tmW);
        prefetch_tensormap(&tmX);
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.sf_full[i], 1);
            mbar_init(&s.empty[i], 1);
            mbar_init(&s.sf_ready[i], kSfWarps * 32);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.acc_full[i], 1);
            mbar_init(&s.acc_empty[i], kEpiWarps * 32);
        }
        mbar_init(s.drain, 1);
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
    const uint32_t tmem_base = *s.tmem_holder;
    pdl_wait();   // routes, scales, tile map and tile count come from earlier kernels

    const int row_bytes = p.kdim / 2;
    const int kblocks = row_bytes / 32;                        // 32-byte MMA steps = scale atoms per 128 rows
    const int nchunks = (row_bytes + kChunk - 1) / kChunk;
    const int rb_per_expert = p.n / 128;
    TileMap tm;
    tm.n_wt = (rb_per_expert + 1) / 2;
    const int total = p.meta[3] * tm.n_wt;

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_normal();
            int stage = 0;
            uint32_t phase = 0;
            for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
                int m, h, wt;
                tm.decode(p, tile, m, h, wt);
                const int e = p.tile_expert[m];
                if (e < 0 || e >= p.num_experts) {
                    atomicOr(p.status, kStatusBadExpert);
                    *s.abort = 1;
                    break;
                }
                const int blk0 = e * rb_per_expert + 2 * wt;
                const int nblk = min(2, rb_per_expert - 2 * wt);
                for (int ks = 0; ks < nchunks; ++ks) {
                    if (!mbar_wait(&s.empty[stage], phase ^ 1u, s.abort, p.status, kStatusTimeoutProducer)) goto done;
                    const int n_at = min(4, kblocks - 4 * ks);
                    const uint32_t sfb = (uint32_t)n_at * kAtom;
                    uint8_t* sf = s.sf + stage * kSlotSf;
                    mbar_arrive_expect_tx(&s.sf_full[stage], (uint32_t)(nblk + 1) * sfb);
                    for (int b = 0; b < nblk; ++b)
                        bulk_load(sf + b * kSfBlock, p.sfb + ((size_t)(blk0 + b) * kblocks + 4 * ks) * kAtom, sfb,
                                  &s.sf_full[stage], pol);
                    bulk_load(sf + 2 * kSfBlock, p.sfa + ((size_t)m * kblocks + 4 * ks) * kAtom, sfb, &s.sf_full[stage],
                              pol);
                    mbar_arrive_expect_tx(&s.full[stage], (uint32_t)(kSlotW + kXBytes));
                    for (int o = 0; o < kOps; ++o)
                        tma_load_3d(s.w + stage * kSlotW + o * kWBytes, &tmW, &s.full[stage], ks * kChunk, 64 * o, blk0,
                                    pol);
                    tma_load_2d(s.x + stage * kXBytes, &tmX, &s.full[stage], ks * kChunk, m * kTileM + kNR * h, pol);
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            const uint32_t idesc = idesc_nvf4(kNW, kNR);
            for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
                int m, h, wt;
                tm.decode(p, tile, m, h, wt);
                if (!mbar_wait(&s.acc_empty[acc], acc_phase ^ 1u, s.abort, p.status, kStatusTimeoutMma)) goto done;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kAccCols);
                for (int ks = 0; ks < nchunks; ++ks) {
                    if (!mbar_wait(&s.full[stage], phase, s.abort, p.status, kStatusTimeoutMma)) goto done;
                    if (!mbar_wait(&s.sf_ready[stage], phase, s.abort, p.status, kStatusTimeoutMma)) goto done;
                    tc_fence_after();
                    const int nkb = min(4, kblocks - 4 * ks);
                    const uint32_t sf_t = tmem_base + kSfColBase + (uint32_t)stage * kSfColsPerStage;
                    // descriptor start addresses count 16-byte units
                    const uint64_t wdesc0 = sdesc_kmajor_sw128(smem_u32(s.w + stage * kSlotW));
                    const uint64_t bdesc0 = sdesc_kmajor_sw128(smem_u32(s.x + stage * kXBytes));
                    auto issue = [&](int j) {
#pragma unroll
                        for (int o = 0; o < kOps; ++o)
                            tc_mma_nvf4(d_tmem + o * kNR, wdesc0 + (uint64_t)o * (kWBytes / 16) + 2u * j, bdesc0 + 2u * j,
                                        idesc, sf_t + 16 * o + 4 * j, sf_t + 32 + 4 * j, (ks | j) != 0);
                    };
                    if (nkb == 4) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) issue(j);   // a full stage: constant descriptor offsets
                    } else {
                        for (int j = 0; j < nkb; ++j) issue(j);
                    }
                    tc_commit(&s.empty[stage]);
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
                tc_commit(&s.acc_full[acc]);
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
        }
    } else if (warp < kEpiWarp0) {
        // scale writer for lane quadrant warp % 4 (each quadrant holds a copy)
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        int stage = 0;
        uint32_t phase = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            int m, h, wt;
            tm.decode(p, tile, m, h, wt);
            for (int ks = 0; ks < nchunks; ++ks) {
                if (!__all_sync(0xffffffffu,
                                mbar_wait(&s.sf_full[stage], phase, s.abort, p.status, kStatusTimeoutMma)))
                    goto done;
                const uint8_t* sf = s.sf + stage * kSlotSf;
                const uint32_t sf_t = tmem_base + kSfColBase + (uint32_t)stage * kSfColsPerStage;
                uint32_t wo0[16], wo1[16], wx[16];
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    // atoms beyond the chunk's K steps or a missing second block
                    // hold stale bytes: the MMAs never read them / their rows
                    // are ignored by the epilogue
                    const uint4 b0 = *reinterpret_cast<const uint4*>(sf + a * kAtom + lane * 16);
                    const uint4 b1 = *reinterpret_cast<const uint4*>(sf + kSfBlock + a * kAtom + lane * 16);
                    const uint4 xa = *reinterpret_cast<const uint4*>(sf + 2 * kSfBlock + a * kAtom + lane * 16);
                    uint32_t w[3][4];
                    compose_sf(b0, b1, xa, h, w);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        wo0[4 * a + q] = w[0][q];
                        wo1[4 * a + q] = w[1][q];
                        wx[4 * a + q] = w[2][q];
                    }
                }
                tmem_st_n<16>(sf_t + lane_off, wo0);
                tmem_st_n<16>(sf_t + 16 + lane_off, wo1);
                tmem_st_n<16>(sf_t + 32 + lane_off, wx);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(&s.sf_ready[stage]);
                if (++stage == kStages) { stage = 0; phase ^= 1u; }
            }
        }
    } else {
        // epilogue: warp quadrant q, thread = weight row r = 32 q + lane of each
        // operand; warp half `half` takes route columns 32 half .. +31,
        // broadcast lane by lane
        const int q = warp & 3;
        const int half = (warp - kEpiWarp0) >> 2;
        const int r = 32 * q + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            int m, h, wt;
            tm.decode(p, tile, m, h, wt);
            const int e = p.tile_expert[m];
            if (e < 0 || e >= p.num_experts) break;
            // this lane's route column (32 half + lane): route, scale and route
            // weight, loaded before the accumulator is ready so that their L2
            // round trips hide under the MMAs
            const float gw = p.gw[e];
            const int rb = m * kTileM + kNR * h + 32 * half;   // first route row of this warp's columns
            const int my_route = p.route_of_row[rb + lane];
            const int my_token = my_route >= 0 ? my_route / p.topk : 0;
            float g_act;
            if (EPI == kEpiFc1Quant || EPI == kEpiFc1F32) g_act = p.g_act_per_token ? p.g_act[my_token] : p.g_act[0];
            else g_act = p.g_act_per_token == 2 ? p.g_act[rb + lane] : p.g_act[0];
            float my_pw = 1.0f;
            if (my_route >= 0 && (((EPI == kEpiFc1Quant || EPI == kEpiFc1F32) && p.weight_on_input) ||
                                  (EPI == kEpiFc2Scatter && p.weight_on_output)))
                my_pw = p.topk_w[my_route];
            float my_alpha = __fmul_rn(g_act, gw);
            if (EPI == kEpiFc2Scatter && p.weight_on_output) my_alpha = my_alpha * my_pw;
            if (!__all_sync(0xffffffffu, mbar_wait(&s.acc_full[acc], acc_phase, s.abort, p.status,
                                                   kStatusTimeoutEpilogue)))
                break;
            tc_fence_after();
            // output column of weight row r in operand o (gated: operand 1 is
            // the up half of the same outputs)
            const int col0 = GATED ? 128 * wt + r : 256 * wt + 128 * (r >> 6) + (r & 63);
            const uint32_t tbase =
                tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * kAccCols) + (uint32_t)(32 * half);
            // columns in groups of 8 with a runtime loop: a fully unrolled body
            // (the requantization inlined per column) was tens of KB of code,
            // fetched cold by every SM at every launch.  An expert's routes
            // fill its rows from the start, so this warp's live columns are a
            // prefix: only the groups holding one are visited; inside them
            // every column is computed and only the stores are predicated, so
            // that the broadcasts of consecutive columns overlap.
            const uint32_t live_mask = __ballot_sync(0xffffffffu, my_route >= 0);
            const int ngroups = (32 - __clz(live_mask) + 7) / 8;
#pragma unroll 1
            for (int g = 0; g < ngroups; ++g) {
                float a0[8], a1[8];
                tmem_ld8(tbase + 8 * g, a0);
                tmem_ld8(tbase + kNR + 8 * g, a1);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int src = 8 * g + j;
                    const bool live = __shfl_sync(0xffffffffu, my_route, src) >= 0;   // pad rows: no store
                    const int row = rb + src;
                    const float alpha = __shfl_sync(0xffffffffu, my_alpha, src);
                    if (EPI == kEpiFc1Quant || EPI == kEpiFc1F32) {
                        const float pw = __shfl_sync(0xffffffffu, my_pw, src);
                        if (GATED) {
                            // silu(z) as in the standard epilogue (ex2-based exponential,
                            // approximate division)
                            const float zg = a0[j] * alpha, zu = a1[j] * alpha;
                            const float hv = __fdividef(zg, 1.0f + __expf(-zg)) * zu * pw;
                            if (EPI == kEpiFc1F32) {
                                if (live) p.out_f32[(size_t)row * p.out_cols + col0] = hv;
                            } else {
                                requant_lane(p, hv, p.g2[0], row, col0, live);
                            }
                        } else {
#pragma unroll
                            for (int o = 0; o < kOps; ++o) {
                                const int col = col0 + 64 * o;
                                if (col - lane >= p.n) continue;  // past the segment: uniform across the warp
                                const float z = fmaxf((o ? a1[j] : a0[j]) * alpha, 0.0f);
                                const float hv = z * z * pw;
                                if (EPI == kEpiFc1F32) {
                                    if (live) p.out_f32[(size_t)row * p.out_cols + col] = hv;
                                } else {
                                    requant_lane(p, hv, p.g2[0], row, col, live);
                                }
                            }
                        }
                    } else {
                        const int token = __shfl_sync(0xffffffffu, my_token, src);
#pragma unroll
                        for (int o = 0; o < kOps; ++o) {
                            const int col = col0 + 64 * o;
                            if (col - lane >= p.n || !live) continue;
                            const float v = (o ? a1[j] : a0[j]) * alpha;
                            if (EPI == kEpiFc2Store) p.out_bf16[(size_t)row * p.out_cols + col] = __float2bfloat16_rn(v);
                            else red_add_f32(p.out_f32 + (size_t)token * p.out_cols + col, v);
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&s.acc_empty[acc]);
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
    }
done:
    {
        // after an abort let in-flight copies land and retire issued MMAs and
        // tensor-memory stores before the tensor memory is freed
        volatile int no_abort = 0;
        if (*s.abort) {
            if (warp == 1 && lane == 0) {
                tc_commit(s.drain);
                mbar_wait(s.drain, 0, &no_abort, p.status, kStatusTimeoutMma);
            }
            if (warp >= 2 && warp < kEpiWarp0) tmem_st_wait();
            for (int i = 0; i < 100; ++i) __nanosleep(10000);
        }
    }
    tc_fence_before();
    __syncthreads();
    pdl_launch_dependents();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

template <int EPI, bool GATED>
static cudaError_t set_smem_one() {
    return cudaFuncSetAttribute(gemm_swap_kernel<EPI, GATED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmemBytes);
}

}  // namespace swapab

cudaError_t setup_gemm_swap_kernels() {
    using namespace swapab;
    cudaError_t e;
    if ((e = set_smem_one<kEpiFc1Quant, true>())) return e;
    if ((e = set_smem_one<kEpiFc1F32, true>())) return e;
    if ((e = set_smem_one<kEpiFc1Quant, false>())) return e;
    if ((e = set_smem_one<kEpiFc1F32, false>())) return e;
    if ((e = set_smem_one<kEpiFc2Store, false>())) return e;
    return set_smem_one<kEpiFc2Scatter, false>();
}

cudaError_t launch_gemm_swap(const LaunchCtx& c, int epilogue, bool gated, const CUtensorMap& tmW,
                             const CUtensorMap& tmX, const GemmParams& p, int num_sms) {
    using namespace swapab;
    const dim3 grid(num_sms), block(kNumThreads);
    const size_t smem = kSmemBytes;
    if (gated) {
        switch (epilogue) {
            case kEpiFc1Quant: return c.launch(gemm_swap_kernel<kEpiFc1Quant, true>, grid, block, smem, tmW, tmX, p);
            case kEpiFc1F32: return c.launch(gemm_swap_kernel<kEpiFc1F32, true>, grid, block, smem, tmW, tmX, p);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (epilogue) {
        case kEpiFc1Quant: return c.launch(gemm_swap_kernel<kEpiFc1Quant, false>, grid, block, smem, tmW, tmX, p);
        case kEpiFc1F32: return c.launch(gemm_swap_kernel<kEpiFc1F32, false>, grid, block, smem, tmW, tmX, p);
        case kEpiFc2Store: return c.launch(gemm_swap_kernel<kEpiFc2Store, false>, grid, block, smem, tmW, tmX, p);
        case kEpiFc2Scatter: return c.launch(gemm_swap_kernel<kEpiFc2Scatter, false>, grid, block, smem, tmW, tmX, p);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace moe
