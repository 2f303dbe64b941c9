// Grouped W4A16 GEMMs with the operands swapped: the expert's weights,
// widened to BF16 on chip, are the MMA's M side (two 128-row operands per
// tile) and the expert's routes its N side (one 64-route half of an M tile),
// for experts that hold few routes [newruntime post on FlashInfer PR #5319,
// "Retrieval answer": W4A16 with BF16 activations on the prepared NVFP4
// weights].
//
//   D^T[w, r] = sum_k W_e[w, k] * X[r, k]         (r: routes of expert e)
//
// Why: in the standard orientation (gemm_w4a16.cu) a tile is 128 activation
// rows, padded per expert, so at a few dozen routes per expert most of
// every MMA, and of every activation tile read from memory, is padding,
// while each weight element is still widened once per M tile.  Here the MMA
// work and the activation bytes follow the routes (64-route halves, only
// those holding routes are tiled), and the widening cost -- the same once
// per weight element and route half -- is what the tile is sized for.
//
// Tile = two weight operands of 128 rows x one 64-route half.  The E2M1
// codes come from one 3-D tensor map over the prepared weights viewed as
// [128-row blocks][128 rows][K bytes], box 64 B x 64 rows x 2 blocks:
// operand 0 = rows 0-63 of blocks 2t and 2t+1, operand 1 = rows 64-127.
// With the SwiGLU interleave of the prepared FC1 weights (64 gate rows then
// 64 up rows per block) operand 0 is 128 gate rows and operand 1 the 128 up
// rows of the same outputs, so gate and up land in the same tensor-memory
// lane of two accumulators; without a gate the operands are 256 consecutive
// output columns (lane r of operand o = column 128 (r / 64) + 64 o + r % 64
// of the tile).
//
// The widened weights never touch shared memory: each converter thread
// owns one weight row, i.e. one tensor-memory lane, and stores its 128
// BF16 of a stage as 64 columns with tcgen05.st; the MMA reads its A operand from
// tensor memory.  (Through shared memory a stage moved ~100 KB -- codes,
// route tile, the widened weights written and read back, the route tile read
// once per operand; keeping the widened weights in tensor memory cut the
// shared-memory wavefronts threefold and the GEMM time by ~8 %.)  Two
// rings: a six-deep copy ring in shared memory (per stage of 128 K
// elements: the route tile as two 64 x 64 BF16 sub-tiles, 128-byte swizzle,
// the two 8 KB code tiles and each weight block's two scale atoms) and two
// slots of widened weights in tensor memory (2 operands x 64 columns each).
// Stages of 128 elements make the code copies 64-byte row segments: with
// 64-element stages (32-byte segments) the copies bounded the kernel, and
// doubling the segment cut the GEMM time by a further ~17 %.
//
// Tensor memory (512 columns): accumulators at 0-255 (two buffers of 2
// operands x 64 route columns), widened-weight slots at 256-511.
//
// Roles (576 threads, one persistent CTA per SM): warp 0 TMA producer, warp
// 1 tensor-memory allocation and MMA issuer (per 16-element K step one
// 128 x 64 x 16 kind::f16 MMA per operand, A from tensor memory), warps 2-9
// converters (thread = one weight row of one operand, on its own lane: 128
// codes x their 8 scales per stage), warps 10-17 epilogue (thread = weight
// row, one column per route: two warps per lane quadrant, 32 route columns
// each).  The epilogue arithmetic is
// that of epilogue.cuh (W4A16: no activation global scale), element for
// element.  Every wait is bounded (1 s); a timeout sets a status bit and all
// roles drain and exit.
#include "common.cuh"
#include "kernels.h"
#include "w4a16_convert.cuh"
#include "w4a16_swap.h"

namespace moe {
namespace swap16 {

constexpr int kNW = 128;                         // weight rows per operand (MMA M)
constexpr int kNR = 64;                          // route rows per tile (MMA N)
constexpr int kOps = 2;
constexpr int kKStage = 128;                     // K elements per stage
constexpr int kLoadStages = 6;
constexpr int kConvSlots = 2;
constexpr int kXHalf = kNR * 128;                // 64 routes x 64 BF16: one 128-byte-swizzled sub-tile
constexpr int kXBytes = 2 * kXHalf;              // 64 routes x 128 BF16
constexpr int kQBytes = kNW * kKStage / 2;       // one operand's codes: 128 rows x 128 E2M1
constexpr int kAtom = 512;                       // one scale atom: 128 rows x 4 scales (64 K elements)
constexpr int kSfBytes = 2 * kAtom;              // one weight block's scales of a stage
constexpr int kConvWarps = 8;
constexpr int kEpiWarp0 = 2 + kConvWarps;
constexpr int kEpiWarps = 8;
constexpr int kNumThreads = (kEpiWarp0 + kEpiWarps) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = kOps * kNR;        // one accumulator buffer
constexpr uint32_t kACol0 = 2 * kAccCols;        // first widened-weight column
constexpr uint32_t kAOpCols = kKStage / 2;       // 128 BF16 of one row per stage, two per column
constexpr uint32_t kASlotCols = kOps * kAOpCols;
static_assert(kACol0 + kConvSlots * kASlotCols <= kTmemCols, "tensor memory budget");
constexpr int kSmemBytes = kLoadStages * (kXBytes + kOps * kQBytes + 2 * kSfBytes) + 1024 + 256;
static_assert(kConvWarps * 32 == kOps * kNW, "one converter thread per weight row of each operand");
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Smem {
    uint8_t* x;          // [kLoadStages][2 sub-tiles][64][128 B], 128-byte swizzle
    uint8_t* q;          // [kLoadStages][2 operands][128][64 B]
    uint8_t* sf;         // [kLoadStages][2 blocks][2 atoms][512 B]
    uint64_t* full;      // copies of a stage landed
    uint64_t* empty;     // MMAs of a stage done (its route tile and codes free)
    uint64_t* conv_full; // a slot's widened weights written
    uint64_t* conv_empty;
    uint64_t* acc_full;
    uint64_t* acc_empty;
    uint64_t* drain;
    uint32_t* tmem_holder;
    volatile int* abort;
};

__device__ __forceinline__ Smem carve(uint8_t* raw) {
    Smem s;
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    s.x = base;
    s.q = s.x + kLoadStages * kXBytes;
    s.sf = s.q + kLoadStages * kOps * kQBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(s.sf + kLoadStages * 2 * kSfBytes);
    s.full = bars;
    s.empty = bars + kLoadStages;
    s.conv_full = bars + 2 * kLoadStages;
    s.conv_empty = s.conv_full + kConvSlots;
    s.acc_full = s.conv_empty + kConvSlots;
    s.acc_empty = s.acc_full + 2;
    s.drain = s.acc_empty + 2;
    s.tmem_holder = reinterpret_cast<uint32_t*>(s.drain + 1);
    s.abort = reinterpret_cast<volatile int*>(s.tmem_holder + 1);
    return s;
}

// tile -> (occupied 64-route half of an M tile, from the scan's list, and
// weight tile of 256 rows), weight tiles fastest: CTAs running at the same
// time share the route rows and walk one expert's weights
struct TileMap {
    int n_wt;
    __device__ __forceinline__ void decode(const GemmParams& p, int tile, int& m, int& h, int& wt) const {
        const int entry = p.tile_half[tile / n_wt];
        m = entry >> 1;
        h = entry & 1;
        wt = tile % n_wt;
    }
};

// kind::f16 MMA with the A operand (M x 16 BF16) in tensor memory
__device__ __forceinline__ void tc_mma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                                   uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void red_add_f32(float* addr, float v) {
    asm volatile("red.relaxed.gpu.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

template <int EPI, bool GATED>
__global__ void __launch_bounds__(kNumThreads, 1)
    gemm_w4a16_swap_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                           const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    const Smem s = carve(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        prefetch_tensormap(&tmW);
        prefetch_tensormap(&tmX);
        for (int i = 0; i < kLoadStages; ++i) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.empty[i], 1);
        }
        for (int i = 0; i < kConvSlots; ++i) {
            mbar_init(&s.conv_full[i], kConvWarps);
            mbar_init(&s.conv_empty[i], 1);
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
    pdl_wait();   // routes, tile lists and the gathered activations come from earlier kernels

    const int kblocks = p.kdim / 64;                 // 64-element K blocks (scale atoms per weight block)
    const int ksteps = p.kdim / kKStage;             // stages per tile
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
                for (int ks = 0; ks < ksteps; ++ks) {
                    if (!mbar_wait(&s.empty[stage], phase ^ 1u, s.abort, p.status, kStatusTimeoutProducer)) goto done;
                    mbar_arrive_expect_tx(&s.full[stage],
                                          (uint32_t)(kXBytes + kOps * kQBytes + nblk * kSfBytes));
                    for (int xh = 0; xh < 2; ++xh)
                        tma_load_2d(s.x + stage * kXBytes + xh * kXHalf, &tmX, &s.full[stage], ks * 256 + xh * 128,
                                    m * kTileM + kNR * h, pol);
                    for (int o = 0; o < kOps; ++o)
                        tma_load_3d(s.q + (stage * kOps + o) * kQBytes, &tmW, &s.full[stage], ks * (kKStage / 2), 64 * o,
                                    blk0, pol);
                    // the two atoms of K blocks 2 ks, 2 ks + 1 are adjacent
                    for (int b = 0; b < nblk; ++b)
                        bulk_load(s.sf + (stage * 2 + b) * kSfBytes,
                                  p.sfb + ((size_t)(blk0 + b) * kblocks + 2 * ks) * kAtom, kSfBytes, &s.full[stage], pol);
                    if (++stage == kLoadStages) { stage = 0; phase ^= 1u; }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0, slot = 0, acc = 0;
            uint32_t phase = 0, cphase = 0, acc_phase = 0;
            const uint32_t idesc = idesc_bf16(kNW, kNR);
            for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
                if (!mbar_wait(&s.acc_empty[acc], acc_phase ^ 1u, s.abort, p.status, kStatusTimeoutMma)) goto done;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kAccCols);
                for (int ks = 0; ks < ksteps; ++ks) {
                    if (!mbar_wait(&s.full[stage], phase, s.abort, p.status, kStatusTimeoutMma)) goto done;
                    if (!mbar_wait(&s.conv_full[slot], cphase, s.abort, p.status, kStatusTimeoutMma)) goto done;
                    tc_fence_after();
                    // descriptor start addresses count 16-byte units: 32 bytes = one K
                    // step; in tensor memory one K step of A is 8 columns
                    const uint32_t a0 = tmem_base + kACol0 + (uint32_t)slot * kASlotCols;
                    const uint64_t xdesc0 = sdesc_kmajor_sw128(smem_u32(s.x + stage * kXBytes));
#pragma unroll
                    for (int j = 0; j < kKStage / 16; ++j)
#pragma unroll
                        for (int o = 0; o < kOps; ++o)
                            tc_mma_bf16_tmem_a(d_tmem + o * kNR, a0 + (uint32_t)(o * kAOpCols + 8 * j),
                                               xdesc0 + (uint64_t)((j >> 2) * (kXHalf / 16) + 2 * (j & 3)), idesc,
                                               (ks | j) != 0);
                    tc_commit(&s.empty[stage]);
                    tc_commit(&s.conv_empty[slot]);
                    if (++stage == kLoadStages) { stage = 0; phase ^= 1u; }
                    if (++slot == kConvSlots) { slot = 0; cphase ^= 1u; }
                }
                tc_commit(&s.acc_full[acc]);
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
        }
    } else if (warp < kEpiWarp0) {
        // converter: thread (o, r) widens row r of operand o, i.e. row
        // 64 o + r % 64 of weight block 2t + r / 64, into tensor-memory lane
        // r (a warp reaches the lanes of quadrant warp % 4 only)
        const int q = warp & 3;
        const int o = (warp - 2) >> 2, r = 32 * q + lane;
        const int rr = 64 * o + (r & 63);
        const uint32_t sf_off = (uint32_t)(r >> 6) * kSfBytes + (uint32_t)(rr & 31) * 16u + (uint32_t)(rr >> 5) * 4u;
        const uint32_t t_row = tmem_base + ((uint32_t)(32 * q) << 16) + kACol0 + (uint32_t)(o * kAOpCols);
        int stage = 0, slot = 0;
        uint32_t phase = 0, cphase = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            for (int ks = 0; ks < ksteps; ++ks) {
                if (!__all_sync(0xffffffffu,
                                mbar_wait(&s.full[stage], phase, s.abort, p.status, kStatusTimeoutProducer)))
                    goto done;
                if (!__all_sync(0xffffffffu, mbar_wait(&s.conv_empty[slot], cphase ^ 1u, s.abort, p.status,
                                                       kStatusTimeoutProducer)))
                    goto done;
                tc_fence_after();                      // the slot's last MMAs are complete
                const uint8_t* qrow = s.q + (stage * kOps + o) * kQBytes + r * (kKStage / 2);
                // two 64-element halves: codes from 32 bytes, scales from one atom each
#pragma unroll
                for (int a = 0; a < 2; ++a) {
                    const uint4 c0 = *reinterpret_cast<const uint4*>(qrow + 32 * a);
                    const uint4 c1 = *reinterpret_cast<const uint4*>(qrow + 32 * a + 16);
                    const uint32_t sfw =
                        *reinterpret_cast<const uint32_t*>(s.sf + stage * 2 * kSfBytes + a * kAtom + sf_off);
                    const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                    uint32_t wv[32];                   // column i = elements 2i (low half), 2i + 1
#pragma unroll
                    for (int c = 0; c < 8; ++c) {      // elements 8c .. 8c+7 of the half
                        const __half2 sc = __float2half2_rn(e4m3_to_f32((sfw >> (8 * (c >> 1))) & 0xFFu));
                        const uint4 v = dequant8(words[c], sc);
                        wv[4 * c] = v.x;
                        wv[4 * c + 1] = v.y;
                        wv[4 * c + 2] = v.z;
                        wv[4 * c + 3] = v.w;
                    }
                    tmem_st32(t_row + (uint32_t)slot * kASlotCols + (uint32_t)(32 * a), wv);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s.conv_full[slot]);
                if (++stage == kLoadStages) { stage = 0; phase ^= 1u; }
                if (++slot == kConvSlots) { slot = 0; cphase ^= 1u; }
            }
        }
    } else {
        // epilogue: lane quadrant q, thread = weight row r = 32 q + lane of
        // each operand; warp half `half` takes route columns 32 half .. +31,
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
            // this lane's route column (32 half + lane): route, token and the
            // epilogue scalars of epi_row (no activation global scale),
            // loaded before the accumulator is ready
            const int rb = m * kTileM + kNR * h + 32 * half;   // first route row of this warp's columns
            const int my_route = p.route_of_row[rb + lane];
            const int my_token = my_route >= 0 ? my_route / p.topk : 0;
            float my_alpha = __fmul_rn(1.0f, p.gw[e]);
            float my_pw = 1.0f;
            if (EPI == kEpiFc1Bf16 && p.weight_on_input && my_route >= 0) my_pw = p.topk_w[my_route];
            if (EPI == kEpiFc2Scatter && p.weight_on_output && my_route >= 0) my_alpha = my_alpha * p.topk_w[my_route];
            if (!__all_sync(0xffffffffu, mbar_wait(&s.acc_full[acc], acc_phase, s.abort, p.status,
                                                   kStatusTimeoutEpilogue)))
                break;
            tc_fence_after();
            const int col0 = GATED ? 128 * wt + r : 256 * wt + 128 * (r >> 6) + (r & 63);
            const uint32_t tbase =
                tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * kAccCols) + (uint32_t)(32 * half);
            // an expert's routes fill its rows from the start: this warp's
            // live columns are a prefix, only the groups of 8 holding one
            // are visited
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
                    if (EPI == kEpiFc1Bf16) {
                        const float pw = __shfl_sync(0xffffffffu, my_pw, src);
                        if (GATED) {
                            // silu as in fc1_act32 (ex2-based exponential, approximate division)
                            const float zg = a0[j] * alpha, zu = a1[j] * alpha;
                            const float hv = __fdividef(zg, 1.0f + __expf(-zg)) * zu * pw;
                            if (live) p.out_bf16[(size_t)row * p.out_cols + col0] = __float2bfloat16_rn(hv);
                        } else {
#pragma unroll
                            for (int oo = 0; oo < kOps; ++oo) {
                                const int col = col0 + 64 * oo;
                                if (col - lane >= p.n || !live) continue;   // past the segment: uniform
                                const float z = fmaxf((oo ? a1[j] : a0[j]) * alpha, 0.0f);
                                p.out_bf16[(size_t)row * p.out_cols + col] = __float2bfloat16_rn(z * z * pw);
                            }
                        }
                    } else {
                        const int token = __shfl_sync(0xffffffffu, my_token, src);
#pragma unroll
                        for (int oo = 0; oo < kOps; ++oo) {
                            const int col = col0 + 64 * oo;
                            if (col - lane >= p.n || !live) continue;
                            const float v = (oo ? a1[j] : a0[j]) * alpha;
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
cudaError_t set_smem_one() {
    return cudaFuncSetAttribute(gemm_w4a16_swap_kernel<EPI, GATED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kSmemBytes);
}

}  // namespace swap16

cudaError_t setup_gemm_w4a16_swap_kernels() {
    using namespace swap16;
    cudaError_t e;
    if ((e = set_smem_one<kEpiFc1Bf16, true>())) return e;
    if ((e = set_smem_one<kEpiFc1Bf16, false>())) return e;
    if ((e = set_smem_one<kEpiFc2Store, false>())) return e;
    return set_smem_one<kEpiFc2Scatter, false>();
}

cudaError_t launch_gemm_w4a16_swap(const LaunchCtx& c, int epilogue, bool gated, const CUtensorMap& tmW,
                                   const CUtensorMap& tmX, const GemmParams& p, int num_sms) {
    using namespace swap16;
    const dim3 grid(num_sms), block(kNumThreads);
    const size_t smem = kSmemBytes;
    if (gated)
        return epilogue == kEpiFc1Bf16
                   ? c.launch(gemm_w4a16_swap_kernel<kEpiFc1Bf16, true>, grid, block, smem, tmW, tmX, p)
                   : cudaErrorInvalidValue;
    switch (epilogue) {
        case kEpiFc1Bf16: return c.launch(gemm_w4a16_swap_kernel<kEpiFc1Bf16, false>, grid, block, smem, tmW, tmX, p);
        case kEpiFc2Store: return c.launch(gemm_w4a16_swap_kernel<kEpiFc2Store, false>, grid, block, smem, tmW, tmX, p);
        case kEpiFc2Scatter:
            return c.launch(gemm_w4a16_swap_kernel<kEpiFc2Scatter, false>, grid, block, smem, tmW, tmX, p);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace moe
