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
#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"

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

// 8 E2M1 codes (4 bytes, low nibble first) times scale s -> 8 BF16.
__device__ __forceinline__ uint4 dequant8(uint32_t codes, float s) {
    uint32_t h2[4];
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}\n"
        : "=r"(h2[0]), "=r"(h2[1]), "=r"(h2[2]), "=r"(h2[3])
        : "r"(codes));
    uint32_t out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 hv = *reinterpret_cast<const __half2*>(&h2[i]);
        const float2 f = __half22float2(hv);
        const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * s, f.y * s);   // exact
        out[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
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
                    const float sc = e4m3_to_f32((sfw >> (8 * (c >> 1))) & 0xFFu);
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
            if (EPI == kEpiFc1Bf16) epilogue_fc1<EPI>(p, taddr, row, meta, n_tile);
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

}  // namespace moe
