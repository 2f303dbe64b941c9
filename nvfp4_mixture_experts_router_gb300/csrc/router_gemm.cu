// Router logits on the tensor cores, the optional first stage of the layer:
//
//   logits[t][e] = sum_h x[t][h] * Wg[e][h]       (BF16 in, FP32 accumulate)
//
// [FlashInfer PR #4366, "Motivation": the MoE wrapper is handed routing that
// was computed upstream from the gate projection; here the projection is the
// layer's own first kernel, feeding the router.]  Products of two BF16 values
// are exact in FP32; the tensor core accumulates them in FP32 (tcgen05.mma
// kind::f16 with BF16 operands, K = 16 per instruction).
//
// One CTA per output tile of 128 tokens x NT experts (NT = the expert count
// rounded up to 16, at most 256; more experts take further tiles), 192
// threads:
//   warp 0      TMA producer: per 64-element K chunk one 128 x 64 x tile
//               and one NT x 64 W_g tile (128-byte swizzle, K-major), four
//               stages; rows past T or E are filled with zeros by the TMA.
//   warp 1      allocates 256 tensor-memory columns; lane 0 issues four
//               128 x NT x 16 MMAs per chunk into one FP32 accumulator and
//               commits each stage back to the producer.
//   warps 2-5   epilogue: tcgen05.ld of the accumulator (one token row per
//               thread), FP32 stores of the valid columns.
// Every wait is bounded (1 s); a timeout sets a status bit and all roles
// drain and exit.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kRBM = 128;
constexpr int kRStages = 4;
constexpr int kRTileA = kRBM * 128;            // 64 BF16 per row
constexpr int kRMaxN = 256;
constexpr int kRTileBMax = kRMaxN * 128;
constexpr int kRThreads = 6 * 32;
constexpr uint32_t kRTmemCols = 256;
constexpr int kRSmemBytes = kRStages * (kRTileA + kRTileBMax) + 1024 + 256;
static_assert(kRSmemBytes <= 232448, "shared memory budget");

__global__ void __launch_bounds__(kRThreads, 1)
    router_gemm_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, int T, int E,
                       int H, int nt, float* __restrict__ logits, unsigned int* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sa = base;
    uint8_t* sb = sa + kRStages * kRTileA;
    uint64_t* full = reinterpret_cast<uint64_t*>(sb + kRStages * kRTileBMax);
    uint64_t* empty = full + kRStages;
    uint64_t* acc_full = empty + kRStages;
    uint64_t* drain = acc_full + 1;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_holder + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * kRBM, n0 = blockIdx.y * kRMaxN;
    const int chunks = H / 64;
    const uint32_t tile_b = (uint32_t)nt * 128u;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kRStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(drain, 1);
        *abort = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmX);
        prefetch_tensormap(&tmW);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, kRTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    pdl_wait();

    if (warp == 0) {
        if (lane == 0) {
            // x is read once: evict it first; W_g is shared by every CTA
            const uint64_t pol_x = policy_evict_first(), pol_w = policy_evict_last();
            int stage = 0;
            uint32_t phase = 0;
            for (int c = 0; c < chunks; ++c) {
                if (!mbar_wait(&empty[stage], phase ^ 1u, abort, status, kStatusTimeoutProducer)) break;
                mbar_arrive_expect_tx(&full[stage], (uint32_t)kRTileA + tile_b);
                // byte coordinates: a chunk is 128 bytes (64 BF16) of a row
                tma_load_2d(sa + stage * kRTileA, &tmX, &full[stage], c * 128, m0, pol_x);
                tma_load_2d(sb + stage * kRTileBMax, &tmW, &full[stage], c * 128, n0, pol_w);
                if (++stage == kRStages) { stage = 0; phase ^= 1u; }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(kRBM, nt);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int c = 0; c < chunks && ok; ++c) {
                if (!mbar_wait(&full[stage], phase, abort, status, kStatusTimeoutMma)) { ok = false; break; }
                tc_fence_after();
                const uint32_t a_s = smem_u32(sa + stage * kRTileA), b_s = smem_u32(sb + stage * kRTileBMax);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    tc_mma_bf16(tmem_base, sdesc_kmajor_sw128(a_s) + 2u * j, sdesc_kmajor_sw128(b_s) + 2u * j, idesc,
                                (c | j) != 0);
                tc_commit(&empty[stage]);
                if (++stage == kRStages) { stage = 0; phase ^= 1u; }
            }
            if (ok) tc_commit(acc_full);
        }
    } else {
        const int q = warp & 3;   // tensor-memory lane quadrant of this warp
        if (__all_sync(0xffffffffu, mbar_wait(acc_full, 0, abort, status, kStatusTimeoutEpilogue))) {
            tc_fence_after();
            const int t = m0 + 32 * q + lane;
            const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16);
            float* out = logits + (size_t)t * E;
            const bool vec = (E & 3) == 0;
            for (int c8 = 0; c8 < nt / 8; ++c8) {
                float v[8];
                tmem_ld8(taddr + 8 * c8, v);
                tmem_ld_wait();
                const int e0 = n0 + 8 * c8;
                if (t >= T || e0 >= E) continue;
                if (vec && e0 + 8 <= E) {
                    reinterpret_cast<float4*>(out + e0)[0] = make_float4(v[0], v[1], v[2], v[3]);
                    reinterpret_cast<float4*>(out + e0)[1] = make_float4(v[4], v[5], v[6], v[7]);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (e0 + i < E) out[e0 + i] = v[i];
                }
            }
        }
    }
    {
        // after an abort let in-flight copies land and retire issued MMAs
        volatile int no_abort = 0;
        if (*abort) {
            if (warp == 1 && lane == 0) {
                tc_commit(drain);
                mbar_wait(drain, 0, &no_abort, status, kStatusTimeoutMma);
            }
            for (int i = 0; i < 100; ++i) __nanosleep(10000);
        }
    }
    tc_fence_before();
    __syncthreads();
    pdl_launch_dependents();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kRTmemCols);
    }
}

}  // namespace

cudaError_t setup_router_gemm_kernel() {
    return cudaFuncSetAttribute(router_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRSmemBytes);
}

int router_gemm_tile_n(int E) {
    const int n = ((E + 15) / 16) * 16;
    return n < kRMaxN ? n : kRMaxN;
}

cudaError_t launch_router_gemm(const LaunchCtx& c, const CUtensorMap& tmX, const CUtensorMap& tmW, int T, int E,
                               int H, float* logits, unsigned int* status) {
    const int nt = router_gemm_tile_n(E);
    const dim3 grid((unsigned)((T + kRBM - 1) / kRBM), (unsigned)((E + kRMaxN - 1) / kRMaxN));
    return c.launch(router_gemm_kernel, grid, dim3(kRThreads), (size_t)kRSmemBytes, tmX, tmW, T, E, H, nt, logits,
                    status);
}

}  // namespace moe
