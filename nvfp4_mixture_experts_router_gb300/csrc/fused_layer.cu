// The whole W4A4 layer forward as ONE persistent kernel (MOE_FUSED_LAYER),
// the single-GPU form of the MegaMoE design ["MegaMoE" blog, "Our approach":
// one persistent kernel per forward pass runs the quantization, both grouped
// GEMMs and the combine].  Meant for small token counts, where the six or
// seven launches of the default path and the ramp-up and drain of each cost
// more than the work.
//
// One CTA per SM (cooperative launch, so that every CTA is resident) with the
// grouped GEMM's warp roles and shared-memory pipeline (gemm_nvf4.cuh,
// 128-wide tiles) and grid-wide barriers between the phases:
//   1 router or given ids + per-unit expert masks  (units of 32 tokens)
//   2 scan: offsets, tile map, pairs, unit rows     (CTA 0)
//   3 x quantization + row scatter + y_acc zeroing  (tokens)
//   4 FC1 tiles (SwiGLU / ReLU2, route weight, requant or FP32 store)
//   5 per-token FC2-input quantization              (rows; per-token mode)
//   6 FC2 tiles (BF16 per-route rows or FP32 scatter)
//   7 finalize                                      (tokens / elements)
// Every phase computes what the kernel of the default path for that step
// computes, with the same device arithmetic, so both paths give the same
// bits (up to the order of the fused finalize's FP32 atomic additions).
// The GEMM pipeline position carries over from FC1 to FC2.
//
// A grid barrier is a counter (zeroed before the launch) that each CTA
// increments once per barrier (release) and polls (acquire); the generic ->
// async proxy fences around it make the operands written by the previous
// phase visible to the TMA copies of the next.  Data written inside the
// kernel is read with plain or L2 (.cg) loads, never through the read-only
// path.  Every wait is bounded (1 s): a CTA that gives up raises
// kStatusGridAbort, and the others stop at their next barrier.
#include "gemm_nvf4.cuh"
#include "kernels.h"
#include "routing.cuh"

namespace moe {

namespace {

using FC = grouped::Cfg<128, 0>;   // one pipeline configuration for both GEMMs
constexpr int kFusedThreads = FC::kNumThreads;
constexpr int kFusedWarps = kFusedThreads / 32;
constexpr int kFusedEpl = kFusedMaxExperts / 32;   // router: experts per lane

__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int* p) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// generic -> async proxy, global and shared memory: the TMA copies of the
// next phase read global data and overwrite shared scratch written by the
// generic proxy before
__device__ __forceinline__ void fence_proxy_async_all() { asm volatile("fence.proxy.async;" ::: "memory"); }

// Grid-wide barrier number n (1, 2, ...).  Returns false (and sets the CTA's
// abort flag) if this CTA arrives failed or another CTA has failed.
__device__ bool grid_barrier(const FusedParams& fp, unsigned int n, volatile int* abort) {
    __shared__ int s_ok;
    fence_proxy_async_all();
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = *abort == 0;
        if (ok) {
            __threadfence();
            atomicAdd(fp.sync, 1u);
            const unsigned int target = n * gridDim.x;
            const uint64_t t0 = global_timer_ns();
            while (ld_acquire_gpu(fp.sync) < target) {
                if (ld_acquire_gpu(fp.status) & kStatusGridAbort) { ok = 0; break; }
                if (global_timer_ns() - t0 > kWaitLimitNs) {
                    atomicOr(fp.status, kStatusTimeoutGrid | kStatusGridAbort);
                    ok = 0;
                    break;
                }
                __nanosleep(32);
            }
        } else {
            atomicOr(fp.status, kStatusGridAbort);
        }
        if (!ok) *abort = 1;
        s_ok = ok;
    }
    __syncthreads();
    fence_proxy_async_all();
    return s_ok != 0;
}

// Phase 1: per unit of 32 tokens (one unit per CTA at a time) the routes and
// the unit's token mask of every expert (route_count_kernel /
// route_given_kernel).
__device__ void phase_route(const FusedParams& fp, uint32_t* s_mask) {
    const int U = (fp.T + kUnitTokens - 1) / kUnitTokens;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int u = blockIdx.x; u < U; u += gridDim.x) {
        for (int e = threadIdx.x; e < fp.E; e += blockDim.x) s_mask[e] = 0u;
        __syncthreads();
        if (fp.ids_in == nullptr) {
            for (int j = warp; j < kUnitTokens; j += kFusedWarps) {   // one warp per token
                const int t = u * kUnitTokens + j;
                if (t < fp.T) {
                    const int e = route_token<kFusedEpl>(t, fp.E, fp.K, fp.logits, fp.bias, fp.renorm, fp.ids,
                                                         fp.topk_w);
                    if (e >= 0) atomicOr(&s_mask[e], 1u << j);
                }
            }
        } else if (warp == 0) {                                        // one lane per token
            const int t = u * kUnitTokens + lane;
            if (t < fp.T) {
                bool bad = false;
                for (int k = 0; k < fp.K; ++k) {
                    const size_t r = (size_t)t * fp.K + k;
                    int e = fp.ids_in[r];
                    if (e >= 0 && e < fp.E) {
                        // a repeat of an earlier kept id finds its bit set
                        if (atomicOr(&s_mask[e], 1u << lane) & (1u << lane)) e = -1;
                    } else {
                        e = -1;
                    }
                    bad |= e < 0;
                    fp.ids[r] = e;
                    fp.topk_w[r] = fp.w_in[r];
                }
                if (bad) atomicOr(fp.status, kStatusBadExpert);
            }
        }
        __syncthreads();
        for (int e = threadIdx.x; e < fp.E; e += blockDim.x) {
            const uint32_t m = s_mask[e];
            fp.unit_base[(size_t)e * U + u] = __popc(m);
            fp.unit_mask[(size_t)e * U + u] = m;
        }
        __syncthreads();
    }
}

// Phase 2 (CTA 0): per-expert totals, exclusive offsets of the counts, the
// 128-padded counts and the M-tile pairs; the per-(expert, unit) starting
// rows in place of the counts; tile map, pair list and -1 in the pad rows
// (permute_scan_kernel).
__device__ void phase_scan(const FusedParams& fp, int* s_cnt, int* s_pad, int* s_pair) {
    const int U = (fp.T + kUnitTokens - 1) / kUnitTokens;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int e = warp; e < fp.E; e += kFusedWarps) {
        int sum = 0;
        for (int u = lane; u < U; u += 32) sum += fp.unit_base[(size_t)e * U + u];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane == 0) s_cnt[e] = sum;
    }
    __syncthreads();
    if (warp == 0) {
        int cc = 0, cp = 0, cq = 0;   // running totals of the earlier 32-expert groups
        for (int e0 = 0; e0 < fp.E; e0 += 32) {
            const int e = e0 + lane;
            const int c = e < fp.E ? s_cnt[e] : 0;
            const int p = (c + kTileM - 1) / kTileM * kTileM;
            const int q = (p / kTileM + 1) / 2;
            int ic = c, ip = p, iq = q;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int a = __shfl_up_sync(0xffffffffu, ic, o);
                const int b = __shfl_up_sync(0xffffffffu, ip, o);
                const int d = __shfl_up_sync(0xffffffffu, iq, o);
                if (lane >= o) { ic += a; ip += b; iq += d; }
            }
            if (e < fp.E) {
                fp.count[e] = c;
                fp.offsets[e] = cc + ic - c;
                fp.padded_offsets[e] = cp + ip - p;
                s_pad[e] = cp + ip - p;
                s_pair[e] = cq + iq - q;
            }
            cc += __shfl_sync(0xffffffffu, ic, 31);
            cp += __shfl_sync(0xffffffffu, ip, 31);
            cq += __shfl_sync(0xffffffffu, iq, 31);
        }
        if (lane == 0) {
            fp.offsets[fp.E] = cc;
            fp.padded_offsets[fp.E] = cp;
            fp.meta[0] = cp;
            fp.meta[1] = cp / kTileM;
            fp.meta[2] = cq;
        }
    }
    __syncthreads();
    for (int e = warp; e < fp.E; e += kFusedWarps) {
        int carry = s_pad[e];
        for (int u0 = 0; u0 < U; u0 += 32) {
            const int u = u0 + lane;
            const int v = u < U ? fp.unit_base[(size_t)e * U + u] : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int a = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += a;
            }
            if (u < U) fp.unit_base[(size_t)e * U + u] = carry + incl - v;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        const int cnt = s_cnt[e];
        const int pcnt = (cnt + kTileM - 1) / kTileM * kTileM;
        const int r0 = s_pad[e];
        for (int r = r0 + cnt + lane; r < r0 + pcnt; r += 32) fp.route_of_row[r] = -1;
        for (int tl = r0 / kTileM + lane; tl < (r0 + pcnt) / kTileM; tl += 32) fp.tile_expert[tl] = e;
        const int nt = pcnt / kTileM;
        for (int i = lane; 2 * i < nt; i += 32)
            fp.tile_pair[s_pair[e] + i] = ((r0 / kTileM + 2 * i) << 1) | (2 * i + 1 < nt ? 1 : 0);
    }
}

__device__ __forceinline__ void load16_bf16_plain(const __nv_bfloat16* p, float (&v)[16]) {
    const uint4 a = *reinterpret_cast<const uint4*>(p);
    const uint4 b = *reinterpret_cast<const uint4*>(p + 8);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// Scales of four consecutive blocks (four consecutive lanes) packed into the
// first lane's word.
__device__ __forceinline__ uint32_t pack_sf4_fused(uint32_t s) {
    const uint32_t s1 = __shfl_down_sync(0xffffffffu, s, 1);
    const uint32_t s2 = __shfl_down_sync(0xffffffffu, s, 2);
    const uint32_t s3 = __shfl_down_sync(0xffffffffu, s, 3);
    return s | (s1 << 8) | (s2 << 16) | (s3 << 24);
}

// CTA-wide maximum of v (every thread gets it); s_red holds kFusedWarps floats.
__device__ __forceinline__ float cta_max(float v, float* s_red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_max(v);
    if (lane == 0) s_red[warp] = v;
    __syncthreads();
    float m = lane < kFusedWarps ? s_red[lane] : 0.0f;
    m = warp_max(m);
    __syncthreads();                                   // s_red is reused
    return m;
}

// Phase 3: x quantization into the token's K permuted rows, the row scatter
// (step 3 of the permutation) and the zeroing of the token's fused-finalize
// accumulator row (quantize_x_kernel).
template <bool kFourSix>
__device__ void phase_quantize_x(const FusedParams& fp, int* s_rows, float* s_red) {
    const int U = (fp.T + kUnitTokens - 1) / kUnitTokens;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = fp.H, K = fp.K, nblk = H / 16;
    for (int t = blockIdx.x; t < fp.T; t += gridDim.x) {
        if (warp == 0 && lane < K) {
            const int r = t * K + lane;
            const int e = fp.ids[r];
            int row = -1;
            if (e >= 0 && e < fp.E) {
                const size_t idx = (size_t)e * U + t / kUnitTokens;
                const uint32_t below = (1u << (t % kUnitTokens)) - 1u;
                row = __ldcg(fp.unit_base + idx) + __popc(__ldcg(fp.unit_mask + idx) & below);
                fp.route_of_row[row] = r;
            }
            fp.row_of_route[r] = row;
            s_rows[lane] = row;
        }
        const __nv_bfloat16* xr = fp.x + (size_t)t * H;
        float G;
        if (fp.per_token) {
            float amax = 0.0f;
            for (int b = tid; b < nblk; b += blockDim.x) {
                float v[16];
                load16_bf16_plain(xr + 16 * b, v);
#pragma unroll
                for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
            }
            const float m = cta_max(amax, s_red);
            G = kFourSix ? global_scale_from_amax_4over6(m) : global_scale_from_amax(m);
            if (tid == 0) fp.g1[t] = G;
        } else {
            G = __ldg(fp.g1_in);
            __syncthreads();                                // s_rows
        }
        for (int b0 = 0; b0 < nblk; b0 += blockDim.x) {   // uniform across the CTA
            const int b = b0 + tid;
            const bool active = b < nblk;
            uint32_t q[2] = {0u, 0u};
            uint32_t s = 0;
            if (active) {
                float v[16];
                load16_bf16_plain(xr + 16 * b, v);
                s = kFourSix ? quant_block16_4over6(v, G, q) : quant_block16(v, G, q);
            }
            const uint32_t word = pack_sf4_fused(s);
            if (active) {
                for (int k = 0; k < K; ++k) {
                    const int row = s_rows[k];
                    if (row < 0) continue;
                    *reinterpret_cast<uint2*>(fp.xq_codes + (size_t)row * (H / 2) + 8 * b) = make_uint2(q[0], q[1]);
                    if ((lane & 3) == 0) *reinterpret_cast<uint32_t*>(fp.xq_sf + sf_offset(row, b, H)) = word;
                }
            }
        }
        if (!fp.det) {
            float* yr = fp.y_acc + (size_t)t * H;
            for (int c = tid * 4; c < H; c += blockDim.x * 4)
                *reinterpret_cast<float4*>(yr + c) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        __syncthreads();                                    // s_rows is reused by the next token
    }
}

// Phase 5 (per-token mode): each valid FC2 input row -> G2 = amax / 2688
// (or / 1536 with 4-over-6 blocks) and NVFP4 codes and scales
// (quantize_h_kernel).
template <bool kFourSix>
__device__ void phase_quantize_h(const FusedParams& fp, float* s_red) {
    const int tid = threadIdx.x, lane = tid & 31;
    const int I = fp.I, nblk = I / 16;
    const int rows = fp.meta[0];
    for (int row = blockIdx.x; row < rows; row += gridDim.x) {
        if (fp.route_of_row[row] < 0) continue;   // pad row (uniform across the CTA)
        const float* hr = fp.h_f32 + (size_t)row * I;
        float amax = 0.0f;
        for (int b = tid; b < nblk; b += blockDim.x) {
            const float4* p4 = reinterpret_cast<const float4*>(hr + 16 * b);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float4 q = p4[j];
                amax = fmaxf(amax, fmaxf(fmaxf(fabsf(q.x), fabsf(q.y)), fmaxf(fabsf(q.z), fabsf(q.w))));
            }
        }
        const float m = cta_max(amax, s_red);
        const float G = kFourSix ? global_scale_from_amax_4over6(m) : global_scale_from_amax(m);
        if (tid == 0) fp.g2[row] = G;
        for (int b0 = 0; b0 < nblk; b0 += blockDim.x) {
            const int b = b0 + tid;
            const bool active = b < nblk;
            uint32_t q[2] = {0u, 0u};
            uint32_t s = 0;
            if (active) {
                float v[16];
                const float4* p4 = reinterpret_cast<const float4*>(hr + 16 * b);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float4 x4 = p4[j];
                    v[4 * j] = x4.x; v[4 * j + 1] = x4.y; v[4 * j + 2] = x4.z; v[4 * j + 3] = x4.w;
                }
                s = kFourSix ? quant_block16_4over6(v, G, q) : quant_block16(v, G, q);
            }
            const uint32_t word = pack_sf4_fused(s);
            if (active) {
                *reinterpret_cast<uint2*>(fp.hq_codes + (size_t)row * (I / 2) + 8 * b) = make_uint2(q[0], q[1]);
                if ((lane & 3) == 0) *reinterpret_cast<uint32_t*>(fp.hq_sf + sf_offset(row, b, I)) = word;
            }
        }
    }
}

// Phase 7: finalize (finalize_fused_kernel / finalize_det_kernel).
__device__ void phase_finalize(const FusedParams& fp) {
    const int H = fp.H, K = fp.K;
    if (!fp.det) {
        const int64_t n8 = (int64_t)fp.T * H / 8;
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
            const float4 a = __ldcg(reinterpret_cast<const float4*>(fp.y_acc) + 2 * i);
            const float4 b = __ldcg(reinterpret_cast<const float4*>(fp.y_acc) + 2 * i + 1);
            const __nv_bfloat162 p0 = __floats2bfloat162_rn(a.x, a.y), p1 = __floats2bfloat162_rn(a.z, a.w);
            const __nv_bfloat162 p2 = __floats2bfloat162_rn(b.x, b.y), p3 = __floats2bfloat162_rn(b.z, b.w);
            reinterpret_cast<uint4*>(fp.y)[i] =
                make_uint4(*reinterpret_cast<const uint32_t*>(&p0), *reinterpret_cast<const uint32_t*>(&p1),
                           *reinterpret_cast<const uint32_t*>(&p2), *reinterpret_cast<const uint32_t*>(&p3));
        }
        return;
    }
    for (int t = blockIdx.x; t < fp.T; t += gridDim.x) {
        for (int c = threadIdx.x; c < H / 8; c += blockDim.x) {
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int k = 0; k < K; ++k) {
                const int row = fp.row_of_route[(size_t)t * K + k];
                if (row < 0) continue;   // dropped route
                const float w = fp.weight_on_output ? fp.topk_w[(size_t)t * K + k] : 1.0f;
                const uint4 v = __ldcg(reinterpret_cast<const uint4*>(fp.o_bf16 + (size_t)row * H) + c);
                const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[2 * i] = fmaf(w, __uint_as_float(u[i] << 16), acc[2 * i]);
                    acc[2 * i + 1] = fmaf(w, __uint_as_float(u[i] & 0xFFFF0000u), acc[2 * i + 1]);
                }
            }
            uint32_t out[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
                out[i] = *reinterpret_cast<const uint32_t*>(&b);
            }
            reinterpret_cast<uint4*>(fp.y + (size_t)t * H)[c] = make_uint4(out[0], out[1], out[2], out[3]);
        }
    }
}

}  // namespace

template <bool kFourSix>
__global__ void __launch_bounds__(kFusedThreads, 1)
    fused_layer_kernel(const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
                       const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2,
                       const __grid_constant__ FusedParams fp) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ int s_rows[32];
    __shared__ float s_red[32];
    const grouped::Smem s = grouped::carve<128, 0>(smem_raw);
    // the operand ring is idle until FC1: phases 1 and 2 keep their
    // per-expert scratch in it
    uint32_t* s_mask = reinterpret_cast<uint32_t*>(s.a);
    int* s_cnt = reinterpret_cast<int*>(s.a) + kFusedMaxExperts;
    int* s_pad = s_cnt + kFusedMaxExperts;
    int* s_pair = s_pad + kFusedMaxExperts;
    if (threadIdx.x == 0) {
        prefetch_tensormap(&tmA1);
        prefetch_tensormap(&tmB1);
        prefetch_tensormap(&tmA2);
        prefetch_tensormap(&tmB2);
    }
    const uint32_t tmem_base = grouped::gemm_init<128, 0>(s);
    grouped::RingState rs;
    unsigned int nb = 0;

    phase_route(fp, s_mask);
    bool ok = grid_barrier(fp, ++nb, s.abort);
    if (ok) {
        if (blockIdx.x == 0) phase_scan(fp, s_cnt, s_pad, s_pair);
        ok = grid_barrier(fp, ++nb, s.abort);
    }
    if (ok) {
        phase_quantize_x<kFourSix>(fp, s_rows, s_red);
        ok = grid_barrier(fp, ++nb, s.abort);
    }
    if (ok) {
        if (fp.per_token) grouped::gemm_tiles<kEpiFc1F32, 128, 0>(s, tmem_base, &tmA1, &tmB1, fp.fc1, rs);
        else grouped::gemm_tiles<kEpiFc1Quant, 128, 0>(s, tmem_base, &tmA1, &tmB1, fp.fc1, rs);
        ok = grid_barrier(fp, ++nb, s.abort);   // fails if the tile loop set the abort flag
    }
    if (ok && fp.per_token) {
        phase_quantize_h<kFourSix>(fp, s_red);
        ok = grid_barrier(fp, ++nb, s.abort);
    }
    if (ok) {
        if (fp.det) grouped::gemm_tiles<kEpiFc2Store, 128, 0>(s, tmem_base, &tmA2, &tmB2, fp.fc2, rs);
        else grouped::gemm_tiles<kEpiFc2Scatter, 128, 0>(s, tmem_base, &tmA2, &tmB2, fp.fc2, rs);
        ok = grid_barrier(fp, ++nb, s.abort);
    }
    if (ok) phase_finalize(fp);

    grouped::gemm_drain<128, 0>(s, fp.status);
    tc_fence_before();
    __syncthreads();
    grouped::gemm_free_tmem(tmem_base);
}

cudaError_t setup_fused_layer_kernel() {
    cudaError_t e = cudaFuncSetAttribute(fused_layer_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         FC::kSmemBytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(fused_layer_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                FC::kSmemBytes);
}

cudaError_t launch_fused_layer(cudaStream_t stream, int num_sms, const CUtensorMap& tmA1, const CUtensorMap& tmB1,
                               const CUtensorMap& tmA2, const CUtensorMap& tmB2, const FusedParams& fp,
                               bool four_six) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)num_sms);
    cfg.blockDim = dim3(kFusedThreads);
    cfg.dynamicSmemBytes = FC::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;   // every CTA resident: the grid barriers rely on it
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return four_six ? cudaLaunchKernelEx(&cfg, fused_layer_kernel<true>, tmA1, tmB1, tmA2, tmB2, fp)
                    : cudaLaunchKernelEx(&cfg, fused_layer_kernel<false>, tmA1, tmB1, tmA2, tmB2, fp);
}

}  // namespace moe
