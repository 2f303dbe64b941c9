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
//   1 routes + per-unit expert token masks   (one warp per token; masks by
//                                             atomicOr, zeroed before launch)
//   2 scan, redundantly in every CTA: expert totals, offsets, padded offsets
//     and tile pairs in shared memory; the per-expert outputs (unit starting
//     rows, tile map, pair list, pad rows) spread over the grid
//   3 x quantization + row scatter + y_acc zeroing (a CTA per token when
//                                             T <= grid, else a warp per token)
//   4 FC1 tiles (SwiGLU / ReLU2, route weight, requant or FP32 store)
//   5 per-token FC2-input quantization        (one warp per row)
//   6 FC2 tiles (BF16 per-route rows or FP32 scatter)
//   7 finalize                                (grid-stride over elements)
// Phases 2 and 3 share one barrier interval when T <= 32 * kDirectUnits:
// a token's row is then its expert's padded offset (in every CTA's shared
// memory) plus the population counts of at most kDirectUnits unit masks.
// Every phase computes what the kernel of the default path for that step
// computes, with the same device arithmetic, so both paths give the same
// bits (up to the order of the fused finalize's FP32 atomic additions).
// The GEMM pipeline position carries over from FC1 to FC2.
//
// The row phases hand work out per warp over the whole grid (1 CTA per SM
// leaves only ten warps per SM, so per-CTA rows with CTA-wide reductions
// were latency-bound: a first version spent 33 us quantizing the mid
// workload's FC2 input, against 10 us for the standalone kernel), except
// that a token's x row is spread over a whole CTA when T is below the grid
// size (a single warp walking a 7168-wide row took ~14 dependent memory
// round trips), and every load loop keeps two blocks per thread in flight.
//
// A grid barrier is a counter (zeroed before the launch) that each CTA
// increments once per barrier (release) and polls (acquire); the generic ->
// async proxy fences around it make the operands written by the previous
// phase visible to the TMA copies of the next.  Data written inside the
// kernel by other CTAs is read with L2 (.cg) loads, never through the
// read-only path.  Every wait is bounded (1 s): a CTA that gives up raises
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
constexpr int kDirectUnits = 4;                    // phases 2 + 3 fused up to 4 units of 32 tokens

__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int* p) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// generic -> async proxy, global and shared memory: the TMA copies of the
// next phase read global data and overwrite shared scratch written by the
// generic proxy before
__device__ __forceinline__ void fence_proxy_async_all() { asm volatile("fence.proxy.async;" ::: "memory"); }

__device__ __forceinline__ int global_warp() { return blockIdx.x * kFusedWarps + (threadIdx.x >> 5); }
__device__ __forceinline__ int num_warps() { return gridDim.x * kFusedWarps; }

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

__device__ __forceinline__ void load16_f32_cg(const float* p, float (&v)[16]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 q = __ldcg(reinterpret_cast<const float4*>(p) + i);
        v[4 * i] = q.x; v[4 * i + 1] = q.y; v[4 * i + 2] = q.z; v[4 * i + 3] = q.w;
    }
}

// Scales of four consecutive blocks (four consecutive lanes) packed into the
// first lane's word; every lane of the warp takes part.
__device__ __forceinline__ uint32_t pack_sf4_fused(uint32_t s) {
    const uint32_t s1 = __shfl_down_sync(0xffffffffu, s, 1);
    const uint32_t s2 = __shfl_down_sync(0xffffffffu, s, 2);
    const uint32_t s3 = __shfl_down_sync(0xffffffffu, s, 3);
    return s | (s1 << 8) | (s2 << 16) | (s3 << 24);
}

// Phase 1: the routes of every token and the unit token masks of every
// expert (route_count_kernel / route_given_kernel).  Router: one warp per
// token.  Given ids: one warp per unit of 32 tokens, one lane per token,
// slots in order, so that a repeat of an earlier kept id finds its bit set.
__device__ void phase_route(const FusedParams& fp) {
    const int U = (fp.T + kUnitTokens - 1) / kUnitTokens;
    const int lane = threadIdx.x & 31;
    if (fp.ids_in == nullptr) {
        for (int t = global_warp(); t < fp.T; t += num_warps()) {
            const int e = route_token<kFusedEpl>(t, fp.E, fp.K, fp.logits, fp.bias, fp.renorm, fp.ids, fp.topk_w);
            if (e >= 0) atomicOr(fp.unit_mask + (size_t)e * U + t / kUnitTokens, 1u << (t % kUnitTokens));
        }
        return;
    }
    for (int u = global_warp(); u < U; u += num_warps()) {
        const int t = u * kUnitTokens + lane;
        if (t >= fp.T) continue;
        bool bad = false;
        for (int k = 0; k < fp.K; ++k) {
            const size_t r = (size_t)t * fp.K + k;
            int e = fp.ids_in[r];
            if (e >= 0 && e < fp.E) {
                if (atomicOr(fp.unit_mask + (size_t)e * U + u, 1u << lane) & (1u << lane)) e = -1;
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

// Phase 2 (permute_scan_kernel), in every CTA: the per-expert totals (the
// population counts of the unit masks), exclusive scans of the counts, the
// 128-padded counts and the M-tile pairs into shared memory (s_cnt, s_pad,
// s_pair); CTA 0 publishes count / offsets / padded_offsets / meta.  Then
// the per-expert outputs, expert e on CTA e % grid: the per-(expert, unit)
// starting rows, the tile map, the pair list and -1 in the pad rows.
__device__ void phase_scan(const FusedParams& fp, int* s_cnt, int* s_pad, int* s_pair, int* s_half) {
    const int U = (fp.T + kUnitTokens - 1) / kUnitTokens;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (U < 32) {
        // few units: a thread per expert, its loads independent (a warp per
        // expert would chain E / 10 dependent L2 round trips per warp)
        for (int e = threadIdx.x; e < fp.E; e += blockDim.x) {
            int sum = 0;
#pragma unroll 4
            for (int u = 0; u < U; ++u) sum += __popc(__ldcg(fp.unit_mask + (size_t)e * U + u));
            s_cnt[e] = sum;
        }
    } else {
        for (int e = warp; e < fp.E; e += kFusedWarps) {
            int sum = 0;
            for (int u = lane; u < U; u += 32) sum += __popc(__ldcg(fp.unit_mask + (size_t)e * U + u));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            if (lane == 0) s_cnt[e] = sum;
        }
    }
    __syncthreads();
    if (warp == 0) {
        int cc = 0, cp = 0, cq = 0, ch = 0;   // running totals of the earlier 32-expert groups
        for (int e0 = 0; e0 < fp.E; e0 += 32) {
            const int e = e0 + lane;
            const int c = e < fp.E ? s_cnt[e] : 0;
            const int p = (c + kTileM - 1) / kTileM * kTileM;
            const int q = (p / kTileM + 1) / 2;
            const int hv = (c + kTileM / 2 - 1) / (kTileM / 2);
            int ic = c, ip = p, iq = q, ih = hv;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int a = __shfl_up_sync(0xffffffffu, ic, o);
                const int b = __shfl_up_sync(0xffffffffu, ip, o);
                const int d = __shfl_up_sync(0xffffffffu, iq, o);
                const int f = __shfl_up_sync(0xffffffffu, ih, o);
                if (lane >= o) { ic += a; ip += b; iq += d; ih += f; }
            }
            if (e < fp.E) {
                s_pad[e] = cp + ip - p;
                s_pair[e] = cq + iq - q;
                s_half[e] = ch + ih - hv;
                if (blockIdx.x == 0) {
                    fp.count[e] = c;
                    fp.offsets[e] = cc + ic - c;
                    fp.padded_offsets[e] = cp + ip - p;
                }
            }
            cc += __shfl_sync(0xffffffffu, ic, 31);
            cp += __shfl_sync(0xffffffffu, ip, 31);
            cq += __shfl_sync(0xffffffffu, iq, 31);
            ch += __shfl_sync(0xffffffffu, ih, 31);
        }
        if (lane == 0) {
            s_pad[fp.E] = cp;
            if (blockIdx.x == 0) {
                fp.offsets[fp.E] = cc;
                fp.padded_offsets[fp.E] = cp;
                fp.meta[0] = cp;
                fp.meta[1] = cp / kTileM;
                fp.meta[2] = cq;
                fp.meta[3] = ch;
            }
        }
    }
    __syncthreads();
    for (int e = blockIdx.x + gridDim.x * warp; e < fp.E; e += gridDim.x * kFusedWarps) {
        int carry = s_pad[e];
        for (int u0 = 0; u0 < U; u0 += 32) {
            const int u = u0 + lane;
            const int v = u < U ? __popc(__ldcg(fp.unit_mask + (size_t)e * U + u)) : 0;
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
        const int nh = (cnt + kTileM / 2 - 1) / (kTileM / 2);
        for (int j = lane; j < nh; j += 32) fp.tile_half[s_half[e] + j] = ((r0 / kTileM + (j >> 1)) << 1) | (j & 1);
    }
}

// Rows of token t's routes (step 3 of the permutation), lane k < K of the
// calling warp taking route t*K+k; records both directions of the map and
// returns the row (-1 for a dropped route and for lanes >= K).  direct: the
// scan's unit starting rows are not published yet; the row is the expert's
// padded offset (s_pad) plus the counts of the token's earlier units.
__device__ __forceinline__ int token_route_row(const FusedParams& fp, int t, const int* s_pad, bool direct) {
    const int lane = threadIdx.x & 31;
    if (lane >= fp.K) return -1;
    const int U = (fp.T + kUnitTokens - 1) / kUnitTokens;
    const int r = t * fp.K + lane;
    const int e = __ldcg(fp.ids + r);
    int row = -1;
    if (e >= 0 && e < fp.E) {
        const int u = t / kUnitTokens;
        const size_t idx = (size_t)e * U + u;
        const uint32_t below = (1u << (t % kUnitTokens)) - 1u;
        int start;
        if (direct) {
            start = s_pad[e];
            for (int v = 0; v < u; ++v) start += __popc(__ldcg(fp.unit_mask + (size_t)e * U + v));
        } else {
            start = __ldcg(fp.unit_base + idx);
        }
        row = start + __popc(__ldcg(fp.unit_mask + idx) & below);
        fp.route_of_row[row] = r;
    }
    fp.row_of_route[r] = row;
    return row;
}

// Largest |x| of token t's row over the blocks g, g + kGroup, ... (two
// blocks per thread in flight).
template <int kGroup>
__device__ __forceinline__ float token_row_amax(const FusedParams& fp, int t, int g) {
    const int nblk = fp.H / 16;
    const __nv_bfloat16* xr = fp.x + (size_t)t * fp.H;
    float amax = 0.0f;
    for (int b0 = g; b0 < nblk; b0 += 2 * kGroup) {
        float v[2][16];
        const bool second = b0 + kGroup < nblk;
        load16_bf16_plain(xr + 16 * b0, v[0]);
        if (second) load16_bf16_plain(xr + 16 * (b0 + kGroup), v[1]);
#pragma unroll
        for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[0][j]));
        if (second) {
#pragma unroll
            for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[1][j]));
        }
    }
    return amax;
}

// NVFP4 codes and scales of token t's x row written to its K rows (rows[],
// shared memory) by a group of kGroup threads (a warp or the CTA), thread g
// of the group on blocks g, g + kGroup, ...; two blocks per thread in
// flight per step (explicit: the byte stores could alias x, so the compiler
// would not move a later load above them).
template <bool kFourSix, int kGroup>
__device__ __forceinline__ void quantize_token_row(const FusedParams& fp, int t, int g, float G, const int* rows) {
    const int H = fp.H, K = fp.K, nblk = H / 16, lane = threadIdx.x & 31;
    const __nv_bfloat16* xr = fp.x + (size_t)t * H;
    for (int b0 = 0; b0 < nblk; b0 += 2 * kGroup) {   // uniform across the group
        float v[2][16];
        bool act[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int b = b0 + i * kGroup + g;
            act[i] = b < nblk;
            if (act[i]) load16_bf16_plain(xr + 16 * b, v[i]);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            if (b0 + i * kGroup >= nblk) break;           // uniform: the group's first block
            const int b = b0 + i * kGroup + g;
            uint32_t q[2] = {0u, 0u};
            uint32_t s = 0;
            if (act[i]) s = kFourSix ? quant_block16_4over6(v[i], G, q) : quant_block16(v[i], G, q);
            const uint32_t word = pack_sf4_fused(s);
            if (!act[i]) continue;
            for (int k = 0; k < K; ++k) {
                const int row = rows[k];
                if (row < 0) continue;
                *reinterpret_cast<uint2*>(fp.xq_codes + (size_t)row * (H / 2) + 8 * b) = make_uint2(q[0], q[1]);
                if ((lane & 3) == 0) *reinterpret_cast<uint32_t*>(fp.xq_sf + sf_offset(row, b, H)) = word;
            }
        }
    }
}

// Phase 3 (quantize_x_kernel): the token's rows, the per-token G1 from the
// row amax (per-token mode), the NVFP4 codes and scales in each of the K
// rows, the zeroing of the fused-finalize accumulator row.  A CTA per token
// when the tokens fit the grid (small T: the row's blocks spread over 320
// threads), else a warp per token.  s_rows: [kFusedWarps][32], s_red:
// [kFusedWarps].
template <bool kFourSix>
__device__ void phase_quantize_x(const FusedParams& fp, const int* s_pad, bool direct, int* s_rows, float* s_red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int H = fp.H;
    if (fp.T <= (int)gridDim.x) {
        const int t = blockIdx.x;
        if (t >= fp.T) return;                           // uniform across the CTA
        if (warp == 0) {
            const int row = token_route_row(fp, t, s_pad, direct);
            if (lane < fp.K) s_rows[lane] = row;
        }
        float G;
        if (fp.per_token) {
            float amax = warp_max(token_row_amax<kFusedThreads>(fp, t, threadIdx.x));
            if (lane == 0) s_red[warp] = amax;
            __syncthreads();
            amax = s_red[0];
#pragma unroll
            for (int w = 1; w < kFusedWarps; ++w) amax = fmaxf(amax, s_red[w]);
            G = kFourSix ? global_scale_from_amax_4over6(amax) : global_scale_from_amax(amax);
            if (threadIdx.x == 0) fp.g1[t] = G;
        } else {
            G = __ldg(fp.g1_in);
            __syncthreads();                             // s_rows
        }
        quantize_token_row<kFourSix, kFusedThreads>(fp, t, threadIdx.x, G, s_rows);
        if (!fp.det) {
            float* yr = fp.y_acc + (size_t)t * H;
            for (int c = threadIdx.x * 4; c < H; c += kFusedThreads * 4)
                *reinterpret_cast<float4*>(yr + c) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        return;
    }
    int* rows = s_rows + warp * 32;
    for (int t = global_warp(); t < fp.T; t += num_warps()) {
        const int row = token_route_row(fp, t, s_pad, direct);
        if (lane < fp.K) rows[lane] = row;
        __syncwarp();
        float G;
        if (fp.per_token) {
            const float amax = warp_max(token_row_amax<32>(fp, t, lane));
            G = kFourSix ? global_scale_from_amax_4over6(amax) : global_scale_from_amax(amax);
            if (lane == 0) fp.g1[t] = G;
        } else {
            G = __ldg(fp.g1_in);
        }
        quantize_token_row<kFourSix, 32>(fp, t, lane, G, rows);
        if (!fp.det) {
            float* yr = fp.y_acc + (size_t)t * H;
            for (int c = lane * 4; c < H; c += 128) *reinterpret_cast<float4*>(yr + c) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        __syncwarp();                                    // rows is reused by the next token
    }
}

// Phase 5 (per-token mode; quantize_h_kernel), one warp per padded row: the
// valid FC2 input rows -> G2 = amax / 2688 (or / 1536 with 4-over-6 blocks)
// and NVFP4 codes and scales; two blocks per lane in flight per step.
template <bool kFourSix>
__device__ void phase_quantize_h(const FusedParams& fp) {
    const int lane = threadIdx.x & 31;
    const int I = fp.I, nblk = I / 16;
    const int rows = __ldcg(fp.meta);
    for (int row = global_warp(); row < rows; row += num_warps()) {
        if (__ldcg(fp.route_of_row + row) < 0) continue;   // pad row (uniform across the warp)
        const float* hr = fp.h_f32 + (size_t)row * I;
        float amax = 0.0f;
        for (int b0 = lane; b0 < nblk; b0 += 64) {
            float v[2][16];
            const bool second = b0 + 32 < nblk;
            load16_f32_cg(hr + 16 * b0, v[0]);
            if (second) load16_f32_cg(hr + 16 * (b0 + 32), v[1]);
#pragma unroll
            for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[0][j]));
            if (second) {
#pragma unroll
                for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[1][j]));
            }
        }
        amax = warp_max(amax);
        const float G = kFourSix ? global_scale_from_amax_4over6(amax) : global_scale_from_amax(amax);
        if (lane == 0) fp.g2[row] = G;
        for (int b0 = 0; b0 < nblk; b0 += 64) {        // uniform across the warp
            float v[2][16];
            bool act[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int b = b0 + 32 * i + lane;
                act[i] = b < nblk;
                if (act[i]) load16_f32_cg(hr + 16 * b, v[i]);
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                if (b0 + 32 * i >= nblk) break;
                const int b = b0 + 32 * i + lane;
                uint32_t q[2] = {0u, 0u};
                uint32_t s = 0;
                if (act[i]) s = kFourSix ? quant_block16_4over6(v[i], G, q) : quant_block16(v[i], G, q);
                const uint32_t word = pack_sf4_fused(s);
                if (act[i]) {
                    *reinterpret_cast<uint2*>(fp.hq_codes + (size_t)row * (I / 2) + 8 * b) = make_uint2(q[0], q[1]);
                    if ((lane & 3) == 0) *reinterpret_cast<uint32_t*>(fp.hq_sf + sf_offset(row, b, I)) = word;
                }
            }
        }
    }
}

// Phase 7 (finalize_fused_kernel / finalize_det_kernel), grid-stride over
// groups of 8 output elements.
__device__ void phase_finalize(const FusedParams& fp) {
    const int H = fp.H, K = fp.K, H8 = H / 8;
    const int64_t n8 = (int64_t)fp.T * H8;
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    if (!fp.det) {
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += step) {
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
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += step) {
        const int t = (int)(i / H8), c = (int)(i % H8);
        float acc[8];
        finalize_det_group(t, c, H, K, fp.row_of_route, fp.topk_w, fp.weight_on_output, fp.o_bf16, acc);
        reinterpret_cast<uint4*>(fp.y)[i] = pack_bf16x8(acc);
    }
}

}  // namespace

template <bool kFourSix>
__global__ void __launch_bounds__(kFusedThreads, 1)
    fused_layer_kernel(const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
                       const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2,
                       const __grid_constant__ FusedParams fp) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ int s_rows[kFusedWarps * 32];
    __shared__ float s_red[kFusedWarps];
    const grouped::Smem s = grouped::carve<128, 0>(smem_raw);
    // the operand ring is idle until FC1: the scan keeps its per-expert
    // tables in it (the TMA copies of FC1 start after a grid barrier, whose
    // proxy fence orders these generic writes before them)
    int* s_cnt = reinterpret_cast<int*>(s.a);
    int* s_pad = s_cnt + kFusedMaxExperts;          // E + 1 entries
    int* s_pair = s_pad + kFusedMaxExperts + 1;
    int* s_half = s_pair + kFusedMaxExperts;
    if (threadIdx.x == 0) {
        prefetch_tensormap(&tmA1);
        prefetch_tensormap(&tmB1);
        prefetch_tensormap(&tmA2);
        prefetch_tensormap(&tmB2);
    }
    const uint32_t tmem_base = grouped::gemm_init<128, 0>(s);
    grouped::RingState rs;
    unsigned int nb = 0;
    const bool direct = (fp.T + kUnitTokens - 1) / kUnitTokens <= kDirectUnits;

    phase_route(fp);
    bool ok = grid_barrier(fp, ++nb, s.abort);
    if (ok) {
        phase_scan(fp, s_cnt, s_pad, s_pair, s_half);
        if (!direct) ok = grid_barrier(fp, ++nb, s.abort);
    }
    if (ok) {
        phase_quantize_x<kFourSix>(fp, s_pad, direct, s_rows, s_red);
        ok = grid_barrier(fp, ++nb, s.abort);
    }
    if (ok) {
        if (fp.per_token) grouped::gemm_tiles<kEpiFc1F32, 128, 0>(s, tmem_base, &tmA1, &tmB1, fp.fc1, rs);
        else grouped::gemm_tiles<kEpiFc1Quant, 128, 0>(s, tmem_base, &tmA1, &tmB1, fp.fc1, rs);
        ok = grid_barrier(fp, ++nb, s.abort);   // fails if the tile loop set the abort flag
    }
    if (ok && fp.per_token) {
        phase_quantize_h<kFourSix>(fp);
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
