// Router (softmax + top-K) and token permutation by expert.
//
// Router ["MegaMoE" blog, "The problem": each token goes to its top-K
// experts]: one warp per token, the E logits spread over the lanes
// (expert e = lane + 32 i), K rounds of a warp-wide arg-max.  Selection on
// l = logit + bias, ties to the lower expert index; the order of l is the
// order of the softmax probabilities.  Weights: softmax over the K selected
// (default) or the full softmax over E evaluated at the selected experts.
//
// Permutation [FlashInfer PR #4366: the grouped GEMM reads each expert's
// routes as one contiguous, tile-padded segment; "Tests": cluster padding
// and partial tiles]: a stable counting sort.  Tokens are cut into units of
// 32; (1) each unit counts its routes per expert, (2) one block scans the
// counts into per-expert totals, offsets, 128-row padded offsets and a
// per-(expert, unit) starting row, (3) each unit walks its tokens in order
// and hands out consecutive rows.  Within an expert the routes therefore sit
// in ascending token order, which makes the permutation unique.
#include "common.cuh"
#include "kernels.h"

namespace moe {

template <int EPL>
__global__ void __launch_bounds__(256) router_topk_kernel(int T, int E, int K, const float* __restrict__ logits,
                                                          const float* __restrict__ bias, int renorm,
                                                          int* __restrict__ topk_ids, float* __restrict__ topk_w,
                                                          unsigned int* status_reset) {
    pdl_wait();
    // the first kernel of a forward clears the device status word
    if (status_reset && blockIdx.x == 0 && threadIdx.x == 0) *status_reset = 0u;
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    float l[EPL];
    uint32_t taken = 0;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E) {
            float v = __ldg(logits + (size_t)t * E + e);
            if (bias) v = __fadd_rn(v, __ldg(bias + e));
            l[i] = v;
        } else {
            l[i] = -INFINITY;
            taken |= 1u << i;
        }
    }
    float sel_v[32];
    int sel_e[32];
    for (int k = 0; k < K; ++k) {
        float bv = -INFINITY;
        int be = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            if (!(taken & (1u << i)) && (be == 0x7fffffff || l[i] > bv)) {
                bv = l[i];
                be = lane + 32 * i;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oe = __shfl_xor_sync(0xffffffffu, be, o);
            if (oe != 0x7fffffff && (be == 0x7fffffff || ov > bv || (ov == bv && oe < be))) {
                bv = ov;
                be = oe;
            }
        }
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        sel_v[k] = bv;
        sel_e[k] = be;
    }
    const float lmax = sel_v[0];
    float den = 0.0f;
    if (renorm) {
        for (int k = 0; k < K; ++k) den += expf(sel_v[k] - lmax);
    } else {
        float part = 0.0f;
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if (lane + 32 * i < E) part += expf(l[i] - lmax);
        den = warp_sum(part);
    }
    for (int k = lane; k < K; k += 32) {
        // register arrays indexed by a lane-dependent k: select by loop
        float v = 0.0f;
        int e = 0;
        for (int j = 0; j < K; ++j)
            if (j == k) { v = sel_v[j]; e = sel_e[j]; }
        topk_ids[(size_t)t * K + k] = e;
        topk_w[(size_t)t * K + k] = expf(v - lmax) / den;
    }
    pdl_launch_dependents();
}

// (1) per-unit histogram: warp w of the block handles unit blockIdx.x*8+w.
__global__ void __launch_bounds__(256) permute_count_kernel(int T, int E, int K, const int* __restrict__ topk_ids,
                                                            int* __restrict__ unit_cnt /* [E][U] */,
                                                            unsigned int* status) {
    extern __shared__ int s_hist[];  // [8][E]
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int U = (T + kUnitTokens - 1) / kUnitTokens;
    const int u = blockIdx.x * 8 + warp;
    int* h = s_hist + warp * E;
    for (int e = lane; e < E; e += 32) h[e] = 0;
    __syncwarp();
    if (u < U) {
        const int t = u * kUnitTokens + lane;
        if (t < T) {
            for (int k = 0; k < K; ++k) {
                const int e = topk_ids[(size_t)t * K + k];
                if (e >= 0 && e < E) atomicAdd(&h[e], 1);
                else atomicOr(status, kStatusBadExpert);
            }
        }
        __syncwarp();
        for (int e = lane; e < E; e += 32) unit_cnt[(size_t)e * U + u] = h[e];
    }
    pdl_launch_dependents();
}

// (2) one block of 1024 threads: totals, offsets, padded offsets, per-unit
// starting rows, M-tile -> expert map, pad rows of route_of_row set to -1.
__global__ void __launch_bounds__(1024) permute_scan_kernel(int T, int E, int* __restrict__ unit_base /* [E][U] */,
                                                            int* __restrict__ count, int* __restrict__ offsets,
                                                            int* __restrict__ padded_offsets, int* __restrict__ meta,
                                                            int* __restrict__ tile_expert,
                                                            int* __restrict__ route_of_row) {
    __shared__ int s_cnt[1024];
    __shared__ int s_pad[1024];
    __shared__ int s_warp[2][32];
    pdl_wait();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int U = (T + kUnitTokens - 1) / kUnitTokens;
    // totals per expert
    for (int e = warp; e < E; e += 32) {
        int s = 0;
        for (int u = lane; u < U; u += 32) s += unit_base[(size_t)e * U + u];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) s_cnt[e] = s;
    }
    __syncthreads();
    // exclusive scans over experts of count and of the padded count
    const int c = tid < E ? s_cnt[tid] : 0;
    const int p = tid < E ? (c + kTileM - 1) / kTileM * kTileM : 0;
    int ic = c, ip = p;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, ic, o);
        const int b = __shfl_up_sync(0xffffffffu, ip, o);
        if (lane >= o) { ic += a; ip += b; }
    }
    if (lane == 31) { s_warp[0][warp] = ic; s_warp[1][warp] = ip; }
    __syncthreads();
    if (warp == 0) {
        int a = s_warp[0][lane], b = s_warp[1][lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int x = __shfl_up_sync(0xffffffffu, a, o);
            const int y = __shfl_up_sync(0xffffffffu, b, o);
            if (lane >= o) { a += x; b += y; }
        }
        s_warp[0][lane] = a;
        s_warp[1][lane] = b;
    }
    __syncthreads();
    const int base_c = warp > 0 ? s_warp[0][warp - 1] : 0;
    const int base_p = warp > 0 ? s_warp[1][warp - 1] : 0;
    const int ex_c = base_c + ic - c, ex_p = base_p + ip - p;
    if (tid < E) {
        count[tid] = c;
        offsets[tid] = ex_c;
        padded_offsets[tid] = ex_p;
        s_pad[tid] = ex_p;
    }
    if (tid == E - 1) {
        offsets[E] = ex_c + c;
        padded_offsets[E] = ex_p + p;
        meta[0] = ex_p + p;
        meta[1] = (ex_p + p) / kTileM;
    }
    __syncthreads();
    // per-(expert, unit) starting rows, tile map, pad rows
    for (int e = warp; e < E; e += 32) {
        int carry = s_pad[e];
        for (int u0 = 0; u0 < U; u0 += 32) {
            const int u = u0 + lane;
            const int v = u < U ? unit_base[(size_t)e * U + u] : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int a = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += a;
            }
            if (u < U) unit_base[(size_t)e * U + u] = carry + incl - v;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        const int cnt = s_cnt[e];
        const int pcnt = (cnt + kTileM - 1) / kTileM * kTileM;
        const int r0 = s_pad[e];
        for (int r = r0 + cnt + lane; r < r0 + pcnt; r += 32) route_of_row[r] = -1;
        for (int tl = r0 / kTileM + lane; tl < (r0 + pcnt) / kTileM; tl += 32) tile_expert[tl] = e;
    }
    pdl_launch_dependents();
}

// (3) scatter: one warp per unit walks its 32 tokens in order.
__global__ void __launch_bounds__(256) permute_scatter_kernel(int T, int E, int K, const int* __restrict__ topk_ids,
                                                              const int* __restrict__ unit_base,
                                                              int* __restrict__ row_of_route,
                                                              int* __restrict__ route_of_row) {
    extern __shared__ int s_next[];  // [8][E]
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int U = (T + kUnitTokens - 1) / kUnitTokens;
    const int u = blockIdx.x * 8 + warp;
    if (u >= U) return;
    int* nx = s_next + warp * E;
    for (int e = lane; e < E; e += 32) nx[e] = unit_base[(size_t)e * U + u];
    __syncwarp();
    const int t_end = min(T, (u + 1) * kUnitTokens);
    for (int t = u * kUnitTokens; t < t_end; ++t) {
        for (int k = lane; k < K; k += 32) {
            const int e = topk_ids[(size_t)t * K + k];
            if (e >= 0 && e < E) {
                const int row = nx[e];      // experts of one token are distinct
                nx[e] = row + 1;
                row_of_route[(size_t)t * K + k] = row;
                route_of_row[row] = t * K + k;
            }
        }
        __syncwarp();
    }
    pdl_launch_dependents();
}

cudaError_t launch_router(const LaunchCtx& c, int T, int E, int K, const float* logits, const float* bias,
                          int renorm, int* ids, float* w, unsigned int* st) {
    const int warps = 8;
    dim3 grid((T + warps - 1) / warps), block(32 * warps);
    const int epl = (E + 31) / 32;
    if (epl <= 1) return c.launch(router_topk_kernel<1>, grid, block, 0, T, E, K, logits, bias, renorm, ids, w, st);
    if (epl <= 2) return c.launch(router_topk_kernel<2>, grid, block, 0, T, E, K, logits, bias, renorm, ids, w, st);
    if (epl <= 4) return c.launch(router_topk_kernel<4>, grid, block, 0, T, E, K, logits, bias, renorm, ids, w, st);
    if (epl <= 8) return c.launch(router_topk_kernel<8>, grid, block, 0, T, E, K, logits, bias, renorm, ids, w, st);
    if (epl <= 16) return c.launch(router_topk_kernel<16>, grid, block, 0, T, E, K, logits, bias, renorm, ids, w, st);
    return c.launch(router_topk_kernel<32>, grid, block, 0, T, E, K, logits, bias, renorm, ids, w, st);
}

cudaError_t launch_permute(const LaunchCtx& c, int T, int E, int K, const int* ids, int* unit_base, int* count,
                           int* offsets, int* padded_offsets, int* meta, int* tile_expert, int* row_of_route,
                           int* route_of_row, unsigned int* status) {
    const int U = (T + kUnitTokens - 1) / kUnitTokens;
    const size_t smem = (size_t)8 * E * sizeof(int);
    cudaError_t err;
    err = c.launch(permute_count_kernel, dim3((U + 7) / 8), dim3(256), smem, T, E, K, ids, unit_base, status);
    if (err != cudaSuccess) return err;
    err = c.launch(permute_scan_kernel, dim3(1), dim3(1024), 0, T, E, unit_base, count, offsets, padded_offsets,
                   meta, tile_expert, route_of_row);
    if (err != cudaSuccess) return err;
    return c.launch(permute_scatter_kernel, dim3((U + 7) / 8), dim3(256), smem, T, E, K, ids,
                    (const int*)unit_base, row_of_route, route_of_row);
}

cudaError_t setup_routing_kernels() {
    const int smem = 8 * 1024 * (int)sizeof(int);
    cudaError_t e = cudaFuncSetAttribute(permute_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(permute_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

}  // namespace moe
