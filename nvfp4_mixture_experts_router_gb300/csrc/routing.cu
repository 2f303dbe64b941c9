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
// and partial tiles]: a stable counting sort over units of 32 tokens.
//   (1) per unit and expert, a 32-bit mask of the unit's tokens that chose
//       the expert (bit j = token u*32+j) and its population count;
//   (2) one block scans the counts into per-expert totals, offsets, 128-row
//       padded offsets and a per-(expert, unit) starting row;
//   (3) a route's row = its (expert, unit) start + popc(mask below its bit):
//       routes of an expert sit in ascending token order, which makes the
//       permutation unique.  Step (3) is a few integer operations per route,
//       so the forward folds it into the kernel that consumes the rows
//       (quantize_x / gather), see rowops.cu.
// The forward also folds (1) into the router kernel (route_count_kernel).
#include "common.cuh"
#include "kernels.h"
#include "routing.cuh"

namespace moe {


// Router only (the allocation-free routing entry point uses it).
template <int EPL>
__global__ void __launch_bounds__(256) router_topk_kernel(int T, int E, int K, const float* __restrict__ logits,
                                                          const float* __restrict__ bias, int renorm,
                                                          int* __restrict__ topk_ids, float* __restrict__ topk_w,
                                                          unsigned int* status_reset) {
    pdl_wait();
    // the first kernel of a forward clears the device status word
    if (status_reset && blockIdx.x == 0 && threadIdx.x == 0) *status_reset = 0u;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t < T) route_token<EPL>(t, E, K, logits, bias, renorm, topk_ids, topk_w);
    pdl_launch_dependents();
}

// Router fused with step (1): one block of 32 warps per unit of 32 tokens.
template <int EPL>
__global__ void __launch_bounds__(1024) route_count_kernel(int T, int E, int K, const float* __restrict__ logits,
                                                           const float* __restrict__ bias, int renorm,
                                                           int* __restrict__ topk_ids, float* __restrict__ topk_w,
                                                           int* __restrict__ unit_cnt, uint32_t* __restrict__ unit_mask,
                                                           unsigned int* status_reset) {
    __shared__ uint32_t s_mask[1024];
    pdl_wait();
    if (status_reset && blockIdx.x == 0 && threadIdx.x == 0) *status_reset = 0u;
    const int U = (T + kUnitTokens - 1) / kUnitTokens;
    const int u = blockIdx.x;
    const int w = threadIdx.x >> 5;
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_mask[e] = 0u;
    __syncthreads();
    const int t = u * kUnitTokens + w;
    if (t < T) {
        const int e = route_token<EPL>(t, E, K, logits, bias, renorm, topk_ids, topk_w);
        if (e >= 0) atomicOr(&s_mask[e], 1u << w);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const uint32_t m = s_mask[e];
        unit_cnt[(size_t)e * U + u] = __popc(m);
        unit_mask[(size_t)e * U + u] = m;
    }
    pdl_launch_dependents();
}

// Step (1) from given expert ids: warp w of the block handles unit blockIdx.x*8+w.
__global__ void __launch_bounds__(256) permute_count_kernel(int T, int E, int K, const int* __restrict__ topk_ids,
                                                            int* __restrict__ unit_cnt,
                                                            uint32_t* __restrict__ unit_mask, unsigned int* status) {
    extern __shared__ uint32_t s_masks[];  // [8][E]
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int U = (T + kUnitTokens - 1) / kUnitTokens;
    const int u = blockIdx.x * 8 + warp;
    uint32_t* m = s_masks + warp * E;
    for (int e = lane; e < E; e += 32) m[e] = 0u;
    __syncwarp();
    if (u < U) {
        const int t = u * kUnitTokens + lane;
        if (t < T) {
            for (int k = 0; k < K; ++k) {
                const int e = topk_ids[(size_t)t * K + k];
                if (e >= 0 && e < E) atomicOr(&m[e], 1u << lane);
                else atomicOr(status, kStatusBadExpert);
            }
        }
        __syncwarp();
        for (int e = lane; e < E; e += 32) {
            unit_cnt[(size_t)e * U + u] = __popc(m[e]);
            unit_mask[(size_t)e * U + u] = m[e];
        }
    }
    pdl_launch_dependents();
}

// Caller-supplied routing [FlashInfer PR #4366, "Motivation": precomputed
// top-K ids and weights] in place of the router, fused with step (1): warp w
// of the block handles unit blockIdx.x*8+w, one lane per token.  Copies the
// ids and weights into the workspace; an id outside [0, E) or repeating an
// earlier kept id of the same token becomes -1 (a dropped route: no row, no
// contribution) and sets kStatusBadExpert.  A repeat shows up as this
// token's bit already set in the expert's unit mask.
__global__ void __launch_bounds__(256) route_given_kernel(int T, int E, int K, const int* __restrict__ ids_in,
                                                          const float* __restrict__ w_in, int* __restrict__ topk_ids,
                                                          float* __restrict__ topk_w, int* __restrict__ unit_cnt,
                                                          uint32_t* __restrict__ unit_mask, unsigned int* status) {
    extern __shared__ uint32_t s_masks[];  // [8][E]
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int U = (T + kUnitTokens - 1) / kUnitTokens;
    const int u = blockIdx.x * 8 + warp;
    uint32_t* m = s_masks + warp * E;
    for (int e = lane; e < E; e += 32) m[e] = 0u;
    __syncwarp();
    if (u < U) {
        const int t = u * kUnitTokens + lane;
        if (t < T) {
            bool bad = false;
            for (int k = 0; k < K; ++k) {
                const size_t r = (size_t)t * K + k;
                int e = ids_in[r];
                if (e >= 0 && e < E) {
                    // only this lane sets this bit, so the old value tells
                    // whether an earlier slot of the token took expert e
                    if (atomicOr(&m[e], 1u << lane) & (1u << lane)) e = -1;
                } else {
                    e = -1;
                }
                bad |= e < 0;
                topk_ids[r] = e;
                topk_w[r] = w_in[r];
            }
            if (bad) atomicOr(status, kStatusBadExpert);
        }
        __syncwarp();
        for (int e = lane; e < E; e += 32) {
            unit_cnt[(size_t)e * U + u] = __popc(m[e]);
            unit_mask[(size_t)e * U + u] = m[e];
        }
    }
    pdl_launch_dependents();
}

// Outputs of the permutation scan (step 2).  tile_pair / tile_half may be
// null (then only meta[2] / meta[3] count them).
struct ScanOut {
    int* count;
    int* offsets;
    int* padded_offsets;
    int* meta;
    int* tile_expert;
    int* tile_pair;
    int* tile_half;
    int* route_of_row;
};

// By a block of 1024 threads, given the per-expert route counts s_cnt[E]:
// exclusive scans over experts of the count, the 128-padded count, the
// number of M-tile pairs (ceil(tiles / 2)) and the number of 64-row halves
// holding routes (ceil(count / 64)); publishes count / offsets /
// padded_offsets / meta and leaves the padded offsets, pair and half
// offsets in shared memory (ends with a block barrier).
__device__ __forceinline__ void scan_experts_block(int E, const int* s_cnt, int* s_pad, int* s_pair, int* s_half,
                                                   int (*s_warp)[32], const ScanOut& o) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = tid < E ? s_cnt[tid] : 0;
    const int p = tid < E ? (c + kTileM - 1) / kTileM * kTileM : 0;
    const int q = (p / kTileM + 1) / 2;
    const int hv = (c + kTileM / 2 - 1) / (kTileM / 2);
    int ic = c, ip = p, iq = q, ih = hv;
#pragma unroll
    for (int k = 1; k < 32; k <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, ic, k);
        const int b = __shfl_up_sync(0xffffffffu, ip, k);
        const int d = __shfl_up_sync(0xffffffffu, iq, k);
        const int f = __shfl_up_sync(0xffffffffu, ih, k);
        if (lane >= k) { ic += a; ip += b; iq += d; ih += f; }
    }
    if (lane == 31) { s_warp[0][warp] = ic; s_warp[1][warp] = ip; s_warp[2][warp] = iq; s_warp[3][warp] = ih; }
    __syncthreads();
    if (warp == 0) {
        int a = s_warp[0][lane], b = s_warp[1][lane], d = s_warp[2][lane], f = s_warp[3][lane];
#pragma unroll
        for (int k = 1; k < 32; k <<= 1) {
            const int x = __shfl_up_sync(0xffffffffu, a, k);
            const int y = __shfl_up_sync(0xffffffffu, b, k);
            const int z = __shfl_up_sync(0xffffffffu, d, k);
            const int w = __shfl_up_sync(0xffffffffu, f, k);
            if (lane >= k) { a += x; b += y; d += z; f += w; }
        }
        s_warp[0][lane] = a;
        s_warp[1][lane] = b;
        s_warp[2][lane] = d;
        s_warp[3][lane] = f;
    }
    __syncthreads();
    const int base_c = warp > 0 ? s_warp[0][warp - 1] : 0;
    const int base_p = warp > 0 ? s_warp[1][warp - 1] : 0;
    const int base_q = warp > 0 ? s_warp[2][warp - 1] : 0;
    const int base_h = warp > 0 ? s_warp[3][warp - 1] : 0;
    const int ex_c = base_c + ic - c, ex_p = base_p + ip - p, ex_q = base_q + iq - q, ex_h = base_h + ih - hv;
    if (tid < E) {
        o.count[tid] = c;
        o.offsets[tid] = ex_c;
        o.padded_offsets[tid] = ex_p;
        s_pad[tid] = ex_p;
        s_pair[tid] = ex_q;
        s_half[tid] = ex_h;
    }
    if (tid == E - 1) {
        o.offsets[E] = ex_c + c;
        o.padded_offsets[E] = ex_p + p;
        o.meta[0] = ex_p + p;
        o.meta[1] = (ex_p + p) / kTileM;
        o.meta[2] = ex_q + q;
        o.meta[3] = ex_h + hv;
    }
    __syncthreads();
}

// Per-expert outputs of the scan, a warp per expert: -1 in the pad rows of
// its segment, the M-tile -> expert map, its M-tile pairs and its occupied
// 64-row halves.
__device__ __forceinline__ void expert_outputs_block(int E, const int* s_cnt, const int* s_pad, const int* s_pair,
                                                     const int* s_half, const ScanOut& o) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    for (int e = warp; e < E; e += nwarps) {
        const int cnt = s_cnt[e];
        const int pcnt = (cnt + kTileM - 1) / kTileM * kTileM;
        const int r0 = s_pad[e];
        for (int r = r0 + cnt + lane; r < r0 + pcnt; r += 32) o.route_of_row[r] = -1;
        for (int tl = r0 / kTileM + lane; tl < (r0 + pcnt) / kTileM; tl += 32) o.tile_expert[tl] = e;
        if (o.tile_pair != nullptr) {
            // pairs of consecutive M tiles of this expert; an odd count leaves
            // the last tile alone
            const int nt = pcnt / kTileM;
            for (int i = lane; 2 * i < nt; i += 32)
                o.tile_pair[s_pair[e] + i] = ((r0 / kTileM + 2 * i) << 1) | (2 * i + 1 < nt ? 1 : 0);
        }
        if (o.tile_half != nullptr) {
            // the 64-row halves of this expert's M tiles that hold routes, in order
            const int nh = (cnt + kTileM / 2 - 1) / (kTileM / 2);
            for (int j = lane; j < nh; j += 32) o.tile_half[s_half[e] + j] = ((r0 / kTileM + (j >> 1)) << 1) | (j & 1);
        }
    }
}

// (2) one block of 1024 threads: totals, offsets, padded offsets, per-unit
// starting rows (in place of the counts), M-tile -> expert map, pad rows of
// route_of_row set to -1.
__global__ void __launch_bounds__(1024) permute_scan_kernel(int T, int E, int* __restrict__ unit_base /* [E][U] */,
                                                            const ScanOut o) {
    __shared__ int s_cnt[1024];
    __shared__ int s_pad[1024];
    __shared__ int s_pair[1024];
    __shared__ int s_half[1024];
    __shared__ int s_warp[4][32];
    pdl_wait();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int U = (T + kUnitTokens - 1) / kUnitTokens;
    // totals per expert.  Up to kSmallU units (T <= 512): a thread per
    // expert holds its unit counts in registers (independent loads) and
    // later writes the unit starting rows from them; a warp per expert
    // would chain E/32 dependent round trips per warp, twice.
    constexpr int kSmallU = 16;
    const bool small = U <= kSmallU;
    // rows of a whole number of int4 (every row 16-byte aligned: the region
    // is): each lane takes four consecutive units per access, a quarter of
    // the instructions of a unit a lane
    const bool vec = (U & 3) == 0;
    int ucnt[kSmallU];
    if (small) {
        if (tid < E) {
            int sum = 0;
#pragma unroll
            for (int u = 0; u < kSmallU; ++u) {
                ucnt[u] = u < U ? unit_base[(size_t)tid * U + u] : 0;
                sum += ucnt[u];
            }
            s_cnt[tid] = sum;
        }
    } else {
        for (int e = warp; e < E; e += 32) {
            int s = 0;
            if (vec) {
                const int4* row4 = reinterpret_cast<const int4*>(unit_base + (size_t)e * U);
#pragma unroll 4
                for (int i = lane; i < U / 4; i += 32) {
                    const int4 v = row4[i];
                    s += v.x + v.y + v.z + v.w;
                }
            } else {
                for (int u = lane; u < U; u += 32) s += unit_base[(size_t)e * U + u];
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (lane == 0) s_cnt[e] = s;
        }
    }
    __syncthreads();
    scan_experts_block(E, s_cnt, s_pad, s_pair, s_half, s_warp, o);
    // per-(expert, unit) starting rows
    if (small && tid < E) {
        int run = s_pad[tid];
#pragma unroll
        for (int u = 0; u < kSmallU; ++u) {
            if (u < U) unit_base[(size_t)tid * U + u] = run;
            run += ucnt[u];
        }
    }
    for (int e = warp; !small && vec && e < E; e += 32) {
        int carry = s_pad[e];
        int4* row4 = reinterpret_cast<int4*>(unit_base + (size_t)e * U);
        const int n4 = U / 4;
#pragma unroll 2
        for (int i0 = 0; i0 < n4; i0 += 32) {
            const int i = i0 + lane;
            const int4 v = i < n4 ? row4[i] : make_int4(0, 0, 0, 0);
            const int sum = v.x + v.y + v.z + v.w;
            int incl = sum;
#pragma unroll
            for (int o2 = 1; o2 < 32; o2 <<= 1) {
                const int a = __shfl_up_sync(0xffffffffu, incl, o2);
                if (lane >= o2) incl += a;
            }
            const int b = carry + incl - sum;
            if (i < n4) row4[i] = make_int4(b, b + v.x, b + v.x + v.y, b + v.x + v.y + v.z);
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
    }
    for (int e = warp; !small && !vec && e < E; e += 32) {
        int carry = s_pad[e];
        for (int u0 = 0; u0 < U; u0 += 32) {
            const int u = u0 + lane;
            const int v = u < U ? unit_base[(size_t)e * U + u] : 0;
            int incl = v;
#pragma unroll
            for (int o2 = 1; o2 < 32; o2 <<= 1) {
                const int a = __shfl_up_sync(0xffffffffu, incl, o2);
                if (lane >= o2) incl += a;
            }
            if (u < U) unit_base[(size_t)e * U + u] = carry + incl - v;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
    }
    expert_outputs_block(E, s_cnt, s_pad, s_pair, s_half, o);
    pdl_launch_dependents();
}

// Steps (1) and (2) in one block for T <= 32 (a single unit of tokens):
// the router (a warp per token), the expert token masks in shared memory,
// their counts and the scan, without the masks' round trip through memory
// and the second launch.  Same outputs as route_count_kernel followed by
// permute_scan_kernel.
template <int EPL>
__global__ void __launch_bounds__(1024) route_scan_small_kernel(int T, int E, int K, const float* __restrict__ logits,
                                                                const float* __restrict__ bias, int renorm,
                                                                int* __restrict__ topk_ids, float* __restrict__ topk_w,
                                                                int* __restrict__ unit_base, uint32_t* __restrict__ unit_mask,
                                                                const ScanOut o, unsigned int* status_reset) {
    __shared__ uint32_t s_mask[1024];
    __shared__ int s_cnt[1024];
    __shared__ int s_pad[1024];
    __shared__ int s_pair[1024];
    __shared__ int s_half[1024];
    __shared__ int s_warp[4][32];
    pdl_wait();
    if (status_reset && threadIdx.x == 0) *status_reset = 0u;
    const int tid = threadIdx.x, warp = tid >> 5;
    for (int e = tid; e < E; e += blockDim.x) s_mask[e] = 0u;
    __syncthreads();
    if (warp < T) {
        const int e = route_token<EPL>(warp, E, K, logits, bias, renorm, topk_ids, topk_w);
        if (e >= 0) atomicOr(&s_mask[e], 1u << warp);
    }
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) {
        const uint32_t m = s_mask[e];
        unit_mask[e] = m;            // [E][1]
        s_cnt[e] = __popc(m);
    }
    __syncthreads();
    scan_experts_block(E, s_cnt, s_pad, s_pair, s_half, s_warp, o);
    for (int e = tid; e < E; e += blockDim.x) unit_base[e] = s_pad[e];   // one unit: its start is the segment's
    expert_outputs_block(E, s_cnt, s_pad, s_pair, s_half, o);
    pdl_launch_dependents();
}

// (3) standalone: one thread per route.
__global__ void __launch_bounds__(256) permute_scatter_kernel(int T, int E, int K, const int* __restrict__ topk_ids,
                                                              const int* __restrict__ unit_base,
                                                              const uint32_t* __restrict__ unit_mask,
                                                              int* __restrict__ row_of_route,
                                                              int* __restrict__ route_of_row) {
    pdl_wait();
    const int U = (T + kUnitTokens - 1) / kUnitTokens;
    const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (r < (int64_t)T * K) {
        const int e = topk_ids[r];
        if (e >= 0 && e < E) {
            const int row = route_row((int)(r / K), e, U, unit_base, unit_mask);
            row_of_route[r] = row;
            route_of_row[row] = (int)r;
        }
    }
    pdl_launch_dependents();
}

#define MOE_EPL_DISPATCH(E, KERNEL, ...)                                  \
    do {                                                                  \
        const int epl_ = ((E) + 31) / 32;                                 \
        if (epl_ <= 1) return c.launch(KERNEL<1>, __VA_ARGS__);           \
        if (epl_ <= 2) return c.launch(KERNEL<2>, __VA_ARGS__);           \
        if (epl_ <= 4) return c.launch(KERNEL<4>, __VA_ARGS__);           \
        if (epl_ <= 8) return c.launch(KERNEL<8>, __VA_ARGS__);           \
        if (epl_ <= 16) return c.launch(KERNEL<16>, __VA_ARGS__);         \
        return c.launch(KERNEL<32>, __VA_ARGS__);                         \
    } while (0)

cudaError_t launch_router(const LaunchCtx& c, int T, int E, int K, const float* logits, const float* bias,
                          int renorm, int* ids, float* w, unsigned int* st) {
    const dim3 grid((T + 7) / 8), block(256);
    MOE_EPL_DISPATCH(E, router_topk_kernel, grid, block, 0, T, E, K, logits, bias, renorm, ids, w, st);
}

cudaError_t launch_route_count(const LaunchCtx& c, int T, int E, int K, const float* logits, const float* bias,
                               int renorm, int* ids, float* w, int* unit_cnt, uint32_t* unit_mask,
                               unsigned int* st) {
    const int U = (T + kUnitTokens - 1) / kUnitTokens;
    MOE_EPL_DISPATCH(E, route_count_kernel, dim3(U), dim3(1024), 0, T, E, K, logits, bias, renorm, ids, w, unit_cnt,
                     unit_mask, st);
}

cudaError_t launch_permute_scan(const LaunchCtx& c, int T, int E, int* unit_base, int* count, int* offsets,
                                int* padded_offsets, int* meta, int* tile_expert, int* tile_pair, int* tile_half,
                                int* route_of_row) {
    const ScanOut o{count, offsets, padded_offsets, meta, tile_expert, tile_pair, tile_half, route_of_row};
    return c.launch(permute_scan_kernel, dim3(1), dim3(1024), 0, T, E, unit_base, o);
}

cudaError_t launch_route_scan_small(const LaunchCtx& c, int T, int E, int K, const float* logits, const float* bias,
                                    int renorm, int* ids, float* w, int* unit_base, uint32_t* unit_mask, int* count,
                                    int* offsets, int* padded_offsets, int* meta, int* tile_expert, int* tile_pair,
                                    int* tile_half, int* route_of_row, unsigned int* status_reset) {
    if (T > kUnitTokens) return cudaErrorInvalidValue;
    const ScanOut o{count, offsets, padded_offsets, meta, tile_expert, tile_pair, tile_half, route_of_row};
    MOE_EPL_DISPATCH(E, route_scan_small_kernel, dim3(1), dim3(1024), 0, T, E, K, logits, bias, renorm, ids, w,
                     unit_base, unit_mask, o, status_reset);
}

cudaError_t launch_permute(const LaunchCtx& c, int T, int E, int K, const int* ids, int* unit_base,
                           uint32_t* unit_mask, int* count, int* offsets, int* padded_offsets, int* meta,
                           int* tile_expert, int* row_of_route, int* route_of_row, unsigned int* status) {
    const int U = (T + kUnitTokens - 1) / kUnitTokens;
    const size_t smem = (size_t)8 * E * sizeof(uint32_t);
    cudaError_t err;
    err = c.launch(permute_count_kernel, dim3((U + 7) / 8), dim3(256), smem, T, E, K, ids, unit_base, unit_mask,
                   status);
    if (err != cudaSuccess) return err;
    err = launch_permute_scan(c, T, E, unit_base, count, offsets, padded_offsets, meta, tile_expert, nullptr, nullptr,
                              route_of_row);
    if (err != cudaSuccess) return err;
    const int64_t routes = (int64_t)T * K;
    return c.launch(permute_scatter_kernel, dim3((unsigned)((routes + 255) / 256)), dim3(256), 0, T, E, K, ids,
                    (const int*)unit_base, (const uint32_t*)unit_mask, row_of_route, route_of_row);
}

cudaError_t launch_route_given(const LaunchCtx& c, int T, int E, int K, const int* ids_in, const float* w_in,
                               int* ids, float* w, int* unit_cnt, uint32_t* unit_mask, unsigned int* status) {
    const int U = (T + kUnitTokens - 1) / kUnitTokens;
    const size_t smem = (size_t)8 * E * sizeof(uint32_t);
    return c.launch(route_given_kernel, dim3((U + 7) / 8), dim3(256), smem, T, E, K, ids_in, w_in, ids, w, unit_cnt,
                    unit_mask, status);
}

cudaError_t setup_routing_kernels() {
    const int smem = 8 * 1024 * (int)sizeof(uint32_t);
    const cudaError_t e = cudaFuncSetAttribute(permute_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(route_given_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

}  // namespace moe
