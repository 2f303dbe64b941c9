// Device-side router of one token (shared by the router kernels and the
// fused layer kernel).
#pragma once
#include "common.cuh"

namespace moe {

// Route one token (the calling warp): writes ids / weights (lanes < K) and
// returns this lane's selected expert (slot = lane) or -1 for lane >= K.
template <int EPL>
__device__ __forceinline__ int route_token(int t, int E, int K, const float* __restrict__ logits,
                                           const float* __restrict__ bias, int renorm, int* __restrict__ topk_ids,
                                           float* __restrict__ topk_w) {
    const int lane = threadIdx.x & 31;
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
    float my_v = 0.0f, lmax = 0.0f, den = 0.0f;
    int my_e = -1;
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
        if (k == 0) lmax = bv;
        if (renorm) den += expf(bv - lmax);      // same order on every lane
        if (k == lane) {
            my_v = bv;
            my_e = be;
        }
    }
    if (!renorm) {
        float part = 0.0f;
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if (lane + 32 * i < E) part += expf(l[i] - lmax);
        den = warp_sum(part);
    }
    if (lane < K) {
        topk_ids[(size_t)t * K + lane] = my_e;
        topk_w[(size_t)t * K + lane] = expf(my_v - lmax) / den;
    }
    return lane < K ? my_e : -1;
}


}  // namespace moe
