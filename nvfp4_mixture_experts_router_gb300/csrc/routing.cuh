// Device-side router of one token (shared by the router kernels and the
// fused layer kernel).
#pragma once
#include "common.cuh"

namespace moe {

// Selection key of expert e with router score v: the score's order-
// preserving bits above the complemented expert index, so that the larger
// key is the larger score and, among equal scores, the lower expert index
// (-0 is read as +0 so that equal values tie; a NaN score ranks below every
// number).  An absent expert (e >= E) has key 0, below every present one.
__device__ __forceinline__ uint64_t route_key(float v, int e) {
    v = __fadd_rn(v, 0.0f);                                  // -0 -> +0
    uint32_t u = __float_as_uint(v);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    if (v != v) u = 0u;
    return ((uint64_t)u << 32) | (uint64_t)(~(uint32_t)e);
}
__device__ __forceinline__ float route_key_value(uint64_t k) {
    const uint32_t u = (uint32_t)(k >> 32);
    return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}
__device__ __forceinline__ uint64_t max_u64(uint64_t a, uint64_t b) { return a > b ? a : b; }

// The same selection by rounds of a per-lane scan and a warp arg-max over
// (value, index) pairs: fewer registers than the keys below, used for more
// than 256 experts (16 or 32 scores a lane), where 64-bit keys would spill.
template <int EPL>
__device__ __forceinline__ int route_token_scan(int t, int E, int K, const float* __restrict__ logits,
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

// Selection by keys (up to 256 experts): expert e lives in lane e % 32,
// register e / 32.  K rounds: the warp's largest key (one 64-bit max
// reduction) is the next expert; the lane that held it drops it and
// recomputes its own largest.  The weights' softmax denominator adds the
// selected experts' terms in selection order.
template <int EPL>
__device__ __forceinline__ int route_token_keys(int t, int E, int K, const float* __restrict__ logits,
                                                const float* __restrict__ bias, int renorm,
                                                int* __restrict__ topk_ids, float* __restrict__ topk_w) {
    const int lane = threadIdx.x & 31;
    float l[EPL];
    uint64_t key[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E) {
            float v = __ldg(logits + (size_t)t * E + e);
            if (bias) v = __fadd_rn(v, __ldg(bias + e));
            l[i] = v;
            key[i] = route_key(v, e);
        } else {
            l[i] = -INFINITY;
            key[i] = 0;
        }
    }
    uint64_t best = key[0];
#pragma unroll
    for (int i = 1; i < EPL; ++i) best = max_u64(best, key[i]);
    float my_v = 0.0f, lmax = 0.0f;
    int my_e = -1;
    for (int k = 0; k < K; ++k) {
        uint64_t w = best;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) w = max_u64(w, __shfl_xor_sync(0xffffffffu, w, o));
        const int e = (int)(~(uint32_t)w);
        const float v = route_key_value(w);
        if (k == 0) lmax = v;
        if (k == lane) {
            my_v = v;
            my_e = e;
        }
        // the holder drops the key and recomputes its largest (every lane
        // runs the same selects, the others with nothing to drop)
        const int drop = (e & 31) == lane ? (e >> 5) : -1;
        uint64_t b = 0;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            key[i] = i == drop ? 0 : key[i];
            b = max_u64(b, key[i]);
        }
        best = b;
    }
    float den;
    if (renorm) {
        // sum in selection order, as the selected terms come
        const float term = lane < K ? expf(my_v - lmax) : 0.0f;
        den = 0.0f;
        for (int k = 0; k < K; ++k) den += __shfl_sync(0xffffffffu, term, k);
    } else {
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


// Route one token (the calling warp): writes ids / weights (lanes < K) and
// returns this lane's selected expert (slot = lane) or -1 for lane >= K.
template <int EPL>
__device__ __forceinline__ int route_token(int t, int E, int K, const float* __restrict__ logits,
                                           const float* __restrict__ bias, int renorm, int* __restrict__ topk_ids,
                                           float* __restrict__ topk_w) {
    if constexpr (EPL > 8)
        return route_token_scan<EPL>(t, E, K, logits, bias, renorm, topk_ids, topk_w);
    else
        return route_token_keys<EPL>(t, E, K, logits, bias, renorm, topk_ids, topk_w);
}

}  // namespace moe
