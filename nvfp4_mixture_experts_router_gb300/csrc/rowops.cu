// Row-parallel kernels around the grouped GEMMs: NVFP4 quantization of x
// (scattered straight into the permuted rows), per-row quantization of the
// FC2 input (per-token mode), the W4A16 gather, both finalize variants and
// weight preparation.  All of them are HBM-bound: one warp per row, 16-byte
// vector loads and stores, lanes on consecutive 16-element blocks.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

__device__ __forceinline__ void load16_bf16(const __nv_bfloat16* p, float (&v)[16]) {
    const uint4 a = *reinterpret_cast<const uint4*>(p);
    const uint4 b = *reinterpret_cast<const uint4*>(p + 8);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ void load16_f32(const float* p, float (&v)[16]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 q = reinterpret_cast<const float4*>(p)[i];
        v[4 * i] = q.x; v[4 * i + 1] = q.y; v[4 * i + 2] = q.z; v[4 * i + 3] = q.w;
    }
}

// Four consecutive lanes hold the scales of four consecutive blocks; the
// first of them gets the packed 32-bit word (byte j%4 = scale of block j).
__device__ __forceinline__ uint32_t pack_sf4(uint32_t s) {
    const uint32_t s1 = __shfl_down_sync(0xffffffffu, s, 1);
    const uint32_t s2 = __shfl_down_sync(0xffffffffu, s, 2);
    const uint32_t s3 = __shfl_down_sync(0xffffffffu, s, 3);
    return s | (s1 << 8) | (s2 << 16) | (s3 << 24);
}

// Step 3 of the permutation for token t, lane k < K handling route t*K+k:
// compute the route's padded row, record both directions of the map, and
// return the row (0 for lanes >= K).
// Returns the route's padded row, or -1 for lanes >= K and dropped routes.
__device__ __forceinline__ int scatter_token_routes(int t, int T, int K, int lane, const RouteScatter& rs) {
    if (lane >= K) return -1;
    const int U = (T + kUnitTokens - 1) / kUnitTokens;
    const int r = t * K + lane;
    const int e = rs.topk_ids[r];
    if (e < 0 || e >= rs.E) {
        rs.row_of_route[r] = -1;
        return -1;
    }
    const int row = route_row(t, e, U, rs.unit_base, rs.unit_mask);
    rs.row_of_route[r] = row;
    rs.route_of_row[row] = r;
    return row;
}

__device__ __forceinline__ void zero_row_f32(float* p, int n, int lane) {
    for (int c = lane * 4; c < n; c += 128) *reinterpret_cast<float4*>(p + c) = make_float4(0.f, 0.f, 0.f, 0.f);
}

}  // namespace

// x [T][H] BF16 -> NVFP4 codes/scales written to each of the token's K
// permuted rows.  One CTA per token, one thread per 16-element block (a
// single read of the row; per-token mode reduces the row amax in the CTA and
// derives G1 = amax/2688).  Also hands out the token's permuted rows (step 3
// of the permutation) and zeroes its row of the fused-finalize accumulator.
// kMaxPer: 16-element blocks per thread (rows up to kMaxPer * 16K elements);
// kFourSix: 4-over-6 blocks (a compile-time choice, so that the default
// kernels carry none of its code)
template <int kMaxPer, bool kFourSix>
__global__ void __launch_bounds__(1024) quantize_x_kernel(int T, int H, int K, const __nv_bfloat16* __restrict__ x,
                                                          const float* __restrict__ g1_in, int per_token,
                                                          float* __restrict__ g1_out, const RouteScatter rs,
                                                          uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                                                          float* __restrict__ y_acc_zero) {
    __shared__ float s_red[32];
    __shared__ int s_rows[32];
    pdl_wait();
    const int t = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nblk = H / 16;
    if (warp == 0) {
        const int row = scatter_token_routes(t, T, K, lane, rs);
        if (lane < K) s_rows[lane] = row;
    }
    const __nv_bfloat16* xr = x + (size_t)t * H;
    float v[kMaxPer][16];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < kMaxPer; ++i) {
        const int b = tid + i * blockDim.x;
        if (b < nblk) {
            load16_bf16(xr + 16 * b, v[i]);
#pragma unroll
            for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[i][j]));
        }
    }
    float G;
    if (per_token) {
        amax = warp_max(amax);
        if (lane == 0) s_red[warp] = amax;
        __syncthreads();
        if (warp == 0) {
            float m = lane < (int)(blockDim.x >> 5) ? s_red[lane] : 0.0f;
            m = warp_max(m);
            if (lane == 0) s_red[0] = kFourSix ? global_scale_from_amax_4over6(m) : global_scale_from_amax(m);
        }
        __syncthreads();
        G = s_red[0];
        if (tid == 0) g1_out[t] = G;
    } else {
        G = __ldg(g1_in);
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < kMaxPer; ++i) {
        const int b0 = i * blockDim.x;              // uniform across the warp
        if (b0 >= nblk) break;
        const int b = tid + b0;
        const bool active = b < nblk;
        uint32_t q[2] = {0u, 0u};
        uint32_t s = 0;
        if (active) s = kFourSix ? quant_block16_4over6(v[i], G, q) : quant_block16(v[i], G, q);
        const uint32_t word = pack_sf4(s);
        if (active) {
            for (int k = 0; k < K; ++k) {
                const int row = s_rows[k];
                if (row < 0) continue;
                *reinterpret_cast<uint2*>(codes + (size_t)row * (H / 2) + 8 * b) = make_uint2(q[0], q[1]);
                if ((lane & 3) == 0) *reinterpret_cast<uint32_t*>(sf + sf_offset(row, b, H)) = word;
            }
        }
    }
    if (y_acc_zero) {
        float* yr = y_acc_zero + (size_t)t * H;
        for (int c = tid * 4; c < H; c += blockDim.x * 4) *reinterpret_cast<float4*>(yr + c) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    pdl_launch_dependents();
}

// MXFP8: x [T][H] BF16 -> E4M3 codes (a byte each) and E8M0 scales per 32
// elements, written to each of the token's K permuted rows.  One CTA per
// token, one thread per 32-element block (blocks are independent: no row
// reduction); hands out the permuted rows and zeroes the token's row of the
// fused-finalize accumulator like quantize_x_kernel.
__global__ void __launch_bounds__(1024) quantize_x_mx_kernel(int T, int H, int K, const __nv_bfloat16* __restrict__ x,
                                                             const RouteScatter rs, uint8_t* __restrict__ codes,
                                                             uint8_t* __restrict__ sf, float* __restrict__ y_acc_zero) {
    __shared__ int s_rows[32];
    pdl_wait();
    const int t = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (warp == 0) {
        const int row = scatter_token_routes(t, T, K, lane, rs);
        if (lane < K) s_rows[lane] = row;
    }
    __syncthreads();
    const int nblk = H / 32;
    const __nv_bfloat16* xr = x + (size_t)t * H;
    for (int b0 = 0; b0 < nblk; b0 += blockDim.x) {      // uniform across the CTA
        const int b = b0 + tid;
        const bool active = b < nblk;
        uint32_t q[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        uint32_t s = 0;
        if (active) {
            float v[32];
            float h16[16];
            load16_bf16(xr + 32 * b, h16);
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = h16[i];
            load16_bf16(xr + 32 * b + 16, h16);
#pragma unroll
            for (int i = 0; i < 16; ++i) v[16 + i] = h16[i];
            s = quant_block32_mx(v, q);
        }
        const uint32_t word = pack_sf4(s);
        if (active) {
            for (int k = 0; k < K; ++k) {
                const int row = s_rows[k];
                if (row < 0) continue;
                uint4* dst = reinterpret_cast<uint4*>(codes + (size_t)row * H + 32 * b);
                dst[0] = make_uint4(q[0], q[1], q[2], q[3]);
                dst[1] = make_uint4(q[4], q[5], q[6], q[7]);
                if ((lane & 3) == 0) *reinterpret_cast<uint32_t*>(sf + sf_offset_mx(row, b, H)) = word;
            }
        }
    }
    if (y_acc_zero) {
        float* yr = y_acc_zero + (size_t)t * H;
        for (int c = tid * 4; c < H; c += blockDim.x * 4)
            *reinterpret_cast<float4*>(yr + c) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    pdl_launch_dependents();
}

// W4A16: copy each token's BF16 row to its K permuted rows.
__global__ void __launch_bounds__(256) gather_x_bf16_kernel(int T, int H, int K, const __nv_bfloat16* __restrict__ x,
                                                            const RouteScatter rs,
                                                            __nv_bfloat16* __restrict__ x_perm,
                                                            float* __restrict__ y_acc_zero) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    const int my_row = scatter_token_routes(t, T, K, lane, rs);
    for (int base = 0; base < H / 8; base += 32) {
        const int c = base + lane;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (c < H / 8) v = src[c];
        for (int k = 0; k < K; ++k) {
            const int row = __shfl_sync(0xffffffffu, my_row, k);
            if (c < H / 8 && row >= 0) reinterpret_cast<uint4*>(x_perm + (size_t)row * H)[c] = v;
        }
    }
    if (y_acc_zero) zero_row_f32(y_acc_zero + (size_t)t * H, H, lane);
    pdl_launch_dependents();
}

// Per-token W4A4: FC2 input row (FP32) -> G2 = amax/2688, NVFP4 codes/scales.
// One CTA per row at a time (grid-stride over the padded rows, pad rows
// skipped), one thread per 16-element block.
template <int kMaxPer, bool kFourSix>
__global__ void __launch_bounds__(1024) quantize_h_kernel(int I, const int* __restrict__ meta,
                                                          const int* __restrict__ route_of_row,
                                                          const float* __restrict__ h, float* __restrict__ g2,
                                                          uint8_t* __restrict__ codes, uint8_t* __restrict__ sf) {
    __shared__ float s_red[32];
    pdl_wait();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rows = meta[0];
    for (int row = blockIdx.x; row < rows; row += gridDim.x) {
    if (route_of_row[row] < 0) continue;      // pad row (uniform across the CTA)
    const int nblk = I / 16;
    const float* hr = h + (size_t)row * I;
    float v[kMaxPer][16];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < kMaxPer; ++i) {
        const int b = tid + i * blockDim.x;
        if (b < nblk) {
            load16_f32(hr + 16 * b, v[i]);
#pragma unroll
            for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[i][j]));
        }
    }
    amax = warp_max(amax);
    if (lane == 0) s_red[warp] = amax;
    __syncthreads();
    if (warp == 0) {
        float m = lane < (int)(blockDim.x >> 5) ? s_red[lane] : 0.0f;
        m = warp_max(m);
        if (lane == 0) s_red[0] = kFourSix ? global_scale_from_amax_4over6(m) : global_scale_from_amax(m);
    }
    __syncthreads();
    const float G = s_red[0];
    __syncthreads();                         // s_red is reused by the next row
    if (tid == 0) g2[row] = G;
#pragma unroll
    for (int i = 0; i < kMaxPer; ++i) {
        const int b0 = i * blockDim.x;
        if (b0 >= nblk) break;
        const int b = tid + b0;
        const bool active = b < nblk;
        uint32_t q[2] = {0u, 0u};
        uint32_t s = 0;
        if (active) s = kFourSix ? quant_block16_4over6(v[i], G, q) : quant_block16(v[i], G, q);
        const uint32_t word = pack_sf4(s);
        if (active) {
            *reinterpret_cast<uint2*>(codes + (size_t)row * (I / 2) + 8 * b) = make_uint2(q[0], q[1]);
            if ((lane & 3) == 0) *reinterpret_cast<uint32_t*>(sf + sf_offset(row, b, I)) = word;
        }
    }
    }
    pdl_launch_dependents();
}

// Deterministic finalize: y[t] = BF16( sum_k w'_k * o[row(t,k)] ), k in
// ascending order, FP32 accumulation; w' = router weight (output side) or 1.
// One thread per 8 output elements of a token (the whole grid shares the
// T x H/8 groups, so a few tokens still spread over many SMs); the K rows
// are loaded four at a time to keep loads in flight.
__global__ void __launch_bounds__(256) finalize_det_kernel(int T, int H, int K, const int* __restrict__ row_of_route,
                                                           const float* __restrict__ topk_w, int weight_on_output,
                                                           const __nv_bfloat16* __restrict__ o,
                                                           __nv_bfloat16* __restrict__ y) {
    pdl_wait();
    const int H8 = H / 8;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < (int64_t)T * H8) {
        const int t = (int)(i / H8), c = (int)(i % H8);
        float acc[8];
        finalize_det_group(t, c, H, K, row_of_route, topk_w, weight_on_output, o, acc);
        reinterpret_cast<uint4*>(y)[i] = pack_bf16x8(acc);
    }
    pdl_launch_dependents();
}

// Fused finalize tail: the FC2 epilogue accumulated y in FP32; round to BF16.
__global__ void __launch_bounds__(256) finalize_fused_kernel(int64_t n8, const float* __restrict__ y_acc,
                                                             __nv_bfloat16* __restrict__ y) {
    pdl_wait();
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
        const float4 a = reinterpret_cast<const float4*>(y_acc)[2 * i];
        const float4 b = reinterpret_cast<const float4*>(y_acc)[2 * i + 1];
        const __nv_bfloat162 p0 = __floats2bfloat162_rn(a.x, a.y), p1 = __floats2bfloat162_rn(a.z, a.w);
        const __nv_bfloat162 p2 = __floats2bfloat162_rn(b.x, b.y), p3 = __floats2bfloat162_rn(b.z, b.w);
        reinterpret_cast<uint4*>(y)[i] =
            make_uint4(*reinterpret_cast<const uint32_t*>(&p0), *reinterpret_cast<const uint32_t*>(&p1),
                       *reinterpret_cast<const uint32_t*>(&p2), *reinterpret_cast<const uint32_t*>(&p3));
    }
    pdl_launch_dependents();
}

// ---------------------------------------------------------------------------
// weight preparation
// ---------------------------------------------------------------------------
__global__ void prep_zero_kernel(uint32_t* amax_bits, int n) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) amax_bits[i] = 0u;
}

// blockIdx.y = expert, blockIdx.z = matrix (0: W1, 1: W2); grid-stride chunks.
__global__ void __launch_bounds__(256) prep_amax_kernel(int E, int64_t n1, int64_t n2,
                                                        const __nv_bfloat16* __restrict__ w1,
                                                        const __nv_bfloat16* __restrict__ w2,
                                                        uint32_t* __restrict__ amax_bits) {
    const int e = blockIdx.y, which = blockIdx.z;
    const int64_t n = which ? n2 : n1;
    const __nv_bfloat16* w = which ? w2 + (size_t)e * n2 : w1 + (size_t)e * n1;
    float m = 0.0f;
    for (int64_t i = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) * 8; i < n; i += (int64_t)gridDim.x * blockDim.x * 8) {
        const uint4 v = *reinterpret_cast<const uint4*>(w + i);
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
            m = fmaxf(m, fmaxf(fabsf(__uint_as_float(u[k] << 16)), fabsf(__uint_as_float(u[k] & 0xFFFF0000u))));
    }
    m = warp_max(m);
    __shared__ float s_m[8];
    if ((threadIdx.x & 31) == 0) s_m[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float b = 0.0f;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) b = fmaxf(b, s_m[i]);
        atomicMax(amax_bits + which * E + e, __float_as_uint(b));   // non-negative: uint order = float order
    }
}

__global__ void prep_scales_kernel(int E, const uint32_t* __restrict__ amax_bits, float* __restrict__ gw1,
                                   float* __restrict__ gw2) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < 2 * E) {
        const float G = global_scale_from_amax(__uint_as_float(amax_bits[i]));
        if (i < E) gw1[i] = G;
        else gw2[i - E] = G;
    }
}

// MXFP8 weights: one warp per weight row (W1 rows first, then W2 rows), one
// lane per 32-element block; Gw1 = Gw2 = 1 (no global scales).
__global__ void __launch_bounds__(256) prep_quant_mx_kernel(int E, int N1, int H, int I, int act,
                                                            const __nv_bfloat16* __restrict__ w1,
                                                            const __nv_bfloat16* __restrict__ w2,
                                                            float* __restrict__ gw1, float* __restrict__ gw2,
                                                            uint8_t* __restrict__ w1c, uint8_t* __restrict__ w1s,
                                                            uint8_t* __restrict__ w2c, uint8_t* __restrict__ w2s) {
    const int lane = threadIdx.x & 31;
    const int64_t gr = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (gr < 2 * (int64_t)E && lane == 0) {
        if (gr < E) gw1[gr] = 1.0f;
        else gw2[gr - E] = 1.0f;
    }
    const int64_t rows1 = (int64_t)E * N1, rows2 = (int64_t)E * H;
    if (gr >= rows1 + rows2) return;
    const bool first = gr < rows1;
    const int64_t r = first ? gr : gr - rows1;
    const int Nrows = first ? N1 : H;
    const int Kd = first ? H : I;
    const int e = (int)(r / Nrows), rr = (int)(r % Nrows);
    const __nv_bfloat16* src = first ? w1 + (size_t)r * H : w2 + (size_t)r * I;
    const int prow = first ? prepared_w1_row(rr, I, act) : rr;
    uint8_t* codes = first ? w1c + (size_t)e * N1 * H : w2c + (size_t)e * H * I;
    uint8_t* sf = first ? w1s + (size_t)e * N1 * (H / 32) : w2s + (size_t)e * H * (I / 32);
    for (int base = 0; base < Kd; base += 1024) {          // uniform across the warp
        const int c = base + lane * 32;
        const bool active = c < Kd;
        uint32_t q[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        uint32_t s = 0;
        if (active) {
            float v[32], h16[16];
            load16_bf16(src + c, h16);
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = h16[i];
            load16_bf16(src + c + 16, h16);
#pragma unroll
            for (int i = 0; i < 16; ++i) v[16 + i] = h16[i];
            s = quant_block32_mx(v, q);
        }
        const uint32_t word = pack_sf4(s);
        if (active) {
            uint4* dst = reinterpret_cast<uint4*>(codes + (size_t)prow * Kd + c);
            dst[0] = make_uint4(q[0], q[1], q[2], q[3]);
            dst[1] = make_uint4(q[4], q[5], q[6], q[7]);
            if ((lane & 3) == 0) *reinterpret_cast<uint32_t*>(sf + sf_offset_mx(prow, c / 32, Kd)) = word;
        }
    }
}

// One warp per weight row (W1 rows first, then W2 rows).
__global__ void __launch_bounds__(256) prep_quant_kernel(int E, int N1, int H, int I, int act,
                                                         const __nv_bfloat16* __restrict__ w1,
                                                         const __nv_bfloat16* __restrict__ w2,
                                                         const float* __restrict__ gw1, const float* __restrict__ gw2,
                                                         uint8_t* __restrict__ w1c, uint8_t* __restrict__ w1s,
                                                         uint8_t* __restrict__ w2c, uint8_t* __restrict__ w2s) {
    const int lane = threadIdx.x & 31;
    const int64_t gr = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int64_t rows1 = (int64_t)E * N1, rows2 = (int64_t)E * H;
    if (gr >= rows1 + rows2) return;
    const bool first = gr < rows1;
    const int64_t r = first ? gr : gr - rows1;
    const int Nrows = first ? N1 : H;
    const int Kd = first ? H : I;
    const int e = (int)(r / Nrows), rr = (int)(r % Nrows);
    const __nv_bfloat16* src = first ? w1 + (size_t)r * H : w2 + (size_t)r * I;
    const float G = first ? gw1[e] : gw2[e];
    const int prow = first ? prepared_w1_row(rr, I, act) : rr;
    uint8_t* codes = first ? w1c + (size_t)e * N1 * (H / 2) : w2c + (size_t)e * H * (I / 2);
    uint8_t* sf = first ? w1s + (size_t)e * N1 * (H / 16) : w2s + (size_t)e * H * (I / 16);
    for (int base = 0; base < Kd; base += 512) {
        const int c = base + lane * 16;
        const bool active = c < Kd;
        float v[16];
        uint32_t q[2] = {0u, 0u};
        uint32_t s = 0;
        if (active) {
            load16_bf16(src + c, v);
            s = quant_block16(v, G, q);
        }
        const uint32_t word = pack_sf4(s);
        if (active) {
            *reinterpret_cast<uint2*>(codes + (size_t)prow * (Kd / 2) + c / 2) = make_uint2(q[0], q[1]);
            if ((lane & 3) == 0) *reinterpret_cast<uint32_t*>(sf + sf_offset(prow, c / 16, Kd)) = word;
        }
    }
}

__global__ void debug_convert_kernel(const float* __restrict__ in, int64_t n, uint8_t* __restrict__ e4m3,
                                     uint8_t* __restrict__ e2m1) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const float v = in[i];
        uint16_t r;
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
        e4m3[i] = (uint8_t)(r & 0xFF);
        e2m1[i] = (uint8_t)(f32x2_to_e2m1x2(v, 0.0f) & 0xF);
    }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
// Threads of a one-row-per-CTA kernel: one per 16-element block, a whole
// number of warps, at most 1024 (rows longer than 16K elements loop).
static unsigned row_threads(int n) {
    int t = (n / 16 + 31) / 32 * 32;
    if (t > 1024) t = 1024;
    return (unsigned)t;
}

cudaError_t launch_quantize_x(const LaunchCtx& c, int T, int H, int K, const void* x, const float* g1_in,
                              int per_token, float* g1_out, const RouteScatter& rs, uint8_t* codes, uint8_t* sf,
                              float* y_acc_zero) {
    const int per = (H / 16 + 1023) / 1024;
    const dim3 grid(T), block(row_threads(H));
    const __nv_bfloat16* xb = (const __nv_bfloat16*)x;
    // per_token 2 = per-token with 4-over-6 blocks
#define MOE_QX(P, F) \
    c.launch(quantize_x_kernel<P, F>, grid, block, 0, T, H, K, xb, g1_in, per_token, g1_out, rs, codes, sf, y_acc_zero)
    if (per_token == 2) return per <= 1 ? MOE_QX(1, true) : per <= 2 ? MOE_QX(2, true) : MOE_QX(4, true);
    return per <= 1 ? MOE_QX(1, false) : per <= 2 ? MOE_QX(2, false) : MOE_QX(4, false);
#undef MOE_QX
}

cudaError_t launch_gather_x_bf16(const LaunchCtx& c, int T, int H, int K, const void* x, const RouteScatter& rs,
                                 void* x_perm, float* y_acc_zero) {
    return c.launch(gather_x_bf16_kernel, dim3((T + 7) / 8), dim3(256), 0, T, H, K, (const __nv_bfloat16*)x, rs,
                    (__nv_bfloat16*)x_perm, y_acc_zero);
}

cudaError_t launch_quantize_h(const LaunchCtx& c, uint64_t rows_cap, int I, const int* meta,
                              const int* route_of_row, const float* h, float* g2, uint8_t* codes, uint8_t* sf,
                              int four_six) {
    const int per = (I / 16 + 1023) / 1024;
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const uint64_t want = (uint64_t)sms * (2048 / row_threads(I));   // enough CTAs to fill every SM
    const dim3 grid((unsigned)(rows_cap < want ? rows_cap : want)), block(row_threads(I));
#define MOE_QH(P, F) c.launch(quantize_h_kernel<P, F>, grid, block, 0, I, meta, route_of_row, h, g2, codes, sf)
    if (four_six) return per <= 1 ? MOE_QH(1, true) : per <= 2 ? MOE_QH(2, true) : MOE_QH(4, true);
    return per <= 1 ? MOE_QH(1, false) : per <= 2 ? MOE_QH(2, false) : MOE_QH(4, false);
#undef MOE_QH
}

cudaError_t launch_finalize_deterministic(const LaunchCtx& c, int T, int H, int K, const int* row_of_route,
                                          const float* topk_w, int weight_on_output, const void* o, void* y) {
    const int64_t groups = (int64_t)T * (H / 8);
    return c.launch(finalize_det_kernel, dim3((unsigned)((groups + 255) / 256)), dim3(256), 0, T, H, K, row_of_route,
                    topk_w, weight_on_output, (const __nv_bfloat16*)o, (__nv_bfloat16*)y);
}

cudaError_t launch_finalize_fused(const LaunchCtx& c, int T, int H, const float* y_acc, void* y) {
    const int64_t n8 = (int64_t)T * H / 8;
    int64_t blocks = (n8 + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    return c.launch(finalize_fused_kernel, dim3((unsigned)blocks), dim3(256), 0, n8, y_acc, (__nv_bfloat16*)y);
}

cudaError_t launch_prepare(cudaStream_t s, int E, int N1, int H, int I, int act, const void* w1, const void* w2,
                           uint8_t* prepared, uint64_t gw1, uint64_t gw2, uint64_t w1c, uint64_t w1s, uint64_t w2c,
                           uint64_t w2s) {
    // per-matrix amax words (2E uint32) are kept at the start of the W1 code
    // region, which the final quantization kernel overwrites afterwards
    uint32_t* scratch = reinterpret_cast<uint32_t*>(prepared + w1c);
    prep_zero_kernel<<<(2 * E + 255) / 256, 256, 0, s>>>(scratch, 2 * E);
    const int64_t n1 = (int64_t)N1 * H, n2 = (int64_t)H * I;
    int64_t chunks = (n1 / 8 + 255) / 256;
    if (chunks > 64) chunks = 64;
    prep_amax_kernel<<<dim3((unsigned)chunks, E, 2), 256, 0, s>>>(E, n1, n2, (const __nv_bfloat16*)w1,
                                                                  (const __nv_bfloat16*)w2, scratch);
    prep_scales_kernel<<<(2 * E + 255) / 256, 256, 0, s>>>(E, scratch, reinterpret_cast<float*>(prepared + gw1),
                                                          reinterpret_cast<float*>(prepared + gw2));
    const int64_t rows = (int64_t)E * (N1 + H);
    prep_quant_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(
        E, N1, H, I, act, (const __nv_bfloat16*)w1, (const __nv_bfloat16*)w2,
        reinterpret_cast<const float*>(prepared + gw1), reinterpret_cast<const float*>(prepared + gw2),
        prepared + w1c, prepared + w1s, prepared + w2c, prepared + w2s);
    return cudaGetLastError();
}

cudaError_t launch_prepare_mx(cudaStream_t s, int E, int N1, int H, int I, int act, const void* w1, const void* w2,
                              uint8_t* prepared, uint64_t gw1, uint64_t gw2, uint64_t w1c, uint64_t w1s, uint64_t w2c,
                              uint64_t w2s) {
    const int64_t rows = (int64_t)E * (N1 + H);
    prep_quant_mx_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(
        E, N1, H, I, act, (const __nv_bfloat16*)w1, (const __nv_bfloat16*)w2, reinterpret_cast<float*>(prepared + gw1),
        reinterpret_cast<float*>(prepared + gw2), prepared + w1c, prepared + w1s, prepared + w2c, prepared + w2s);
    return cudaGetLastError();
}

cudaError_t launch_quantize_x_mx(const LaunchCtx& c, int T, int H, int K, const void* x, const RouteScatter& rs,
                                 uint8_t* codes, uint8_t* sf, float* y_acc_zero) {
    int threads = ((H / 32 + 31) / 32) * 32;
    if (threads > 1024) threads = 1024;
    return c.launch(quantize_x_mx_kernel, dim3(T), dim3(threads), 0, T, H, K, (const __nv_bfloat16*)x, rs, codes,
                    sf, y_acc_zero);
}

cudaError_t launch_debug_convert(cudaStream_t s, const float* in, int64_t n, uint8_t* e4m3, uint8_t* e2m1) {
    int64_t blocks = (n + 255) / 256;
    if (blocks > 8192) blocks = 8192;
    if (blocks < 1) blocks = 1;
    debug_convert_kernel<<<(unsigned)blocks, 256, 0, s>>>(in, n, e4m3, e2m1);
    return cudaGetLastError();
}

}  // namespace moe
