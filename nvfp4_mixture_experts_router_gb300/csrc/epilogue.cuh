// Fused GEMM epilogues shared by the NVFP4 (gemm_nvf4.cu) and W4A16
// (gemm_w4a16.cu) grouped GEMMs.  One thread owns one output row (one
// tensor-memory lane) and reads 128 FP32 accumulator columns of its tile.
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace moe {

// Per-row scalars of an epilogue: the route of the row (-1 in pad rows), its
// token, the product of the activation and weight global scales, the router
// weight applied to the FC1 output (input side), and the per-tensor FC2-input
// scale.  They depend only on the tile map and the routing, not on the
// accumulator: the epilogue loops load them before waiting for the
// accumulator, so that their (dependent) global-memory round trips overlap
// the main loop instead of delaying the accumulator's release.
struct EpiRow {
    int route;
    int token;
    float alpha;   // FC1: G_act(token) * Gw1[e]; FC2: G_act(row) * Gw2[e] (* route weight when scattering)
    float pw;      // FC1: route weight on the input side, else 1
    float g2;      // FC1 per-tensor requantization: the FC2-input scale
};

template <int EPI>
__device__ __forceinline__ EpiRow epi_row(const GemmParams& p, int row, int e) {
    constexpr bool kFc1 = EPI == kEpiFc1Quant || EPI == kEpiFc1F32 || EPI == kEpiFc1Bf16 || EPI == kEpiFc1Mx;
    EpiRow m;
    m.route = row >= 0 ? p.route_of_row[row] : -1;
    m.token = m.route >= 0 ? m.route / p.topk : 0;
    float g_act;
    if (kFc1) g_act = p.g_act == nullptr ? 1.0f : (p.g_act_per_token ? p.g_act[m.token] : p.g_act[0]);
    else g_act = p.g_act_per_token == 2 ? p.g_act[row] : (p.g_act ? p.g_act[0] : 1.0f);
    m.alpha = __fmul_rn(g_act, p.gw[e]);
    m.pw = (kFc1 && p.weight_on_input && m.route >= 0) ? p.topk_w[m.route] : 1.0f;
    if (EPI == kEpiFc2Scatter && m.route >= 0 && p.weight_on_output) m.alpha = m.alpha * p.topk_w[m.route];
    m.g2 = EPI == kEpiFc1Quant ? p.g2[0] : 1.0f;
    return m;
}

// FC1 activation of 32 columns in place.  SwiGLU: h holds 32 gate and u the
// matching 32 up accumulators; h <- silu(alpha g) (alpha u) pw.  ReLU2
// (u unused): h <- max(alpha h, 0)^2 pw.
__device__ __forceinline__ void fc1_act32(float (&h)[32], const float (&u)[32], bool swiglu, float alpha, float pw) {
    if (swiglu) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            // silu(z) = z / (1 + e^-z) with the ex2-based exponential and
            // the approximate division (relative error ~1e-6; for z below
            // about -88 the denominator is +inf and the result 0).  The
            // IEEE division + full-range expf, or a correctly rounded
            // reciprocal, cost 3-6x this epilogue and made FC1
            // epilogue-bound.
            const float zg = h[i] * alpha, zu = u[i] * alpha;
            h[i] = __fdividef(zg, 1.0f + __expf(-zg)) * zu * pw;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float z = fmaxf(h[i] * alpha, 0.0f);
            h[i] = z * z * pw;
        }
    }
}

// Store 32 activated FC1 outputs of route row `row` at columns col0..col0+31
// in the FC2-input format of EPI.
template <int EPI>
__device__ __forceinline__ void fc1_emit32(const GemmParams& p, const float (&h)[32], int row, int col0, float g2) {
    if (EPI == kEpiFc1Mx) {
        // one MXFP8 block per 32 columns: 32 E4M3 bytes and an E8M0 byte
        uint32_t q[8];
        const uint32_t sc = quant_block32_mx(h, q);
        uint4* dst = reinterpret_cast<uint4*>(p.out_codes + (size_t)row * p.out_cols + col0);
        dst[0] = make_uint4(q[0], q[1], q[2], q[3]);
        dst[1] = make_uint4(q[4], q[5], q[6], q[7]);
        p.out_sf[sf_offset_mx(row, col0 / 32, p.out_cols)] = (uint8_t)sc;
    } else if (EPI == kEpiFc1Quant) {
        uint32_t q[4];
        float blk[16];
        uint32_t c2[2];
#pragma unroll
        for (int i = 0; i < 16; ++i) blk[i] = h[i];
        const uint32_t s0 = quant_block16(blk, g2, c2);
        q[0] = c2[0]; q[1] = c2[1];
#pragma unroll
        for (int i = 0; i < 16; ++i) blk[i] = h[16 + i];
        const uint32_t s1 = quant_block16(blk, g2, c2);
        q[2] = c2[0]; q[3] = c2[1];
        *reinterpret_cast<uint4*>(p.out_codes + (size_t)row * (p.out_cols / 2) + col0 / 2) =
            make_uint4(q[0], q[1], q[2], q[3]);
        // two scales per 32 columns: a 16-bit store at an even scale index
        *reinterpret_cast<uint16_t*>(p.out_sf + sf_offset(row, col0 / 16, p.out_cols)) = (uint16_t)(s0 | (s1 << 8));
    } else if (EPI == kEpiFc1Bf16) {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(h[2 * i], h[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t*>(&b);
        }
        uint4* dst = reinterpret_cast<uint4*>(p.out_bf16 + (size_t)row * p.out_cols + col0);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    } else {
        float4* dst = reinterpret_cast<float4*>(p.out_f32 + (size_t)row * p.out_cols + col0);
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i] = make_float4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
    }
}

// SwiGLU tile: columns 0..63 gate, 64..127 up (prepared-weight interleave);
// yields 64 FC2-input values.  ReLU2 tile: 128 values.  Reads the
// accumulator chunk by chunk from tensor memory.
// COLS > 0 (BF16 output only): the BF16 rows go out through the warp's
// staging block stg in whole sectors (see staged_rows), every lane taking
// part; rows without a route write nothing.
template <int COLS, int NW, class Op>
__device__ __forceinline__ void staged_rows(uint32_t* stg, const uint32_t (&w)[NW], Op op);

template <int EPI, int COLS = 0>
__device__ __forceinline__ void epilogue_fc1(const GemmParams& p, uint32_t taddr, int row, const EpiRow& m,
                                             int n_tile, uint32_t* stg = nullptr) {
    const bool swiglu = p.act == MOE_ACT_SWIGLU;
    const int chunks = swiglu ? 2 : 4;
    for (int ch = 0; ch < chunks; ++ch) {
        float h[32], u[32];
        tmem_ld32(taddr + ch * 32, h);
        if (swiglu) tmem_ld32(taddr + 64 + ch * 32, u);
        tmem_ld_wait();
        fc1_act32(h, u, swiglu, m.alpha, m.pw);
        const int col0 = (swiglu ? n_tile * 64 : n_tile * 128) + ch * 32;
        if constexpr (COLS > 0 && EPI == kEpiFc1Bf16) {
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const __nv_bfloat162 b = __floats2bfloat162_rn(h[2 * i], h[2 * i + 1]);
                w[i] = *reinterpret_cast<const uint32_t*>(&b);
            }
            const int row0 = row - (threadIdx.x & 31);
            const int route = m.route;
            staged_rows<COLS>(stg, w, [&](int r, int w0, uint4 v) {
                if (__shfl_sync(0xffffffffu, route, r) >= 0)
                    *reinterpret_cast<uint4*>(p.out_bf16 + (size_t)(row0 + r) * p.out_cols + col0 + 2 * w0) = v;
            });
        } else {
            if (m.route >= 0) fc1_emit32<EPI>(p, h, row, col0, m.g2);
        }
    }
}

// The same epilogue on a slice the caller has already copied out of tensor
// memory (acc[c] = accumulator column c of the thread's row), so that the
// accumulator can be handed back to the MMA before this work starts.  COLS >
// 0 (FP32 output only): the rows go out through the warp's staging block stg
// (see staged_rows), every lane taking part; rows without a route write
// nothing.
template <int EPI, int COLS = 0>
__device__ __forceinline__ void epilogue_fc1_held(const GemmParams& p, const float (&acc)[128], int row,
                                                  const EpiRow& m, int n_tile, uint32_t* stg = nullptr) {
    auto emit = [&](const float (&h)[32], int col0) {
        if constexpr (COLS > 0 && EPI == kEpiFc1F32) {
            uint32_t w[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(h[i]);
            const int row0 = row - (threadIdx.x & 31);
            const int route = m.route;
            staged_rows<COLS>(stg, w, [&](int r, int w0, uint4 v) {
                if (__shfl_sync(0xffffffffu, route, r) >= 0)
                    *reinterpret_cast<uint4*>(p.out_f32 + (size_t)(row0 + r) * p.out_cols + col0 + w0) = v;
            });
        } else {
            if (m.route >= 0) fc1_emit32<EPI>(p, h, row, col0, m.g2);
        }
    };
    if (p.act == MOE_ACT_SWIGLU) {
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
            float h[32], u[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                h[i] = acc[ch * 32 + i];
                u[i] = acc[64 + ch * 32 + i];
            }
            fc1_act32(h, u, true, m.alpha, m.pw);
            emit(h, n_tile * 64 + ch * 32);
        }
    } else {
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
            float h[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) h[i] = acc[ch * 32 + i];
            fc1_act32(h, h, false, m.alpha, m.pw);
            emit(h, n_tile * 128 + ch * 32);
        }
    }
}

// Row segments through a per-warp shared-memory block.  After the
// tensor-memory load, lane r holds the words of route row r, so a global
// access issued straight from registers sends the 32 lanes to 32 different
// rows, 16 bytes each: every 32-byte L2 sector of a red or a store then
// carries half a sector.  Here each warp writes COLS words of its 32 rows
// into its block, row by row, and reads them back with COLS/4 lanes per row,
// so that one instruction covers whole COLS*4-byte segments of 32*4/COLS
// rows.  The 16-byte slots of a row are XOR-swizzled so that both the
// row-wise writes and the segment-wise reads are free of bank conflicts
// (a quarter warp touches eight distinct 16-byte bank groups either way).
// op(r, w0, v) gets row r of the warp, the word offset w0 of v in the row's
// NW words and the four words v; it runs on every lane (shuffles allowed).
template <int COLS, int NW, class Op>
__device__ __forceinline__ void staged_rows(uint32_t* stg, const uint32_t (&w)[NW], Op op) {
    static_assert(COLS == 8 || COLS == 16, "staging block of 8 or 16 words per row");
    static_assert(NW % COLS == 0, "whole staging blocks");
    constexpr int NQ = COLS / 4;          // 16-byte slots per row
    constexpr int RPL = 8 / NQ;           // rows per 128 bytes of the block
    constexpr int RPI = 32 / NQ;          // rows per read instruction
    const int lane = threadIdx.x & 31;
    uint4* blk = reinterpret_cast<uint4*>(stg);
#pragma unroll
    for (int sc = 0; sc < NW / COLS; ++sc) {
        __syncwarp();
#pragma unroll
        for (int j = 0; j < NQ; ++j)
            blk[lane * NQ + (j ^ ((lane / RPL) % NQ))] =
                make_uint4(w[sc * COLS + 4 * j], w[sc * COLS + 4 * j + 1], w[sc * COLS + 4 * j + 2],
                           w[sc * COLS + 4 * j + 3]);
        __syncwarp();
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
            const int r = i * RPI + lane / NQ, q = lane % NQ;
            op(r, sc * COLS + 4 * q, blk[r * NQ + (q ^ ((r / RPL) % NQ))]);
        }
    }
    __syncwarp();
}

// FC2 output of 32 columns (accumulators o, columns col0..col0+31 of the
// output row): BF16 per-route row (store) or alpha-scaled FP32 reduction
// into the token's row (scatter).  COLS > 0: through staged_rows with the
// warp's staging block stg (32 rows x COLS words), every lane taking part;
// COLS = 0 writes straight from registers.
template <int EPI, int COLS>
__device__ __forceinline__ void fc2_emit32(const GemmParams& p, const float (&o)[32], int row, const EpiRow& m,
                                           int col0, uint32_t* stg) {
    const int route = m.route;
    const float alpha = m.alpha;
    if constexpr (COLS > 0) {
        // rows without a route write nothing
        if constexpr (EPI == kEpiFc2Store) {
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const __nv_bfloat162 b = __floats2bfloat162_rn(o[2 * i] * alpha, o[2 * i + 1] * alpha);
                w[i] = *reinterpret_cast<const uint32_t*>(&b);
            }
            const int row0 = row - (threadIdx.x & 31);
            staged_rows<COLS>(stg, w, [&](int r, int w0, uint4 v) {
                if (__shfl_sync(0xffffffffu, route, r) >= 0)
                    *reinterpret_cast<uint4*>(p.out_bf16 + (size_t)(row0 + r) * p.out_cols + col0 + 2 * w0) = v;
            });
        } else {
            uint32_t w[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(o[i] * alpha);
            const int tk_lane = route >= 0 ? m.token : -1;
            staged_rows<COLS>(stg, w, [&](int r, int w0, uint4 v) {
                const int tk = __shfl_sync(0xffffffffu, tk_lane, r);
                if (tk >= 0)
                    red_add_f32x4(reinterpret_cast<float4*>(p.out_f32 + (size_t)tk * p.out_cols + col0 + w0),
                                  __uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z),
                                  __uint_as_float(v.w));
            });
        }
        return;
    }
    if (route < 0) return;
    if (EPI == kEpiFc2Store) {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(o[2 * i] * alpha, o[2 * i + 1] * alpha);
            w[i] = *reinterpret_cast<const uint32_t*>(&b);
        }
        uint4* dst = reinterpret_cast<uint4*>(p.out_bf16 + (size_t)row * p.out_cols + col0);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    } else {
        float4* dst = reinterpret_cast<float4*>(p.out_f32 + (size_t)m.token * p.out_cols + col0);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            red_add_f32x4(dst + i, o[4 * i] * alpha, o[4 * i + 1] * alpha, o[4 * i + 2] * alpha,
                          o[4 * i + 3] * alpha);
    }
}

// FC2 epilogue of a 128-column slice, read chunk by chunk from tensor memory.
template <int EPI, int COLS = 0>
__device__ __forceinline__ void epilogue_fc2(const GemmParams& p, uint32_t taddr, int row, const EpiRow& m,
                                             int n_tile, uint32_t* stg = nullptr) {
    for (int ch = 0; ch < 4; ++ch) {
        float o[32];
        tmem_ld32(taddr + ch * 32, o);
        tmem_ld_wait();
        fc2_emit32<EPI, COLS>(p, o, row, m, n_tile * 128 + ch * 32, stg);
    }
}

// The same on a slice already copied out of tensor memory (see
// epilogue_fc1_held).
template <int EPI, int COLS = 0>
__device__ __forceinline__ void epilogue_fc2_held(const GemmParams& p, const float (&acc)[128], int row,
                                                  const EpiRow& m, int n_tile, uint32_t* stg = nullptr) {
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
        float o[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = acc[ch * 32 + i];
        fc2_emit32<EPI, COLS>(p, o, row, m, n_tile * 128 + ch * 32, stg);
    }
}

}  // namespace moe
