// Layout arithmetic shared by the host orchestrator and the kernels:
// workspace and prepared-weight offsets, the 128x4 scale-factor atom, and
// the SwiGLU gate/up row interleave of the prepared FC1 weights.
#pragma once
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe_nvfp4.h"

#if defined(__CUDACC__)
#define MOE_HD __host__ __device__ __forceinline__
#else
#define MOE_HD inline
#endif

namespace moe {

constexpr int kTileM = 128;        // routes per M tile (expert segments padded to this)
constexpr int kTileN = 128;        // output columns per N tile
constexpr int kGluChunk = 64;      // SwiGLU: 64 gate rows then 64 up rows per 128-row tile
constexpr int kUnitTokens = 32;    // tokens per permute unit

MOE_HD uint64_t align_up(uint64_t v, uint64_t a) { return (v + a - 1) / a * a; }

MOE_HD int act_of(uint32_t flags) { return (int)(flags & MOE_ACT_MASK); }
MOE_HD int mode_of(uint32_t flags) { return (int)((flags & MOE_MODE_MASK) >> 2); }
constexpr int kModePerTensor = 0, kModePerToken = 1, kModeW4A16 = 2, kModeMxfp8 = 3;

MOE_HD int n1_of(int I, uint32_t flags) { return act_of(flags) == MOE_ACT_SWIGLU ? 2 * I : I; }

// Padded-row capacity: every expert holding at least one route adds at most
// kTileM-1 pad rows.
MOE_HD uint64_t rows_capacity(int T, int K, int E) {
    const uint64_t R = (uint64_t)T * (uint64_t)K;
    const uint64_t busy = R < (uint64_t)E ? R : (uint64_t)E;
    return align_up(R + busy * (kTileM - 1), kTileM);
}

// Byte offset of scale j of row r inside a scale tensor laid out as
// [rows/128][cols/64][512]: a 512-byte atom holds 128 rows x 4 scales,
// byte (r%32)*16 + ((r/32)%4)*4 + j%4.  This is the layout tcgen05.cp
// (32x128b, warpx4) moves into tensor memory for a 128-row block-scaled MMA.
MOE_HD uint64_t sf_offset(uint64_t r, uint64_t j, uint64_t cols) {
    return ((r >> 7) * (cols >> 6) + (j >> 2)) * 512u + (r & 31u) * 16u + ((r >> 5) & 3u) * 4u + (j & 3u);
}

// The same atom layout for MXFP8 scales (one E8M0 per 32 elements): an
// atom holds 128 rows x 4 scales covering 128 elements of K, so `j` (the
// 32-element block) groups by four as above and `cols` counts elements.
MOE_HD uint64_t sf_offset_mx(uint64_t r, uint64_t j, uint64_t cols) {
    return ((r >> 7) * (cols >> 7) + (j >> 2)) * 512u + (r & 31u) * 16u + ((r >> 5) & 3u) * 4u + (j & 3u);
}

// Prepared FC1 row of checkpoint row `r` (SwiGLU: rows [0, I) gate, [I, 2I) up).
MOE_HD int prepared_w1_row(int r, int I, int act) {
    if (act != MOE_ACT_SWIGLU) return r;
    const bool up = r >= I;
    const int j = up ? r - I : r;
    return (j / kGluChunk) * (2 * kGluChunk) + (up ? kGluChunk : 0) + (j % kGluChunk);
}

struct PreparedLayout {
    uint64_t gw1, gw2, w1_codes, w1_sf, w2_codes, w2_sf, total;
    uint64_t w1_codes_per_expert, w1_sf_per_expert, w2_codes_per_expert, w2_sf_per_expert;
};

// NVFP4 weights (every mode but MXFP8): half a byte per element and a scale
// per 16; MXFP8 weights: a byte per element and a scale per 32.
MOE_HD PreparedLayout prepared_layout(moe_shape s, uint32_t flags) {
    PreparedLayout L{};
    const uint64_t E = (uint64_t)s.E, H = (uint64_t)s.H, I = (uint64_t)s.I;
    const uint64_t N1 = (uint64_t)n1_of(s.I, flags);
    const bool mx = mode_of(flags) == kModeMxfp8;
    const uint64_t cdiv = mx ? 1 : 2, sdiv = mx ? 32 : 16;
    L.w1_codes_per_expert = N1 * H / cdiv;
    L.w1_sf_per_expert = N1 * H / sdiv;
    L.w2_codes_per_expert = H * I / cdiv;
    L.w2_sf_per_expert = H * I / sdiv;
    uint64_t o = 0;
    L.gw1 = o; o = align_up(o + 4 * E, 256);
    L.gw2 = o; o = align_up(o + 4 * E, 256);
    L.w1_codes = o; o = align_up(o + E * L.w1_codes_per_expert, 256);
    L.w1_sf = o; o = align_up(o + E * L.w1_sf_per_expert, 256);
    L.w2_codes = o; o = align_up(o + E * L.w2_codes_per_expert, 256);
    L.w2_sf = o; o = align_up(o + E * L.w2_sf_per_expert, 256);
    L.total = o;
    return L;
}

inline moe_workspace_layout workspace_layout(moe_shape s, uint32_t flags) {
    moe_workspace_layout L;
    {   // regions a mode does not use keep the marker UINT64_MAX
        uint64_t* f = reinterpret_cast<uint64_t*>(&L);
        for (size_t i = 0; i < sizeof(L) / sizeof(uint64_t); ++i) f[i] = ~0ull;
    }
    const uint64_t T = (uint64_t)s.T, H = (uint64_t)s.H, I = (uint64_t)s.I;
    const uint64_t E = (uint64_t)s.E, K = (uint64_t)s.K;
    const uint64_t cap = rows_capacity(s.T, s.K, s.E);
    const uint64_t units = (T + kUnitTokens - 1) / kUnitTokens;
    const int mode = mode_of(flags);
    const bool det = (flags & MOE_FINALIZE_DETERMINISTIC) != 0;
    L.rows_cap = cap;
    uint64_t o = 0;
    auto take = [&](uint64_t bytes) { uint64_t at = o; o = align_up(o + bytes, 256); return at; };
    L.status = take(16);
    // the unit masks follow the status word: the single-kernel forward
    // zeroes both with one memset before its launch
    L.unit_mask = take(4 * E * units);
    L.topk_ids = take(4 * T * K);
    L.topk_w = take(4 * T * K);
    L.count = take(4 * E);
    L.offsets = take(4 * (E + 1));
    L.padded_offsets = take(4 * (E + 1));
    L.meta = take(16);
    L.unit_base = take(4 * E * units);
    L.row_of_route = take(4 * T * K);
    L.route_of_row = take(4 * cap);
    L.tile_expert = take(4 * (cap / kTileM));
    L.tile_pair = take(4 * (cap / kTileM));
    L.tile_half = take(4 * 2 * (cap / kTileM));
    if (mode == kModeMxfp8) {
        // E4M3 codes, E8M0 scales per 32 (no global scales)
        L.xq_codes = take(cap * H);
        L.xq_sf = take(cap * H / 32);
        L.hq_codes = take(cap * I);
        L.hq_sf = take(cap * I / 32);
    } else if (mode != kModeW4A16) {
        L.g1 = take(4 * T);
        L.xq_codes = take(cap * H / 2);
        L.xq_sf = take(cap * H / 16);
        L.hq_codes = take(cap * I / 2);
        L.hq_sf = take(cap * I / 16);
        if (mode == kModePerToken) {
            L.h_f32 = take(4 * cap * I);
            L.g2 = take(4 * cap);
        }
    } else {
        L.x_bf16_perm = take(2 * cap * H);
        L.h_bf16 = take(2 * cap * I);
    }
    if (det) L.o_bf16 = take(2 * cap * H);
    else L.y_acc = take(4 * T * H);
    if (flags & MOE_ROUTER_GEMM) L.logits = take(4 * T * E);
    L.total = o;
    return L;
}

}  // namespace moe
