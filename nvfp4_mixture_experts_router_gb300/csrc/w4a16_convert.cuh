// Weight widening of the W4A16 GEMMs (gemm_w4a16.cu, gemm_w4a16_swap.cu):
// E2M1 codes times their E4M3 block scale, written as BF16 into the
// 128-byte-swizzled K-major shared-memory layout the tensor core reads.
#pragma once
#include "common.cuh"

namespace moe {

// 8 E2M1 codes (4 bytes, low nibble first) times scale s -> 8 BF16, given
// s2 = s in both halves of an f16x2 (exact: E4M3 values are normal f16).
// Each code pair is widened to f16x2 and multiplied by s2 in f16 -- exact,
// the product has at most 6 significant bits and lies in [2^-10, 2688] --
// then widened to FP32 and packed to BF16 (exact again).
__device__ __forceinline__ uint4 dequant8(uint32_t codes, __half2 s2) {
    uint32_t h2[4];
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}\n"
        : "=r"(h2[0]), "=r"(h2[1]), "=r"(h2[2]), "=r"(h2[3])
        : "r"(codes));
    uint32_t out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 p = __hmul2(*reinterpret_cast<const __half2*>(&h2[i]), s2);   // exact
        const float2 f = __half22float2(p);
        const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);                    // exact
        out[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace moe
