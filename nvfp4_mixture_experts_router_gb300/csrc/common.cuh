// Device-side building blocks for sm_103a: NVFP4 conversions, mbarriers with
// bounded waits, TMA (cp.async.bulk[.tensor]) loads, and the tcgen05 tensor
// core / tensor-memory instructions, all as inline PTX.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "layout.h"

namespace moe {

// ---------------------------------------------------------------------------
// status word bits (workspace status[0])
// ---------------------------------------------------------------------------
constexpr uint32_t kStatusTimeoutProducer = 1u << 0;
constexpr uint32_t kStatusTimeoutMma = 1u << 1;
constexpr uint32_t kStatusTimeoutEpilogue = 1u << 2;
constexpr uint32_t kStatusBadExpert = 1u << 3;
constexpr uint32_t kStatusBadRow = 1u << 4;
constexpr uint32_t kStatusTimeoutGrid = 1u << 5;   // fused layer: a grid barrier gave up
constexpr uint32_t kStatusGridAbort = 1u << 6;     // fused layer: a CTA stopped early

// One bounded wait gives up after this many nanoseconds of %globaltimer.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// NVFP4 conversions (round-to-nearest-even, saturating)
// ---------------------------------------------------------------------------
// E4M3 code of a non-negative float (low byte of cvt.rn.satfinite.e4m3x2).
__device__ __forceinline__ uint32_t f32_to_e4m3(float v) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
    return r & 0xFFu;
}

// Two E4M3 codes (signed, satfinite): `lo` -> bits 0-7, `hi` -> bits 8-15.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Exact float value of an E4M3 code (finite codes; 0x7F/0xFF give NaN).
__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
    uint32_t r;
    asm("{\n .reg .b16 lo;\n .reg .f16x2 h2;\n cvt.u16.u32 lo, %1;\n"
        " cvt.rn.f16x2.e4m3x2 h2, lo;\n mov.b32 %0, h2;\n}\n"
        : "=r"(r) : "r"(code & 0xFFu));
    return __half2float(__ushort_as_half(static_cast<unsigned short>(r & 0xFFFFu)));
}

// Two E2M1 codes in one byte: `lo` -> bits 0-3, `hi` -> bits 4-7.
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float lo, float hi) {
    uint32_t r;
    asm("{\n .reg .b8 b;\n cvt.rn.satfinite.e2m1x2.f32 b, %1, %2;\n cvt.u32.u8 %0, b;\n}\n"
        : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Quantize 16 consecutive values (one NVFP4 block) with global scale G:
//   s = E4M3((amax / G) / 6); inv = s == 0 ? 0 : 1 / (s * G); q = E2M1(v * inv)
// every step rounded to float32 nearest-even (explicit _rn intrinsics keep the
// compiler from contracting or approximating them).  Returns the scale code;
// writes 8 code bytes (two per byte, even element in the low nibble).
__device__ __forceinline__ uint32_t quant_block16(const float (&v)[16], float G, uint32_t (&codes)[2]) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const uint32_t s = f32_to_e4m3(__fdiv_rn(__fdiv_rn(amax, G), 6.0f));
    const float sv = e4m3_to_f32(s);
    const float inv = (sv == 0.0f) ? 0.0f : __fdiv_rn(1.0f, __fmul_rn(sv, G));
#pragma unroll
    for (int w = 0; w < 2; ++w) {
        uint32_t word = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int i = w * 8 + b * 2;
            word |= f32x2_to_e2m1x2(__fmul_rn(v[i], inv), __fmul_rn(v[i + 1], inv)) << (8 * b);
        }
        codes[w] = word;
    }
    return s;
}

// Global scale of a row from its amax: amax / 2688 (6 * 448), 1 if zero.
__device__ __forceinline__ float global_scale_from_amax(float amax) {
    return amax == 0.0f ? 1.0f : __fdiv_rn(amax, 2688.0f);
}
// Under 4-over-6 quantization: amax / 1536 (6 * 256), so that the larger
// max-4 block scale (at most 384) stays inside the E4M3 range.
constexpr float kScaleDiv4over6 = 1536.0f;
__device__ __forceinline__ float global_scale_from_amax_4over6(float amax) {
    return amax == 0.0f ? 1.0f : __fdiv_rn(amax, kScaleDiv4over6);
}

// E2M1 value of a 4-bit code (sign in bit 3), without a table in local
// memory: magnitude codes 2..7 are 2^((c>>1)-1) * (1 + (c&1)/2), i.e. float32
// exponent field 126 + (c>>1) and mantissa bit 22 = c&1; codes 0 and 1 are
// 0 and 0.5.
__device__ __forceinline__ float e2m1_to_f32(uint32_t c) {
    const uint32_t m = c & 7u;
    const float mag = m >= 2u ? __uint_as_float(((126u + (m >> 1)) << 23) | ((m & 1u) << 22)) : 0.5f * (float)m;
    return (c & 8u) ? -mag : mag;
}

// MXFP8 (OCP MX, block 32, E4M3 elements, E8M0 scale): shared exponent
// floor(log2 amax) - 8, clamped to [-127, 127]; -127 for an all-zero block.
__device__ __forceinline__ int mx_block_exp(float amax) {
    const uint32_t b = __float_as_uint(amax);
    if (!(amax > 0.0f) || (b >> 23) >= 255u) return -127;
    const int fl = (b >> 23) == 0 ? (31 - __clz((int)(b & 0x7FFFFFu))) - 149 : (int)(b >> 23) - 127;
    return max(-127, min(127, fl - 8));
}
// 2^k as a float for k in [-127, 127] (2^-127 is subnormal).
__device__ __forceinline__ float pow2f(int k) {
    return k >= -126 ? __uint_as_float((uint32_t)(k + 127) << 23) : __uint_as_float(0x00400000u);
}
// Quantize 32 consecutive values: 32 E4M3 codes (element 4w+b in byte b of
// word w) and the returned E8M0 code e + 127.  v * 2^-e is an exact
// power-of-two scaling.
__device__ __forceinline__ uint32_t quant_block32_mx(const float (&v)[32], uint32_t (&codes)[8]) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const int e = mx_block_exp(amax);
    const float sc = pow2f(-e);
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const uint32_t lo = f32x2_to_e4m3x2(__fmul_rn(v[4 * w], sc), __fmul_rn(v[4 * w + 1], sc));
        const uint32_t hi = f32x2_to_e4m3x2(__fmul_rn(v[4 * w + 2], sc), __fmul_rn(v[4 * w + 3], sc));
        codes[w] = lo | (hi << 16);
    }
    return (uint32_t)(e + 127);
}

// One candidate of 4-over-6: the block quantized with its maximum mapped to
// M (t = amax / G), and the float32 squared dequantization error summed in
// element order (d_i = v_i - (e2m1_i * s) * G, every step rounded to nearest).
__device__ __forceinline__ float quant_candidate16(const float (&v)[16], float G, float t, float M,
                                                   uint32_t (&codes)[2], uint32_t& s_out) {
    const uint32_t s = f32_to_e4m3(__fdiv_rn(t, M));
    const float sv = e4m3_to_f32(s);
    const float inv = (sv == 0.0f) ? 0.0f : __fdiv_rn(1.0f, __fmul_rn(sv, G));
    float err = 0.0f;
#pragma unroll
    for (int w = 0; w < 2; ++w) {
        uint32_t word = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int i = w * 8 + b * 2;
            const uint32_t pair = f32x2_to_e2m1x2(__fmul_rn(v[i], inv), __fmul_rn(v[i + 1], inv));
            word |= pair << (8 * b);
            const float d0 = __fsub_rn(v[i], __fmul_rn(__fmul_rn(e2m1_to_f32(pair & 15u), sv), G));
            const float d1 = __fsub_rn(v[i + 1], __fmul_rn(__fmul_rn(e2m1_to_f32(pair >> 4), sv), G));
            err = __fadd_rn(err, __fmul_rn(d0, d0));
            err = __fadd_rn(err, __fmul_rn(d1, d1));
        }
        codes[w] = word;
    }
    s_out = s;
    return err;
}

// 4-over-6 block quantization: the max-6 and the max-4 candidates, keeping
// the one with the smaller squared error (ties keep max-6).
__device__ __forceinline__ uint32_t quant_block16_4over6(const float (&v)[16], float G, uint32_t (&codes)[2]) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const float t = __fdiv_rn(amax, G);
    uint32_t c6[2], c4[2], s6, s4;
    const float e6 = quant_candidate16(v, G, t, 6.0f, c6, s6);
    const float e4 = quant_candidate16(v, G, t, 4.0f, c4, s4);
    const bool four = e4 < e6;
    codes[0] = four ? c4[0] : c6[0];
    codes[1] = four ? c4[1] : c6[1];
    return four ? s4 : s6;
}

// Padded row of token t's route to expert e: the (expert, unit) starting row
// plus the number of the unit's earlier tokens that chose e (bit j of the
// unit's mask of e is token u*32+j).
__device__ __forceinline__ int route_row(int t, int e, int U, const int* __restrict__ unit_base,
                                         const uint32_t* __restrict__ unit_mask) {
    const int u = t / kUnitTokens, j = t % kUnitTokens;
    const size_t idx = (size_t)e * U + u;
    return unit_base[idx] + __popc(unit_mask[idx] & ((1u << j) - 1u));
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// CLUSTER = true: acquire at cluster scope, for phases completed by arrivals
// from the other CTA of a pair.
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    if (CLUSTER)
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(smem_u32(bar)), "r"(parity)
            : "memory");
    else
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(smem_u32(bar)), "r"(parity)
            : "memory");
    return ok != 0;
}

// Bounded wait for the phase with `parity`.  Gives up (returns false) when
// *abort is set by another role or after kWaitLimitNs; in the latter case it
// sets *abort and ORs `err_bit` into the global status word.
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          unsigned int* status, uint32_t err_bit) {
    if (mbar_try_wait<CLUSTER>(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait<CLUSTER>(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                *abort = 1;
                if (status) atomicOr(status, err_bit);
                return false;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// TMA
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
        : "memory");
}

// 3-D tile copy: {x, y, z} coordinates of the box's first element.
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory, MMA, copies
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_result, uint32_t ncols) {  // whole warp
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_result)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {  // whole warp
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrive on `bar` once all previously issued tcgen05 async ops of this thread complete.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address >> 4 in
// bits 0-13, leading byte offset >> 4 in 16-29, stride byte offset >> 4 in
// 32-45, descriptor version 1 in 46-47, swizzle mode in 61-63.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swizzle) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)swizzle << 61;
    return d;
}
constexpr uint32_t kSwizzleNone = 0, kSwizzle128B = 2;

// K-major operand tile of 128-byte rows, 128-byte swizzle (8-row atoms of 1 KB).
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t saddr) {
    return sdesc(saddr, 16, 1024, kSwizzle128B);
}

// Instruction descriptor, block-scaled MMA kind::mxf4nvf4 with E2M1 A and B
// (format code 1 at bits 7-9 / 10-12), K-major both, UE4M3 scales (bit 23 =
// 0), N >> 3 at bits 17-22, M >> 4 at bits 24-28, scale-factor ids 0.
__host__ __device__ constexpr uint32_t idesc_nvf4(int M, int N) {
    return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// Instruction descriptor, block-scaled MMA kind::mxf8f6f4 with E4M3 A and B
// (format code 0), UE8M0 scales (bit 23), scale-factor byte ids at bits
// 29-30 (A) and 4-5 (B): with one scale per 32 elements (scale_vec::1X) the
// four K = 32 MMAs of a 128-element chunk share one scale word per row and
// pick byte `sf_id` of it.
__host__ __device__ constexpr uint32_t idesc_mxf8(int M, int N, int sf_id) {
    return ((uint32_t)sf_id << 4) | ((uint32_t)(N >> 3) << 17) | (1u << 23) | ((uint32_t)(M >> 4) << 24) |
           ((uint32_t)sf_id << 29);
}
// Instruction descriptor, kind::f16 with BF16 A/B (format 1) and FP32 D
// (bits 4-5 = 1), K-major both.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
        " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n}\n" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_mma_mxf8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
        " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n}\n" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// ---------------------------------------------------------------------------
// CTA pairs (thread-block clusters of 2) and the pair-wide tcgen05 forms
// ---------------------------------------------------------------------------
// In a kernel that uses cta_group::2 every tcgen05 instruction carrying a
// cta_group qualifier (alloc, dealloc, relinquish, mma, commit) uses ::2.
__device__ __forceinline__ uint32_t cluster_cta_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// All threads of both CTAs (warp-uniform call sites only).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// shared::cluster address of this CTA's shared-memory object `p` in CTA `rank`.
__device__ __forceinline__ uint32_t cluster_map(const void* p, uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
    return a;
}
// Arrive on an mbarrier of any CTA of the cluster, without release
// semantics.  Used only where what the arrival announces is already complete
// and visible (landed TMA copies, waited-for tensor-memory loads and stores):
// a release at cluster scope made each such arrival wait for the SM's
// outstanding memory traffic (0.5-3 us measured).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// Arrive on the other CTA's mbarrier after writes to this CTA's own shared
// memory that the pair MMA (issued by the other CTA) reads: release at CTA
// scope orders the writes (and, after __syncwarp, the warp's) before the
// arrival without the cluster-wide fence of a cluster-scope release, which
// waits for the SM's outstanding memory traffic (microseconds under load).
// The writer issues fence.proxy.async first, for the tensor core's reads.
__device__ __forceinline__ void mbar_arrive_remote_cta_release(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
// Both CTAs of the pair each run this in one warp; the two allocations are
// made together and sit at the same tensor-memory address in both.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* smem_result, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_result)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// M = 256 block-scaled MMA over the CTA pair, issued by the even CTA: rows
// 0..127 of A, D and the A scales live in the even CTA, rows 128..255 in the
// odd one (same shared-memory / tensor-memory addresses); B is split by rows
// (first half in the even CTA) and every CTA's tensor memory holds the B
// scales of all N rows.
__device__ __forceinline__ void tc_mma_nvf4_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
        " tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n}\n" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}
// Tile copies whose completion is counted on an mbarrier of either CTA of the
// pair (`bar` a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "l"(policy)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(void* smem_dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                                 int z, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z), "l"(policy)
        : "memory");
}

// M = 256 BF16 MMA over the CTA pair (kind::f16, FP32 accumulate), issued by
// the even CTA; operand halves split as in tc_mma_nvf4_pair, no scales.
__device__ __forceinline__ void tc_mma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive on the mbarrier at `bar`'s offset in every CTA of `cta_mask` once all
// previously issued pair MMAs of this thread have completed.
__device__ __forceinline__ void tc_commit_pair_mc(uint64_t* bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// Load 32 consecutive FP32 columns of this warp's 32 lanes.
// 8 consecutive accumulator columns of this thread's lane.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Store 16 / 32 consecutive 32-bit columns of this warp's 32 lanes.
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t (&r)[4]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(r[0]), "r"(r[1]),
                 "r"(r[2]), "r"(r[3])
                 : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
// N consecutive columns, N in {4, 8, 16, 32}.
template <int N>
__device__ __forceinline__ void tmem_st_n(uint32_t taddr, const uint32_t (&r)[N]) {
    static_assert(N == 4 || N == 8 || N == 16 || N == 32, "tcgen05.st width");
    if constexpr (N == 4) tmem_st4(taddr, r);
    else if constexpr (N == 8) tmem_st8(taddr, r);
    else if constexpr (N == 16) tmem_st16(taddr, r);
    else tmem_st32(taddr, r);
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Per-warpgroup register budget (all four warps of a warpgroup execute the
// same instruction).  An increase waits until the block's pool, fixed at
// launch (threads x registers per thread), has the registers free, so the
// kernels that use these check the launch register count on the host.
template <uint32_t N>
__device__ __forceinline__ void regs_release() {
    static_assert(N % 8 == 0 && N >= 24 && N <= 256, "setmaxnreg range");
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_claim() {
    static_assert(N % 8 == 0 && N >= 24 && N <= 256, "setmaxnreg range");
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// Programmatic dependent launch: wait for the preceding grid's results /
// allow the next grid to start its prologue.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Fire-and-forget FP32 vector reduction into global memory (red, no
// returned value).  Stated explicitly: the same float4 atomicAdd was
// measured to become a returning atomic in one kernel and a reduction in
// another, and the returning form halved the throughput of the scatter
// epilogue.
__device__ __forceinline__ void red_add_f32x4(float4* addr, float a, float b, float c, float d) {
    asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c),
                 "f"(d)
                 : "memory");
}

// Deterministic finalize of 8 output elements: acc = sum over the K routes
// of token t, k ascending, of w'_k * o[row(t, k)][8c .. 8c+8) with FP32 fma
// (w' = the router weight on the output side, else 1; dropped routes,
// row -1, skipped).  The rows are loaded four at a time (L2 loads: the
// inputs may come from other CTAs of the same kernel).
__device__ __forceinline__ void finalize_det_group(int t, int c, int H, int K, const int* row_of_route,
                                                   const float* topk_w, int weight_on_output,
                                                   const __nv_bfloat16* o, float (&acc)[8]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    for (int k0 = 0; k0 < K; k0 += 4) {
        int row[4];
        float w[4];
        uint4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int k = k0 + j;
            row[j] = k < K ? __ldcg(row_of_route + (size_t)t * K + k) : -1;
            w[j] = (k < K && weight_on_output) ? __ldcg(topk_w + (size_t)t * K + k) : 1.0f;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
            v[j] = row[j] >= 0 ? __ldcg(reinterpret_cast<const uint4*>(o + (size_t)row[j] * H) + c)
                               : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (row[j] < 0) continue;
            const uint32_t u[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[2 * i] = fmaf(w[j], __uint_as_float(u[i] << 16), acc[2 * i]);
                acc[2 * i + 1] = fmaf(w[j], __uint_as_float(u[i] & 0xFFFF0000u), acc[2 * i + 1]);
            }
        }
    }
}

// Eight FP32 values rounded to BF16 (nearest even), packed in order.
__device__ __forceinline__ uint4 pack_bf16x8(const float (&a)[8]) {
    uint32_t out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(a[2 * i], a[2 * i + 1]);
        out[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

}  // namespace moe
