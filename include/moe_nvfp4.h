/*
 * moe_nvfp4.h — C ABI of libmoe_nvfp4.so: a single-GPU NVFP4 Mixture-of-
 * Experts layer forward for NVIDIA GB300 (sm_103a).
 *
 * The layer (sources cited by page title and section):
 *   router softmax + top-K            ["MegaMoE" blog, "The problem"]
 *   token permutation by expert       [FlashInfer PR #4366: the "contiguous
 *                                      gather" grouped GEMM; "Tests": cluster
 *                                      padding and partial tiles]
 *   activation quantization to NVFP4  ["MegaMoE", "Our approach": W4A4 with
 *   (E2M1 + E4M3 block-16 scales +     block-16 scaling; newruntime post on
 *   FP32 per-tensor or per-token       PR #5319, "Retrieval answer": W4A4
 *   global scale)                      per-tensor or per-token, W4A16]
 *   grouped GEMM FC1 (gate|up) + SwiGLU or ReLU2, router weight on the FC2
 *   input or at the output reduction, requantization to NVFP4
 *                                     [PR #4366, "Motivation"]
 *   grouped GEMM FC2
 *   finalize: unpermute + weighted top-K reduction, fused into the FC2
 *   epilogue or a separate deterministic kernel
 *                                     [PR #5319 post, "Retrieval answer":
 *                                      fused vs --no-fused-finalize]
 *   W4A16 variant: NVFP4 weights, BF16 activations.
 *
 * Conventions for every entry point:
 *   - All data pointers are DEVICE pointers owned by the caller; the library
 *     never allocates device memory and keeps no pointer after returning.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Every
 *     entry point except moe_nvfp4_last_device_status only enqueues work on
 *     `stream` and returns without synchronizing.
 *   - Arguments are validated on the host before anything is launched; an
 *     invalid call returns an error code and enqueues nothing.  Device-side
 *     faults are never used to report errors.
 *   - Numeric contract: see the per-function comments; results do not depend
 *     on the stream, the launch order of other work, or the SM count, except
 *     the fused finalize (floating-point atomics; not bit-reproducible).
 */
#ifndef MOE_NVFP4_H
#define MOE_NVFP4_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* bad shape, flag, null or misaligned pointer */
    MOE_ERR_UNSUPPORTED = 2,   /* valid request this build/device cannot run  */
    MOE_ERR_WORKSPACE = 3,     /* buffer smaller than the *_bytes() query     */
    MOE_ERR_CUDA = 4,          /* a CUDA runtime call failed                  */
    MOE_ERR_TIMEOUT = 5        /* a device-side wait gave up (see status word)*/
} moe_status;

/* ---- flags (one uint32_t) ------------------------------------------------ */
/* bits 0-1: activation of FC1 */
#define MOE_ACT_SWIGLU 0u            /* h = silu(gate) * up, W1 = [gate; up] */
#define MOE_ACT_RELU2 1u             /* h = max(z, 0)^2, non-gated          */
#define MOE_ACT_MASK 3u
/* bits 2-3: precision mode */
#define MOE_W4A4_PER_TENSOR (0u << 2) /* caller-supplied FP32 global scales   */
#define MOE_W4A4_PER_TOKEN (1u << 2)  /* per-row amax/2688 global scales      */
#define MOE_W4A16 (2u << 2)           /* BF16 activations, NVFP4 weights      */
/* MXFP8 W8A8 [MegaMoE, "Our approach": 8-bit weights and activations with
 * block-32 scaling]: E4M3 elements, one E8M0 (power-of-two) scale per 32
 * elements along K, 2^(floor(log2 amax) - 8); no global scales (the
 * act_scale arguments must be NULL).  Weights are prepared in this format. */
#define MOE_W8A8_MXFP8 (3u << 2)
#define MOE_MODE_MASK (3u << 2)
/* bit 4: router weight applied to the FC2 input (after the activation,
 * before the FC2-input quantization or BF16 store) instead of at the output
 * reduction (default) [PR #4366, "Motivation"]. */
#define MOE_ROUTER_W_ON_INPUT (1u << 4)
/* bit 5: deterministic two-stage finalize (FC2 stores per-route rows, a
 * fixed-order reduction kernel sums them) instead of the fused FC2-epilogue
 * scatter (default). */
#define MOE_FINALIZE_DETERMINISTIC (1u << 5)
/* bit 6: router weights are the full softmax over all E experts evaluated
 * at the selected ones, instead of the softmax over the K selected. */
#define MOE_ROUTE_NO_RENORM (1u << 6)
/* bits 7-8: GEMM tile scheduling (W4A4 NVFP4 and W4A16; ignored by MXFP8;
 * results are the same either way up to FP32 accumulation order).  A GEMM
 * whose weight height is a multiple of 256 runs on CTA pairs (cta_group::2
 * MMAs, 256 x 256 tiles over two 128-row M tiles of one expert) when the
 * experts holding routes hold at least 256 on average (T*K >= 256 *
 * min(E, T*K)), else on single CTAs; MOE_GEMM_PAIRS_ALWAYS /
 * MOE_GEMM_PAIRS_NEVER force pairs / single CTAs.  Setting both is
 * invalid. */
#define MOE_GEMM_PAIRS_NEVER (1u << 7)
#define MOE_GEMM_PAIRS_ALWAYS (1u << 8)
/* bit 9: 4-over-6 activation quantization (per-token W4A4 only) [PR #4366
 * post, "Performance benchmark": the per-token activation contract runs with
 * NVFP4_4OVER6, NVFP4_4OVER6_E4M3_USE_256 and NVFP4_4OVER6_ERR_MODE=MSE].
 * Every 16-element block of x and of the FC2 input is quantized with its
 * maximum mapped to 6 and to 4; the candidate with the smaller float32
 * squared dequantization error is kept (ties keep 6).  Per-row global
 * scales become amax/1536 (6 * 256).  The decode, and so the GEMMs, are
 * unchanged. */
#define MOE_QUANT_4OVER6 (1u << 9)
/* bit 10: the whole forward as one persistent kernel (one CTA per SM,
 * cooperative launch) [MegaMoE, "Our approach": a single persistent kernel
 * per forward pass runs the quantization, the grouped GEMMs and the
 * combine]: routing, permutation, x quantization, FC1, the FC2-input
 * quantization, FC2 and the finalize run as phases separated by grid-wide
 * barriers, with the same arithmetic as the default launch sequence (same
 * bits, up to the order of the fused finalize's FP32 additions).  Meant for
 * small T, where launch and ramp-up latency dominate.  W4A4 modes only
 * (per-tensor or per-token, optionally 4-over-6), E <= 256, 128-wide GEMM
 * tiles; invalid with MOE_GEMM_PAIRS_ALWAYS.  Needs every SM free for one
 * resident CTA (otherwise the launch fails: MOE_ERR_CUDA).  The staged entry
 * point records all eight events around the one kernel. */
#define MOE_FUSED_LAYER (1u << 10)
/* bits 11-12: GEMM operand orientation (W4A4 and W4A16 launch sequence;
 * results are the same either way up to FP32 accumulation order).  The
 * swapped orientation puts the expert's weights on the MMA's M side (W4A16:
 * widened to BF16 on chip) and 64 of its routes on the N side, so that
 * experts with few routes do not stream 128-row activation tiles that are
 * mostly padding.  Default: swapped when the mean number of routes per
 * expert holding any (T*K / min(E, T*K)) is at most 64 and T*K >= 64.
 * MOE_GEMM_SWAP_NEVER / _ALWAYS force a choice; setting both, or _ALWAYS
 * with MOE_GEMM_PAIRS_ALWAYS, MOE_FUSED_LAYER or MOE_W8A8_MXFP8, is
 * invalid. */
#define MOE_GEMM_SWAP_NEVER (1u << 11)
#define MOE_GEMM_SWAP_ALWAYS (1u << 12)
/* bit 13: test hook for the bounded waits.  The producer warp of the first
 * CTA of the FC1 GEMM skips its first pipeline stage: it issues neither that
 * stage's copies nor its barrier arrival, so no copy is ever in flight
 * against the barrier the MMA thread then waits on.  That wait gives up
 * after its limit (1 s), every role of the CTA drains and exits, the forward
 * returns MOE_OK and moe_nvfp4_last_device_status reports MOE_ERR_TIMEOUT;
 * y is undefined.  Valid only on the launch sequence with the standard GEMM
 * orientation: a W4A4 mode together with MOE_GEMM_SWAP_NEVER, without
 * MOE_GEMM_PAIRS_ALWAYS or MOE_FUSED_LAYER. */
#define MOE_DEBUG_FC1_SKIP_STAGE (1u << 13)
/* bit 14: the router logits are computed by the layer itself from the gate
 * projection, logits = x . W_g^T (moe_nvfp4_forward_gate; required by it,
 * invalid with every other forward entry point and with MOE_FUSED_LAYER).
 * The workspace then holds the FP32 logits [T][E]. */
#define MOE_ROUTER_GEMM (1u << 14)
#define MOE_FLAGS_KNOWN 0x7FFFu

/* ---- shapes ---------------------------------------------------------------- */
typedef struct {
    int T;  /* tokens, >= 1                                                  */
    int H;  /* hidden size, multiple of 128                                  */
    int I;  /* per-expert intermediate size, multiple of 128                 */
    int E;  /* experts, 1..1024                                              */
    int K;  /* experts per token (top-K), 1..min(E, 32)                      */
} moe_shape;

/* ---- weight preparation ------------------------------------------------------ */
/* Size in bytes of the prepared-weight buffer for this shape, activation and
 * weight format (only the activation bits and whether the precision mode is
 * MOE_W8A8_MXFP8 matter).  0 if the shape is invalid. */
MOE_API size_t moe_nvfp4_prepared_bytes(moe_shape s, uint32_t flags);

/* Quantize BF16 checkpoint weights to NVFP4 (or, with MOE_W8A8_MXFP8, to
 * MXFP8) and reorder them into the prepared layout consumed by
 * moe_nvfp4_forward ["MegaMoE", "Usage": weights accepted in checkpoint
 * layout, quantized and reordered by the layer; PR #5319 post: W4A4 and
 * W4A16 share the NVFP4 layout].
 *   w1_bf16  [E][N1][H] row-major, N1 = 2I for SwiGLU (rows 0..I-1 gate,
 *            I..2I-1 up), N1 = I for ReLU2.  16-byte aligned.
 *   w2_bf16  [E][H][I] row-major.  16-byte aligned.
 *   prepared output, `prepared_bytes` >= moe_nvfp4_prepared_bytes(); 256-byte
 *            aligned.  Per expert and matrix: global scale amax/2688 (1 if the
 *            matrix is zero), E4M3 scale per 16 elements along the reduction
 *            dimension, E2M1 codes.  Layout (versioned, MOE_PREPARED_VERSION):
 *              Gw1[E] f32 | Gw2[E] f32 | W1 codes [E][N1][H/2] |
 *              W1 scales [E][N1/128][H/64][512] | W2 codes [E][H][I/2] |
 *              W2 scales [E][H/128][I/64][512]
 *            each region 256-byte aligned.  W1 rows are reordered for SwiGLU
 *            so that every 128-row tile holds 64 gate rows then the 64
 *            matching up rows.  A 512-byte scale atom holds 128 rows x 4
 *            scales: byte (r%32)*16 + (r/32)*4 + j for row r, scale j.
 *            MXFP8: Gw1 = Gw2 = 1, codes are E4M3 bytes ([E][N1][H],
 *            [E][H][I]) and the scales E8M0 per 32 elements in the same atom
 *            layout over 128 elements of K ([E][N1/128][H/128][512],
 *            [E][H/128][I/128][512]).
 * Errors: MOE_ERR_INVALID_ARG (shape, flags, null/misaligned pointer),
 * MOE_ERR_WORKSPACE (prepared_bytes too small), MOE_ERR_CUDA.  Enqueues two
 * kernels on `stream`; the input buffers must stay valid until they finish. */
MOE_API moe_status moe_nvfp4_prepare_weights(moe_shape s, uint32_t flags,
                                     const void* w1_bf16, const void* w2_bf16,
                                     void* prepared, size_t prepared_bytes,
                                     void* stream);

#define MOE_PREPARED_VERSION 1

/* ---- forward ------------------------------------------------------------------- */
/* Size in bytes of the workspace moe_nvfp4_forward needs.  0 if invalid. */
MOE_API size_t moe_nvfp4_workspace_bytes(moe_shape s, uint32_t flags);

/* The layer forward, y = MoE(x).
 *   x_bf16        [T][H] BF16, 16-byte aligned.
 *   router_logits [T][E] FP32 (finite), 16-byte aligned.
 *   router_bias   [E] FP32 added to the logits before selection, or NULL.
 *   act_scale_fc1 per-tensor W4A4: device FP32[1], the FC1-input global scale
 *                 G1 (> 0, decode direction: x ~ q * s * G1); else NULL.
 *   act_scale_fc2 per-tensor W4A4: device FP32[1], FC2-input scale G2 (> 0);
 *                 else NULL.
 *   prepared      output of moe_nvfp4_prepare_weights for the same shape
 *                 and activation.
 *   workspace     >= moe_nvfp4_workspace_bytes(), 256-byte aligned; holds
 *                 the intermediates (layout: moe_nvfp4_workspace_layout).
 *   y_bf16        [T][H] BF16 output, overwritten; 16-byte aligned; must not
 *                 alias any input.
 * Selection: the K largest logit+bias, ties to the lower expert index.
 * Bit-exact, on every device and at every size: expert ids, counts, offsets,
 * the permutation and the NVFP4 codes/scales of x.  Floating-point: router
 * weights (expf), FC outputs and y (tensor-core FP32 accumulation).
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_WORKSPACE, MOE_ERR_UNSUPPORTED (no
 * sm_103a/sm_100-family device), MOE_ERR_CUDA.  Nothing is synchronized. */
MOE_API moe_status moe_nvfp4_forward(moe_shape s, uint32_t flags,
                             const void* x_bf16, const float* router_logits,
                             const float* router_bias,
                             const float* act_scale_fc1, const float* act_scale_fc2,
                             const void* prepared,
                             void* workspace, size_t workspace_bytes,
                             void* y_bf16, void* stream);

/* The layer forward on caller-supplied routing instead of router logits
 * [FlashInfer PR #4366, "Motivation": the fused-MoE wrapper takes the top-K
 * expert ids and their final scales precomputed; "Existing SM120 status":
 * they must be device tensors of the right dtype and shape].
 *   topk_ids      [T][K] int32, device, 4-byte aligned: expert of slot k of
 *                 token t.  An id outside [0, E), or repeating the id of an
 *                 earlier kept slot of the same token, is a dropped route:
 *                 it gets no row and contributes nothing (like a route of
 *                 weight 0), and moe_nvfp4_last_device_status then reports
 *                 MOE_ERR_INVALID_ARG.
 *   topk_weights  [T][K] FP32, device, 4-byte aligned: used as given (no
 *                 softmax, no renormalization), at the output reduction or
 *                 on the FC2 input per MOE_ROUTER_W_ON_INPUT.
 * Every other argument, the workspace and its layout are those of
 * moe_nvfp4_forward; the workspace's topk_ids / topk_w regions receive the
 * ids (dropped routes as -1) and the weights.  MOE_ROUTE_NO_RENORM is
 * rejected (there is no router).  Neither routing array may overlap y or the
 * workspace.  Errors as moe_nvfp4_forward.  Nothing is synchronized. */
MOE_API moe_status moe_nvfp4_forward_routed(moe_shape s, uint32_t flags,
                                            const void* x_bf16, const int32_t* topk_ids,
                                            const float* topk_weights,
                                            const float* act_scale_fc1, const float* act_scale_fc2,
                                            const void* prepared,
                                            void* workspace, size_t workspace_bytes,
                                            void* y_bf16, void* stream);

/* Router logits from the gate projection on the tensor cores [FlashInfer
 * PR #4366, "Motivation": the MoE wrapper is handed routing that was computed
 * upstream from the gate projection; this is that projection]:
 *   logits[t][e] = sum_h x[t][h] * gate_w[e][h]
 *   x_bf16       [T][H] BF16, device, 16-byte aligned (H % 128 == 0)
 *   gate_w_bf16  [E][H] BF16, device, 16-byte aligned (1 <= E <= 1024)
 *   logits       [T][E] FP32, device, 16-byte aligned, caller-owned output;
 *                may not overlap x or gate_w.
 * BF16 products are exact; the sum is accumulated in FP32 by the tensor cores
 * (order unspecified), so it may differ from the exactly rounded sum by a few
 * FP32 roundings of partial sums.  Enqueues one kernel on `stream`; nothing is
 * synchronized; a timed-out internal wait leaves the output undefined and is
 * not reported (use moe_nvfp4_forward_gate for a status).
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA. */
MOE_API moe_status moe_nvfp4_router_logits(int T, int E, int H, const void* x_bf16,
                                           const void* gate_w_bf16, float* logits,
                                           void* stream);

/* The layer forward from the gate projection instead of router logits: the
 * logits kernel of moe_nvfp4_router_logits writes into the workspace's logits
 * region, then the forward of moe_nvfp4_forward runs on them (router bias,
 * softmax and top-K as there).  flags must include MOE_ROUTER_GEMM (which
 * sizes the workspace for the logits) and not MOE_FUSED_LAYER.  gate_w_bf16
 * [E][H] BF16, device, 16-byte aligned, not overlapping the workspace.  Every
 * other argument as moe_nvfp4_forward; the device status also reports a
 * timeout of the logits kernel.  Nothing is synchronized. */
MOE_API moe_status moe_nvfp4_forward_gate(moe_shape s, uint32_t flags,
                                          const void* x_bf16, const void* gate_w_bf16,
                                          const float* router_bias,
                                          const float* act_scale_fc1, const float* act_scale_fc2,
                                          const void* prepared,
                                          void* workspace, size_t workspace_bytes,
                                          void* y_bf16, void* stream);

/* Same as moe_nvfp4_forward, and records caller-created CUDA events
 * (cudaEvent_t, created with timing enabled) on `stream` at the stage
 * boundaries, for per-stage timing:
 *   events[0] before the router, [1] after the router, [2] after the
 *   permutation (recorded right after [1] when T <= 32: one launch does
 *   both), [3] after the activation quantization (W4A4) or gather
 *   (W4A16), [4] after FC1, [5] after the FC2-input quantization (recorded
 *   right after [4] when the mode has none), [6] after FC2, [7] after the
 *   finalize.  MOE_NUM_STAGE_EVENTS events, none NULL.
 * The recordings serialize the stages (no programmatic dependent launch),
 * so the sum of the stages can exceed the plain forward's time. */
#define MOE_NUM_STAGE_EVENTS 8
MOE_API moe_status moe_nvfp4_forward_staged(moe_shape s, uint32_t flags,
                                            const void* x_bf16, const float* router_logits,
                                            const float* router_bias,
                                            const float* act_scale_fc1, const float* act_scale_fc2,
                                            const void* prepared,
                                            void* workspace, size_t workspace_bytes,
                                            void* y_bf16, void* stream, void* const* events);

/* Number of kernel launches one moe_nvfp4_forward enqueues for this shape
 * and flags (-1 if invalid): 6 (7 with per-token scales: the FC2-input
 * quantization), one fewer for T <= 32 (router and permutation scan in one
 * launch), 1 for MOE_FUSED_LAYER.  moe_nvfp4_forward_routed always launches
 * the scan separately.  Pure host call. */
MOE_API int moe_nvfp4_forward_launches(moe_shape s, uint32_t flags);

/* Byte offsets of the intermediates inside the workspace (for tests and
 * debugging; MOE_WORKSPACE_VERSION).  Each entry is 256-byte aligned.
 * rows_cap = the padded-row capacity (a multiple of 128).               */
typedef struct {
    uint64_t rows_cap;       /* padded-row capacity                          */
    uint64_t status;         /* uint32[4]: [0] error bits of the last run,   */
                             /*   [1] grid-barrier counter (fused layer)     */
    uint64_t topk_ids;       /* int32 [T][K]                                 */
    uint64_t topk_w;         /* f32   [T][K]                                 */
    uint64_t count;          /* int32 [E]   routes per expert                */
    uint64_t offsets;        /* int32 [E+1] exclusive prefix of count        */
    uint64_t padded_offsets; /* int32 [E+1] prefix of count rounded up to 128*/
    uint64_t meta;           /* int32 [4]: [0] padded rows, [1] M tiles,     */
                             /*   [2] M-tile pairs (tile_pair entries),      */
                             /*   [3] occupied halves (tile_half entries)    */
    uint64_t unit_base;      /* int32 [E][ceil(T/32)] per-unit starting rows */
    uint64_t unit_mask;      /* uint32 [E][ceil(T/32)] per-unit token masks  */
    uint64_t row_of_route;   /* int32 [T*K] padded row of route t*K+k        */
    uint64_t route_of_row;   /* int32 [rows_cap] route of a row, -1 in pads  */
    uint64_t tile_expert;    /* int32 [rows_cap/128] expert of each M tile   */
    uint64_t tile_pair;      /* int32 [rows_cap/128] M-tile pairs of one     */
                             /*   expert: (first tile << 1) | has_second     */
    uint64_t tile_half;      /* int32 [2*rows_cap/128] 64-row halves of M    */
                             /*   tiles holding routes: (M tile << 1) | half */
    uint64_t g1;             /* f32   [T] FC1-input global scale per token   */
    uint64_t xq_codes;       /* u8    [rows_cap][H/2] permuted x codes       */
    uint64_t xq_sf;          /* u8    [rows_cap/128][H/64][512] x scales     */
    uint64_t h_f32;          /* f32   [rows_cap][I] FC2 input before quant   */
    uint64_t g2;             /* f32   [rows_cap] FC2-input scale per row     */
    uint64_t hq_codes;       /* u8    [rows_cap][I/2] FC2-input codes        */
    uint64_t hq_sf;          /* u8    [rows_cap/128][I/64][512]              */
    uint64_t x_bf16_perm;    /* bf16  [rows_cap][H] permuted x (W4A16)       */
    uint64_t h_bf16;         /* bf16  [rows_cap][I] FC2 input (W4A16)        */
    uint64_t o_bf16;         /* bf16  [rows_cap][H] per-route FC2 output     */
    uint64_t y_acc;          /* f32   [T][H] fused-finalize accumulator      */
    uint64_t logits;         /* f32   [T][E] router logits (MOE_ROUTER_GEMM) */
    uint64_t total;          /* workspace bytes                              */
} moe_workspace_layout;

#define MOE_WORKSPACE_VERSION 6

/* Fill `out` with the workspace layout for this shape and flags.  Regions a
 * mode does not use have offset UINT64_MAX.  Pure host call, no CUDA. */
MOE_API moe_status moe_nvfp4_workspace_layout(moe_shape s, uint32_t flags,
                                      moe_workspace_layout* out);

/* Debug: wait for `stream`, then read and clear the device status word that
 * the most recent forward on `workspace` left (each forward clears it first).
 * Returns MOE_OK; MOE_ERR_TIMEOUT if a kernel's bounded wait (1 s) gave up
 * (for the fused layer also a grid barrier, or a CTA that stopped early);
 * MOE_ERR_INVALID_ARG if a kernel met an out-of-range expert id; or
 * MOE_ERR_CUDA.  Synchronizes `stream`. */
MOE_API moe_status moe_nvfp4_last_device_status(void* workspace, void* stream);

/* Test hook: convert n FP32 values with the library's device conversions,
 * E4M3 (round-to-nearest-even, saturating; one byte per value) and E2M1
 * (same rounding; the 4-bit code in the low nibble of one byte per value).
 * All pointers are device pointers.  Enqueues one kernel on `stream`. */
MOE_API moe_status moe_nvfp4_debug_convert(const float* in, int64_t n, uint8_t* e4m3,
                                   uint8_t* e2m1, void* stream);

/* ---- routing without any caller-allocated scratch ------------------------- */
/* No counterpart on the pages: this entry point exists for callers that
 * cannot allocate device memory (for example code running inside another
 * engine's fixed memory budget, or a latency-critical loop that must not
 * call cudaMalloc), yet need the routing stage on its own.
 *
 * Runs the router (softmax + top-K, selection and weights as in
 * moe_nvfp4_forward) and the stable permutation by expert, writing only
 * into the caller's output buffers (device pointers, 4-byte aligned):
 *   topk_ids [T*K] int32, topk_w [T*K] f32, count [E], offsets [E+1],
 *   padded_offsets [E+1] (prefix of the counts rounded up to 128),
 *   row_of_route [T*K] (padded row of route t*K+k),
 *   route_of_row [rows_cap] with rows_cap = round_up(T*K + min(E, T*K)*127,
 *   128) (the workspace layout's rows_cap); entries [0, padded_offsets[E])
 *   are written (-1 in pad rows), the rest are left untouched.
 * flags: 0 or MOE_ROUTE_NO_RENORM.  Results are bit-identical to the routing
 * intermediates moe_nvfp4_forward leaves in its workspace.
 *
 * Scratch: a fixed MOE_NOALLOC_SCRATCH_BYTES array in device memory, part of
 * the library image, which every GPU that loads the library holds until the
 * process exits.  It allocates nothing (no cudaMalloc/cudaFree, no
 * allocating library call).  Shapes whose scratch need (8 + rows_cap/128 +
 * 2*E*ceil(T/32) int32, plus alignment) exceeds the array return
 * MOE_ERR_WORKSPACE before anything is launched; E = 256 fits up to about
 * 16 000 tokens.  All calls share the one array (it keeps the last call's
 * contents; every entry a call reads is written by that call first), so calls
 * whose work may overlap on the GPU (different streams, or other host
 * threads) race and must be serialized by the caller.  The first call on each
 * device looks up the array's device address (cudaGetSymbolAddress) and
 * prepares the kernels; make that first call before any stream capture (a
 * CUDA error during that look-up is returned and the look-up retried on the
 * next call).  There is no device status to read back: the status word of
 * the kernels lives in the shared array, and the router only produces ids in
 * [0, E), so the permutation's bad-id checks cannot trigger.
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_WORKSPACE, MOE_ERR_UNSUPPORTED,
 * MOE_ERR_CUDA.  Enqueues four kernels on `stream`; does not synchronize. */
#define MOE_NOALLOC_SCRATCH_BYTES (1 << 20)
MOE_API moe_status moe_nvfp4_route_noalloc(int T, int E, int K, uint32_t flags,
                                           const float* router_logits,
                                           const float* router_bias,
                                           int32_t* topk_ids, float* topk_w,
                                           int32_t* count, int32_t* offsets,
                                           int32_t* padded_offsets,
                                           int32_t* row_of_route,
                                           int32_t* route_of_row, void* stream);

/* Library version string, e.g. "moe_nvfp4 1.0 sm_103a". */
MOE_API const char* moe_nvfp4_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_NVFP4_H */
