/*
 * CPU oracle for the NVFP4 Mixture-of-Experts layer forward.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow, obviously correct
 * restatement of what the layer computes, used to check the CUDA library.
 * Only the test-suite, the smoke entry point and the benchmark's CPU
 * baseline may load it.  It shares no code with the CUDA library.
 *
 * Floating point: FP64 accumulation for GEMMs and reductions; the NVFP4
 * encodings are emulated bit-exactly with IEEE float32 round-to-nearest-even
 * steps in a fixed order (built with -ffp-contract=off, no fast-math).
 *
 * Sources (page title, section):
 *  [MegaMoE]  "MegaMoE" (flashinfer.ai blog): "The problem" (top-K routing),
 *             "Our approach" (NVFP4 W4A4 with block-16 scaling), "Usage"
 *             (weights accepted in checkpoint layout, quantized and reordered).
 *  [PR4366]   FlashInfer PR #4366 page: "Motivation" (router-weight
 *             placement algebra, post-activation placement, FC2-input
 *             quantization boundary), "Existing SM120 status" (pre-activation
 *             counter-example), "Tests" (finalize / padding matrix).
 *  [PR5319]   "Disaggregated deployments can assign precision by serving
 *             phase ..." (newruntime post): "Retrieval answer" (per-tensor or
 *             per-token W4A4, W4A16, fused vs unfused finalize).
 *
 * Readings of points the pages leave open are stated beside each function.
 * Every function here is pinned by tests/test_oracle_pins.py except where a
 * comment says "parity unpinned".
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- number formats -------------------------------------------------- */
uint8_t orc_f32_to_e4m3(float v);   /* RN-even, saturate to +-448, NaN->0x7F */
float   orc_e4m3_to_f32(uint8_t b);
uint8_t orc_f32_to_e2m1(float v);   /* RN-even, saturate to +-6, 4-bit code   */
float   orc_e2m1_to_f32(uint8_t c);
uint16_t orc_f64_to_bf16(double v); /* RN-even, single rounding               */
uint16_t orc_f32_to_bf16(float v);  /* RN-even                                */
double  orc_bf16_to_f64(uint16_t b);
void orc_f32_to_e4m3_n(const float* v, uint8_t* out, int64_t n);
void orc_f32_to_e2m1_n(const float* v, uint8_t* out, int64_t n);
void orc_f64_to_bf16_n(const double* v, uint16_t* out, int64_t n);
void orc_f32_to_bf16_n(const float* v, uint16_t* out, int64_t n);

/* ---- NVFP4 row quantization ------------------------------------------ */
/* Global (decode-direction) scale of one row: amax/2688, or 1 if amax==0. */
float orc_row_global_scale(const float* x, int64_t n);
/* Quantize `rows` rows of length n (n % 16 == 0) with per-row global scale
 * G[r]: codes [rows][n/2] (low nibble = even element), scales [rows][n/16]
 * (E4M3, row-major: the canonical view, not any kernel layout). */
void orc_quant_rows(const float* x, int64_t rows, int64_t n, const float* G,
                    uint8_t* codes, uint8_t* sf);
/* Decode q*s (without the global scale) into FP64, exact. */
/* 4-over-6: per 16-element block, the better (float32 squared error) of
 * scaling the block maximum to 6 or to 4; ties keep 6.  G as above. */
void orc_quant_rows_4over6(const float* x, int64_t rows, int64_t n, const float* G,
                           uint8_t* codes, uint8_t* sf);
/* amax / div (1 for an all-zero row). */
float orc_row_global_scale_div(const float* x, int64_t n, float div);
/* MXFP8 rows: E4M3 codes [rows][n], E8M0 scales [rows][n/32] (block 32;
 * scale 2^(floor(log2 amax) - 8), 2^-127 for an all-zero block). */
int orc_mx_block_exp(float amax);
void orc_quant_rows_mx(const float* x, int64_t rows, int64_t n, uint8_t* codes, uint8_t* sf);
void orc_dequant_rows_mx(const uint8_t* codes, const uint8_t* sf, int64_t rows, int64_t n, double* out);
void orc_prepare_matrix_mx(const uint16_t* w_bf16, int64_t N, int64_t Kd, uint8_t* codes, uint8_t* sf);
void orc_dequant_rows(const uint8_t* codes, const uint8_t* sf, int64_t rows,
                      int64_t n, double* out);

/* ---- router ----------------------------------------------------------- */
/* Softmax + top-K. Selection on l = logit + bias (float32 add), descending,
 * ties to the lower expert index. Weights in FP64: softmax over the K
 * selected (renorm != 0) or over all E experts (renorm == 0). */
void orc_router(int64_t T, int E, int K, const float* logits, const float* bias,
                int renorm, int32_t* ids, double* w);

/* ---- grouping (token permutation by expert) -------------------------- */
/* Stable counting sort of routes by expert; expert segments padded to a
 * multiple of `pad` rows.  route r = t*K + k.  row_of_route gives the padded
 * row; route_of_row (length rows_cap) gets -1 in pad rows and past the end.
 * A negative id is a dropped route: it has no row (row_of_route -1).
 * Returns the padded row total, -1 if it exceeds rows_cap, -2 if an id is
 * >= E. */
int64_t orc_group(int64_t T, int E, int K, const int32_t* ids, int pad,
                  int32_t* count, int32_t* offsets, int32_t* padded_offsets,
                  int32_t* row_of_route, int32_t* route_of_row, int64_t rows_cap);

/* ---- weight preparation (canonical view) ----------------------------- */
/* One expert matrix W [N][Kd] BF16 -> codes [N][Kd/2], sf [N][Kd/16],
 * global scale G = amax(W)/2688 (1 if zero).  Returns G. */
float orc_prepare_matrix(const uint16_t* w_bf16, int64_t N, int64_t Kd,
                         uint8_t* codes, uint8_t* sf);

/* ---- expert MLP steps -------------------------------------------------- */
/* FC1 + activation for `rows` rows of one expert.
 *  a      : [rows][H] FP64 activation operand (q*s for W4A4, BF16 value for
 *           W4A16, raw value in exact mode)
 *  alpha  : [rows] FP64 factor applied to the accumulator (G1_row * Gw1)
 *  w1     : [N1][H] FP64 weight operand (q*s, or raw in exact mode),
 *           checkpoint row order (SwiGLU: gate rows then up rows)
 *  p      : [rows] route weight applied after the activation, or NULL
 *  h      : [rows][I] FP64 output */
void orc_fc1(const double* a, const double* alpha, int64_t rows, int64_t H,
             const double* w1, int64_t I, int act, const double* p, double* h);
/* FC2: o[r][n] = (sum_k a[r][k] * w2[n][k]) * alpha[r]. */
void orc_fc2(const double* a, const double* alpha, int64_t rows, int64_t I,
             const double* w2, int64_t H, double* o);
/* Finalize for n_tok tokens: y[t] = sum_k wk[t][k] * o[o_index[t*K+k]]
 * (k ascending, FP64).  o_index maps each route to its row of o.
 * wk == NULL means weight 1 for every route (input-side placement). */
void orc_finalize(int64_t n_tok, int K, int64_t H, const int64_t* o_index,
                  const double* wk, const double* o, double* y);

/* Host threads of the parallel loops above (timing only: every result is
 * the same for any thread count).  n < 1 restores the default. */
void orc_set_threads(int n);
int  orc_max_threads(void);

#ifdef __cplusplus
}
#endif
#endif
