/*
 * CPU oracle for the NVFP4 Mixture-of-Experts layer forward.
 * TEST INFRASTRUCTURE ONLY (see moe_oracle.h).  Plain loops, FP64
 * accumulation, bit-exact emulation of the NVFP4 encodings.
 * Build: g++ -O2 -std=c++17 -ffp-contract=off -fopenmp -fPIC -shared.
 */
#include "moe_oracle.h"

#include <omp.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>

/* ======================================================================
 * Number formats.
 *
 * NVFP4 stores each element as E2M1 (1 sign, 2 exponent, 1 mantissa bit,
 * magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}) with one E4M3 scale per 16
 * consecutive elements and an FP32 global scale [MegaMoE, "Our approach":
 * "4-bit weights and activations using block-16 scaling"].
 * E4M3 here is the "fn" variant: bias 7, no infinities, 0x7F/0xFF = NaN,
 * largest finite 448, subnormals m*2^-9.
 * Rounding is round-to-nearest-even with saturation to the largest finite
 * magnitude ("satfinite").  Zero keeps the sign of its input (-0 -> code 8
 * for E2M1, 0x80 for E4M3); the scales are never negative.
 * ==================================================================== */

uint8_t orc_f32_to_e4m3(float v) {
    if (std::isnan(v)) return 0x7F;
    const uint8_t sign = std::signbit(v) ? 0x80 : 0x00;
    const float a = std::fabs(v);
    if (a >= 448.0f) return sign | 0x7E;               /* saturate */
    int code;
    if (a < 0x1p-6f) {
        /* subnormal range, quantum 2^-9; a*512 is exact, 8 -> min normal */
        code = (int)std::nearbyint(a * 512.0f);
    } else {
        int e2;
        std::frexp(a, &e2);
        int E = e2 - 1;                                 /* a in [2^E, 2^(E+1)) */
        int m = (int)std::nearbyint((std::ldexp(a, -E) - 1.0f) * 8.0f);
        if (m == 8) { E += 1; m = 0; }
        code = ((E + 7) << 3) | m;
        if (code > 0x7E) code = 0x7E;
    }
    return (uint8_t)(sign | code);
}

float orc_e4m3_to_f32(uint8_t b) {
    const int E = (b >> 3) & 15, m = b & 7;
    float v;
    if (E == 15 && m == 7) v = NAN;
    else if (E == 0) v = std::ldexp((float)m, -9);
    else v = std::ldexp(1.0f + (float)m / 8.0f, E - 7);
    return (b & 0x80) ? -v : v;
}

uint8_t orc_f32_to_e2m1(float v) {
    if (std::isnan(v)) return 0x7;     /* outside the input contract */
    const uint8_t sign = std::signbit(v) ? 0x8 : 0x0;
    const float a = std::fabs(v);
    int code;
    if (a >= 6.0f) code = 7;
    else if (a < 1.0f) code = (int)std::nearbyint(a * 2.0f);                 /* 0, .5, 1 */
    else if (a < 2.0f) code = 2 + (int)std::nearbyint((a - 1.0f) * 2.0f);    /* 1, 1.5, 2 */
    else if (a < 4.0f) code = 4 + (int)std::nearbyint((a * 0.5f - 1.0f) * 2.0f); /* 2, 3, 4 */
    else code = 6 + (int)std::nearbyint((a * 0.25f - 1.0f) * 2.0f);           /* 4, 6 */
    if (code > 7) code = 7;
    return (uint8_t)(sign | code);
}

float orc_e2m1_to_f32(uint8_t c) {
    static const float mag[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
    const float v = mag[c & 7];
    return (c & 8) ? -v : v;
}

uint16_t orc_f32_to_bf16(float v) {
    uint32_t u;
    std::memcpy(&u, &v, 4);
    if (std::isnan(v)) return (uint16_t)((u >> 16) | 0x40);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

uint16_t orc_f64_to_bf16(double v) {
    if (std::isnan(v)) return 0x7FC0;
    const uint16_t sign = std::signbit(v) ? 0x8000 : 0;
    const double a = std::fabs(v);
    if (a == 0.0) return sign;
    if (std::isinf(a)) return sign | 0x7F80;
    int e2;
    std::frexp(a, &e2);
    const int E = e2 - 1;
    const int qexp = (E < -126) ? -133 : E - 7;        /* BF16 has 8 significant bits */
    const double r = std::ldexp(std::nearbyint(std::ldexp(a, -qexp)), qexp);
    if (r >= 0x1p128) return sign | 0x7F80;
    const float f = (float)r;                           /* exact */
    uint32_t u;
    std::memcpy(&u, &f, 4);
    return (uint16_t)(sign | (u >> 16));
}

double orc_bf16_to_f64(uint16_t b) {
    const uint32_t u = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return (double)f;
}

void orc_f32_to_e4m3_n(const float* v, uint8_t* out, int64_t n) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_e4m3(v[i]);
}

void orc_f32_to_e2m1_n(const float* v, uint8_t* out, int64_t n) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_e2m1(v[i]);
}

void orc_f64_to_bf16_n(const double* v, uint16_t* out, int64_t n) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f64_to_bf16(v[i]);
}

void orc_f32_to_bf16_n(const float* v, uint16_t* out, int64_t n) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_bf16(v[i]);
}

/* ======================================================================
 * NVFP4 quantization of one row (the activation boundary before FC1 and,
 * in W4A4, before FC2 [PR4366, "Motivation": W4A4 FC2-input quantization
 * boundary]; per-tensor or per-token global scale [PR5319, "Retrieval
 * answer"]).
 *
 * Reading (the pages fix no operation order; this fixed float32 sequence is
 * the one both sides follow):
 *   G   = caller's scale (per-tensor) or amax_row/2688 (per-token; 1 if 0),
 *         so that x ~= q * s * G and the largest element maps to 6*448;
 *   s_b = E4M3( (amax_b / G) / 6 )                       per 16-block
 *   inv = s_b == 0 ? 0 : 1 / (s_b * G)
 *   q_i = E2M1( x_i * inv )
 * every arithmetic step rounded to float32 nearest-even.
 * ==================================================================== */

float orc_row_global_scale(const float* x, int64_t n) {
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) amax = std::max(amax, std::fabs(x[i]));
    if (amax == 0.0f) return 1.0f;
    return amax / 2688.0f;
}

static void quant_row(const float* x, int64_t n, float G, uint8_t* codes, uint8_t* sf) {
    for (int64_t b = 0; b < n / 16; ++b) {
        const float* xb = x + 16 * b;
        float amax = 0.0f;
        for (int i = 0; i < 16; ++i) amax = std::max(amax, std::fabs(xb[i]));
        const float t = amax / G;
        const uint8_t s = orc_f32_to_e4m3(t / 6.0f);
        sf[b] = s;
        const float sv = orc_e4m3_to_f32(s);
        const float denom = sv * G;
        const float inv = (sv == 0.0f) ? 0.0f : 1.0f / denom;
        for (int i = 0; i < 16; i += 2) {
            const float p0 = xb[i] * inv;
            const float p1 = xb[i + 1] * inv;
            const uint8_t lo = orc_f32_to_e2m1(p0);
            const uint8_t hi = orc_f32_to_e2m1(p1);
            codes[8 * b + i / 2] = (uint8_t)(lo | (hi << 4));
        }
    }
}

void orc_quant_rows(const float* x, int64_t rows, int64_t n, const float* G,
                    uint8_t* codes, uint8_t* sf) {
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < rows; ++r)
        quant_row(x + r * n, n, G[r], codes + r * (n / 2), sf + r * (n / 16));
}

float orc_row_global_scale_div(const float* x, int64_t n, float div) {
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) amax = std::max(amax, std::fabs(x[i]));
    if (amax == 0.0f) return 1.0f;
    return amax / div;
}

/* ======================================================================
 * 4-over-6 block quantization [FlashInfer PR #4366 post, "Performance
 * benchmark": the per-token activation contract run with NVFP4_4OVER6,
 * NVFP4_4OVER6_E4M3_USE_256 and NVFP4_4OVER6_ERR_MODE=MSE; the page gives
 * only these switch names].  Reading: each 16-element block is quantized
 * twice with the procedure above, once scaling the block maximum to 6 (the
 * default) and once to 4 (scale amax/G/4), and keeps the candidate whose
 * squared dequantization error is smaller (ties keep 6).  The error is
 * computed in float32 with round-to-nearest-even at every step in a fixed
 * order: d_i = x_i - (v_i * s) * G, err = (((d_0^2 + d_1^2) + d_2^2) ...),
 * so that the choice is reproducible.  E4M3_USE_256: the per-row global
 * scale is amax / (6 * 256) = amax / 1536, which keeps the larger max-4
 * block scale (at most 384) inside the E4M3 range.
 * ==================================================================== */
static float block_candidate(const float* xb, float G, float t, float M, uint8_t* codes, uint8_t* s_out) {
    const uint8_t s = orc_f32_to_e4m3(t / M);
    const float sv = orc_e4m3_to_f32(s);
    const float inv = (sv == 0.0f) ? 0.0f : 1.0f / (sv * G);
    float err = 0.0f;
    for (int i = 0; i < 16; i += 2) {
        const uint8_t lo = orc_f32_to_e2m1(xb[i] * inv);
        const uint8_t hi = orc_f32_to_e2m1(xb[i + 1] * inv);
        codes[i / 2] = (uint8_t)(lo | (hi << 4));
        const float d0 = xb[i] - (orc_e2m1_to_f32(lo) * sv) * G;
        const float d1 = xb[i + 1] - (orc_e2m1_to_f32(hi) * sv) * G;
        err = err + d0 * d0;
        err = err + d1 * d1;
    }
    *s_out = s;
    return err;
}

static void quant_row_4over6(const float* x, int64_t n, float G, uint8_t* codes, uint8_t* sf) {
    for (int64_t b = 0; b < n / 16; ++b) {
        const float* xb = x + 16 * b;
        float amax = 0.0f;
        for (int i = 0; i < 16; ++i) amax = std::max(amax, std::fabs(xb[i]));
        const float t = amax / G;
        uint8_t c6[8], c4[8], s6, s4;
        const float e6 = block_candidate(xb, G, t, 6.0f, c6, &s6);
        const float e4 = block_candidate(xb, G, t, 4.0f, c4, &s4);
        const bool four = e4 < e6;
        for (int i = 0; i < 8; ++i) codes[8 * b + i] = four ? c4[i] : c6[i];
        sf[b] = four ? s4 : s6;
    }
}

void orc_quant_rows_4over6(const float* x, int64_t rows, int64_t n, const float* G,
                           uint8_t* codes, uint8_t* sf) {
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < rows; ++r)
        quant_row_4over6(x + r * n, n, G[r], codes + r * (n / 2), sf + r * (n / 16));
}

void orc_dequant_rows(const uint8_t* codes, const uint8_t* sf, int64_t rows,
                      int64_t n, double* out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t i = 0; i < n; ++i) {
            const uint8_t byte = codes[r * (n / 2) + i / 2];
            const uint8_t c = (i & 1) ? (byte >> 4) : (byte & 15);
            out[r * n + i] = (double)orc_e2m1_to_f32(c) * (double)orc_e4m3_to_f32(sf[r * (n / 16) + i / 16]);
        }
}

/* ======================================================================
 * Router: softmax over the expert logits and top-K selection
 * [MegaMoE, "The problem": each token is routed to a top-K subset of
 * experts].  Reading: the K experts with the largest l = logit + bias
 * (ties to the lower index; the order of l equals the order of the softmax
 * probabilities), slot k holding the k-th largest; weights are the softmax
 * over the K selected logits (renormalised top-K) or, with renorm == 0, the
 * full softmax over all E experts evaluated at the selected ones.
 * ==================================================================== */
void orc_router(int64_t T, int E, int K, const float* logits, const float* bias,
                int renorm, int32_t* ids, double* w) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        std::vector<float> l(E);
        std::vector<char> taken(E, 0);
        for (int e = 0; e < E; ++e)
            l[e] = bias ? (logits[t * E + e] + bias[e]) : logits[t * E + e];
        for (int k = 0; k < K; ++k) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e;
            }
            taken[best] = 1;
            ids[t * K + k] = best;
        }
        const double lmax = (double)l[ids[t * K]];
        double den = 0.0;
        if (renorm) {
            for (int k = 0; k < K; ++k) den += std::exp((double)l[ids[t * K + k]] - lmax);
        } else {
            for (int e = 0; e < E; ++e) den += std::exp((double)l[e] - lmax);
        }
        for (int k = 0; k < K; ++k)
            w[t * K + k] = std::exp((double)l[ids[t * K + k]] - lmax) / den;
    }
}

/* ======================================================================
 * Grouping: routes of each expert made contiguous for the grouped GEMM
 * (the "contiguous gather" grouped GEMM of FlashInfer PR #4366, "Outside
 * diff" file list), each expert segment padded to whole tiles [PR4366,
 * "Tests": finalize handles cluster padding and partial tiles].
 * Reading: stable counting sort (routes of an expert in ascending token
 * order), padding granularity `pad` rows.
 * ==================================================================== */
int64_t orc_group(int64_t T, int E, int K, const int32_t* ids, int pad,
                  int32_t* count, int32_t* offsets, int32_t* padded_offsets,
                  int32_t* row_of_route, int32_t* route_of_row, int64_t rows_cap) {
    for (int e = 0; e < E; ++e) count[e] = 0;
    for (int64_t r = 0; r < T * K; ++r) {
        if (ids[r] < 0) continue;          /* a dropped route has no row */
        if (ids[r] >= E) return -2;
        count[ids[r]] += 1;
    }
    offsets[0] = 0;
    padded_offsets[0] = 0;
    for (int e = 0; e < E; ++e) {
        offsets[e + 1] = offsets[e] + count[e];
        padded_offsets[e + 1] = padded_offsets[e] + (count[e] + pad - 1) / pad * pad;
    }
    const int64_t total = padded_offsets[E];
    if (total > rows_cap) return -1;
    for (int64_t r = 0; r < rows_cap; ++r) route_of_row[r] = -1;
    std::vector<int64_t> next(padded_offsets, padded_offsets + E);
    for (int64_t t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k) {
            const int e = ids[t * K + k];
            if (e < 0) {
                row_of_route[t * K + k] = -1;
                continue;
            }
            const int64_t row = next[e]++;
            row_of_route[t * K + k] = (int32_t)row;
            route_of_row[row] = (int32_t)(t * K + k);
        }
    return total;
}

/* ======================================================================
 * Weight preparation, canonical view [MegaMoE, "Usage": weights accepted in
 * checkpoint layout, quantized and reordered by the layer; PR5319: W4A4 and
 * W4A16 consume the same prepared NVFP4 layout].  Reading: one FP32 global
 * scale per expert matrix (FC1 gate and up share it), amax/2688; rows
 * quantized along the reduction dimension with the row procedure above.
 * ==================================================================== */
float orc_prepare_matrix(const uint16_t* w_bf16, int64_t N, int64_t Kd,
                         uint8_t* codes, uint8_t* sf) {
    const int64_t n = N * Kd;
    std::vector<float> wf(n);
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        wf[i] = (float)orc_bf16_to_f64(w_bf16[i]);
        amax = std::max(amax, std::fabs(wf[i]));
    }
    const float G = (amax == 0.0f) ? 1.0f : amax / 2688.0f;
    std::vector<float> g(N, G);
    orc_quant_rows(wf.data(), N, Kd, g.data(), codes, sf);
    return G;
}

/* ======================================================================
 * MXFP8 (W8A8, block 32) [MegaMoE, "Our approach": an MXFP8 (W8A8) backend
 * with 8-bit weights and activations and block-32 scaling].  The page names
 * the format only.  Reading: the OCP Microscaling definition with E4M3
 * elements and one E8M0 (power-of-two) scale per 32 consecutive elements
 * along the reduction dimension: X = 2^(floor(log2(amax)) - 8), 8 being the
 * exponent of the largest E4M3 normal (448 = 1.75 * 2^8); elements are
 * E4M3_RN_satfinite(v / X) (the scaling by a power of two is exact); an
 * all-zero block gets X = 2^-127 (code 0); the exponent is clamped to
 * [-127, 127] (E8M0 codes 0..254, 255 is NaN).  There is no global scale.
 * ==================================================================== */
int orc_mx_block_exp(float amax) {
    if (!(amax > 0.0f) || !std::isfinite(amax)) return -127;
    int ex = 0;
    std::frexp(amax, &ex);                 /* amax = m * 2^ex, m in [0.5, 1) */
    const int e = (ex - 1) - 8;
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}

void orc_quant_rows_mx(const float* x, int64_t rows, int64_t n, uint8_t* codes, uint8_t* sf) {
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < n / 32; ++b) {
            const float* xb = x + r * n + 32 * b;
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs(xb[i]));
            const int e = orc_mx_block_exp(amax);
            sf[r * (n / 32) + b] = (uint8_t)(e + 127);
            for (int i = 0; i < 32; ++i) codes[r * n + 32 * b + i] = orc_f32_to_e4m3(std::ldexp(xb[i], -e));
        }
    }
}

void orc_dequant_rows_mx(const uint8_t* codes, const uint8_t* sf, int64_t rows, int64_t n, double* out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t i = 0; i < n; ++i)
            out[r * n + i] = std::ldexp((double)orc_e4m3_to_f32(codes[r * n + i]), (int)sf[r * (n / 32) + i / 32] - 127);
}

void orc_prepare_matrix_mx(const uint16_t* w_bf16, int64_t N, int64_t Kd, uint8_t* codes, uint8_t* sf) {
    std::vector<float> wf(N * Kd);
    for (int64_t i = 0; i < N * Kd; ++i) wf[i] = (float)orc_bf16_to_f64(w_bf16[i]);
    orc_quant_rows_mx(wf.data(), N, Kd, codes, sf);
}

/* ======================================================================
 * Expert MLP.  FC1 (gate|up), activation, optional input-side router
 * weight applied after the activation [PR4366, "Motivation": the flag
 * scales the post-activation FC2 input and never the FC1 pre-activation],
 * FC2.  GEMMs are naive FP64 loops with ascending k.
 *   SwiGLU: h_j = silu(z_j) * z_{I+j}, silu(z) = z / (1 + exp(-z))
 *   ReLU2 : h_j = max(z_j, 0)^2          [PR4366, "Existing SM120 status"]
 * ==================================================================== */
void orc_fc1(const double* a, const double* alpha, int64_t rows, int64_t H,
             const double* w1, int64_t I, int act, const double* p, double* h) {
    const int64_t N1 = (act == 0) ? 2 * I : I;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < rows; ++r) {
        std::vector<double> z(N1);
        const double* ar = a + r * H;
        for (int64_t j = 0; j < N1; ++j) {
            const double* wj = w1 + j * H;
            double acc = 0.0;
            for (int64_t k = 0; k < H; ++k) acc += ar[k] * wj[k];
            z[j] = acc * alpha[r];
        }
        for (int64_t j = 0; j < I; ++j) {
            double v;
            if (act == 0) {
                const double g = z[j], u = z[I + j];
                v = g / (1.0 + std::exp(-g)) * u;
            } else {
                const double zz = z[j] > 0.0 ? z[j] : 0.0;
                v = zz * zz;
            }
            if (p) v *= p[r];
            h[r * I + j] = v;
        }
    }
}

void orc_fc2(const double* a, const double* alpha, int64_t rows, int64_t I,
             const double* w2, int64_t H, double* o) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < rows; ++r) {
        const double* ar = a + r * I;
        for (int64_t n = 0; n < H; ++n) {
            const double* wn = w2 + n * I;
            double acc = 0.0;
            for (int64_t k = 0; k < I; ++k) acc += ar[k] * wn[k];
            o[r * H + n] = acc * alpha[r];
        }
    }
}

/* Finalize: unpermute and weighted top-K reduction, k ascending
 * [PR5319, "Retrieval answer": fused or unfused (deterministic) finalize;
 * PR4366, "Motivation": sum_r p_r * W2_r(a_r), or sum_r W2_r(p_r * a_r) with
 * the finalize weight neutral when the weight was applied on the input]. */
void orc_finalize(int64_t n_tok, int K, int64_t H, const int64_t* o_index,
                  const double* wk, const double* o, double* y) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n_tok; ++t)
        for (int64_t n = 0; n < H; ++n) {
            double acc = 0.0;
            for (int k = 0; k < K; ++k) {
                const double wt = wk ? wk[t * K + k] : 1.0;
                acc += wt * o[o_index[t * K + k] * H + n];
            }
            y[t * H + n] = acc;
        }
}

static int g_default_threads = 0;

void orc_set_threads(int n) {
    if (g_default_threads == 0) g_default_threads = omp_get_max_threads();
    omp_set_num_threads(n >= 1 ? n : g_default_threads);
}

int orc_max_threads(void) { return omp_get_max_threads(); }
