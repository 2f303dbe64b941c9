// Kernel launchers (host side) used by the orchestrator in moe_api.cu.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// Launch helper: every launch goes through cudaLaunchKernelEx so that the
// programmatic-dependent-launch and cluster attributes can be set uniformly.
struct LaunchCtx {
    cudaStream_t stream = nullptr;
    bool pdl = false;
    int cluster = 1;   // CTAs per thread-block cluster (x)

    template <typename... KArgs, typename... Args>
    cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, Args... args) const {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = block;
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[2];
        unsigned n = 0;
        if (pdl) {
            attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[n].val.programmaticStreamSerializationAllowed = 1;
            ++n;
        }
        if (cluster > 1) {
            attr[n].id = cudaLaunchAttributeClusterDimension;
            attr[n].val.clusterDim.x = (unsigned)cluster;
            attr[n].val.clusterDim.y = 1;
            attr[n].val.clusterDim.z = 1;
            ++n;
        }
        cfg.attrs = attr;
        cfg.numAttrs = n;
        return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
    }
};

// routing.cu
cudaError_t setup_routing_kernels();
cudaError_t launch_router(const LaunchCtx& c, int T, int E, int K, const float* logits, const float* bias,
                          int renorm, int* ids, float* w, unsigned int* status_reset);
cudaError_t launch_route_count(const LaunchCtx& c, int T, int E, int K, const float* logits, const float* bias,
                               int renorm, int* ids, float* w, int* unit_cnt, uint32_t* unit_mask,
                               unsigned int* status_reset);
// Caller-supplied ids / weights in place of the router (fused with the unit
// masks); out-of-range or repeated ids become dropped routes (-1).
cudaError_t launch_route_given(const LaunchCtx& c, int T, int E, int K, const int* ids_in, const float* w_in,
                               int* ids, float* w, int* unit_cnt, uint32_t* unit_mask, unsigned int* status);
// T <= 32 (one unit of tokens): router, unit masks and the scan in one
// block (the outputs of launch_route_count + launch_permute_scan)
cudaError_t launch_route_scan_small(const LaunchCtx& c, int T, int E, int K, const float* logits, const float* bias,
                                    int renorm, int* ids, float* w, int* unit_base, uint32_t* unit_mask, int* count,
                                    int* offsets, int* padded_offsets, int* meta, int* tile_expert, int* tile_pair,
                                    int* tile_half, int* route_of_row, unsigned int* status_reset);
// tile_pair / tile_half may be null (then only meta[2] / meta[3] count them)
cudaError_t launch_permute_scan(const LaunchCtx& c, int T, int E, int* unit_base, int* count, int* offsets,
                                int* padded_offsets, int* meta, int* tile_expert, int* tile_pair, int* tile_half,
                                int* route_of_row);
cudaError_t launch_permute(const LaunchCtx& c, int T, int E, int K, const int* ids, int* unit_base,
                           uint32_t* unit_mask, int* count, int* offsets, int* padded_offsets, int* meta,
                           int* tile_expert, int* row_of_route, int* route_of_row, unsigned int* status);

// Where a row-parallel kernel hands out the permuted rows itself (step 3 of
// the permutation fused in): the routing intermediates it reads and writes.
struct RouteScatter {
    const int* topk_ids;        // [T*K]
    const int* unit_base;       // [E][U] starting rows
    const uint32_t* unit_mask;  // [E][U] token masks
    int E;
    int* row_of_route;          // [T*K] out
    int* route_of_row;          // [rows_cap] out (valid rows)
};

// rowops.cu
cudaError_t launch_quantize_x(const LaunchCtx& c, int T, int H, int K, const void* x, const float* g1_in,
                              int per_token, float* g1_out, const RouteScatter& rs, uint8_t* codes, uint8_t* sf,
                              float* y_acc_zero);
// MXFP8 mode: x quantized to E4M3 / E8M0 per 32 into the token's permuted rows
cudaError_t launch_quantize_x_mx(const LaunchCtx& c, int T, int H, int K, const void* x, const RouteScatter& rs,
                                 uint8_t* codes, uint8_t* sf, float* y_acc_zero);
cudaError_t launch_gather_x_bf16(const LaunchCtx& c, int T, int H, int K, const void* x, const RouteScatter& rs,
                                 void* x_perm, float* y_acc_zero);
// per_token (quantize_x): 0 caller's per-tensor scale, 1 per-token, 2 per-token
// with 4-over-6 blocks; four_six (quantize_h): 4-over-6 blocks
cudaError_t launch_quantize_h(const LaunchCtx& c, uint64_t rows_cap, int I, const int* meta,
                              const int* route_of_row, const float* h, float* g2, uint8_t* codes, uint8_t* sf,
                              int four_six);
cudaError_t launch_finalize_deterministic(const LaunchCtx& c, int T, int H, int K, const int* row_of_route,
                                          const float* topk_w, int weight_on_output, const void* o, void* y);
cudaError_t launch_finalize_fused(const LaunchCtx& c, int T, int H, const float* y_acc, void* y);
cudaError_t launch_prepare(cudaStream_t s, int E, int N1, int H, int I, int act, const void* w1, const void* w2,
                           uint8_t* prepared, uint64_t gw1, uint64_t gw2, uint64_t w1c, uint64_t w1s, uint64_t w2c,
                           uint64_t w2s);
cudaError_t launch_prepare_mx(cudaStream_t s, int E, int N1, int H, int I, int act, const void* w1, const void* w2,
                              uint8_t* prepared, uint64_t gw1, uint64_t gw2, uint64_t w1c, uint64_t w1s, uint64_t w2c,
                              uint64_t w2s);
cudaError_t launch_debug_convert(cudaStream_t s, const float* in, int64_t n, uint8_t* e4m3, uint8_t* e2m1);

// gemm_nvf4.cu — grouped block-scaled GEMMs on tcgen05
enum GemmEpilogue : int {
    kEpiFc1Quant = 0,   // FC1: activation, route weight, NVFP4 requant with per-tensor G2
    kEpiFc1F32 = 1,     // FC1: activation, route weight, FP32 store (per-token G2 later)
    kEpiFc2Store = 2,   // FC2: BF16 per-route rows (deterministic finalize)
    kEpiFc2Scatter = 3, // FC2: weighted FP32 atomic add into the token row (fused finalize)
    kEpiFc1Bf16 = 4,    // FC1 (W4A16): activation, route weight, BF16 store
    kEpiFc1Mx = 5       // FC1 (MXFP8): activation, route weight, MXFP8 requant (block 32)
};

struct GemmParams {
    // operands
    const uint8_t* sfa;          // A scales [rows_cap/128][kdim/64][512]
    const uint8_t* sfb;          // B scales [E][N/128][kdim/64][512]
    int kdim;                    // reduction length (elements)
    int chunk_maps;              // 1: tmA / tmB are 3-D chunk maps (rows of a multiple of 128 bytes)
    int n;                       // output columns per expert (B rows per expert)
    int n_slab;                  // > 0: walk the output width in slabs of n_slab N tiles (standard kernel)
    const int* meta;             // meta[1] = number of M tiles, meta[2] = M-tile pairs
    const int* tile_expert;      // expert of each M tile
    const int* tile_pair;        // (first M tile << 1) | has_second, per pair (pair kernel)
    const int* tile_half;        // (M tile << 1) | half, per occupied 64-row half (swapped GEMM; meta[3] entries)
    const int* route_of_row;     // route of each padded row, -1 in pad rows
    int num_experts;             // E (bounds check of tile_expert)
    unsigned int* status;
    // epilogue
    int act;                     // MOE_ACT_*
    int topk;                    // K
    const float* gw;             // per-expert weight global scale [E]
    const float* g_act;          // activation global scale: per-tensor [1] or per-token/row array
    int g_act_per_token;         // 0: g_act[0]; 1 (FC1): g_act[token]; 2 (FC2): g_act[row]
    const float* topk_w;         // [T*K] router weights
    int weight_on_input;         // FC1: multiply h by the route weight
    int weight_on_output;        // FC2 scatter: multiply o by the route weight
    const float* g2;             // FC1 quant: per-tensor FC2-input scale [1]
    int out_cols;                // width of the output row (I for FC1, H for FC2)
    uint8_t* out_codes;          // FC1 quant: [rows_cap][I/2] (MXFP8: [rows_cap][I])
    uint8_t* out_sf;             // FC1 quant: [rows_cap/128][I/64][512] (MXFP8: [..][I/128][512])
    float* out_f32;              // FC1 F32: [rows_cap][I]; FC2 scatter: y_acc [T][H]
                                 // (g_act == nullptr: no activation global scale, W4A16)
    __nv_bfloat16* out_bf16;     // FC2 store: [rows_cap][H]; FC1 BF16: [rows_cap][I]
    int debug_skip_first_stage;  // test hook: CTA 0's producer skips its first stage (standard GEMM)
};

cudaError_t setup_gemm_kernels();
cudaError_t setup_gemm_w4a16_kernels();
cudaError_t launch_gemm_w4a16(const LaunchCtx& c, int epilogue, const CUtensorMap& tmA, const CUtensorMap& tmBq,
                              const GemmParams& p, int num_sms);
// The same on CTA pairs (256 x 256 pair tiles over pairs of M tiles of one
// expert, p.tile_pair / meta[2]); needs n % 256 == 0, the same 128-row maps.
// setup sizes the persistent grid for `device`.
cudaError_t setup_gemm_w4a16_pair_kernels(int device, int num_sms);
cudaError_t launch_gemm_w4a16_pair(const LaunchCtx& c, int epilogue, const CUtensorMap& tmA,
                                   const CUtensorMap& tmBq, const GemmParams& p, int device);
// tile_n = gemm_nvf4_tile_n(kdim, n) (128 or 256); tmB's box must be tile_n rows high.
// kind 0: NVFP4 operands (kind::mxf4nvf4); 1: MXFP8 operands (kind::mxf8f6f4).
int gemm_nvf4_tile_n(int kdim, int n);
cudaError_t launch_gemm_nvf4(const LaunchCtx& c, int epilogue, const CUtensorMap& tmA, const CUtensorMap& tmB,
                             const GemmParams& p, int num_sms, int tile_n, int kind);
// gemm_nvf4_pair.cu — the same GEMMs on CTA pairs (256 x 256 pair tiles over
// pairs of M tiles of one expert); needs n % 256 == 0 and tmA / tmB boxes of
// 128 rows (2-D one-chunk maps, or 3-D chunk maps when p.chunk_maps).
// Epilogues kEpiFc1Quant / F32, kEpiFc2Store / Scatter.
// setup sizes the persistent grid for `device`.
cudaError_t setup_gemm_pair_kernels(int device, int num_sms);
int gemm_pair_chunks();           // 128-byte K chunks per pipeline stage (1: 2-D maps; 2: 3-D chunk maps)
int gemm_pair_grid(int device);   // CTAs of the persistent pair grid (0 before setup)
cudaError_t launch_gemm_nvf4_pair(const LaunchCtx& c, int epilogue, const CUtensorMap& tmA, const CUtensorMap& tmB,
                                  const GemmParams& p, int device);

// router_gemm.cu — logits = x . W_g^T on the tensor cores (BF16, FP32
// accumulate).  tmX: 2-D uint8 map over x [T][2H] bytes, box 128 B x 128
// rows; tmW: over W_g [E][2H] bytes, box 128 B x router_gemm_tile_n(E) rows.
// status may be null.
cudaError_t setup_router_gemm_kernel();
int router_gemm_tile_n(int E);
cudaError_t launch_router_gemm(const LaunchCtx& c, const CUtensorMap& tmX, const CUtensorMap& tmW, int T, int E,
                               int H, float* logits, unsigned int* status);

// gemm_swap.cu — the W4A4 GEMMs with the weights on the MMA's M side (128
// rows per operand, two operands per tile) and 64 routes on its N side, for
// experts with few routes.  tmW: 3-D map over the prepared weights
// (row bytes, 128 rows, blocks of 128 rows), box 128 B x 64 x 2; tmX: 2-D
// map over the activation codes, box 128 B x 64 rows.  gated: FC1 SwiGLU
// (needs n % 256 == 0).  Epilogues kEpiFc1Quant / kEpiFc1F32 / kEpiFc2Store /
// kEpiFc2Scatter.
cudaError_t setup_gemm_swap_kernels();
cudaError_t launch_gemm_swap(const LaunchCtx& c, int epilogue, bool gated, const CUtensorMap& tmW,
                             const CUtensorMap& tmX, const GemmParams& p, int num_sms);

// fused_layer.cu — the whole W4A4 forward as one cooperative persistent
// kernel (one CTA per SM); E <= kFusedMaxExperts.
constexpr int kFusedMaxExperts = 256;
struct FusedParams {
    int T, H, I, E, K;
    // routing input: router logits (+ bias) or, when ids_in is set, given ids / weights
    const float* logits;
    const float* bias;
    int renorm;
    const int* ids_in;
    const float* w_in;
    // routing and permutation (workspace)
    int* ids;
    float* topk_w;
    int* unit_base;
    uint32_t* unit_mask;
    int* count;
    int* offsets;
    int* padded_offsets;
    int* meta;
    int* tile_expert;
    int* tile_pair;
    int* tile_half;
    int* row_of_route;
    int* route_of_row;
    // activations
    const __nv_bfloat16* x;
    int per_token;               // per-token G1 / G2 (else the caller's per-tensor scales)
    const float* g1_in;          // per-tensor: the caller's FC1 input scale
    float* g1;                   // per-token: [T]
    uint8_t* xq_codes;
    uint8_t* xq_sf;
    float* h_f32;                // per-token: FC1 output before quantization
    float* g2;                   // per-token: [rows_cap]
    uint8_t* hq_codes;
    uint8_t* hq_sf;
    // output
    int det;                     // deterministic finalize (FC2 stores BF16 rows)
    int weight_on_output;
    float* y_acc;                // fused finalize: [T][H] FP32
    const __nv_bfloat16* o_bf16; // deterministic finalize: [rows_cap][H]
    __nv_bfloat16* y;
    GemmParams fc1, fc2;         // the two GEMMs (128-wide tiles)
    unsigned int* status;        // status word (zeroed before the launch)
    unsigned int* sync;          // grid-barrier counter (zeroed before the launch)
};
cudaError_t setup_fused_layer_kernel();
// cooperative launch of num_sms CTAs; four_six: 4-over-6 blocks (per-token mode)
cudaError_t launch_fused_layer(cudaStream_t stream, int num_sms, const CUtensorMap& tmA1, const CUtensorMap& tmB1,
                               const CUtensorMap& tmA2, const CUtensorMap& tmB2, const FusedParams& fp,
                               bool four_six);

}  // namespace moe
