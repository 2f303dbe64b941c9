// Host side of libmoe_nvfp4.so: argument validation, workspace carving,
// tensor-map encoding and the launch sequence of the layer forward.  No
// host synchronization and no allocation on the forward path: the expert
// counts never leave the device (the GEMM tile schedulers read them).
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "../../include/moe_nvfp4.h"
#include "common.cuh"
#include "kernels.h"
#include "w4a16_swap.h"
#include "layout.h"

using namespace moe;

namespace {

struct DeviceState {
    bool ready = false;
    moe_status status = MOE_ERR_UNSUPPORTED;
    int sms = 0;
};

std::mutex g_mu;
DeviceState g_dev[64];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

moe_status device_state(int* sms, int* device = nullptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState& d = g_dev[dev];
    if (!d.ready) {
        d.ready = true;
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            d.status = MOE_ERR_CUDA;
        } else if (major != 10 || minor != 3) {
            d.status = MOE_ERR_UNSUPPORTED;  // the binary carries sm_103a code only
        } else if (setup_routing_kernels() != cudaSuccess || setup_gemm_kernels() != cudaSuccess ||
                   setup_gemm_w4a16_kernels() != cudaSuccess || setup_gemm_pair_kernels(dev, d.sms) != cudaSuccess ||
                   setup_gemm_w4a16_pair_kernels(dev, d.sms) != cudaSuccess ||
                   setup_fused_layer_kernel() != cudaSuccess || setup_gemm_swap_kernels() != cudaSuccess ||
                   setup_gemm_w4a16_swap_kernels() != cudaSuccess ||
                   setup_router_gemm_kernel() != cudaSuccess) {
            d.status = MOE_ERR_CUDA;
        } else {
            d.status = MOE_OK;
        }
        if (d.status == MOE_OK && g_encode == nullptr) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || fn == nullptr) {
                d.status = MOE_ERR_CUDA;
            } else {
                g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
            }
        }
    }
    *sms = d.sms;
    if (device) *device = dev;
    return d.status;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

moe_status validate_shape(moe_shape s, uint32_t flags) {
    if (flags & ~MOE_FLAGS_KNOWN) return MOE_ERR_INVALID_ARG;
    if ((flags & MOE_GEMM_PAIRS_NEVER) && (flags & MOE_GEMM_PAIRS_ALWAYS)) return MOE_ERR_INVALID_ARG;
    if ((flags & MOE_QUANT_4OVER6) && mode_of(flags) != kModePerToken) return MOE_ERR_INVALID_ARG;
    if ((flags & MOE_GEMM_SWAP_NEVER) && (flags & MOE_GEMM_SWAP_ALWAYS)) return MOE_ERR_INVALID_ARG;
    if ((flags & MOE_GEMM_SWAP_ALWAYS) &&
        (mode_of(flags) == kModeMxfp8 || (flags & (MOE_GEMM_PAIRS_ALWAYS | MOE_FUSED_LAYER))))
        return MOE_ERR_INVALID_ARG;
    if (flags & MOE_FUSED_LAYER) {
        // one persistent kernel: the NVFP4 activation modes, the router's
        // register layout (E <= 256) and single-CTA GEMM tiles
        const int m = mode_of(flags);
        if ((m != kModePerTensor && m != kModePerToken) || s.E > kFusedMaxExperts || (flags & MOE_GEMM_PAIRS_ALWAYS))
            return MOE_ERR_INVALID_ARG;
    }
    if ((flags & MOE_ROUTER_GEMM) && (flags & MOE_FUSED_LAYER)) return MOE_ERR_INVALID_ARG;
    if (flags & MOE_DEBUG_FC1_SKIP_STAGE) {
        const int m = mode_of(flags);
        if ((m != kModePerTensor && m != kModePerToken) || !(flags & MOE_GEMM_SWAP_NEVER) ||
            (flags & (MOE_GEMM_PAIRS_ALWAYS | MOE_FUSED_LAYER)))
            return MOE_ERR_INVALID_ARG;
    }
    if (act_of(flags) > 1) return MOE_ERR_INVALID_ARG;
    if (s.T < 1 || s.T > (1 << 22)) return MOE_ERR_INVALID_ARG;
    if (s.H < 128 || s.H % 128 != 0 || s.H > 65536) return MOE_ERR_INVALID_ARG;
    if (s.I < 128 || s.I % 128 != 0 || s.I > 65536) return MOE_ERR_INVALID_ARG;
    if (s.E < 1 || s.E > 1024) return MOE_ERR_INVALID_ARG;
    if (s.K < 1 || s.K > 32 || s.K > s.E) return MOE_ERR_INVALID_ARG;
    if ((int64_t)s.T * s.K > (1 << 26)) return MOE_ERR_INVALID_ARG;
    // every row count that reaches a TMA coordinate must stay below 2^31
    const uint64_t N1 = (uint64_t)n1_of(s.I, flags);
    if ((uint64_t)s.E * N1 >= (1ull << 31) || (uint64_t)s.E * (uint64_t)s.H >= (1ull << 31)) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

// 2-D uint8 tensor map over a row-major [rows][row_bytes] array with
// box_bytes x 128-row boxes.  128-byte boxes use the 128-byte swizzle (the
// canonical K-major UMMA operand layout); narrower boxes are unswizzled.
bool encode_operand_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t row_bytes,
                        uint32_t box_bytes = 128, uint32_t box_rows = 128) {
    const cuuint64_t dims[2] = {row_bytes, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_bytes, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                box_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3-D uint8 tensor map over a row-major [rows][row_bytes] array, row_bytes a
// multiple of 128: x = byte inside a 128-byte chunk, y = row, z = chunk.  A
// box of two chunks x box_rows rows lands in shared memory as two
// consecutive 128-byte-swizzled [box_rows][128 B] tiles (one TMA copy for
// what would otherwise be two).
bool encode_chunk_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t row_bytes, uint32_t box_rows) {
    const cuuint64_t dims[3] = {128, rows, row_bytes / 128};
    const cuuint64_t strides[2] = {row_bytes, 128};
    const cuuint32_t box[3] = {128, box_rows, 2};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3-D uint8 tensor map over prepared weight codes [rows][row_bytes] viewed
// as [rows/128 blocks][128 rows][row_bytes], box box_bytes x 64 rows x 2
// blocks (the swapped-orientation GEMMs' weight operands): 128-byte boxes
// with the 128-byte swizzle (NVFP4 operands), narrower ones unswizzled
// (W4A16 codes, widened by the converter warps).
bool encode_swap_weight_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t row_bytes,
                            uint32_t box_bytes = 128) {
    const cuuint64_t dims[3] = {row_bytes, 128, rows / 128};
    const cuuint64_t strides[2] = {row_bytes, 128 * row_bytes};
    const cuuint32_t box[3] = {box_bytes, 64, 2};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                box_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Run the W4A4 (and W4A16) GEMMs in the swapped orientation?  When asked to, or by
// default when the experts that hold routes hold at most 64 on average
// (their 128-row activation tiles would be half padding or more) and there
// are at least 64 routes in all.  With fewer (a decode step of one token,
// the 16-token tiny case) every CTA runs a single tile and the standard
// kernel's 256-wide tile has the shorter fixed latency (measured on GB300:
// T = 1 at the DSV3 shape 68.6 us standard vs 72.3 us swapped; T = 16
// 452.7 vs 440.8; the mid workload 77.8 vs 74.9; T = 4096: 128 routes per
// expert, standard).  W4A16 (H = 4096, I = 1536, E = 128, top-8): T = 16
// step 385 -> 273 us, T = 512 532 -> 389 us swapped.
constexpr uint64_t kSlabAccBytes = 48ull << 20;   // FC2 accumulator slice kept in L2 (of 129 MB)
constexpr int64_t kSwapMaxRoutesPerExpert = 64;
constexpr int64_t kSwapMinRoutes = 64;
bool use_swap_gemm(moe_shape s, uint32_t flags) {
    if (flags & MOE_GEMM_SWAP_ALWAYS) return true;
    if (flags & (MOE_GEMM_SWAP_NEVER | MOE_GEMM_PAIRS_ALWAYS)) return false;
    const int64_t routes = (int64_t)s.T * s.K;
    const int64_t busy = routes < s.E ? routes : s.E;
    return routes >= kSwapMinRoutes && routes <= kSwapMaxRoutesPerExpert * busy;
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Run a W4A4 GEMM with `n` weight rows per expert on CTA pairs?  Pair tiles
// cover 256 routes of one expert; by default they are used when the experts
// that hold routes hold at least 256 on average (measured on GB300, standard
// vs pairs: prefill T = 16384 step 4.12 vs 3.68 ms, DSV3 shape T = 8192 FC1
// 1094 vs 1025 us, 16 experts x 2048 routes FC1 442 vs 374 us; below that a
// pair's second M tile is mostly padding).  MOE_GEMM_PAIRS_ALWAYS / _NEVER
// force either.  The W4A16 GEMMs follow the same rule (measured on GB300 at
// H = 4096, I = 1536, E = 128, top-8: T = 4096 (256 routes per expert) FC1
// 650 -> 455 us and FC2 663 -> 486 us on pairs; T = 512 (32 per expert)
// 275 -> 329 and 262 -> 330 us when forced, i.e. slower).
constexpr int64_t kPairMinRoutesPerExpert = 256;
bool use_pair_gemm(moe_shape s, uint32_t flags, int n) {
    if (n % 256 != 0 || (flags & MOE_GEMM_PAIRS_NEVER)) return false;
    if (flags & MOE_GEMM_PAIRS_ALWAYS) return true;
    const int64_t routes = (int64_t)s.T * s.K;
    const int64_t busy = routes < s.E ? routes : s.E;
    return routes >= kPairMinRoutesPerExpert * busy;
}

}  // namespace

extern "C" {

const char* moe_nvfp4_version(void) { return "moe_nvfp4 1.5 sm_103a (prepared v1, workspace v6)"; }

size_t moe_nvfp4_prepared_bytes(moe_shape s, uint32_t flags) {
    if (validate_shape(s, flags) != MOE_OK) return 0;
    return (size_t)prepared_layout(s, flags).total;
}

size_t moe_nvfp4_workspace_bytes(moe_shape s, uint32_t flags) {
    if (validate_shape(s, flags) != MOE_OK) return 0;
    return (size_t)workspace_layout(s, flags).total;
}

moe_status moe_nvfp4_workspace_layout(moe_shape s, uint32_t flags, moe_workspace_layout* out) {
    if (!out) return MOE_ERR_INVALID_ARG;
    const moe_status st = validate_shape(s, flags);
    if (st != MOE_OK) return st;
    *out = workspace_layout(s, flags);
    return MOE_OK;
}

moe_status moe_nvfp4_prepare_weights(moe_shape s, uint32_t flags, const void* w1_bf16, const void* w2_bf16,
                                     void* prepared, size_t prepared_bytes, void* stream) {
    moe_status st = validate_shape(s, flags);
    if (st != MOE_OK) return st;
    if (!w1_bf16 || !w2_bf16 || !prepared) return MOE_ERR_INVALID_ARG;
    if (!aligned(w1_bf16, 16) || !aligned(w2_bf16, 16) || !aligned(prepared, 256)) return MOE_ERR_INVALID_ARG;
    const PreparedLayout L = prepared_layout(s, flags);
    if (prepared_bytes < L.total) return MOE_ERR_WORKSPACE;
    int sms = 0;
    st = device_state(&sms);
    if (st != MOE_OK) return st;
    const int N1 = n1_of(s.I, flags);
    auto prep = mode_of(flags) == kModeMxfp8 ? launch_prepare_mx : launch_prepare;
    return cuda_status(prep(static_cast<cudaStream_t>(stream), s.E, N1, s.H, s.I, act_of(flags), w1_bf16, w2_bf16,
                            static_cast<uint8_t*>(prepared), L.gw1, L.gw2, L.w1_codes, L.w1_sf, L.w2_codes,
                            L.w2_sf));
}

// Routing input of a forward: router logits (+ bias), or caller-supplied
// top-K ids and weights.
struct RoutingIn {
    const float* logits = nullptr;
    const float* bias = nullptr;
    const int32_t* ids = nullptr;
    const float* w = nullptr;
    bool status_cleared = false;   // an earlier kernel of this forward may have raised status bits
};

// MOE_FUSED_LAYER: every step in one cooperative persistent launch.  The
// operands and GemmParams are the default path's with 128-wide tiles.
static moe_status forward_fused(moe_shape s, uint32_t flags, const void* x_bf16, const RoutingIn& rin,
                                const float* act_scale_fc1, const float* act_scale_fc2, const PreparedLayout& P,
                                const uint8_t* pw, const moe_workspace_layout& W, uint8_t* ws, void* y_bf16,
                                int sms, cudaStream_t stream, void* const* events) {
    auto wsp = [&](uint64_t off) { return ws + off; };
    const bool per_token = mode_of(flags) == kModePerToken;
    const bool det = (flags & MOE_FINALIZE_DETERMINISTIC) != 0;
    const bool on_input = (flags & MOE_ROUTER_W_ON_INPUT) != 0;
    const int N1 = n1_of(s.I, flags);
    FusedParams f{};
    f.T = s.T; f.H = s.H; f.I = s.I; f.E = s.E; f.K = s.K;
    f.logits = rin.logits;
    f.bias = rin.bias;
    f.renorm = (flags & MOE_ROUTE_NO_RENORM) ? 0 : 1;
    f.ids_in = rin.ids;
    f.w_in = rin.w;
    f.ids = reinterpret_cast<int*>(wsp(W.topk_ids));
    f.topk_w = reinterpret_cast<float*>(wsp(W.topk_w));
    f.unit_base = reinterpret_cast<int*>(wsp(W.unit_base));
    f.unit_mask = reinterpret_cast<uint32_t*>(wsp(W.unit_mask));
    f.count = reinterpret_cast<int*>(wsp(W.count));
    f.offsets = reinterpret_cast<int*>(wsp(W.offsets));
    f.padded_offsets = reinterpret_cast<int*>(wsp(W.padded_offsets));
    f.meta = reinterpret_cast<int*>(wsp(W.meta));
    f.tile_expert = reinterpret_cast<int*>(wsp(W.tile_expert));
    f.tile_pair = reinterpret_cast<int*>(wsp(W.tile_pair));
    f.tile_half = reinterpret_cast<int*>(wsp(W.tile_half));
    f.row_of_route = reinterpret_cast<int*>(wsp(W.row_of_route));
    f.route_of_row = reinterpret_cast<int*>(wsp(W.route_of_row));
    f.x = static_cast<const __nv_bfloat16*>(x_bf16);
    f.per_token = per_token ? 1 : 0;
    f.g1_in = act_scale_fc1;
    f.g1 = reinterpret_cast<float*>(wsp(W.g1));
    f.xq_codes = wsp(W.xq_codes);
    f.xq_sf = wsp(W.xq_sf);
    f.h_f32 = per_token ? reinterpret_cast<float*>(wsp(W.h_f32)) : nullptr;
    f.g2 = per_token ? reinterpret_cast<float*>(wsp(W.g2)) : nullptr;
    f.hq_codes = wsp(W.hq_codes);
    f.hq_sf = wsp(W.hq_sf);
    f.det = det ? 1 : 0;
    f.weight_on_output = on_input ? 0 : 1;
    f.y_acc = det ? nullptr : reinterpret_cast<float*>(wsp(W.y_acc));
    f.o_bf16 = det ? reinterpret_cast<const __nv_bfloat16*>(wsp(W.o_bf16)) : nullptr;
    f.y = static_cast<__nv_bfloat16*>(y_bf16);
    unsigned int* status = reinterpret_cast<unsigned int*>(wsp(W.status));
    f.status = status;
    f.sync = status + 1;

    const uint64_t rbx = (uint64_t)s.H / 2, rbh = (uint64_t)s.I / 2;
    const bool ch1 = rbx % 128 == 0, ch2 = rbh % 128 == 0;
    CUtensorMap tmA1, tmB1, tmA2, tmB2;
    const bool ok1 = ch1 ? (encode_chunk_map(&tmA1, f.xq_codes, W.rows_cap, rbx, 128) &&
                            encode_chunk_map(&tmB1, pw + P.w1_codes, (uint64_t)s.E * N1, rbx, 128))
                         : (encode_operand_map(&tmA1, f.xq_codes, W.rows_cap, rbx) &&
                            encode_operand_map(&tmB1, pw + P.w1_codes, (uint64_t)s.E * N1, rbx));
    const bool ok2 = ch2 ? (encode_chunk_map(&tmA2, f.hq_codes, W.rows_cap, rbh, 128) &&
                            encode_chunk_map(&tmB2, pw + P.w2_codes, (uint64_t)s.E * s.H, rbh, 128))
                         : (encode_operand_map(&tmA2, f.hq_codes, W.rows_cap, rbh) &&
                            encode_operand_map(&tmB2, pw + P.w2_codes, (uint64_t)s.E * s.H, rbh));
    if (!ok1 || !ok2) return MOE_ERR_CUDA;

    GemmParams& a = f.fc1;
    a.sfa = f.xq_sf;
    a.sfb = pw + P.w1_sf;
    a.kdim = s.H;
    a.chunk_maps = ch1 ? 1 : 0;
    a.n = N1;
    a.meta = f.meta;
    a.tile_expert = f.tile_expert;
    a.tile_pair = f.tile_pair;
    a.route_of_row = f.route_of_row;
    a.num_experts = s.E;
    a.status = status;
    a.act = act_of(flags);
    a.topk = s.K;
    a.gw = reinterpret_cast<const float*>(pw + P.gw1);
    a.topk_w = f.topk_w;
    a.weight_on_input = on_input ? 1 : 0;
    a.out_cols = s.I;
    if (per_token) {
        a.g_act = f.g1;
        a.g_act_per_token = 1;
        a.out_f32 = f.h_f32;
    } else {
        a.g_act = act_scale_fc1;
        a.g2 = act_scale_fc2;
        a.out_codes = f.hq_codes;
        a.out_sf = f.hq_sf;
    }
    GemmParams& b = f.fc2;
    b.sfa = f.hq_sf;
    b.sfb = pw + P.w2_sf;
    b.kdim = s.I;
    b.chunk_maps = ch2 ? 1 : 0;
    b.n = s.H;
    b.meta = f.meta;
    b.tile_expert = f.tile_expert;
    b.tile_pair = f.tile_pair;
    b.route_of_row = f.route_of_row;
    b.num_experts = s.E;
    b.status = status;
    b.act = act_of(flags);
    b.topk = s.K;
    b.gw = reinterpret_cast<const float*>(pw + P.gw2);
    b.topk_w = f.topk_w;
    b.weight_on_output = on_input ? 0 : 1;
    b.out_cols = s.H;
    b.g_act = per_token ? f.g2 : act_scale_fc2;
    b.g_act_per_token = per_token ? 2 : 0;
    if (det) b.out_bf16 = reinterpret_cast<__nv_bfloat16*>(wsp(W.o_bf16));
    else b.out_f32 = f.y_acc;

    auto mark = [&](int i) -> bool {
        return events == nullptr || cudaEventRecord(static_cast<cudaEvent_t>(events[i]), stream) == cudaSuccess;
    };
    if (!mark(0)) return MOE_ERR_CUDA;
    // status word, grid-barrier counter and the unit masks (built by
    // atomicOr) start at zero; the masks follow the status word
    const uint64_t units = ((uint64_t)s.T + kUnitTokens - 1) / kUnitTokens;
    const size_t zero_bytes = (size_t)(W.unit_mask + 4 * (uint64_t)s.E * units - W.status);
    if (W.unit_mask < W.status || cudaMemsetAsync(status, 0, zero_bytes, stream) != cudaSuccess) return MOE_ERR_CUDA;
    if (launch_fused_layer(stream, sms, tmA1, tmB1, tmA2, tmB2, f, (flags & MOE_QUANT_4OVER6) != 0) != cudaSuccess)
        return MOE_ERR_CUDA;
    for (int i = 1; i < MOE_NUM_STAGE_EVENTS; ++i)
        if (!mark(i)) return MOE_ERR_CUDA;
    return MOE_OK;
}

static moe_status forward_impl(moe_shape s, uint32_t flags, const void* x_bf16, const RoutingIn& rin,
                               const float* act_scale_fc1, const float* act_scale_fc2, const void* prepared,
                               void* workspace, size_t workspace_bytes, void* y_bf16, void* stream,
                               void* const* events) {
    moe_status st = validate_shape(s, flags);
    if (st != MOE_OK) return st;
    const int mode = mode_of(flags);
    const bool given = rin.ids != nullptr;
    if (!x_bf16 || !prepared || !workspace || !y_bf16) return MOE_ERR_INVALID_ARG;
    if (!aligned(x_bf16, 16) || !aligned(y_bf16, 16) || !aligned(prepared, 256) || !aligned(workspace, 256))
        return MOE_ERR_INVALID_ARG;
    if (given) {
        // caller-supplied routing: no router, so its options do not apply
        if (!rin.w || !aligned(rin.ids, 4) || !aligned(rin.w, 4) || (flags & MOE_ROUTE_NO_RENORM))
            return MOE_ERR_INVALID_ARG;
    } else {
        if (!rin.logits || !aligned(rin.logits, 16)) return MOE_ERR_INVALID_ARG;
        if (rin.bias && !aligned(rin.bias, 4)) return MOE_ERR_INVALID_ARG;
    }
    if (mode == kModePerTensor) {
        if (!act_scale_fc1 || !act_scale_fc2 || !aligned(act_scale_fc1, 4) || !aligned(act_scale_fc2, 4))
            return MOE_ERR_INVALID_ARG;
    }
    if (mode == kModeMxfp8 && (act_scale_fc1 || act_scale_fc2)) return MOE_ERR_INVALID_ARG;   // no global scales
    const moe_workspace_layout W = workspace_layout(s, flags);
    if (workspace_bytes < W.total) return MOE_ERR_WORKSPACE;
    const size_t y_bytes = (size_t)s.T * s.H * 2;
    if (overlaps(y_bf16, y_bytes, workspace, W.total) || overlaps(y_bf16, y_bytes, x_bf16, y_bytes))
        return MOE_ERR_INVALID_ARG;
    if (!given && overlaps(y_bf16, y_bytes, rin.logits, (size_t)s.T * s.E * 4)) return MOE_ERR_INVALID_ARG;
    if (given && (overlaps(y_bf16, y_bytes, rin.ids, (size_t)s.T * s.K * 4) ||
                  overlaps(y_bf16, y_bytes, rin.w, (size_t)s.T * s.K * 4) ||
                  overlaps(workspace, W.total, rin.ids, (size_t)s.T * s.K * 4) ||
                  overlaps(workspace, W.total, rin.w, (size_t)s.T * s.K * 4)))
        return MOE_ERR_INVALID_ARG;

    int sms = 0, device = 0;
    st = device_state(&sms, &device);
    if (st != MOE_OK) return st;

    const PreparedLayout P = prepared_layout(s, flags);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const uint8_t* pw = static_cast<const uint8_t*>(prepared);
    auto wsp = [&](uint64_t off) { return ws + off; };
    unsigned int* status = reinterpret_cast<unsigned int*>(wsp(W.status));
    int* ids = reinterpret_cast<int*>(wsp(W.topk_ids));
    float* topk_w = reinterpret_cast<float*>(wsp(W.topk_w));
    int* meta = reinterpret_cast<int*>(wsp(W.meta));
    int* row_of_route = reinterpret_cast<int*>(wsp(W.row_of_route));
    int* route_of_row = reinterpret_cast<int*>(wsp(W.route_of_row));
    int* tile_expert = reinterpret_cast<int*>(wsp(W.tile_expert));
    const bool det = (flags & MOE_FINALIZE_DETERMINISTIC) != 0;
    const bool on_input = (flags & MOE_ROUTER_W_ON_INPUT) != 0;
    const int act = act_of(flags);
    const int N1 = n1_of(s.I, flags);
    float* y_acc = det ? nullptr : reinterpret_cast<float*>(wsp(W.y_acc));

    if (flags & MOE_FUSED_LAYER)
        return forward_fused(s, flags, x_bf16, rin, act_scale_fc1, act_scale_fc2, P, pw, W, ws, y_bf16, sms,
                             static_cast<cudaStream_t>(stream), events);

    // GEMM variants of the W4A4 / W8A8 modes (host decisions only)
    const bool mx = mode == kModeMxfp8;
    const bool per_token = mode == kModePerToken;
    const bool swap = mode != kModeW4A16 && !mx && use_swap_gemm(s, flags);
    const bool pair1 = mode != kModeW4A16 && !mx && !swap && use_pair_gemm(s, flags, N1),
               pair2 = mode != kModeW4A16 && !mx && !swap && use_pair_gemm(s, flags, s.H);
    const int tn1 = pair1 ? 128 : gemm_nvf4_tile_n(s.H, N1), tn2 = pair2 ? 128 : gemm_nvf4_tile_n(s.I, s.H);
    LaunchCtx c;
    c.stream = static_cast<cudaStream_t>(stream);
    c.pdl = events == nullptr;   // stage events between kernels would serialize them anyway
    cudaError_t e;
    auto mark = [&](int i) -> bool {
        return events == nullptr ||
               cudaEventRecord(static_cast<cudaEvent_t>(events[i]), c.stream) == cudaSuccess;
    };
    if (!mark(0)) return MOE_ERR_CUDA;

    if (given) {
        // the given-routing kernel reports bad ids in the status word, so the
        // word is cleared before it rather than by it
        if (cudaMemsetAsync(status, 0, 16, c.stream) != cudaSuccess) return MOE_ERR_CUDA;
        LaunchCtx c0 = c;
        c0.pdl = false;
        e = launch_route_given(c0, s.T, s.E, s.K, rin.ids, rin.w, ids, topk_w,
                               reinterpret_cast<int*>(wsp(W.unit_base)), reinterpret_cast<uint32_t*>(wsp(W.unit_mask)),
                               status);
    } else if (s.T <= kUnitTokens) {
        // one unit of tokens: router and scan in one block
        e = launch_route_scan_small(c, s.T, s.E, s.K, rin.logits, rin.bias, (flags & MOE_ROUTE_NO_RENORM) ? 0 : 1,
                                    ids, topk_w, reinterpret_cast<int*>(wsp(W.unit_base)),
                                    reinterpret_cast<uint32_t*>(wsp(W.unit_mask)), reinterpret_cast<int*>(wsp(W.count)),
                                    reinterpret_cast<int*>(wsp(W.offsets)), reinterpret_cast<int*>(wsp(W.padded_offsets)),
                                    meta, tile_expert, reinterpret_cast<int*>(wsp(W.tile_pair)),
                                    reinterpret_cast<int*>(wsp(W.tile_half)), route_of_row,
                                    rin.status_cleared ? nullptr : status);
    } else {
        e = launch_route_count(c, s.T, s.E, s.K, rin.logits, rin.bias, (flags & MOE_ROUTE_NO_RENORM) ? 0 : 1, ids,
                               topk_w, reinterpret_cast<int*>(wsp(W.unit_base)),
                               reinterpret_cast<uint32_t*>(wsp(W.unit_mask)), rin.status_cleared ? nullptr : status);
    }
    if (e != cudaSuccess || !mark(1)) return MOE_ERR_CUDA;
    if (given || s.T > kUnitTokens) {
        e = launch_permute_scan(c, s.T, s.E, reinterpret_cast<int*>(wsp(W.unit_base)),
                                reinterpret_cast<int*>(wsp(W.count)), reinterpret_cast<int*>(wsp(W.offsets)),
                                reinterpret_cast<int*>(wsp(W.padded_offsets)), meta, tile_expert,
                                reinterpret_cast<int*>(wsp(W.tile_pair)), reinterpret_cast<int*>(wsp(W.tile_half)),
                                route_of_row);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
    }
    if (!mark(2)) return MOE_ERR_CUDA;
    // the quantize / gather kernel hands out the permuted rows itself
    RouteScatter rs;
    rs.topk_ids = ids;
    rs.unit_base = reinterpret_cast<const int*>(wsp(W.unit_base));
    rs.unit_mask = reinterpret_cast<const uint32_t*>(wsp(W.unit_mask));
    rs.E = s.E;
    rs.row_of_route = row_of_route;
    rs.route_of_row = route_of_row;

    if (mode == kModeW4A16) {
        // ---- W4A16: BF16 activations, weights widened on chip ----
        __nv_bfloat16* x_perm = reinterpret_cast<__nv_bfloat16*>(wsp(W.x_bf16_perm));
        __nv_bfloat16* h_bf16 = reinterpret_cast<__nv_bfloat16*>(wsp(W.h_bf16));
        e = launch_gather_x_bf16(c, s.T, s.H, s.K, x_bf16, rs, x_perm, y_acc);
        if (e != cudaSuccess || !mark(3)) return MOE_ERR_CUDA;
        // few routes per expert: weights on the MMA's M side, 64-route halves on N
        const bool swap16 = use_swap_gemm(s, flags);
        CUtensorMap tA1, tB1, tA2, tB2;
        const bool maps_ok =
            swap16 ? (encode_operand_map(&tA1, x_perm, W.rows_cap, (uint64_t)s.H * 2, 128, 64) &&
                      encode_swap_weight_map(&tB1, pw + P.w1_codes, (uint64_t)s.E * N1, (uint64_t)s.H / 2, 64) &&
                      encode_operand_map(&tA2, h_bf16, W.rows_cap, (uint64_t)s.I * 2, 128, 64) &&
                      encode_swap_weight_map(&tB2, pw + P.w2_codes, (uint64_t)s.E * s.H, (uint64_t)s.I / 2, 64))
                   : (encode_operand_map(&tA1, x_perm, W.rows_cap, (uint64_t)s.H * 2) &&
                      encode_operand_map(&tB1, pw + P.w1_codes, (uint64_t)s.E * N1, (uint64_t)s.H / 2, 32) &&
                      encode_operand_map(&tA2, h_bf16, W.rows_cap, (uint64_t)s.I * 2) &&
                      encode_operand_map(&tB2, pw + P.w2_codes, (uint64_t)s.E * s.H, (uint64_t)s.I / 2, 32));
        if (!maps_ok) return MOE_ERR_CUDA;
        int* tile_half16 = reinterpret_cast<int*>(wsp(W.tile_half));
        GemmParams a{};
        a.sfb = pw + P.w1_sf;
        a.kdim = s.H;
        a.n = N1;
        a.meta = meta;
        a.tile_expert = tile_expert;
        a.route_of_row = route_of_row;
        a.num_experts = s.E;
        a.status = status;
        a.act = act;
        a.topk = s.K;
        a.gw = reinterpret_cast<const float*>(pw + P.gw1);
        a.topk_w = topk_w;
        a.weight_on_input = on_input ? 1 : 0;
        a.out_cols = s.I;
        a.out_bf16 = h_bf16;
        a.tile_pair = reinterpret_cast<int*>(wsp(W.tile_pair));
        a.tile_half = tile_half16;
        e = swap16 ? launch_gemm_w4a16_swap(c, kEpiFc1Bf16, act == MOE_ACT_SWIGLU, tB1, tA1, a, sms)
            : use_pair_gemm(s, flags, N1) ? launch_gemm_w4a16_pair(c, kEpiFc1Bf16, tA1, tB1, a, device)
                                          : launch_gemm_w4a16(c, kEpiFc1Bf16, tA1, tB1, a, sms);
        if (e != cudaSuccess || !mark(4) || !mark(5)) return MOE_ERR_CUDA;
        GemmParams b{};
        b.sfb = pw + P.w2_sf;
        b.kdim = s.I;
        b.n = s.H;
        b.meta = meta;
        b.tile_expert = tile_expert;
        b.route_of_row = route_of_row;
        b.num_experts = s.E;
        b.status = status;
        b.act = act;
        b.topk = s.K;
        b.gw = reinterpret_cast<const float*>(pw + P.gw2);
        b.topk_w = topk_w;
        b.weight_on_output = on_input ? 0 : 1;
        b.out_cols = s.H;
        int epi2;
        if (det) {
            b.out_bf16 = reinterpret_cast<__nv_bfloat16*>(wsp(W.o_bf16));
            epi2 = kEpiFc2Store;
        } else {
            b.out_f32 = y_acc;
            epi2 = kEpiFc2Scatter;
        }
        b.tile_pair = reinterpret_cast<int*>(wsp(W.tile_pair));
        b.tile_half = tile_half16;
        e = swap16 ? launch_gemm_w4a16_swap(c, epi2, false, tB2, tA2, b, sms)
            : use_pair_gemm(s, flags, s.H) ? launch_gemm_w4a16_pair(c, epi2, tA2, tB2, b, device)
                                           : launch_gemm_w4a16(c, epi2, tA2, tB2, b, sms);
        if (e != cudaSuccess || !mark(6)) return MOE_ERR_CUDA;
        if (det)
            e = launch_finalize_deterministic(c, s.T, s.H, s.K, row_of_route, topk_w, on_input ? 0 : 1,
                                              wsp(W.o_bf16), y_bf16);
        else
            e = launch_finalize_fused(c, s.T, s.H, y_acc, y_bf16);
        if (e != cudaSuccess || !mark(7)) return MOE_ERR_CUDA;
        return MOE_OK;
    }

    // ---- W4A4 (NVFP4) and W8A8 (MXFP8) ----
    float* g1 = mx ? nullptr : reinterpret_cast<float*>(wsp(W.g1));
    uint8_t* xq_codes = wsp(W.xq_codes);
    uint8_t* xq_sf = wsp(W.xq_sf);
    uint8_t* hq_codes = wsp(W.hq_codes);
    uint8_t* hq_sf = wsp(W.hq_sf);
    const bool four_six = (flags & MOE_QUANT_4OVER6) != 0;
    if (mx)
        e = launch_quantize_x_mx(c, s.T, s.H, s.K, x_bf16, rs, xq_codes, xq_sf, y_acc);
    else
        e = launch_quantize_x(c, s.T, s.H, s.K, x_bf16, act_scale_fc1, per_token ? (four_six ? 2 : 1) : 0, g1, rs,
                              xq_codes, xq_sf, y_acc);
    if (e != cudaSuccess || !mark(3)) return MOE_ERR_CUDA;

    // operand rows: NVFP4 half a byte per element, MXFP8 a byte
    const uint64_t rbx = mx ? (uint64_t)s.H : (uint64_t)s.H / 2, rbh = mx ? (uint64_t)s.I : (uint64_t)s.I / 2;
    // single-CTA GEMMs with 128-wide tiles over rows of a multiple of 128
    // bytes copy two chunks per TMA instruction (3-D maps); the others use
    // 2-D maps
    const bool pch = gemm_pair_chunks() > 1;   // pair kernel with multi-chunk stages (3-D maps)
    const bool ch1 = pair1 ? (pch && rbx % 128 == 0) : (tn1 == 128 && rbx % 128 == 0);
    const bool ch2 = pair2 ? (pch && rbh % 128 == 0) : (tn2 == 128 && rbh % 128 == 0);
    CUtensorMap tmA1, tmB1, tmA2, tmB2;
    const bool ok1 = swap ? (encode_operand_map(&tmA1, xq_codes, W.rows_cap, rbx, 128, 64) &&
                             encode_swap_weight_map(&tmB1, pw + P.w1_codes, (uint64_t)s.E * N1, rbx))
                   : ch1 ? (encode_chunk_map(&tmA1, xq_codes, W.rows_cap, rbx, 128) &&
                            encode_chunk_map(&tmB1, pw + P.w1_codes, (uint64_t)s.E * N1, rbx, tn1))
                         : (encode_operand_map(&tmA1, xq_codes, W.rows_cap, rbx) &&
                            encode_operand_map(&tmB1, pw + P.w1_codes, (uint64_t)s.E * N1, rbx, 128, tn1));
    const bool ok2 = swap ? (encode_operand_map(&tmA2, hq_codes, W.rows_cap, rbh, 128, 64) &&
                             encode_swap_weight_map(&tmB2, pw + P.w2_codes, (uint64_t)s.E * s.H, rbh))
                   : ch2 ? (encode_chunk_map(&tmA2, hq_codes, W.rows_cap, rbh, 128) &&
                            encode_chunk_map(&tmB2, pw + P.w2_codes, (uint64_t)s.E * s.H, rbh, tn2))
                         : (encode_operand_map(&tmA2, hq_codes, W.rows_cap, rbh) &&
                            encode_operand_map(&tmB2, pw + P.w2_codes, (uint64_t)s.E * s.H, rbh, 128, tn2));
    if (!ok1 || !ok2) return MOE_ERR_CUDA;
    int* tile_pair = reinterpret_cast<int*>(wsp(W.tile_pair));
    int* tile_half = reinterpret_cast<int*>(wsp(W.tile_half));

    GemmParams g1p{};
    g1p.sfa = xq_sf;
    g1p.sfb = pw + P.w1_sf;
    g1p.kdim = s.H;
    g1p.chunk_maps = ch1 ? 1 : 0;
    g1p.n = N1;
    g1p.meta = meta;
    g1p.tile_expert = tile_expert;
    g1p.tile_pair = tile_pair;
    g1p.tile_half = tile_half;
    g1p.route_of_row = route_of_row;
    g1p.num_experts = s.E;
    g1p.status = status;
    g1p.act = act;
    g1p.topk = s.K;
    g1p.gw = reinterpret_cast<const float*>(pw + P.gw1);
    g1p.topk_w = topk_w;
    g1p.weight_on_input = on_input ? 1 : 0;
    g1p.out_cols = s.I;
    g1p.debug_skip_first_stage = (flags & MOE_DEBUG_FC1_SKIP_STAGE) ? 1 : 0;
    int epi1;
    if (mx) {
        g1p.g_act = nullptr;           // MXFP8: no activation global scale
        g1p.out_codes = hq_codes;
        g1p.out_sf = hq_sf;
        epi1 = kEpiFc1Mx;
    } else if (per_token) {
        g1p.g_act = g1;
        g1p.g_act_per_token = 1;
        g1p.out_f32 = reinterpret_cast<float*>(wsp(W.h_f32));
        epi1 = kEpiFc1F32;
    } else {
        g1p.g_act = act_scale_fc1;
        g1p.g_act_per_token = 0;
        g1p.g2 = act_scale_fc2;
        g1p.out_codes = hq_codes;
        g1p.out_sf = hq_sf;
        epi1 = kEpiFc1Quant;
    }
    e = swap    ? launch_gemm_swap(c, epi1, act == MOE_ACT_SWIGLU, tmB1, tmA1, g1p, sms)
        : pair1 ? launch_gemm_nvf4_pair(c, epi1, tmA1, tmB1, g1p, device)
                : launch_gemm_nvf4(c, epi1, tmA1, tmB1, g1p, sms, tn1, mx ? 1 : 0);
    if (e != cudaSuccess || !mark(4)) return MOE_ERR_CUDA;
    if (per_token) {
        e = launch_quantize_h(c, W.rows_cap, s.I, meta, route_of_row, reinterpret_cast<const float*>(wsp(W.h_f32)),
                              reinterpret_cast<float*>(wsp(W.g2)), hq_codes, hq_sf, four_six ? 1 : 0);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
    }
    if (!mark(5)) return MOE_ERR_CUDA;

    GemmParams g2p{};
    g2p.sfa = hq_sf;
    g2p.sfb = pw + P.w2_sf;
    g2p.kdim = s.I;
    g2p.chunk_maps = ch2 ? 1 : 0;
    g2p.n = s.H;
    g2p.meta = meta;
    g2p.tile_expert = tile_expert;
    g2p.tile_pair = tile_pair;
    g2p.tile_half = tile_half;
    g2p.route_of_row = route_of_row;
    g2p.num_experts = s.E;
    g2p.status = status;
    g2p.act = act;
    g2p.topk = s.K;
    g2p.gw = reinterpret_cast<const float*>(pw + P.gw2);
    g2p.topk_w = topk_w;
    g2p.weight_on_output = on_input ? 0 : 1;
    g2p.out_cols = s.H;
    if (mx) {
        g2p.g_act = nullptr;
        g2p.g_act_per_token = 0;
    } else if (per_token) {
        g2p.g_act = reinterpret_cast<const float*>(wsp(W.g2));
        g2p.g_act_per_token = 2;
    } else {
        g2p.g_act = act_scale_fc2;
        g2p.g_act_per_token = 0;
    }
    int epi2;
    if (det) {
        g2p.out_bf16 = reinterpret_cast<__nv_bfloat16*>(wsp(W.o_bf16));
        epi2 = kEpiFc2Store;
    } else {
        g2p.out_f32 = y_acc;
        epi2 = kEpiFc2Scatter;
        // an accumulator beyond 48 MB: walk FC2's output width in slabs whose
        // accumulator slice stays in L2 (T x slab x 4 B <= 48 MB), so that a
        // token's K reductions do not each go through HBM
        const uint64_t slab_bytes_per_tile = (uint64_t)s.T * (uint64_t)(pair2 ? 256 : tn2) * 4u;
        if (!swap && (uint64_t)s.T * s.H * 4u > kSlabAccBytes) {
            const uint64_t ns = kSlabAccBytes / slab_bytes_per_tile;
            g2p.n_slab = (int)(ns < 1 ? 1 : ns);
        }
    }
    e = swap    ? launch_gemm_swap(c, epi2, false, tmB2, tmA2, g2p, sms)
        : pair2 ? launch_gemm_nvf4_pair(c, epi2, tmA2, tmB2, g2p, device)
                : launch_gemm_nvf4(c, epi2, tmA2, tmB2, g2p, sms, tn2, mx ? 1 : 0);
    if (e != cudaSuccess || !mark(6)) return MOE_ERR_CUDA;

    if (det)
        e = launch_finalize_deterministic(c, s.T, s.H, s.K, row_of_route, topk_w, on_input ? 0 : 1, wsp(W.o_bf16),
                                          y_bf16);
    else
        e = launch_finalize_fused(c, s.T, s.H, y_acc, y_bf16);
    if (e != cudaSuccess || !mark(7)) return MOE_ERR_CUDA;
    return MOE_OK;
}

moe_status moe_nvfp4_forward(moe_shape s, uint32_t flags, const void* x_bf16, const float* router_logits,
                             const float* router_bias, const float* act_scale_fc1, const float* act_scale_fc2,
                             const void* prepared, void* workspace, size_t workspace_bytes, void* y_bf16,
                             void* stream) {
    if (flags & MOE_ROUTER_GEMM) return MOE_ERR_INVALID_ARG;   // logits come from the caller here
    RoutingIn rin;
    rin.logits = router_logits;
    rin.bias = router_bias;
    return forward_impl(s, flags, x_bf16, rin, act_scale_fc1, act_scale_fc2, prepared, workspace, workspace_bytes,
                        y_bf16, stream, nullptr);
}

moe_status moe_nvfp4_forward_routed(moe_shape s, uint32_t flags, const void* x_bf16, const int32_t* topk_ids,
                                    const float* topk_weights, const float* act_scale_fc1,
                                    const float* act_scale_fc2, const void* prepared, void* workspace,
                                    size_t workspace_bytes, void* y_bf16, void* stream) {
    if (!topk_ids || (flags & MOE_ROUTER_GEMM)) return MOE_ERR_INVALID_ARG;
    RoutingIn rin;
    rin.ids = topk_ids;
    rin.w = topk_weights;
    return forward_impl(s, flags, x_bf16, rin, act_scale_fc1, act_scale_fc2, prepared, workspace, workspace_bytes,
                        y_bf16, stream, nullptr);
}

moe_status moe_nvfp4_forward_staged(moe_shape s, uint32_t flags, const void* x_bf16, const float* router_logits,
                                    const float* router_bias, const float* act_scale_fc1,
                                    const float* act_scale_fc2, const void* prepared, void* workspace,
                                    size_t workspace_bytes, void* y_bf16, void* stream, void* const* events) {
    if (!events || (flags & MOE_ROUTER_GEMM)) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < MOE_NUM_STAGE_EVENTS; ++i)
        if (!events[i]) return MOE_ERR_INVALID_ARG;
    RoutingIn rin;
    rin.logits = router_logits;
    rin.bias = router_bias;
    return forward_impl(s, flags, x_bf16, rin, act_scale_fc1, act_scale_fc2, prepared, workspace, workspace_bytes,
                        y_bf16, stream, events);
}

// 2-D uint8 maps of the router GEMM's BF16 operands (rows of 2H bytes,
// 128-byte boxes, 128-byte swizzle).
static bool encode_router_maps(CUtensorMap* tmX, CUtensorMap* tmW, const void* x, const void* gate_w, int T, int E,
                               int H) {
    return encode_operand_map(tmX, x, (uint64_t)T, (uint64_t)H * 2, 128, 128) &&
           encode_operand_map(tmW, gate_w, (uint64_t)E, (uint64_t)H * 2, 128, (uint32_t)router_gemm_tile_n(E));
}

static bool router_gemm_args_ok(int T, int E, int H, const void* x, const void* gate_w, const void* logits) {
    if (T < 1 || T > (1 << 22) || E < 1 || E > 1024 || H < 128 || H % 128 != 0 || H > 65536) return false;
    if (!x || !gate_w || !logits || !aligned(x, 16) || !aligned(gate_w, 16) || !aligned(logits, 16)) return false;
    const size_t lb = (size_t)T * E * 4;
    return !overlaps(logits, lb, x, (size_t)T * H * 2) && !overlaps(logits, lb, gate_w, (size_t)E * H * 2);
}

moe_status moe_nvfp4_router_logits(int T, int E, int H, const void* x_bf16, const void* gate_w_bf16, float* logits,
                                   void* stream) {
    if (!router_gemm_args_ok(T, E, H, x_bf16, gate_w_bf16, logits)) return MOE_ERR_INVALID_ARG;
    int sms = 0;
    const moe_status st = device_state(&sms);
    if (st != MOE_OK) return st;
    CUtensorMap tmX, tmW;
    if (!encode_router_maps(&tmX, &tmW, x_bf16, gate_w_bf16, T, E, H)) return MOE_ERR_CUDA;
    LaunchCtx c;
    c.stream = static_cast<cudaStream_t>(stream);
    return cuda_status(launch_router_gemm(c, tmX, tmW, T, E, H, logits, nullptr));
}

moe_status moe_nvfp4_forward_gate(moe_shape s, uint32_t flags, const void* x_bf16, const void* gate_w_bf16,
                                  const float* router_bias, const float* act_scale_fc1, const float* act_scale_fc2,
                                  const void* prepared, void* workspace, size_t workspace_bytes, void* y_bf16,
                                  void* stream) {
    if (!(flags & MOE_ROUTER_GEMM)) return MOE_ERR_INVALID_ARG;
    moe_status st = validate_shape(s, flags);
    if (st != MOE_OK) return st;
    if (!workspace || !aligned(workspace, 256)) return MOE_ERR_INVALID_ARG;
    const moe_workspace_layout W = workspace_layout(s, flags);
    if (workspace_bytes < W.total) return MOE_ERR_WORKSPACE;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    float* logits = reinterpret_cast<float*>(ws + W.logits);
    if (!router_gemm_args_ok(s.T, s.E, s.H, x_bf16, gate_w_bf16, logits) ||
        overlaps(gate_w_bf16, (size_t)s.E * s.H * 2, workspace, W.total))
        return MOE_ERR_INVALID_ARG;
    int sms = 0;
    st = device_state(&sms);
    if (st != MOE_OK) return st;
    CUtensorMap tmX, tmW;
    if (!encode_router_maps(&tmX, &tmW, x_bf16, gate_w_bf16, s.T, s.E, s.H)) return MOE_ERR_CUDA;
    LaunchCtx c;
    c.stream = static_cast<cudaStream_t>(stream);
    unsigned int* status = reinterpret_cast<unsigned int*>(ws + W.status);
    // the status word is cleared here, before the logits kernel (which can
    // raise a timeout bit), rather than by the router
    if (cudaMemsetAsync(status, 0, 16, c.stream) != cudaSuccess) return MOE_ERR_CUDA;
    if (launch_router_gemm(c, tmX, tmW, s.T, s.E, s.H, logits, status) != cudaSuccess) return MOE_ERR_CUDA;
    RoutingIn rin;
    rin.logits = logits;
    rin.bias = router_bias;
    rin.status_cleared = true;
    return forward_impl(s, flags, x_bf16, rin, act_scale_fc1, act_scale_fc2, prepared, workspace, workspace_bytes,
                        y_bf16, stream, nullptr);
}

int moe_nvfp4_forward_launches(moe_shape s, uint32_t flags) {
    if (validate_shape(s, flags) != MOE_OK) return -1;
    if (flags & MOE_FUSED_LAYER) return 1;
    const int extra = mode_of(flags) == kModePerToken ? 1 : 0;   // the FC2-input quantization
    // T <= 32: router and scan in one launch
    if (s.T <= kUnitTokens) return 5 + extra;
    // router + unit counts, scan, quantize or gather (+ row scatter), FC1, [FC2-input quant], FC2, finalize
    return 6 + extra;
}

moe_status moe_nvfp4_last_device_status(void* workspace, void* stream) {
    if (!workspace || !aligned(workspace, 256)) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned int word = 0;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemset(workspace, 0, sizeof(word)) != cudaSuccess) return MOE_ERR_CUDA;
    if (word & (kStatusTimeoutProducer | kStatusTimeoutMma | kStatusTimeoutEpilogue | kStatusTimeoutGrid)) return MOE_ERR_TIMEOUT;
    if (word & (kStatusBadExpert | kStatusBadRow)) return MOE_ERR_INVALID_ARG;
    if (word & kStatusGridAbort) return MOE_ERR_TIMEOUT;   // raised only together with a reason above
    return MOE_OK;
}

moe_status moe_nvfp4_debug_convert(const float* in, int64_t n, uint8_t* e4m3, uint8_t* e2m1, void* stream) {
    if (n < 0 || (n > 0 && (!in || !e4m3 || !e2m1))) return MOE_ERR_INVALID_ARG;
    if (n == 0) return MOE_OK;
    int sms = 0;
    const moe_status st = device_state(&sms);
    if (st != MOE_OK) return st;
    return cuda_status(launch_debug_convert(static_cast<cudaStream_t>(stream), in, n, e4m3, e2m1));
}

}  // extern "C"
