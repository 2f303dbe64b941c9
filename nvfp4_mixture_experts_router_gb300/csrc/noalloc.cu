// Routing and token permutation without any caller-provided scratch.
//
// moe_nvfp4_forward needs a workspace that the caller allocates.  Some
// callers cannot allocate device memory at all: code that runs inside
// another engine's fixed memory budget (a plugin handed only its inputs and
// outputs), or a latency-critical loop where a cudaMalloc and the device
// synchronization it can imply are not acceptable.  For them this file
// offers the routing stage (softmax + top-K, then the stable permutation by
// expert) with its only scratch -- per-unit expert counts and token masks,
// the M-tile map and a status word -- in a fixed array in device memory that
// every GPU loading the library holds until the process exits.  It computes
// exactly what the routing stage of moe_nvfp4_forward computes, with the
// router, the unit masks, the scan and the row scatter as four kernels.
#include <mutex>

#include "../../include/moe_nvfp4.h"
#include "common.cuh"
#include "kernels.h"
#include "layout.h"

namespace {

// 1 MiB of int32 scratch, shared by every call on a device.
constexpr int64_t kScratchInts = MOE_NOALLOC_SCRATCH_BYTES / 4;
static __device__ __align__(256) int g_route_scratch[kScratchInts];

// Host-side addresses of g_route_scratch, looked up once per device (the
// array's name in host code is only a stand-in for the symbol, not a device
// address).
// A device's outcome is kept once it is final (the address found, or the
// GPU is not one this library runs on); a CUDA error during the look-up (for
// example a first call made inside a stream capture) is returned but not
// kept, so that a later call tries again.
std::mutex g_mu;
int* g_scratch_ptr[64] = {};
moe_status g_state[64] = {};
bool g_ready[64] = {};

moe_status scratch_for_current_device(int** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_ready[dev]) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            g_state[dev] = MOE_ERR_CUDA;
        } else if (major != 10 || minor != 3) {
            g_state[dev] = MOE_ERR_UNSUPPORTED;
        } else if (moe::setup_routing_kernels() != cudaSuccess) {
            g_state[dev] = MOE_ERR_CUDA;
        } else {
            void* p = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&p, g_route_scratch);
            if (e != cudaSuccess || p == nullptr) {
                g_state[dev] = MOE_ERR_CUDA;
            } else {
                g_scratch_ptr[dev] = static_cast<int*>(p);
                g_state[dev] = MOE_OK;
            }
        }
        g_ready[dev] = g_state[dev] != MOE_ERR_CUDA;
    }
    *out = g_scratch_ptr[dev];
    return g_state[dev];
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" {

moe_status moe_nvfp4_route_noalloc(int T, int E, int K, uint32_t flags, const float* router_logits,
                                   const float* router_bias, int32_t* topk_ids, float* topk_w, int32_t* count,
                                   int32_t* offsets, int32_t* padded_offsets, int32_t* row_of_route,
                                   int32_t* route_of_row, void* stream) {
    if ((flags & ~MOE_ROUTE_NO_RENORM) != 0) return MOE_ERR_INVALID_ARG;
    if (T < 1 || T > (1 << 22) || E < 1 || E > 1024 || K < 1 || K > 32 || K > E) return MOE_ERR_INVALID_ARG;
    if ((int64_t)T * K > (1 << 26)) return MOE_ERR_INVALID_ARG;
    if (!router_logits || !topk_ids || !topk_w || !count || !offsets || !padded_offsets || !row_of_route ||
        !route_of_row)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(router_logits, 4) || (router_bias && !aligned(router_bias, 4)) || !aligned(topk_ids, 4) ||
        !aligned(topk_w, 4) || !aligned(count, 4) || !aligned(offsets, 4) || !aligned(padded_offsets, 4) ||
        !aligned(row_of_route, 4) || !aligned(route_of_row, 4))
        return MOE_ERR_INVALID_ARG;

    // scratch layout (int32): [0,4) status, [4,8) meta, [8, 8+tiles) M-tile
    // map, then at the next 64-int boundary the per-(expert, unit) starting
    // rows and the per-(expert, unit) token masks
    const int64_t units = (T + moe::kUnitTokens - 1) / moe::kUnitTokens;
    const int64_t tiles = (int64_t)(moe::rows_capacity(T, K, E) / moe::kTileM);
    const int64_t base_units = (8 + tiles + 63) / 64 * 64;
    if (base_units + 2 * (int64_t)E * units > kScratchInts) return MOE_ERR_WORKSPACE;

    int* scratch = nullptr;
    const moe_status st = scratch_for_current_device(&scratch);
    if (st != MOE_OK) return st;
    unsigned int* status = reinterpret_cast<unsigned int*>(scratch);
    int* meta = scratch + 4;
    int* tile_expert = scratch + 8;
    int* unit_base = scratch + base_units;
    uint32_t* unit_mask = reinterpret_cast<uint32_t*>(unit_base + (int64_t)E * units);

    moe::LaunchCtx c;
    c.stream = static_cast<cudaStream_t>(stream);
    c.pdl = false;
    // the router clears the status word; every other scratch entry is fully
    // written by a kernel before any kernel reads it
    cudaError_t e = moe::launch_router(c, T, E, K, router_logits, router_bias,
                                       (flags & MOE_ROUTE_NO_RENORM) ? 0 : 1, topk_ids, topk_w, status);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    e = moe::launch_permute(c, T, E, K, topk_ids, unit_base, unit_mask, count, offsets, padded_offsets, meta,
                            tile_expert, row_of_route, route_of_row, status);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // extern "C"
