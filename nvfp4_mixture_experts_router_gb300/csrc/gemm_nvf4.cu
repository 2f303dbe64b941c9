// One grouped GEMM per launch on the engine of gemm_nvf4.cuh.
#include "gemm_nvf4.cuh"

namespace moe {

using grouped::Cfg;

template <int EPI, int BN, int KIND>
__global__ void __launch_bounds__(Cfg<BN, KIND>::kNumThreads, 1)
    gemm_nvf4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    const grouped::Smem s = grouped::carve<BN, KIND>(smem_raw);
    if (threadIdx.x == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    const uint32_t tmem_base = grouped::gemm_init<BN, KIND>(s);
    pdl_wait();  // A operand, tile map and tile count come from earlier kernels
    grouped::RingState rs;
    grouped::gemm_tiles<EPI, BN, KIND>(s, tmem_base, &tmA, &tmB, p, rs);
    grouped::gemm_drain<BN, KIND>(s, p.status);
    tc_fence_before();
    __syncthreads();
    pdl_launch_dependents();
    grouped::gemm_free_tmem(tmem_base);
}

template <int EPI, int BN, int KIND>
static cudaError_t set_smem_one() {
    return cudaFuncSetAttribute(gemm_nvf4_kernel<EPI, BN, KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Cfg<BN, KIND>::kSmemBytes);
}

template <int BN>
static cudaError_t set_smem_all() {
    cudaError_t e;
    if ((e = set_smem_one<kEpiFc1Quant, BN, 0>())) return e;
    if ((e = set_smem_one<kEpiFc1F32, BN, 0>())) return e;
    if ((e = set_smem_one<kEpiFc2Store, BN, 0>())) return e;
    if ((e = set_smem_one<kEpiFc2Scatter, BN, 0>())) return e;
    if ((e = set_smem_one<kEpiFc1Mx, BN, 1>())) return e;
    if ((e = set_smem_one<kEpiFc2Store, BN, 1>())) return e;
    return set_smem_one<kEpiFc2Scatter, BN, 1>();
}

cudaError_t setup_gemm_kernels() {
    const cudaError_t e = set_smem_all<128>();
    if (e != cudaSuccess) return e;
    return set_smem_all<256>();
}

template <int EPI, int BN, int KIND>
static cudaError_t launch_one(const LaunchCtx& c, const CUtensorMap& tmA, const CUtensorMap& tmB,
                              const GemmParams& p, int num_sms) {
    using C = Cfg<BN, KIND>;
    return c.launch(gemm_nvf4_kernel<EPI, BN, KIND>, dim3(num_sms), dim3(C::kNumThreads), (size_t)C::kSmemBytes, tmA,
                    tmB, p);
}

template <int BN>
static cudaError_t launch_bn(const LaunchCtx& c, int epilogue, int kind, const CUtensorMap& tmA,
                             const CUtensorMap& tmB, const GemmParams& p, int num_sms) {
    if (kind == 0) {
        switch (epilogue) {
            case kEpiFc1Quant: return launch_one<kEpiFc1Quant, BN, 0>(c, tmA, tmB, p, num_sms);
            case kEpiFc1F32: return launch_one<kEpiFc1F32, BN, 0>(c, tmA, tmB, p, num_sms);
            case kEpiFc2Store: return launch_one<kEpiFc2Store, BN, 0>(c, tmA, tmB, p, num_sms);
            case kEpiFc2Scatter: return launch_one<kEpiFc2Scatter, BN, 0>(c, tmA, tmB, p, num_sms);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (epilogue) {
        case kEpiFc1Mx: return launch_one<kEpiFc1Mx, BN, 1>(c, tmA, tmB, p, num_sms);
        case kEpiFc2Store: return launch_one<kEpiFc2Store, BN, 1>(c, tmA, tmB, p, num_sms);
        case kEpiFc2Scatter: return launch_one<kEpiFc2Scatter, BN, 1>(c, tmA, tmB, p, num_sms);
        default: return cudaErrorInvalidValue;
    }
}

int gemm_nvf4_tile_n(int kdim, int n) {
    // a 256-wide tile halves the MMA issues per weight byte but leaves room for
    // only one accumulator, so its epilogue is not overlapped: worth it when the
    // main loop per tile is long
    // (measured: 256 wins for K = 7168, loses for K <= 2048)
    return (kdim >= 4096 && n >= 256) ? 256 : 128;
}

cudaError_t launch_gemm_nvf4(const LaunchCtx& c, int epilogue, const CUtensorMap& tmA, const CUtensorMap& tmB,
                             const GemmParams& p, int num_sms, int tile_n, int kind) {
    return tile_n == 256 ? launch_bn<256>(c, epilogue, kind, tmA, tmB, p, num_sms)
                         : launch_bn<128>(c, epilogue, kind, tmA, tmB, p, num_sms);
}

}  // namespace moe
