// gemm_w4a16_swap.cu — the W4A16 GEMMs in the swapped orientation: the
// weights widened to BF16 on chip on the M side, 64 BF16 route rows on N.
// tmW: 3-D map over the prepared weight codes (row bytes, 128 rows, blocks
// of 128 rows), box 64 B x 64 x 2, unswizzled; tmX: 2-D map over the BF16
// activations, box 128 B x 64 rows, 128-byte swizzle.  gated: FC1 SwiGLU.
// Epilogues kEpiFc1Bf16 / kEpiFc2Store / kEpiFc2Scatter.
#pragma once
#include "kernels.h"

namespace moe {

cudaError_t setup_gemm_w4a16_swap_kernels();
cudaError_t launch_gemm_w4a16_swap(const LaunchCtx& c, int epilogue, bool gated, const CUtensorMap& tmW,
                                   const CUtensorMap& tmX, const GemmParams& p, int num_sms);

}  // namespace moe
