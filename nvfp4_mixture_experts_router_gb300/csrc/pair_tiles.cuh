// Tile order of the CTA-pair GEMMs (gemm_nvf4_pair.cu, gemm_w4a16.cu): a
// pair tile is two consecutive 128-row M tiles of one expert (listed by the
// permutation scan in tile_pair as (first << 1) | has_second) x 256 weight
// rows.
#pragma once
#include "kernels.h"

namespace moe {

// Pair tile -> (M tile of this CTA, the pair's first M tile, N tile), N
// tiles fastest; with slabs of p.n_slab N tiles the output width is walked
// slab by slab, every pair within a slab before the next (the fused-finalize
// scatter then keeps adding into one slab of the accumulator, which stays in
// L2).  m_tile is -1 for rank 1 of a pair without a second M tile.
__device__ __forceinline__ void decode_pair(const GemmParams& p, int tile, int n_tiles, int num_pairs, uint32_t rank,
                                            int& m_tile, int& m0, int& n_tile) {
    int pr;
    if (p.n_slab <= 0) {
        pr = tile / n_tiles;
        n_tile = tile % n_tiles;
    } else {
        const int per_slab = num_pairs * p.n_slab;
        const int slab = tile / per_slab, rem = tile % per_slab;
        const int width = min(p.n_slab, n_tiles - slab * p.n_slab);   // the last slab may be narrower
        pr = rem / width;
        n_tile = slab * p.n_slab + rem % width;
    }
    const int v = p.tile_pair[pr];
    m0 = v >> 1;
    m_tile = rank == 0 ? m0 : ((v & 1) ? m0 + 1 : -1);
}


}  // namespace moe
