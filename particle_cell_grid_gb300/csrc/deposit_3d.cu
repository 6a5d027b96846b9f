// deposit_3d.cu -- 3D instantiations of the tiled deposit kernel.
#include "deposit_tiled.cuh"

namespace pcg {
pcg_status deposit_tiled_3d(int order, int tile, int halo, const dep::Geom &g, long long n,
                            const dep::Particles &P, const uint32_t *offs, float *J,
                            const dep::Counters &ctr, unsigned *chunk_tile, long long chunk,
                            int block, cudaStream_t s) {
    return dep::dispatch_tiled<3>(order, tile, halo, g, n, P, offs, J, ctr, chunk_tile, chunk,
                                  block, s);
}
}  // namespace pcg
