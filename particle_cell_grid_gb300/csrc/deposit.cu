// deposit.cu -- C ABI of the current deposit: argument checks, J zeroing, the
// chunk-to-tile map, the flat (all-global-reduction) kernel and the tiled
// dispatch.  See deposit.cuh for the method and its sources.
#include <mutex>

#include "deposit.cuh"

namespace pcg {
namespace {

using dep::Counters;
using dep::Geom;
using dep::Particles;

// Zero J, map every chunk of the sorted array to the tile holding its first
// slot, and check that tile_offsets is a valid layout.  One launch.
__global__ void __launch_bounds__(256)
    prep_kernel(float *__restrict__ J, size_t nJ, const uint32_t *__restrict__ offs,
                unsigned n_tiles, long long n, long long chunk, unsigned *__restrict__ chunk_tile,
                long long nchunks, unsigned *__restrict__ flags) {
    const size_t tid = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    // J is 16-byte aligned (checked on the host) and nJ = 3 * ncells
    float4 *J4 = reinterpret_cast<float4 *>(J);
    const size_t n4 = nJ / 4;
    for (size_t i = tid; i < n4; i += stride) J4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (tid < nJ - n4 * 4) J[n4 * 4 + tid] = 0.f;
    if (offs == nullptr) return;
    for (size_t b = tid; b < (size_t)nchunks; b += stride) {
        const unsigned long long target = (unsigned long long)b * (unsigned long long)chunk;
        unsigned lo = 0, hi = n_tiles;  // largest t in [0, n_tiles] with offs[t] <= target
        while (lo < hi) {
            const unsigned mid = lo + (hi - lo + 1) / 2;
            if ((unsigned long long)offs[mid] <= target) lo = mid;
            else hi = mid - 1;
        }
        chunk_tile[b] = lo;
    }
    bool bad = false;
    for (size_t t = tid; t < n_tiles; t += stride) bad |= offs[t] > offs[t + 1];
    if (tid == 0) bad |= (offs[0] != 0u) | ((long long)offs[n_tiles] > n);
    if (bad && flags) atomicOr(flags, PCG_FLAG_BAD_LAYOUT);
}

template <int DIM, int ORDER>
__global__ void __launch_bounds__(256)
    deposit_flat_kernel(Geom g, Particles P, long long n, float *__restrict__ J, Counters ctr) {
    unsigned n_inv = 0;
    for (long long p = blockIdx.x * (long long)blockDim.x + threadIdx.x; p < n;
         p += (long long)gridDim.x * blockDim.x) {
        const float x = P.x[p], y = P.y[p], z = DIM == 3 ? P.z[p] : 0.f;
        if (!dep::in_domain<DIM>(g, x, y, z)) {
            ++n_inv;
            continue;
        }
        const float q = P.q[p];
        dep::deposit_global<DIM, ORDER>(g, J, x, y, z, q * P.vx[p], q * P.vy[p], q * P.vz[p]);
    }
    warp_add_u64(ctr.n_invalid, n_inv);
}

}  // namespace

// Particles per CTA of the tiled kernel: a power of two in [1024, 16384], about
// 16 chunks per SM so that the last wave is short.
long long chunk_for(long long n) {
    long long target = n / ((long long)num_sms() * 16);
    long long c = 1024;
    while (c < target && c < 16384) c <<= 1;
    return c;
}

// The 3D quadratic kernel flushes its window of 11^3 nodes at every tile
// segment end, so it takes larger chunks (fewer segments split across chunks);
// never smaller than chunk_for(n), so the workspace sized by chunk_for holds
// its chunk map.
constexpr long long kQuadChunkMax = 65536;
long long chunk_for_shape(long long n, int dim, int order, int tile, bool tiled) {
    long long c = chunk_for(n);
    if (!(tiled && dim == 3 && order == 2 && tile == 8)) return c;
    const long long target = n / ((long long)num_sms() * 8);
    while (c < target && c < kQuadChunkMax) c <<= 1;
    return c;
}

bool geom_from(int32_t dim, const int32_t *grid, int tile, Geom *g) {
    TileGrid tg;
    if (!make_tile_grid(dim, grid, tile < 1 ? 1 : tile, &tg)) return false;
    g->ncells = 1;
    for (int mu = 0; mu < 3; ++mu) {
        g->N[mu] = tg.N[mu];
        g->nt[mu] = tg.nt[mu];
        g->Nf[mu] = (float)tg.N[mu];
        g->ncells *= tg.N[mu];
    }
    g->n_tiles = (unsigned)tg.n_tiles;
    return true;
}

pcg_status launch_prep(float *J, const Geom &g, const uint32_t *tile_offsets, long long n, long long chunk,
                       unsigned *chunk_tile, unsigned *flags, cudaStream_t s) {
    const long long nchunks = (n + chunk - 1) / chunk;
    const size_t nJ = 3 * (size_t)g.ncells;
    size_t work = nJ / 4 > (size_t)nchunks ? nJ / 4 : (size_t)nchunks;
    if (tile_offsets != nullptr && (size_t)g.n_tiles > work) work = g.n_tiles;
    size_t blocks = (work + 255) / 256;
    const size_t cap = (size_t)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    prof::Mark mk("deposit_prep", s);
    prep_kernel<<<(unsigned)blocks, 256, 0, s>>>(J, nJ, tile_offsets, g.n_tiles, n, chunk, chunk_tile, nchunks,
                                                flags);
    return launch_status();
}

}  // namespace pcg

extern "C" pcg_status pcg_deposit_current_workspace_size(int32_t dim, const int32_t *grid,
                                                         int32_t tile, int64_t n, size_t *bytes) {
    using namespace pcg;
    Geom g;
    if (bytes == nullptr || n < 0 || n >= 0xffffffffll || !geom_from(dim, grid, tile, &g))
        return PCG_ERR_INVALID_ARG;
    const long long chunk = chunk_for(n);
    *bytes = align_up((size_t)((n + chunk - 1) / chunk) * sizeof(unsigned), 256);
    return PCG_OK;
}

namespace pcg {
namespace {

// Host checks shared by pcg_deposit_current and pcg_deposit_current_noalloc,
// made before anything else (workspace, scratch lookup, launches).
pcg_status check_current_args(int32_t dim, const int32_t *grid, int32_t order, int32_t tile, int32_t halo,
                              int32_t block, int64_t n, const float *const *pos, const float *const *vel,
                              const float *q, bool tiled, const float *J, Geom *g) {
    if (n < 0 || n >= 0xffffffffll) return PCG_ERR_INVALID_ARG;
    if (order != 1 && order != 2) return PCG_ERR_INVALID_ARG;
    if (tiled && (tile < 1 || tile > 64 || halo < 0)) return PCG_ERR_INVALID_ARG;
    if (!geom_from(dim, grid, tiled ? tile : 1, g)) return PCG_ERR_INVALID_ARG;
    if (block != 0 && block != 128 && block != 256 && block != 512) return PCG_ERR_INVALID_ARG;
    if (J == nullptr || !aligned16(J)) return PCG_ERR_INVALID_ARG;
    if (n > 0) {
        if (pos == nullptr || vel == nullptr || q == nullptr) return PCG_ERR_INVALID_ARG;
        for (int mu = 0; mu < dim; ++mu)
            if (pos[mu] == nullptr) return PCG_ERR_INVALID_ARG;
        for (int c = 0; c < 3; ++c)
            if (vel[c] == nullptr) return PCG_ERR_INVALID_ARG;
    }
    if (tiled && ((tile != 4 && tile != 8) || halo > 2)) return PCG_ERR_UNSUPPORTED;
    return PCG_OK;
}

}  // namespace
}  // namespace pcg

extern "C" pcg_status pcg_deposit_current(int32_t dim, const int32_t *grid, int32_t order,
                                          int32_t tile, int32_t halo, int32_t block, int64_t n,
                                          const float *const *pos, const float *const *vel,
                                          const float *q, const uint32_t *tile_offsets, float *J,
                                          pcg_stats *stats, void *workspace,
                                          size_t workspace_bytes, void *stream) {
    using namespace pcg;
    const bool tiled = tile_offsets != nullptr;
    Geom g;
    {
        const pcg_status st = check_current_args(dim, grid, order, tile, halo, block, n, pos, vel, q, tiled, J, &g);
        if (st != PCG_OK) return st;
    }
    const long long chunk = chunk_for_shape(n, dim, order, tile, tiled);
    const long long nchunks = (n + chunk - 1) / chunk;
    const size_t need = tiled ? align_up((size_t)nchunks * sizeof(unsigned), 256) : 0;
    if (workspace_bytes < need || (need > 0 && workspace == nullptr)) return PCG_ERR_WORKSPACE;

    cudaStream_t s = as_stream(stream);
    Particles P{};
    if (n > 0) {
        P.x = pos[0];
        P.y = pos[1];
        P.z = dim == 3 ? pos[2] : pos[0];
        P.vx = vel[0];
        P.vy = vel[1];
        P.vz = vel[2];
        P.q = q;
    }
    Counters ctr{stats ? &stats->n_escaped : nullptr, stats ? &stats->n_invalid : nullptr,
                 stats ? &stats->error_flags : nullptr};
    unsigned *chunk_tile = static_cast<unsigned *>(workspace);
    {
        const pcg_status st = launch_prep(J, g, tiled ? tile_offsets : nullptr, n, chunk, chunk_tile, ctr.flags, s);
        if (st != PCG_OK) return st;
    }
    if (n == 0) return PCG_OK;
    if (!tiled) {
        const long long want = (n + 255) / 256;
        const long long cap = (long long)num_sms() * 16;
        const unsigned blocks = (unsigned)(want < cap ? want : cap);
        prof::Mark mk("deposit_flat", s);
        if (dim == 2) {
            if (order == 1) deposit_flat_kernel<2, 1><<<blocks, 256, 0, s>>>(g, P, n, J, ctr);
            else deposit_flat_kernel<2, 2><<<blocks, 256, 0, s>>>(g, P, n, J, ctr);
        } else {
            if (order == 1) deposit_flat_kernel<3, 1><<<blocks, 256, 0, s>>>(g, P, n, J, ctr);
            else deposit_flat_kernel<3, 2><<<blocks, 256, 0, s>>>(g, P, n, J, ctr);
        }
        return launch_status();
    }
    const int threads = block == 0 ? 256 : block;
    return dim == 2 ? deposit_tiled_2d(order, tile, halo, g, n, P, tile_offsets, J, ctr, chunk_tile,
                                       chunk, threads, s)
                    : deposit_tiled_3d(order, tile, halo, g, n, P, tile_offsets, J, ctr, chunk_tile,
                                       chunk, threads, s);
}

// ---------------------------------------------------------------------------
// Allocation-free variant of pcg_deposit_current.
//
// Some callers cannot allocate device memory at all: code running inside a
// host callback or a custom allocator, plugins handed only their input and
// output buffers by a host application, or a pool that forbids cudaMalloc at
// run time.  This entry point takes exactly the arguments of
// pcg_deposit_current except the workspace: the only scratch the tiled path
// needs, the chunk-to-tile map (one 32-bit entry per chunk of particles), lives
// in the fixed device array below, which every GPU that loads the library holds
// until the process exits.
//
// Host code must not pass the array's name to a kernel: on the host it is only
// a stand-in for the symbol.  Its device address is looked up once per device,
// with that device current, by the first call made on that device.
namespace pcg {
namespace {

constexpr size_t kNoAllocChunks = 65536;  // 256 KB: up to 65536 chunks of <= 16384 particles
static __device__ __align__(256) unsigned g_chunk_tile[kNoAllocChunks];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
unsigned *g_chunk_tile_addr[kMaxDevices] = {};

// Device address of g_chunk_tile on the current device (set up on first use).
pcg_status noalloc_scratch(unsigned **out) {
    int dev = 0;
    PCG_CHECK_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return PCG_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_chunk_tile_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_chunk_tile) != cudaSuccess || p == nullptr) {
            (void)cudaGetLastError();
            return PCG_ERR_CUDA;
        }
        g_chunk_tile_addr[dev] = static_cast<unsigned *>(p);
    }
    *out = g_chunk_tile_addr[dev];
    return PCG_OK;
}

}  // namespace
}  // namespace pcg

extern "C" pcg_status pcg_deposit_current_noalloc(int32_t dim, const int32_t *grid, int32_t order,
                                                  int32_t tile, int32_t halo, int32_t block,
                                                  int64_t n, const float *const *pos,
                                                  const float *const *vel, const float *q,
                                                  const uint32_t *tile_offsets, float *J,
                                                  pcg_stats *stats, void *stream) {
    using namespace pcg;
    {
        // the same argument checks as pcg_deposit_current, before the size limit
        // and before the scratch array's address is looked up
        Geom g;
        const pcg_status st = check_current_args(dim, grid, order, tile, halo, block, n, pos, vel, q,
                                                 tile_offsets != nullptr, J, &g);
        if (st != PCG_OK) return st;
    }
    const long long chunk = chunk_for_shape(n, dim, order, tile, tile_offsets != nullptr);
    const long long nchunks = (n + chunk - 1) / chunk;
    if (tile_offsets != nullptr && (size_t)nchunks > kNoAllocChunks) return PCG_ERR_WORKSPACE;
    unsigned *scratch = nullptr;
    if (tile_offsets != nullptr && n > 0) {
        pcg_status st = noalloc_scratch(&scratch);
        if (st != PCG_OK) return st;
    }
    // every entry the kernels read is written by this call's prep kernel first,
    // so the array needs no clearing between calls
    return pcg_deposit_current(dim, grid, order, tile, halo, block, n, pos, vel, q, tile_offsets, J,
                               stats, scratch, scratch ? kNoAllocChunks * sizeof(unsigned) : 0,
                               stream);
}
