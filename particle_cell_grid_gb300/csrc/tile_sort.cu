// tile_sort.cu -- counting sort of particles into spatial tiles.
//
// Method: "Tiled current deposit" (Entity wiki), section "The tile-based
// spatial sort": ntiles = ceil(N / T) per axis, a tile key per particle,
// invalid particles parked in a sentinel bin after the last tile, tile_offsets
// as the prefix sum of the per-tile counts, and the SoA members physically
// permuted into tile order.  The page uses a vendor sort_by_key or a bin sort;
// here it is a hand-written counting sort, since the keys are small integers.
//
// GB300 design (bins B = n_tiles + 1):
//  * B <= kSmemBins: "chunked" sort.  G CTAs (a multiple of the 152 SMs) each
//    own a contiguous chunk of particles.  (1) count: block-private histogram in
//    shared memory, written out as counts[g][b]; (2) colscan: one thread per bin
//    scans its column over the G chunks (coalesced) giving each (chunk, bin)
//    its start inside the bin, and the bin totals; (3) a one-CTA exclusive scan
//    of the totals gives tile_offsets; (4) scatter: every CTA loads its
//    (chunk, bin) cursors into shared memory and places each particle with a
//    shared-memory atomic.  A chunk's particles of one tile land contiguously.
//  * B > kSmemBins (for example one bin per cell of a 64^3 grid): counts and
//    cursors live in global memory and are bumped with global atomics.
// No step waits on another CTA; kernel boundaries order the phases.
#include "common.cuh"

namespace pcg {
namespace {

constexpr unsigned kSmemBins = 32769;  // 128 KB + 4 B of shared counters
constexpr int kSortThreads = 512;
constexpr int kMaxPayload = 16;

struct KeyGeom {
    int nt0, nt1;  // tiles along x and y
    unsigned n_tiles;
    float N0, N1, N2;  // domain extent per axis (exact in fp32 up to 2^24)
    int tile;
};

struct Payload {
    const unsigned *in[kMaxPayload];
    unsigned *out[kMaxPayload];
};

template <int TILE>
__device__ __forceinline__ int tdiv(int i, int tile) {
    if (TILE > 0) return i / (TILE > 0 ? TILE : 1);  // constant divisor
    return i / tile;
}

// Tile key of one particle (sentinel n_tiles when any coordinate is outside [0, N)).
template <int DIM, int TILE>
__device__ __forceinline__ unsigned tile_key(const KeyGeom &g, float x, float y, float z) {
    bool ok = (x >= 0.f) & (x < g.N0) & (y >= 0.f) & (y < g.N1);
    if (DIM == 3) ok &= (z >= 0.f) & (z < g.N2);
    if (!ok) return g.n_tiles;
    int tx = tdiv<TILE>((int)x, g.tile);
    int ty = tdiv<TILE>((int)y, g.tile);
    int tz = DIM == 3 ? tdiv<TILE>((int)z, g.tile) : 0;
    return (unsigned)((tz * g.nt1 + ty) * g.nt0 + tx);
}

template <int DIM, int TILE>
__global__ void __launch_bounds__(kSortThreads)
    count_chunked_kernel(KeyGeom g, const float *__restrict__ kx, const float *__restrict__ ky,
                         const float *__restrict__ kz, long long n, long long chunk,
                         unsigned *__restrict__ counts, unsigned B,
                         unsigned long long *__restrict__ n_invalid) {
    extern __shared__ unsigned hist[];
    for (unsigned b = threadIdx.x; b < B; b += blockDim.x) hist[b] = 0;
    __syncthreads();
    const long long p0 = (long long)blockIdx.x * chunk;
    const long long p1 = min(n, p0 + chunk);
    unsigned inval = 0;
    for (long long p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
        const unsigned k = tile_key<DIM, TILE>(g, kx[p], ky[p], DIM == 3 ? kz[p] : 0.f);
        atomicAdd(&hist[k], 1u);
        inval += (k == g.n_tiles);
    }
    warp_add_u64(n_invalid, inval);
    __syncthreads();
    unsigned *row = counts + (size_t)blockIdx.x * B;
    for (unsigned b = threadIdx.x; b < B; b += blockDim.x) row[b] = hist[b];
}

// counts[g][b] -> exclusive start of chunk g inside bin b (in place); totals[b].
__global__ void __launch_bounds__(256)
    colscan_kernel(unsigned *__restrict__ counts, unsigned *__restrict__ totals, unsigned G,
                   unsigned B) {
    const unsigned b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    unsigned run = 0;
    for (unsigned gi = 0; gi < G; ++gi) {
        unsigned *c = counts + (size_t)gi * B + b;
        const unsigned v = *c;
        *c = run;
        run += v;
    }
    totals[b] = run;
}

// Exclusive scan of in[0..L) into out[0..L) by one CTA of 1024 threads; optional
// second output copy.  Handles any L in segments of 1024 * 8 elements.
__global__ void __launch_bounds__(1024)
    scan_one_cta_kernel(const unsigned *__restrict__ in, unsigned *__restrict__ out,
                        unsigned *__restrict__ out2, unsigned L) {
    constexpr int kItems = 8;
    __shared__ unsigned warp_sums[32];
    __shared__ unsigned carry_s;
    if (threadIdx.x == 0) carry_s = 0;
    __syncthreads();
    const unsigned lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (unsigned seg = 0; seg < L; seg += 1024u * kItems) {
        unsigned v[kItems];
        unsigned sum = 0;
        const unsigned base = seg + threadIdx.x * kItems;
#pragma unroll
        for (int i = 0; i < kItems; ++i) {
            v[i] = (base + i < L) ? in[base + i] : 0u;
            sum += v[i];
        }
        // inclusive warp scan of the per-thread sums
        unsigned incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            unsigned t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= (unsigned)o) incl += t;
        }
        if (lane == 31) warp_sums[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            unsigned ws = warp_sums[lane];
            unsigned wi = ws;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                unsigned t = __shfl_up_sync(0xffffffffu, wi, o);
                if (lane >= (unsigned)o) wi += t;
            }
            warp_sums[lane] = wi - ws;  // exclusive prefix of warp totals
        }
        __syncthreads();
        unsigned run = carry_s + warp_sums[warp] + (incl - sum);
#pragma unroll
        for (int i = 0; i < kItems; ++i) {
            if (base + i < L) {
                out[base + i] = run;
                if (out2) out2[base + i] = run;
            }
            run += v[i];
        }
        __syncthreads();
        if (threadIdx.x == 1023) carry_s = run;  // last thread holds the segment total
        __syncthreads();
    }
}

template <int DIM, int TILE>
__global__ void __launch_bounds__(kSortThreads)
    scatter_chunked_kernel(KeyGeom g, const float *__restrict__ kx, const float *__restrict__ ky,
                           const float *__restrict__ kz, long long n, long long chunk,
                           const unsigned *__restrict__ starts, const unsigned *__restrict__ offs,
                           unsigned B, Payload pl, int np) {
    extern __shared__ unsigned cursor[];
    const unsigned *row = starts + (size_t)blockIdx.x * B;
    for (unsigned b = threadIdx.x; b < B; b += blockDim.x) cursor[b] = offs[b] + row[b];
    __syncthreads();
    const long long p0 = (long long)blockIdx.x * chunk;
    const long long p1 = min(n, p0 + chunk);
    for (long long p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
        const unsigned k = tile_key<DIM, TILE>(g, kx[p], ky[p], DIM == 3 ? kz[p] : 0.f);
        const unsigned slot = atomicAdd(&cursor[k], 1u);
        for (int f = 0; f < np; ++f) pl.out[f][slot] = pl.in[f][p];
    }
}

template <int DIM, int TILE>
__global__ void __launch_bounds__(256)
    count_global_kernel(KeyGeom g, const float *__restrict__ kx, const float *__restrict__ ky,
                        const float *__restrict__ kz, long long n, unsigned *__restrict__ totals,
                        unsigned long long *__restrict__ n_invalid) {
    unsigned inval = 0;
    for (long long p = blockIdx.x * (long long)blockDim.x + threadIdx.x; p < n;
         p += (long long)gridDim.x * blockDim.x) {
        const unsigned k = tile_key<DIM, TILE>(g, kx[p], ky[p], DIM == 3 ? kz[p] : 0.f);
        atomicAdd(&totals[k], 1u);
        inval += (k == g.n_tiles);
    }
    warp_add_u64(n_invalid, inval);
}

template <int DIM, int TILE>
__global__ void __launch_bounds__(256)
    scatter_global_kernel(KeyGeom g, const float *__restrict__ kx, const float *__restrict__ ky,
                          const float *__restrict__ kz, long long n, unsigned *__restrict__ cursor,
                          Payload pl, int np) {
    for (long long p = blockIdx.x * (long long)blockDim.x + threadIdx.x; p < n;
         p += (long long)gridDim.x * blockDim.x) {
        const unsigned k = tile_key<DIM, TILE>(g, kx[p], ky[p], DIM == 3 ? kz[p] : 0.f);
        const unsigned slot = atomicAdd(&cursor[k], 1u);
        for (int f = 0; f < np; ++f) pl.out[f][slot] = pl.in[f][p];
    }
}

struct Plan {
    bool chunked;
    unsigned B;
    unsigned G;        // chunks (chunked path)
    long long chunk;   // particles per chunk
    size_t bytes;      // workspace bytes
    size_t smem;       // dynamic shared memory of count / scatter
};

Plan make_plan(const TileGrid &tg, long long n) {
    Plan p{};
    p.B = (unsigned)(tg.n_tiles + 1);
    p.chunked = p.B <= kSmemBins;
    if (p.chunked) {
        p.smem = (size_t)p.B * sizeof(unsigned);
        // resident CTAs per SM allowed by shared memory (228 KB per SM, 1 KB reserved per CTA)
        long long per_sm = (228 * 1024) / (long long)(p.smem + 1024);
        if (per_sm < 1) per_sm = 1;
        if (per_sm > 4) per_sm = 4;
        long long G = (long long)kNumSMs * per_sm;
        long long max_g = (n + 1023) / 1024;  // at least ~1024 particles per chunk
        if (max_g < 1) max_g = 1;
        if (G > max_g) G = max_g;
        p.G = (unsigned)G;
        p.chunk = (n + G - 1) / G;
        if (p.chunk < 1) p.chunk = 1;
        p.bytes = align_up((size_t)G * p.B * sizeof(unsigned), 256) +
                  align_up((size_t)p.B * sizeof(unsigned), 256);
    } else {
        p.smem = 0;
        p.G = 0;
        p.chunk = 0;
        p.bytes = 2 * align_up((size_t)p.B * sizeof(unsigned), 256);
    }
    return p;
}

template <int DIM, int TILE>
pcg_status run_sort(const TileGrid &tg, const Plan &pl, long long n, const float *const *kp,
                    const Payload &py, int np, uint32_t *offs, unsigned long long *n_invalid,
                    unsigned char *ws, cudaStream_t s) {
    KeyGeom g;
    g.nt0 = tg.nt[0];
    g.nt1 = tg.nt[1];
    g.n_tiles = (unsigned)tg.n_tiles;
    g.N0 = (float)tg.N[0];
    g.N1 = (float)tg.N[1];
    g.N2 = (float)tg.N[2];
    g.tile = tg.tile;
    const float *kz = DIM == 3 ? kp[2] : kp[0];
    if (pl.chunked) {
        unsigned *counts = reinterpret_cast<unsigned *>(ws);
        unsigned *totals = reinterpret_cast<unsigned *>(
            ws + align_up((size_t)pl.G * pl.B * sizeof(unsigned), 256));
        if (pl.smem > 48 * 1024) {
            PCG_CHECK_CUDA(cudaFuncSetAttribute(count_chunked_kernel<DIM, TILE>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                (int)pl.smem));
            PCG_CHECK_CUDA(cudaFuncSetAttribute(scatter_chunked_kernel<DIM, TILE>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                (int)pl.smem));
        }
        {
            prof::Mark mk("sort_count", s);
            count_chunked_kernel<DIM, TILE><<<pl.G, kSortThreads, pl.smem, s>>>(
                g, kp[0], kp[1], kz, n, pl.chunk, counts, pl.B, n_invalid);
        }
        PCG_CHECK_LAUNCH();
        {
            prof::Mark mk("sort_colscan", s);
            colscan_kernel<<<(pl.B + 255) / 256, 256, 0, s>>>(counts, totals, pl.G, pl.B);
        }
        PCG_CHECK_LAUNCH();
        {
            prof::Mark mk("sort_scan", s);
            scan_one_cta_kernel<<<1, 1024, 0, s>>>(totals, offs, nullptr, pl.B);
        }
        PCG_CHECK_LAUNCH();
        prof::Mark mk("sort_scatter", s);
        scatter_chunked_kernel<DIM, TILE><<<pl.G, kSortThreads, pl.smem, s>>>(
            g, kp[0], kp[1], kz, n, pl.chunk, counts, offs, pl.B, py, np);
        return launch_status();
    }
    unsigned *totals = reinterpret_cast<unsigned *>(ws);
    unsigned *cursor =
        reinterpret_cast<unsigned *>(ws + align_up((size_t)pl.B * sizeof(unsigned), 256));
    pcg_status st = zero_f32(reinterpret_cast<float *>(totals), pl.B, s);
    if (st != PCG_OK) return st;
    const unsigned grid = (unsigned)kNumSMs * 8;
    {
        prof::Mark mk("sort_count_global", s);
        count_global_kernel<DIM, TILE><<<grid, 256, 0, s>>>(g, kp[0], kp[1], kz, n, totals, n_invalid);
    }
    PCG_CHECK_LAUNCH();
    {
        prof::Mark mk("sort_scan", s);
        scan_one_cta_kernel<<<1, 1024, 0, s>>>(totals, offs, cursor, pl.B);
    }
    PCG_CHECK_LAUNCH();
    prof::Mark mk("sort_scatter_global", s);
    scatter_global_kernel<DIM, TILE><<<grid, 256, 0, s>>>(g, kp[0], kp[1], kz, n, cursor, py, np);
    return launch_status();
}

template <int DIM>
pcg_status dispatch_tile(const TileGrid &tg, const Plan &pl, long long n, const float *const *kp,
                         const Payload &py, int np, uint32_t *offs, unsigned long long *ni,
                         unsigned char *ws, cudaStream_t s) {
    switch (tg.tile) {
        case 1: return run_sort<DIM, 1>(tg, pl, n, kp, py, np, offs, ni, ws, s);
        case 4: return run_sort<DIM, 4>(tg, pl, n, kp, py, np, offs, ni, ws, s);
        case 8: return run_sort<DIM, 8>(tg, pl, n, kp, py, np, offs, ni, ws, s);
        default: return run_sort<DIM, 0>(tg, pl, n, kp, py, np, offs, ni, ws, s);
    }
}

bool valid_sort_args(int32_t dim, const int32_t *grid, int32_t tile, int64_t n, TileGrid *tg) {
    if (n < 0 || n >= 0xffffffffll) return false;
    if (tile < 1 || tile > 64) return false;
    return make_tile_grid(dim, grid, tile, tg);
}

}  // namespace
}  // namespace pcg

extern "C" pcg_status pcg_tile_sort_workspace_size(int32_t dim, const int32_t *grid, int32_t tile,
                                                   int64_t n, size_t *bytes) {
    using namespace pcg;
    TileGrid tg;
    if (bytes == nullptr || !valid_sort_args(dim, grid, tile, n, &tg)) return PCG_ERR_INVALID_ARG;
    *bytes = make_plan(tg, n).bytes;
    return PCG_OK;
}

extern "C" pcg_status pcg_tile_sort(int32_t dim, const int32_t *grid, int32_t tile, int64_t n,
                                    const float *const *key_pos, int32_t n_payload,
                                    const void *const *payload_in, void *const *payload_out,
                                    uint32_t *tile_offsets, pcg_stats *stats, void *workspace,
                                    size_t workspace_bytes, void *stream) {
    using namespace pcg;
    TileGrid tg;
    if (!valid_sort_args(dim, grid, tile, n, &tg)) return PCG_ERR_INVALID_ARG;
    if (tile_offsets == nullptr || key_pos == nullptr) return PCG_ERR_INVALID_ARG;
    if (n_payload < 1 || n_payload > kMaxPayload || payload_in == nullptr || payload_out == nullptr)
        return PCG_ERR_INVALID_ARG;
    Payload py{};
    for (int f = 0; f < n_payload; ++f) {
        if (n > 0 && (payload_in[f] == nullptr || payload_out[f] == nullptr))
            return PCG_ERR_INVALID_ARG;
        py.in[f] = static_cast<const unsigned *>(payload_in[f]);
        py.out[f] = static_cast<unsigned *>(payload_out[f]);
    }
    for (int mu = 0; mu < dim; ++mu)
        if (n > 0 && key_pos[mu] == nullptr) return PCG_ERR_INVALID_ARG;
    const Plan pl = make_plan(tg, n);
    if (workspace_bytes < pl.bytes || (pl.bytes > 0 && workspace == nullptr))
        return PCG_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return PCG_ERR_WORKSPACE;
    cudaStream_t s = as_stream(stream);
    if (n == 0) return zero_f32(reinterpret_cast<float *>(tile_offsets), (size_t)tg.n_tiles + 1, s);
    unsigned long long *ni = stats ? &stats->n_invalid : nullptr;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    return dim == 2 ? dispatch_tile<2>(tg, pl, n, key_pos, py, n_payload, tile_offsets, ni, ws, s)
                    : dispatch_tile<3>(tg, pl, n, key_pos, py, n_payload, tile_offsets, ni, ws, s);
}
