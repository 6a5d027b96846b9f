// deposit_zigzag.cu -- charge-conserving zigzag current deposit (3D, CIC charge).
//
// Method.  "Tiled current deposit" (Entity wiki), section "Halo sizing", names
// the O == 0 zigzag deposit: it writes at most 2 cells above min(i, i_prev).
// The scheme is the relay split of Umeda, Omura, Tominaga & Matsumoto, Comput.
// Phys. Commun. 156 (2003) 73.  Per axis, with cells i1 = floor(x1),
// i2 = floor(x2) (|i2 - i1| <= 1 after the periodic minimum image):
//   relay  xr = min(min(i1, i2) + 1, max(max(i1, i2), (x1 + x2) / 2)),
//   moves  D1 = xr - x1,  D2 = x2 - xr,  fluxes F_s = q D_s / dt,
//   shape  W1 = (x1 + xr) / 2 - i1,  W2 = (xr + x2) / 2 - i2.
// Segment s adds to J^c on the four c-edges of its cell that start at
// (cell + a e_u + b e_v), u and v the transverse axes, the flux F_s^c times
//   w_a(W_s^u) w_b(W_s^v) + (a == b ? 1 : -1) D_s^u D_s^v / 12,
// w_0(W) = 1 - W, w_1(W) = W: the bilinear weight averaged along the straight
// segment, which keeps (rho(x2) - rho(x1)) / dt + div J = 0 exact in 3D (the
// D D / 12 term vanishes when a segment moves along at most two axes, where
// the weight is Umeda's midpoint one).  J[c] at node index (k*Ny + j)*Nx + i is
// the c-current on the edge from node (i, j, k) towards +e_c.
//
// Tiled path ("How a tile deposit runs", "Halo sizing", "Correctness is
// independent of the halo").  The particles are sorted by the tile of their
// previous position (the page keys on min(i, i_prev) to put the whole halo on
// the high side; the previous cell is at most one cell above that minimum, so a
// halo of 2 on both sides holds every stencil of a particle that has not left
// its tile).  Each CTA owns a fixed-size chunk of the sorted array; for every
// tile segment inside it, it zeroes a 3 x (T + 4)^3 scratch window in shared
// memory, adds each particle's edges there with shared-memory reductions when
// its 3 x 3 x 3 node footprint fits the window, or sends the whole particle to
// J with global reductions when it does not (the escape valve), and flushes
// the window once.
#include "deposit_tiled.cuh"

namespace pcg {
namespace {

using dep::Counters;
using dep::Geom;

struct ZParticles {
    const float *x1[3];  // previous positions
    const float *x2[3];  // current positions
    const float *q;
};

// One particle's zigzag split: the lower cell of the move (per axis, in
// [-1, N)), each segment's cell relative to it (0 or 1), the fluxes, the
// segment midpoints relative to their cells and the segment moves.
struct Zig {
    int base[3];
    int cell[2][3];
    float F[2][3], W[2][3], D[2][3];
    bool same;  // both segments in one cell
};

__device__ __forceinline__ bool zigzag_split(const Geom &g, const float (&x1)[3], const float (&x2)[3], float q,
                                             float inv_dt, Zig &z) {
    bool ok = true;
    z.same = true;
#pragma unroll
    for (int mu = 0; mu < 3; ++mu) {
        const float a1 = x1[mu], a2 = x2[mu];
        ok &= (a1 >= 0.f) & (a1 < g.Nf[mu]) & (a2 >= 0.f) & (a2 < g.Nf[mu]);
        const int i1 = (int)a1, i2 = (int)a2;  // floor: both are >= 0 when ok
        int di = i2 - i1;                       // periodic minimum image
        if (2 * di > g.N[mu]) di -= g.N[mu];
        if (2 * di < -g.N[mu]) di += g.N[mu];
        ok &= (di >= -1) & (di <= 1);
        const int lo = di < 0 ? di : 0;
        const int a = -lo, b = di - lo;
        const float X1 = (float)a + (a1 - (float)i1);
        const float X2 = (float)b + (a2 - (float)i2);
        const float xr = fminf(1.f, fmaxf((float)(a > b ? a : b), 0.5f * (X1 + X2)));
        z.base[mu] = i1 + lo;
        z.cell[0][mu] = a;
        z.cell[1][mu] = b;
        z.same &= a == b;
        z.D[0][mu] = xr - X1;
        z.D[1][mu] = X2 - xr;
        z.F[0][mu] = q * z.D[0][mu] * inv_dt;
        z.F[1][mu] = q * z.D[1][mu] * inv_dt;
        z.W[0][mu] = 0.5f * (X1 + xr) - (float)a;
        z.W[1][mu] = 0.5f * (xr + X2) - (float)b;
    }
    return ok;
}

// The four edge weights of component c for segment s, times its flux:
// out[b][a] for the edge at cell + a e_u + b e_v.
template <int C>
__device__ __forceinline__ void edge_values(const Zig &z, int s, float (&out)[2][2]) {
    constexpr int U = (C + 1) % 3, V = (C + 2) % 3;
    const float wu = z.W[s][U], wv = z.W[s][V];
    const float avg = z.D[s][U] * z.D[s][V] * (1.f / 12.f);
    const float F = z.F[s][C];
    out[0][0] = F * ((1.f - wu) * (1.f - wv) + avg);
    out[0][1] = F * (wu * (1.f - wv) - avg);
    out[1][0] = F * ((1.f - wu) * wv - avg);
    out[1][1] = F * (wu * wv + avg);
}

// Visit the 12 (same cell) or 24 edge values of a particle:
// put(c, dx, dy, dz, value) with (dx, dy, dz) the edge's start node relative
// to base, each in {0, 1, 2}.
template <class Put>
__device__ __forceinline__ void zigzag_edges(const Zig &z, Put put) {
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        if (s == 1 && z.same) break;
        const int cx = z.cell[s][0], cy = z.cell[s][1], cz = z.cell[s][2];
        float v[2][2];
        // J^x: edges (cx, cy + a, cz + b)
        edge_values<0>(z, s, v);
        if (z.same) {
            float w[2][2];
            edge_values<0>(z, 1, w);
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i >> 1][i & 1] += w[i >> 1][i & 1];
        }
#pragma unroll
        for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int a = 0; a < 2; ++a) put(0, cx, cy + a, cz + b, v[b][a]);
        // J^y: U = z, V = x: edges (cx + b, cy, cz + a)
        edge_values<1>(z, s, v);
        if (z.same) {
            float w[2][2];
            edge_values<1>(z, 1, w);
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i >> 1][i & 1] += w[i >> 1][i & 1];
        }
#pragma unroll
        for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int a = 0; a < 2; ++a) put(1, cx + b, cy, cz + a, v[b][a]);
        // J^z: U = x, V = y: edges (cx + a, cy + b, cz)
        edge_values<2>(z, s, v);
        if (z.same) {
            float w[2][2];
            edge_values<2>(z, 1, w);
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i >> 1][i & 1] += w[i >> 1][i & 1];
        }
#pragma unroll
        for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int a = 0; a < 2; ++a) put(2, cx + a, cy + b, cz, v[b][a]);
    }
}

__device__ __forceinline__ int wrap_once(int i, int N) { return i < 0 ? i + N : (i >= N ? i - N : i); }

// All edges of one particle into J with global reductions (periodic wrap).
__device__ __forceinline__ void zigzag_global(const Geom &g, float *__restrict__ J, const Zig &z) {
    zigzag_edges(z, [&](int c, int dx, int dy, int dz, float v) {
        // base in [-1, N), d <= 2 and N >= 3: at most one correction
        const int gx = wrap_once(z.base[0] + dx, g.N[0]);
        const int gy = wrap_once(z.base[1] + dy, g.N[1]);
        const int gz = wrap_once(z.base[2] + dz, g.N[2]);
        const long long node = ((long long)gz * g.N[1] + gy) * g.N[0] + gx;
        if (PCG_IN(node, g.ncells)) red_add_f32(J + c * g.ncells + node, v);
    });
}

__device__ __forceinline__ void load_particle(const ZParticles &P, long long p, float (&x1)[3], float (&x2)[3],
                                              float &q) {
#pragma unroll
    for (int mu = 0; mu < 3; ++mu) {
        x1[mu] = P.x1[mu][p];
        x2[mu] = P.x2[mu][p];
    }
    q = P.q[p];
}

__global__ void __launch_bounds__(256)
    zigzag_flat_kernel(Geom g, ZParticles P, long long n, float inv_dt, float *__restrict__ J, Counters ctr) {
    unsigned n_inv = 0;
    for (long long p = blockIdx.x * (long long)blockDim.x + threadIdx.x; p < n;
         p += (long long)gridDim.x * blockDim.x) {
        float x1[3], x2[3], q;
        load_particle(P, p, x1, x2, q);
        Zig z;
        if (!zigzag_split(g, x1, x2, q, inv_dt, z)) {
            ++n_inv;
            continue;
        }
        zigzag_global(g, J, z);
    }
    warp_add_u64(ctr.n_invalid, n_inv);
}

// General path of one particle in a tile segment: the full split, then its
// 12 or 24 edges into the scratch window when its 3 x 3 x 3 footprint fits,
// else into J (the escape valve).  Out of line: it serves the cell-crossing
// particles, which the hot loop of the tiled kernel only lists.
template <int TILE, int HALO>
__device__ __noinline__ void zigzag_general(const Geom g, const ZParticles P, long long p, float inv_dt,
                                            float *scratch, float *J, int ox, int oy, int oz, unsigned *n_esc) {
    using C = dep::TileCfg<3, 1, TILE, HALO>;
    constexpr int TE = C::TE;
    float x1[3], x2[3], q;
    load_particle(P, p, x1, x2, q);
    Zig z;
    if (!zigzag_split(g, x1, x2, q, inv_dt, z)) return;  // counted by the caller
    const int lx = dep::local_index<3, TILE, HALO>(z.base[0], ox, g.N[0]);
    const int ly = dep::local_index<3, TILE, HALO>(z.base[1], oy, g.N[1]);
    const int lz = dep::local_index<3, TILE, HALO>(z.base[2], oz, g.N[2]);
    const bool fits = (lx >= -HALO) & (lx + 2 < TILE + HALO) & (ly >= -HALO) & (ly + 2 < TILE + HALO) &
                      (lz >= -HALO) & (lz + 2 < TILE + HALO);
    if (!fits) {
        ++*n_esc;
        zigzag_global(g, J, z);
        return;
    }
    const int b0 = ((lz + HALO) * TE + (ly + HALO)) * TE + (lx + HALO);
    if (!PCG_IN(b0, C::CELLS) || !PCG_IN(b0 + (2 * TE + 2) * TE + 2, C::CELLS)) return;
    float *w0 = scratch + b0;
    zigzag_edges(z, [&](int c, int dx, int dy, int dz, float v) {
        red_shared_add_f32(w0 + c * C::CELLS + (dz * TE + dy) * TE + dx, v);
    });
}

// Tiled kernel.  Each round gives every thread one particle.  A particle that
// stays inside its cell moves along a straight line, so its two zigzag
// segments add up to the single-segment current: with f1, f2 its offsets in
// the cell, D = f2 - f1, m = (f1 + f2) / 2 and F = q D / dt, the c-edges at
// (cell + a e_u + b e_v) get F^c (w_a(m^u) w_b(m^v) + (a == b ? 1 : -1) D^u D^v / 12),
// 12 shared reductions from a few multiplies.  Particles that cross a cell
// face (about 11 % at v ~ N(0, 0.05^2)) are only listed, and taken after the
// loop by the general path in compact warps, so that the loop's warps stay
// converged and issue 12 reductions per particle instead of 24.
constexpr int kCrossCap = 2048;

template <int TILE, int HALO>
__global__ void __launch_bounds__(256, 3)
    zigzag_tiled_kernel(Geom g, ZParticles P, long long n, float inv_dt, const uint32_t *__restrict__ offs,
                        const unsigned *__restrict__ chunk_tile, long long chunk, float *__restrict__ J,
                        Counters ctr) {
    using C = dep::TileCfg<3, 1, TILE, HALO>;
    constexpr int TE = C::TE;
    extern __shared__ __align__(16) float scratch[];  // [3][CELLS]
    __shared__ unsigned cross[kCrossCap];             // segment-relative indices of crossing particles
    __shared__ unsigned n_cross;

    const int lane = threadIdx.x & 31;
    const long long c0 = (long long)blockIdx.x * chunk;
    const long long c1 = min(n, c0 + chunk);
    unsigned n_esc = 0, n_inv = 0;
    unsigned t = chunk_tile[blockIdx.x];
    if (t > g.n_tiles) t = g.n_tiles;
    for (;; ++t) {
        long long s = (long long)offs[t];
        if (s < c0) s = c0;
        if (s >= c1) break;
        long long e = (t < g.n_tiles) ? (long long)offs[t + 1] : c1;
        if (e > c1) e = c1;
        if (t == g.n_tiles) {
            // tail pass: slots after the last tile go straight to J
            for (long long p = s + threadIdx.x; p < e; p += 256) {
                float x1[3], x2[3], q;
                load_particle(P, p, x1, x2, q);
                Zig z;
                if (!zigzag_split(g, x1, x2, q, inv_dt, z)) {
                    ++n_inv;
                    continue;
                }
                zigzag_global(g, J, z);
            }
            break;
        }
        if (e <= s) continue;  // empty tile
        const int tx = (int)(t % (unsigned)g.nt[0]);
        const int ty = (int)((t / (unsigned)g.nt[0]) % (unsigned)g.nt[1]);
        const int tz = (int)(t / ((unsigned)g.nt[0] * (unsigned)g.nt[1]));
        const int ox = tx * TILE, oy = ty * TILE, oz = tz * TILE;

        for (int i = threadIdx.x; i < C::FLOATS; i += 256) scratch[i] = 0.f;
        if (threadIdx.x == 0) n_cross = 0;
        __syncthreads();

        for (long long r = s; r < e; r += 256) {
            const long long p = r + threadIdx.x;
            const bool live = p < e;
            float x1[3], x2[3], q = 0.f;
            if (live) load_particle(P, p, x1, x2, q);
            bool ok = live, same = true;
            int ic[3];
            float f1[3], f2[3];
#pragma unroll
            for (int mu = 0; mu < 3; ++mu) {
                const float a1 = live ? x1[mu] : 0.f, a2 = live ? x2[mu] : 0.f;
                ok &= (a1 >= 0.f) & (a1 < g.Nf[mu]) & (a2 >= 0.f) & (a2 < g.Nf[mu]);
                const int i1 = (int)a1, i2 = (int)a2;
                int di = i2 - i1;
                if (2 * di > g.N[mu]) di -= g.N[mu];
                if (2 * di < -g.N[mu]) di += g.N[mu];
                ok &= (di >= -1) & (di <= 1);
                same &= di == 0;
                ic[mu] = i1;
                f1[mu] = a1 - (float)i1;
                f2[mu] = a2 - (float)i2;
            }
            n_inv += live & !ok;
            const bool crossing = ok & !same;
            const unsigned m = __ballot_sync(0xffffffffu, crossing);
            if (m != 0u) {
                unsigned base = 0;
                if (lane == 0) base = atomicAdd(&n_cross, (unsigned)__popc(m));
                base = __shfl_sync(0xffffffffu, base, 0);
                if (crossing) {
                    const unsigned slot = base + __popc(m & ((1u << lane) - 1u));
                    if (slot < kCrossCap) cross[slot] = (unsigned)(p - s);
                    else zigzag_general<TILE, HALO>(g, P, p, inv_dt, scratch, J, ox, oy, oz, &n_esc);
                }
            }
            if (!(ok & same)) continue;
            const int lx = dep::local_index<2, TILE, HALO>(ic[0], ox, g.N[0]);
            const int ly = dep::local_index<2, TILE, HALO>(ic[1], oy, g.N[1]);
            const int lz = dep::local_index<2, TILE, HALO>(ic[2], oz, g.N[2]);
            const bool fits = (lx >= -HALO) & (lx + 1 < TILE + HALO) & (ly >= -HALO) & (ly + 1 < TILE + HALO) &
                              (lz >= -HALO) & (lz + 1 < TILE + HALO);
            if (!fits) {
                zigzag_general<TILE, HALO>(g, P, p, inv_dt, scratch, J, ox, oy, oz, &n_esc);
                continue;
            }
            float D[3], mid[3], F[3];
#pragma unroll
            for (int mu = 0; mu < 3; ++mu) {
                D[mu] = f2[mu] - f1[mu];
                mid[mu] = 0.5f * (f1[mu] + f2[mu]);
                F[mu] = q * D[mu] * inv_dt;
            }
            const int b0 = ((lz + HALO) * TE + (ly + HALO)) * TE + (lx + HALO);
            if (!PCG_IN(b0, C::CELLS) || !PCG_IN(b0 + (TE + 1) * TE + 1, C::CELLS)) continue;
            float *w0 = scratch + b0;
#pragma unroll
            for (int c = 0; c < 3; ++c) {
                const int u = (c + 1) % 3, v = (c + 2) % 3;
                const float wu = mid[u], wv = mid[v];
                const float avg = D[u] * D[v] * (1.f / 12.f);
                const float val[2][2] = {{F[c] * ((1.f - wu) * (1.f - wv) + avg), F[c] * (wu * (1.f - wv) - avg)},
                                         {F[c] * ((1.f - wu) * wv - avg), F[c] * (wu * wv + avg)}};
                // the edge at cell + a e_u + b e_v
                constexpr int stride[3] = {1, TE, TE * TE};
#pragma unroll
                for (int b = 0; b < 2; ++b)
#pragma unroll
                    for (int a = 0; a < 2; ++a)
                        red_shared_add_f32(w0 + c * C::CELLS + a * stride[u] + b * stride[v], val[b][a]);
            }
        }
        __syncthreads();
        const unsigned nc = min(n_cross, (unsigned)kCrossCap);
        for (unsigned i = threadIdx.x; i < nc; i += 256)
            zigzag_general<TILE, HALO>(g, P, s + cross[i], inv_dt, scratch, J, ox, oy, oz, &n_esc);
        __syncthreads();
        dep::flush_scratch<3, TILE, HALO, 256>(g, scratch, J, ox, oy, oz);
        __syncthreads();
    }
    warp_add_u64(ctr.n_escaped, n_esc);
    warp_add_u64(ctr.n_invalid, n_inv);
}

}  // namespace
}  // namespace pcg

extern "C" pcg_status pcg_deposit_zigzag(const int32_t *grid, int32_t tile, int64_t n, const float *const *pos_prev,
                                         const float *const *pos, const float *q, double dt,
                                         const uint32_t *tile_offsets, float *J, pcg_stats *stats, void *workspace,
                                         size_t workspace_bytes, void *stream) {
    using namespace pcg;
    const bool tiled = tile_offsets != nullptr;
    if (n < 0 || n >= 0xffffffffll || grid == nullptr) return PCG_ERR_INVALID_ARG;
    for (int mu = 0; mu < 3; ++mu)
        if (grid[mu] < 3) return PCG_ERR_INVALID_ARG;
    if (!(dt > 0.0) || !(dt < 1e300)) return PCG_ERR_INVALID_ARG;
    if (tiled && tile != 8) return tile < 1 || tile > 64 ? PCG_ERR_INVALID_ARG : PCG_ERR_UNSUPPORTED;
    Geom g;
    if (!geom_from(3, grid, tiled ? tile : 1, &g)) return PCG_ERR_INVALID_ARG;
    if (J == nullptr || !aligned16(J)) return PCG_ERR_INVALID_ARG;
    ZParticles P{};
    if (n > 0) {
        if (pos_prev == nullptr || pos == nullptr || q == nullptr) return PCG_ERR_INVALID_ARG;
        for (int mu = 0; mu < 3; ++mu) {
            if (pos_prev[mu] == nullptr || pos[mu] == nullptr) return PCG_ERR_INVALID_ARG;
            P.x1[mu] = pos_prev[mu];
            P.x2[mu] = pos[mu];
        }
        P.q = q;
    }
    const long long chunk = chunk_for(n);
    const long long nchunks = (n + chunk - 1) / chunk;
    const size_t need = tiled ? align_up((size_t)nchunks * sizeof(unsigned), 256) : 0;
    if (workspace_bytes < need || (need > 0 && workspace == nullptr)) return PCG_ERR_WORKSPACE;

    cudaStream_t s = as_stream(stream);
    Counters ctr{stats ? &stats->n_escaped : nullptr, stats ? &stats->n_invalid : nullptr,
                 stats ? &stats->error_flags : nullptr};
    unsigned *chunk_tile = static_cast<unsigned *>(workspace);
    pcg_status st = launch_prep(J, g, tiled ? tile_offsets : nullptr, n, chunk, chunk_tile, ctr.flags, s);
    if (st != PCG_OK || n == 0) return st;
    const float inv_dt = (float)(1.0 / dt);
    if (!tiled) {
        const long long want = (n + 255) / 256;
        const long long cap = (long long)num_sms() * 16;
        prof::Mark mk("deposit_zigzag_flat", s);
        zigzag_flat_kernel<<<(unsigned)(want < cap ? want : cap), 256, 0, s>>>(g, P, n, inv_dt, J, ctr);
        return launch_status();
    }
    using C = dep::TileCfg<3, 1, 8, 2>;
    const size_t smem = C::FLOATS * sizeof(float);
    prof::Mark mk("deposit_zigzag", s);
    zigzag_tiled_kernel<8, 2><<<(unsigned)nchunks, 256, smem, s>>>(g, P, n, inv_dt, tile_offsets, chunk_tile, chunk,
                                                                    J, ctr);
    return launch_status();
}
