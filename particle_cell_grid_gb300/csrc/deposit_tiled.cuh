// deposit_tiled.cuh -- the tiled deposit kernel template (instantiated per
// dimension in deposit_2d.cu and deposit_3d.cu to keep compile units small).
#pragma once

#include "deposit.cuh"

namespace pcg {
namespace dep {

template <int DIM, int ORDER, int TILE, int HALO>
struct TileCfg {
    static constexpr int S = ORDER + 1;                 // stencil nodes per axis
    static constexpr int TE = TILE + 2 * HALO;          // scratch edge
    static constexpr int TEZ = DIM == 3 ? TE : 1;
    static constexpr int CELLS = TE * TE * TEZ;         // scratch nodes
    static constexpr int FLOATS = 3 * CELLS;
};

// Deposit one particle of tile (ox, oy, oz) into the scratch window, or escape.
template <int DIM, int ORDER, int TILE, int HALO>
__device__ __forceinline__ void deposit_one(const Geom &g, float *__restrict__ scratch,
                                            float *__restrict__ J, int ox, int oy, int oz, float x,
                                            float y, float z, float vx, float vy, float vz, float q,
                                            unsigned &n_esc, unsigned &n_inv) {
    using C = TileCfg<DIM, ORDER, TILE, HALO>;
    constexpr int S = C::S;
    if (!in_domain<DIM>(g, x, y, z)) {
        ++n_inv;
        return;
    }
    const float qvx = q * vx, qvy = q * vy, qvz = q * vz;
    float wx[S], wy[S], wz[S];
    const int fx = axis_weights<ORDER>(x, wx);
    const int fy = axis_weights<ORDER>(y, wy);
    int fz = 0;
    if (DIM == 3) fz = axis_weights<ORDER>(z, wz);
    else wz[0] = 1.f;
    const int lx = local_index<S, TILE, HALO>(fx, ox, g.N[0]);
    const int ly = local_index<S, TILE, HALO>(fy, oy, g.N[1]);
    const int lz = DIM == 3 ? local_index<S, TILE, HALO>(fz, oz, g.N[2]) : 0;
    // fit test: every stencil node inside [-HALO, TILE + HALO) on every axis
    bool fits = (lx >= -HALO) & (lx + S - 1 < TILE + HALO) & (ly >= -HALO) &
                (ly + S - 1 < TILE + HALO);
    if (DIM == 3) fits &= (lz >= -HALO) & (lz + S - 1 < TILE + HALO);
    if (!fits) {
        ++n_esc;
        deposit_global<DIM, ORDER>(g, J, x, y, z, qvx, qvy, qvz);
        return;
    }
    constexpr int SZ = DIM == 3 ? S : 1;
    const int base = ((DIM == 3 ? (lz + HALO) * C::TE : 0) + (ly + HALO)) * C::TE + (lx + HALO);
#pragma unroll
    for (int kz = 0; kz < SZ; ++kz) {
#pragma unroll
        for (int ky = 0; ky < S; ++ky) {
            const float wyz = wy[ky] * wz[kz];
            float *row = scratch + base + (kz * C::TE + ky) * C::TE;
#pragma unroll
            for (int kx = 0; kx < S; ++kx) {
                const float W = wyz * wx[kx];
                red_shared_add_f32(row + kx, qvx * W);
                red_shared_add_f32(row + C::CELLS + kx, qvy * W);
                red_shared_add_f32(row + 2 * C::CELLS + kx, qvz * W);
            }
        }
    }
}

template <int DIM, int ORDER, int TILE, int HALO>
__global__ void __launch_bounds__(512)
    deposit_tiled_kernel(Geom g, Particles P, long long n, const uint32_t *__restrict__ offs,
                         const unsigned *__restrict__ chunk_tile, long long chunk,
                         float *__restrict__ J, Counters ctr, bool vec4) {
    using C = TileCfg<DIM, ORDER, TILE, HALO>;
    __shared__ float scratch[C::FLOATS];
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
            for (long long p = s + threadIdx.x; p < e; p += blockDim.x) {
                const float x = P.x[p], y = P.y[p], z = DIM == 3 ? P.z[p] : 0.f;
                if (!in_domain<DIM>(g, x, y, z)) {
                    ++n_inv;
                    continue;
                }
                const float q = P.q[p];
                deposit_global<DIM, ORDER>(g, J, x, y, z, q * P.vx[p], q * P.vy[p], q * P.vz[p]);
            }
            break;
        }
        if (e <= s) continue;  // empty tile
        const int tx = (int)(t % (unsigned)g.nt[0]);
        const int ty = (int)((t / (unsigned)g.nt[0]) % (unsigned)g.nt[1]);
        const int tz = DIM == 3 ? (int)(t / ((unsigned)g.nt[0] * (unsigned)g.nt[1])) : 0;
        const int ox = tx * TILE, oy = ty * TILE, oz = tz * TILE;

        for (int i = threadIdx.x; i < C::FLOATS; i += blockDim.x) scratch[i] = 0.f;
        __syncthreads();

        if (vec4) {
            // groups of four consecutive slots, 16-byte loads; slots outside [s, e) masked
            const long long g0 = s >> 2, g1 = (e + 3) >> 2;
            for (long long gi = g0 + threadIdx.x; gi < g1; gi += blockDim.x) {
                const long long p = gi << 2;
                float xs[4], ys[4], zs[4], vxs[4], vys[4], vzs[4], qs[4];
                if (p + 3 < n) {
                    const float4 a = *reinterpret_cast<const float4 *>(P.x + p);
                    const float4 b = *reinterpret_cast<const float4 *>(P.y + p);
                    const float4 c = DIM == 3 ? *reinterpret_cast<const float4 *>(P.z + p)
                                              : make_float4(0.f, 0.f, 0.f, 0.f);
                    const float4 d = *reinterpret_cast<const float4 *>(P.vx + p);
                    const float4 f = *reinterpret_cast<const float4 *>(P.vy + p);
                    const float4 h = *reinterpret_cast<const float4 *>(P.vz + p);
                    const float4 k = *reinterpret_cast<const float4 *>(P.q + p);
                    xs[0] = a.x; xs[1] = a.y; xs[2] = a.z; xs[3] = a.w;
                    ys[0] = b.x; ys[1] = b.y; ys[2] = b.z; ys[3] = b.w;
                    zs[0] = c.x; zs[1] = c.y; zs[2] = c.z; zs[3] = c.w;
                    vxs[0] = d.x; vxs[1] = d.y; vxs[2] = d.z; vxs[3] = d.w;
                    vys[0] = f.x; vys[1] = f.y; vys[2] = f.z; vys[3] = f.w;
                    vzs[0] = h.x; vzs[1] = h.y; vzs[2] = h.z; vzs[3] = h.w;
                    qs[0] = k.x; qs[1] = k.y; qs[2] = k.z; qs[3] = k.w;
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const long long pj = p + j < n ? p + j : n - 1;
                        xs[j] = P.x[pj]; ys[j] = P.y[pj]; zs[j] = DIM == 3 ? P.z[pj] : 0.f;
                        vxs[j] = P.vx[pj]; vys[j] = P.vy[pj]; vzs[j] = P.vz[pj]; qs[j] = P.q[pj];
                    }
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const long long pj = p + j;
                    if (pj < s || pj >= e) continue;
                    deposit_one<DIM, ORDER, TILE, HALO>(g, scratch, J, ox, oy, oz, xs[j], ys[j],
                                                        zs[j], vxs[j], vys[j], vzs[j], qs[j],
                                                        n_esc, n_inv);
                }
            }
        } else {
            for (long long p = s + threadIdx.x; p < e; p += blockDim.x) {
                deposit_one<DIM, ORDER, TILE, HALO>(g, scratch, J, ox, oy, oz, P.x[p], P.y[p],
                                                    DIM == 3 ? P.z[p] : 0.f, P.vx[p], P.vy[p],
                                                    P.vz[p], P.q[p], n_esc, n_inv);
            }
        }
        __syncthreads();

        // flush: one global reduction per non-zero scratch cell, periodic wrap
        for (int i = threadIdx.x; i < C::FLOATS; i += blockDim.x) {
            const float val = scratch[i];
            if (val == 0.f) continue;
            const int c = i / C::CELLS;
            const int r = i - c * C::CELLS;
            const int sx = r % C::TE;
            const int sy = (r / C::TE) % C::TE;
            const int sz = DIM == 3 ? r / (C::TE * C::TE) : 0;
            const int gx = wrap_index(ox - HALO + sx, g.N[0]);
            const int gy = wrap_index(oy - HALO + sy, g.N[1]);
            const int gz = DIM == 3 ? wrap_index(oz - HALO + sz, g.N[2]) : 0;
            red_add_f32(J + c * g.ncells + ((long long)gz * g.N[1] + gy) * g.N[0] + gx, val);
        }
        __syncthreads();  // scratch is reused by the next segment
    }
    warp_add_u64(ctr.n_escaped, n_esc);
    warp_add_u64(ctr.n_invalid, n_inv);
}

template <int DIM, int ORDER, int TILE, int HALO>
pcg_status launch_tiled(const Geom &g, long long n, const Particles &P, const uint32_t *offs,
                        float *J, const Counters &ctr, const unsigned *chunk_tile, long long chunk,
                        int block, cudaStream_t s) {
    const long long nchunks = (n + chunk - 1) / chunk;
    if (nchunks == 0) return PCG_OK;
    const bool vec4 = aligned16(P.x) && aligned16(P.y) && (DIM == 2 || aligned16(P.z)) &&
                      aligned16(P.vx) && aligned16(P.vy) && aligned16(P.vz) && aligned16(P.q);
    prof::Mark mk("deposit_tiled", s);
    deposit_tiled_kernel<DIM, ORDER, TILE, HALO>
        <<<(unsigned)nchunks, block, 0, s>>>(g, P, n, offs, chunk_tile, chunk, J, ctr, vec4);
    return launch_status();
}

template <int DIM, int ORDER, int TILE>
pcg_status dispatch_halo(int halo, const Geom &g, long long n, const Particles &P,
                         const uint32_t *offs, float *J, const Counters &ctr,
                         const unsigned *chunk_tile, long long chunk, int block, cudaStream_t s) {
    switch (halo) {
        case 0: return launch_tiled<DIM, ORDER, TILE, 0>(g, n, P, offs, J, ctr, chunk_tile, chunk, block, s);
        case 1: return launch_tiled<DIM, ORDER, TILE, 1>(g, n, P, offs, J, ctr, chunk_tile, chunk, block, s);
        case 2: return launch_tiled<DIM, ORDER, TILE, 2>(g, n, P, offs, J, ctr, chunk_tile, chunk, block, s);
        default: return PCG_ERR_UNSUPPORTED;
    }
}

template <int DIM>
pcg_status dispatch_tiled(int order, int tile, int halo, const Geom &g, long long n,
                          const Particles &P, const uint32_t *offs, float *J, const Counters &ctr,
                          unsigned *chunk_tile, long long chunk, int block, cudaStream_t s) {
    if (order == 1 && tile == 8) return dispatch_halo<DIM, 1, 8>(halo, g, n, P, offs, J, ctr, chunk_tile, chunk, block, s);
    if (order == 1 && tile == 4) return dispatch_halo<DIM, 1, 4>(halo, g, n, P, offs, J, ctr, chunk_tile, chunk, block, s);
    if (order == 2 && tile == 8) return dispatch_halo<DIM, 2, 8>(halo, g, n, P, offs, J, ctr, chunk_tile, chunk, block, s);
    if (order == 2 && tile == 4) return dispatch_halo<DIM, 2, 4>(halo, g, n, P, offs, J, ctr, chunk_tile, chunk, block, s);
    return PCG_ERR_UNSUPPORTED;
}

}  // namespace dep
}  // namespace pcg
