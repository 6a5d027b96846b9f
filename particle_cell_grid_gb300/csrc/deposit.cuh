// deposit.cuh -- current deposit J^c_g = sum_p q_p v^c_p W(x_p - x_g) (tiled and flat).
//
// Shape: tensor-product B-splines (Pennati & Markidis, Sec. 2.3, Eq. (12)).
// order 1 (cloud-in-cell): nodes i, i+1 with weights 1 - xi, xi.
// order 2 (quadratic): nearest node k = i + (xi >= 1/2), s = x - k in [-1/2, 1/2),
//   nodes k-1, k, k+1 with weights (1/2 - s)^2 / 2, 3/4 - s^2, (1/2 + s)^2 / 2;
//   i.e. {j-1, j, j+1} when xi < 1/2 and {j, j+1, j+2} otherwise.
//
// Tiled deposit: "Tiled current deposit" (Entity wiki), sections "How a tile
// deposit runs", "Halo sizing" and "Correctness is independent of the halo".
// Each CTA owns a fixed-size chunk of the tile-sorted particle array.  For every
// tile segment inside its chunk it zeroes a haloed scratch tile of
// 3 x (T + 2*HALO)^D floats in shared memory, adds each particle's stencil
// there with shared-memory reductions when the whole stencil fits the window
// (the fit test), or sends the whole particle to J with global reductions when
// it does not (the escape valve), and finally flushes every non-zero scratch
// cell once into J with a global reduction, wrapping periodically.  Fixed-size
// chunks instead of one CTA per tile give every CTA the same particle count,
// so dense tiles (a 10x density bump) split across CTAs without a work list.
#pragma once

#include "common.cuh"

namespace pcg {
namespace dep {

struct Geom {
    int N[3];      // nodes per axis (1 on unused axes)
    int nt[3];     // tiles per axis
    float Nf[3];   // domain extents
    long long ncells;
    unsigned n_tiles;
};

struct Particles {
    const float *x, *y, *z;
    const float *vx, *vy, *vz;
    const float *q;
};

struct Counters {
    unsigned long long *n_escaped;
    unsigned long long *n_invalid;
    unsigned *flags;
};

// One axis of the B-spline support: first node and ORDER+1 weights.
template <int ORDER>
__device__ __forceinline__ int axis_weights(float x, float (&w)[ORDER + 1]) {
    const int i = (int)x;  // x >= 0 here
    const float xi = x - (float)i;
    if (ORDER == 1) {
        w[0] = 1.f - xi;
        w[1] = xi;
        return i;
    } else {
        const int k = i + (xi >= 0.5f ? 1 : 0);
        const float s = x - (float)k;  // exact: x and k are within a factor two
        const float a = 0.5f - s, b = 0.5f + s;
        w[0] = 0.5f * a * a;
        w[1] = 0.75f - s * s;
        w[2] = 0.5f * b * b;
        return k - 1;
    }
}

template <int DIM>
__device__ __forceinline__ bool in_domain(const Geom &g, float x, float y, float z) {
    bool ok = (x >= 0.f) & (x < g.Nf[0]) & (y >= 0.f) & (y < g.Nf[1]);
    if (DIM == 3) ok &= (z >= 0.f) & (z < g.Nf[2]);
    return ok;
}

// Whole stencil of one particle into J with global reductions (periodic wrap).
template <int DIM, int ORDER>
__device__ __forceinline__ void deposit_global(const Geom &g, float *__restrict__ J, float x,
                                               float y, float z, float qvx, float qvy, float qvz) {
    constexpr int S = ORDER + 1;
    constexpr int SZ = DIM == 3 ? S : 1;
    float wx[S], wy[S], wz[S];
    const int fx = axis_weights<ORDER>(x, wx);
    const int fy = axis_weights<ORDER>(y, wy);
    int fz = 0;
    if (DIM == 3) fz = axis_weights<ORDER>(z, wz);
    else wz[0] = 1.f;
#pragma unroll
    for (int kz = 0; kz < SZ; ++kz) {
        const int gz = DIM == 3 ? wrap_index(fz + kz, g.N[2]) : 0;
#pragma unroll
        for (int ky = 0; ky < S; ++ky) {
            const int gy = wrap_index(fy + ky, g.N[1]);
            const float wyz = wy[ky] * wz[kz];
            const long long row = ((long long)gz * g.N[1] + gy) * g.N[0];
#pragma unroll
            for (int kx = 0; kx < S; ++kx) {
                const long long node = row + wrap_index(fx + kx, g.N[0]);
                if (!PCG_IN(node, g.ncells)) continue;
                const float W = wyz * wx[kx];
                red_add_f32(J + node, qvx * W);
                red_add_f32(J + g.ncells + node, qvy * W);
                red_add_f32(J + 2 * g.ncells + node, qvz * W);
            }
        }
    }
}

// Tile-local coordinate of a stencil's first node (S nodes per axis) relative to
// the tile origin, taken periodically: the non-negative offset when the stencil
// then ends inside the scratch window [-HALO, TILE + HALO), else the offset one
// period below (a particle that drifted across the lower periodic boundary).
template <int S, int TILE, int HALO>
__device__ __forceinline__ int local_index(int f, int origin, int N) {
    // f in [-1, N) (a first node of an in-domain particle) and origin in [0, N),
    // so f - origin lies in [-N - 1, N) and at most two corrections reduce it
    int d = f - origin;
    if (d < 0) d += N;
    if (d < 0) d += N;
    return d + S - 1 < TILE + HALO ? d : d - N;
}

}  // namespace dep

// host-side helpers shared by the deposit entry points (deposit.cu)
long long chunk_for(long long n);
bool geom_from(int32_t dim, const int32_t *grid, int tile, dep::Geom *g);
// zero J (3 * ncells floats, 16-byte aligned), and with tile_offsets given,
// map every chunk of the sorted array to its first tile and check the layout
pcg_status launch_prep(float *J, const dep::Geom &g, const uint32_t *tile_offsets, long long n, long long chunk,
                       unsigned *chunk_tile, unsigned *flags, cudaStream_t s);

// host-side dispatchers (deposit_2d.cu / deposit_3d.cu)
pcg_status deposit_tiled_2d(int order, int tile, int halo, const dep::Geom &g, long long n,
                            const dep::Particles &P, const uint32_t *offs, float *J,
                            const dep::Counters &ctr, unsigned *chunk_tile, long long chunk,
                            int block, cudaStream_t s);
pcg_status deposit_tiled_3d(int order, int tile, int halo, const dep::Geom &g, long long n,
                            const dep::Particles &P, const uint32_t *offs, float *J,
                            const dep::Counters &ctr, unsigned *chunk_tile, long long chunk,
                            int block, cudaStream_t s);

}  // namespace pcg
