// mass_tsc.cuh -- pieces shared by the second-order (TSC) ECSIM mass-matrix
// kernels: the CUDA-core one (mass_tsc.cu) and the tcgen05 one (mass_tsc_tc.cu).
//
// Pennati & Markidis, "Mass Matrix Assembly on Tensor Cores for Implicit
// Particle-In-Cell Methods": Eqs. (4)-(6) (M^{ij}_{gg'} = sum_p w_p alpha_p^{ij}
// W_pg W_pg'), Sec. 2.3 (quadratic B-spline weights and the base-offset rule),
// Sec. 3.4 (offset storage, here all 125 displacements in {-2..2}^3 kept:
// M[g][o][ij], o = (dz+2)*25 + (dy+2)*5 + (dx+2)).
#pragma once

#include "common.cuh"
#include "mass_common.cuh"

namespace pcg {
namespace tsc {

struct Args {
    int N[3];
    long long ncells;
    const float *x, *y, *z, *w, *ox, *oy, *oz;
    const uint32_t *offs;
    long long n;
    float *M;
    unsigned *flags;
    unsigned long long *n_invalid;
};

// Quadratic B-spline support of one coordinate: first node k - 1 with
// k = i + (xi >= 1/2), and the weights at k-1, k, k+1 for s = x - k.
__device__ __forceinline__ int tsc_axis(float x, float (&w)[3]) {
    const int i = (int)x;  // x >= 0
    const int k = i + (x - (float)i >= 0.5f ? 1 : 0);
    const float s = x - (float)k;
    const float a = 0.5f - s, b = 0.5f + s;
    w[0] = 0.5f * a * a;
    w[1] = 0.75f - s * s;
    w[2] = 0.5f * b * b;
    return k - 1;
}

__device__ __forceinline__ int wrapi(int i, int N) { return i >= N ? i - N : (i < 0 ? i + N : i); }

__device__ __forceinline__ bool in_grid(const Args &A, float x, float y, float z) {
    return x >= 0.f && x < (float)A.N[0] && y >= 0.f && y < (float)A.N[1] && z >= 0.f && z < (float)A.N[2];
}

// A particle not inside the cell it is listed under: all 27 x 27 x 9
// contributions straight to global M.
static __device__ __noinline__ void particle_global(const Args A, float x, float y, float z, float wq, float ox, float oy,
                                             float oz) {
    float wx[3], wy[3], wz[3], s[9];
    const int fx = tsc_axis(x, wx), fy = tsc_axis(y, wy), fz = tsc_axis(z, wz);
    alpha_w(wq, ox, oy, oz, s);
    for (int a = 0; a < 27; ++a) {
        const int ax = a % 3, ay = (a / 3) % 3, az = a / 9;
        const long long g = ((long long)wrapi(fz + az, A.N[2]) * A.N[1] + wrapi(fy + ay, A.N[1])) * A.N[0] +
                            wrapi(fx + ax, A.N[0]);
        const float Wa = wx[ax] * wy[ay] * wz[az];
        for (int b = 0; b < 27; ++b) {
            const int bx = b % 3, by = (b / 3) % 3, bz = b / 9;
            const int o = (bz - az + 2) * 25 + (by - ay + 2) * 5 + (bx - ax + 2);
            const float WW = Wa * wx[bx] * wy[by] * wz[bz];
            for (int c = 0; c < 9; ++c) red_add_f32(A.M + (g * 125 + o) * 9 + c, s[c] * WW);
        }
    }
}

// The tail pass: slots [offs[ncells], n) are listed under no cell (the sort's
// sentinel bin of invalid particles, or particles appended after the sort);
// valid ones go to M by the global path, invalid ones are counted.
__device__ __forceinline__ void tail_pass(const Args &A, unsigned &n_inv) {
    for (long long p = (long long)A.offs[A.ncells] + (long long)blockIdx.x * blockDim.x + threadIdx.x; p < A.n;
         p += (long long)gridDim.x * blockDim.x) {
        const float x = A.x[p], y = A.y[p], z = A.z[p];
        if (in_grid(A, x, y, z)) particle_global(A, x, y, z, A.w[p], A.ox[p], A.oy[p], A.oz[p]);
        else ++n_inv;
    }
}

// M (float[ncells][125][9]) must be zeroed by the caller; grid edges >= 5.
pcg_status launch_mass_tsc(const Args &A, cudaStream_t s);                    // CUDA cores (mass_tsc.cu)
pcg_status launch_mass_tsc_tc(const Args &A, int precision, cudaStream_t s);  // tcgen05 (mass_tsc_tc.cu)

}  // namespace tsc
}  // namespace pcg
