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

constexpr int kMidOffset = 62;  // offset of the displacement (0, 0, 0); see "Stored half" below

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
        if (!PCG_IN(g, A.ncells)) continue;
        for (int b = 0; b < 27; ++b) {
            const int bx = b % 3, by = (b / 3) % 3, bz = b / 9;
            const int o = (bz - az + 2) * 25 + (by - ay + 2) * 5 + (bx - ax + 2);
            if (o < kMidOffset) continue;  // the mirror half is copied afterwards
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

// Stored half.  M is symmetric per component, M[g][o] = M[g + d][124 - o] for
// the displacement d of offset o (Eq. (11) of Pennati & Markidis: each
// component block is symmetric in (g, g')).  The assembly kernels add only the
// offsets o >= 62 (d >= 0 in (dz, dy, dx) lexicographic order, the canonical
// half of Sec. 3.4) and a streaming kernel then copies the mirror half.
// One x-run of partners of a node at union x-position ax (0..3): the partners
// bx = lo .. lo + cnt - 1 of the 4-node union row with |bx - ax| <= 2 that lie
// in the stored half for the row's (dy, dz); o0 is the offset of the first.
// False when the row stores nothing.
struct Run {
    int lo, cnt, o0;
};
__device__ __forceinline__ bool stored_run(int ax, int dy, int dz, Run &r) {
    if (dy < -2 || dy > 2 || dz < -2 || dz > 2) return false;
    if (dz < 0 || (dz == 0 && dy < 0)) return false;
    const int last = ax == 0 ? 2 : 3;
    r.lo = (dz == 0 && dy == 0) ? ax : (ax == 3 ? 1 : 0);
    r.cnt = last - r.lo + 1;
    r.o0 = (dz + 2) * 25 + (dy + 2) * 5 + (r.lo - ax + 2);
    return true;
}

// A lane's staging slot for the flush: 40 floats (ten 16-byte quads) of shared
// memory, 16-byte aligned.
constexpr int kSlot = 40;

// Add one run of M: floats [start, start + L) (L <= 36) get val(k) for
// k = k0 .. k0 + L - 1, val a compile-time-indexable source of 36 values.  The
// run is placed in this lane's slot at the same 16-byte phase as M, with zeros
// around it, and goes out as aligned 16-byte vector reductions of the quads
// that hold a non-zero (a zero added to a neighbouring entry leaves it
// unchanged); a quad that would reach past float `total` of M goes out as
// scalars.  The loop is the same for every lane (no divergent dispatch on the
// run's start, length or phase); `active` false adds nothing.
template <class V>
__device__ __forceinline__ void flush_slot(float *M, long long total, float *slot, long long start, int k0, int L,
                                           bool active, const V &val) {
    float4 *q = reinterpret_cast<float4 *>(slot);
#pragma unroll
    for (int i = 0; i < kSlot / 4; ++i) q[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    active = active && PCG_IN(start, total) && PCG_IN(start + L - 1, total);
    const int mis = (int)(start & 3);
#pragma unroll
    for (int k = 0; k < 36; ++k)
        if (active && k >= k0 && k < k0 + L) slot[mis + k - k0] = val(k);
    const long long base = start - mis;
#pragma unroll
    for (int i = 0; i < kSlot / 4; ++i) {
        const float4 v = q[i];
        if (!active || (v.x == 0.f && v.y == 0.f && v.z == 0.f && v.w == 0.f)) continue;
        const long long a = base + 4 * i;
        if (a + 4 <= total) {
            red_add_v4_f32(M + a, v.x, v.y, v.z, v.w);
        } else {
            if (a < total && v.x != 0.f) red_add_f32(M + a, v.x);
            if (a + 1 < total && v.y != 0.f) red_add_f32(M + a + 1, v.y);
            if (a + 2 < total && v.z != 0.f) red_add_f32(M + a + 2, v.z);
        }
    }
}

// M (float[ncells][125][9]) must be zeroed by the caller; grid edges >= 5.
// The assembly fills the stored half; launch_mass_tsc_mirror the rest.
pcg_status launch_mass_tsc(const Args &A, cudaStream_t s);                    // CUDA cores (mass_tsc.cu)
pcg_status launch_mass_tsc_tc(const Args &A, int precision, cudaStream_t s);  // tcgen05 (mass_tsc_tc.cu)
pcg_status launch_mass_tsc_mirror(const Args &A, cudaStream_t s);             // mass_tsc.cu

}  // namespace tsc
}  // namespace pcg
