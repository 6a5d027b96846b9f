// mass_tsc.cu -- ECSIM block mass matrix with second-order (TSC) B-splines, on
// CUDA cores.
//
// Method: Pennati & Markidis, "Mass Matrix Assembly on Tensor Cores for
// Implicit Particle-In-Cell Methods".
//   Eqs. (4)-(6): M^{ij}_{gg'} = sum_p w_p alpha_p^{ij} W_pg W_pg'.
//   Sec. 2.3:     quadratic B-spline weights per axis; a coordinate whose
//                 fractional part is < 1/2 uses nodes j-1..j+1, else j..j+2.
//   Sec. 3.3:     particles of one cell with the same node set form a support
//                 group (up to 8); the alternative the section names, one
//                 product over the union of the groups' nodes with zero weights
//                 outside each particle's own 27, is what this kernel does.
//   Sec. 3.4:     displacements in {-2..2}^3: 125 offsets per node, all kept.
//
// GB300 design (CUDA cores; the A/B baseline of the tcgen05 kernel in
// mass_tsc_tc.cu).  One 512-thread CTA per cell: the union of the supports of
// the cell's particles is the 4x4x4 node block starting one node below the
// cell.  Thread (a, h) owns union node a (0..63) and the 8 partner nodes
// b = 8h..8h+7, i.e. 72 accumulators (8 pairs x 9 components) in registers, for
// every particle of the cell.  Particles are staged 64 at a time: their
// per-node weights (64 x 64 floats, zero outside their 27 nodes) and
// coefficients w alpha in shared memory.  At the end of the cell the pairs in
// the stored half of M (displacement >= 0; the mirror half is copied by
// mirror_kernel afterwards) are added to M: each thread's 4 partners along x
// are consecutive offsets, one run of up to 36 consecutive floats of M, which
// goes out through the thread's shared-memory slot as aligned 16-byte vector
// reductions (flush_slot: the same loop in every lane).  The cells are walked
// in order so that the rows they share stay in L2.
#include "mass_tsc.cuh"

namespace pcg {
namespace tsc {
namespace {

constexpr int kThreads = 512;
constexpr int KB = 64;     // particles per staged batch
constexpr int NU = 64;     // union nodes (4 x 4 x 4)


// Row ROW (partners 4 ROW .. 4 ROW + 3 of this thread, one x-row of the union)
// of node (ax, ay, az): its stored part (offsets >= 62) as one run of M,
// flushed through the thread's slot.
template <int ROW>
__device__ __forceinline__ void flush_row(float *M, long long total, float *slot, long long g, int ax, int ay,
                                          int az, int h, const float (&acc)[8][9]) {
    const int b0 = 8 * h + 4 * ROW;
    Run r{0, 0, 0};
    const bool act = stored_run(ax, ((b0 >> 2) & 3) - ay, (b0 >> 4) - az, r);
    flush_slot(M, total, slot, (g * 125 + r.o0) * 9, 9 * r.lo, 9 * r.cnt, act,
               [&](int k) { return acc[4 * ROW + k / 9][k % 9]; });
}

// The mirror half: M[g][o] = M[g + d(o)][124 - o] for every offset o < 62,
// a streaming copy within M (reads the stored half, writes the other).
__global__ void mirror_kernel(float *__restrict__ M, int Nx, int Ny, int Nz, long long ncells) {
    const long long total = ncells * (kMidOffset * 9);
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long g = i / (kMidOffset * 9);
        const int r = (int)(i - g * (kMidOffset * 9));
        const int o = r / 9, c = r - 9 * (r / 9);
        const int dx = o % 5 - 2, dy = (o / 5) % 5 - 2, dz = o / 25 - 2;
        const int gx = (int)(g % Nx), gy = (int)((g / Nx) % Ny), gz = (int)(g / ((long long)Nx * Ny));
        const long long gp = ((long long)wrapi(gz + dz, Nz) * Ny + wrapi(gy + dy, Ny)) * Nx + wrapi(gx + dx, Nx);
        if (PCG_IN(gp, ncells)) M[(g * 125 + o) * 9 + c] = M[(gp * 125 + (124 - o)) * 9 + c];
    }
}

__global__ void __launch_bounds__(kThreads, 1) mass_tsc_kernel(Args A) {
    __shared__ __align__(16) float Wt[KB][NU];  // per-node weights of the staged particles
    __shared__ float S[KB][9];        // w alpha
    __shared__ int rel[KB][3];        // first node relative to the union, -1 = skip
    __shared__ float wax[KB][3][3];   // per-axis weights
    extern __shared__ __align__(16) float slots[];  // kSlot floats per thread, for the flush
    float *slot = slots + kSlot * threadIdx.x;

    const int tid = threadIdx.x;
    const int a = tid >> 3, h = tid & 7;
    const int ax = a & 3, ay = (a >> 2) & 3, az = a >> 4;
    unsigned n_inv = 0;

    for (long long cell = blockIdx.x; cell < A.ncells; cell += gridDim.x) {
        const int cx = (int)(cell % A.N[0]);
        const int cy = (int)((cell / A.N[0]) % A.N[1]);
        const int cz = (int)(cell / ((long long)A.N[0] * A.N[1]));
        long long s0 = A.offs[cell], s1 = A.offs[cell + 1];
        if (s1 < s0 || s1 > A.n) {
            if (tid == 0 && A.flags) atomicOr(A.flags, PCG_FLAG_BAD_LAYOUT);
            continue;  // uniform
        }
        if (s1 == s0) continue;

        float acc[8][9];
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int c = 0; c < 9; ++c) acc[j][c] = 0.f;

        for (long long b0 = s0; b0 < s1; b0 += KB) {
            const int len = (int)min((long long)KB, s1 - b0);
            // ---- stage: per particle its union-relative support and coefficients ----
            if (tid < len) {
                const long long p = b0 + tid;
                const float x = A.x[p], y = A.y[p], z = A.z[p];
                const float wq = A.w[p], ox = A.ox[p], oy = A.oy[p], oz = A.oz[p];
                const bool inside = x >= (float)cx && x < (float)(cx + 1) && y >= (float)cy &&
                                    y < (float)(cy + 1) && z >= (float)cz && z < (float)(cz + 1);
                if (inside) {
                    float w3[3];
                    rel[tid][0] = tsc_axis(x, w3) - (cx - 1);
                    for (int e = 0; e < 3; ++e) wax[tid][0][e] = w3[e];
                    rel[tid][1] = tsc_axis(y, w3) - (cy - 1);
                    for (int e = 0; e < 3; ++e) wax[tid][1][e] = w3[e];
                    rel[tid][2] = tsc_axis(z, w3) - (cz - 1);
                    for (int e = 0; e < 3; ++e) wax[tid][2][e] = w3[e];
                    float sv[9];
                    alpha_w(wq, ox, oy, oz, sv);
                    for (int c = 0; c < 9; ++c) S[tid][c] = sv[c];
                } else {
                    rel[tid][0] = -1;
                    for (int c = 0; c < 9; ++c) S[tid][c] = 0.f;
                    const bool ok = x >= 0.f && x < (float)A.N[0] && y >= 0.f && y < (float)A.N[1] && z >= 0.f &&
                                    z < (float)A.N[2];
                    if (ok) {
                        particle_global(A, x, y, z, wq, ox, oy, oz);
                        if (A.flags) atomicOr(A.flags, PCG_FLAG_CELL_MISMATCH);
                    } else {
                        ++n_inv;  // outside the domain or NaN: skipped
                    }
                }
            }
            __syncthreads();
            // ---- per-node weights, zero outside each particle's 27 nodes ----
            for (int e = tid; e < KB * NU; e += kThreads) {
                const int k = e / NU, nd = e % NU;
                float W = 0.f;
                if (k < len && rel[k][0] >= 0) {
                    const int dx = (nd & 3) - rel[k][0], dy = ((nd >> 2) & 3) - rel[k][1], dz = (nd >> 4) - rel[k][2];
                    if ((unsigned)dx < 3u && (unsigned)dy < 3u && (unsigned)dz < 3u)
                        W = wax[k][0][dx] * wax[k][1][dy] * wax[k][2][dz];
                }
                Wt[k][nd] = W;
            }
            __syncthreads();
            // ---- accumulate the 8 pairs (a, 8h + j) of this thread ----
            for (int k = 0; k < len; ++k) {
                const float wa = Wt[k][a];
                if (wa == 0.f) continue;
                const float4 p0 = *reinterpret_cast<const float4 *>(&Wt[k][8 * h]);
                const float4 p1 = *reinterpret_cast<const float4 *>(&Wt[k][8 * h + 4]);
                const float wb[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
                float sv[9];
#pragma unroll
                for (int c = 0; c < 9; ++c) sv[c] = S[k][c];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float wab = wa * wb[j];
#pragma unroll
                    for (int c = 0; c < 9; ++c) acc[j][c] = fmaf(wab, sv[c], acc[j][c]);
                }
            }
            __syncthreads();  // staging is reused by the next batch
        }

        // ---- flush the pairs within +-2 nodes per axis: two x-rows per thread ----
        const long long g = ((long long)wrapi(cz - 1 + az, A.N[2]) * A.N[1] + wrapi(cy - 1 + ay, A.N[1])) * A.N[0] +
                            wrapi(cx - 1 + ax, A.N[0]);
        flush_row<0>(A.M, A.ncells * 1125, slot, g, ax, ay, az, h, acc);
        flush_row<1>(A.M, A.ncells * 1125, slot, g, ax, ay, az, h, acc);
    }
    tail_pass(A, n_inv);
    warp_add_u64(A.n_invalid, n_inv);
}

}  // namespace

pcg_status launch_mass_tsc_mirror(const Args &A, cudaStream_t s) {
    const long long total = A.ncells * (kMidOffset * 9);
    long long blocks = (total + 255) / 256;
    const long long cap = (long long)num_sms() * 16;
    if (blocks > cap) blocks = cap;
    prof::Mark mk("mass_tsc_mirror", s);
    mirror_kernel<<<(unsigned)blocks, 256, 0, s>>>(A.M, A.N[0], A.N[1], A.N[2], A.ncells);
    return launch_status();
}

pcg_status launch_mass_tsc(const Args &A, cudaStream_t s) {
    const long long cap = num_sms();
    const long long ctas = A.ncells < cap ? A.ncells : cap;
    prof::Mark mk("mass_tsc_simt", s);
    constexpr int kSlotBytes = kSlot * 4 * kThreads;
    PCG_CHECK_CUDA(cudaFuncSetAttribute(mass_tsc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSlotBytes));
    mass_tsc_kernel<<<(unsigned)ctas, kThreads, kSlotBytes, s>>>(A);
    return launch_status();
}

}  // namespace tsc
}  // namespace pcg
