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
// GB300 design (first version, CUDA cores).  One 512-thread CTA per cell: the
// union of the supports of the cell's particles is the 4x4x4 node block
// starting one node below the cell.  Thread (a, h) owns union node a (0..63)
// and the 8 partner nodes b = 8h..8h+7, i.e. 72 accumulators (8 pairs x 9
// components) in registers, for every particle of the cell.  Particles are
// staged 64 at a time: their per-node weights (64 x 64 floats, zero outside
// their 27 nodes) and coefficients w alpha in shared memory.  At the end of the
// cell every pair within +-2 nodes per axis is added to M: each thread's 4
// partners along x are 4 consecutive offsets, i.e. a run of up to 36
// consecutive floats of M, which goes out as 16-byte vector reductions between
// a scalar head and tail: 9-12 reductions per run instead of 27-36 (32^3 x 64
// ppc: 6.64 -> 5.80 ms).  The cells are walked in order so that the rows they
// share stay in L2.
#include "mass_tsc.cuh"

namespace pcg {
namespace tsc {
namespace {

constexpr int kThreads = 512;
constexpr int KB = 64;     // particles per staged batch
constexpr int NU = 64;     // union nodes (4 x 4 x 4)


// One run of the flush: the partners bx = LO .. LO + L/9 - 1 of one row, i.e.
// L consecutive floats of M starting at dst (= (g*125 + o)*9 floats into the
// 16-byte-aligned M).  HEAD = floats up to the next 16-byte boundary: scalar
// reductions for the head and the tail, 16-byte vector reductions between, so
// every vector address is 16-byte aligned.  All-zero quads are skipped.
template <int ROW, int LO, int L, int HEAD>
__device__ __forceinline__ void flush_run(float *dst, const float (&acc)[8][9]) {
#define PCG_TSC_V(e) acc[4 * ROW + LO + (e) / 9][(e) % 9]
#pragma unroll
    for (int e = 0; e < HEAD && e < L; ++e)
        if (PCG_TSC_V(e) != 0.f) red_add_f32(dst + e, PCG_TSC_V(e));
#pragma unroll
    for (int e = HEAD; e + 4 <= L; e += 4) {
        const float v0 = PCG_TSC_V(e), v1 = PCG_TSC_V(e + 1), v2 = PCG_TSC_V(e + 2), v3 = PCG_TSC_V(e + 3);
        if (v0 != 0.f || v1 != 0.f || v2 != 0.f || v3 != 0.f) red_add_v4_f32(dst + e, v0, v1, v2, v3);
    }
#pragma unroll
    for (int e = HEAD + (L - HEAD) / 4 * 4; e < L; ++e)
        if (e >= HEAD && PCG_TSC_V(e) != 0.f) red_add_f32(dst + e, PCG_TSC_V(e));
#undef PCG_TSC_V
}

// Row ROW (partners 4 ROW .. 4 ROW + 3 of this thread, one x-row of the union)
// of node (ax, ay, az) into M: the partners within +-2 along x are bx = 0..2
// (ax = 0), 1..3 (ax = 3) or 0..3.
template <int ROW>
__device__ __forceinline__ void flush_row(float *M, long long g, int ax, int ay, int az, int h,
                                          const float (&acc)[8][9]) {
    const int b0 = 8 * h + 4 * ROW;
    const int dy = ((b0 >> 2) & 3) - ay, dz = (b0 >> 4) - az;
    if (dy < -2 || dy > 2 || dz < -2 || dz > 2) return;
    const int lo = ax == 3 ? 1 : 0;
    const int o = (dz + 2) * 25 + (dy + 2) * 5 + (lo - ax + 2);
    const long long start = (g * 125 + o) * 9;
    const int head = (int)((4 - (start & 3)) & 3);
    float *dst = M + start;
    const int kind = ax == 0 ? 1 : (ax == 3 ? 2 : 0);  // 0: 4 partners from bx 0; 1: 3 from 0; 2: 3 from 1
    switch (kind * 4 + head) {
        case 0: flush_run<ROW, 0, 36, 0>(dst, acc); break;
        case 1: flush_run<ROW, 0, 36, 1>(dst, acc); break;
        case 2: flush_run<ROW, 0, 36, 2>(dst, acc); break;
        case 3: flush_run<ROW, 0, 36, 3>(dst, acc); break;
        case 4: flush_run<ROW, 0, 27, 0>(dst, acc); break;
        case 5: flush_run<ROW, 0, 27, 1>(dst, acc); break;
        case 6: flush_run<ROW, 0, 27, 2>(dst, acc); break;
        case 7: flush_run<ROW, 0, 27, 3>(dst, acc); break;
        case 8: flush_run<ROW, 1, 27, 0>(dst, acc); break;
        case 9: flush_run<ROW, 1, 27, 1>(dst, acc); break;
        case 10: flush_run<ROW, 1, 27, 2>(dst, acc); break;
        default: flush_run<ROW, 1, 27, 3>(dst, acc); break;
    }
}

__global__ void __launch_bounds__(kThreads, 1) mass_tsc_kernel(Args A) {
    __shared__ __align__(16) float Wt[KB][NU];  // per-node weights of the staged particles
    __shared__ float S[KB][9];        // w alpha
    __shared__ int rel[KB][3];        // first node relative to the union, -1 = skip
    __shared__ float wax[KB][3][3];   // per-axis weights

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
        flush_row<0>(A.M, g, ax, ay, az, h, acc);
        flush_row<1>(A.M, g, ax, ay, az, h, acc);
    }
    tail_pass(A, n_inv);
    warp_add_u64(A.n_invalid, n_inv);
}

}  // namespace

pcg_status launch_mass_tsc(const Args &A, cudaStream_t s) {
    const long long cap = num_sms();
    const long long ctas = A.ncells < cap ? A.ncells : cap;
    prof::Mark mk("mass_tsc_simt", s);
    mass_tsc_kernel<<<(unsigned)ctas, kThreads, 0, s>>>(A);
    return launch_status();
}

}  // namespace tsc
}  // namespace pcg
