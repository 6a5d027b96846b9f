// mass_cic.cuh -- pieces of the first-order (CIC) ECSIM mass-matrix assembly
// shared by the tcgen05 pipeline (mass_cic_tc.cu) and the CUDA-core kernel
// (mass_matrix.cu): work blocks and their node window, operand layout, the
// per-particle weights and coefficients, the slow and tail paths, the window
// flush.
//
// Pennati & Markidis, "Mass Matrix Assembly on Tensor Cores for Implicit
// Particle-In-Cell Methods": Eqs. (4)-(6), Sec. 3.1-3.2 (per-cell products over
// zero-padded batches of particles), Sec. 3.4 (offset storage, all 27 kept).
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"
#include "mass_common.cuh"
#include "tcgen05.cuh"

namespace pcg {
namespace mm {


constexpr int KB = 64;             // particles per batch: the K extent of one cell product
constexpr int G = 2;               // batches (cell products) per iteration
// a CTA walks blocks of BCX x BCY x BCZ cells
constexpr int BCX = 4, BCY = 4, BCZ = 2;
constexpr int NCELL = BCX * BCY * BCZ;
constexpr int WNX = BCX + 1, WNY = BCY + 1, WNZ = BCZ + 1;  // node window
constexpr int NROWS = WNY * WNZ;                            // window rows (x runs)
// Node blocks: 27 offsets x NC components (NC = 9 for the ECSIM tensor, 1 for
// the scalar matrix).  A window row of 5 node blocks starts 0-3 floats into its
// slot, so that it has the same alignment modulo 16 bytes as its place in M.
template <int NC>
struct Win {
    static constexpr int NB = 27 * NC;                                   // floats per node block
    static constexpr int ACC_ROW = (WNX * NB + 3 + 3) / 4 * 4;           // 1220 (NC 9), 140 (NC 1)
    static constexpr int ACC_FLOATS = NROWS * ACC_ROW;
    static constexpr int ACC_BYTES = (ACC_FLOATS * 4 + 1023) / 1024 * 1024;
};
constexpr uint32_t kMaxPolls = 1u << 22;

enum Mode { TF32 = 0, BF16 = 1, SIMT = 2 };

// Staging of one batch (128-byte swizzle, K-major), NC components:
//   TF32: K = 64 x 4 B = 256 B per row = two 128-byte K-atoms; per K-atom the
//         8 NC A rows are NC atoms of 8 rows, B's 8 rows one atom (1 KB).
//         [A k0 | A k1 | B k0 | B k1] = 20 KB for NC = 9, 4 KB for NC = 1.
//   BF16: K = 64 x 2 B = one K-atom.  [A | B].
template <int MODE, int NC, int GG = G>
struct Op {
    static constexpr int KATOMS = MODE == TF32 ? 2 : 1;
    static constexpr int A_KSTRIDE = NC * 1024;              // A bytes per K-atom
    static constexpr int A_BYTES = KATOMS * A_KSTRIDE;
    static constexpr int B_BYTES = KATOMS * 1024;
    static constexpr int BATCH = A_BYTES + B_BYTES;
    static constexpr int STAGING = GG * BATCH;               // GG batches staged together
    // the MMA reads 16 row atoms of A and 2 of B from each K-atom base, past the
    // last batch's own rows; those reads land in the memory that follows (never
    // read back) and must stay inside the CTA's shared memory
    static constexpr int READ_END_A = (GG - 1) * BATCH + (KATOMS - 1) * A_KSTRIDE + 16 * 1024;
    static constexpr int READ_END_B = (GG - 1) * BATCH + A_BYTES + (KATOMS - 1) * 1024 + 2 * 1024;
    static constexpr int READ_END = READ_END_A > READ_END_B ? READ_END_A : READ_END_B;
    static constexpr int KSTEPS = MODE == TF32 ? KB / 8 : KB / 16;
    static constexpr int EB = MODE == TF32 ? 4 : 2;           // element bytes
};

template <int NC, int GG>
struct Op<SIMT, NC, GG> {
    static constexpr int STAGING = GG * KB * (8 + NC) * 4;  // per particle: W[8], s[NC]
    static constexpr int READ_END = 0;
};

struct Args {
    int N[3];
    long long ncells;
    int nb[3];  // cell blocks per axis
    const float *x, *y, *z, *w, *ox, *oy, *oz;
    const uint32_t *offs;
    long long n;
    float *M;
    unsigned *flags;
    unsigned long long *n_invalid;
};

struct Batch {
    int ci;      // cell index inside the block (0..63), -1 = none
    unsigned start, len;
};


// Per-particle coefficients: w alpha (NC = 9) or w (NC = 1, the scalar case of Eq. (6)).
template <int NC>
__device__ __forceinline__ void coeffs(float w, float ox, float oy, float oz, float (&s)[NC]) {
    if constexpr (NC == 9) alpha_w(w, ox, oy, oz, s);
    else s[0] = w;
}

__device__ __forceinline__ float corner_w(int a, float fx, float fy, float fz) {
    return ((a & 1) ? fx : 1.f - fx) * ((a & 2) ? fy : 1.f - fy) * ((a & 4) ? fz : 1.f - fz);
}

__device__ __forceinline__ int wrapi(int i, int N) { return i >= N ? i - N : (i < 0 ? i + N : i); }

// Slow path for a particle not inside the cell it is listed under: all 8x8xNC
// contributions straight to global M.
template <int NC>
__device__ void particle_global(const Args &A, float x, float y, float z, float w, float ox,
                                float oy, float oz) {
    const int ix = (int)x, iy = (int)y, iz = (int)z;
    const float fx = x - ix, fy = y - iy, fz = z - iz;
    float s[NC];
    coeffs<NC>(w, ox, oy, oz, s);
    for (int a = 0; a < 8; ++a) {
        const int gx = wrapi(ix + (a & 1), A.N[0]);
        const int gy = wrapi(iy + ((a >> 1) & 1), A.N[1]);
        const int gz = wrapi(iz + (a >> 2), A.N[2]);
        const long long g = ((long long)gz * A.N[1] + gy) * A.N[0] + gx;
        const float Wa = corner_w(a, fx, fy, fz);
        for (int b = 0; b < 8; ++b) {
            const int o = (((b >> 2) - (a >> 2)) + 1) * 9 + ((((b >> 1) & 1) - ((a >> 1) & 1)) + 1) * 3 +
                          ((b & 1) - (a & 1)) + 1;
            const float WW = Wa * corner_w(b, fx, fy, fz);
            if (!PCG_IN(g, A.ncells)) continue;
            for (int c = 0; c < NC; ++c) red_add_f32(A.M + (g * 27 + o) * NC + c, s[c] * WW);
        }
    }
}

// This thread's particle of the batch group: raw fields, loaded ahead of use.
struct Raw {
    float x, y, z, w, ox, oy, oz;
    bool live;
};

template <int NC>
__device__ __forceinline__ Raw load_raw(const Args &A, const Batch &b, int k) {
    Raw r;
    r.live = b.ci >= 0 && k < (int)b.len;
    if (r.live) {
        const unsigned p = b.start + k;
        r.x = A.x[p];
        r.y = A.y[p];
        r.z = A.z[p];
        r.w = A.w[p];
        if (NC == 9) {
            r.ox = A.ox[p];
            r.oy = A.oy[p];
            r.oz = A.oz[p];
        } else {
            r.ox = r.oy = r.oz = 0.f;
        }
    } else {
        r.x = r.y = r.z = r.w = r.ox = r.oy = r.oz = 0.f;
    }
    return r;
}

// Weights and coefficients of a loaded particle for the cell (cx, cy, cz); a
// particle outside that cell is flagged, deposited by the slow path and
// contributes zeros here.
template <int NC>
__device__ __forceinline__ bool prepare(const Args &A, const Raw &r, int cx, int cy, int cz,
                                        bool owner, float (&W)[8], float (&s)[NC], unsigned &n_inv) {
    bool use = r.live;
    if (use) {
        const bool inside = r.x >= (float)cx && r.x < (float)(cx + 1) && r.y >= (float)cy &&
                            r.y < (float)(cy + 1) && r.z >= (float)cz && r.z < (float)(cz + 1);
        if (!inside) {
            const bool ok = r.x >= 0.f && r.x < (float)A.N[0] && r.y >= 0.f && r.y < (float)A.N[1] &&
                            r.z >= 0.f && r.z < (float)A.N[2];
            if (owner) {  // once per particle, by one of the threads sharing it
                if (ok) {
                    particle_global<NC>(A, r.x, r.y, r.z, r.w, r.ox, r.oy, r.oz);
                    if (A.flags) atomicOr(A.flags, PCG_FLAG_CELL_MISMATCH);
                } else {
                    ++n_inv;  // outside the domain or NaN: skipped
                }
            }
            use = false;
        }
    }
    if (!use) {
#pragma unroll
        for (int a = 0; a < 8; ++a) W[a] = 0.f;
#pragma unroll
        for (int c = 0; c < NC; ++c) s[c] = 0.f;
        return false;
    }
    const float fx = r.x - (float)cx, fy = r.y - (float)cy, fz = r.z - (float)cz;
    const float gx = 1.f - fx, gy = 1.f - fy, gz = 1.f - fz;
    const float yz00 = gy * gz, yz10 = fy * gz, yz01 = gy * fz, yz11 = fy * fz;
    W[0] = gx * yz00;
    W[1] = fx * yz00;
    W[2] = gx * yz10;
    W[3] = fx * yz10;
    W[4] = gx * yz01;
    W[5] = fx * yz01;
    W[6] = gx * yz11;
    W[7] = fx * yz11;
    coeffs<NC>(r.w, r.ox, r.oy, r.oz, s);
    return true;
}

// The tail pass: slots [offs[ncells], n) are listed under no cell (the sort's
// sentinel bin of invalid particles, or particles appended after the sort).
// Valid ones go to M by the global path, invalid ones are counted.
template <int NC>
__device__ void tail_pass(const Args &A, unsigned &n_inv) {
    const long long t0 = A.offs[A.ncells];
    for (long long p = t0 + (long long)blockIdx.x * blockDim.x + threadIdx.x; p < A.n;
         p += (long long)gridDim.x * blockDim.x) {
        const float x = A.x[p], y = A.y[p], z = A.z[p];
        const bool ok = x >= 0.f && x < (float)A.N[0] && y >= 0.f && y < (float)A.N[1] && z >= 0.f &&
                        z < (float)A.N[2];
        if (!ok) {
            ++n_inv;
            continue;
        }
        if (NC == 9) particle_global<NC>(A, x, y, z, A.w[p], A.ox[p], A.oy[p], A.oz[p]);
        else particle_global<NC>(A, x, y, z, A.w[p], 0.f, 0.f, 0.f);
    }
}

// The G batches starting at cursor (cur, cur_k); identical in every thread.
__device__ __forceinline__ bool next_batches(const unsigned *cstart, const unsigned *ccount, int &cur,
                                             unsigned &cur_k, Batch (&bt)[G]) {
    bool any = false;
#pragma unroll
    for (int j = 0; j < G; ++j) {
        while (cur < NCELL && cur_k >= ccount[cur]) {
            ++cur;
            cur_k = 0;
        }
        if (cur < NCELL) {
            const unsigned rem = ccount[cur] - cur_k;
            bt[j] = Batch{cur, cstart[cur] + cur_k, rem < (unsigned)KB ? rem : (unsigned)KB};
            cur_k += KB;
            any = true;
        } else {
            bt[j] = Batch{-1, 0, 0};
        }
    }
    return any;
}


// Row shift of window row `row` of block (bx, by, bz): the row's first node
// block starts this many floats into its slot, so that the row has the same
// 16-byte phase in shared memory as its place in M.
template <int NC>
__device__ __forceinline__ int row_shift(const Args &A, int bx, int by, int bz, int row) {
    int gy = by * BCY + row % WNY, gz = bz * BCZ + row / WNY, gx = bx * BCX;
    if (gy >= A.N[1]) gy -= A.N[1];  // a window reaches at most one node past the grid's end
    if (gz >= A.N[2]) gz -= A.N[2];
    if (gx >= A.N[0]) gx -= A.N[0];
    const long long node = ((long long)gz * A.N[1] + gy) * A.N[0] + gx;
    return (int)((node * Win<NC>::NB) & 3);
}

// Flush the node window `acc` of block (bx, by, bz) into M: each window row of 5
// node blocks is contiguous in M and goes out as one asynchronous bulk
// reduce-add (TMA engine) issued by thread 0 of the THREADS taking part (`tid`
// is the caller's index among them), the < 4-float head and tail by threads
// 1..7; the part of a row after a periodic wrap in x (shared and
// global alignment then differ) by plain global reductions.  The caller fences
// the window's shared-memory writes for the async proxy and synchronises
// before, and commits and waits on thread 0's bulk group after.
template <int NC, int THREADS>
__device__ __forceinline__ void flush_window(const Args &A, const float *acc, const int *rsh, int bx, int by,
                                             int bz, int tid = threadIdx.x) {
    constexpr int NB = Win<NC>::NB, ACC_ROW = Win<NC>::ACC_ROW;
    for (int row = 0; row < NROWS; ++row) {
        int gy = by * BCY + row % WNY, gz = bz * BCZ + row / WNY;
        if (gy >= A.N[1]) gy -= A.N[1];
        if (gz >= A.N[2]) gz -= A.N[2];
        const float *src = acc + row * ACC_ROW + rsh[row];
        int nx0 = 0;
        while (nx0 < WNX) {
            int gx0 = bx * BCX + nx0;
            if (gx0 >= A.N[0]) gx0 -= A.N[0];
            int len = WNX - nx0;
            if (gx0 + len > A.N[0]) len = A.N[0] - gx0;  // the row wraps at the x boundary
            if (!PCG_IN(((long long)gz * A.N[1] + gy) * A.N[0] + gx0 + len - 1, A.ncells)) break;
            float *dst = A.M + (((long long)gz * A.N[1] + gy) * A.N[0] + gx0) * NB;
            const float *sp = src + nx0 * NB;
            const int L = len * NB;
            const int head = min((int)((16 - (reinterpret_cast<uintptr_t>(dst) & 15)) & 15) / 4, L);
            const bool same = ((reinterpret_cast<uintptr_t>(sp + head) & 15) == 0) &&
                              ((reinterpret_cast<uintptr_t>(dst + head) & 15) == 0);
            if (same) {
                // aligned body: one bulk reduce-add; head and tail (< 4 floats each) by threads
                const int body = (L - head) & ~3;
                if (tid == 0 && body > 0) tc::bulk_reduce_add_f32(dst + head, sp + head, (uint32_t)body * 4);
                const int e = tid - 1;  // threads 1..7
                if (e >= 0 && e < head) red_add_f32(dst + e, sp[e]);
                const int t = head + body + (e - 3);
                if (e >= 3 && e < 7 && t < L) red_add_f32(dst + t, sp[t]);
            } else {
                for (int i = tid; i < L; i += THREADS)
                    if (sp[i] != 0.f) red_add_f32(dst + i, sp[i]);
            }
            nx0 += len;
        }
    }
}

// The software-pipelined tcgen05 assembly (mass_cic_tc.cu), MODE TF32 or BF16.
template <int MODE, int NC>
pcg_status launch_tc(const Args &A, cudaStream_t s);

}  // namespace mm
}  // namespace pcg
