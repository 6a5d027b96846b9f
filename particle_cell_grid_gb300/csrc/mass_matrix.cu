// mass_matrix.cu -- ECSIM block mass matrix with CIC shapes on tcgen05 tensor cores.
//
// Method: Pennati & Markidis, "Mass Matrix Assembly on Tensor Cores for
// Implicit Particle-In-Cell Methods".
//   Eqs. (4)-(6): M^{ij}_{gg'} = sum_p s_p^{ij} W_pg W_pg',  s_p = w_p alpha_p,
//                 alpha_p = (I - C(omega_p) + omega_p omega_p^T) / (1 + |omega_p|^2).
//   Sec. 3.1, Eqs. (14)-(15): with particles sorted by cell, every CIC particle
//                 of a cell shares the cell's 8 corner nodes, so the cell's
//                 contribution is the local product  M^ij = (W S^ij) W^T.
//   Sec. 3.2, Eqs. (16)-(20): the particles of a cell are cut into batches of K
//                 (zero-padded), and D <- D + A B accumulates in place.
//   Sec. 3.4:     the 8x8 local block is scattered into offset-indexed storage.
//
// GB300 design.
//  * One tcgen05.mma per K-step computes all nine tensor components of a cell
//    batch at once: A stacks the nine 8 x K blocks W S^{ij} into its rows (row
//    r = 8*(3i+j) + a; 72 of the 128 rows of an M = 128 MMA), B = W^T is K x 8
//    (N = 16).  Rows 72..127 of A and columns 8..15 of B are never read back, so
//    their shared-memory footprint overlaps the next buffer instead of being
//    zeroed.  TF32 (kind::tf32, K = 8 per instruction) or BF16 (kind::f16,
//    K = 16), fp32 accumulation in tensor memory; one thread issues, the result
//    comes back with tcgen05.ld (32 lanes x 8 columns per warp).
//  * Operands use the 128-byte-swizzled K-major layout.  Two threads own one
//    particle (one K column of A and B; tensor components 0-4 and B, or 5-8):
//    a warp's 32 consecutive particles write a full 128-byte row per store
//    instruction, all 32 banks, with the row index a compile-time constant, so
//    the particle's corner weights and coefficients stay in registers.
//  * The next batch group's particles are loaded into registers while the
//    tensor core runs on the current one.
//  * A CTA of 256 threads walks 4x4x2-cell blocks; each block's 5x5x3 node
//    window of 243-float blocks (71 KB) is accumulated in shared memory and
//    flushed once to global M, ~2.3 node blocks of reductions per cell instead
//    of 8: each window row (5 nodes, contiguous in M) goes out as one
//    asynchronous bulk reduce-add on the TMA engine, issued by one thread.
//    Two CTAs share an SM (113 KB of shared memory each for TF32), so that one
//    CTA's staging and epilogue run while the other waits on its MMAs.  One
//    512-thread CTA per SM with 4x4x4 blocks was 1.42x slower (TF32, 64^3 x 64
//    ppc: 2.28 vs 1.60 ms), bound by the barriers and waits of its serial
//    stage -> MMA -> epilogue loop (37 % issue-active, 16 warps per SM).
//  * precision 2 computes the same local products on CUDA cores (fp32 FMAs),
//    the A/B baseline of the tensor-core kernel.
#include <cuda_bf16.h>

#include "common.cuh"
#include "mass_common.cuh"
#include "tcgen05.cuh"
#include "mass_tsc.cuh"

namespace pcg {
namespace mm {

constexpr int kThreads = 256;
constexpr int KB = 64;             // particles per batch: the K extent of one cell product
constexpr int G = 2;               // batches (cell products) per iteration
// a CTA walks blocks of BCX x BCY x BCZ cells; two CTAs share an SM
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
constexpr uint32_t kTmemCols = 32;  // G accumulators of 16 columns
constexpr uint32_t kMaxPolls = 1u << 22;

enum Mode { TF32 = 0, BF16 = 1, SIMT = 2 };

// Staging of one batch (128-byte swizzle, K-major), NC components:
//   TF32: K = 64 x 4 B = 256 B per row = two 128-byte K-atoms; per K-atom the
//         8 NC A rows are NC atoms of 8 rows, B's 8 rows one atom (1 KB).
//         [A k0 | A k1 | B k0 | B k1] = 20 KB for NC = 9, 4 KB for NC = 1.
//   BF16: K = 64 x 2 B = one K-atom.  [A | B].
template <int MODE, int NC>
struct Op {
    static constexpr int KATOMS = MODE == TF32 ? 2 : 1;
    static constexpr int A_KSTRIDE = NC * 1024;              // A bytes per K-atom
    static constexpr int A_BYTES = KATOMS * A_KSTRIDE;
    static constexpr int B_BYTES = KATOMS * 1024;
    static constexpr int BATCH = A_BYTES + B_BYTES;
    static constexpr int STAGING = G * BATCH;
    // the MMA reads 16 row atoms of A and 2 of B from each K-atom base, past the
    // last batch's own rows; those reads land in the node window that follows
    // (never read back) and must stay inside the CTA's shared memory
    static constexpr int READ_END_A = (G - 1) * BATCH + (KATOMS - 1) * A_KSTRIDE + 16 * 1024;
    static constexpr int READ_END_B = (G - 1) * BATCH + A_BYTES + (KATOMS - 1) * 1024 + 2 * 1024;
    static constexpr int READ_END = READ_END_A > READ_END_B ? READ_END_A : READ_END_B;
    static constexpr int KSTEPS = MODE == TF32 ? KB / 8 : KB / 16;
    static constexpr int EB = MODE == TF32 ? 4 : 2;           // element bytes
};

template <int NC>
struct Op<SIMT, NC> {
    static constexpr int STAGING = G * KB * (8 + NC) * 4;  // per particle: W[8], s[NC]
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

template <int MODE, int NC>
__global__ void __launch_bounds__(kThreads, 2) mass_kernel(Args A) {
    using Wn = Win<NC>;
    constexpr int NB = Wn::NB, ACC_ROW = Wn::ACC_ROW, ACC_FLOATS = Wn::ACC_FLOATS;
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char *stage = smem;  // 1024-aligned operand staging first
    float *acc = reinterpret_cast<float *>(smem + Op<MODE, NC>::STAGING);
    unsigned *cstart = reinterpret_cast<unsigned *>(smem + Op<MODE, NC>::STAGING + Wn::ACC_BYTES);
    unsigned *ccount = cstart + 64;
    int *rsh = reinterpret_cast<int *>(ccount + 64);  // window row shifts (floats)
    uint64_t *mbar = reinterpret_cast<uint64_t *>(rsh + 32);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mbar + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int pme = tid % (G * KB), half = tid / (G * KB);
    const int jme = pme / KB, kme = pme % KB;  // this thread's batch, particle and half
    uint32_t tmem = 0;
    if (MODE != SIMT) {
        if (warp == 0) tc::tmem_alloc(tmem_slot, kTmemCols);
        if (tid == 0) tc::mbar_init(mbar, 1);
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        tmem = *tmem_slot;
    }
    for (int i = tid; i < ACC_FLOATS; i += kThreads) acc[i] = 0.f;
    uint32_t phase = 0;
    bool timed_out = false;
    unsigned n_inv = 0;

    const long long nblocks = (long long)A.nb[0] * A.nb[1] * A.nb[2];
    for (long long blk = blockIdx.x; blk < nblocks && !timed_out; blk += gridDim.x) {
        const int bx = (int)(blk % A.nb[0]);
        const int by = (int)((blk / A.nb[0]) % A.nb[1]);
        const int bz = (int)(blk / ((long long)A.nb[0] * A.nb[1]));
        __syncthreads();  // previous block's flush finished with cstart/ccount
        if (tid < NCELL) {
            const int cx = bx * BCX + tid % BCX, cy = by * BCY + (tid / BCX) % BCY,
                      cz = bz * BCZ + tid / (BCX * BCY);
            unsigned s = 0, c = 0;
            if (cx < A.N[0] && cy < A.N[1] && cz < A.N[2]) {
                const long long cell = ((long long)cz * A.N[1] + cy) * A.N[0] + cx;
                unsigned a0 = A.offs[cell], a1 = A.offs[cell + 1];
                if (a1 < a0 || (long long)a1 > A.n) {
                    if (A.flags) atomicOr(A.flags, PCG_FLAG_BAD_LAYOUT);
                    a1 = a0 = 0;
                }
                s = a0;
                c = a1 - a0;
            }
            cstart[tid] = s;
            ccount[tid] = c;
        } else if (tid < NCELL + NROWS) {
            const int row = tid - NCELL;
            const int gy = (by * BCY + row % WNY) % A.N[1], gz = (bz * BCZ + row / WNY) % A.N[2];
            const long long node = ((long long)gz * A.N[1] + gy) * A.N[0] + (bx * BCX) % A.N[0];
            rsh[row] = (int)((node * NB) & 3);
        }
        __syncthreads();

        int cur = 0;
        unsigned cur_k = 0;
        Batch bt[G];
        bool any = next_batches(cstart, ccount, cur, cur_k, bt);
        Raw raw = load_raw<NC>(A, bt[jme], kme);
        while (any) {
            const Batch mine = bt[jme];
            const int cx = bx * BCX + mine.ci % BCX, cy = by * BCY + (mine.ci / BCX) % BCY,
                      cz = bz * BCZ + mine.ci / (BCX * BCY);
            float W[8], s[NC];
            prepare<NC>(A, raw, cx, cy, cz, half == 0, W, s, n_inv);

            float d[2][8];   // this thread's rows of up to two batches
            int dj[2] = {-1, -1};
            Batch nbt[G];
            bool nany;
            if constexpr (MODE != SIMT) {
                using O = Op<MODE, NC>;
                // ---- this particle's column of A = [W S^ij] and B = W^T (128-byte swizzle) ----
                {
                    unsigned char *Aj = stage + jme * O::BATCH;
                    unsigned char *Bj = Aj + O::A_BYTES;
                    const int katom = (kme * O::EB) >> 7;               // which 128-byte K-atom
                    const int kin = (kme * O::EB) & 127;                // byte inside the row
                    const int chunk = kin >> 4, inb = kin & 15;
                    unsigned char *abase = Aj + katom * O::A_KSTRIDE + inb;
                    unsigned char *bbase = Bj + katom * 1024 + inb;
#pragma unroll
                    for (int a = 0; a < 8; ++a) {
                        const int off = a * 128 + ((chunk ^ a) << 4);
#pragma unroll
                        for (int c = 0; c < NC; ++c) {
                            // components split between the particle's two threads
                            if ((c < (NC + 1) / 2) != (half == 0)) continue;
                            const float v = s[c] * W[a];
                            unsigned char *dst = abase + c * 1024 + off;
                            if (MODE == TF32) *reinterpret_cast<uint32_t *>(dst) = tc::to_tf32(v);
                            else *reinterpret_cast<__nv_bfloat16 *>(dst) = __float2bfloat16_rn(v);
                        }
                        if (half == 0) {
                            unsigned char *dstb = bbase + off;
                            if (MODE == TF32) *reinterpret_cast<uint32_t *>(dstb) = tc::to_tf32(W[a]);
                            else *reinterpret_cast<__nv_bfloat16 *>(dstb) = __float2bfloat16_rn(W[a]);
                        }
                    }
                }
                tc::fence_proxy_async_smem();
                tc::fence_before_sync();
                __syncthreads();

                // ---- one thread issues the MMAs of the valid batches ----
                if (tid == 0) {
                    tc::fence_after_sync();
                    constexpr uint32_t idesc = tc::instr_desc(MODE == TF32 ? 2u : 1u, 128, 16);
                    const uint64_t ad0 = tc::smem_desc_sw128(tc::smem_addr(stage), 1024);
                    const uint64_t bd0 = tc::smem_desc_sw128(tc::smem_addr(stage + O::A_BYTES), 1024);
                    // batch-major: consecutive instructions chain on one accumulator
                    // (measured faster than interleaving the G accumulators)
#pragma unroll
                    for (int jj = 0; jj < G; ++jj) {
                        if (bt[jj].ci < 0) continue;
                        const uint64_t joff = (uint64_t)(jj * O::BATCH) >> 4;  // descriptor units
#pragma unroll
                        for (int ks = 0; ks < O::KSTEPS; ++ks) {
                            // 32 bytes of K per instruction: K-atom ks*32/128, offset inside it
                            const uint32_t kb = ks * 32;
                            const uint32_t ka = (kb >> 7), ko = kb & 127;
                            const uint64_t aoff = (ka * O::A_KSTRIDE + ko) >> 4;
                            const uint64_t boff = (ka * 1024 + ko) >> 4;
                            tc::mma<MODE == TF32>(tmem + 16 * jj, ad0 + joff + aoff, bd0 + joff + boff,
                                                  idesc, ks > 0);
                        }
                    }
                    tc::commit(mbar);
                }
                // the next group's particles load while the tensor core works
                nany = next_batches(cstart, ccount, cur, cur_k, nbt);
                raw = load_raw<NC>(A, nbt[jme], kme);

                const bool late = __syncthreads_or(!tc::mbar_wait(mbar, phase, kMaxPolls));
                if (late) {
                    timed_out = true;
                    if (tid == 0 && A.flags) atomicOr(A.flags, PCG_FLAG_TIMEOUT);
                    break;
                }
                phase ^= 1;
                tc::fence_after_sync();

                // ---- read the accumulators back: warp quadrant q holds rows 32q..32q+31 ----
                const int q = warp & 3;
                const int jj = warp >> 2;  // one batch per warp: warps 4j..4j+3 cover its 128 lanes
                if (32 * q < 8 * NC && bt[jj].ci >= 0) {  // warp-uniform
                    tc::tmem_ld8(tmem + ((uint32_t)(32 * q) << 16) + 16 * jj, d[0]);
                    dj[0] = jj;
                }
                tc::fence_before_sync();
            } else {
                // ---- CUDA-core baseline: per-particle W and s staged in shared memory ----
                constexpr int PS = 8 + NC;                      // floats per particle
                float *ps = reinterpret_cast<float *>(stage);  // [G][KB][PS]
                if (half == 0) {
                    float *dst = ps + (size_t)pme * PS;
#pragma unroll
                    for (int a = 0; a < 8; ++a) dst[a] = W[a];
#pragma unroll
                    for (int c = 0; c < NC; ++c) dst[8 + c] = s[c];
                }
                nany = next_batches(cstart, ccount, cur, cur_k, nbt);
                raw = load_raw<NC>(A, nbt[jme], kme);
                __syncthreads();
                const int q = warp & 3;
                const int r = 32 * q + lane;
#pragma unroll
                for (int h = 0; h < 1; ++h) {
                    const int jj = warp >> 2;
                    if (32 * q >= 8 * NC || bt[jj].ci < 0) continue;
                    dj[h] = jj;
#pragma unroll
                    for (int nn = 0; nn < 8; ++nn) d[h][nn] = 0.f;
                    if (r < 8 * NC) {
                        const int c = r >> 3, a = r & 7;
                        const float *pj = ps + (size_t)jj * KB * PS;
                        for (int k = 0; k < KB; ++k) {
                            const float f = pj[k * PS + 8 + c] * pj[k * PS + a];
#pragma unroll
                            for (int nn = 0; nn < 8; ++nn) d[h][nn] = fmaf(f, pj[k * PS + nn], d[h][nn]);
                        }
                    }
                }
            }

            // ---- epilogue: add the 8x8 block rows into the node window ----
            {
                const int r = 32 * (warp & 3) + lane;
                if (r < 8 * NC) {
                    const int c = r >> 3, a = r & 7;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (dj[h] < 0) continue;
                        const int ci = bt[dj[h]].ci;
                        const int nx = ci % BCX + (a & 1), ny = (ci / BCX) % BCY + ((a >> 1) & 1),
                                  nz = ci / (BCX * BCY) + (a >> 2);
                        const int wr = nz * WNY + ny;
                        float *row = acc + wr * ACC_ROW + rsh[wr] + nx * NB + c;
#pragma unroll
                        for (int nn = 0; nn < 8; ++nn) {
                            const int o = ((nn >> 2) - (a >> 2) + 1) * 9 +
                                          (((nn >> 1) & 1) - ((a >> 1) & 1) + 1) * 3 +
                                          ((nn & 1) - (a & 1) + 1);
                            red_shared_add_f32(row + o * NC, d[h][nn]);
                        }
                    }
                }
            }
            __syncthreads();  // staging, TMEM slots and the batch list are reused
            if (MODE != SIMT) tc::fence_after_sync();
#pragma unroll
            for (int j = 0; j < G; ++j) bt[j] = nbt[j];
            any = nany;
        }

        // ---- flush the node window: each row of 5 node blocks is contiguous in M ----
        tc::fence_proxy_async_smem();  // the window's shared-memory reductions, for the TMA
        __syncthreads();
        for (int row = 0; row < NROWS; ++row) {
            const int gy = (by * BCY + row % WNY) % A.N[1];
            const int gz = (bz * BCZ + row / WNY) % A.N[2];
            const float *src = acc + row * ACC_ROW + rsh[row];
            int nx0 = 0;
            while (nx0 < WNX) {
                const int gx0 = (bx * BCX + nx0) % A.N[0];
                int len = WNX - nx0;
                if (gx0 + len > A.N[0]) len = A.N[0] - gx0;  // the row wraps at the x boundary
                float *dst = A.M + (((long long)gz * A.N[1] + gy) * A.N[0] + gx0) * NB;
                const float *sp = src + nx0 * NB;
                const int L = len * NB;
                const int head = min((int)((16 - (reinterpret_cast<uintptr_t>(dst) & 15)) & 15) / 4, L);
                const bool same = ((reinterpret_cast<uintptr_t>(sp + head) & 15) == 0) &&
                                  ((reinterpret_cast<uintptr_t>(dst + head) & 15) == 0);
                if (same) {
                    // aligned body: one bulk reduce-add; head and tail (< 4 floats each) by threads
                    const int body = (L - head) & ~3;
                    if (tid == 0 && body > 0)
                        tc::bulk_reduce_add_f32(dst + head, sp + head, (uint32_t)body * 4);
                    const int e = tid - 1;  // threads 1..7
                    if (e >= 0 && e < head) red_add_f32(dst + e, sp[e]);
                    const int t = head + body + (e - 3);
                    if (e >= 3 && e < 7 && t < L) red_add_f32(dst + t, sp[t]);
                } else {
                    // the part after a wrap: shared and global alignment differ
                    for (int i = tid; i < L; i += kThreads)
                        if (sp[i] != 0.f) red_add_f32(dst + i, sp[i]);
                }
                nx0 += len;
            }
        }
        if (tid == 0) {
            tc::bulk_commit();
            tc::bulk_wait_read_all();  // the window may be cleared once the TMA has read it
        }
        __syncthreads();
        for (int i = tid; i < ACC_FLOATS; i += kThreads) acc[i] = 0.f;
    }

    if (!timed_out) tail_pass<NC>(A, n_inv);
    warp_add_u64(A.n_invalid, n_inv);
    if (tid == 0) tc::bulk_wait_all();
    if (MODE != SIMT) {
        // after a timeout, give the outstanding MMAs one more bounded wait
        if (timed_out) (void)tc::mbar_wait(mbar, phase, kMaxPolls);
        tc::fence_before_sync();
        __syncthreads();
        if (warp == 0) {
            tc::fence_after_sync();
            tc::tmem_dealloc(tmem, kTmemCols);
        }
    }
}

template <int MODE, int NC>
size_t smem_bytes() {
    const size_t used = Op<MODE, NC>::STAGING + Win<NC>::ACC_BYTES + 64 * 8 + 32 * 4 + 16;
    const size_t reads = Op<MODE, NC>::READ_END;
    return used > reads ? used : reads;
}

template <int MODE, int NC>
pcg_status launch(const Args &A, cudaStream_t s) {
    const size_t smem = smem_bytes<MODE, NC>();
    PCG_CHECK_CUDA(cudaFuncSetAttribute(mass_kernel<MODE, NC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)smem));
    const long long nblocks = (long long)A.nb[0] * A.nb[1] * A.nb[2];
    const long long cap = 2ll * num_sms();  // two CTAs per SM
    const long long grid = nblocks < cap ? nblocks : cap;
    static const char *const names[2][3] = {
        {"mass_matrix_tf32", "mass_matrix_bf16", "mass_matrix_simt"},
        {"mass_scalar_tf32", "mass_scalar_bf16", "mass_scalar_simt"}};
    prof::Mark mk(names[NC == 1][MODE], s);
    mass_kernel<MODE, NC><<<(unsigned)grid, kThreads, smem, s>>>(A);
    return launch_status();
}

}  // namespace mm
}  // namespace pcg

extern "C" pcg_status pcg_assemble_mass_matrix_workspace_size(const int32_t *grid, int64_t n,
                                                              size_t *bytes) {
    if (grid == nullptr || bytes == nullptr || n < 0) return PCG_ERR_INVALID_ARG;
    *bytes = 0;
    return PCG_OK;
}

namespace pcg {
namespace mm {
namespace {

// Shared body of the tensor (NC = 9) and scalar (NC = 1) entry points.
template <int NC>
pcg_status assemble(const int32_t *grid, int32_t order, int32_t precision, int64_t n, const float *const *pos,
                    const float *w, const float *const *omega, const uint32_t *cell_offsets, float *M,
                    pcg_stats *stats, void *stream) {
    if (grid == nullptr || n < 0 || n >= 0xffffffffll) return PCG_ERR_INVALID_ARG;
    if (order != 1 && !(order == 2 && NC == 9)) return PCG_ERR_INVALID_ARG;
    if (precision < 0 || precision > 2) return PCG_ERR_INVALID_ARG;
    const int min_edge = order == 2 ? 5 : 3;  // the 27 or 125 offsets must be distinct nodes
    long long ncells = 1;
    for (int mu = 0; mu < 3; ++mu) {
        if (grid[mu] < min_edge || grid[mu] > (1 << 20)) return PCG_ERR_INVALID_ARG;
        ncells *= grid[mu];
    }
    if (ncells >= (1ll << 31)) return PCG_ERR_INVALID_ARG;
    if (M == nullptr || !aligned16(M) || cell_offsets == nullptr) return PCG_ERR_INVALID_ARG;
    if (n > 0 && (pos == nullptr || w == nullptr || pos[0] == nullptr || pos[1] == nullptr || pos[2] == nullptr))
        return PCG_ERR_INVALID_ARG;
    if (NC == 9 && n > 0 &&
        (omega == nullptr || omega[0] == nullptr || omega[1] == nullptr || omega[2] == nullptr))
        return PCG_ERR_INVALID_ARG;
    Args A{};
    for (int mu = 0; mu < 3; ++mu) {
        A.N[mu] = grid[mu];
        A.nb[mu] = (grid[mu] + (mu == 0 ? BCX : mu == 1 ? BCY : BCZ) - 1) / (mu == 0 ? BCX : mu == 1 ? BCY : BCZ);
    }
    A.ncells = ncells;
    if (n > 0) {
        A.x = pos[0];
        A.y = pos[1];
        A.z = pos[2];
        A.w = w;
        if (NC == 9) {
            A.ox = omega[0];
            A.oy = omega[1];
            A.oz = omega[2];
        }
    }
    A.offs = cell_offsets;
    A.n = n;
    A.M = M;
    A.flags = stats ? &stats->error_flags : nullptr;
    A.n_invalid = stats ? &stats->n_invalid : nullptr;
    cudaStream_t s = as_stream(stream);
    pcg_status st = zero_f32(M, (size_t)ncells * (order == 2 ? 1125 : Win<NC>::NB), s);
    if (st != PCG_OK || n == 0) return st;
    if (order == 2) {
        tsc::Args T{};
        for (int mu = 0; mu < 3; ++mu) T.N[mu] = grid[mu];
        T.ncells = ncells;
        T.x = A.x;
        T.y = A.y;
        T.z = A.z;
        T.w = A.w;
        T.ox = A.ox;
        T.oy = A.oy;
        T.oz = A.oz;
        T.offs = cell_offsets;
        T.n = n;
        T.M = M;
        T.flags = A.flags;
        T.n_invalid = A.n_invalid;
        st = precision == 2 ? tsc::launch_mass_tsc(T, s) : tsc::launch_mass_tsc_tc(T, precision, s);
        return st == PCG_OK ? tsc::launch_mass_tsc_mirror(T, s) : st;
    }
    switch (precision) {
        case 0: return launch<TF32, NC>(A, s);
        case 1: return launch<BF16, NC>(A, s);
        default: return launch<SIMT, NC>(A, s);
    }
}

}  // namespace
}  // namespace mm
}  // namespace pcg

extern "C" pcg_status pcg_assemble_mass_matrix(const int32_t *grid, int32_t order,
                                               int32_t precision, int64_t n,
                                               const float *const *pos, const float *w,
                                               const float *const *omega,
                                               const uint32_t *cell_offsets, float *M,
                                               pcg_stats *stats, void *workspace,
                                               size_t workspace_bytes, void *stream) {
    (void)workspace;
    (void)workspace_bytes;
    return pcg::mm::assemble<9>(grid, order, precision, n, pos, w, omega, cell_offsets, M, stats, stream);
}

extern "C" pcg_status pcg_assemble_mass_matrix_scalar(const int32_t *grid, int32_t order, int32_t precision,
                                                      int64_t n, const float *const *pos, const float *w,
                                                      const uint32_t *cell_offsets, float *M, pcg_stats *stats,
                                                      void *stream) {
    return pcg::mm::assemble<1>(grid, order, precision, n, pos, w, nullptr, cell_offsets, M, stats, stream);
}
