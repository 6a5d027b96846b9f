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
//    at once: A stacks the nine 8 x K blocks W S^{ij} into its rows (row
//    r = 8*(3i+j) + a; 72 of the 128 rows of an M = 128 MMA), B = W^T is K x 8
//    (N = 16; columns 8..15 and rows 72..127 are never read back, so their
//    shared-memory footprint overlaps the next buffer instead of being zeroed).
//    TF32 (kind::tf32, K = 8 per instruction) or BF16 (kind::f16, K = 16), fp32
//    accumulation in tensor memory; one thread issues, the result comes back
//    with tcgen05.ld (32 lanes x 8 columns per warp).
//  * A CTA walks 4x4x4-cell blocks; each block's 5x5x5 node window of
//    243-float blocks (121.5 KB) is accumulated in shared memory and flushed
//    once to global M with 16-byte vector reductions, so global reduction
//    traffic is ~1.95 node blocks per cell instead of 8.
//  * Operands are written in the canonical K-major no-swizzle layout (8 rows x
//    16 bytes per core matrix) with a rotated row order per thread, so each
//    8-thread store phase hits 32 distinct banks.
//  * precision 2 computes the same local products on CUDA cores (fp32 FMAs),
//    the A/B baseline of the tensor-core kernel.
#include <cuda_bf16.h>

#include "common.cuh"
#include "tcgen05.cuh"

namespace pcg {
namespace mm {

constexpr int kThreads = 256;
constexpr int KB = 64;             // particles per batch: the K extent of one cell product
constexpr int G = 4;               // batches (cell products) per iteration
constexpr int BC = 4;              // cell-block edge
constexpr int WN = BC + 1;         // node-window edge
constexpr int WNODES = WN * WN * WN;
constexpr int ACC_FLOATS = WNODES * 243;
constexpr int ACC_BYTES = (ACC_FLOATS * 4 + 1023) / 1024 * 1024;
constexpr uint32_t kTmemCols = 64;  // G accumulators of 16 columns
constexpr uint32_t kMaxPolls = 1u << 22;
constexpr unsigned kFlagTimeout = 4u;

enum Mode { TF32 = 0, BF16 = 1, SIMT = 2 };

template <int MODE>
struct Op {
    static constexpr int EPC = MODE == TF32 ? 4 : 8;  // K elements per 16-byte core-matrix row
    static constexpr int KG = KB / EPC;               // core matrices along K
    static constexpr int SBO = KG * 128;              // stride between 8-row groups
    static constexpr int A_BYTES = 9 * SBO;           // rows 0..71
    static constexpr int B_BYTES = SBO;               // N rows 0..7
    static constexpr int BATCH = A_BYTES + B_BYTES;
    static constexpr int STAGING = G * BATCH + 7 * SBO;  // rows 72..127 of the last A stay inside
    static constexpr int KSTEPS = MODE == TF32 ? KB / 8 : KB / 16;
    static constexpr int PARTS = kThreads / (G * KG);  // threads sharing one k-group
};

template <>
struct Op<SIMT> {
    static constexpr int STAGING = G * KB * 17 * 4;  // per particle: W[8], s[9]
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
};

struct Batch {
    int ci;      // cell index inside the block (0..63), -1 = none
    unsigned start, len;
};

__device__ __forceinline__ void alpha_w(float w, float ox, float oy, float oz, float (&s)[9]) {
    const float n2 = ox * ox + oy * oy + oz * oz;
    const float f = w / (1.f + n2);
    s[0] = f * (1.f + ox * ox);
    s[1] = f * (oz + ox * oy);
    s[2] = f * (-oy + ox * oz);
    s[3] = f * (-oz + oy * ox);
    s[4] = f * (1.f + oy * oy);
    s[5] = f * (ox + oy * oz);
    s[6] = f * (oy + oz * ox);
    s[7] = f * (-ox + oz * oy);
    s[8] = f * (1.f + oz * oz);
}

__device__ __forceinline__ float corner_w(int a, float fx, float fy, float fz) {
    return ((a & 1) ? fx : 1.f - fx) * ((a & 2) ? fy : 1.f - fy) * ((a & 4) ? fz : 1.f - fz);
}

__device__ __forceinline__ int wrapi(int i, int N) { return i >= N ? i - N : (i < 0 ? i + N : i); }

// Slow path for a particle not inside the cell it is listed under: all 8x8x9
// contributions straight to global M.
__device__ void particle_global(const Args &A, float x, float y, float z, float w, float ox,
                                float oy, float oz) {
    const int ix = (int)x, iy = (int)y, iz = (int)z;
    const float fx = x - ix, fy = y - iy, fz = z - iz;
    float s[9];
    alpha_w(w, ox, oy, oz, s);
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
            for (int c = 0; c < 9; ++c) red_add_f32(A.M + (g * 27 + o) * 9 + c, s[c] * WW);
        }
    }
}

// Load one particle; returns false (weights zero) when it is padding.  A
// particle outside its listed cell is flagged and deposited by the slow path
// (only by the thread with `owner` set, so exactly once).
__device__ __forceinline__ bool load_particle(const Args &A, const Batch &b, int k, int cx, int cy,
                                              int cz, bool owner, float &fx, float &fy, float &fz,
                                              float (&s)[9]) {
    if (b.ci < 0 || k >= (int)b.len) return false;
    const unsigned p = b.start + k;
    const float x = A.x[p], y = A.y[p], z = A.z[p];
    const float w = A.w[p], ox = A.ox[p], oy = A.oy[p], oz = A.oz[p];
    const bool inside = x >= (float)cx && x < (float)(cx + 1) && y >= (float)cy &&
                        y < (float)(cy + 1) && z >= (float)cz && z < (float)(cz + 1);
    if (!inside) {
        if (owner) {
            const bool ok = x >= 0.f && x < (float)A.N[0] && y >= 0.f && y < (float)A.N[1] &&
                            z >= 0.f && z < (float)A.N[2];
            if (ok) particle_global(A, x, y, z, w, ox, oy, oz);
            if (A.flags) atomicOr(A.flags, PCG_FLAG_CELL_MISMATCH);
        }
        return false;
    }
    fx = x - (float)cx;
    fy = y - (float)cy;
    fz = z - (float)cz;
    alpha_w(w, ox, oy, oz, s);
    return true;
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) mass_kernel(Args A) {
    extern __shared__ __align__(1024) unsigned char smem[];
    float *acc = reinterpret_cast<float *>(smem);
    unsigned char *stage = smem + ACC_BYTES;
    unsigned *cstart = reinterpret_cast<unsigned *>(stage + Op<MODE>::STAGING);
    unsigned *ccount = cstart + 64;
    uint64_t *mbar = reinterpret_cast<uint64_t *>(ccount + 64);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mbar + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
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

    const long long nblocks = (long long)A.nb[0] * A.nb[1] * A.nb[2];
    for (long long blk = blockIdx.x; blk < nblocks && !timed_out; blk += gridDim.x) {
        const int bx = (int)(blk % A.nb[0]);
        const int by = (int)((blk / A.nb[0]) % A.nb[1]);
        const int bz = (int)(blk / ((long long)A.nb[0] * A.nb[1]));
        __syncthreads();  // previous block's flush finished with cstart/ccount
        if (tid < 64) {
            const int cx = bx * BC + (tid & 3), cy = by * BC + ((tid >> 2) & 3), cz = bz * BC + (tid >> 4);
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
        }
        __syncthreads();

        int cur = 0;
        unsigned cur_k = 0;
        while (true) {
            // the next G batches (identical in every thread)
            Batch bt[G];
            bool any = false;
#pragma unroll
            for (int j = 0; j < G; ++j) {
                while (cur < 64 && cur_k >= ccount[cur]) {
                    ++cur;
                    cur_k = 0;
                }
                if (cur < 64) {
                    const unsigned rem = ccount[cur] - cur_k;
                    bt[j] = Batch{cur, cstart[cur] + cur_k, rem < (unsigned)KB ? rem : (unsigned)KB};
                    cur_k += KB;
                    any = true;
                } else {
                    bt[j] = Batch{-1, 0, 0};
                }
            }
            if (!any) break;

            float d[2][8];  // this thread's rows of up to two batches
            int dj[2] = {-1, -1};
            if constexpr (MODE != SIMT) {
                // ---- build A = [W S^ij] and B = W^T in the core-matrix layout ----
                using O = Op<MODE>;
                const int unit = tid % (G * O::KG);
                const int part = tid / (G * O::KG);
                const int j = unit / O::KG, kg = unit % O::KG;
                const Batch b = bt[j];
                const int cx = bx * BC + (b.ci & 3), cy = by * BC + ((b.ci >> 2) & 3),
                          cz = bz * BC + (b.ci >> 4);
                float fx[O::EPC], fy[O::EPC], fz[O::EPC], s[O::EPC][9];
                bool live[O::EPC];
#pragma unroll
                for (int e = 0; e < O::EPC; ++e)
                    live[e] = load_particle(A, b, kg * O::EPC + e, cx, cy, cz, part == 0, fx[e],
                                            fy[e], fz[e], s[e]);
                unsigned char *Aj = stage + j * O::BATCH;
                unsigned char *Bj = Aj + O::A_BYTES;
#pragma unroll
                for (int c = 0; c < 9; ++c) {
                    if (c % O::PARTS != part) continue;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int a = (i + kg) & 7;  // rotated row order: conflict-free phases
                        float v[O::EPC];
#pragma unroll
                        for (int e = 0; e < O::EPC; ++e)
                            v[e] = live[e] ? s[e][c] * corner_w(a, fx[e], fy[e], fz[e]) : 0.f;
                        unsigned char *dst = Aj + c * O::SBO + kg * 128 + a * 16;
                        if (MODE == TF32) {
                            *reinterpret_cast<uint4 *>(dst) = make_uint4(
                                tc::to_tf32(v[0]), tc::to_tf32(v[1]), tc::to_tf32(v[2]), tc::to_tf32(v[3]));
                        } else {
                            uint32_t pk[4];
#pragma unroll
                            for (int h = 0; h < 4; ++h) {
                                __nv_bfloat162 t2 = __floats2bfloat162_rn(v[2 * h], v[2 * h + 1]);
                                pk[h] = *reinterpret_cast<uint32_t *>(&t2);
                            }
                            *reinterpret_cast<uint4 *>(dst) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        }
                    }
                }
                if (part == O::PARTS - 1) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int nn = (i + kg) & 7;
                        float v[O::EPC];
#pragma unroll
                        for (int e = 0; e < O::EPC; ++e)
                            v[e] = live[e] ? corner_w(nn, fx[e], fy[e], fz[e]) : 0.f;
                        unsigned char *dst = Bj + kg * 128 + nn * 16;
                        if (MODE == TF32) {
                            *reinterpret_cast<uint4 *>(dst) = make_uint4(
                                tc::to_tf32(v[0]), tc::to_tf32(v[1]), tc::to_tf32(v[2]), tc::to_tf32(v[3]));
                        } else {
                            uint32_t pk[4];
#pragma unroll
                            for (int h = 0; h < 4; ++h) {
                                __nv_bfloat162 t2 = __floats2bfloat162_rn(v[2 * h], v[2 * h + 1]);
                                pk[h] = *reinterpret_cast<uint32_t *>(&t2);
                            }
                            *reinterpret_cast<uint4 *>(dst) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
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
                    for (int jj = 0; jj < G; ++jj) {
                        if (bt[jj].ci < 0) continue;
                        const uint32_t a0 = tc::smem_addr(stage + jj * O::BATCH);
                        const uint32_t b0 = a0 + O::A_BYTES;
#pragma unroll
                        for (int ks = 0; ks < O::KSTEPS; ++ks) {
                            const uint64_t ad = tc::smem_desc(a0 + ks * 256, 128, O::SBO);
                            const uint64_t bd = tc::smem_desc(b0 + ks * 256, 128, O::SBO);
                            tc::mma<MODE == TF32>(tmem + 16 * jj, ad, bd, idesc, ks > 0);
                        }
                    }
                    tc::commit(mbar);
                }
                // bounded wait; the verdict is made uniform across the CTA
                const bool late = __syncthreads_or(!tc::mbar_wait(mbar, phase, kMaxPolls));
                if (late) {
                    timed_out = true;
                    if (tid == 0 && A.flags) atomicOr(A.flags, kFlagTimeout);
                    break;
                }
                phase ^= 1;
                tc::fence_after_sync();

                // ---- read the accumulators back: warp quadrant q holds rows 32q..32q+31 ----
                const int q = warp & 3;
                if (q < 3) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int jj = (warp >> 2) + 2 * h;
                        if (bt[jj].ci < 0) continue;  // warp-uniform
                        tc::tmem_ld8(tmem + ((uint32_t)(32 * q) << 16) + 16 * jj, d[h]);
                        dj[h] = jj;
                    }
                }
                tc::fence_before_sync();
            } else {
                // ---- CUDA-core baseline: per-particle W and s staged in shared memory ----
                float *ps = reinterpret_cast<float *>(stage);  // [G][KB][17]
                for (int u = tid; u < G * KB; u += kThreads) {
                    const int j = u / KB, k = u % KB;
                    const Batch b = bt[j];
                    const int cx = bx * BC + (b.ci & 3), cy = by * BC + ((b.ci >> 2) & 3),
                              cz = bz * BC + (b.ci >> 4);
                    float fx = 0.f, fy = 0.f, fz = 0.f, s[9];
                    const bool live = load_particle(A, b, k, cx, cy, cz, true, fx, fy, fz, s);
                    float *dst = ps + (size_t)u * 17;
#pragma unroll
                    for (int a = 0; a < 8; ++a) dst[a] = live ? corner_w(a, fx, fy, fz) : 0.f;
#pragma unroll
                    for (int c = 0; c < 9; ++c) dst[8 + c] = live ? s[c] : 0.f;
                }
                __syncthreads();
                // thread -> (batch, row); rows 0..71 of batches {warp>>2, warp>>2 + 2}
                const int q = warp & 3;
                const int r = 32 * q + lane;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int jj = (warp >> 2) + 2 * h;
                    if (q >= 3 || bt[jj].ci < 0) continue;
                    dj[h] = jj;
#pragma unroll
                    for (int nn = 0; nn < 8; ++nn) d[h][nn] = 0.f;
                    if (r < 72) {
                        const int c = r >> 3, a = r & 7;
                        const float *pj = ps + (size_t)jj * KB * 17;
                        for (int k = 0; k < KB; ++k) {
                            const float f = pj[k * 17 + 8 + c] * pj[k * 17 + a];
#pragma unroll
                            for (int nn = 0; nn < 8; ++nn) d[h][nn] = fmaf(f, pj[k * 17 + nn], d[h][nn]);
                        }
                    }
                }
            }

            // ---- epilogue: add the 8x8 block rows into the node window ----
            {
                const int r = 32 * (warp & 3) + lane;
                if (r < 72) {
                    const int c = r >> 3, a = r & 7;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (dj[h] < 0) continue;
                        const int ci = bt[dj[h]].ci;
                        const int nx = (ci & 3) + (a & 1), ny = ((ci >> 2) & 3) + ((a >> 1) & 1),
                                  nz = (ci >> 4) + (a >> 2);
                        float *row = acc + ((nz * WN + ny) * WN + nx) * 243 + c;
#pragma unroll
                        for (int nn = 0; nn < 8; ++nn) {
                            const int o = ((nn >> 2) - (a >> 2) + 1) * 9 +
                                          (((nn >> 1) & 1) - ((a >> 1) & 1) + 1) * 3 +
                                          ((nn & 1) - (a & 1) + 1);
                            red_shared_add_f32(row + o * 9, d[h][nn]);
                        }
                    }
                }
            }
            __syncthreads();  // staging, TMEM slots and the batch cursor are reused
            if (MODE != SIMT) tc::fence_after_sync();
        }

        // ---- flush the node window: contiguous x-runs of node blocks, vector reductions ----
        __syncthreads();
        for (int row = 0; row < WN * WN; ++row) {
            const int ny = row % WN, nz = row / WN;
            const int gy = (by * BC + ny) % A.N[1];
            const int gz = (bz * BC + nz) % A.N[2];
            int nx0 = 0;
            while (nx0 < WN) {
                const int gx0 = (bx * BC + nx0) % A.N[0];
                int len = WN - nx0;
                if (gx0 + len > A.N[0]) len = A.N[0] - gx0;
                const long long g0 = (((long long)gz * A.N[1] + gy) * A.N[0] + gx0) * 243;
                const float *src = acc + (row * WN + nx0) * 243;
                const int L = len * 243;
                const int head = (int)((4 - (g0 & 3)) & 3) < L ? (int)((4 - (g0 & 3)) & 3) : L;
                const int nvec = (L - head) / 4;
                for (int i = tid; i < head; i += kThreads)
                    if (src[i] != 0.f) red_add_f32(A.M + g0 + i, src[i]);
                for (int i = tid; i < nvec; i += kThreads) {
                    const float *sv = src + head + 4 * i;
                    const float v0 = sv[0], v1 = sv[1], v2 = sv[2], v3 = sv[3];
                    if (v0 != 0.f || v1 != 0.f || v2 != 0.f || v3 != 0.f)
                        red_add_v4_f32(A.M + g0 + head + 4 * i, v0, v1, v2, v3);
                }
                for (int i = head + 4 * nvec + tid; i < L; i += kThreads)
                    if (src[i] != 0.f) red_add_f32(A.M + g0 + i, src[i]);
                nx0 += len;
            }
        }
        __syncthreads();
        for (int i = tid; i < ACC_FLOATS; i += kThreads) acc[i] = 0.f;
    }

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

template <int MODE>
size_t smem_bytes() {
    return ACC_BYTES + Op<MODE>::STAGING + 64 * 8 + 16;
}

template <int MODE>
pcg_status launch(const Args &A, cudaStream_t s) {
    const size_t smem = smem_bytes<MODE>();
    PCG_CHECK_CUDA(cudaFuncSetAttribute(mass_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)smem));
    const long long nblocks = (long long)A.nb[0] * A.nb[1] * A.nb[2];
    const long long grid = nblocks < kNumSMs ? nblocks : kNumSMs;
    prof::Mark mk(MODE == TF32 ? "mass_matrix_tf32" : MODE == BF16 ? "mass_matrix_bf16" : "mass_matrix_simt", s);
    mass_kernel<MODE><<<(unsigned)grid, kThreads, smem, s>>>(A);
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

extern "C" pcg_status pcg_assemble_mass_matrix(const int32_t *grid, int32_t order,
                                               int32_t precision, int64_t n,
                                               const float *const *pos, const float *w,
                                               const float *const *omega,
                                               const uint32_t *cell_offsets, float *M,
                                               pcg_stats *stats, void *workspace,
                                               size_t workspace_bytes, void *stream) {
    using namespace pcg;
    (void)workspace;
    (void)workspace_bytes;
    if (grid == nullptr || order != 1 || n < 0 || n >= 0xffffffffll) return PCG_ERR_INVALID_ARG;
    if (precision < 0 || precision > 2) return PCG_ERR_INVALID_ARG;
    long long ncells = 1;
    for (int mu = 0; mu < 3; ++mu) {
        if (grid[mu] < 3 || grid[mu] > (1 << 20)) return PCG_ERR_INVALID_ARG;
        ncells *= grid[mu];
    }
    if (ncells >= (1ll << 31)) return PCG_ERR_INVALID_ARG;
    if (M == nullptr || !aligned16(M) || cell_offsets == nullptr) return PCG_ERR_INVALID_ARG;
    if (n > 0 && (pos == nullptr || omega == nullptr || w == nullptr || pos[0] == nullptr ||
                  pos[1] == nullptr || pos[2] == nullptr || omega[0] == nullptr ||
                  omega[1] == nullptr || omega[2] == nullptr))
        return PCG_ERR_INVALID_ARG;
    mm::Args A{};
    for (int mu = 0; mu < 3; ++mu) {
        A.N[mu] = grid[mu];
        A.nb[mu] = (grid[mu] + mm::BC - 1) / mm::BC;
    }
    A.ncells = ncells;
    if (n > 0) {
        A.x = pos[0];
        A.y = pos[1];
        A.z = pos[2];
        A.w = w;
        A.ox = omega[0];
        A.oy = omega[1];
        A.oz = omega[2];
    }
    A.offs = cell_offsets;
    A.n = n;
    A.M = M;
    A.flags = stats ? &stats->error_flags : nullptr;
    cudaStream_t s = as_stream(stream);
    pcg_status st = zero_f32(M, (size_t)ncells * 243, s);
    if (st != PCG_OK || n == 0) return st;
    switch (precision) {
        case 0: return mm::launch<mm::TF32>(A, s);
        case 1: return mm::launch<mm::BF16>(A, s);
        default: return mm::launch<mm::SIMT>(A, s);
    }
}
