// mass_matrix.cu -- ECSIM block mass matrix: the entry points, and the CIC
// assembly on CUDA cores (the A/B baseline of the tensor-core kernels).
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
// Kernels behind pcg_assemble_mass_matrix(_scalar):
//  * order 1 on tcgen05 (TF32, BF16): mass_cic_tc.cu, a warp-specialised pipeline;
//  * order 2 on tcgen05: mass_tsc_tc.cu; order 2 on CUDA cores: mass_tsc.cu;
//  * order 1 on CUDA cores: mass_simt_kernel below.  Two 256-thread CTAs per SM
//    walk 4x4x2-cell blocks; per iteration two cell batches of 64 particles are
//    staged (W and w alpha per particle) in shared memory, the thread of row
//    (component c, corner a) sums s^c W_a W_b over the batch for the 8 partners
//    b with fp32 FMAs, and the rows are added into the block's 5x5x3 node window
//    in shared memory, which goes to M by bulk reduce-adds on the TMA engine.
#include "mass_cic.cuh"
#include "mass_tsc.cuh"

namespace pcg {
namespace mm {

constexpr int kThreads = 256;

template <int NC>
__global__ void __launch_bounds__(kThreads, 2) mass_simt_kernel(Args A) {
    using Wn = Win<NC>;
    constexpr int NB = Wn::NB, ACC_ROW = Wn::ACC_ROW, ACC_FLOATS = Wn::ACC_FLOATS;
    extern __shared__ __align__(16) unsigned char smem[];
    float *ps = reinterpret_cast<float *>(smem);  // [G][KB][8 + NC]: W and s of the staged particles
    float *acc = reinterpret_cast<float *>(smem + Op<SIMT, NC>::STAGING);
    unsigned *cstart = reinterpret_cast<unsigned *>(smem + Op<SIMT, NC>::STAGING + Wn::ACC_BYTES);
    unsigned *ccount = cstart + 64;
    int *rsh = reinterpret_cast<int *>(ccount + 64);  // window row shifts (floats)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int pme = tid % (G * KB), half = tid / (G * KB);
    const int jme = pme / KB, kme = pme % KB;  // this thread's batch, particle and half
    for (int i = tid; i < ACC_FLOATS; i += kThreads) acc[i] = 0.f;
    unsigned n_inv = 0;

    const int nblocks = A.nb[0] * A.nb[1] * A.nb[2];
    for (int blk = blockIdx.x; blk < nblocks; blk += gridDim.x) {
        const int bx = blk % A.nb[0], by = (blk / A.nb[0]) % A.nb[1], bz = blk / (A.nb[0] * A.nb[1]);
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
            rsh[tid - NCELL] = row_shift<NC>(A, bx, by, bz, tid - NCELL);
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
            // ---- per-particle W and s staged in shared memory ----
            constexpr int PS = 8 + NC;  // floats per particle
            if (half == 0) {
                float *dst = ps + (size_t)pme * PS;
#pragma unroll
                for (int a = 0; a < 8; ++a) dst[a] = W[a];
#pragma unroll
                for (int c = 0; c < NC; ++c) dst[8 + c] = s[c];
            }
            Batch nbt[G];
            const bool nany = next_batches(cstart, ccount, cur, cur_k, nbt);
            raw = load_raw<NC>(A, nbt[jme], kme);  // the next batches load while this one is summed
            __syncthreads();
            // ---- row (c, a) of batch jj: the 8 partner sums on CUDA cores ----
            const int q = warp & 3, jj = warp >> 2;
            const int r = 32 * q + lane;
            if (32 * q < 8 * NC && bt[jj].ci >= 0 && r < 8 * NC) {
                const int c = r >> 3, a = r & 7;
                const float *pj = ps + (size_t)jj * KB * PS;
                float d[8];
#pragma unroll
                for (int nn = 0; nn < 8; ++nn) d[nn] = 0.f;
                for (int k = 0; k < KB; ++k) {
                    const float f = pj[k * PS + 8 + c] * pj[k * PS + a];
#pragma unroll
                    for (int nn = 0; nn < 8; ++nn) d[nn] = fmaf(f, pj[k * PS + nn], d[nn]);
                }
                // ---- into the node window ----
                const int ci = bt[jj].ci;
                const int nx = ci % BCX + (a & 1), ny = (ci / BCX) % BCY + ((a >> 1) & 1), nz = ci / (BCX * BCY) + (a >> 2);
                const int wr = nz * WNY + ny;
                const int ri = wr * ACC_ROW + rsh[wr] + nx * NB + c;
                float *row = acc + ri;
                // (no early exit here: the barrier below is reached by every thread)
                if (PCG_IN(ri, ACC_FLOATS) && PCG_IN(ri + 26 * NC, ACC_FLOATS)) {
#pragma unroll
                    for (int nn = 0; nn < 8; ++nn) {
                        const int o = ((nn >> 2) - (a >> 2) + 1) * 9 + (((nn >> 1) & 1) - ((a >> 1) & 1) + 1) * 3 +
                                      ((nn & 1) - (a & 1) + 1);
                        red_shared_add_f32(row + o * NC, d[nn]);
                    }
                }
            }
            __syncthreads();  // staging and the batch list are reused
#pragma unroll
            for (int j = 0; j < G; ++j) bt[j] = nbt[j];
            any = nany;
        }

        // ---- flush the node window: each row of 5 node blocks is contiguous in M ----
        tc::fence_proxy_async_smem();  // the window's shared-memory reductions, for the TMA
        __syncthreads();
        flush_window<NC, kThreads>(A, acc, rsh, bx, by, bz);
        if (tid == 0) {
            tc::bulk_commit();
            tc::bulk_wait_read_all();  // the window may be cleared once the TMA has read it
        }
        __syncthreads();
        for (int i = tid; i < ACC_FLOATS; i += kThreads) acc[i] = 0.f;
    }

    tail_pass<NC>(A, n_inv);
    warp_add_u64(A.n_invalid, n_inv);
    if (tid == 0) tc::bulk_wait_all();
}

template <int NC>
pcg_status launch_simt(const Args &A, cudaStream_t s) {
    const size_t smem = Op<SIMT, NC>::STAGING + Win<NC>::ACC_BYTES + 64 * 8 + 32 * 4;
    PCG_CHECK_CUDA(cudaFuncSetAttribute(mass_simt_kernel<NC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)smem));
    const long long nblocks = (long long)A.nb[0] * A.nb[1] * A.nb[2];
    const long long cap = 2ll * num_sms();  // two CTAs per SM
    const long long grid = nblocks < cap ? nblocks : cap;
    prof::Mark mk(NC == 1 ? "mass_scalar_simt" : "mass_matrix_simt", s);
    mass_simt_kernel<NC><<<(unsigned)grid, kThreads, smem, s>>>(A);
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
        case 0: return launch_tc<TF32, NC>(A, s);
        case 1: return launch_tc<BF16, NC>(A, s);
        default: return launch_simt<NC>(A, s);
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
