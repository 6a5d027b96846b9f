// mass_tsc_tc.cu -- ECSIM block mass matrix with second-order (TSC) B-splines on
// tcgen05 tensor cores (TF32 or BF16 operands, fp32 accumulation in tensor
// memory).
//
// Method: Pennati & Markidis, "Mass Matrix Assembly on Tensor Cores for
// Implicit Particle-In-Cell Methods".
//   Eqs. (4)-(6): M^{ij}_{gg'} = sum_p w_p alpha_p^{ij} W_pg W_pg'.
//   Sec. 3.1-3.2: per cell, the local product D = W S W^T over batches of
//                 particles, accumulated in place.
//   Sec. 3.3:     a TSC cell's particles fall into up to 8 support groups (node
//                 sets); the alternative the section names is taken: one
//                 product over the union of the groups' supports (the 4 x 4 x 4
//                 nodes from one node below the cell), each particle's weights
//                 zero outside its own 27 nodes.
//   Sec. 3.4:     displacements in {-2..2}^3, all 125 offsets stored.
//
// GB300 design.
//  * Two neighbouring cells along x form one tcgen05 product of M = 128 rows:
//    row 64 j + a is union node a of cell j.  Their particles are the K columns,
//    32 of each cell per 64-particle chunk, and A is block-diagonal (cell j's
//    weights only in its own K half; the other half holds static zeros), so one
//    accumulator serves both cells with every row in use.
//  * Columns are partner nodes b of one z-plane of the union times the nine
//    tensor components, c fastest: N = 4 rows (by) x 40 (4 bx x 9 c, 4 padding
//    columns) = 160.  B = [w alpha^c W_b] per particle.  A thread's 36 columns of
//    one by-row are then the 4 (or 3) consecutive offsets along x of its node,
//    i.e. one run of 36 (or 27) consecutive floats of M, which goes out as
//    16-byte vector reductions between a scalar head and tail.
//  * The 4 planes are 4 passes; a pass accumulates every chunk of the pair.  The
//    accumulator of a plane (160 columns) lives in one of two tensor-memory
//    buffers, so the flush of plane k runs while the tensor core computes plane
//    k + 1, and operand staging of chunk i + 1 runs while chunk i multiplies
//    (two staging buffers, each released by an mbarrier the MMAs commit to).
//  * Operands use the 128-byte-swizzled K-major layout; a warp's 32 lanes are 32
//    particles of one cell and write 128 contiguous bytes of one row per store.
//  * Every mbarrier wait is bounded; a timeout sets PCG_FLAG_TIMEOUT and ends
//    the kernel after one more bounded wait for the MMAs in flight.
#include <cuda_bf16.h>

#include "mass_tsc.cuh"
#include "tcgen05.cuh"

namespace pcg {
namespace tsc {
namespace {

constexpr int kThreads = 256;         // 8 warps
constexpr int KC = 64;                // particles per chunk: 32 of each cell
constexpr int NROW = 40;              // columns per by-row: 4 bx x 9 components + 4 padding
constexpr int NPL = 4 * NROW;         // N = 160 columns per plane
constexpr uint32_t kTmemCols = 512;   // two plane accumulators at columns 0 and 256
constexpr uint32_t kMaxPolls = 1u << 22;

enum { TF32 = 0, BF16 = 1 };

template <int MODE>
struct Lay {
    static constexpr int EB = MODE == TF32 ? 4 : 2;          // element bytes
    static constexpr int KATOMS = KC * EB / 128;              // 2 (TF32) or 1 (BF16)
    static constexpr int A_ATOM = 128 * 128;                  // 128 rows x 128 bytes
    static constexpr int B_ATOM = NPL * 128;                  // 160 rows x 128 bytes
    static constexpr int A_BYTES = KATOMS * A_ATOM;
    static constexpr int B_BYTES = KATOMS * B_ATOM;
    static constexpr int STAGE = A_BYTES + B_BYTES;           // 72 KB (TF32), 36 KB (BF16)
    static constexpr int KSTEPS = KC * EB / 32;               // 32 bytes of K per instruction
    // one CTA per SM: the CTA takes all 512 tensor-memory columns, so shared
    // memory is sized to leave no room for a second CTA
    static constexpr int USED = 2 * STAGE + kSlot * 4 * kThreads + 64;
    static constexpr int SMEM = USED > 120 * 1024 ? USED : 120 * 1024;
};

// Byte offset of (row r, K column kk) inside an operand of K-atoms of `atom`
// bytes (128-byte swizzle: 16-byte chunk c of row r stored at chunk c ^ (r % 8)).
template <int MODE>
__device__ __forceinline__ int sw_off(int r, int kk, int atom) {
    const int kb = kk * Lay<MODE>::EB;
    const int at = kb >> 7, in = kb & 127;
    return at * atom + (r >> 3) * 1024 + (r & 7) * 128 + ((((in >> 4) ^ (r & 7))) << 4) + (in & 15);
}

template <int MODE>
__device__ __forceinline__ void put(unsigned char *p, float v) {
    if (MODE == TF32) *reinterpret_cast<uint32_t *>(p) = tc::to_tf32(v);
    else *reinterpret_cast<__nv_bfloat16 *>(p) = __float2bfloat16_rn(v);
}

// Per-axis weights of a coordinate over the 4 union nodes u = 0..3 of its cell
// (the union starts one node below the cell); zero outside its 3-node support.
__device__ __forceinline__ void union_axis(float x, int cell, float (&U)[4]) {
    float w[3];
    const int r = tsc_axis(x, w) - (cell - 1);  // 0 or 1 for a particle inside the cell
    U[0] = r == 0 ? w[0] : 0.f;
    U[1] = r == 0 ? w[1] : w[0];
    U[2] = r == 0 ? w[2] : w[1];
    U[3] = r == 0 ? 0.f : w[2];
}

// A cell pair: cells (cx0 + j, cy, cz), j = 0, 1; n[j] particles from s[j].
struct Pair {
    int cx0, cy, cz;
    unsigned s[2], n[2];
    int nch;  // 64-particle chunks
};

__device__ __forceinline__ Pair load_pair(const Args &A, long long P) {
    const int npx = (A.N[0] + 1) / 2;
    Pair pr;
    pr.cx0 = (int)(P % npx) * 2;
    pr.cy = (int)((P / npx) % A.N[1]);
    pr.cz = (int)(P / ((long long)npx * A.N[1]));
    int nch = 0;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        pr.s[j] = 0;
        pr.n[j] = 0;
        const int cx = pr.cx0 + j;
        if (cx < A.N[0]) {
            const long long cell = ((long long)pr.cz * A.N[1] + pr.cy) * A.N[0] + cx;
            const unsigned a0 = A.offs[cell], a1 = A.offs[cell + 1];
            if (a1 < a0 || (long long)a1 > A.n) {
                if (threadIdx.x == 0 && A.flags) atomicOr(A.flags, PCG_FLAG_BAD_LAYOUT);
            } else {
                pr.s[j] = a0;
                pr.n[j] = a1 - a0;
            }
        }
        const int c = (int)((pr.n[j] + 31) / 32);
        nch = c > nch ? c : nch;
    }
    pr.nch = nch;
    return pr;
}

// Stage chunk `ch` of the pair for plane p: this thread's particle (cell j =
// warp & 1, slot = lane) writes its A rows of union plane uz = q = warp >> 1
// (16 rows) and its B rows of by-row q of plane p (4 bx x 9 components).
// Particles not inside their listed cell contribute zeros; at plane 0 (once per
// particle, by the q = 0 warp) they go to M by the global path, or are counted
// invalid.
template <int MODE>
__device__ __forceinline__ void stage(const Args &A, const Pair &pr, int p, int ch, unsigned char *Ab,
                                      unsigned char *Bb, unsigned &n_inv) {
    using L = Lay<MODE>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j = warp & 1, q = warp >> 1;
    const unsigned k = (unsigned)ch * 32 + lane;
    const int kk = 32 * j + lane;  // K column of this particle in the chunk
    float Ux[4] = {0.f, 0.f, 0.f, 0.f}, Uy[4] = {0.f, 0.f, 0.f, 0.f}, Uz[4] = {0.f, 0.f, 0.f, 0.f};
    float s[9];
#pragma unroll
    for (int c = 0; c < 9; ++c) s[c] = 0.f;
    if (k < pr.n[j]) {
        const long long pi = (long long)pr.s[j] + k;
        const float x = A.x[pi], y = A.y[pi], z = A.z[pi];
        const int cx = pr.cx0 + j;
        const bool inside = x >= (float)cx && x < (float)(cx + 1) && y >= (float)pr.cy && y < (float)(pr.cy + 1) &&
                            z >= (float)pr.cz && z < (float)(pr.cz + 1);
        if (inside) {
            union_axis(x, cx, Ux);
            union_axis(y, pr.cy, Uy);
            union_axis(z, pr.cz, Uz);
            alpha_w(A.w[pi], A.ox[pi], A.oy[pi], A.oz[pi], s);
        } else if (p == 0 && q == 0) {
            if (in_grid(A, x, y, z)) {
                particle_global(A, x, y, z, A.w[pi], A.ox[pi], A.oy[pi], A.oz[pi]);
                if (A.flags) atomicOr(A.flags, PCG_FLAG_CELL_MISMATCH);
            } else {
                ++n_inv;
            }
        }
    }
    // A: rows 64 j + (16 q + 4 uy + ux), weight Uz[q] Uy[uy] Ux[ux]
    const float wz = Uz[q];
#pragma unroll
    for (int uy = 0; uy < 4; ++uy) {
        const float wyz = wz * Uy[uy];
#pragma unroll
        for (int ux = 0; ux < 4; ++ux) {
            const int r = 64 * j + 16 * q + 4 * uy + ux;
            put<MODE>(Ab + sw_off<MODE>(r, kk, L::A_ATOM), wyz * Ux[ux]);
        }
    }
    // B: rows NROW q + 9 bx + c of plane p, value w alpha^c Uz[p] Uy[q] Ux[bx]
    const float wpq = Uz[p] * Uy[q];
#pragma unroll
    for (int bx = 0; bx < 4; ++bx) {
        const float wb = wpq * Ux[bx];
#pragma unroll
        for (int c = 0; c < 9; ++c) put<MODE>(Bb + sw_off<MODE>(NROW * q + 9 * bx + c, kk, L::B_ATOM), s[c] * wb);
    }
}

// The MMAs of one staged chunk into the plane accumulator at column `dcol`.
template <int MODE>
__device__ __forceinline__ void issue(uint32_t tmem, uint32_t dcol, const unsigned char *Ab,
                                      const unsigned char *Bb, bool acc_first) {
    using L = Lay<MODE>;
    constexpr uint32_t idesc = tc::instr_desc(MODE == TF32 ? 2u : 1u, 128, NPL);
    const uint32_t a0 = tc::smem_addr(Ab), b0 = tc::smem_addr(Bb);
#pragma unroll
    for (int ks = 0; ks < L::KSTEPS; ++ks) {
        const uint32_t kb = ks * 32, at = kb >> 7, ko = kb & 127;
        const uint64_t ad = tc::smem_desc_sw128(a0 + at * L::A_ATOM + ko, 1024);
        const uint64_t bd = tc::smem_desc_sw128(b0 + at * L::B_ATOM + ko, 1024);
        tc::mma<MODE == TF32>(tmem + dcol, ad, bd, idesc, acc_first || ks > 0);
    }
}

// Read one plane's accumulator back and add its stored half to M.  Warp w reads
// lane quadrant w & 3 (rows 32 (w & 3) .. +31: cell j = row / 64, union node
// a = row % 64) and by-rows 2 (w >> 2), 2 (w >> 2) + 1; each row of a node is
// one run of M, flushed through the lane's slot.
__device__ __forceinline__ void drain(const Args &A, const Pair &pr, int p, uint32_t tmem, uint32_t dcol,
                                      float *slot) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = 32 * (warp & 3) + lane;
    const int j = row >> 6, a = row & 63;
    if (pr.n[j] == 0) return;  // warp-uniform: a warp's rows belong to one cell
    const int ax = a & 3, ay = (a >> 2) & 3, az = a >> 4;
    const int gx = wrapi(pr.cx0 + j - 1 + ax, A.N[0]);
    const int gy = wrapi(pr.cy - 1 + ay, A.N[1]);
    const int gz = wrapi(pr.cz - 1 + az, A.N[2]);
    const long long g = ((long long)gz * A.N[1] + gy) * A.N[0] + gx;
    const long long total = A.ncells * 1125;
    const uint32_t lanebase = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + dcol;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int by = 2 * (warp >> 2) + h;
        uint32_t v[NROW];
#pragma unroll
        for (int m = 0; m < NROW / 8; ++m) tc::tmem_ld8_async(lanebase + NROW * by + 8 * m, v + 8 * m);
        tc::tmem_wait_ld(v);
        Run r{0, 0, 0};
        const bool act = stored_run(ax, by - ay, p - az, r);
        flush_slot(A.M, total, slot, (g * 125 + r.o0) * 9, 9 * r.lo, 9 * r.cnt, act,
                   [&](int k) { return __uint_as_float(v[k]); });
    }
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) mass_tsc_tc_kernel(Args A) {
    using L = Lay<MODE>;
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char *const stg0 = smem, *const stg1 = smem + L::STAGE;
    float *slots = reinterpret_cast<float *>(smem + 2 * L::STAGE);       // kSlot floats per thread
    uint64_t *bar = reinterpret_cast<uint64_t *>(slots + kSlot * kThreads);  // [0, 1] staging, [2, 3] planes
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 4);
    const int tid = threadIdx.x, warp = tid >> 5;

    // both staging buffers start at zero: the other cell's half of A and the
    // padding rows of B are never written again
    for (int i = tid; i < 2 * L::STAGE / 16; i += kThreads) reinterpret_cast<uint4 *>(smem)[i] = make_uint4(0, 0, 0, 0);
    if (warp == 0) tc::tmem_alloc(tslot, kTmemCols);
    if (tid == 0)
        for (int i = 0; i < 4; ++i) tc::mbar_init(&bar[i], 1);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tslot;

    uint32_t sph[2] = {0u, 0u}, tph[2] = {0u, 0u};  // parity of each barrier's next completion
    unsigned n_inv = 0;
    bool timed_out = false;
    long long it = 0;  // staging iterations (buffer it & 1)
    int pl = 0;        // planes issued (accumulator pl & 1)
    Pair pend{};       // the plane whose accumulator waits to be drained
    int pend_p = -1, pend_tb = 0;

    auto drain_pending = [&]() {
        const bool late = __syncthreads_or(!tc::mbar_wait(&bar[2 + pend_tb], tph[pend_tb], kMaxPolls));
        if (late) {
            timed_out = true;
            return;
        }
        tph[pend_tb] ^= 1u;
        tc::fence_after_sync();
        drain(A, pend, pend_p, tmem, 256u * pend_tb, slots + kSlot * threadIdx.x);
        tc::fence_before_sync();
        pend_p = -1;
    };

    const long long npairs = (long long)((A.N[0] + 1) / 2) * A.N[1] * A.N[2];
    for (long long P = blockIdx.x; P < npairs && !timed_out; P += gridDim.x) {
        const Pair pr = load_pair(A, P);
        if (pr.nch == 0) continue;
        for (int p = 0; p < 4 && !timed_out; ++p) {
            const int tb = pl & 1;
            for (int ch = 0; ch < pr.nch; ++ch) {
                const int sb = (int)(it & 1);
                unsigned char *Ab = sb ? stg1 : stg0;
                if (it >= 2) {  // the MMAs that read this buffer two iterations ago are done
                    const bool late = __syncthreads_or(!tc::mbar_wait(&bar[sb], sph[sb], kMaxPolls));
                    if (late) {
                        timed_out = true;
                        break;
                    }
                    sph[sb] ^= 1u;
                }
                stage<MODE>(A, pr, p, ch, Ab, Ab + L::A_BYTES, n_inv);
                tc::fence_proxy_async_smem();
                tc::fence_before_sync();
                __syncthreads();
                if (tid == 0) {
                    tc::fence_after_sync();
                    issue<MODE>(tmem, 256u * tb, Ab, Ab + L::A_BYTES, ch > 0);
                    tc::commit(&bar[sb]);
                    if (ch == pr.nch - 1) tc::commit(&bar[2 + tb]);
                }
                ++it;
            }
            if (timed_out) break;
            // the previous plane's flush runs while the tensor core works on this one
            if (pend_p >= 0) drain_pending();
            pend = pr;
            pend_p = p;
            pend_tb = tb;
            ++pl;
        }
    }
    if (!timed_out && pend_p >= 0) drain_pending();

    if (timed_out) {
        if (tid == 0 && A.flags) atomicOr(A.flags, PCG_FLAG_TIMEOUT);
        // one more bounded wait for the last group of MMAs (its commit implies all earlier ones)
        if (it > 0) {
            const int sb = (int)((it - 1) & 1);
            (void)tc::mbar_wait(&bar[sb], sph[sb], kMaxPolls);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
    if (!timed_out) tail_pass(A, n_inv);
    warp_add_u64(A.n_invalid, n_inv);
}

template <int MODE>
pcg_status launch_t(const Args &A, cudaStream_t s) {
    using L = Lay<MODE>;
    PCG_CHECK_CUDA(cudaFuncSetAttribute(mass_tsc_tc_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        L::SMEM));
    const long long npairs = (long long)((A.N[0] + 1) / 2) * A.N[1] * A.N[2];
    const long long cap = num_sms();
    const long long grid = npairs < cap ? npairs : cap;
    prof::Mark mk(MODE == TF32 ? "mass_tsc_tf32" : "mass_tsc_bf16", s);
    mass_tsc_tc_kernel<MODE><<<(unsigned)grid, kThreads, L::SMEM, s>>>(A);
    return launch_status();
}

}  // namespace

pcg_status launch_mass_tsc_tc(const Args &A, int precision, cudaStream_t s) {
    return precision == 0 ? launch_t<TF32>(A, s) : launch_t<BF16>(A, s);
}

}  // namespace tsc
}  // namespace pcg
