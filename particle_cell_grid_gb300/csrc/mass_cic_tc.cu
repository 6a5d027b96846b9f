// mass_cic_tc.cu -- ECSIM block mass matrix (CIC, tensor and scalar forms) on
// tcgen05 tensor cores, as a warp-specialised pipeline.
//
// Method: Pennati & Markidis, "Mass Matrix Assembly on Tensor Cores for
// Implicit Particle-In-Cell Methods".
//   Eqs. (4)-(6): M^{ij}_{gg'} = sum_p s_p^{ij} W_pg W_pg',  s_p = w_p alpha_p.
//   Sec. 3.1-3.2, Eqs. (14)-(20): per cell the local product (W S^ij) W^T over
//                 zero-padded batches of particles, accumulated in place.
//   Sec. 3.4:     the 8x8 local block scattered into offset-indexed storage.
//
// GB300 design.
//  * The cell product: A stacks the NC components' 8 x K blocks W S^{ij} (72 of
//    the 128 rows of an M = 128 tcgen05.mma for the tensor, 8 for the scalar
//    matrix), B = W^T (N = 16, 8 used), K = 64 particles per batch, TF32 or BF16
//    operands in the 128-byte-swizzled K-major layout, fp32 accumulation in
//    tensor memory.
//  * One 512-thread CTA per SM, warp-specialised, over iterations of GP = 3 cell
//    batches:
//      - producer warps 0-11 stage iteration i's operands into staging buffer
//        i % 2 (two threads per particle; the particles were loaded into
//        registers two iterations earlier) and arrive on full[i % 2];
//      - one thread of warp 15 waits for that, issues the MMAs into accumulator
//        i % 2 and commits to empty[i % 2] (the buffer may be restaged) and to
//        tfull[i % 2];
//      - warps 12-14 (tensor-memory lane quadrants 0-2, the rows in use) wait
//        for tfull, read the accumulators back (tcgen05.ld), add them into the
//        node window and arrive on tempty[i % 2] (the accumulator may be
//        overwritten).
//    Staging, the tensor core and the read-back of different iterations run at
//    the same time.  Every role walks the same sequence of iterations with its
//    own cursor, so no descriptors pass between them.
//  * Cells are walked in 4x4x2 blocks; a block's 5x5x3 node window lives in
//    shared memory and is flushed to M by bulk reduce-adds on the TMA engine.
//    The window is cleared for the next block once that bulk copy has read it.
//    Window adds are plain read-add-writes: an entry (node, offset, component)
//    has one writer at a time (a component belongs to one warp, a cell's 8
//    corners are 8 different nodes, a lane takes its batches in turn).
//  * Every mbarrier wait is bounded.  A role that times out raises a shared
//    abort flag and stops; the others stop at their next wait (each role
//    decides together, through a barrier reduction, so no thread is left at a
//    named barrier), PCG_FLAG_TIMEOUT is set, and the tensor memory is freed
//    after one more bounded wait for the MMAs in flight.
#include "mass_cic.cuh"

namespace pcg {
namespace mm {
namespace {

// Warp roles of the 512-thread CTA.
constexpr int kPThreads = 512;
constexpr int GP = 3;              // cell batches per iteration
constexpr int kProdWarps = 12;     // warps 0-11: operand staging, two threads per particle
constexpr int kEpiWarp0 = 12;      // warps 12-14: read-back, tensor-memory lane quadrants 0-2
constexpr int kEpiThreads = 96;
constexpr int kMmaWarp = 15;       // warp 15: the MMA thread (lane quadrant 3 holds no rows in use)
constexpr int kProdThreads = kProdWarps * 32;
static_assert(kProdThreads == 2 * GP * KB, "two producer threads per particle of an iteration");
constexpr uint32_t kPTmemCols = 128;  // 2 accumulators x GP batches x 16 columns, rounded up
constexpr int kEpiBar = 1, kProdBar = 2;  // named barriers of the roles (0 is the CTA-wide one)
// role waits suspend for up to kSleepNs per poll; at most ~1 s in all
constexpr uint32_t kSleepNs = 1000, kSleepPolls = 1u << 20;

// A role's table of the current block's cell ranges.
struct Tab {
    unsigned start[NCELL], count[NCELL];
};

template <int MODE, int NC>
struct PLay {
    using O = Op<MODE, NC, GP>;
    static constexpr int STAGE = (O::STAGING + 1023) / 1024 * 1024;
    static constexpr int WIN_OFF = 2 * STAGE;
    static constexpr int BAR_OFF = WIN_OFF + Win<NC>::ACC_BYTES;
    static constexpr int TAB_OFF = BAR_OFF + 128;                 // 8 mbarriers, tensor-memory address, abort flag
    static constexpr int RS_OFF = TAB_OFF + 3 * (int)sizeof(Tab);  // a cell table per role
    static constexpr int USED = RS_OFF + 16 * 4;                    // window row shifts of the current block
    // the MMAs of the second staging buffer read past it (rows of A and B that
    // are never read back); those reads must stay inside the allocation
    static constexpr int READ_END = STAGE + O::READ_END;
    static constexpr int SMEM = USED > READ_END ? USED : READ_END;
};

// One pipeline iteration: up to GP batches of one block of cells.
struct Iter {
    Batch bt[GP];
    int blk;
    int bx, by, bz;  // the block's coordinates in blocks
    bool first;      // first iteration of its block
    bool valid;
};

// bt[j] with a runtime j, through constant indices (keeps the batches in registers).
__device__ __forceinline__ Batch pick(const Iter &it, int j) {
    return j == 0 ? it.bt[0] : (j == 1 ? it.bt[1] : it.bt[2]);
}

// Particles of cell ci of block (bx, by, bz): [start, start + count).  A bad
// layout is flagged and the cell treated as empty.
__device__ __forceinline__ void cell_range(const Args &A, int bx, int by, int bz, int ci, unsigned &start,
                                           unsigned &count) {
    start = count = 0;
    const int cx = bx * BCX + ci % BCX, cy = by * BCY + (ci / BCX) % BCY, cz = bz * BCZ + ci / (BCX * BCY);
    if (cx >= A.N[0] || cy >= A.N[1] || cz >= A.N[2]) return;
    const long long cell = ((long long)cz * A.N[1] + cy) * A.N[0] + cx;
    const unsigned a0 = A.offs[cell], a1 = A.offs[cell + 1];
    if (a1 < a0 || (long long)a1 > A.n) {
        if (threadIdx.x == 0 && A.flags) atomicOr(A.flags, PCG_FLAG_BAD_LAYOUT);
        return;
    }
    start = a0;
    count = a1 - a0;
}

// The walk of a CTA over its blocks and their batches.  Each role walks the same
// sequence with its own cursor and its own table of the current block's cell
// ranges, filled once per block by the role's threads between two of the role's
// named barriers (a warp-wide sync for the MMA warp).
struct Cursor {
    int blk;         // current block
    int bx, by, bz;  // its coordinates
    int ci;          // current cell of the block
    unsigned k;      // next particle of that cell
    int prev_blk;
};

template <int BAR, int NT>
__device__ __forceinline__ void role_sync() {
    if (NT == 32) __syncwarp();
    else asm volatile("bar.sync %0, %1;" ::"n"(BAR), "n"(NT) : "memory");
}

// A role-wide OR (the same result in every thread of the role), so that the
// role leaves its loop together.
template <int BAR, int NT>
__device__ __forceinline__ bool role_any(bool v) {
    if (NT == 32) return __any_sync(0xffffffffu, v);
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, %2, %3, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(BAR), "n"(NT)
        : "memory");
    return r != 0;
}

// Enter block blk (32-bit arithmetic: there are fewer blocks than cells, < 2^31):
// the role's NT threads (index lt) fill its table.
template <int BAR, int NT>
__device__ __forceinline__ void enter_block(const Args &A, int blk, Cursor &cu, Tab &tab, int lt) {
    cu.blk = blk;
    cu.ci = 0;
    cu.k = 0;
    cu.bx = blk % A.nb[0];
    cu.by = (blk / A.nb[0]) % A.nb[1];
    cu.bz = blk / (A.nb[0] * A.nb[1]);
    role_sync<BAR, NT>();  // every thread of the role is done with the previous table
    for (int ci = lt; ci < NCELL; ci += NT) cell_range(A, cu.bx, cu.by, cu.bz, ci, tab.start[ci], tab.count[ci]);
    role_sync<BAR, NT>();
}

template <int BAR, int NT>
__device__ __forceinline__ void cursor_start(const Args &A, int nblocks, Cursor &cu, Tab &tab, int lt) {
    cu.blk = nblocks;
    cu.prev_blk = -1;
    if ((int)blockIdx.x < nblocks) enter_block<BAR, NT>(A, (int)blockIdx.x, cu, tab, lt);
}

template <int BAR, int NT>
__device__ __forceinline__ Iter next_iter(const Args &A, int nblocks, Cursor &cu, Tab &tab, int lt) {
    Iter it;
    it.valid = false;
    while (cu.blk < nblocks) {
        int nb = 0;
#pragma unroll
        for (int j = 0; j < GP; ++j) it.bt[j] = Batch{-1, 0, 0};
        while (nb < GP && cu.ci < NCELL) {
            const unsigned cnt = tab.count[cu.ci];
            if (cu.k >= cnt) {  // next cell
                ++cu.ci;
                cu.k = 0;
                continue;
            }
            const unsigned rem = cnt - cu.k;
            const Batch b{cu.ci, tab.start[cu.ci] + cu.k, rem < (unsigned)KB ? rem : (unsigned)KB};
            if (nb == 0) it.bt[0] = b;
            else if (nb == 1) it.bt[1] = b;
            else it.bt[2] = b;
            ++nb;
            cu.k += KB;
        }
        if (nb > 0) {
            it.valid = true;
            it.blk = cu.blk;
            it.bx = cu.bx;
            it.by = cu.by;
            it.bz = cu.bz;
            it.first = cu.blk != cu.prev_blk;
            cu.prev_blk = cu.blk;
            return it;
        }
        // the block is exhausted: the next one of this CTA
        const int nxt = cu.blk + (int)gridDim.x;
        if (nxt < nblocks) enter_block<BAR, NT>(A, nxt, cu, tab, lt);
        else cu.blk = nblocks;
    }
    return it;
}

// Part PART (0, 1) of one particle's K column: A rows of components [C0, C1)
// and, for one of the two parts, the B column (W^T), 128-byte swizzle.
template <int MODE, int NC, int PART>
__device__ __forceinline__ void stage_part(unsigned char *abase, unsigned char *bbase, int chunk,
                                           const float (&W)[8], const float (&s)[NC]) {
    constexpr int C0 = NC == 9 ? (PART == 0 ? 0 : 4) : 0;  // 4 components + B, or 5 components
    constexpr int C1 = NC == 9 ? (PART == 0 ? 4 : 9) : (PART == 0 ? 1 : 0);
    constexpr bool BPART = PART == (NC == 9 ? 0 : 1);
#pragma unroll
    for (int a = 0; a < 8; ++a) {
        const int off = a * 128 + ((chunk ^ a) << 4);
#pragma unroll
        for (int c = C0; c < C1; ++c) {
            const float v = s[c] * W[a];
            unsigned char *dst = abase + c * 1024 + off;
            if (MODE == TF32) *reinterpret_cast<uint32_t *>(dst) = tc::to_tf32(v);
            else *reinterpret_cast<__nv_bfloat16 *>(dst) = __float2bfloat16_rn(v);
        }
        if (BPART) {
            unsigned char *dstb = bbase + off;
            if (MODE == TF32) *reinterpret_cast<uint32_t *>(dstb) = tc::to_tf32(W[a]);
            else *reinterpret_cast<__nv_bfloat16 *>(dstb) = __float2bfloat16_rn(W[a]);
        }
    }
}

template <int MODE, int NC>
__global__ void __launch_bounds__(kPThreads, 1) mass_tc_kernel(Args A) {
    using L = PLay<MODE, NC>;
    using O = Op<MODE, NC, GP>;
    using Wn = Win<NC>;
    constexpr int NB = Wn::NB, ACC_ROW = Wn::ACC_ROW, ACC_FLOATS = Wn::ACC_FLOATS;
    extern __shared__ __align__(1024) unsigned char smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::BAR_OFF);
    uint64_t *full = bars, *empty = bars + 2, *tfull = bars + 4, *tempty = bars + 6;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    Tab *tabs = reinterpret_cast<Tab *>(smem + L::TAB_OFF);  // [0] producers, [1] MMA warp, [2] read-back
    float *acc = reinterpret_cast<float *>(smem + L::WIN_OFF);
    int *rsh = reinterpret_cast<int *>(smem + L::RS_OFF);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (warp == 0) tc::tmem_alloc(tmem_slot, kPTmemCols);
    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&full[b], kProdThreads);    // every producer thread arrives
            tc::mbar_init(&empty[b], 1);              // tcgen05.commit
            tc::mbar_init(&tfull[b], 1);              // tcgen05.commit
            tc::mbar_init(&tempty[b], kEpiThreads);   // every read-back thread arrives
        }
        *abort_flag = 0;
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    const int nblocks = A.nb[0] * A.nb[1] * A.nb[2];
    unsigned n_inv = 0;
    bool timed_out = false;
    Cursor cu;

    if (warp < kProdWarps) {
        // ---- producers: stage the operands of every iteration ----
        const int pme = tid % (GP * KB), half = tid / (GP * KB);
        const int jme = pme / KB, kme = pme % KB;  // this thread's batch and particle
        auto produce = [&](long long i, const Iter &it, const Raw &raw) -> bool {
            const int s = (int)(i & 1);
            const bool ok = i < 2 || (tc::mbar_wait_sleep(&empty[s], (uint32_t)((i - 2) >> 1) & 1u, kSleepPolls, kSleepNs) &&
                                      !*abort_flag);
            if (role_any<kProdBar, kProdThreads>(!ok)) return false;
            const Batch mine = pick(it, jme);
            const int cx = it.bx * BCX + mine.ci % BCX, cy = it.by * BCY + (mine.ci / BCX) % BCY,
                      cz = it.bz * BCZ + mine.ci / (BCX * BCY);
            float W[8], sc[NC];
            prepare<NC>(A, raw, cx, cy, cz, half == 0, W, sc, n_inv);
            unsigned char *Aj = smem + s * L::STAGE + jme * O::BATCH;
            const int katom = (kme * O::EB) >> 7, kin = (kme * O::EB) & 127;
            const int chunk = kin >> 4, inb = kin & 15;
            unsigned char *abase = Aj + katom * O::A_KSTRIDE + inb;
            unsigned char *bbase = Aj + O::A_BYTES + katom * 1024 + inb;
            if (half == 0) stage_part<MODE, NC, 0>(abase, bbase, chunk, W, sc);
            else stage_part<MODE, NC, 1>(abase, bbase, chunk, W, sc);
            tc::fence_proxy_async_smem();  // the staged operands, for the tensor core
            tc::mbar_arrive(&full[s]);
            return true;
        };
        cursor_start<kProdBar, kProdThreads>(A, nblocks, cu, tabs[0], tid);
        // two iterations in registers: the particles of iteration i + 2 load while
        // iteration i + 1 is staged
        Iter it0 = next_iter<kProdBar, kProdThreads>(A, nblocks, cu, tabs[0], tid);
        Raw r0 = load_raw<NC>(A, pick(it0, jme), kme);
        Iter it1 = next_iter<kProdBar, kProdThreads>(A, nblocks, cu, tabs[0], tid);
        Raw r1 = load_raw<NC>(A, pick(it1, jme), kme);
        for (long long i = 0; it0.valid; i += 2) {
            if (!produce(i, it0, r0)) {
                timed_out = true;
                break;
            }
            it0 = next_iter<kProdBar, kProdThreads>(A, nblocks, cu, tabs[0], tid);
            r0 = load_raw<NC>(A, pick(it0, jme), kme);
            if (!it1.valid) break;
            if (!produce(i + 1, it1, r1)) {
                timed_out = true;
                break;
            }
            it1 = next_iter<kProdBar, kProdThreads>(A, nblocks, cu, tabs[0], tid);
            r1 = load_raw<NC>(A, pick(it1, jme), kme);
        }
    } else if (warp == kMmaWarp) {
        // ---- warp 15: the whole warp walks the cursor (its 32 lanes fill the cell
        // table of a new block at once); lane 0 waits, issues the MMAs and commits ----
        cursor_start<0, 32>(A, nblocks, cu, tabs[1], lane);
        Iter cur = next_iter<0, 32>(A, nblocks, cu, tabs[1], lane);
        long long i = 0;
        for (; cur.valid; ++i) {
            const int s = (int)(i & 1);
            bool ok = true;
            if (lane == 0) {
                ok = tc::mbar_wait_sleep(&full[s], (uint32_t)(i >> 1) & 1u, kSleepPolls, kSleepNs) && !*abort_flag &&
                     (i < 2 || tc::mbar_wait_sleep(&tempty[s], (uint32_t)((i - 2) >> 1) & 1u, kSleepPolls, kSleepNs));
                if (ok) {
                    tc::fence_after_sync();
                    constexpr uint32_t idesc = tc::instr_desc(MODE == TF32 ? 2u : 1u, 128, 16);
                    // descriptors of stage s: a base plus compile-time offsets
                    // (in 16-byte units) per batch and K step
                    const uint64_t ad0 = tc::smem_desc_sw128(tc::smem_addr(smem + s * L::STAGE), 1024);
                    const uint64_t bd0 = ad0 + (uint64_t)(O::A_BYTES >> 4);
                    const uint32_t dcol = tmem + 64u * s;
#pragma unroll
                    for (int jj = 0; jj < GP; ++jj) {
                        if (pick(cur, jj).ci < 0) continue;
#pragma unroll
                        for (int ks = 0; ks < O::KSTEPS; ++ks) {
                            const int kb = ks * 32, ka = kb >> 7, ko = kb & 127;
                            const uint64_t aoff = (uint64_t)((jj * O::BATCH + ka * O::A_KSTRIDE + ko) >> 4);
                            const uint64_t boff = (uint64_t)((jj * O::BATCH + ka * 1024 + ko) >> 4);
                            tc::mma<MODE == TF32>(dcol + 16u * jj, ad0 + aoff, bd0 + boff, idesc, ks > 0);
                        }
                    }
                    tc::commit(&empty[s]);
                    tc::commit(&tfull[s]);
                }
            }
            if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
                timed_out = true;
                break;
            }
            cur = next_iter<0, 32>(A, nblocks, cu, tabs[1], lane);
        }
        if (timed_out && lane == 0 && i > 0) {
            // the MMAs issued last complete before their commit arrives
            const long long l = i - 1;
            (void)tc::mbar_wait(&tfull[l & 1], (uint32_t)(l >> 1) & 1u, kMaxPolls);
        }
        __syncwarp();
    } else {
        // ---- warps 12-14: accumulators into the node window, the window into M ----
        const int et = tid - kEpiWarp0 * 32;  // 0..95
        const int q = warp & 3;               // lane quadrant of this warp
        cursor_start<kEpiBar, kEpiThreads>(A, nblocks, cu, tabs[2], et);
        Iter cur = next_iter<kEpiBar, kEpiThreads>(A, nblocks, cu, tabs[2], et);
        for (long long i = 0; cur.valid; ++i) {
            const int s = (int)(i & 1);
            const Iter nxt = next_iter<kEpiBar, kEpiThreads>(A, nblocks, cu, tabs[2], et);
            const bool last = !nxt.valid || nxt.blk != cur.blk;
            if (cur.first) {
                // clear the window once the previous block's bulk copy has read it
                if (et == 0) tc::bulk_wait_read_all();
                role_sync<kEpiBar, kEpiThreads>();
                for (int e = et; e < ACC_FLOATS / 4; e += kEpiThreads)
                    reinterpret_cast<float4 *>(acc)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (et < NROWS) rsh[et] = row_shift<NC>(A, cur.bx, cur.by, cur.bz, et);
                role_sync<kEpiBar, kEpiThreads>();
            }
            const bool ok = tc::mbar_wait_sleep(&tfull[s], (uint32_t)(i >> 1) & 1u, kSleepPolls, kSleepNs) && !*abort_flag;
            if (role_any<kEpiBar, kEpiThreads>(!ok)) {
                timed_out = true;
                break;
            }
            tc::fence_after_sync();
            const int r = 32 * q + lane;
            if (32 * q < 8 * NC) {  // warp-uniform: this quadrant holds rows in use
                // the accumulators of all batches first, then one wait
                uint32_t d[GP * 8];
#pragma unroll
                for (int jj = 0; jj < GP; ++jj)
                    if (pick(cur, jj).ci >= 0)
                        tc::tmem_ld8_async(tmem + ((uint32_t)(32 * q) << 16) + 64u * s + 16u * jj, d + 8 * jj);
                tc::tmem_wait_ld(d);
                if (r < 8 * NC) {
                    const int c = r >> 3, a = r & 7;
                    // offset of partner nn from corner a: P(nn) - P(a) + 13 with
                    // P(x) = 9 (x >> 2) + 3 ((x >> 1) & 1) + (x & 1)
                    const int pa = (a >> 2) * 9 + ((a >> 1) & 1) * 3 + (a & 1);
#pragma unroll
                    for (int jj = 0; jj < GP; ++jj) {
                        const int ci = pick(cur, jj).ci;
                        if (ci < 0) continue;
                        const int nx = ci % BCX + (a & 1), ny = (ci / BCX) % BCY + ((a >> 1) & 1),
                                  nz = ci / (BCX * BCY) + (a >> 2);
                        const int wr = nz * WNY + ny;
                        const int bi = wr * ACC_ROW + rsh[wr] + nx * NB + c - (pa - 13) * NC;
                        // partners at base + P(nn) NC, P(nn) in [0, 13]
                        if (!PCG_IN(bi, ACC_FLOATS) || !PCG_IN(bi + 13 * NC, ACC_FLOATS)) continue;
                        float *base = acc + bi;
                        float old[8];
#pragma unroll
                        for (int nn = 0; nn < 8; ++nn)
                            old[nn] = base[((nn >> 2) * 9 + ((nn >> 1) & 1) * 3 + (nn & 1)) * NC];
#pragma unroll
                        for (int nn = 0; nn < 8; ++nn)
                            base[((nn >> 2) * 9 + ((nn >> 1) & 1) * 3 + (nn & 1)) * NC] =
                                old[nn] + __uint_as_float(d[8 * jj + nn]);
                    }
                }
            }
            tc::fence_before_sync();
            tc::mbar_arrive(&tempty[s]);
            if (last) {
                tc::fence_proxy_async_smem();  // this thread's window writes, for the TMA
                role_sync<kEpiBar, kEpiThreads>();
                flush_window<NC, kEpiThreads>(A, acc, rsh, cur.bx, cur.by, cur.bz, et);
                if (et == 0) tc::bulk_commit();
            }
            cur = nxt;
        }
        if (et == 0) tc::bulk_wait_all();
    }

    if (timed_out) {
        *abort_flag = 1;
        if (A.flags) atomicOr(A.flags, PCG_FLAG_TIMEOUT);
    }
    tc::fence_before_sync();
    __syncthreads();
    const bool aborted = *abort_flag != 0;
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kPTmemCols);
    }
    if (!aborted) tail_pass<NC>(A, n_inv);
    warp_add_u64(A.n_invalid, n_inv);
}

}  // namespace

template <int MODE, int NC>
pcg_status launch_tc(const Args &A, cudaStream_t s) {
    using L = PLay<MODE, NC>;
    PCG_CHECK_CUDA(cudaFuncSetAttribute(mass_tc_kernel<MODE, NC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        L::SMEM));
    const long long nblocks = (long long)A.nb[0] * A.nb[1] * A.nb[2];
    const long long cap = num_sms();
    const long long grid = nblocks < cap ? nblocks : cap;
    static const char *const names[2][2] = {{"mass_matrix_tf32", "mass_matrix_bf16"},
                                            {"mass_scalar_tf32", "mass_scalar_bf16"}};
    prof::Mark mk(names[NC == 1][MODE], s);
    mass_tc_kernel<MODE, NC><<<(unsigned)grid, kPThreads, L::SMEM, s>>>(A);
    return launch_status();
}

template pcg_status launch_tc<TF32, 9>(const Args &, cudaStream_t);
template pcg_status launch_tc<BF16, 9>(const Args &, cudaStream_t);
template pcg_status launch_tc<TF32, 1>(const Args &, cudaStream_t);
template pcg_status launch_tc<BF16, 1>(const Args &, cudaStream_t);

}  // namespace mm
}  // namespace pcg
