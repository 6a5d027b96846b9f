// tile_sort.cu -- counting sort of particles into spatial tiles.
//
// Method: "Tiled current deposit" (Entity wiki), section "The tile-based
// spatial sort": ntiles = ceil(N / T) per axis, a tile key per particle,
// invalid particles parked in a sentinel bin after the last tile, tile_offsets
// as the prefix sum of the per-tile counts, and the SoA members physically
// permuted into tile order.  The page uses a vendor sort_by_key or a bin sort;
// here it is a hand-written counting sort, since the keys are small integers.
//
// GB300 design (bins B = n_tiles + 1):
//  * B <= kSmemBins: "chunked" sort.  G CTAs (a multiple of the 152 SMs) each
//    own a contiguous chunk of particles.  (1) count: block-private histogram in
//    shared memory, written out as counts[g][b]; (2) colscan: one thread per bin
//    scans its column over the G chunks (coalesced) giving each (chunk, bin)
//    its start inside the bin, and the bin totals; (3) a one-CTA exclusive scan
//    of the totals gives tile_offsets; (4) scatter: every CTA loads its
//    (chunk, bin) cursors into shared memory and places each particle with a
//    shared-memory atomic.  A chunk's particles of one tile land contiguously.
//  * B > kSmemBins (for example one bin per cell of a 64^3 grid): counts and
//    cursors live in global memory and are bumped with global atomics.
// No step waits on another CTA; kernel boundaries order the phases.
#include <cmath>

#include "common.cuh"
#include "tcgen05.cuh"

namespace pcg {
namespace {

constexpr unsigned kSmemBins = 32769;  // 128 KB + 4 B of shared counters
constexpr int kSortThreads = 512;
constexpr int kMaxPayload = 16;

struct KeyGeom {
    int nt0, nt1;  // tiles along x and y
    unsigned n_tiles;
    float N0, N1, N2;  // domain extent per axis (exact in fp32 up to 2^24)
    int tile;
};

struct Payload {
    const unsigned *in[kMaxPayload];
    unsigned *out[kMaxPayload];
};

template <int TILE>
__device__ __forceinline__ int tdiv(int i, int tile) {
    if (TILE > 0) return i / (TILE > 0 ? TILE : 1);  // constant divisor
    return i / tile;
}

// Tile key of one particle (sentinel n_tiles when any coordinate is outside [0, N)).
template <int DIM, int TILE>
__device__ __forceinline__ unsigned tile_key(const KeyGeom &g, float x, float y, float z) {
    bool ok = (x >= 0.f) & (x < g.N0) & (y >= 0.f) & (y < g.N1);
    if (DIM == 3) ok &= (z >= 0.f) & (z < g.N2);
    if (!ok) return g.n_tiles;
    int tx = tdiv<TILE>((int)x, g.tile);
    int ty = tdiv<TILE>((int)y, g.tile);
    int tz = DIM == 3 ? tdiv<TILE>((int)z, g.tile) : 0;
    return (unsigned)((tz * g.nt1 + ty) * g.nt0 + tx);
}

template <int DIM, int TILE>
__global__ void __launch_bounds__(kSortThreads)
    count_chunked_kernel(KeyGeom g, const float *__restrict__ kx, const float *__restrict__ ky,
                         const float *__restrict__ kz, long long n, long long chunk,
                         unsigned *__restrict__ counts, unsigned B,
                         unsigned long long *__restrict__ n_invalid) {
    extern __shared__ unsigned hist[];
    for (unsigned b = threadIdx.x; b < B; b += blockDim.x) hist[b] = 0;
    __syncthreads();
    const long long p0 = (long long)blockIdx.x * chunk;
    const long long p1 = min(n, p0 + chunk);
    unsigned inval = 0;
    // U independent particles per thread per round keep enough loads in flight
    constexpr int U = 8;
    for (long long q = p0 + threadIdx.x; q < p1; q += (long long)U * blockDim.x) {
        float x[U], y[U], z[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long p = q + (long long)u * blockDim.x;
            const bool in = p < p1;
            x[u] = in ? kx[p] : -1.f;
            y[u] = in ? ky[p] : 0.f;
            z[u] = (DIM == 3 && in) ? kz[p] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (q + (long long)u * blockDim.x >= p1) break;
            const unsigned k = tile_key<DIM, TILE>(g, x[u], y[u], z[u]);
            if (PCG_IN(k, B)) atomicAdd(&hist[k], 1u);
            inval += (k == g.n_tiles);
        }
    }
    warp_add_u64(n_invalid, inval);
    __syncthreads();
    unsigned *row = counts + (size_t)blockIdx.x * B;
    for (unsigned b = threadIdx.x; b < B; b += blockDim.x) row[b] = hist[b];
}

// counts[g][b] -> exclusive start of chunk g inside bin b (in place); totals[b].
__global__ void __launch_bounds__(256)
    colscan_kernel(unsigned *__restrict__ counts, unsigned *__restrict__ totals, unsigned G,
                   unsigned B) {
    const unsigned b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    unsigned run = 0;
    for (unsigned gi = 0; gi < G; ++gi) {
        unsigned *c = counts + (size_t)gi * B + b;
        const unsigned v = *c;
        *c = run;
        run += v;
    }
    totals[b] = run;
}

// Exclusive scan of in[0..L) into out[0..L) by one CTA of 1024 threads; optional
// second output copy.  Handles any L in segments of 1024 * 8 elements.
__global__ void __launch_bounds__(1024)
    scan_one_cta_kernel(const unsigned *__restrict__ in, unsigned *__restrict__ out,
                        unsigned *__restrict__ out2, unsigned L) {
    constexpr int kItems = 8;
    __shared__ unsigned warp_sums[32];
    __shared__ unsigned carry_s;
    if (threadIdx.x == 0) carry_s = 0;
    __syncthreads();
    const unsigned lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (unsigned seg = 0; seg < L; seg += 1024u * kItems) {
        unsigned v[kItems];
        unsigned sum = 0;
        const unsigned base = seg + threadIdx.x * kItems;
#pragma unroll
        for (int i = 0; i < kItems; ++i) {
            v[i] = (base + i < L) ? in[base + i] : 0u;
            sum += v[i];
        }
        // inclusive warp scan of the per-thread sums
        unsigned incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            unsigned t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= (unsigned)o) incl += t;
        }
        if (lane == 31) warp_sums[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            unsigned ws = warp_sums[lane];
            unsigned wi = ws;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                unsigned t = __shfl_up_sync(0xffffffffu, wi, o);
                if (lane >= (unsigned)o) wi += t;
            }
            warp_sums[lane] = wi - ws;  // exclusive prefix of warp totals
        }
        __syncthreads();
        unsigned run = carry_s + warp_sums[warp] + (incl - sum);
#pragma unroll
        for (int i = 0; i < kItems; ++i) {
            if (base + i < L) {
                out[base + i] = run;
                if (out2) out2[base + i] = run;
            }
            run += v[i];
        }
        __syncthreads();
        if (threadIdx.x == 1023) carry_s = run;  // last thread holds the segment total
        __syncthreads();
    }
}

template <int DIM, int TILE>
__global__ void __launch_bounds__(kSortThreads)
    scatter_chunked_kernel(KeyGeom g, const float *__restrict__ kx, const float *__restrict__ ky,
                           const float *__restrict__ kz, long long n, long long chunk,
                           const unsigned *__restrict__ starts, const unsigned *__restrict__ offs,
                           unsigned B, Payload pl, int np) {
    extern __shared__ unsigned cursor[];
    const unsigned *row = starts + (size_t)blockIdx.x * B;
    for (unsigned b = threadIdx.x; b < B; b += blockDim.x) cursor[b] = offs[b] + row[b];
    __syncthreads();
    const long long p0 = (long long)blockIdx.x * chunk;
    const long long p1 = min(n, p0 + chunk);
    for (long long p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
        const unsigned k = tile_key<DIM, TILE>(g, kx[p], ky[p], DIM == 3 ? kz[p] : 0.f);
        if (!PCG_IN(k, B)) continue;
        const unsigned slot = atomicAdd(&cursor[k], 1u);
        if (!PCG_IN(slot, n)) continue;
        for (int f = 0; f < np; ++f) pl.out[f][slot] = pl.in[f][p];
    }
}

template <int DIM, int TILE>
__global__ void __launch_bounds__(256)
    count_global_kernel(KeyGeom g, const float *__restrict__ kx, const float *__restrict__ ky,
                        const float *__restrict__ kz, long long n, unsigned *__restrict__ totals,
                        unsigned long long *__restrict__ n_invalid) {
    unsigned inval = 0;
    for (long long p = blockIdx.x * (long long)blockDim.x + threadIdx.x; p < n;
         p += (long long)gridDim.x * blockDim.x) {
        const unsigned k = tile_key<DIM, TILE>(g, kx[p], ky[p], DIM == 3 ? kz[p] : 0.f);
        if (PCG_IN(k, g.n_tiles + 1u)) atomicAdd(&totals[k], 1u);
        inval += (k == g.n_tiles);
    }
    warp_add_u64(n_invalid, inval);
}

template <int DIM, int TILE>
__global__ void __launch_bounds__(256)
    scatter_global_kernel(KeyGeom g, const float *__restrict__ kx, const float *__restrict__ ky,
                          const float *__restrict__ kz, long long n, unsigned *__restrict__ cursor,
                          Payload pl, int np) {
    for (long long p = blockIdx.x * (long long)blockDim.x + threadIdx.x; p < n;
         p += (long long)gridDim.x * blockDim.x) {
        const unsigned k = tile_key<DIM, TILE>(g, kx[p], ky[p], DIM == 3 ? kz[p] : 0.f);
        if (!PCG_IN(k, g.n_tiles + 1u)) continue;
        const unsigned slot = atomicAdd(&cursor[k], 1u);
        if (!PCG_IN(slot, n)) continue;
        for (int f = 0; f < np; ++f) pl.out[f][slot] = pl.in[f][p];
    }
}

// ---------------------------------------------------------------------------
// Two-pass partition for outputs larger than L2 (MSD order).
// Pass 1 moves every particle into one of <= 256 coarse buckets of `tpb`
// consecutive tiles, pass 2 into its tile inside the bucket.  One persistent
// CTA per SM walks batches of `bs` consecutive input rows (4096 where shared
// memory allows), dealt round-robin:
//  * a producer warp copies the batch's fields global -> shared, one bulk
//    (TMA) copy per field, into a single staging buffer, and refills a field
//    for the next batch as soon as every worker warp has finished reading it
//    (an mbarrier per field each way: "full" when the copy has landed, "free"
//    when the 16 worker warps are done with it).  The key inputs come first,
//    so the next batch can be ranked while this one is still being written;
//  * 16 worker warps count the digits in shared memory (the counting atomic's
//    return value is the particle's rank inside its digit), scan them, reserve
//    one contiguous output run per non-empty digit with one global atomic, and
//    list the batch in digit order in a 16-bit permutation;
//  * consecutive threads then write consecutive output slots field by field,
//    so every digit's run leaves the SM as contiguous stores, and the open
//    sectors are one per bucket or tile frontier (the runs of successive
//    batches, from any CTA, abut).
// Measured on GB300: the store phase costs about the same per run of a digit
// whatever its length, so the batch is as large as shared memory allows.
// Every mbarrier wait is bounded; a timeout sets PCG_FLAG_TIMEOUT, and the
// workers leave together at their next barrier (before any further global
// write), the producer after its copies in flight have landed.
constexpr int kPartWorkers = 512;
constexpr int kPartThreads = kPartWorkers + 32;  // + the producer warp
constexpr int kWorkerWarps = kPartWorkers / 32;
constexpr int kMaxBatch = 4096;
constexpr int kItems = kMaxBatch / kPartWorkers;
constexpr unsigned kMaxPassBins = 2048;
// Pass-1 buckets.  A batch's runs are about bs / digits rows long and the
// store phase costs about the same per run, so the two passes' digit counts
// are balanced: 128 buckets (257 tiles each at 256^3 / 8) measured best among
// 96, 128, 160, 181 and 256 (pass 1 writes one field more than pass 2).  Up to
// kMaxBuckets when the tiles per bucket would exceed kMaxPassBins.
constexpr unsigned kBuckets = 128;
constexpr unsigned kMaxBuckets = 256;
constexpr int kMaxRows = kMaxPayload + 3;
constexpr uint32_t kPartPolls = 1u << 20;  // bounded waits: about 1 s with the 1 us suspend hint
constexpr uint32_t kPartSleepNs = 1000;
constexpr int kWorkBar = 1;  // named barrier of the worker warps

__device__ __forceinline__ void work_sync() {
    asm volatile("bar.sync %0, %1;" ::"n"(kWorkBar), "n"(kPartWorkers) : "memory");
}
// OR over the worker threads, the same in all of them (and a worker barrier)
__device__ __forceinline__ bool work_any(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, %2, %3, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(kWorkBar), "n"(kPartWorkers)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *mbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(tc::smem_addr(mbar)), "r"(bytes)
                 : "memory");
}
// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned)
// global -> shared, completing on `mbar`'s transaction count.
__device__ __forceinline__ void bulk_g2s(void *sdst, const void *gsrc, uint32_t bytes, uint64_t *mbar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            tc::smem_addr(sdst)),
        "l"(gsrc), "r"(bytes), "r"(tc::smem_addr(mbar))
        : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// out[0..nb) = exclusive scan of in[0..nb) (nb <= kMaxPassBins) by the worker
// warps; in is read after the caller's barrier, out is ready after the last one.
__device__ void work_exclusive_scan(const unsigned *in, unsigned *out, unsigned nb, unsigned *warp_tot) {
    constexpr int PER = kMaxPassBins / kPartWorkers;
    const unsigned lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned loc[PER];
    unsigned sum = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const unsigned b = threadIdx.x * PER + i;
        loc[i] = b < nb ? in[b] : 0u;
        sum += loc[i];
    }
    unsigned incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= (unsigned)o) incl += t;
    }
    if (lane == 31) warp_tot[warp] = incl;
    work_sync();
    if (warp == 0) {
        const unsigned w = lane < (unsigned)kWorkerWarps ? warp_tot[lane] : 0u;
        unsigned wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned t = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= (unsigned)o) wi += t;
        }
        if (lane < (unsigned)kWorkerWarps) warp_tot[lane] = wi - w;
    }
    work_sync();
    unsigned run = warp_tot[warp] + incl - sum;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const unsigned b = threadIdx.x * PER + i;
        if (b < nb) out[b] = run;
        run += loc[i];
    }
    work_sync();
}

// One batch: input rows [b0, b0 + len), digits [base, base + nb).
struct BatchGeo {
    long long b0;
    unsigned len, base, nb;
};

struct PartArgs {
    KeyGeom g;
    const float *kx, *ky, *kz;
    long long n;
    Payload pl;
    int np;
    const unsigned *in_key;     // pass 2: tile keys written by pass 1
    unsigned *out_key;          // pass 1 of two: tile keys for pass 2
    const uint32_t *offs;       // tile offsets (bin starts)
    unsigned *gcursor;          // next free output slot per bin (pass 1: per bucket)
    const unsigned *batch_off;  // pass 2: first batch of each bucket
    unsigned *flags;            // pcg_stats error flags (may be null)
    unsigned tpb, B, nb1, nbcap, bs, nbatch;
};

// PASS 1: digit = bucket of the tile key computed from key positions; writes the
//         payload and the key to the intermediate arrays (or, with FINAL, the
//         payload straight to the output when one pass suffices).
// PASS 2: digit = tile inside the batch's bucket; key read from the
//         intermediate arrays; writes the final payload.
// Shared memory: nr = np + NK fields of (bs + 4) words (payload, then the key
// inputs; pass 1 of two overwrites the x field with the tile key) | hist |
// lstart | gbase ([nbcap] each) | bucket starts and batch offsets ([nb1 + 1]
// each, pass 2) | perm[bs] | sdig[bs] (16-bit).
template <int DIM, int TILE, int PASS, bool FINAL>
__global__ void __launch_bounds__(kPartThreads, 1) partition_kernel(const PartArgs a) {
    extern __shared__ __align__(16) unsigned sm[];
    __shared__ __align__(8) uint64_t full[kMaxRows], freeb[kMaxRows];
    __shared__ BatchGeo s_geo[4];
    __shared__ unsigned warp_tot[kWorkerWarps];
    constexpr bool kKey = PASS == 1 && !FINAL;
    constexpr int NK = PASS == 1 ? DIM : 1;  // key fields: positions, or the key
    const int np = a.np, nr = np + NK;
    const long long n = a.n;
    const unsigned bs = a.bs, row = bs + 4;
    unsigned *hist = sm + (size_t)nr * row;  // counts, then ranks
    unsigned *lstart = hist + a.nbcap;       // local exclusive starts
    unsigned *gbase = lstart + a.nbcap;      // reserved global starts
    unsigned *bstart = gbase + a.nbcap;      // pass 2: bucket b = [bstart[b], bstart[b+1])
    unsigned *boff = bstart + (PASS == 2 ? a.nb1 + 1 : 0u);  // pass 2: first batch of bucket b
    unsigned short *perm = reinterpret_cast<unsigned short *>(boff + (PASS == 2 ? a.nb1 + 1 : 0u));
    unsigned short *sdig = perm + bs;
    const unsigned tid = threadIdx.x, lane = tid & 31;

    if (tid == 0) {
        for (int r = 0; r < nr; ++r) {
            tc::mbar_init(&full[r], 1);
            tc::mbar_init(&freeb[r], kWorkerWarps);
        }
        fence_mbar_init();
    }
    for (unsigned d = tid; d < a.nbcap; d += kPartThreads) hist[d] = 0;
    if (PASS == 2) {
        for (unsigned b = tid; b <= a.nb1; b += kPartThreads) {
            const unsigned long long t = (unsigned long long)b * a.tpb;
            bstart[b] = t < a.B ? a.offs[t] : (unsigned)n;
            boff[b] = a.batch_off[b];
        }
    }
    __syncthreads();

    if (tid >= (unsigned)kPartWorkers) {
        // ---- producer warp ----
        auto geometry = [&](unsigned k, BatchGeo &o) {
            o.len = 0;
            o.b0 = 0;
            o.base = 0;
            o.nb = 1;
            if (k >= a.nbatch) return;
            if (PASS == 1) {
                o.b0 = (long long)k * bs;
                const long long rem = n - o.b0;
                o.len = rem < (long long)bs ? (unsigned)(rem > 0 ? rem : 0) : bs;
                o.nb = FINAL ? a.B : a.nb1;
            } else {
                // bucket of batch k: largest b with boff[b] <= k
                unsigned lo = 0, hi = a.nb1;
                while (lo < hi) {
                    const unsigned mid = (lo + hi + 1) / 2;
                    if (boff[mid] <= k) lo = mid;
                    else hi = mid - 1;
                }
                if (lo >= a.nb1) return;
                o.b0 = (long long)bstart[lo] + (long long)(k - boff[lo]) * bs;
                const long long rem = (long long)bstart[lo + 1] - o.b0;
                o.len = rem < (long long)bs ? (unsigned)(rem > 0 ? rem : 0) : bs;
                o.base = lo * a.tpb;
                o.nb = min(a.tpb, a.B - o.base);
            }
        };
        auto source = [&](int r) -> const unsigned * {
            if (r < np) return a.pl.in[r];
            if (PASS == 2) return a.in_key;
            const int q = r - np;
            return reinterpret_cast<const unsigned *>(q == 0 ? a.kx : (q == 1 ? a.ky : a.kz));
        };
        // field r of batch o into its staging row: element b0 lands at row[b0 % 4];
        // one bulk copy from the 16-byte boundary at or below b0 to the one at
        // or below the end, plain loads for the rest (all of it when the array
        // is not 16-byte aligned)
        auto stage = [&](int r, const BatchGeo &o) {
            const unsigned *src = source(r);
            unsigned *dst = sm + (size_t)r * row;
            const long long a0 = o.b0 & ~3ll;
            const int sh = (int)(o.b0 - a0);
            const long long e = o.b0 + o.len;
            const bool al = (reinterpret_cast<uintptr_t>(src) & 15) == 0;
            long long e16 = al ? (e & ~3ll) : a0;
            if (e16 < a0) e16 = a0;
            const long long t0 = e16 > o.b0 ? e16 : o.b0;
            for (long long t = t0 + lane; t < e; t += 32) dst[sh + (t - o.b0)] = src[t];
            __syncwarp();
            if (lane == 0) {
                const uint32_t bytes = (uint32_t)(e16 - a0) * 4u;
                if (bytes) {
                    mbar_expect_tx(&full[r], bytes);
                    bulk_g2s(dst, src + a0, bytes, &full[r]);
                } else {
                    tc::mbar_arrive(&full[r]);
                }
            }
        };
        bool ok = true;
        unsigned k = 0;
        uint32_t issued = 0;  // fields of batch k already issued (bit r)
        for (;; ++k) {
            BatchGeo o;
            geometry(blockIdx.x + k * gridDim.x, o);
            if (lane == 0) s_geo[k & 3] = o;
            issued = 0;
            // the key fields first: the workers rank with them before they need the payload
            for (int q = 0; q < nr && ok; ++q) {
                const int r = q < NK ? np + q : q - NK;
                if (k > 0) {
                    // the workers are done with this field of the previous batch
                    bool w = true;
                    if (lane == 0) w = tc::mbar_wait_sleep(&freeb[r], (k - 1) & 1, kPartPolls, kPartSleepNs);
                    ok = __shfl_sync(0xffffffffu, w, 0);
                    if (!ok) break;
                }
                if (o.len == 0) {
                    // no batch left: complete the key fields' phases so that
                    // the workers read the empty geometry and leave
                    if (q < NK) {
                        if (lane == 0) tc::mbar_arrive(&full[r]);
                        issued |= 1u << r;
                    }
                    continue;
                }
                stage(r, o);
                issued |= 1u << r;
            }
            if (!ok || o.len == 0) break;
        }
        if (!ok) {
            // leave only after the copies in flight have landed
            if (lane == 0) {
                for (int r = 0; r < nr; ++r) {
                    if (issued & (1u << r)) (void)tc::mbar_wait_sleep(&full[r], k & 1, kPartPolls, kPartSleepNs);
                    else if (k > 0) (void)tc::mbar_wait_sleep(&full[r], (k - 1) & 1, kPartPolls, kPartSleepNs);
                }
                if (a.flags) atomicOr(a.flags, PCG_FLAG_TIMEOUT);
            }
        }
        return;
    }

    // ---- worker warps ----
    bool bad = false;  // this thread gave up a wait
    for (unsigned k = 0;; ++k) {
        const uint32_t par = k & 1;
        for (int q = 0; q < NK; ++q)
            bad |= !tc::mbar_wait_sleep(&full[np + q], par, kPartPolls, kPartSleepNs);
        BatchGeo cur = s_geo[k & 3];
        // (after a timeout the geometry may be stale: keep every index in range
        // until the workers leave together below)
        if (cur.len > bs) cur.len = bs;
        if (cur.nb < 1 || cur.nb > a.nbcap) cur.nb = 1;
        const int sh = (int)(cur.b0 & 3);
        unsigned *keyrow = sm + (size_t)np * row + sh;
        unsigned dig[kItems], rk[kItems];
#pragma unroll
        for (int j = 0; j < kItems; ++j) {
            const unsigned i = tid + j * kPartWorkers;
            dig[j] = 0xffffffffu;
            if (i < cur.len) {
                unsigned key;
                if (PASS == 1) {
                    const float x = __uint_as_float(keyrow[i]);
                    const float y = __uint_as_float(keyrow[row + i]);
                    const float z = DIM == 3 ? __uint_as_float(keyrow[2 * row + i]) : 0.f;
                    key = tile_key<DIM, TILE>(a.g, x, y, z);
                    if (kKey) keyrow[i] = key;  // the x field now holds the key
                } else {
                    key = keyrow[i];
                }
                unsigned d = (PASS == 1) ? (FINAL ? key : key / a.tpb) : key - cur.base;
                if (d >= cur.nb) d = cur.nb - 1;  // defensive: never index outside the histogram
                dig[j] = d;
                rk[j] = atomicAdd(&hist[d], 1u);
            }
        }
        // key fields that are not written out are free for the next batch
        __syncwarp();
        if (lane == 0)
            for (int q = kKey ? 1 : 0; q < NK; ++q) tc::mbar_arrive(&freeb[np + q]);
        if (work_any(bad || cur.len == 0)) break;  // uniform: done, or a wait gave up
        work_exclusive_scan(hist, lstart, cur.nb, warp_tot);
        for (unsigned d = tid; d < cur.nb; d += kPartWorkers) {
            const unsigned c = hist[d];
            gbase[d] = c ? atomicAdd(&a.gcursor[cur.base + d], c) : 0u;
            hist[d] = 0;  // ready for the next batch
        }
#pragma unroll
        for (int j = 0; j < kItems; ++j) {
            if (dig[j] == 0xffffffffu) continue;
            const unsigned slot = lstart[dig[j]] + rk[j];
            perm[slot] = (unsigned short)(tid + j * kPartWorkers);
            sdig[slot] = (unsigned short)dig[j];
        }
        work_sync();
        // this thread's output slots: source row and global position
        unsigned src[kItems], gpos[kItems];
#pragma unroll
        for (int j = 0; j < kItems; ++j) {
            const unsigned s = tid + j * kPartWorkers;
            src[j] = 0xffffffffu;
            if (s < cur.len) {
                const unsigned i = perm[s], d = sdig[s];
                const unsigned gp = gbase[d] + (s - lstart[d]);
                if (PCG_IN(gp, n) && (long long)gp < n && PCG_IN(i, cur.len)) {
                    src[j] = i;
                    gpos[j] = gp;
                }
            }
        }
        // write every digit's run with consecutive threads, field by field,
        // releasing each field to the producer as soon as this warp is done
        if (kKey) {
#pragma unroll
            for (int j = 0; j < kItems; ++j)
                if (src[j] != 0xffffffffu) a.out_key[gpos[j]] = keyrow[src[j]];
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&freeb[np]);
        }
        for (int f = 0; f < np; ++f) {
            bad |= !tc::mbar_wait_sleep(&full[f], par, kPartPolls, kPartSleepNs);
            const unsigned *fr = sm + (size_t)f * row + sh;
            unsigned *out = a.pl.out[f];
#pragma unroll
            for (int j = 0; j < kItems; ++j)
                if (src[j] != 0xffffffffu) out[gpos[j]] = fr[src[j]];
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&freeb[f]);
        }
    }
    if (bad && a.flags) atomicOr(a.flags, PCG_FLAG_TIMEOUT);
}

size_t partition_smem(int DIM, int pass, bool final_, int np, unsigned nbcap, unsigned nb1, unsigned bs) {
    const int nk = pass == 1 ? DIM : 1;
    const size_t row = (size_t)(bs + 4) * 4;
    size_t b = (size_t)(np + nk) * row;
    b += (size_t)3 * nbcap * 4;
    if (pass == 2) b += (size_t)2 * (nb1 + 1) * 4;
    b += (size_t)bs * 4;  // perm + sdig
    return b;
}

// Largest batch (<= kMaxBatch, a multiple of kPartWorkers) whose buffers fit.
unsigned partition_batch(int DIM, int pass, bool final_, int np, unsigned nbcap, unsigned nb1) {
    constexpr size_t kSmemCap = 227 * 1024 - 1024;  // less the static shared memory
    for (unsigned bs = kMaxBatch; bs > (unsigned)kPartWorkers; bs /= 2)
        if (partition_smem(DIM, pass, final_, np, nbcap, nb1, bs) <= kSmemCap) return bs;
    return kPartWorkers;
}

// cursor1[b] = start of bucket b; cursor2[t] = start of tile t (written by the
// scan); batch_off = exclusive scan of the per-bucket batch counts.
__global__ void __launch_bounds__(1024)
    bucket_setup_kernel(const uint32_t *__restrict__ offs, long long n, unsigned B, unsigned tpb,
                        unsigned nb1, unsigned bs, unsigned *__restrict__ cursor1,
                        unsigned *__restrict__ batch_off) {
    __shared__ unsigned cnt[kMaxBuckets + 1];
    const unsigned b = threadIdx.x;
    if (b < nb1) {
        const unsigned t0 = b * tpb, t1 = min(t0 + tpb, B);
        const long long start = offs[t0];
        const long long end = t1 < B ? (long long)offs[t1] : n;
        cursor1[b] = (unsigned)start;
        const long long size = end > start ? end - start : 0;
        cnt[b] = (unsigned)((size + bs - 1) / bs);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned run = 0;
        for (unsigned i = 0; i < nb1; ++i) {
            batch_off[i] = run;
            run += cnt[i];
        }
        batch_off[nb1] = run;
    }
}

enum Path { kChunked = 0, kGlobal = 1, kTwoPass = 2 };

struct Plan {
    int path;
    unsigned B;
    unsigned G;        // chunks (chunked path and the chunked count of the two-pass path)
    long long chunk;   // particles per chunk
    unsigned tpb, nb1; // two-pass: tiles per bucket, buckets (1 = single pass)
    unsigned bs1, bs2; // two-pass: batch rows of pass 1 and pass 2
    size_t smem1, smem2;
    size_t bytes;      // workspace bytes
    size_t smem;       // dynamic shared memory of the chunked count / scatter
    // workspace layout (byte offsets)
    size_t o_counts, o_totals, o_cursor, o_cursor1, o_batch, o_inter, o_key;
    size_t inter_stride;  // bytes between the intermediate payload arrays
};

// Path choice.  The chunked path writes each (chunk, bin) run 4 bytes at a
// time as its particles arrive, so every run keeps one partly written sector
// per payload field open; that is fine while the whole output stays in L2.  For
// larger outputs the open sectors are evicted half written and DRAM does
// read-modify-write on every sector, so the two-pass partition is used.
constexpr double kL2Resident = 96.0 * 1024 * 1024;

Plan make_plan(const TileGrid &tg, long long n, int n_payload, int dim) {
    Plan p{};
    p.B = (unsigned)(tg.n_tiles + 1);
    const double out = (double)n * n_payload * 4.0;
    const bool small_bins = p.B <= kSmemBins;
    if (out <= kL2Resident) p.path = small_bins ? kChunked : kGlobal;
    else p.path = kTwoPass;
    if (p.path == kTwoPass) {
        if (p.B <= kMaxPassBins) {
            p.nb1 = 1;
            p.tpb = p.B;
        } else {
            p.tpb = (p.B + kBuckets - 1) / kBuckets;
            if (p.tpb > kMaxPassBins) p.tpb = (p.B + kMaxBuckets - 1) / kMaxBuckets;
            if (p.tpb > kMaxPassBins) p.path = kGlobal;  // too many bins for two passes
            p.nb1 = (p.B + p.tpb - 1) / p.tpb;
        }
    }
    // chunked counting (used by the chunked path and to count for the two-pass path)
    if (small_bins) {
        p.smem = (size_t)p.B * sizeof(unsigned);
        long long per_sm = (228 * 1024) / (long long)(p.smem + 1024);
        if (per_sm < 1) per_sm = 1;
        if (per_sm > 4) per_sm = 4;
        long long G = (long long)num_sms() * per_sm;
        long long max_g = (n + 1023) / 1024;
        if (max_g < 1) max_g = 1;
        if (G > max_g) G = max_g;
        p.G = (unsigned)G;
        p.chunk = align_up((size_t)((n + G - 1) / G), 4);  // chunks start 16-byte aligned
        if (p.chunk < 4) p.chunk = 4;
    }
    if (p.path == kTwoPass) {
        const bool fin = p.nb1 == 1;
        const unsigned cap1 = fin ? p.B : p.nb1;
        p.bs1 = partition_batch(dim, 1, fin, n_payload, cap1, p.nb1);
        p.smem1 = partition_smem(dim, 1, fin, n_payload, cap1, p.nb1, p.bs1);
        if (!fin) {
            p.bs2 = partition_batch(dim, 2, false, n_payload, p.tpb, p.nb1);
            p.smem2 = partition_smem(dim, 2, false, n_payload, p.tpb, p.nb1, p.bs2);
        }
    }
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o += align_up(bytes, 256);
        return at;
    };
    const size_t b4 = (size_t)p.B * sizeof(unsigned);
    if (p.path == kChunked) {
        p.o_counts = take((size_t)p.G * b4);
        p.o_totals = take(b4);
    } else if (p.path == kGlobal) {
        p.o_totals = take(b4);
        p.o_cursor = take(b4);
    } else {
        if (small_bins) p.o_counts = take((size_t)p.G * b4);
        p.o_totals = take(b4);
        p.o_cursor = take(b4);
        p.o_cursor1 = take((kMaxBuckets + 1) * sizeof(unsigned));
        p.o_batch = take((kMaxBuckets + 1) * sizeof(unsigned));
        if (p.nb1 > 1) {
            p.inter_stride = align_up((size_t)n * 4 + 16, 256);
            p.o_inter = take(p.inter_stride * n_payload);
            p.o_key = take((size_t)n * 4 + 16);
        }
    }
    p.bytes = o;
    return p;
}

template <int DIM, int TILE>
pcg_status count_into_totals(const KeyGeom &g, const Plan &pl, long long n, const float *const *kp,
                             unsigned char *ws, unsigned long long *n_invalid, cudaStream_t s) {
    const float *kz = DIM == 3 ? kp[2] : kp[0];
    unsigned *totals = reinterpret_cast<unsigned *>(ws + pl.o_totals);
    if (pl.B <= kSmemBins) {
        unsigned *counts = reinterpret_cast<unsigned *>(ws + pl.o_counts);
        if (pl.smem > 48 * 1024)
            PCG_CHECK_CUDA(cudaFuncSetAttribute(count_chunked_kernel<DIM, TILE>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                (int)pl.smem));
        {
            prof::Mark mk("sort_count", s);
            count_chunked_kernel<DIM, TILE><<<pl.G, kSortThreads, pl.smem, s>>>(
                g, kp[0], kp[1], kz, n, pl.chunk, counts, pl.B, n_invalid);
        }
        PCG_CHECK_LAUNCH();
        prof::Mark mk("sort_colscan", s);
        colscan_kernel<<<(pl.B + 255) / 256, 256, 0, s>>>(counts, totals, pl.G, pl.B);
        return launch_status();
    }
    pcg_status st = zero_f32(reinterpret_cast<float *>(totals), pl.B, s);
    if (st != PCG_OK) return st;
    prof::Mark mk("sort_count_global", s);
    count_global_kernel<DIM, TILE><<<(unsigned)num_sms() * 8, 256, 0, s>>>(g, kp[0], kp[1], kz, n,
                                                                        totals, n_invalid);
    return launch_status();
}

template <int DIM, int TILE>
pcg_status run_sort(const TileGrid &tg, const Plan &pl, long long n, const float *const *kp,
                    const Payload &py, int np, uint32_t *offs, unsigned long long *n_invalid,
                    unsigned *flags, unsigned char *ws, cudaStream_t s) {
    KeyGeom g;
    g.nt0 = tg.nt[0];
    g.nt1 = tg.nt[1];
    g.n_tiles = (unsigned)tg.n_tiles;
    g.N0 = (float)tg.N[0];
    g.N1 = (float)tg.N[1];
    g.N2 = (float)tg.N[2];
    g.tile = tg.tile;
    const float *kz = DIM == 3 ? kp[2] : kp[0];
    pcg_status st = count_into_totals<DIM, TILE>(g, pl, n, kp, ws, n_invalid, s);
    if (st != PCG_OK) return st;
    unsigned *totals = reinterpret_cast<unsigned *>(ws + pl.o_totals);
    if (pl.path == kChunked) {
        unsigned *counts = reinterpret_cast<unsigned *>(ws + pl.o_counts);
        {
            prof::Mark mk("sort_scan", s);
            scan_one_cta_kernel<<<1, 1024, 0, s>>>(totals, offs, nullptr, pl.B);
        }
        PCG_CHECK_LAUNCH();
        if (pl.smem > 48 * 1024)
            PCG_CHECK_CUDA(cudaFuncSetAttribute(scatter_chunked_kernel<DIM, TILE>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                (int)pl.smem));
        prof::Mark mk("sort_scatter", s);
        scatter_chunked_kernel<DIM, TILE><<<pl.G, kSortThreads, pl.smem, s>>>(
            g, kp[0], kp[1], kz, n, pl.chunk, counts, offs, pl.B, py, np);
        return launch_status();
    }
    unsigned *cursor = reinterpret_cast<unsigned *>(ws + pl.o_cursor);
    {
        prof::Mark mk("sort_scan", s);
        scan_one_cta_kernel<<<1, 1024, 0, s>>>(totals, offs, cursor, pl.B);
    }
    PCG_CHECK_LAUNCH();
    if (pl.path == kGlobal) {
        prof::Mark mk("sort_scatter_global", s);
        scatter_global_kernel<DIM, TILE><<<(unsigned)num_sms() * 8, 256, 0, s>>>(g, kp[0], kp[1], kz, n,
                                                                              cursor, py, np);
        return launch_status();
    }
    const unsigned sms = (unsigned)num_sms();
    PartArgs a{};
    a.g = g;
    a.kx = kp[0];
    a.ky = kp[1];
    a.kz = kz;
    a.n = n;
    a.np = np;
    a.offs = offs;
    a.flags = flags;
    a.B = pl.B;
    a.nb1 = pl.nb1;
    a.tpb = pl.tpb;
    if (pl.nb1 == 1) {
        // one pass: the digits are the tiles
        auto kern = partition_kernel<DIM, TILE, 1, true>;
        PCG_CHECK_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem1));
        a.pl = py;
        a.gcursor = cursor;
        a.nbcap = pl.B;
        a.bs = pl.bs1;
        a.nbatch = (unsigned)((n + pl.bs1 - 1) / pl.bs1);
        prof::Mark mk("sort_partition", s);
        kern<<<min(a.nbatch, sms), kPartThreads, pl.smem1, s>>>(a);
        return launch_status();
    }
    unsigned *cursor1 = reinterpret_cast<unsigned *>(ws + pl.o_cursor1);
    unsigned *batch = reinterpret_cast<unsigned *>(ws + pl.o_batch);
    unsigned *ikey = reinterpret_cast<unsigned *>(ws + pl.o_key);
    PartArgs a1 = a, a2 = a;
    for (int f = 0; f < np; ++f) {
        unsigned *inter = reinterpret_cast<unsigned *>(ws + pl.o_inter + (size_t)f * pl.inter_stride);
        a1.pl.in[f] = py.in[f];
        a1.pl.out[f] = inter;
        a2.pl.in[f] = inter;
        a2.pl.out[f] = py.out[f];
    }
    a1.out_key = ikey;
    a1.gcursor = cursor1;
    a1.nbcap = pl.nb1;
    a1.bs = pl.bs1;
    a1.nbatch = (unsigned)((n + pl.bs1 - 1) / pl.bs1);
    a2.in_key = ikey;
    a2.gcursor = cursor;
    a2.batch_off = batch;
    a2.nbcap = pl.tpb;
    a2.bs = pl.bs2;
    // upper bound on the bucket-aligned batches; the ones past the real count are empty
    a2.nbatch = (unsigned)((n + pl.bs2 - 1) / pl.bs2) + pl.nb1;
    {
        prof::Mark mk("sort_bucket_setup", s);
        bucket_setup_kernel<<<1, 1024, 0, s>>>(offs, n, pl.B, pl.tpb, pl.nb1, pl.bs2, cursor1, batch);
    }
    PCG_CHECK_LAUNCH();
    auto k1 = partition_kernel<DIM, TILE, 1, false>;
    auto k2 = partition_kernel<DIM, TILE, 2, false>;
    PCG_CHECK_CUDA(cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem1));
    PCG_CHECK_CUDA(cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem2));
    {
        prof::Mark mk("sort_partition1", s);
        k1<<<min(a1.nbatch, sms), kPartThreads, pl.smem1, s>>>(a1);
    }
    PCG_CHECK_LAUNCH();
    prof::Mark mk("sort_partition2", s);
    k2<<<min(a2.nbatch, sms), kPartThreads, pl.smem2, s>>>(a2);
    return launch_status();
}

template <int DIM>
pcg_status dispatch_tile(const TileGrid &tg, const Plan &pl, long long n, const float *const *kp,
                         const Payload &py, int np, uint32_t *offs, unsigned long long *ni,
                         unsigned *fl, unsigned char *ws, cudaStream_t s) {
    switch (tg.tile) {
        case 1: return run_sort<DIM, 1>(tg, pl, n, kp, py, np, offs, ni, fl, ws, s);
        case 4: return run_sort<DIM, 4>(tg, pl, n, kp, py, np, offs, ni, fl, ws, s);
        case 8: return run_sort<DIM, 8>(tg, pl, n, kp, py, np, offs, ni, fl, ws, s);
        default: return run_sort<DIM, 0>(tg, pl, n, kp, py, np, offs, ni, fl, ws, s);
    }
}

bool valid_sort_args(int32_t dim, const int32_t *grid, int32_t tile, int64_t n, TileGrid *tg) {
    if (n < 0 || n >= 0xffffffffll) return false;
    if (tile < 1 || tile > 64) return false;
    return make_tile_grid(dim, grid, tile, tg);
}

}  // namespace
}  // namespace pcg

extern "C" pcg_status pcg_tile_sort_workspace_size(int32_t dim, const int32_t *grid, int32_t tile,
                                                   int64_t n, int32_t n_payload, size_t *bytes) {
    using namespace pcg;
    TileGrid tg;
    if (bytes == nullptr || !valid_sort_args(dim, grid, tile, n, &tg)) return PCG_ERR_INVALID_ARG;
    if (n_payload < 1 || n_payload > kMaxPayload) return PCG_ERR_INVALID_ARG;
    *bytes = make_plan(tg, n, n_payload, dim).bytes;
    return PCG_OK;
}

extern "C" pcg_status pcg_tile_sort(int32_t dim, const int32_t *grid, int32_t tile, int64_t n,
                                    const float *const *key_pos, int32_t n_payload,
                                    const void *const *payload_in, void *const *payload_out,
                                    uint32_t *tile_offsets, pcg_stats *stats, void *workspace,
                                    size_t workspace_bytes, void *stream) {
    using namespace pcg;
    TileGrid tg;
    if (!valid_sort_args(dim, grid, tile, n, &tg)) return PCG_ERR_INVALID_ARG;
    if (tile_offsets == nullptr || key_pos == nullptr) return PCG_ERR_INVALID_ARG;
    if (n_payload < 1 || n_payload > kMaxPayload || payload_in == nullptr || payload_out == nullptr)
        return PCG_ERR_INVALID_ARG;
    Payload py{};
    for (int f = 0; f < n_payload; ++f) {
        if (n > 0 && (payload_in[f] == nullptr || payload_out[f] == nullptr))
            return PCG_ERR_INVALID_ARG;
        py.in[f] = static_cast<const unsigned *>(payload_in[f]);
        py.out[f] = static_cast<unsigned *>(payload_out[f]);
    }
    for (int mu = 0; mu < dim; ++mu)
        if (n > 0 && key_pos[mu] == nullptr) return PCG_ERR_INVALID_ARG;
    const Plan pl = make_plan(tg, n, n_payload, dim);
    if (workspace_bytes < pl.bytes || (pl.bytes > 0 && workspace == nullptr))
        return PCG_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return PCG_ERR_WORKSPACE;
    cudaStream_t s = as_stream(stream);
    if (n == 0) return zero_f32(reinterpret_cast<float *>(tile_offsets), (size_t)tg.n_tiles + 1, s);
    unsigned long long *ni = stats ? &stats->n_invalid : nullptr;
    unsigned *fl = stats ? &stats->error_flags : nullptr;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    return dim == 2 ? dispatch_tile<2>(tg, pl, n, key_pos, py, n_payload, tile_offsets, ni, fl, ws, s)
                    : dispatch_tile<3>(tg, pl, n, key_pos, py, n_payload, tile_offsets, ni, fl, ws, s);
}
