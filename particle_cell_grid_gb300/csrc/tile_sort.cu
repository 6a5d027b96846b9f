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
#include "common.cuh"

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
// CTA per SM walks batches of `bs` consecutive particles (<= 2048), two at a
// time in flight:
//  * the next batch's payload and key inputs go global -> shared with
//    asynchronous copies (16 bytes where the arrays are aligned), never through
//    registers, while the current batch is ranked and written;
//  * the digits are counted in shared memory; the counting atomic's return
//    value is the particle's rank inside its digit;
//  * one global atomic per non-empty digit reserves a contiguous output range;
//  * a 16-bit permutation lists the batch in digit order, and consecutive
//    threads write consecutive output slots, so every digit's run leaves the SM
//    as contiguous stores and the open sectors are one per bucket or tile
//    frontier.
constexpr int kPartThreads = 512;
constexpr int kMaxBatch = 2048;
constexpr int kItems = kMaxBatch / kPartThreads;
constexpr unsigned kMaxPassBins = 2048;
constexpr unsigned kMaxBuckets = 256;

__device__ __forceinline__ void cp_async4(unsigned *sdst, const unsigned *gsrc) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                     static_cast<unsigned>(__cvta_generic_to_shared(sdst))),
                 "l"(gsrc)
                 : "memory");
}
__device__ __forceinline__ void cp_async16(unsigned *sdst, const unsigned *gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     static_cast<unsigned>(__cvta_generic_to_shared(sdst))),
                 "l"(gsrc)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most one committed group of this thread is still in flight.
__device__ __forceinline__ void cp_async_wait_one() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Exclusive scan of v[0..nb) in place (nb <= kMaxPassBins) by one CTA of
// kPartThreads threads.
__device__ void block_exclusive_scan(unsigned *v, unsigned nb, unsigned *warp_tot) {
    constexpr int PER = kMaxPassBins / kPartThreads;
    constexpr int NW = kPartThreads / 32;
    const unsigned lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned loc[PER];
    unsigned sum = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const unsigned b = threadIdx.x * PER + i;
        loc[i] = b < nb ? v[b] : 0u;
        sum += loc[i];
    }
    unsigned incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= (unsigned)o) incl += t;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const unsigned w = lane < NW ? warp_tot[lane] : 0u;
        unsigned wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned t = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= (unsigned)o) wi += t;
        }
        if (lane < NW) warp_tot[lane] = wi - w;
    }
    __syncthreads();
    unsigned run = warp_tot[warp] + incl - sum;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const unsigned b = threadIdx.x * PER + i;
        if (b < nb) v[b] = run;
        run += loc[i];
    }
    __syncthreads();
}

// Copy elements [b0, b0 + len) of one 32-bit array (n_arr elements) into
// stage[sh + i], sh = b0 % 4: 16-byte copies where the array is 16-byte aligned
// and the whole vector lies inside the array, 4-byte copies otherwise.  The
// stage row holds len + 4 elements.
__device__ __forceinline__ void stage_field(unsigned *stage, const unsigned *__restrict__ src,
                                            long long b0, unsigned len, long long n_arr) {
    const int sh = (int)(b0 & 3);
    const long long a0 = b0 - sh;
    if ((reinterpret_cast<uintptr_t>(src) & 15) == 0) {
        const unsigned nv = (unsigned)(sh + len + 3) / 4;
        for (unsigned v = threadIdx.x; v < nv; v += kPartThreads) {
            const long long a = a0 + 4ll * v;
            if (a + 4 <= n_arr) {
                cp_async16(stage + 4 * v, src + a);
            } else {
                for (int e = 0; e < 4; ++e)
                    if (a + e < n_arr) cp_async4(stage + 4 * v + e, src + a + e);
            }
        }
    } else {
        for (unsigned i = threadIdx.x; i < len; i += kPartThreads)
            cp_async4(stage + sh + i, src + b0 + i);
    }
}

struct BatchGeo {
    long long b0;
    unsigned len, base, nb;
};

// PASS 1: digit = bucket of the tile key computed from key positions; writes the
//         payload and the key to the intermediate arrays (or, with FINAL, the
//         payload straight to the output when one pass suffices).
// PASS 2: digit = tile inside the batch's bucket; key read from the
//         intermediate arrays; writes the final payload.
// Shared memory: two buffers of nl = np + NK rows of (bs + 4) words (payload,
// then the key inputs) | key row (pass 1 with intermediate output) | hist |
// lstart | gbase ([nbcap] each) | bucket starts and batch offsets ([nb1 + 1]
// each, pass 2) | perm[bs] | sdig[bs] (16-bit).
template <int DIM, int TILE, int PASS, bool FINAL>
__global__ void __launch_bounds__(kPartThreads, 1)
    partition_kernel(KeyGeom g, const float *__restrict__ kx, const float *__restrict__ ky,
                     const float *__restrict__ kz, long long n, Payload pl, int np,
                     const unsigned *__restrict__ in_key, unsigned *__restrict__ out_key,
                     unsigned *__restrict__ gcursor, unsigned tpb, unsigned B,
                     const unsigned *__restrict__ batch_off, const uint32_t *__restrict__ offs,
                     unsigned nb1, unsigned nbcap, unsigned bs, unsigned nbatch) {
    extern __shared__ __align__(16) unsigned sm[];
    __shared__ unsigned warp_tot[kPartThreads / 32];
    __shared__ BatchGeo s_geo[2];
    constexpr bool kKey = PASS == 1 && !FINAL;
    constexpr int NK = PASS == 1 ? DIM : 1;  // staged key inputs: positions, or the key
    const int nl = np + NK;
    const unsigned row = bs + 4;
    const size_t buf_words = (size_t)nl * row;  // buffer b starts at sm + b * buf_words
    unsigned *krow = sm + (size_t)2 * nl * row;
    unsigned *hist = krow + (kKey ? row : 0u);  // counts, then ranks
    unsigned *lstart = hist + nbcap;              // local exclusive starts
    unsigned *gbase = lstart + nbcap;             // reserved global starts
    unsigned *bstart = gbase + nbcap;             // pass 2: bucket b = [bstart[b], bstart[b+1])
    unsigned *boff = bstart + (PASS == 2 ? nb1 + 1 : 0u);  // pass 2: first batch of bucket b
    unsigned short *perm = reinterpret_cast<unsigned short *>(boff + (PASS == 2 ? nb1 + 1 : 0u));
    unsigned short *sdig = perm + bs;
    const unsigned tid = threadIdx.x;

    if (PASS == 2) {
        for (unsigned b = tid; b <= nb1; b += kPartThreads) {
            const unsigned long long t = (unsigned long long)b * tpb;
            bstart[b] = t < B ? offs[t] : (unsigned)n;
            boff[b] = batch_off[b];
        }
        __syncthreads();
    }
    auto geometry = [&](unsigned k, BatchGeo &o) {
        o.len = 0;
        o.b0 = 0;
        o.base = 0;
        o.nb = 1;
        if (k >= nbatch) return;
        if (PASS == 1) {
            o.b0 = (long long)k * bs;
            const long long rem = n - o.b0;
            o.len = rem < (long long)bs ? (unsigned)(rem > 0 ? rem : 0) : bs;
            o.nb = FINAL ? B : nb1;
        } else {
            // bucket of batch k: largest b with boff[b] <= k
            unsigned lo = 0, hi = nb1;
            while (lo < hi) {
                const unsigned mid = (lo + hi + 1) / 2;
                if (boff[mid] <= k) lo = mid;
                else hi = mid - 1;
            }
            if (lo >= nb1) return;
            o.b0 = (long long)bstart[lo] + (long long)(k - boff[lo]) * bs;
            const long long rem = (long long)bstart[lo + 1] - o.b0;
            o.len = rem < (long long)bs ? (unsigned)(rem > 0 ? rem : 0) : bs;
            o.base = lo * tpb;
            o.nb = min(tpb, B - o.base);
        }
    };
    auto issue = [&](const BatchGeo &o, unsigned *dst) {
        if (o.len == 0) return;
        for (int f = 0; f < np; ++f) stage_field(dst + (size_t)f * row, pl.in[f], o.b0, o.len, n);
        if (PASS == 1) {
            stage_field(dst + (size_t)np * row, reinterpret_cast<const unsigned *>(kx), o.b0, o.len, n);
            stage_field(dst + (size_t)(np + 1) * row, reinterpret_cast<const unsigned *>(ky), o.b0, o.len, n);
            if (DIM == 3)
                stage_field(dst + (size_t)(np + 2) * row, reinterpret_cast<const unsigned *>(kz), o.b0,
                            o.len, n);
        } else {
            stage_field(dst + (size_t)np * row, in_key, o.b0, o.len, n);
        }
    };

    if (tid == 0) geometry(blockIdx.x, s_geo[0]);
    __syncthreads();
    issue(s_geo[0], sm);
    cp_async_commit();
    int it = 0;
    for (unsigned k = blockIdx.x; k < nbatch; k += gridDim.x, ++it) {
        const int cb = it & 1;
        if (tid == 0) geometry(k + gridDim.x, s_geo[cb ^ 1]);
        const BatchGeo cur = s_geo[cb];
        for (unsigned d = tid; d < cur.nb; d += kPartThreads) hist[d] = 0;
        __syncthreads();  // next geometry visible, histogram zeroed
        issue(s_geo[cb ^ 1], sm + (cb ^ 1) * buf_words);
        cp_async_commit();
        if (cur.len == 0) break;  // uniform; only trailing batches of pass 2 are empty
        cp_async_wait_one();      // this thread's copies of the current batch
        __syncthreads();          // everyone's copies
        const unsigned *st = sm + cb * buf_words;
        const int sh = (int)(cur.b0 & 3);
        unsigned dig[kItems], rk[kItems];
#pragma unroll
        for (int j = 0; j < kItems; ++j) {
            const unsigned i = tid + j * kPartThreads;
            dig[j] = 0xffffffffu;
            if (i < cur.len) {
                unsigned key;
                if (PASS == 1) {
                    const float x = __uint_as_float(st[(size_t)np * row + sh + i]);
                    const float y = __uint_as_float(st[(size_t)(np + 1) * row + sh + i]);
                    const float z = DIM == 3 ? __uint_as_float(st[(size_t)(np + 2) * row + sh + i]) : 0.f;
                    key = tile_key<DIM, TILE>(g, x, y, z);
                } else {
                    key = st[(size_t)np * row + sh + i];
                }
                if (kKey) krow[i] = key;
                unsigned d = (PASS == 1) ? (FINAL ? key : key / tpb) : key - cur.base;
                if (d >= cur.nb) d = cur.nb - 1;  // defensive: never index outside the histogram
                dig[j] = d;
                rk[j] = atomicAdd(&hist[d], 1u);
            }
        }
        __syncthreads();
        for (unsigned d = tid; d < cur.nb; d += kPartThreads) lstart[d] = hist[d];
        __syncthreads();
        block_exclusive_scan(lstart, cur.nb, warp_tot);
        for (unsigned d = tid; d < cur.nb; d += kPartThreads) {
            const unsigned c = hist[d];
            gbase[d] = c ? atomicAdd(&gcursor[cur.base + d], c) : 0u;
        }
#pragma unroll
        for (int j = 0; j < kItems; ++j) {
            if (dig[j] == 0xffffffffu) continue;
            const unsigned slot = lstart[dig[j]] + rk[j];
            perm[slot] = (unsigned short)(tid + j * kPartThreads);
            sdig[slot] = (unsigned short)dig[j];
        }
        __syncthreads();
        // write every digit's run with consecutive threads; all of a slot's
        // shared-memory loads are issued before its stores
        for (unsigned slot = tid; slot < cur.len; slot += kPartThreads) {
            const unsigned i = perm[slot], d = sdig[slot];
            const unsigned gpos = gbase[d] + (slot - lstart[d]);
            if (!PCG_IN(gpos, n) || !PCG_IN(i, cur.len)) continue;
            const unsigned *src = st + sh + i;
            if (PASS == 2) {
                // measured faster for pass 2: one load-store pair per field
                for (int f = 0; f < np; ++f) pl.out[f][gpos] = src[(size_t)f * row];
            } else {
                // measured faster for pass 1: all loads of the slot before its stores
                unsigned v[kMaxPayload];
#pragma unroll
                for (int f = 0; f < kMaxPayload; ++f)
                    if (f < np) v[f] = src[(size_t)f * row];
                const unsigned kv = kKey ? krow[i] : 0u;
#pragma unroll
                for (int f = 0; f < kMaxPayload; ++f)
                    if (f < np) pl.out[f][gpos] = v[f];
                if (kKey) out_key[gpos] = kv;
            }
        }
        __syncthreads();  // buffer, key row, histogram and permutation are reused
    }
    cp_async_wait_all();
}

size_t partition_smem(int DIM, int pass, bool final_, int np, unsigned nbcap, unsigned nb1, unsigned bs) {
    const int nk = pass == 1 ? DIM : 1;
    const size_t row = (size_t)(bs + 4) * 4;
    size_t b = 2 * (size_t)(np + nk) * row;
    if (pass == 1 && !final_) b += row;
    b += (size_t)3 * nbcap * 4;
    if (pass == 2) b += (size_t)2 * (nb1 + 1) * 4;
    b += (size_t)bs * 4;  // perm + sdig
    return b;
}

// Largest batch (<= kMaxBatch, a multiple of kPartThreads) whose buffers fit.
unsigned partition_batch(int DIM, int pass, bool final_, int np, unsigned nbcap, unsigned nb1) {
    constexpr size_t kSmemCap = 227 * 1024 - 1024;
    for (unsigned bs = kMaxBatch; bs > (unsigned)kPartThreads; bs /= 2)
        if (partition_smem(DIM, pass, final_, np, nbcap, nb1, bs) <= kSmemCap) return bs;
    return kPartThreads;
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

Plan make_plan(const TileGrid &tg, long long n, int n_payload) {
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
            p.tpb = (p.B + kMaxBuckets - 1) / kMaxBuckets;
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
    // two-pass partition with global cursors: one persistent CTA per SM
    if (pl.nb1 == 1) {
        const unsigned bs = partition_batch(DIM, 1, true, np, pl.B, 1);
        const size_t smem = partition_smem(DIM, 1, true, np, pl.B, 1, bs);
        const unsigned nbatch = (unsigned)((n + bs - 1) / bs);
        PCG_CHECK_CUDA(cudaFuncSetAttribute(partition_kernel<DIM, TILE, 1, true>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        prof::Mark mk("sort_partition", s);
        partition_kernel<DIM, TILE, 1, true><<<nbatch < sms ? nbatch : sms, kPartThreads, smem, s>>>(
            g, kp[0], kp[1], kz, n, py, np, nullptr, nullptr, cursor, 1, pl.B, nullptr, offs, 1, pl.B, bs,
            nbatch);
        return launch_status();
    }
    unsigned *cursor1 = reinterpret_cast<unsigned *>(ws + pl.o_cursor1);
    unsigned *batch = reinterpret_cast<unsigned *>(ws + pl.o_batch);
    unsigned *ikey = reinterpret_cast<unsigned *>(ws + pl.o_key);
    Payload p1{}, p2{};
    for (int f = 0; f < np; ++f) {
        unsigned *inter = reinterpret_cast<unsigned *>(ws + pl.o_inter + (size_t)f * pl.inter_stride);
        p1.in[f] = py.in[f];
        p1.out[f] = inter;
        p2.in[f] = inter;
        p2.out[f] = py.out[f];
    }
    const unsigned bs1 = partition_batch(DIM, 1, false, np, pl.nb1, pl.nb1);
    const unsigned bs2 = partition_batch(DIM, 2, false, np, pl.tpb, pl.nb1);
    const size_t smem1 = partition_smem(DIM, 1, false, np, pl.nb1, pl.nb1, bs1);
    const size_t smem2 = partition_smem(DIM, 2, false, np, pl.tpb, pl.nb1, bs2);
    {
        prof::Mark mk("sort_bucket_setup", s);
        bucket_setup_kernel<<<1, 1024, 0, s>>>(offs, n, pl.B, pl.tpb, pl.nb1, bs2, cursor1, batch);
    }
    PCG_CHECK_LAUNCH();
    PCG_CHECK_CUDA(cudaFuncSetAttribute(partition_kernel<DIM, TILE, 1, false>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1));
    PCG_CHECK_CUDA(cudaFuncSetAttribute(partition_kernel<DIM, TILE, 2, false>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2));
    const unsigned nbatch1 = (unsigned)((n + bs1 - 1) / bs1);
    {
        prof::Mark mk("sort_partition1", s);
        partition_kernel<DIM, TILE, 1, false><<<nbatch1 < sms ? nbatch1 : sms, kPartThreads, smem1, s>>>(
            g, kp[0], kp[1], kz, n, p1, np, nullptr, ikey, cursor1, pl.tpb, pl.B, batch, offs, pl.nb1,
            pl.nb1, bs1, nbatch1);
    }
    PCG_CHECK_LAUNCH();
    // upper bound on the bucket-aligned batches; the ones past the real count are empty
    const unsigned nbatch2 = (unsigned)((n + bs2 - 1) / bs2) + pl.nb1;
    prof::Mark mk("sort_partition2", s);
    partition_kernel<DIM, TILE, 2, false><<<nbatch2 < sms ? nbatch2 : sms, kPartThreads, smem2, s>>>(
        g, kp[0], kp[1], kz, n, p2, np, ikey, nullptr, cursor, pl.tpb, pl.B, batch, offs, pl.nb1, pl.tpb,
        bs2, nbatch2);
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
    *bytes = make_plan(tg, n, n_payload).bytes;
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
    const Plan pl = make_plan(tg, n, n_payload);
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
