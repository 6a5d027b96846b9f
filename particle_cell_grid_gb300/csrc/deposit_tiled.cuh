// deposit_tiled.cuh -- the tiled deposit kernel template (instantiated per
// dimension in deposit_2d.cu and deposit_3d.cu to keep compile units small).
//
// Per CTA: a fixed-size chunk of the tile-sorted particle array; for every tile
// segment inside it, a haloed scratch tile of 3 x (T + 2*HALO)^D floats in
// shared memory ("Tiled current deposit", Entity wiki, "How a tile deposit
// runs"), flushed once to J with global reductions.
//
// Inside a segment the particles are taken in sub-batches of 8 per thread.  A
// shared-memory counting sort groups each sub-batch by the first node of its
// stencil (the cell for CIC, the nearest node minus one for the quadratic
// spline): particles with the same first node share the whole stencil (the
// "support group" of Pennati & Markidis, Sec. 3.3), so one thread per group sums
// q v W of its particles in registers and adds each stencil node to the
// scratch tile once per group.  On this GPU a warp-wide fp32 shared-memory
// reduction to random addresses costs ~13 cycles, ~4 when the 32 addresses are
// distinct and in distinct banks; the grouped flush by consecutive threads is of
// the second kind and replaces 8 (CIC) or 27 (quadratic) random reductions per
// particle by that many per group.
//
// Particles whose stencil fits the scratch window but whose first node lies
// outside the tile's own range (they drifted into the halo) add their stencil
// directly with per-particle shared reductions; particles whose stencil leaves
// the window take the escape valve to global J ("Correctness is independent of
// the halo").
#pragma once

#include "deposit.cuh"

namespace pcg {
namespace dep {

template <int DIM, int ORDER, int TILE, int HALO>
struct TileCfg {
    static constexpr int S = ORDER + 1;                 // stencil nodes per axis
    static constexpr int TE = TILE + 2 * HALO;          // scratch edge
    static constexpr int TEZ = DIM == 3 ? TE : 1;
    static constexpr int CELLS = TE * TE * TEZ;         // scratch nodes
    static constexpr int FLOATS = 3 * CELLS;
    static constexpr int SZ = DIM == 3 ? S : 1;
    // grouped ("home") first nodes per axis: those of particles inside the tile
    // ([0, TILE) for CIC, [-1, TILE) for the quadratic spline) whose stencil
    // also fits the window [-HALO, TILE + HALO)
    static constexpr int KLO = -(ORDER - 1) > -HALO ? -(ORDER - 1) : -HALO;
    static constexpr int KHI_A = TILE;
    static constexpr int KHI_B = TILE + HALO - S + 1;
    static constexpr int KHI = KHI_A < KHI_B ? KHI_A : KHI_B;
    static constexpr int KR = KHI - KLO;
    static constexpr int KRZ = DIM == 3 ? KR : 1;
    static constexpr int NKEYS = KR * KR * KRZ;
};

template <int THREADS>
struct BatchCfg {
    static constexpr int PPT = 8;              // particles per thread per sub-batch
    static constexpr int GROUPS = PPT / 4;     // groups of four consecutive slots
    static constexpr int SB = PPT * THREADS;   // sub-batch size
};

// Weights of one axis from the stored offset: CIC offset = x - cell, quadratic
// offset = x - nearest node.
template <int ORDER>
__device__ __forceinline__ void weights_from(float t, float (&w)[ORDER + 1]) {
    if (ORDER == 1) {
        w[0] = 1.f - t;
        w[1] = t;
    } else {
        const float a = 0.5f - t, b = 0.5f + t;
        w[0] = 0.5f * a * a;
        w[1] = 0.75f - t * t;
        w[2] = 0.5f * b * b;
    }
}

// First node and stored offset of one axis (x >= 0).
template <int ORDER>
__device__ __forceinline__ int first_node(float x, float &t) {
    const int i = (int)x;
    const float xi = x - (float)i;
    if (ORDER == 1) {
        t = xi;
        return i;
    }
    const int k = i + (xi >= 0.5f ? 1 : 0);
    t = x - (float)k;  // exact: x and k are within a factor two
    return k - 1;
}

// Exclusive scan of v[0..NB) in place by all THREADS threads of the CTA.
template <int THREADS, int NB>
__device__ __forceinline__ void cta_exclusive_scan(unsigned *v, unsigned *warp_tot) {
    constexpr int PER = (NB + THREADS - 1) / THREADS;
    constexpr int NW = THREADS / 32;
    const unsigned lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned loc[PER];
    unsigned sum = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int b = threadIdx.x * PER + i;
        loc[i] = b < NB ? v[b] : 0u;
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
        const int b = threadIdx.x * PER + i;
        if (b < NB) v[b] = run;
        run += loc[i];
    }
}

// Stencil of one particle with precomputed offsets into the scratch window.
template <int DIM, int ORDER, int TILE, int HALO>
__device__ __forceinline__ void scratch_particle(float *scratch, int lx, int ly, int lz, float tx,
                                                 float ty, float tz, float qvx, float qvy, float qvz) {
    using C = TileCfg<DIM, ORDER, TILE, HALO>;
    constexpr int S = C::S;
    float wx[S], wy[S], wz[S];
    weights_from<ORDER>(tx, wx);
    weights_from<ORDER>(ty, wy);
    if (DIM == 3) weights_from<ORDER>(tz, wz);
    else wz[0] = 1.f;
    const int base = ((DIM == 3 ? (lz + HALO) * C::TE : 0) + (ly + HALO)) * C::TE + (lx + HALO);
    if (!PCG_IN(base, C::CELLS) || !PCG_IN(base + ((C::SZ - 1) * C::TE + S - 1) * C::TE + S - 1, C::CELLS)) return;
#pragma unroll
    for (int kz = 0; kz < C::SZ; ++kz)
#pragma unroll
        for (int ky = 0; ky < S; ++ky) {
            const float wyz = wy[ky] * wz[kz];
            float *row = scratch + base + (kz * C::TE + ky) * C::TE;
#pragma unroll
            for (int kx = 0; kx < S; ++kx) {
                const float W = wyz * wx[kx];
                red_shared_add_f32(row + kx, qvx * W);
                red_shared_add_f32(row + C::CELLS + kx, qvy * W);
                red_shared_add_f32(row + 2 * C::CELLS + kx, qvz * W);
            }
        }
}

// Flush the scratch tile: every row once, as contiguous runs of J (split where
// the periodic wrap breaks them) with 8/16-byte vector reductions; all-zero
// pieces are skipped.
template <int DIM, int TILE, int HALO, int THREADS>
__device__ __forceinline__ void flush_scratch(const Geom &g, const float *scratch, float *J, int ox,
                                              int oy, int oz) {
    using C = TileCfg<DIM, 1, TILE, HALO>;
    for (int row = threadIdx.x; row < 3 * C::TE * C::TEZ; row += THREADS) {
        const int c = row / (C::TE * C::TEZ);
        const int rr = row - c * (C::TE * C::TEZ);
        const int sy = rr % C::TE;
        const int sz = rr / C::TE;
        int gy = oy - HALO + sy;
        gy = gy < 0 ? gy + g.N[1] : (gy >= g.N[1] ? gy - g.N[1] : gy);
        int gz = 0;
        if (DIM == 3) {
            gz = oz - HALO + sz;
            gz = gz < 0 ? gz + g.N[2] : (gz >= g.N[2] ? gz - g.N[2] : gz);
        }
        if (gy < 0 || gy >= g.N[1] || gz < 0 || gz >= g.N[2]) {
            // a grid shorter than the window: wrap each cell on its own
            for (int sx = 0; sx < C::TE; ++sx) {
                const float v = scratch[row * C::TE + sx];
                const long long node = ((long long)wrap_index(oz - HALO + sz, g.N[2]) * g.N[1] +
                                        wrap_index(oy - HALO + sy, g.N[1])) * g.N[0] +
                                       wrap_index(ox - HALO + sx, g.N[0]);
                if (v != 0.f && PCG_IN(node, g.ncells)) red_add_f32(J + c * g.ncells + node, v);
            }
            continue;
        }
        float *jrow = J + c * g.ncells + ((long long)gz * g.N[1] + gy) * g.N[0];
        const float *src = scratch + row * C::TE;
        int sx = 0;
        while (sx < C::TE) {
            int gx = ox - HALO + sx;
            gx = gx < 0 ? gx + g.N[0] : (gx >= g.N[0] ? gx - g.N[0] : gx);
            if (gx < 0 || gx >= g.N[0]) {  // grid shorter than the window along x
                const float v = src[sx];
                if (v != 0.f) red_add_f32(jrow + wrap_index(ox - HALO + sx, g.N[0]), v);
                ++sx;
                continue;
            }
            int run = g.N[0] - gx;            // contiguous in J up to the wrap
            if (run > C::TE - sx) run = C::TE - sx;
            if (!PCG_IN(((long long)gz * g.N[1] + gy) * g.N[0] + gx + run - 1, g.ncells)) break;
            float *dst = jrow + gx;
            const float *sv = src + sx;
            int k = 0;
            while (k < run) {
                const uintptr_t a = reinterpret_cast<uintptr_t>(dst + k);
                if ((a & 15) == 0 && k + 4 <= run) {
                    const float v0 = sv[k], v1 = sv[k + 1], v2 = sv[k + 2], v3 = sv[k + 3];
                    if (v0 != 0.f || v1 != 0.f || v2 != 0.f || v3 != 0.f)
                        red_add_v4_f32(dst + k, v0, v1, v2, v3);
                    k += 4;
                } else if ((a & 7) == 0 && k + 2 <= run) {
                    const float v0 = sv[k], v1 = sv[k + 1];
                    if (v0 != 0.f || v1 != 0.f) red_add_v2_f32(dst + k, v0, v1);
                    k += 2;
                } else {
                    if (sv[k] != 0.f) red_add_f32(dst + k, sv[k]);
                    k += 1;
                }
            }
            sx += run;
        }
    }
}

template <int DIM, int ORDER, int TILE, int HALO, int THREADS>
__global__ void __launch_bounds__(THREADS, 512 / THREADS)
    deposit_tiled_kernel(Geom g, Particles P, long long n, const uint32_t *__restrict__ offs,
                         const unsigned *__restrict__ chunk_tile, long long chunk,
                         float *__restrict__ J, Counters ctr, bool vec4) {
    using C = TileCfg<DIM, ORDER, TILE, HALO>;
    using BC = BatchCfg<THREADS>;
    constexpr int S = C::S;
    constexpr int NK = C::NKEYS;
    extern __shared__ __align__(16) unsigned char dsm[];
    float *scratch = reinterpret_cast<float *>(dsm);                   // [3][CELLS]
    unsigned *cnt = reinterpret_cast<unsigned *>(scratch + C::FLOATS);  // [NK]
    unsigned *start = cnt + NK;                                         // [NK]
    unsigned *cur = start + NK;                                         // [NK]
    float *stage = reinterpret_cast<float *>(cur + NK);                 // [7][SB]
    __shared__ unsigned warp_tot[THREADS / 32];
    __shared__ unsigned n_halo;

    const long long c0 = (long long)blockIdx.x * chunk;
    const long long c1 = min(n, c0 + chunk);
    unsigned n_esc = 0, n_inv = 0;
    unsigned t = chunk_tile[blockIdx.x];
    if (t > g.n_tiles) t = g.n_tiles;
    for (;; ++t) {
        long long s = (long long)offs[t];
        if (s < c0) s = c0;
        if (s >= c1) break;
        long long e = (t < g.n_tiles) ? (long long)offs[t + 1] : c1;
        if (e > c1) e = c1;
        if (t == g.n_tiles) {
            // tail pass: slots after the last tile go straight to J
            for (long long p = s + threadIdx.x; p < e; p += THREADS) {
                const float x = P.x[p], y = P.y[p], z = DIM == 3 ? P.z[p] : 0.f;
                if (!in_domain<DIM>(g, x, y, z)) {
                    ++n_inv;
                    continue;
                }
                const float q = P.q[p];
                deposit_global<DIM, ORDER>(g, J, x, y, z, q * P.vx[p], q * P.vy[p], q * P.vz[p]);
            }
            break;
        }
        if (e <= s) continue;  // empty tile
        const int tx = (int)(t % (unsigned)g.nt[0]);
        const int ty = (int)((t / (unsigned)g.nt[0]) % (unsigned)g.nt[1]);
        const int tz = DIM == 3 ? (int)(t / ((unsigned)g.nt[0] * (unsigned)g.nt[1])) : 0;
        const int ox = tx * TILE, oy = ty * TILE, oz = tz * TILE;

        for (int i = threadIdx.x; i < C::FLOATS; i += THREADS) scratch[i] = 0.f;

        const long long g0 = s >> 2, g1 = (e + 3) >> 2;  // groups of four slots
        for (long long gb = g0; gb < g1; gb += (long long)BC::GROUPS * THREADS) {
            for (int i = threadIdx.x; i < NK; i += THREADS) cnt[i] = 0;
            if (threadIdx.x == 0) n_halo = 0;
            __syncthreads();

            // ---- A: load, classify, count the grouped particles ----
            unsigned key[BC::PPT];
            float off[BC::PPT][3], qv[BC::PPT][3];
#pragma unroll
            for (int gr = 0; gr < BC::GROUPS; ++gr) {
                const long long gi = gb + threadIdx.x + gr * THREADS;
                const long long p = gi << 2;
                float xs[4], ys[4], zs[4], vxs[4], vys[4], vzs[4], qs[4];
                if (gi < g1 && vec4 && p + 3 < n) {
                    const float4 a = *reinterpret_cast<const float4 *>(P.x + p);
                    const float4 b = *reinterpret_cast<const float4 *>(P.y + p);
                    const float4 c = DIM == 3 ? *reinterpret_cast<const float4 *>(P.z + p)
                                              : make_float4(0.f, 0.f, 0.f, 0.f);
                    const float4 d = *reinterpret_cast<const float4 *>(P.vx + p);
                    const float4 f = *reinterpret_cast<const float4 *>(P.vy + p);
                    const float4 h = *reinterpret_cast<const float4 *>(P.vz + p);
                    const float4 k = *reinterpret_cast<const float4 *>(P.q + p);
                    xs[0] = a.x; xs[1] = a.y; xs[2] = a.z; xs[3] = a.w;
                    ys[0] = b.x; ys[1] = b.y; ys[2] = b.z; ys[3] = b.w;
                    zs[0] = c.x; zs[1] = c.y; zs[2] = c.z; zs[3] = c.w;
                    vxs[0] = d.x; vxs[1] = d.y; vxs[2] = d.z; vxs[3] = d.w;
                    vys[0] = f.x; vys[1] = f.y; vys[2] = f.z; vys[3] = f.w;
                    vzs[0] = h.x; vzs[1] = h.y; vzs[2] = h.z; vzs[3] = h.w;
                    qs[0] = k.x; qs[1] = k.y; qs[2] = k.z; qs[3] = k.w;
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const long long pj = (gi < g1 && p + j >= s && p + j < e) ? p + j : s;
                        xs[j] = P.x[pj]; ys[j] = P.y[pj]; zs[j] = DIM == 3 ? P.z[pj] : 0.f;
                        vxs[j] = P.vx[pj]; vys[j] = P.vy[pj]; vzs[j] = P.vz[pj]; qs[j] = P.q[pj];
                    }
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int slot = gr * 4 + j;
                    key[slot] = 0xffffffffu;
                    const long long pj = p + j;
                    if (gi >= g1 || pj < s || pj >= e) continue;
                    const float x = xs[j], y = ys[j], z = zs[j];
                    if (!in_domain<DIM>(g, x, y, z)) {
                        ++n_inv;
                        continue;
                    }
                    const float q = qs[j];
                    const float qvx = q * vxs[j], qvy = q * vys[j], qvz = q * vzs[j];
                    float tx_, ty_, tz_ = 0.f;
                    const int fx = first_node<ORDER>(x, tx_);
                    const int fy = first_node<ORDER>(y, ty_);
                    const int fz = DIM == 3 ? first_node<ORDER>(z, tz_) : 0;
                    const int lx = local_index<S, TILE, HALO>(fx, ox, g.N[0]);
                    const int ly = local_index<S, TILE, HALO>(fy, oy, g.N[1]);
                    const int lz = DIM == 3 ? local_index<S, TILE, HALO>(fz, oz, g.N[2]) : 0;
                    bool home = (lx >= C::KLO) & (lx < C::KHI) & (ly >= C::KLO) & (ly < C::KHI);
                    if (DIM == 3) home &= (lz >= C::KLO) & (lz < C::KHI);
                    if (home) {
                        const unsigned k = (unsigned)(((DIM == 3 ? (lz - C::KLO) * C::KR : 0) +
                                                       (ly - C::KLO)) * C::KR + (lx - C::KLO));
                        key[slot] = k;
                        off[slot][0] = tx_;
                        off[slot][1] = ty_;
                        off[slot][2] = tz_;
                        qv[slot][0] = qvx;
                        qv[slot][1] = qvy;
                        qv[slot][2] = qvz;
                        if (PCG_IN(k, NK)) atomicAdd(&cnt[k], 1u);
                        else key[slot] = 0xffffffffu;
                        continue;
                    }
                    bool fits = (lx >= -HALO) & (lx + S - 1 < TILE + HALO) & (ly >= -HALO) &
                                (ly + S - 1 < TILE + HALO);
                    if (DIM == 3) fits &= (lz >= -HALO) & (lz + S - 1 < TILE + HALO);
                    if (!fits) {
                        ++n_esc;
                        deposit_global<DIM, ORDER>(g, J, x, y, z, qvx, qvy, qvz);
                        continue;
                    }
                    // drifted into the halo: listed at the top of the staging
                    // buffer and deposited after the groups by densely packed threads
                    const unsigned hs = BC::SB - 1 - atomicAdd(&n_halo, 1u);
                    if (!PCG_IN(hs, BC::SB)) continue;
                    stage[0 * BC::SB + hs] = tx_;
                    stage[1 * BC::SB + hs] = ty_;
                    stage[2 * BC::SB + hs] = tz_;
                    stage[3 * BC::SB + hs] = qvx;
                    stage[4 * BC::SB + hs] = qvy;
                    stage[5 * BC::SB + hs] = qvz;
                    stage[6 * BC::SB + hs] = __int_as_float(((lx + HALO) & 255) | (((ly + HALO) & 255) << 8) |
                                                            (((lz + HALO) & 255) << 16));
                }
            }
            __syncthreads();

            // ---- B: group starts ----
            for (int i = threadIdx.x; i < NK; i += THREADS) start[i] = cnt[i];
            __syncthreads();
            cta_exclusive_scan<THREADS, NK>(start, warp_tot);
            __syncthreads();
            for (int i = threadIdx.x; i < NK; i += THREADS) cur[i] = start[i];
            __syncthreads();

            // ---- C: place each grouped particle in its group's slots ----
#pragma unroll
            for (int i = 0; i < BC::PPT; ++i) {
                if (key[i] == 0xffffffffu) continue;
                const unsigned slot = atomicAdd(&cur[key[i]], 1u);
                if (!PCG_IN(slot, BC::SB)) continue;
                stage[0 * BC::SB + slot] = off[i][0];
                stage[1 * BC::SB + slot] = off[i][1];
                stage[2 * BC::SB + slot] = off[i][2];
                stage[3 * BC::SB + slot] = qv[i][0];
                stage[4 * BC::SB + slot] = qv[i][1];
                stage[5 * BC::SB + slot] = qv[i][2];
            }
            __syncthreads();

            // pull the next sub-batch of this segment into L2 while this one is reduced
            if (threadIdx.x == 0 && vec4) {
                const long long nb0 = (gb + (long long)BC::GROUPS * THREADS) << 2;
                long long nb1 = nb0 + BC::SB;
                if (nb1 > (e & ~3ll)) nb1 = e & ~3ll;
                if (nb1 > nb0) {
                    const unsigned bytes = (unsigned)((nb1 - nb0) * 4);
                    prefetch_l2_bulk(P.x + nb0, bytes);
                    prefetch_l2_bulk(P.y + nb0, bytes);
                    if (DIM == 3) prefetch_l2_bulk(P.z + nb0, bytes);
                    prefetch_l2_bulk(P.vx + nb0, bytes);
                    prefetch_l2_bulk(P.vy + nb0, bytes);
                    prefetch_l2_bulk(P.vz + nb0, bytes);
                    prefetch_l2_bulk(P.q + nb0, bytes);
                }
            }

            // ---- D: one thread per group sums its particles, then adds each node once ----
            for (int k = threadIdx.x; k < NK; k += THREADS) {
                const unsigned m = cnt[k];
                if (m == 0) continue;
                const unsigned b0 = start[k];
                if (!PCG_IN(b0 + m - 1, BC::SB)) continue;
                float acc[C::SZ][S][S][3];
#pragma unroll
                for (int kz = 0; kz < C::SZ; ++kz)
#pragma unroll
                    for (int ky = 0; ky < S; ++ky)
#pragma unroll
                        for (int kx = 0; kx < S; ++kx)
                            acc[kz][ky][kx][0] = acc[kz][ky][kx][1] = acc[kz][ky][kx][2] = 0.f;
                for (unsigned u = b0; u < b0 + m; ++u) {
                    float wx[S], wy[S], wz[S];
                    weights_from<ORDER>(stage[u], wx);
                    weights_from<ORDER>(stage[BC::SB + u], wy);
                    if (DIM == 3) weights_from<ORDER>(stage[2 * BC::SB + u], wz);
                    else wz[0] = 1.f;
                    const float a = stage[3 * BC::SB + u], b = stage[4 * BC::SB + u],
                                c = stage[5 * BC::SB + u];
#pragma unroll
                    for (int kz = 0; kz < C::SZ; ++kz)
#pragma unroll
                        for (int ky = 0; ky < S; ++ky) {
                            const float wyz = wy[ky] * wz[kz];
#pragma unroll
                            for (int kx = 0; kx < S; ++kx) {
                                const float W = wyz * wx[kx];
                                acc[kz][ky][kx][0] = fmaf(a, W, acc[kz][ky][kx][0]);
                                acc[kz][ky][kx][1] = fmaf(b, W, acc[kz][ky][kx][1]);
                                acc[kz][ky][kx][2] = fmaf(c, W, acc[kz][ky][kx][2]);
                            }
                        }
                }
                const int kx0 = k % C::KR + C::KLO;
                const int ky0 = (k / C::KR) % C::KR + C::KLO;
                const int kz0 = DIM == 3 ? k / (C::KR * C::KR) + C::KLO : 0;
                const int base =
                    ((DIM == 3 ? (kz0 + HALO) * C::TE : 0) + (ky0 + HALO)) * C::TE + (kx0 + HALO);
#pragma unroll
                for (int kz = 0; kz < C::SZ; ++kz)
#pragma unroll
                    for (int ky = 0; ky < S; ++ky) {
                        float *row = scratch + base + (kz * C::TE + ky) * C::TE;
#pragma unroll
                        for (int kx = 0; kx < S; ++kx) {
                            red_shared_add_f32(row + kx, acc[kz][ky][kx][0]);
                            red_shared_add_f32(row + C::CELLS + kx, acc[kz][ky][kx][1]);
                            red_shared_add_f32(row + 2 * C::CELLS + kx, acc[kz][ky][kx][2]);
                        }
                    }
            }
            // ---- the halo particles listed in phase A ----
            for (unsigned h = threadIdx.x; h < n_halo; h += THREADS) {
                const unsigned hs = BC::SB - 1 - h;
                const int pk = __float_as_int(stage[6 * BC::SB + hs]);
                scratch_particle<DIM, ORDER, TILE, HALO>(
                    scratch, (pk & 255) - HALO, ((pk >> 8) & 255) - HALO, ((pk >> 16) & 255) - HALO,
                    stage[hs], stage[BC::SB + hs], stage[2 * BC::SB + hs], stage[3 * BC::SB + hs],
                    stage[4 * BC::SB + hs], stage[5 * BC::SB + hs]);
            }
            __syncthreads();  // stage and counters are reused by the next sub-batch
        }

        flush_scratch<DIM, TILE, HALO, THREADS>(g, scratch, J, ox, oy, oz);
        __syncthreads();  // scratch is reused by the next segment
    }
    warp_add_u64(ctr.n_escaped, n_esc);
    warp_add_u64(ctr.n_invalid, n_inv);
}

// ---------------------------------------------------------------------------
// 3D CIC with 8^3 tiles, persistent: one CTA of 512 threads per SM walks the
// chunks b, b + grid, ... of the tile-sorted array in rounds of 4096
// particles (8 per thread, loaded as float4 per field).  One thread per cell of
// the tile keeps the cell's 8 corners x 3 components in registers for the
// whole tile segment.  A round is distributed to the cells through a
// transposed staging array of float2 pairs, st[pair][rank][cell]: the placing
// atomic returns the rank, and a warp's 32 cells read rank r from 32
// consecutive 8-byte words (conflict-free).  With 8 particles per cell per
// round on average, a warp's longest cell list is ~1.5x the mean (a round of
// 1024 would leave two thirds of the lanes idle).  A cell holds up to CAP
// particles per round.  Particles the fast path does not take (drifted into the
// halo, beyond CAP in their cell, escaping, invalid) are queued per warp in
// shared memory (ballot-compacted) and taken by the warp one per lane after its
// 8 particles: their general path and global reductions then run once per warp
// instead of inside the unrolled loop whenever any lane of the warp needs it.
// The next round's particles are loaded into registers before this round is
// accumulated, so their latency hides behind the accumulation.
// ---------------------------------------------------------------------------
template <int HALO>
struct Cic5Cfg {
    static constexpr int THREADS = 512;
    static constexpr int PPT = 8;               // particles per thread per round
    static constexpr int R = THREADS * PPT;     // round size
    static constexpr int CAP = 12;              // staged particles per cell and round
    static constexpr int QCAP = PPT * 32;       // queued particles per warp and round: room for all
    using C = TileCfg<3, 1, 8, HALO>;
    static constexpr int NK = C::NKEYS;         // cells of the tile (one thread each)
    static_assert(NK <= THREADS, "one thread per grouped cell");
    static_assert(24 <= 6 * CAP, "the corner values fit in the staging array");
    static constexpr size_t SMEM = (size_t)3 * CAP * NK * 8 + (size_t)(THREADS / 32) * QCAP * 4 + (size_t)NK * 4;
};

// Position of a CTA in its work: chunk, tile segment (tile t, valid particles
// [lo, hi)) and round base rb (a multiple of 4).
struct RoundPos {
    long long c;      // chunk
    long long rb;     // round base
    long long lo, hi; // tile segment inside the chunk
    unsigned t;       // tile (n_tiles: the invalid tail; > n_tiles: no more work)
};

__device__ __forceinline__ bool seg_of_tile(const Geom &g, const uint32_t *__restrict__ offs, long long n,
                                            long long c0, long long c1, unsigned t, RoundPos &r) {
    long long s = (long long)offs[t];
    if (s < c0) s = c0;
    long long e = (t < g.n_tiles) ? (long long)offs[t + 1] : c1;
    if (e > c1) e = c1;
    r.t = t;
    r.lo = s;
    r.hi = e;
    r.rb = s & ~3ll;
    return s < c1;  // false: the tile starts after the chunk
}

// First non-empty tile segment at or after tile t of chunk c, or the next chunk's.
__device__ __forceinline__ void seek(const Geom &g, const uint32_t *__restrict__ offs,
                                     const unsigned *__restrict__ chunk_tile, long long n, long long chunk,
                                     long long nchunks, long long c, unsigned t, RoundPos &r) {
    for (; c < nchunks; c += gridDim.x, t = 0xffffffffu) {
        const long long c0 = c * chunk, c1 = min(n, c0 + chunk);
        if (t == 0xffffffffu) t = min(chunk_tile[c], g.n_tiles);
        r.c = c;
        for (; t <= g.n_tiles; ++t) {
            if (!seg_of_tile(g, offs, n, c0, c1, t, r)) break;
            if (r.hi > r.lo) return;
            if (t == g.n_tiles) break;
        }
    }
    r.c = nchunks;
    r.t = g.n_tiles + 1;
}

// Stencil of one CIC particle at local first node (lx, ly, lz) of the tile at
// (ox, oy, oz) straight into J with global reductions (periodic wrap): the path
// of halo and overflow particles.  On this GPU a shared-memory float reduction
// is a long serial read-modify-write (~87 cycles per dependent op against ~6 for
// an integer shared atomic), while a global reduction is fire-and-forget.
template <int HALO>
__device__ __forceinline__ void stencil_to_global(const Geom &g, float *__restrict__ J, int ox, int oy, int oz,
                                                  int lx, int ly, int lz, float tx, float ty, float tz, float qvx,
                                                  float qvy, float qvz) {
    const float wx[2] = {1.f - tx, tx}, wy[2] = {1.f - ty, ty}, wz[2] = {1.f - tz, tz};
    int gx[2], gy[2], gz[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        gx[k] = ox + lx + k;
        gy[k] = oy + ly + k;
        gz[k] = oz + lz + k;
        while (gx[k] < 0) gx[k] += g.N[0];
        while (gx[k] >= g.N[0]) gx[k] -= g.N[0];
        while (gy[k] < 0) gy[k] += g.N[1];
        while (gy[k] >= g.N[1]) gy[k] -= g.N[1];
        while (gz[k] < 0) gz[k] += g.N[2];
        while (gz[k] >= g.N[2]) gz[k] -= g.N[2];
    }
#pragma unroll
    for (int kz = 0; kz < 2; ++kz)
#pragma unroll
        for (int ky = 0; ky < 2; ++ky) {
            const float wyz = wy[ky] * wz[kz];
            const long long row = ((long long)gz[kz] * g.N[1] + gy[ky]) * g.N[0];
#pragma unroll
            for (int kx = 0; kx < 2; ++kx) {
                const float W = wyz * wx[kx];
                if (!PCG_IN(row + gx[kx], g.ncells)) continue;
                float *j = J + row + gx[kx];
                red_add_f32(j, qvx * W);
                red_add_f32(j + g.ncells, qvy * W);
                red_add_f32(j + 2 * g.ncells, qvz * W);
            }
        }
}

// The escape of a particle whose stencil leaves the window, kept out of line.
static __device__ __noinline__ void escape_to_global(const Geom g, float *J, float x, float y, float z, float qvx,
                                              float qvy, float qvz) {
    deposit_global<3, 1>(g, J, x, y, z, qvx, qvy, qvz);
}
// The general path of one particle of tile (ox, oy, oz) that the fast path did
// not take: 1 invalid (skipped), 2 escaped to J, 0 placed in its own cell (rank
// below CAP) or deposited straight to J (halo, or beyond CAP).  It runs for a
// few percent of the particles, from a warp's queue, outside the unrolled loop.
template <int HALO>
__device__ __forceinline__ int slow_particle(const Geom &g, float *J, float2 *st, unsigned *cnt, int ox, int oy,
                                          int oz, float x, float y, float z, float qvx, float qvy, float qvz) {
    using C = typename Cic5Cfg<HALO>::C;
    constexpr int NK = Cic5Cfg<HALO>::NK, CAP = Cic5Cfg<HALO>::CAP;
    if (!in_domain<3>(g, x, y, z)) return 1;
    float fx_, fy_, fz_;
    const int fx = first_node<1>(x, fx_);
    const int fy = first_node<1>(y, fy_);
    const int fz = first_node<1>(z, fz_);
    const int lx = local_index<2, 8, HALO>(fx, ox, g.N[0]);
    const int ly = local_index<2, 8, HALO>(fy, oy, g.N[1]);
    const int lz = local_index<2, 8, HALO>(fz, oz, g.N[2]);
    const bool home = (lx >= C::KLO) & (lx < C::KHI) & (ly >= C::KLO) & (ly < C::KHI) & (lz >= C::KLO) &
                      (lz < C::KHI);
    if (home) {
        const int k = ((lz - C::KLO) * C::KR + (ly - C::KLO)) * C::KR + (lx - C::KLO);
        if (!PCG_IN(k, NK)) return 0;
        const unsigned r = atomicAdd(&cnt[k], 1u);
        if (r < (unsigned)CAP) {
            float2 *dst = st + r * NK + k;
            dst[0] = make_float2(fx_, fy_);
            dst[CAP * NK] = make_float2(fz_, qvx);
            dst[2 * CAP * NK] = make_float2(qvy, qvz);
            return 0;
        }
        // more than CAP in this cell: straight to J like a halo particle
    } else {
        const bool fits = (lx >= -HALO) & (lx + 1 < 8 + HALO) & (ly >= -HALO) & (ly + 1 < 8 + HALO) &
                          (lz >= -HALO) & (lz + 1 < 8 + HALO);
        if (!fits) {
            deposit_global<3, 1>(g, J, x, y, z, qvx, qvy, qvz);
            return 2;
        }
    }
    stencil_to_global<HALO>(g, J, ox, oy, oz, lx, ly, lz, fx_, fy_, fz_, qvx, qvy, qvz);
    return 0;
}

template <int HALO>
__global__ void __launch_bounds__(512, 1)
    deposit_cic3d_v5_kernel(Geom g, Particles P, long long n, const uint32_t *__restrict__ offs,
                            const unsigned *__restrict__ chunk_tile, long long chunk, long long nchunks,
                            float *__restrict__ J, Counters ctr, bool vec) {
    using K = Cic5Cfg<HALO>;
    using C = typename K::C;
    constexpr int NK = K::NK, CAP = K::CAP, QCAP = K::QCAP;
    extern __shared__ __align__(16) unsigned char dsm[];
    float2 *st = reinterpret_cast<float2 *>(dsm);                              // [3][CAP][NK]
    int *qbuf = reinterpret_cast<int *>(st + 3 * CAP * NK);                    // [warps][QCAP]
    unsigned *cnt = reinterpret_cast<unsigned *>(qbuf + (K::THREADS / 32) * QCAP);  // [NK]

    const int tid = threadIdx.x, lane = tid & 31;
    int *wq = qbuf + (tid >> 5) * QCAP;  // this warp's queue: particle offsets in the round
    unsigned n_esc = 0, n_inv = 0;
    const int kx0 = tid % C::KR + C::KLO, ky0 = (tid / C::KR) % C::KR + C::KLO,
              kz0 = tid / (C::KR * C::KR) + C::KLO;

    if (tid < NK) cnt[tid] = 0;
    float acc[8][3];
#pragma unroll
    for (int a = 0; a < 8; ++a) acc[a][0] = acc[a][1] = acc[a][2] = 0.f;

    // the particles of one round, this thread's 8 slots
    float X[8], Y[8], Z[8], VX[8], VY[8], VZ[8], Q[8];
    auto load_round = [&](const RoundPos &r) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const long long b = r.rb + h * (K::R / 2) + 4 * tid;
            if (vec && b + 3 < n) {
                const float4 a = *reinterpret_cast<const float4 *>(P.x + b);
                const float4 bb = *reinterpret_cast<const float4 *>(P.y + b);
                const float4 c = *reinterpret_cast<const float4 *>(P.z + b);
                const float4 d = *reinterpret_cast<const float4 *>(P.vx + b);
                const float4 e = *reinterpret_cast<const float4 *>(P.vy + b);
                const float4 f = *reinterpret_cast<const float4 *>(P.vz + b);
                const float4 q = *reinterpret_cast<const float4 *>(P.q + b);
                X[4 * h] = a.x; X[4 * h + 1] = a.y; X[4 * h + 2] = a.z; X[4 * h + 3] = a.w;
                Y[4 * h] = bb.x; Y[4 * h + 1] = bb.y; Y[4 * h + 2] = bb.z; Y[4 * h + 3] = bb.w;
                Z[4 * h] = c.x; Z[4 * h + 1] = c.y; Z[4 * h + 2] = c.z; Z[4 * h + 3] = c.w;
                VX[4 * h] = d.x; VX[4 * h + 1] = d.y; VX[4 * h + 2] = d.z; VX[4 * h + 3] = d.w;
                VY[4 * h] = e.x; VY[4 * h + 1] = e.y; VY[4 * h + 2] = e.z; VY[4 * h + 3] = e.w;
                VZ[4 * h] = f.x; VZ[4 * h + 1] = f.y; VZ[4 * h + 2] = f.z; VZ[4 * h + 3] = f.w;
                Q[4 * h] = q.x; Q[4 * h + 1] = q.y; Q[4 * h + 2] = q.z; Q[4 * h + 3] = q.w;
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const long long p = (b + j < n) ? b + j : 0;
                    X[4 * h + j] = P.x[p]; Y[4 * h + j] = P.y[p]; Z[4 * h + j] = P.z[p];
                    VX[4 * h + j] = P.vx[p]; VY[4 * h + j] = P.vy[p]; VZ[4 * h + j] = P.vz[p];
                    Q[4 * h + j] = P.q[p];
                }
            }
        }
    };

    RoundPos cur;
    seek(g, offs, chunk_tile, n, chunk, nchunks, blockIdx.x, 0xffffffffu, cur);
    // the invalid tail and empty work never enter the round loop
    auto tail = [&](const RoundPos &r) {
        for (long long p = r.lo + tid; p < r.hi; p += K::THREADS) {
            const float x = P.x[p], y = P.y[p], z = P.z[p];
            if (!in_domain<3>(g, x, y, z)) {
                ++n_inv;
                continue;
            }
            const float q = P.q[p];
            deposit_global<3, 1>(g, J, x, y, z, q * P.vx[p], q * P.vy[p], q * P.vz[p]);
        }
    };
    while (cur.t == g.n_tiles) {  // a chunk that holds only invalid-tail particles
        tail(cur);
        seek(g, offs, chunk_tile, n, chunk, nchunks, cur.c + gridDim.x, 0xffffffffu, cur);
    }
    if (cur.t > g.n_tiles) {
        warp_add_u64(ctr.n_invalid, n_inv);
        return;
    }
    load_round(cur);
    __syncthreads();  // counters zeroed
    int ox = 0, oy = 0, oz = 0;  // origin of the current tile
    // A particle the fast path does not take (outside the tile's own cells, or
    // beyond CAP in its cell, or invalid) is queued by its warp; the warp then
    // takes its queue with one particle per lane: the general path runs once per
    // warp instead of inside the unrolled loop whenever any lane needs it, and
    // the global reductions of halo and overflow particles are issued there.
    auto slow_count = [&](int rc) {
        n_inv += rc == 1;
        n_esc += rc == 2;
    };
    const unsigned lanes_below = (1u << lane) - 1u;
    while (true) {
        // ---- place the round held in registers (tile cur.t, origin o*) ----
        const int tx = (int)(cur.t % (unsigned)g.nt[0]);
        const int ty = (int)((cur.t / (unsigned)g.nt[0]) % (unsigned)g.nt[1]);
        const int tz = (int)(cur.t / ((unsigned)g.nt[0] * (unsigned)g.nt[1]));
        ox = tx * 8;
        oy = ty * 8;
        oz = tz * 8;
        // the tile's own cells that exist (a last tile may stick out of the grid)
        const unsigned limx = (unsigned)min(C::KHI, g.N[0] - ox), limy = (unsigned)min(C::KHI, g.N[1] - oy),
                       limz = (unsigned)min(C::KHI, g.N[2] - oz);
        int qn = 0;  // particles this warp has queued this round (warp-uniform)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const long long p = cur.rb + (j >> 2) * (K::R / 2) + 4 * tid + (j & 3);
            const bool live = p >= cur.lo && p < cur.hi;
            const float x = X[j], y = Y[j], z = Z[j];
            const float qq = Q[j];
            const float qvx = qq * VX[j], qvy = qq * VY[j], qvz = qq * VZ[j];
            float fx_, fy_, fz_;
            const int fx = first_node<1>(x, fx_);
            const int fy = first_node<1>(y, fy_);
            const int fz = first_node<1>(z, fz_);
            // fast path: the cell is one of the tile's own cells inside the grid
            // and the coordinates are not negative (the conversion truncates
            // towards zero); then x, y, z are in the domain (a NaN fails too)
            const unsigned dx = (unsigned)(fx - ox), dy = (unsigned)(fy - oy), dz = (unsigned)(fz - oz);
            bool slow = live;
            if (live & (C::KLO == 0) & (x >= 0.f) & (y >= 0.f) & (z >= 0.f) & (dx < limx) & (dy < limy) &
                (dz < limz)) {
                const int k = ((int)dz * C::KR + (int)dy) * C::KR + (int)dx;
                const unsigned r = PCG_IN(k, NK) ? atomicAdd(&cnt[k], 1u) : (unsigned)CAP;
                if (r < (unsigned)CAP) {
                    float2 *dst = st + r * NK + k;
                    dst[0] = make_float2(fx_, fy_);
                    dst[CAP * NK] = make_float2(fz_, qvx);
                    dst[2 * CAP * NK] = make_float2(qvy, qvz);
                    slow = false;
                }
            }
            const unsigned m = __ballot_sync(0xffffffffu, slow);
            if (m) {  // warp-uniform
                if (slow && PCG_IN(qn + __popc(m & lanes_below), QCAP)) wq[qn + __popc(m & lanes_below)] = (int)(p - cur.rb);
                qn += __popc(m);
            }
        }
        // the warp's queue, one particle per lane: re-read from memory (it was
        // loaded one round ago and sits in L2), then the general path
        __syncwarp();
        for (int e = lane; e < qn; e += 32) {
            const long long pp = cur.rb + wq[e];
            if (!PCG_IN(pp, n)) continue;
            const float q = P.q[pp];
            slow_count(slow_particle<HALO>(g, J, st, cnt, ox, oy, oz, P.x[pp], P.y[pp], P.z[pp], q * P.vx[pp],
                                           q * P.vy[pp], q * P.vz[pp]));
        }
        __syncwarp();
        // ---- the next round: position, and its particles into registers ----
        RoundPos nxt = cur;
        nxt.rb = cur.rb + K::R;
        if (nxt.rb >= cur.hi) seek(g, offs, chunk_tile, n, chunk, nchunks, cur.c, cur.t + 1, nxt);
        const bool tile_ends = nxt.t != cur.t || nxt.c != cur.c;
        const bool more = nxt.t < g.n_tiles;
        // the next round's loads go out before the barrier, so that the warps
        // issue them as they finish placing instead of all at once after it
        if (more) load_round(nxt);
        __syncthreads();  // the round is staged

        // ---- every cell's thread adds its staged particles in registers ----
        if (tid < NK) {
            const unsigned m0 = cnt[tid];
            const unsigned m = m0 < (unsigned)CAP ? m0 : (unsigned)CAP;
            cnt[tid] = 0;
#pragma unroll 2
            for (unsigned r = 0; r < m; ++r) {
                const float2 a = st[r * NK + tid];
                const float2 b = st[CAP * NK + r * NK + tid];
                const float2 c = st[2 * CAP * NK + r * NK + tid];
                // moments sum qv fx^i fy^j fz^k (i, j, k in {0, 1}) in acc[i + 2j + 4k]
                const float fx = a.x, fy = a.y, fz = b.x;
                const float fxy = fx * fy, fxz = fx * fz, fyz = fy * fz, fxyz = fxy * fz;
                const float mono[8] = {1.f, fx, fy, fxy, fz, fxz, fyz, fxyz};
                const float qv[3] = {b.y, c.x, c.y};
#pragma unroll
                for (int comp = 0; comp < 3; ++comp) {
                    acc[0][comp] += qv[comp];
#pragma unroll
                    for (int i = 1; i < 8; ++i) acc[i][comp] = fmaf(qv[comp], mono[i], acc[i][comp]);
                }
            }
        }
        if (tile_ends) {
            // The tile's flush without shared-memory float atomics: every cell's 8
            // corners x 3 components go to the (now free) staging area with plain
            // stores; after a barrier one thread per node sums the up to 8 cell
            // corners that meet there and adds the total to J once.
            float *corner = reinterpret_cast<float *>(st);  // [24][NK]
            __syncthreads();  // every cell's staged particles have been read
            if (tid < NK) {
                // moments -> corner weights: along each axis the CIC weights are
                // 1 - f and f, so the low corner is M0 - M1 and the high one M1
#pragma unroll
                for (int comp = 0; comp < 3; ++comp)
#pragma unroll
                    for (int bit = 1; bit < 8; bit <<= 1)
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            if (!(i & bit)) acc[i][comp] -= acc[i | bit][comp];
#pragma unroll
                for (int a = 0; a < 8; ++a)
#pragma unroll
                    for (int comp = 0; comp < 3; ++comp) {
                        corner[(a * 3 + comp) * NK + tid] = acc[a][comp];
                        acc[a][comp] = 0.f;
                    }
            }
            __syncthreads();
            constexpr int NR = C::KR + 1;
            for (int nd = tid; nd < NR * NR * NR; nd += K::THREADS) {
                const int nx = nd % NR, ny = (nd / NR) % NR, nz = nd / (NR * NR);
                float sum[3] = {0.f, 0.f, 0.f};
#pragma unroll
                for (int a = 0; a < 8; ++a) {
                    const int cx = nx - (a & 1), cy = ny - ((a >> 1) & 1), cz = nz - (a >> 2);
                    if (cx < 0 || cx >= C::KR || cy < 0 || cy >= C::KR || cz < 0 || cz >= C::KR) continue;
                    const int cell = (cz * C::KR + cy) * C::KR + cx;
#pragma unroll
                    for (int comp = 0; comp < 3; ++comp) sum[comp] += corner[(a * 3 + comp) * NK + cell];
                }
                int gx = ox + C::KLO + nx, gy = oy + C::KLO + ny, gz = oz + C::KLO + nz;
                while (gx >= g.N[0]) gx -= g.N[0];
                while (gy >= g.N[1]) gy -= g.N[1];
                while (gz >= g.N[2]) gz -= g.N[2];
                const long long node = ((long long)gz * g.N[1] + gy) * g.N[0] + gx;
                if (!PCG_IN(node, g.ncells)) continue;
#pragma unroll
                for (int comp = 0; comp < 3; ++comp)
                    if (sum[comp] != 0.f) red_add_f32(J + comp * g.ncells + node, sum[comp]);
            }
        }
        if (!more) {
            // the invalid tail sits at the end of the array: after it come only
            // chunks that are all tail or past the end
            RoundPos r = nxt;
            while (r.t == g.n_tiles) {
                tail(r);
                seek(g, offs, chunk_tile, n, chunk, nchunks, r.c + gridDim.x, 0xffffffffu, r);
            }
            break;
        }
        cur = nxt;
        __syncthreads();  // staging and corner values read
    }
    warp_add_u64(ctr.n_escaped, n_esc);
    warp_add_u64(ctr.n_invalid, n_inv);
}

template <int HALO>
pcg_status launch_cic3d_v5(const Geom &g, long long n, const Particles &P, const uint32_t *offs, float *J,
                           const Counters &ctr, const unsigned *chunk_tile, long long chunk, cudaStream_t s) {
    using K = Cic5Cfg<HALO>;
    const long long nchunks = (n + chunk - 1) / chunk;
    if (nchunks == 0) return PCG_OK;
    const bool vec = aligned16(P.x) && aligned16(P.y) && aligned16(P.z) && aligned16(P.vx) &&
                     aligned16(P.vy) && aligned16(P.vz) && aligned16(P.q);
    const long long sms = num_sms();
    const unsigned grid = (unsigned)(nchunks < sms ? nchunks : sms);
    PCG_CHECK_CUDA(cudaFuncSetAttribute(deposit_cic3d_v5_kernel<HALO>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)K::SMEM));
    prof::Mark mk("deposit_tiled", s);
    deposit_cic3d_v5_kernel<HALO><<<grid, K::THREADS, K::SMEM, s>>>(g, P, n, offs, chunk_tile, chunk, nchunks,
                                                                    J, ctr, vec);
    return launch_status();
}


}  // namespace dep
}  // namespace pcg

#include "deposit_quad3d.cuh"

namespace pcg {
namespace dep {

template <int DIM, int ORDER, int TILE, int HALO, int THREADS>
size_t tiled_smem() {
    using C = TileCfg<DIM, ORDER, TILE, HALO>;
    return (size_t)C::FLOATS * 4 + 3 * (size_t)C::NKEYS * 4 + 7 * (size_t)BatchCfg<THREADS>::SB * 4;
}

template <int DIM, int ORDER, int TILE, int HALO, int THREADS>
pcg_status launch_tiled_t(const Geom &g, long long n, const Particles &P, const uint32_t *offs,
                          float *J, const Counters &ctr, const unsigned *chunk_tile, long long chunk,
                          cudaStream_t s) {
    const long long nchunks = (n + chunk - 1) / chunk;
    if (nchunks == 0) return PCG_OK;
    const bool vec4 = aligned16(P.x) && aligned16(P.y) && (DIM == 2 || aligned16(P.z)) &&
                      aligned16(P.vx) && aligned16(P.vy) && aligned16(P.vz) && aligned16(P.q);
    const size_t smem = tiled_smem<DIM, ORDER, TILE, HALO, THREADS>();
    PCG_CHECK_CUDA(cudaFuncSetAttribute(deposit_tiled_kernel<DIM, ORDER, TILE, HALO, THREADS>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    prof::Mark mk("deposit_tiled", s);
    deposit_tiled_kernel<DIM, ORDER, TILE, HALO, THREADS>
        <<<(unsigned)nchunks, THREADS, smem, s>>>(g, P, n, offs, chunk_tile, chunk, J, ctr, vec4);
    return launch_status();
}

template <int DIM, int ORDER, int TILE, int HALO>
pcg_status launch_tiled(const Geom &g, long long n, const Particles &P, const uint32_t *offs,
                        float *J, const Counters &ctr, const unsigned *chunk_tile, long long chunk,
                        int block, cudaStream_t s) {
    if constexpr (DIM == 3 && ORDER == 1 && TILE == 8) {
        // block 512 asks for one 512-thread CTA per SM with the full register file
        return launch_cic3d_v5<HALO>(g, n, P, offs, J, ctr, chunk_tile, chunk, s);
    } else if constexpr (DIM == 3 && ORDER == 2 && TILE == 8) {
        return launch_quad3d<HALO>(g, n, P, offs, J, ctr, chunk_tile, chunk, s);
    } else {
        if (block == 512)
            return launch_tiled_t<DIM, ORDER, TILE, HALO, 512>(g, n, P, offs, J, ctr, chunk_tile, chunk, s);
        return launch_tiled_t<DIM, ORDER, TILE, HALO, 256>(g, n, P, offs, J, ctr, chunk_tile, chunk, s);
    }
}

template <int DIM, int ORDER, int TILE>
pcg_status dispatch_halo(int halo, const Geom &g, long long n, const Particles &P,
                         const uint32_t *offs, float *J, const Counters &ctr,
                         const unsigned *chunk_tile, long long chunk, int block, cudaStream_t s) {
    switch (halo) {
        case 0: return launch_tiled<DIM, ORDER, TILE, 0>(g, n, P, offs, J, ctr, chunk_tile, chunk, block, s);
        case 1: return launch_tiled<DIM, ORDER, TILE, 1>(g, n, P, offs, J, ctr, chunk_tile, chunk, block, s);
        case 2: return launch_tiled<DIM, ORDER, TILE, 2>(g, n, P, offs, J, ctr, chunk_tile, chunk, block, s);
        default: return PCG_ERR_UNSUPPORTED;
    }
}

template <int DIM>
pcg_status dispatch_tiled(int order, int tile, int halo, const Geom &g, long long n,
                          const Particles &P, const uint32_t *offs, float *J, const Counters &ctr,
                          unsigned *chunk_tile, long long chunk, int block, cudaStream_t s) {
    if (order == 1 && tile == 8) return dispatch_halo<DIM, 1, 8>(halo, g, n, P, offs, J, ctr, chunk_tile, chunk, block, s);
    if (order == 1 && tile == 4) return dispatch_halo<DIM, 1, 4>(halo, g, n, P, offs, J, ctr, chunk_tile, chunk, block, s);
    if (order == 2 && tile == 8) return dispatch_halo<DIM, 2, 8>(halo, g, n, P, offs, J, ctr, chunk_tile, chunk, block, s);
    if (order == 2 && tile == 4) return dispatch_halo<DIM, 2, 4>(halo, g, n, P, offs, J, ctr, chunk_tile, chunk, block, s);
    return PCG_ERR_UNSUPPORTED;
}

}  // namespace dep
}  // namespace pcg
