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
                        atomicAdd(&cnt[k], 1u);
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
                stage[0 * BC::SB + slot] = off[i][0];
                stage[1 * BC::SB + slot] = off[i][1];
                stage[2 * BC::SB + slot] = off[i][2];
                stage[3 * BC::SB + slot] = qv[i][0];
                stage[4 * BC::SB + slot] = qv[i][1];
                stage[5 * BC::SB + slot] = qv[i][2];
            }
            __syncthreads();

            // ---- D: one thread per group sums its particles, then adds each node once ----
            for (int k = threadIdx.x; k < NK; k += THREADS) {
                const unsigned m = cnt[k];
                if (m == 0) continue;
                const unsigned b0 = start[k];
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

        // flush: one global reduction per non-zero scratch cell, periodic wrap
        for (int i = threadIdx.x; i < C::FLOATS; i += THREADS) {
            const float val = scratch[i];
            if (val == 0.f) continue;
            const int c = i / C::CELLS;
            const int r = i - c * C::CELLS;
            const int sx = r % C::TE;
            const int sy = (r / C::TE) % C::TE;
            const int sz = DIM == 3 ? r / (C::TE * C::TE) : 0;
            const int gx = wrap_index(ox - HALO + sx, g.N[0]);
            const int gy = wrap_index(oy - HALO + sy, g.N[1]);
            const int gz = DIM == 3 ? wrap_index(oz - HALO + sz, g.N[2]) : 0;
            red_add_f32(J + c * g.ncells + ((long long)gz * g.N[1] + gy) * g.N[0] + gx, val);
        }
        __syncthreads();  // scratch is reused by the next segment
    }
    warp_add_u64(ctr.n_escaped, n_esc);
    warp_add_u64(ctr.n_invalid, n_inv);
}

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
    if (block == 512)
        return launch_tiled_t<DIM, ORDER, TILE, HALO, 512>(g, n, P, offs, J, ctr, chunk_tile, chunk, s);
    return launch_tiled_t<DIM, ORDER, TILE, HALO, 256>(g, n, P, offs, J, ctr, chunk_tile, chunk, s);
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
