// deposit_zigzag.cu -- charge-conserving zigzag current deposit (3D, CIC charge).
//
// Method.  "Tiled current deposit" (Entity wiki), section "Halo sizing", names
// the O == 0 zigzag deposit: it writes at most 2 cells above min(i, i_prev).
// The scheme is the relay split of Umeda, Omura, Tominaga & Matsumoto, Comput.
// Phys. Commun. 156 (2003) 73.  Per axis, with cells i1 = floor(x1),
// i2 = floor(x2) (|i2 - i1| <= 1 after the periodic minimum image):
//   relay  xr = min(min(i1, i2) + 1, max(max(i1, i2), (x1 + x2) / 2)),
//   moves  D1 = xr - x1,  D2 = x2 - xr,  fluxes F_s = q D_s / dt,
//   shape  W1 = (x1 + xr) / 2 - i1,  W2 = (xr + x2) / 2 - i2.
// Segment s adds to J^c on the four c-edges of its cell that start at
// (cell + a e_u + b e_v), u and v the transverse axes, the flux F_s^c times
//   w_a(W_s^u) w_b(W_s^v) + (a == b ? 1 : -1) D_s^u D_s^v / 12,
// w_0(W) = 1 - W, w_1(W) = W: the bilinear weight averaged along the straight
// segment, which keeps (rho(x2) - rho(x1)) / dt + div J = 0 exact in 3D (the
// D D / 12 term vanishes when a segment moves along at most two axes, where
// the weight is Umeda's midpoint one).  J[c] at node index (k*Ny + j)*Nx + i is
// the c-current on the edge from node (i, j, k) towards +e_c.
//
// Tiled path ("How a tile deposit runs", "Halo sizing", "Correctness is
// independent of the halo").  The particles are sorted by the tile of their
// previous position (the page keys on min(i, i_prev) to put the whole halo on
// the high side; here every segment whose cell lies outside the tile goes to J
// directly, so the key needs no such shift).  A particle whose 3 x 3 x 3 node
// footprint leaves the window of a 2-cell halo around its tile is counted as an
// escape, as the page's escape valve defines it.  The kernel itself is
// described above zigzag_cells_kernel.
#include "deposit_tiled.cuh"

namespace pcg {
namespace {

using dep::Counters;
using dep::Geom;

struct ZParticles {
    const float *x1[3];  // previous positions
    const float *x2[3];  // current positions
    const float *q;
};

// One particle's zigzag split: the lower cell of the move (per axis, in
// [-1, N)), each segment's cell relative to it (0 or 1), the fluxes, the
// segment midpoints relative to their cells and the segment moves.
struct Zig {
    int base[3];
    int cell[2][3];
    float F[2][3], W[2][3], D[2][3];
    bool same;  // both segments in one cell
};

__device__ __forceinline__ bool zigzag_split(const Geom &g, const float (&x1)[3], const float (&x2)[3], float q,
                                             float inv_dt, Zig &z) {
    bool ok = true;
    z.same = true;
#pragma unroll
    for (int mu = 0; mu < 3; ++mu) {
        const float a1 = x1[mu], a2 = x2[mu];
        ok &= (a1 >= 0.f) & (a1 < g.Nf[mu]) & (a2 >= 0.f) & (a2 < g.Nf[mu]);
        const int i1 = (int)a1, i2 = (int)a2;  // floor: both are >= 0 when ok
        int di = i2 - i1;                       // periodic minimum image
        if (2 * di > g.N[mu]) di -= g.N[mu];
        if (2 * di < -g.N[mu]) di += g.N[mu];
        ok &= (di >= -1) & (di <= 1);
        const int lo = di < 0 ? di : 0;
        const int a = -lo, b = di - lo;
        const float X1 = (float)a + (a1 - (float)i1);
        const float X2 = (float)b + (a2 - (float)i2);
        const float xr = fminf(1.f, fmaxf((float)(a > b ? a : b), 0.5f * (X1 + X2)));
        z.base[mu] = i1 + lo;
        z.cell[0][mu] = a;
        z.cell[1][mu] = b;
        z.same &= a == b;
        z.D[0][mu] = xr - X1;
        z.D[1][mu] = X2 - xr;
        z.F[0][mu] = q * z.D[0][mu] * inv_dt;
        z.F[1][mu] = q * z.D[1][mu] * inv_dt;
        z.W[0][mu] = 0.5f * (X1 + xr) - (float)a;
        z.W[1][mu] = 0.5f * (xr + X2) - (float)b;
    }
    return ok;
}

// The four edge weights of component c for segment s, times its flux:
// out[b][a] for the edge at cell + a e_u + b e_v.
template <int C>
__device__ __forceinline__ void edge_values(const Zig &z, int s, float (&out)[2][2]) {
    constexpr int U = (C + 1) % 3, V = (C + 2) % 3;
    const float wu = z.W[s][U], wv = z.W[s][V];
    const float avg = z.D[s][U] * z.D[s][V] * (1.f / 12.f);
    const float F = z.F[s][C];
    out[0][0] = F * ((1.f - wu) * (1.f - wv) + avg);
    out[0][1] = F * (wu * (1.f - wv) - avg);
    out[1][0] = F * ((1.f - wu) * wv - avg);
    out[1][1] = F * (wu * wv + avg);
}

// Visit the 12 (same cell) or 24 edge values of a particle:
// put(c, dx, dy, dz, value) with (dx, dy, dz) the edge's start node relative
// to base, each in {0, 1, 2}.
template <class Put>
__device__ __forceinline__ void zigzag_edges(const Zig &z, Put put) {
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        if (s == 1 && z.same) break;
        const int cx = z.cell[s][0], cy = z.cell[s][1], cz = z.cell[s][2];
        float v[2][2];
        // J^x: edges (cx, cy + a, cz + b)
        edge_values<0>(z, s, v);
        if (z.same) {
            float w[2][2];
            edge_values<0>(z, 1, w);
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i >> 1][i & 1] += w[i >> 1][i & 1];
        }
#pragma unroll
        for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int a = 0; a < 2; ++a) put(0, cx, cy + a, cz + b, v[b][a]);
        // J^y: U = z, V = x: edges (cx + b, cy, cz + a)
        edge_values<1>(z, s, v);
        if (z.same) {
            float w[2][2];
            edge_values<1>(z, 1, w);
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i >> 1][i & 1] += w[i >> 1][i & 1];
        }
#pragma unroll
        for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int a = 0; a < 2; ++a) put(1, cx + b, cy, cz + a, v[b][a]);
        // J^z: U = x, V = y: edges (cx + a, cy + b, cz)
        edge_values<2>(z, s, v);
        if (z.same) {
            float w[2][2];
            edge_values<2>(z, 1, w);
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i >> 1][i & 1] += w[i >> 1][i & 1];
        }
#pragma unroll
        for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int a = 0; a < 2; ++a) put(2, cx + a, cy + b, cz, v[b][a]);
    }
}

__device__ __forceinline__ int wrap_once(int i, int N) { return i < 0 ? i + N : (i >= N ? i - N : i); }

// All edges of one particle into J with global reductions (periodic wrap).
__device__ __forceinline__ void zigzag_global(const Geom &g, float *__restrict__ J, const Zig &z) {
    zigzag_edges(z, [&](int c, int dx, int dy, int dz, float v) {
        // base in [-1, N), d <= 2 and N >= 3: at most one correction
        const int gx = wrap_once(z.base[0] + dx, g.N[0]);
        const int gy = wrap_once(z.base[1] + dy, g.N[1]);
        const int gz = wrap_once(z.base[2] + dz, g.N[2]);
        const long long node = ((long long)gz * g.N[1] + gy) * g.N[0] + gx;
        if (PCG_IN(node, g.ncells)) red_add_f32(J + c * g.ncells + node, v);
    });
}

__device__ __forceinline__ void load_particle(const ZParticles &P, long long p, float (&x1)[3], float (&x2)[3],
                                              float &q) {
#pragma unroll
    for (int mu = 0; mu < 3; ++mu) {
        x1[mu] = P.x1[mu][p];
        x2[mu] = P.x2[mu][p];
    }
    q = P.q[p];
}

__global__ void __launch_bounds__(256)
    zigzag_flat_kernel(Geom g, ZParticles P, long long n, float inv_dt, float *__restrict__ J, Counters ctr) {
    unsigned n_inv = 0;
    for (long long p = blockIdx.x * (long long)blockDim.x + threadIdx.x; p < n;
         p += (long long)gridDim.x * blockDim.x) {
        float x1[3], x2[3], q;
        load_particle(P, p, x1, x2, q);
        Zig z;
        if (!zigzag_split(g, x1, x2, q, inv_dt, z)) {
            ++n_inv;
            continue;
        }
        zigzag_global(g, J, z);
    }
    warp_add_u64(ctr.n_invalid, n_inv);
}

// ---------------------------------------------------------------------------
// Tiled kernel.  A particle's zigzag current is the sum of its segments' (one
// straight segment when it stays in its cell, the two relay segments when it
// crosses a face), and a segment with midpoint m (relative to its cell), move D
// and flux F = q D / dt adds to the c-edges of its cell at cell + a e_u + b e_v
//   F^c (w_a(m^u) w_b(m^v) + (a == b ? 1 : -1) D^u D^v / 12),
// which depends on the segment only through four sums per component:
//   S0 = sum F^c, Su = sum F^c m^u, Sv = sum F^c m^v,
//   Q = sum F^c (m^u m^v + D^u D^v / 12),
// giving the edges (a, b) = (0, 0): S0 - Su - Sv + Q, (1, 0): Su - Q,
// (0, 1): Sv - Q, (1, 1): Q.  So one thread per cell of the 8^3 tile keeps its
// cell's 12 sums in registers for the whole tile segment, as the CIC kernel
// does with its corner moments.
//
// One persistent CTA of 512 threads per SM walks the chunks b, b + grid, ... of
// the array sorted by the tile of the previous position, in rounds of 4096
// particles (8 per thread, float4 loads per field, the next round loaded into
// registers before this one is accumulated).  A round's segments are placed by
// rank (a shared u32 counting atomic) into per-cell lists st[pair][rank][cell]
// that the cell threads read conflict-free.  Particles that stay in one of the
// tile's cells take the fast path (one segment, a few multiplies); the others
// (crossing a face, about 11 % at v ~ N(0, 0.05^2); invalid; outside the tile)
// are queued per warp and taken one per lane after the warp's placements: the
// full relay split, each segment listed when its cell is one of the tile's, or
// added to J with global reductions.  At a tile segment's end every cell thread
// stores its 12 edge values, and one thread per edge adds the <= 4 cells' values
// that meet there and issues one global reduction.  No shared-memory float
// atomics: on this GPU they are a serial read-modify-write.
struct ZzCfg {
    static constexpr int THREADS = 512;
    static constexpr int NC = 512;                // cells of an 8^3 tile, one thread each
    static constexpr int PPT = 8;                 // particles per thread per round
    static constexpr int R = THREADS * PPT;       // round size
    static constexpr int CAP = 14;                // listed segments per cell and round
    static constexpr int QCAP = PPT * 32;         // queued particles per warp and round: room for all
    static constexpr size_t LIST = (size_t)CAP * NC;
    static constexpr size_t SMEM = LIST * 3 * 8 + LIST * 4 + (size_t)(THREADS / 32) * QCAP * 4 + (size_t)NC * 4;
    static_assert(THREADS == NC, "one thread per cell");
    static_assert((size_t)12 * NC * 4 <= LIST * 3 * 8, "the edge values fit in the list area");
};

// List a segment of tile-local cell `cell` (midpoint m, move D, q / dt):
// false when the cell's list is full.
__device__ __forceinline__ bool zz_list(float2 *st, float *sq, unsigned *cnt, int cell, float mx, float my,
                                        float mz, float Dx, float Dy, float Dz, float qdt) {
    using K = ZzCfg;
    if (!PCG_IN(cell, K::NC)) return false;
    const unsigned r = atomicAdd(&cnt[cell], 1u);
    if (r >= (unsigned)K::CAP) return false;
    float2 *e = st + (size_t)r * K::NC + cell;
    e[0] = make_float2(mx, my);
    e[K::LIST] = make_float2(mz, Dx);
    e[2 * K::LIST] = make_float2(Dy, Dz);
    sq[(size_t)r * K::NC + cell] = qdt;
    return true;
}

// The 12 edges of one segment of global cell (cx, cy, cz) (each in [-1, N]) into
// J with global reductions (periodic wrap).
__device__ __forceinline__ void zz_segment_global(const Geom &g, float *__restrict__ J, int cx, int cy, int cz,
                                                  const float (&m)[3], const float (&D)[3], float qdt) {
    const int cell[3] = {cx, cy, cz};
#pragma unroll
    for (int c = 0; c < 3; ++c) {
        const int u = (c + 1) % 3, v = (c + 2) % 3;
        const float F = qdt * D[c];
        const float Su = F * m[u], Sv = F * m[v];
        const float Q = F * (m[u] * m[v] + D[u] * D[v] * (1.f / 12.f));
        const float val[2][2] = {{F - Su - Sv + Q, Su - Q}, {Sv - Q, Q}};  // [b][a]
#pragma unroll
        for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int a = 0; a < 2; ++a) {
                int nd[3] = {cell[0], cell[1], cell[2]};
                nd[u] += a;
                nd[v] += b;
                const int gx = wrap_once(nd[0], g.N[0]), gy = wrap_once(nd[1], g.N[1]),
                          gz = wrap_once(nd[2], g.N[2]);
                const long long node = ((long long)gz * g.N[1] + gy) * g.N[0] + gx;
                if (PCG_IN(node, g.ncells)) red_add_f32(J + c * g.ncells + node, val[b][a]);
            }
    }
}

// The general path of a queued particle of the tile at (ox, oy, oz): the full
// relay split; each segment listed when its cell is one of the tile's (list
// not full), else added to J.  Returns 1 invalid (skipped), 2 escaped (its
// 3 x 3 x 3 node footprint leaves the window [-HALO, 8 + HALO) of the tile, the
// escape valve's definition), 0 otherwise.
template <int HALO>
__device__ __forceinline__ int zz_slow(const Geom &g, float *J, float2 *st, float *sq, unsigned *cnt, int ox,
                                       int oy, int oz, const float (&x1)[3], const float (&x2)[3], float q,
                                       float inv_dt) {
    Zig z;
    if (!zigzag_split(g, x1, x2, q, inv_dt, z)) return 1;
    const int lx = dep::local_index<3, 8, HALO>(z.base[0], ox, g.N[0]);
    const int ly = dep::local_index<3, 8, HALO>(z.base[1], oy, g.N[1]);
    const int lz = dep::local_index<3, 8, HALO>(z.base[2], oz, g.N[2]);
    const bool fits = (lx >= -HALO) & (lx + 2 < 8 + HALO) & (ly >= -HALO) & (ly + 2 < 8 + HALO) &
                      (lz >= -HALO) & (lz + 2 < 8 + HALO);
    const float qdt = q * inv_dt;
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        const int cx = z.base[0] + z.cell[s][0], cy = z.base[1] + z.cell[s][1], cz = z.base[2] + z.cell[s][2];
        const unsigned dx = (unsigned)(cx - ox), dy = (unsigned)(cy - oy), dz = (unsigned)(cz - oz);
        if ((dx < 8u) & (dy < 8u) & (dz < 8u) &&
            zz_list(st, sq, cnt, ((int)dz * 8 + (int)dy) * 8 + (int)dx, z.W[s][0], z.W[s][1], z.W[s][2],
                    z.D[s][0], z.D[s][1], z.D[s][2], qdt))
            continue;
        const float m[3] = {z.W[s][0], z.W[s][1], z.W[s][2]};
        const float D[3] = {z.D[s][0], z.D[s][1], z.D[s][2]};
        zz_segment_global(g, J, cx, cy, cz, m, D, qdt);
    }
    return fits ? 0 : 2;
}

template <int HALO>
__global__ void __launch_bounds__(512, 1)
    zigzag_cells_kernel(Geom g, ZParticles P, long long n, float inv_dt, const uint32_t *__restrict__ offs,
                        const unsigned *__restrict__ chunk_tile, long long chunk, long long nchunks,
                        float *__restrict__ J, Counters ctr, bool vec) {
    using K = ZzCfg;
    constexpr int NC = K::NC, CAP = K::CAP, QCAP = K::QCAP;
    extern __shared__ __align__(16) unsigned char dsm[];
    float2 *st = reinterpret_cast<float2 *>(dsm);                                 // [3][CAP][NC]
    float *sq = reinterpret_cast<float *>(st + 3 * K::LIST);                      // [CAP][NC]: q / dt
    int *qbuf = reinterpret_cast<int *>(sq + K::LIST);                            // [warps][QCAP]
    unsigned *cnt = reinterpret_cast<unsigned *>(qbuf + (K::THREADS / 32) * QCAP);  // [NC]

    const int tid = threadIdx.x, lane = tid & 31;
    int *wq = qbuf + (tid >> 5) * QCAP;
    unsigned n_esc = 0, n_inv = 0;
    cnt[tid] = 0;
    float acc[3][4];  // per component: S0, Su, Sv, Q
#pragma unroll
    for (int c = 0; c < 3; ++c) acc[c][0] = acc[c][1] = acc[c][2] = acc[c][3] = 0.f;

    // the particles of one round, this thread's 8 slots
    float A[3][8], B[3][8], Q[8];  // previous position, position, charge
    auto load_round = [&](const dep::RoundPos &r) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const long long b = r.rb + h * (K::R / 2) + 4 * tid;
            if (vec && b + 3 < n) {
#pragma unroll
                for (int mu = 0; mu < 3; ++mu) {
                    const float4 a = *reinterpret_cast<const float4 *>(P.x1[mu] + b);
                    const float4 c = *reinterpret_cast<const float4 *>(P.x2[mu] + b);
                    A[mu][4 * h] = a.x; A[mu][4 * h + 1] = a.y; A[mu][4 * h + 2] = a.z; A[mu][4 * h + 3] = a.w;
                    B[mu][4 * h] = c.x; B[mu][4 * h + 1] = c.y; B[mu][4 * h + 2] = c.z; B[mu][4 * h + 3] = c.w;
                }
                const float4 q = *reinterpret_cast<const float4 *>(P.q + b);
                Q[4 * h] = q.x; Q[4 * h + 1] = q.y; Q[4 * h + 2] = q.z; Q[4 * h + 3] = q.w;
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const long long p = (b + j < n) ? b + j : 0;
#pragma unroll
                    for (int mu = 0; mu < 3; ++mu) {
                        A[mu][4 * h + j] = P.x1[mu][p];
                        B[mu][4 * h + j] = P.x2[mu][p];
                    }
                    Q[4 * h + j] = P.q[p];
                }
            }
        }
    };
    // slots after the last tile: the flat path, straight to J
    auto tail = [&](const dep::RoundPos &r) {
        for (long long p = r.lo + tid; p < r.hi; p += K::THREADS) {
            float x1[3], x2[3], q;
            load_particle(P, p, x1, x2, q);
            Zig z;
            if (!zigzag_split(g, x1, x2, q, inv_dt, z)) {
                ++n_inv;
                continue;
            }
            zigzag_global(g, J, z);
        }
    };

    dep::RoundPos cur;
    dep::seek(g, offs, chunk_tile, n, chunk, nchunks, blockIdx.x, 0xffffffffu, cur);
    while (cur.t == g.n_tiles) {  // a chunk that holds only invalid-tail particles
        tail(cur);
        dep::seek(g, offs, chunk_tile, n, chunk, nchunks, cur.c + gridDim.x, 0xffffffffu, cur);
    }
    if (cur.t > g.n_tiles) {
        warp_add_u64(ctr.n_invalid, n_inv);
        return;
    }
    load_round(cur);
    __syncthreads();  // counters zeroed
    auto slow_count = [&](int rc) {
        n_inv += rc == 1;
        n_esc += rc == 2;
    };
    const unsigned lanes_below = (1u << lane) - 1u;
    while (true) {
        const int tx = (int)(cur.t % (unsigned)g.nt[0]);
        const int ty = (int)((cur.t / (unsigned)g.nt[0]) % (unsigned)g.nt[1]);
        const int tz = (int)(cur.t / ((unsigned)g.nt[0] * (unsigned)g.nt[1]));
        const int ox = tx * 8, oy = ty * 8, oz = tz * 8;
        // ---- place the round held in registers: one straight segment for a
        // particle that stays in one of the tile's cells ----
        int qn = 0;  // particles this warp has queued this round (warp-uniform)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const long long p = cur.rb + (j >> 2) * (K::R / 2) + 4 * tid + (j & 3);
            const bool live = p >= cur.lo && p < cur.hi;
            bool fast = live;
            int ic[3];
            float f1[3], f2[3];
#pragma unroll
            for (int mu = 0; mu < 3; ++mu) {
                const float a1 = A[mu][j], a2 = B[mu][j];
                // both positions in [0, N) (a NaN fails) and in the same cell
                fast &= (a1 >= 0.f) & (a1 < g.Nf[mu]) & (a2 >= 0.f) & (a2 < g.Nf[mu]);
                const int i1 = (int)a1, i2 = (int)a2;
                fast &= i1 == i2;
                ic[mu] = i1;
                f1[mu] = a1 - (float)i1;
                f2[mu] = a2 - (float)i2;
            }
            const unsigned dx = (unsigned)(ic[0] - ox), dy = (unsigned)(ic[1] - oy), dz = (unsigned)(ic[2] - oz);
            fast &= (dx < 8u) & (dy < 8u) & (dz < 8u);
            bool slow = live;
            if (fast) {
                const float qdt = Q[j] * inv_dt;
                slow = !zz_list(st, sq, cnt, ((int)dz * 8 + (int)dy) * 8 + (int)dx, 0.5f * (f1[0] + f2[0]),
                                0.5f * (f1[1] + f2[1]), 0.5f * (f1[2] + f2[2]), f2[0] - f1[0], f2[1] - f1[1],
                                f2[2] - f1[2], qdt);
            }
            const unsigned m = __ballot_sync(0xffffffffu, slow);
            if (m) {  // warp-uniform
                const int at = qn + __popc(m & lanes_below);
                if (slow && PCG_IN(at, QCAP)) wq[at] = (int)(p - cur.rb);
                qn += __popc(m);
            }
        }
        // the warp's queue, one particle per lane: re-read from memory (it was
        // loaded one round ago and sits in L2), then the general path
        __syncwarp();
        for (int e = lane; e < qn; e += 32) {
            const long long pp = cur.rb + wq[e];
            if (!PCG_IN(pp, n)) continue;
            float x1[3], x2[3], q;
            load_particle(P, pp, x1, x2, q);
            slow_count(zz_slow<HALO>(g, J, st, sq, cnt, ox, oy, oz, x1, x2, q, inv_dt));
        }
        __syncwarp();
        // ---- the next round: position, and its particles into registers ----
        dep::RoundPos nxt = cur;
        nxt.rb = cur.rb + K::R;
        if (nxt.rb >= cur.hi) dep::seek(g, offs, chunk_tile, n, chunk, nchunks, cur.c, cur.t + 1, nxt);
        const bool tile_ends = nxt.t != cur.t || nxt.c != cur.c;
        const bool more = nxt.t < g.n_tiles;
        // issued before the barrier, so that the warps issue them as they finish placing
        if (more) load_round(nxt);
        __syncthreads();  // the round is listed

        // ---- every cell's thread adds its listed segments' sums ----
        {
            const unsigned m0 = cnt[tid];
            const unsigned m = m0 < (unsigned)CAP ? m0 : (unsigned)CAP;
            cnt[tid] = 0;
#pragma unroll 2
            for (unsigned r = 0; r < m; ++r) {
                const float2 a = st[(size_t)r * NC + tid];
                const float2 b = st[K::LIST + (size_t)r * NC + tid];
                const float2 c = st[2 * K::LIST + (size_t)r * NC + tid];
                const float qdt = sq[(size_t)r * NC + tid];
                const float mx = a.x, my = a.y, mz = b.x, Dx = b.y, Dy = c.x, Dz = c.y;
                const float Fx = qdt * Dx, Fy = qdt * Dy, Fz = qdt * Dz;
                // per component c (u, v the next two axes): m^u m^v + D^u D^v / 12
                const float pyz = fmaf(Dy * Dz, 1.f / 12.f, my * mz);
                const float pzx = fmaf(Dz * Dx, 1.f / 12.f, mz * mx);
                const float pxy = fmaf(Dx * Dy, 1.f / 12.f, mx * my);
                acc[0][0] += Fx;
                acc[0][1] = fmaf(Fx, my, acc[0][1]);
                acc[0][2] = fmaf(Fx, mz, acc[0][2]);
                acc[0][3] = fmaf(Fx, pyz, acc[0][3]);
                acc[1][0] += Fy;
                acc[1][1] = fmaf(Fy, mz, acc[1][1]);
                acc[1][2] = fmaf(Fy, mx, acc[1][2]);
                acc[1][3] = fmaf(Fy, pzx, acc[1][3]);
                acc[2][0] += Fz;
                acc[2][1] = fmaf(Fz, mx, acc[2][1]);
                acc[2][2] = fmaf(Fz, my, acc[2][2]);
                acc[2][3] = fmaf(Fz, pxy, acc[2][3]);
            }
        }
        if (tile_ends) {
            // every cell's 12 edge values to the free list area with plain stores;
            // after a barrier one thread per edge adds the <= 4 cells' values that
            // meet there and reduces the total into J once
            float *edge = reinterpret_cast<float *>(st);  // [3][4][NC]: (c, b * 2 + a)
            __syncthreads();  // every list has been read
#pragma unroll
            for (int c = 0; c < 3; ++c) {
                const float S0 = acc[c][0], Su = acc[c][1], Sv = acc[c][2], Qc = acc[c][3];
                edge[(c * 4 + 0) * NC + tid] = S0 - Su - Sv + Qc;
                edge[(c * 4 + 1) * NC + tid] = Su - Qc;
                edge[(c * 4 + 2) * NC + tid] = Sv - Qc;
                edge[(c * 4 + 3) * NC + tid] = Qc;
                acc[c][0] = acc[c][1] = acc[c][2] = acc[c][3] = 0.f;
            }
            __syncthreads();
            // component c's edges start at the nodes [0, 8) along c and [0, 9)
            // along u and v (the edge at node n belongs to cells n - a e_u - b e_v)
            constexpr int NE = 8 * 9 * 9;
            for (int idx = tid; idx < 3 * NE; idx += K::THREADS) {
                const int c = idx / NE, r = idx - c * NE;
                const int u = c == 2 ? 0 : c + 1, v = c == 0 ? 2 : (c == 1 ? 0 : 1);
                const int nc = r % 8, nu = (r / 8) % 9, nv = r / 72;
                float sum = 0.f;
#pragma unroll
                for (int b = 0; b < 2; ++b)
#pragma unroll
                    for (int a = 0; a < 2; ++a) {
                        const int cu = nu - a, cv = nv - b;
                        if (cu < 0 || cu >= 8 || cv < 0 || cv >= 8) continue;
                        int cell3[3];
                        cell3[c] = nc;
                        cell3[u] = cu;
                        cell3[v] = cv;
                        const int cell = (cell3[2] * 8 + cell3[1]) * 8 + cell3[0];
                        sum += edge[(c * 4 + b * 2 + a) * NC + cell];
                    }
                if (sum == 0.f) continue;
                int nd[3];
                nd[c] = nc;
                nd[u] = nu;
                nd[v] = nv;
                int gx = ox + nd[0], gy = oy + nd[1], gz = oz + nd[2];
                while (gx >= g.N[0]) gx -= g.N[0];
                while (gy >= g.N[1]) gy -= g.N[1];
                while (gz >= g.N[2]) gz -= g.N[2];
                const long long node = ((long long)gz * g.N[1] + gy) * g.N[0] + gx;
                if (PCG_IN(node, g.ncells)) red_add_f32(J + c * g.ncells + node, sum);
            }
        }
        if (!more) {
            // the invalid tail sits at the end of the array: after it come only
            // chunks that are all tail or past the end
            dep::RoundPos rr = nxt;
            while (rr.t == g.n_tiles) {
                tail(rr);
                dep::seek(g, offs, chunk_tile, n, chunk, nchunks, rr.c + gridDim.x, 0xffffffffu, rr);
            }
            break;
        }
        cur = nxt;
        __syncthreads();  // lists, counters and edge values read
    }
    warp_add_u64(ctr.n_escaped, n_esc);
    warp_add_u64(ctr.n_invalid, n_inv);
}

}  // namespace
}  // namespace pcg

extern "C" pcg_status pcg_deposit_zigzag(const int32_t *grid, int32_t tile, int64_t n, const float *const *pos_prev,
                                         const float *const *pos, const float *q, double dt,
                                         const uint32_t *tile_offsets, float *J, pcg_stats *stats, void *workspace,
                                         size_t workspace_bytes, void *stream) {
    using namespace pcg;
    const bool tiled = tile_offsets != nullptr;
    if (n < 0 || n >= 0xffffffffll || grid == nullptr) return PCG_ERR_INVALID_ARG;
    for (int mu = 0; mu < 3; ++mu)
        if (grid[mu] < 3) return PCG_ERR_INVALID_ARG;
    if (!(dt > 0.0) || !(dt < 1e300)) return PCG_ERR_INVALID_ARG;
    if (tiled && tile != 8) return tile < 1 || tile > 64 ? PCG_ERR_INVALID_ARG : PCG_ERR_UNSUPPORTED;
    Geom g;
    if (!geom_from(3, grid, tiled ? tile : 1, &g)) return PCG_ERR_INVALID_ARG;
    if (J == nullptr || !aligned16(J)) return PCG_ERR_INVALID_ARG;
    ZParticles P{};
    if (n > 0) {
        if (pos_prev == nullptr || pos == nullptr || q == nullptr) return PCG_ERR_INVALID_ARG;
        for (int mu = 0; mu < 3; ++mu) {
            if (pos_prev[mu] == nullptr || pos[mu] == nullptr) return PCG_ERR_INVALID_ARG;
            P.x1[mu] = pos_prev[mu];
            P.x2[mu] = pos[mu];
        }
        P.q = q;
    }
    const long long chunk = chunk_for(n);
    const long long nchunks = (n + chunk - 1) / chunk;
    const size_t need = tiled ? align_up((size_t)nchunks * sizeof(unsigned), 256) : 0;
    if (workspace_bytes < need || (need > 0 && workspace == nullptr)) return PCG_ERR_WORKSPACE;

    cudaStream_t s = as_stream(stream);
    Counters ctr{stats ? &stats->n_escaped : nullptr, stats ? &stats->n_invalid : nullptr,
                 stats ? &stats->error_flags : nullptr};
    unsigned *chunk_tile = static_cast<unsigned *>(workspace);
    pcg_status st = launch_prep(J, g, tiled ? tile_offsets : nullptr, n, chunk, chunk_tile, ctr.flags, s);
    if (st != PCG_OK || n == 0) return st;
    const float inv_dt = (float)(1.0 / dt);
    if (!tiled) {
        const long long want = (n + 255) / 256;
        const long long cap = (long long)num_sms() * 16;
        prof::Mark mk("deposit_zigzag_flat", s);
        zigzag_flat_kernel<<<(unsigned)(want < cap ? want : cap), 256, 0, s>>>(g, P, n, inv_dt, J, ctr);
        return launch_status();
    }
    bool vec = true;
    for (int mu = 0; mu < 3; ++mu) vec = vec && aligned16(P.x1[mu]) && aligned16(P.x2[mu]);
    vec = vec && aligned16(P.q);
    const long long sms = num_sms();
    const unsigned grid_ = (unsigned)(nchunks < sms ? nchunks : sms);
    PCG_CHECK_CUDA(cudaFuncSetAttribute(zigzag_cells_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)ZzCfg::SMEM));
    prof::Mark mk("deposit_zigzag", s);
    zigzag_cells_kernel<2><<<grid_, ZzCfg::THREADS, ZzCfg::SMEM, s>>>(g, P, n, inv_dt, tile_offsets, chunk_tile,
                                                                       chunk, nchunks, J, ctr, vec);
    return launch_status();
}
