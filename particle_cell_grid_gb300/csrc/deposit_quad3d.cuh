// deposit_quad3d.cuh -- 3D quadratic (27-node B-spline) tiled current deposit
// for 8^3 tiles ("Tiled current deposit", Entity wiki, "How a tile deposit
// runs"; the shape is the second-order B-spline of the pages' deposit).
//
// The quadratic stencil of a particle is fixed by its first node (nearest node
// minus one per axis): the particles of one first node form a support group
// (Pennati & Markidis, Sec. 3.3) and add to the same 27 nodes.  A tile has KR^3
// first nodes (9^3 with a 2-cell halo), each group 27 x 3 sums: 59 K floats,
// the whole register file.  So a thread owns GX consecutive first nodes along x
// (one y, one z): the union of their stencils is (GX + 2) x 3 x 3 nodes.  With
// a 2-cell halo GX = 3: 135 sums for three groups in 243 threads (8 warps, so
// that the register file allows 255 registers a thread; 13 warps of x-pairs
// would be capped at 128 and spill), holding the tile in registers for the
// whole tile segment.
//
// One persistent CTA per SM walks the chunks b, b + grid, ... of the tile-sorted
// array in rounds of THREADS x 16 particles, loaded 8 per thread at a time
// (float4 loads per field) and placed; the first 8 of a round are loaded into
// registers during the previous round's walk, and the round is pulled into L2
// when the previous one starts.  The round is as large as the registers
// (the sums take 135) and the lists allow: the longer the lists, the fewer a
// warp's owners wait for its longest one.  A round is placed by
// rank (a shared u32 counting atomic) into per-group lists st[k][slot][rank]
// [owner] of float2 pairs, which the owners read conflict-free, one list after
// the other, each with its own compile-time x offset into the sums.  At the
// tile's end every owner stores its sums (plain stores into the free staging
// area), and after one barrier one thread per node adds the owner sums that
// meet there and issues one global reduction per component.  Shared-memory float atomics are not used: on this GPU they
// are a serial read-modify-write.
//
// Particles the fast path does not take (outside the tile's first nodes, beyond
// CAP in their list, invalid) are queued per warp and taken one per lane after
// the round's placement: invalid ones are counted, the others add their
// stencil straight to J with global reductions (escapes counted).
#pragma once

namespace pcg {
namespace dep {

template <int HALO>
struct Quad3Cfg {
    using C = TileCfg<3, 2, 8, HALO>;
    static constexpr int KR = C::KR;              // first nodes per axis
    static constexpr int KLO = C::KLO;            // lowest first node (tile-local)
    static constexpr int GX = KR % 3 == 0 ? 3 : 2;  // first nodes per owner along x
    static constexpr int NP = (KR + GX - 1) / GX; // owners per row
    static constexpr int OWN = NP * KR * KR;      // owner threads
    static constexpr int THREADS = (OWN + 31) / 32 * 32;
    static constexpr int PART = 8;                // particles per thread per load
    static constexpr int NPART = 2;               // loads per round
    static constexpr int PPT = PART * NPART;      // particles per thread per round
    static constexpr int R = THREADS * PPT;       // round size
    static constexpr int RP = THREADS * PART;     // particles per load
    static constexpr int CAP = 12;                // listed particles per group and round
    static constexpr int QCAP = PART * 32;        // queued particles per warp and load: room for all
    static constexpr int NACC = (GX + 2) * 3 * 3 * 3;  // sums per owner
    static constexpr int NN = KR + 2;             // window nodes per axis
    static constexpr size_t ST_BYTES = (size_t)3 * GX * CAP * THREADS * 8;
    static constexpr size_t SUM_BYTES = (size_t)NACC * THREADS * 4;
    static constexpr size_t AREA = ST_BYTES > SUM_BYTES ? ST_BYTES : SUM_BYTES;
    static constexpr size_t SMEM = AREA + (size_t)(THREADS / 32) * QCAP * 4 + (size_t)GX * THREADS * 4;
    static_assert(RP % 8 == 0, "a load splits into two float4 halves per thread");
};

// List a particle of tile-local first node (bx, by, bz) in [0, KR)^3 (counted
// from KLO) with offsets (tx, ty, tz): false when its list is full.
template <int HALO>
__device__ __forceinline__ bool quad_list(float2 *st, unsigned *cnt, int bx, int by, int bz, float tx, float ty,
                                          float tz, float qvx, float qvy, float qvz) {
    using K = Quad3Cfg<HALO>;
    const int bq = bx / K::GX;
    const int slot = bx - bq * K::GX;
    const int owner = (bz * K::KR + by) * K::NP + bq;
    if (!PCG_IN(owner, K::OWN)) return false;
    const unsigned r = atomicAdd(&cnt[slot * K::THREADS + owner], 1u);
    if (r >= (unsigned)K::CAP) return false;
    float2 *dst = st + ((size_t)slot * K::CAP + r) * K::THREADS + owner;
    constexpr size_t KS = (size_t)K::GX * K::CAP * K::THREADS;  // stride between the three pairs
    dst[0] = make_float2(tx, ty);
    dst[KS] = make_float2(tz, qvx);
    dst[2 * KS] = make_float2(qvy, qvz);
    return true;
}

// The general path of a queued particle of the tile at (ox, oy, oz): 1 invalid
// (skipped), 2 escaped to J, 0 listed or added to J (outside the tile's first
// nodes but inside the window, or its list full).
template <int HALO>
__device__ __forceinline__ int quad_slow(const Geom &g, float *J, float2 *st, unsigned *cnt, int ox, int oy, int oz,
                                         float x, float y, float z, float qvx, float qvy, float qvz) {
    using K = Quad3Cfg<HALO>;
    using C = typename K::C;
    if (!in_domain<3>(g, x, y, z)) return 1;
    float tx, ty, tz;
    const int fx = first_node<2>(x, tx);
    const int fy = first_node<2>(y, ty);
    const int fz = first_node<2>(z, tz);
    const int lx = local_index<3, 8, HALO>(fx, ox, g.N[0]);
    const int ly = local_index<3, 8, HALO>(fy, oy, g.N[1]);
    const int lz = local_index<3, 8, HALO>(fz, oz, g.N[2]);
    const bool home = (lx >= C::KLO) & (lx < C::KHI) & (ly >= C::KLO) & (ly < C::KHI) & (lz >= C::KLO) &
                      (lz < C::KHI);
    if (home && quad_list<HALO>(st, cnt, lx - C::KLO, ly - C::KLO, lz - C::KLO, tx, ty, tz, qvx, qvy, qvz))
        return 0;
    const bool fits = (lx >= -HALO) & (lx + 2 < 8 + HALO) & (ly >= -HALO) & (ly + 2 < 8 + HALO) &
                      (lz >= -HALO) & (lz + 2 < 8 + HALO);
    deposit_global<3, 2>(g, J, x, y, z, qvx, qvy, qvz);
    return fits ? 0 : 2;
}

// One owner's list of slot P: m particles, added to the sums of the owner's
// union window at x offset P.
template <int HALO, int P>
__device__ __forceinline__ void quad_walk(const float2 *st, int owner, unsigned m,
                                          float (&acc)[Quad3Cfg<HALO>::GX + 2][3][3][3]) {
    using K = Quad3Cfg<HALO>;
    constexpr size_t KS = (size_t)K::GX * K::CAP * K::THREADS;
    const float2 *src = st + (size_t)P * K::CAP * K::THREADS + owner;
    for (unsigned r = 0; r < m; ++r) {
        const float2 a = src[(size_t)r * K::THREADS];
        const float2 b = src[KS + (size_t)r * K::THREADS];
        const float2 c = src[2 * KS + (size_t)r * K::THREADS];
        float wx[3], wy[3], wz[3];
        weights_from<2>(a.x, wx);
        weights_from<2>(a.y, wy);
        weights_from<2>(b.x, wz);
        const float qv[3] = {b.y, c.x, c.y};
#pragma unroll
        for (int k = 0; k < 3; ++k)
#pragma unroll
            for (int j = 0; j < 3; ++j) {
                const float wyz = wy[j] * wz[k];
#pragma unroll
                for (int i = 0; i < 3; ++i) {
                    const float W = wyz * wx[i];
#pragma unroll
                    for (int comp = 0; comp < 3; ++comp)
                        acc[P + i][j][k][comp] = fmaf(qv[comp], W, acc[P + i][j][k][comp]);
                }
            }
    }
}

template <int HALO>
__global__ void __launch_bounds__(Quad3Cfg<HALO>::THREADS, 1)
    deposit_quad3d_kernel(Geom g, Particles P, long long n, const uint32_t *__restrict__ offs,
                          const unsigned *__restrict__ chunk_tile, long long chunk, long long nchunks,
                          float *__restrict__ J, Counters ctr, bool vec) {
    using K = Quad3Cfg<HALO>;
    constexpr int THREADS = K::THREADS, KR = K::KR, NP = K::NP, CAP = K::CAP, QCAP = K::QCAP, GX = K::GX;
    extern __shared__ __align__(16) unsigned char dsm[];
    float2 *st = reinterpret_cast<float2 *>(dsm);                           // lists; at a tile end: sums
    int *qbuf = reinterpret_cast<int *>(dsm + K::AREA);                      // [warps][QCAP]
    unsigned *cnt = reinterpret_cast<unsigned *>(qbuf + (THREADS / 32) * QCAP);  // [GX][THREADS]

    const int tid = threadIdx.x, lane = tid & 31;
    int *wq = qbuf + (tid >> 5) * QCAP;
    unsigned n_esc = 0, n_inv = 0;
    const bool owner = tid < K::OWN;
#pragma unroll
    for (int sl = 0; sl < GX; ++sl) cnt[sl * THREADS + tid] = 0;
    float acc[GX + 2][3][3][3];
#pragma unroll
    for (int i = 0; i < GX + 2; ++i)
#pragma unroll
        for (int j = 0; j < 3; ++j)
#pragma unroll
            for (int k = 0; k < 3; ++k) acc[i][j][k][0] = acc[i][j][k][1] = acc[i][j][k][2] = 0.f;

    float X[8], Y[8], Z[8], VX[8], VY[8], VZ[8], Q[8];
    // part `part` of the round at r: this thread's 8 particles
    auto load_part = [&](const RoundPos &r, int part) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const long long b = r.rb + (long long)part * K::RP + h * (K::RP / 2) + 4 * tid;
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
    auto tail = [&](const RoundPos &r) {
        for (long long p = r.lo + tid; p < r.hi; p += THREADS) {
            const float x = P.x[p], y = P.y[p], z = P.z[p];
            if (!in_domain<3>(g, x, y, z)) {
                ++n_inv;
                continue;
            }
            const float q = P.q[p];
            deposit_global<3, 2>(g, J, x, y, z, q * P.vx[p], q * P.vy[p], q * P.vz[p]);
        }
    };

    RoundPos cur;
    seek(g, offs, chunk_tile, n, chunk, nchunks, blockIdx.x, 0xffffffffu, cur);
    while (cur.t == g.n_tiles) {  // a chunk that holds only invalid-tail particles
        tail(cur);
        seek(g, offs, chunk_tile, n, chunk, nchunks, cur.c + gridDim.x, 0xffffffffu, cur);
    }
    if (cur.t > g.n_tiles) {
        warp_add_u64(ctr.n_invalid, n_inv);
        return;
    }
    load_part(cur, 0);
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
        // the next round's position; its particles are pulled into L2 while
        // this round is placed and walked
        RoundPos nxt = cur;
        nxt.rb = cur.rb + K::R;
        if (nxt.rb >= cur.hi) seek(g, offs, chunk_tile, n, chunk, nchunks, cur.c, cur.t + 1, nxt);
        const bool tile_ends = nxt.t != cur.t || nxt.c != cur.c;
        const bool more = nxt.t < g.n_tiles;
        if (tid == 0 && vec && more) {
            long long e = nxt.rb + K::R;
            if (e > (nxt.hi & ~3ll)) e = nxt.hi & ~3ll;
            if (e > nxt.rb) {
                const unsigned bytes = (unsigned)((e - nxt.rb) * 4);
                prefetch_l2_bulk(P.x + nxt.rb, bytes);
                prefetch_l2_bulk(P.y + nxt.rb, bytes);
                prefetch_l2_bulk(P.z + nxt.rb, bytes);
                prefetch_l2_bulk(P.vx + nxt.rb, bytes);
                prefetch_l2_bulk(P.vy + nxt.rb, bytes);
                prefetch_l2_bulk(P.vz + nxt.rb, bytes);
                prefetch_l2_bulk(P.q + nxt.rb, bytes);
            }
        }
        // ---- place the round: fast path for the tile's own first nodes ----
#pragma unroll 1
        for (int part = 0; part < K::NPART; ++part) {
        if (part > 0) load_part(cur, part);  // part 0 was loaded during the last walk
        int qn = 0;  // particles this warp has queued from this load (warp-uniform)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const long long p = cur.rb + (long long)part * K::RP + (j >> 2) * (K::RP / 2) + 4 * tid + (j & 3);
            const bool live = p >= cur.lo && p < cur.hi;
            const float x = X[j], y = Y[j], z = Z[j];
            const float qq = Q[j];
            const float qvx = qq * VX[j], qvy = qq * VY[j], qvz = qq * VZ[j];
            float fx_, fy_, fz_;
            const int fx = first_node<2>(x, fx_);
            const int fy = first_node<2>(y, fy_);
            const int fz = first_node<2>(z, fz_);
            // in the domain (a NaN fails too) and a first node of the tile,
            // counted from KLO (no periodic wrap: the particle is in the tile)
            const unsigned dx = (unsigned)(fx - ox - K::KLO), dy = (unsigned)(fy - oy - K::KLO),
                           dz = (unsigned)(fz - oz - K::KLO);
            bool slow = live;
            if (live && in_domain<3>(g, x, y, z) && (dx < (unsigned)KR) & (dy < (unsigned)KR) &
                            (dz < (unsigned)KR))
                slow = !quad_list<HALO>(st, cnt, (int)dx, (int)dy, (int)dz, fx_, fy_, fz_, qvx, qvy, qvz);
            const unsigned m = __ballot_sync(0xffffffffu, slow);
            if (m) {  // warp-uniform
                const int at = qn + __popc(m & lanes_below);
                if (slow && PCG_IN(at, QCAP)) wq[at] = (int)(p - cur.rb);
                qn += __popc(m);
            }
        }
        // the warp's queue, one particle per lane (re-read: it sits in L1/L2)
        __syncwarp();
        for (int e = lane; e < qn; e += 32) {
            const long long pp = cur.rb + wq[e];
            if (!PCG_IN(pp, n)) continue;
            const float q = P.q[pp];
            slow_count(quad_slow<HALO>(g, J, st, cnt, ox, oy, oz, P.x[pp], P.y[pp], P.z[pp], q * P.vx[pp],
                                       q * P.vy[pp], q * P.vz[pp]));
        }
        __syncwarp();
        }
        // the next round's first load goes out now: its latency hides behind
        // the walk, which leaves room in the registers for it
        if (more) load_part(nxt, 0);
        __syncthreads();  // the round is listed

        // ---- every owner adds its lists in registers ----
        if (owner) {
            unsigned m[GX];
#pragma unroll
            for (int sl = 0; sl < GX; ++sl) {
                m[sl] = min(cnt[sl * THREADS + tid], (unsigned)CAP);
                cnt[sl * THREADS + tid] = 0;
            }
            quad_walk<HALO, 0>(st, tid, m[0], acc);
            quad_walk<HALO, 1>(st, tid, m[1], acc);
            if constexpr (GX == 3) quad_walk<HALO, 2>(st, tid, m[2], acc);
        }
        if (tile_ends) {
            // every owner's sums to the free staging area, then one thread per
            // node adds the owner sums that meet there and reduces them into J
            float *sums = reinterpret_cast<float *>(st);  // [NACC][THREADS]
            __syncthreads();  // every list has been read
            if (owner) {
#pragma unroll
                for (int i = 0; i < GX + 2; ++i)
#pragma unroll
                    for (int j = 0; j < 3; ++j)
#pragma unroll
                        for (int k = 0; k < 3; ++k)
#pragma unroll
                            for (int comp = 0; comp < 3; ++comp) {
                                sums[(((i * 3 + j) * 3 + k) * 3 + comp) * THREADS + tid] = acc[i][j][k][comp];
                                acc[i][j][k][comp] = 0.f;
                            }
            }
            __syncthreads();
            constexpr int NN = K::NN;
            for (int nd = tid; nd < NN * NN * NN; nd += THREADS) {
                const int nx = nd % NN, ny = (nd / NN) % NN, nz = nd / (NN * NN);
                float s[3] = {0.f, 0.f, 0.f};
                // owners whose union [GX bp, GX bp + GX + 1] x [by, by + 2] x
                // [bz, bz + 2] holds the node
                const int bp0 = nx > GX + 1 ? (nx - 2) / GX : 0, bp1 = min(nx / GX, NP - 1);
                for (int dz = 0; dz < 3; ++dz) {
                    const int bz = nz - dz;
                    if (bz < 0 || bz >= KR) continue;
                    for (int dy = 0; dy < 3; ++dy) {
                        const int by = ny - dy;
                        if (by < 0 || by >= KR) continue;
                        for (int bp = bp0; bp <= bp1; ++bp) {
                            const int ow = (bz * KR + by) * NP + bp;
                            const int v = (((nx - GX * bp) * 3 + dy) * 3 + dz) * 3;
#pragma unroll
                            for (int comp = 0; comp < 3; ++comp) s[comp] += sums[(v + comp) * THREADS + ow];
                        }
                    }
                }
                const int gx = wrap_index(ox + K::KLO + nx, g.N[0]);
                const int gy = wrap_index(oy + K::KLO + ny, g.N[1]);
                const int gz = wrap_index(oz + K::KLO + nz, g.N[2]);
                const long long node = ((long long)gz * g.N[1] + gy) * g.N[0] + gx;
                if (!PCG_IN(node, g.ncells)) continue;
#pragma unroll
                for (int comp = 0; comp < 3; ++comp)
                    if (s[comp] != 0.f) red_add_f32(J + comp * g.ncells + node, s[comp]);
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
        __syncthreads();  // lists, counters and sums read
    }
    warp_add_u64(ctr.n_escaped, n_esc);
    warp_add_u64(ctr.n_invalid, n_inv);
}

template <int HALO>
pcg_status launch_quad3d(const Geom &g, long long n, const Particles &P, const uint32_t *offs, float *J,
                         const Counters &ctr, const unsigned *chunk_tile, long long chunk, cudaStream_t s) {
    using K = Quad3Cfg<HALO>;
    const long long nchunks = (n + chunk - 1) / chunk;
    if (nchunks == 0) return PCG_OK;
    const bool vec = aligned16(P.x) && aligned16(P.y) && aligned16(P.z) && aligned16(P.vx) &&
                     aligned16(P.vy) && aligned16(P.vz) && aligned16(P.q);
    const long long sms = num_sms();
    const unsigned grid = (unsigned)(nchunks < sms ? nchunks : sms);
    PCG_CHECK_CUDA(cudaFuncSetAttribute(deposit_quad3d_kernel<HALO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)K::SMEM));
    prof::Mark mk("deposit_tiled", s);
    deposit_quad3d_kernel<HALO><<<grid, K::THREADS, K::SMEM, s>>>(g, P, n, offs, chunk_tile, chunk, nchunks, J,
                                                                   ctr, vec);
    return launch_status();
}

}  // namespace dep
}  // namespace pcg
