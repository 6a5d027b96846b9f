/*
 * pcg.h -- C ABI of the GB300 (sm_103a) particle-to-grid deposit library.
 *
 * One shared library, libpcg.so.  Every entry point:
 *   - takes plain pointers and sizes (no framework types);
 *   - unless stated otherwise, data pointers are DEVICE pointers owned by the
 *     caller, and "const T* const* name" parameters are HOST arrays holding
 *     device pointers (one per axis / component / payload field);
 *   - enqueues its kernels on `stream` (a cudaStream_t passed as void*; NULL
 *     selects the legacy default stream) and returns without synchronising;
 *   - validates its arguments on the host before launching anything and
 *     returns a pcg_status; on any error nothing is enqueued;
 *   - OVERWRITES its outputs (never accumulates into them), except `stats`,
 *     whose counters are added to;
 *   - never allocates device memory: scratch space is a caller-provided
 *     `workspace` whose size is returned by the matching *_workspace_size query
 *     (a NULL workspace with size 0 is fine where that query returns 0).
 *
 * Conventions.  Positions are in cell units, x in [0, N) per axis; node g sits at
 * integer coordinates and cell i is [i, i+1).  Grids are periodic on every
 * axis.  Arrays over nodes or cells are flattened with x fastest:
 * index = (z * Ny + y) * Nx + x.  Particle arrays are structure-of-arrays fp32.
 * A particle with a coordinate outside [0, N) or NaN is "invalid": it is skipped
 * and counted in stats->n_invalid.
 */
#ifndef PCG_H
#define PCG_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PCG_API __attribute__((visibility("default")))
#else
#define PCG_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pcg_status {
    PCG_OK = 0,
    PCG_ERR_INVALID_ARG = 1, /* null pointer, bad size, unsupported value   */
    PCG_ERR_WORKSPACE = 2,   /* workspace smaller than the size query says  */
    PCG_ERR_UNSUPPORTED = 3, /* valid request without a compiled kernel     */
    PCG_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed        */
    PCG_ERR_TIMEOUT = 5,     /* reserved: a bounded device-side wait gave up */
    PCG_ERR_DOMAIN = 6       /* data-dependent anomaly reported in stats    */
} pcg_status;

/* Device-resident counters, caller-owned; every call ADDS to them.  Zero the
 * struct before the calls whose anomalies you want to count, copy it to the
 * host after synchronising the stream, and map it with pcg_stats_check(). */
typedef struct pcg_stats {
    unsigned long long n_escaped; /* particles deposited through the escape valve */
    unsigned long long n_invalid; /* particles skipped: position outside [0, N) or NaN */
    unsigned int error_flags;     /* bit set of PCG_FLAG_* */
    unsigned int reserved;
} pcg_stats;

#define PCG_FLAG_BAD_LAYOUT 1u /* tile_offsets / cell_offsets not monotone or out of range */
#define PCG_FLAG_CELL_MISMATCH 2u /* mass matrix: a particle not inside the cell it is listed under */
#define PCG_FLAG_TIMEOUT 4u       /* a bounded wait for an asynchronous copy or a tensor-core result
                                     gave up; the call's output is invalid */

/* Index checks.  The library built with -DPCG_CHECKED (the checked build)
 * tests the data-dependent indices of its kernels (from positions, offsets,
 * counts and ranks) before each access they guard; a failed test skips the
 * access and adds one to a device counter (no trap, no assert).  This call
 * synchronises the device, stores the failures counted since the previous call
 * in *failures (HOST) and resets the count; *checked_build (HOST, may be NULL)
 * is set to 1 in the checked build, else 0 (and *failures to 0).
 * PCG_ERR_INVALID_ARG for a NULL failures pointer. */
PCG_API pcg_status pcg_bounds_check_failures(uint64_t *failures, int32_t *checked_build);

/* Library version (major * 10000 + minor * 100 + patch). */
PCG_API int pcg_version(void);

/* Static, NUL-terminated description of a status code. */
PCG_API const char *pcg_status_string(int status);

/* Map a HOST copy of a pcg_stats to PCG_OK or PCG_ERR_DOMAIN (any invalid
 * particle or error flag).  Escapes are normal and do not count as errors. */
PCG_API pcg_status pcg_stats_check(const pcg_stats *host_stats);

/* -------------------------------------------------------------------------
 * 1D windowed cloud-in-cell histogram and its loss.
 * Defined by "03. Compaction and scatter-add" (WEANJ examples), sections
 * "The problem" and "Code" (the loop over t = 1..T with the window test, the
 * taper and the two scatter-adds), and the JAX helpers minimg / taper on the
 * same page.
 *
 * For t = 1..nsteps: c = t/nsteps; x = wrap(x0 + v*(t*dt)) in [0,1);
 * d = x - c - round(d) (periodic minimum image, ties to even); if |d| < halfwidth
 * the particle adds w = (1 - |d|/halfwidth)^2 times the linear CIC weights of
 * g = x*nbins - 1/2 to bins floor(g) mod nbins and floor(g)+1 mod nbins.
 * loss = sum_b (H_b - target_b)^2.
 *
 * The window test, g and floor(g) are evaluated in fp64 with individually
 * rounded operations (no fused multiply-add); the deposits are added in fp32
 * and the loss is accumulated in fp64 from the fp32 histogram.
 *
 *   x0, v    device float[n]: initial positions on [0,1) (any finite value is
 *            wrapped) and velocities.
 *   target   device float[nbins].
 *   H        device float[nbins], output (overwritten).
 *   loss     device double[1], output (overwritten).
 *   n >= 0; 1 <= nbins <= 16384; nsteps >= 1; 0 < halfwidth; dt finite.
 * Up to 16384 particles: one launch of one 8-CTA thread-block cluster.  Above:
 * a memset of H, one full-grid launch and a one-CTA loss launch.  No
 * workspace.  The order of the fp32 additions into H is unspecified.
 */
PCG_API pcg_status pcg_deposit_cic1d(const float *x0, const float *v, int64_t n, const float *target,
                             int32_t nbins, int32_t nsteps, double dt, double halfwidth,
                             float *H, double *loss, void *stream);

/* -------------------------------------------------------------------------
 * Gradient of the 1D windowed CIC loss with respect to the initial positions.
 * Defined by "03. Compaction and scatter-add" (WEANJ examples), section "The
 * problem" (dL/dx0 of the loss above) and section "Code" (the reverse pass is
 * seeded with dL/dH = 2 (H - target)).  The wrap, the window test and floor(g)
 * are piecewise constant and contribute no derivative, so every selected
 * (particle, step) pair adds
 *   G[b0] (w' (1 - f) - w nbins) + G[b1] (w' f + w nbins),
 *   G = 2 (H - target),  w' = -2 (1 - |d|/h) sign(d) / h  (sign(0) = 0),
 * to dx0 of its particle, b0/b1 and f the CIC bins and fraction above.
 *
 * Runs the forward pass of pcg_deposit_cic1d (same arguments, same H and
 * loss), then the gradient, which reads H from the forward.
 *   dx0      device double[n], output (overwritten; zero for particles never
 *            selected).  May be NULL when n == 0.
 * The selection is the forward's fp64 test, so both passes select the same
 * pairs; G and the sum are in fp64 (pairs of one particle are added in an
 * unspecified order).  One launch more than the forward.
 */
PCG_API pcg_status pcg_deposit_cic1d_grad(const float *x0, const float *v, int64_t n, const float *target,
                                  int32_t nbins, int32_t nsteps, double dt, double halfwidth,
                                  float *H, double *loss, double *dx0, void *stream);

/* -------------------------------------------------------------------------
 * Tile counting sort.
 * Defined by "Tiled current deposit" (Entity wiki), section "The tile-based
 * spatial sort" (tile counts ntiles = ceil(N / T) per axis, a per-particle tile
 * key, invalid particles in a sentinel bin after the last tile, the
 * tile_offsets prefix sum, SoA members physically permuted into tile order)
 * and section "How a tile deposit runs" (tile t owns
 * [tile_offsets[t], tile_offsets[t+1])).  With tile = 1 the sort orders
 * particles by cell, the order the mass-matrix assembly assumes (Pennati &
 * Markidis, Sec. 3.1).
 *
 * key of a particle = index of the tile holding cell floor(key_pos), x fastest;
 * n_tiles = prod_mu ceil(grid[mu] / tile).  Invalid key positions go to the
 * sentinel bin n_tiles.
 *
 *   dim        2 or 3.  grid: HOST int32[dim], each in [1, 2^20], and the total
 *              node count below 2^31.
 *   tile       1..64.  n_tiles + 1 must stay below 2^31.
 *   n          number of particles, 0 <= n < 2^32 - 1.
 *   key_pos    HOST array of dim device float[n]: positions defining the key
 *              (for example the sort-time / previous positions).
 *   n_payload  1..16 arrays of 4-byte elements (fp32, int32 or uint32 bits).
 *   payload_in / payload_out   HOST arrays of n_payload device pointers to n
 *              elements each; payload_out[k] receives payload_in[k] permuted
 *              into tile order.  Outputs must not overlap any input.  A
 *              key_pos array may also appear among payload_in.
 *   tile_offsets  device uint32[n_tiles + 1], output: tile t holds slots
 *              [tile_offsets[t], tile_offsets[t+1]); invalid particles fill
 *              [tile_offsets[n_tiles], n).  Order inside a tile is unspecified.
 *   stats      device pcg_stats or NULL; n_invalid counts the sentinel bin.
 *   workspace  device memory of at least pcg_tile_sort_workspace_size() bytes
 *              (same dim, grid, tile, n and n_payload), 256-byte aligned;
 *              contents on entry are irrelevant.  When the permuted payload
 *              does not fit in L2 the sort runs as two partition passes and the
 *              workspace also holds the intermediate arrays, about
 *              4 * (n_payload + 1) * n bytes.
 * Launches: 4 while the output fits in L2 (count, column scan, scan,
 * scatter), 6-7 otherwise (count, scan, bucket set-up, two partition passes).
 */
PCG_API pcg_status pcg_tile_sort_workspace_size(int32_t dim, const int32_t *grid, int32_t tile, int64_t n,
                                        int32_t n_payload, size_t *bytes);
PCG_API pcg_status pcg_tile_sort(int32_t dim, const int32_t *grid, int32_t tile, int64_t n,
                         const float *const *key_pos, int32_t n_payload,
                         const void *const *payload_in, void *const *payload_out,
                         uint32_t *tile_offsets, pcg_stats *stats, void *workspace,
                         size_t workspace_bytes, void *stream);

/* -------------------------------------------------------------------------
 * Current deposit J^c_g = sum_p q_p v^c_p W(x_p - x_g), c in {x, y, z}.
 * Defined by the tensor-product B-spline shape of Pennati & Markidis, Sec. 2.3,
 * Eq. (12) (order 1 = cloud-in-cell, 2 nodes per axis; order 2 = quadratic,
 * nodes {j-1, j, j+1} when the fractional coordinate is below 1/2, else
 * {j, j+1, j+2}), deposited as in "Tiled current deposit" (Entity wiki),
 * sections "How a tile deposit runs" (one team per tile, a haloed
 * (T + 2*HALO)^D x 3 scratch tile, the fit test, a single flush per scratch
 * cell), "Halo sizing" (HALO = stencil reach + drift allowance) and "Correctness
 * is independent of the halo" (a particle whose stencil leaves the scratch
 * window is deposited whole into J through global atomics).
 *
 *   dim        2 or 3 (in 2D the stencil is 2D and vel[2] deposits Jz).
 *   grid       HOST int32[dim], each >= 1.
 *   order      1 or 2.
 *   tile       4 or 8 (the tiled kernels compiled in); ignored when
 *              tile_offsets is NULL.
 *   halo       0, 1 or 2 cells per side; correctness never depends on it.
 *   block      threads per CTA: 0 = automatic, else 128, 256 or 512.
 *   n          number of particles.
 *   pos        HOST array of dim device float[n]: deposit positions.
 *   vel        HOST array of 3 device float[n].
 *   q          device float[n], charges.
 *   tile_offsets  NULL: flat path, one thread per particle straight to global
 *              atomics.  Else device uint32[n_tiles + 1] from pcg_tile_sort
 *              with the same dim, grid and tile: particles of tile t are
 *              [tile_offsets[t], tile_offsets[t+1]) and may have moved since the
 *              sort (drift); slots [tile_offsets[n_tiles], n) are deposited by
 *              the flat path (the tail pass).
 *   J          device float[3][ncells], output (overwritten).
 *   stats      device pcg_stats or NULL: n_escaped, n_invalid, error_flags.
 *   workspace  device memory of pcg_deposit_current_workspace_size() bytes.
 * Launches: 2 (flat) or 3 (tiled).
 */
PCG_API pcg_status pcg_deposit_current_workspace_size(int32_t dim, const int32_t *grid, int32_t tile,
                                              int64_t n, size_t *bytes);
PCG_API pcg_status pcg_deposit_current(int32_t dim, const int32_t *grid, int32_t order, int32_t tile,
                               int32_t halo, int32_t block, int64_t n, const float *const *pos,
                               const float *const *vel, const float *q,
                               const uint32_t *tile_offsets, float *J, pcg_stats *stats,
                               void *workspace, size_t workspace_bytes, void *stream);

/* -------------------------------------------------------------------------
 * pcg_deposit_current without a workspace: for callers that cannot allocate
 * device memory (a host callback, a plugin that is handed only its input and
 * output buffers, an application whose memory pool forbids run-time
 * allocation).  The pages have no counterpart: this is a packaging variant of
 * pcg_deposit_current, which it calls with its own scratch.
 *
 * Arguments, outputs, stats and errors are those of pcg_deposit_current minus
 * the workspace.  The tiled path's scratch (one 32-bit entry per chunk of
 * particles) is a fixed 256 KB device array inside the library, held on every
 * GPU that loads it until the process exits; so this entry point accepts at
 * most 65536 chunks when tile_offsets is given, and returns PCG_ERR_WORKSPACE
 * above that (before launching anything).  Chunks hold up to 16384 particles
 * (up to 65536 for the 3D quadratic deposit on 8^3 tiles), so every
 * n <= 2^30 fits.
 * The flat path (tile_offsets NULL) uses no scratch and has no such limit.
 *
 * Arguments are checked exactly as pcg_deposit_current checks them, before the
 * size limit and before any CUDA call.
 *
 * It allocates nothing.  The first call made on a device looks up the array's
 * device address (cudaGetSymbolAddress) with that device current; make that
 * first call before any stream capture.  The address is kept per device for the
 * life of the process, which assumes the device's primary context (the one the
 * CUDA runtime uses) is never reset: after cudaDeviceReset the kept address is
 * stale, so do not call this entry point in a process that has reset the device.  Every call shares the one array and
 * each call rewrites every entry it reads, so nothing needs clearing between
 * calls; but calls whose kernels overlap on the GPU (different streams, no
 * ordering between them) race on the array and must not be issued.
 */
PCG_API pcg_status pcg_deposit_current_noalloc(int32_t dim, const int32_t *grid, int32_t order,
                                               int32_t tile, int32_t halo, int32_t block, int64_t n,
                                               const float *const *pos, const float *const *vel,
                                               const float *q, const uint32_t *tile_offsets, float *J,
                                               pcg_stats *stats, void *stream);

/* -------------------------------------------------------------------------
 * Charge-conserving zigzag current deposit, 3D.
 * Named by "Tiled current deposit" (Entity wiki), section "Halo sizing" (the
 * O == 0 zigzag deposit, writing at most 2 cells above min(i, i_prev)) and run
 * the way "How a tile deposit runs" and "Correctness is independent of the
 * halo" describe; the scheme is Umeda, Omura, Tominaga & Matsumoto, Comput.
 * Phys. Commun. 156 (2003) 73.  Per axis, cells i1 = floor(x1), i2 = floor(x2):
 *   xr = min(min(i1,i2) + 1, max(max(i1,i2), (x1 + x2)/2)),
 *   D1 = xr - x1, D2 = x2 - xr, F_s = q D_s / dt,
 *   W1 = (x1 + xr)/2 - i1, W2 = (xr + x2)/2 - i2;
 * segment s adds F_s^c (w_a(W_s^u) w_b(W_s^v) + (a == b ? 1 : -1) D_s^u D_s^v / 12)
 * to the c-edge starting at its cell + a e_u + b e_v (u, v the transverse axes,
 * w_0(W) = 1 - W, w_1(W) = W).  The D D / 12 term (the weight averaged along
 * the straight segment) makes (rho(x2) - rho(x1)) / dt + div J = 0 exact for
 * the CIC charge rho; it is zero when a segment moves along at most two axes.
 *
 * Output layout: J float[3][Nz][Ny][Nx]; J[c] at node (i, j, k) is the
 * c-current on the edge from that node towards +e_c.  Periodic on every axis.
 *
 *   grid       HOST int32[3], each in [3, 2^20].
 *   tile       8 (with tile_offsets); ignored when tile_offsets is NULL.
 *   n          number of particles, 0 <= n < 2^32 - 1.
 *   pos_prev, pos  HOST arrays of 3 device float[n]: the positions before and
 *              after the move, both in [0, N).  The move is the periodic
 *              minimum image of the cell change, so a particle may cross the
 *              periodic boundary.
 *   q          device float[n]; dt > 0.
 *   tile_offsets  NULL (flat: every particle through global reductions) or the
 *              output of pcg_tile_sort with tile 8 keyed on pos_prev and with
 *              pos_prev, pos and q among its payload.  Particles whose 3x3x3
 *              footprint leaves their tile's window (tile + 2 cells per side)
 *              take the escape valve (stats->n_escaped).
 *   J          device float[3 * ncells], 16-byte aligned, output (overwritten).
 *   stats      device pcg_stats or NULL: n_invalid counts particles with a
 *              coordinate outside [0, N) or NaN, or whose cell changes by more
 *              than one along an axis (beyond the scheme's CFL limit); they are
 *              skipped.
 *   workspace  pcg_deposit_current_workspace_size(3, grid, 8, n) bytes when
 *              tiled, else may be NULL.
 * Launches: 2 (zero J + chunk map, deposit).  Errors: PCG_ERR_INVALID_ARG for
 * bad sizes, pointers or dt; PCG_ERR_UNSUPPORTED for a tile other than 8.
 */
PCG_API pcg_status pcg_deposit_zigzag(const int32_t *grid, int32_t tile, int64_t n,
                                      const float *const *pos_prev, const float *const *pos,
                                      const float *q, double dt, const uint32_t *tile_offsets,
                                      float *J, pcg_stats *stats, void *workspace,
                                      size_t workspace_bytes, void *stream);

/* -------------------------------------------------------------------------
 * ECSIM block mass matrix with first-order (CIC) or second-order (TSC)
 * B-splines.
 * Defined by Pennati & Markidis, Sec. 2.1, Eqs. (4)-(6):
 *   M^{ij}_{g g'} = sum_p s_p^{ij} W_pg W_pg',  s_p = w_p alpha_p,
 *   alpha_p = (I - C(omega_p) + omega_p omega_p^T) / (1 + |omega_p|^2),
 *   C(omega) u = omega x u,
 * with every constant prefactor absorbed into w (sigma = 1), assembled cell by
 * cell as in Sec. 3.1-3.2, Eqs. (14)-(20) (A = W S^{ij}, B = W^T over batches of
 * particles, accumulated in place), and stored by stencil offset as in Sec. 3.4
 * with all 27 offsets kept.
 *
 * Output layout, order 1: M[g][o][i][j], g the row node,
 * o = (dz+1)*9 + (dy+1)*3 + (dx+1) the offset of the column node
 * g' = g + (dx, dy, dz) (periodic), i, j the tensor component;
 * float[ncells][27][3][3].
 * Order 2 (Sec. 2.3: per axis nodes j-1..j+1 when the fractional part is
 * < 1/2, else j..j+2; Sec. 3.3-3.4: up to 8 support groups per cell,
 * displacements in {-2..2}^3): o = (dz+2)*25 + (dy+2)*5 + (dx+2);
 * float[ncells][125][3][3], every offset kept.
 *
 *   grid       HOST int32[3], each >= 3 for order 1 and >= 5 for order 2 (so
 *              that the offsets are distinct nodes).
 *   order      1 or 2.
 *   precision  0 = TF32 tensor cores (tcgen05.mma kind::tf32, fp32 accumulate
 *              in tensor memory); 1 = BF16 tensor cores (kind::f16); 2 = fp32
 *              CUDA cores (no tensor cores; the A/B baseline).  Both orders run
 *              on all three.
 *   n          number of particles.
 *   pos        HOST array of 3 device float[n]; w device float[n] (q^2/m);
 *   omega      HOST array of 3 device float[n] (omega = beta_s B(x_p) / c).
 *   cell_offsets  device uint32[ncells + 1] from pcg_tile_sort with tile = 1:
 *              the particles listed under cell c are [cell_offsets[c],
 *              cell_offsets[c+1]).  A particle whose position is not inside the
 *              cell it is listed under is still deposited correctly (through
 *              global atomics) and flagged with PCG_FLAG_CELL_MISMATCH.  Slots
 *              [cell_offsets[ncells], n) (the sort's sentinel bin, or particles
 *              appended after the sort) are deposited through global atomics
 *              (the tail pass).
 *   M          device float[ncells * 243] (order 1) or [ncells * 1125]
 *              (order 2), 16-byte aligned, output (overwritten).
 *   stats      device pcg_stats or NULL: n_invalid counts the particles skipped
 *              for a coordinate outside [0, N) or NaN, wherever they are listed
 *              (a pcg_tile_sort into the same stats has counted those of its
 *              sentinel bin already).
 *   workspace  pcg_assemble_mass_matrix_workspace_size() bytes (currently 0).
 */
PCG_API pcg_status pcg_assemble_mass_matrix_workspace_size(const int32_t *grid, int64_t n, size_t *bytes);
PCG_API pcg_status pcg_assemble_mass_matrix(const int32_t *grid, int32_t order, int32_t precision,
                                    int64_t n, const float *const *pos, const float *w,
                                    const float *const *omega, const uint32_t *cell_offsets,
                                    float *M, pcg_stats *stats, void *workspace,
                                    size_t workspace_bytes, void *stream);

/* -------------------------------------------------------------------------
 * Scalar mass matrix with first-order (CIC) B-splines.
 * Defined by Pennati & Markidis, Sec. 2.1 after Eq. (6): the scalar case
 * s_p^{ij} = q_p delta^{ij} (e.g. the MPM mass matrix), one component per node
 * pair:  M_{g g'} = sum_p w_p W_pg W_pg'  (sigma = 1), assembled and stored as
 * for pcg_assemble_mass_matrix (Sec. 3.1-3.4) with NC = 1.
 *
 * Output layout: M[g][o], o as above; float[ncells][27].
 *   grid, order, precision, n, pos, cell_offsets, stats: as for
 *              pcg_assemble_mass_matrix (precision 0 = TF32 and 1 = BF16 tensor
 *              cores, 2 = fp32 CUDA cores).
 *   w          device float[n] (the per-particle coefficient, e.g. the mass).
 *   M          device float[ncells * 27], 16-byte aligned, output (overwritten).
 * Launches: 2 (zero M + assembly).  No workspace.
 */
PCG_API pcg_status pcg_assemble_mass_matrix_scalar(const int32_t *grid, int32_t order, int32_t precision,
                                                   int64_t n, const float *const *pos, const float *w,
                                                   const uint32_t *cell_offsets, float *M,
                                                   pcg_stats *stats, void *stream);

/* -------------------------------------------------------------------------
 * Kernel timing (tracing aid; no counterpart in the method).
 * While enabled, every kernel the library launches is bracketed by two CUDA
 * events recorded on its launch stream.  pcg_profile_collect() waits for the
 * recorded events, aggregates them by kernel name and forgets them:
 *   names     HOST char[max_entries][64], NUL-terminated kernel names;
 *   launches  HOST int64[max_entries], total_ms HOST double[max_entries];
 *   n_entries HOST int32: number of distinct kernels seen (may exceed
 *             max_entries; only the first max_entries are written).
 * Returns PCG_ERR_CUDA if some event could not be timed.  Thread-safe; the
 * state is process-wide.  Recording costs two event records per launch.
 */
PCG_API pcg_status pcg_profile_enable(int32_t enable);
PCG_API pcg_status pcg_profile_collect(int32_t max_entries, char *names, int64_t *launches,
                                       double *total_ms, int32_t *n_entries);

#ifdef __cplusplus
}
#endif

#endif /* PCG_H */
