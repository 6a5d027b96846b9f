/*
 * pcg_oracle.c -- plain, slow, obviously-correct fp64 CPU oracle for the
 * particle-to-grid deposit path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header or constant with the CUDA library.
 *
 * Every floating-point quantity is double.  Inputs arrive as float and are
 * promoted exactly.  Compile with -ffp-contract=off so that each operation is
 * rounded on its own (the 1D window test below is an integer decision taken in
 * fp64; the CUDA side takes it with the same sequence of rounded operations).
 *
 * Sources (page title, section / equation):
 *  - "03. Compaction and scatter-add" (WEANJ examples), sections "The problem"
 *    and "Code": the 1D windowed cloud-in-cell histogram and its loss.
 *  - "Mass Matrix Assembly on Tensor Cores for Implicit Particle-In-Cell
 *    Methods" (Pennati & Markidis), Sec. 2.1 Eqs. (4)-(6) (mass matrix and the
 *    rotation-response tensor), Sec. 2.3 Eq. (12) (tensor-product B-spline
 *    shape, TSC base-offset rule), Sec. 3.4 (offset-indexed stencil storage).
 *  - "Tiled current deposit" (Entity wiki), sections "How a tile deposit runs"
 *    and "The tile-based spatial sort": tile counts ceil(n/T) per axis, tile
 *    key, tile_offsets prefix sum; section "Halo sizing" names the O == 0
 *    zigzag deposit, whose scheme is the published one of Umeda et al. (2003).
 *
 * Parity pins: every function here is pinned by the CPU tests against brute
 * force, closed forms or invariants (see tests/test_oracle_pins.py).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_VERSION 1

int oracle_version(void) { return ORACLE_VERSION; }

/* Julia's mod(j, n) for n > 0: result in [0, n). */
static int64_t mod_floor(int64_t j, int64_t n) {
    int64_t r = j % n;
    return r < 0 ? r + n : r;
}

/* Periodic minimum image on the unit interval: d - round(d), ties to even
 * (the JAX helper on the WEANJ page uses jnp.round). */
static double minimg(double d) { return d - nearbyint(d); }

/* ------------------------------------------------------------------------ */
/* 1D windowed CIC histogram ("03. Compaction and scatter-add", "Code")       */
/* ------------------------------------------------------------------------ */
/*
 * For t = 1..nsteps: c = t/nsteps, x = wrap(x0 + v*(t*dt)),
 * d = minimg(x - c); particles with |d| < hw are deposited with weight
 * w = (1 - |d|/hw)^2 and linear CIC weights on g = x*nb - 1/2 into bins
 * j mod nb and (j+1) mod nb.  loss = sum_b (H_b - target_b)^2.
 * H (double[nbins]) is overwritten.  Returns the number of (particle, step)
 * deposits made.
 */
int64_t oracle_cic1d(const float *x0, const float *v, int64_t n,
                     const float *target, int32_t nbins, int32_t nsteps,
                     double dt, double hw, double *H, double *loss) {
    int64_t nsel = 0;
    for (int32_t b = 0; b < nbins; ++b) H[b] = 0.0;
    for (int32_t t = 1; t <= nsteps; ++t) {
        double c = (double)t / (double)nsteps;      /* window centre */
        double s = (double)t * dt;                  /* elapsed time  */
        for (int64_t p = 0; p < n; ++p) {
            double xu = (double)x0[p] + (double)v[p] * s;
            double x = xu - floor(xu);                 /* wrap to [0,1) */
            double d = minimg(x - c);
            if (!(fabs(d) < hw)) continue;             /* window test   */
            double u = 1.0 - fabs(d) / hw;
            double w = u * u;                          /* taper         */
            double g = x * (double)nbins - 0.5;        /* CIC position  */
            double jf = floor(g);
            double f = g - jf;
            int64_t j = (int64_t)jf;
            H[mod_floor(j, nbins)] += w * (1.0 - f);
            H[mod_floor(j + 1, nbins)] += w * f;
            ++nsel;
        }
    }
    double L = 0.0;
    for (int32_t b = 0; b < nbins; ++b) {
        double e = H[b] - (double)target[b];
        L += e * e;
    }
    *loss = L;
    return nsel;
}

/* Gradient of the 1D loss with respect to the initial positions, the
 * quantity the page differentiates ("03. Compaction and scatter-add", "The
 * problem": d L / d x0; "Code": the reverse pass is seeded with
 * dL/dH = 2 (H - target)).  The window test, the wrap and floor(g) are
 * piecewise constant; along x = wrap(x0 + v s) the derivative of every
 * selected (particle, step) term follows from
 *   d = minimg(x - c):  dd/dx0 = 1,
 *   w = (1 - |d|/h)^2:  dw/dd  = -2 (1 - |d|/h) sign(d) / h   (sign(0) = 0),
 *   f = x*nb - 1/2 - floor(.):  df/dx0 = nb,
 * so the pair H[j] += w (1 - f), H[j+1] += w f contributes
 *   G[j] (w' (1 - f) - w nb) + G[j+1] (w' f + w nb),  G = 2 (H - target).
 * H is the fp64 forward result of oracle_cic1d; dx0 is written for every
 * particle (zero for particles never selected).  Returns the selected count. */
int64_t oracle_cic1d_grad(const float *x0, const float *v, int64_t n,
                          const float *target, int32_t nbins, int32_t nsteps,
                          double dt, double hw, double *H, double *loss, double *dx0) {
    int64_t nsel = oracle_cic1d(x0, v, n, target, nbins, nsteps, dt, hw, H, loss);
    for (int64_t p = 0; p < n; ++p) dx0[p] = 0.0;
    for (int32_t t = 1; t <= nsteps; ++t) {
        double c = (double)t / (double)nsteps;
        double s = (double)t * dt;
        for (int64_t p = 0; p < n; ++p) {
            double xu = (double)x0[p] + (double)v[p] * s;
            double x = xu - floor(xu);
            double d = minimg(x - c);
            if (!(fabs(d) < hw)) continue;
            double u = 1.0 - fabs(d) / hw;
            double w = u * u;
            double sgn = d > 0.0 ? 1.0 : (d < 0.0 ? -1.0 : 0.0);
            double dw = -2.0 * u * sgn / hw;
            double g = x * (double)nbins - 0.5;
            double jf = floor(g);
            double f = g - jf;
            int64_t j = (int64_t)jf;
            double G0 = 2.0 * (H[mod_floor(j, nbins)] - (double)target[mod_floor(j, nbins)]);
            double G1 = 2.0 * (H[mod_floor(j + 1, nbins)] - (double)target[mod_floor(j + 1, nbins)]);
            dx0[p] += G0 * (dw * (1.0 - f) - w * (double)nbins) + G1 * (dw * f + w * (double)nbins);
        }
    }
    return nsel;
}

/* ------------------------------------------------------------------------ */
/* 1D B-spline weights (Pennati & Markidis, Sec. 2.3, Eq. (12))              */
/* ------------------------------------------------------------------------ */
/* Order-1 B-spline (CIC): phi(s) = 1 - |s| on |s| <= 1. */
static double bspline1(double s) {
    double a = fabs(s);
    return a < 1.0 ? 1.0 - a : 0.0;
}

/* Order-2 B-spline (TSC / quadratic): 3/4 - s^2 on |s| <= 1/2,
 * (3/2 - |s|)^2 / 2 on 1/2 <= |s| <= 3/2. */
static double bspline2(double s) {
    double a = fabs(s);
    if (a <= 0.5) return 0.75 - a * a;
    if (a <= 1.5) return 0.5 * (1.5 - a) * (1.5 - a);
    return 0.0;
}

/*
 * Support of one axis: first node and the per-node weights.
 * order 1: nodes i, i+1 (i = floor x).
 * order 2: nodes i-1..i+1 when xi < 1/2, else i..i+2 (the base-offset rule of
 * Sec. 2.3); weights are phi(x - node).
 * Returns the number of support nodes.
 */
static int axis_support(int order, double x, int64_t *first, double wts[3]) {
    double fi = floor(x);
    double xi = x - fi;
    int64_t i = (int64_t)fi;
    if (order == 1) {
        *first = i;
        wts[0] = bspline1(x - (double)i);
        wts[1] = bspline1(x - (double)(i + 1));
        return 2;
    }
    int64_t base = (xi < 0.5) ? i - 1 : i;
    *first = base;
    for (int k = 0; k < 3; ++k) wts[k] = bspline2(x - (double)(base + k));
    return 3;
}

/* A position is inside the periodic domain when 0 <= x < N (NaN is not). */
static int in_domain(double x, int32_t N) { return x >= 0.0 && x < (double)N; }

/* exported for the pin tests: the per-axis support of one coordinate */
int oracle_axis_support(int32_t order, double x, int64_t *first, double *wts) {
    if (order != 1 && order != 2) return -1;
    return axis_support(order, x, first, wts);
}

/* ------------------------------------------------------------------------ */
/* Current deposit J^c_g = sum_p q_p v^c_p W(x_p - x_g)                      */
/* ------------------------------------------------------------------------ */
/*
 * dim = 2 or 3, order = 1 (CIC) or 2 (quadratic).  grid[0..dim) = (Nx, Ny[, Nz]).
 * pos[0..dim) are positions in cell units; vel[0..3) always three components
 * (in 2D, vz deposits Jz on the 2D stencil).  J is double[3][ncells] with the
 * flattened node index (z*Ny + y)*Nx + x; it is overwritten.  Periodic on every
 * axis.  Particles with a coordinate outside [0, N) (or NaN) are skipped and
 * counted.  Returns that count.
 */
int64_t oracle_deposit_current(int32_t dim, const int32_t *grid, int32_t order,
                               int64_t n, const float *const *pos,
                               const float *const *vel, const float *q,
                               double *J) {
    int32_t Nx = grid[0], Ny = grid[1], Nz = (dim == 3) ? grid[2] : 1;
    int64_t ncells = (int64_t)Nx * Ny * Nz;
    memset(J, 0, sizeof(double) * 3 * (size_t)ncells);
    int64_t n_invalid = 0;
    for (int64_t p = 0; p < n; ++p) {
        double x = pos[0][p], y = pos[1][p], z = (dim == 3) ? (double)pos[2][p] : 0.0;
        if (!in_domain(x, Nx) || !in_domain(y, Ny) || (dim == 3 && !in_domain(z, Nz))) {
            ++n_invalid;
            continue;
        }
        int64_t fx, fy, fz = 0;
        double wx[3], wy[3], wz[3] = {1.0, 0.0, 0.0};
        int sx = axis_support(order, x, &fx, wx);
        int sy = axis_support(order, y, &fy, wy);
        int sz = 1;
        if (dim == 3) sz = axis_support(order, z, &fz, wz);
        double qv[3];
        for (int c = 0; c < 3; ++c) qv[c] = (double)q[p] * (double)vel[c][p];
        for (int kz = 0; kz < sz; ++kz) {
            int64_t gz = mod_floor(fz + kz, Nz);
            for (int ky = 0; ky < sy; ++ky) {
                int64_t gy = mod_floor(fy + ky, Ny);
                for (int kx = 0; kx < sx; ++kx) {
                    int64_t gx = mod_floor(fx + kx, Nx);
                    double W = wx[kx] * wy[ky] * wz[kz];
                    int64_t g = (gz * Ny + gy) * Nx + gx;
                    for (int c = 0; c < 3; ++c) J[c * ncells + g] += qv[c] * W;
                }
            }
        }
    }
    return n_invalid;
}

/* ------------------------------------------------------------------------ */
/* Charge-conserving zigzag current deposit                                  */
/* ------------------------------------------------------------------------ */
/*
 * The O == 0 deposit of "Tiled current deposit" (Entity wiki), section "Halo
 * sizing": it writes at most 2 cells above min(i, i_prev).  The page names the
 * scheme without defining it; this is the zigzag scheme of Umeda, Omura,
 * Tominaga & Matsumoto, Comput. Phys. Commun. 156 (2003) 73, for unit cells:
 *
 * per axis, with cells i1 = floor(x1), i2 = floor(x2) (|i2 - i1| <= 1),
 *   relay  xr = min(min(i1, i2) + 1, max(max(i1, i2), (x1 + x2) / 2)),
 *   moves  D1 = xr - x1,  D2 = x2 - xr,  fluxes F_s = q D_s / dt,
 *   shape  W1 = (x1 + xr) / 2 - i1,  W2 = (xr + x2) / 2 - i2;
 * segment s (cell (i_s, j_s, k_s)) adds to J^x at the four edges
 * (i_s + 1/2, j_s + a, k_s + b), a, b in {0, 1}, the flux F_s^x times the
 * bilinear weight of (W_s^y, W_s^z) averaged along the straight segment:
 *   w_a(W^y) w_b(W^z) + (a == b ? +1 : -1) D_s^y D_s^z / 12,
 * w_0(W) = 1 - W, w_1(W) = W; likewise for y and z.  The D D / 12 term is the
 * exact path average of the product (Villasenor & Buneman); it vanishes when
 * the segment moves along at most two axes, where the expression is Umeda's.
 * With rho the CIC charge at the nodes, this J satisfies
 * (rho(x2) - rho(x1)) / dt + div J = 0 exactly, div taken with backward
 * differences of the edge currents.
 *
 * Layout: J is double[3][ncells]; J[c][(k*Ny + j)*Nx + i] holds the c-current
 * on the edge from node (i, j, k) towards +e_c.  Periodic on every axis.
 *
 * Inputs: pos_prev = x1 and pos = x2, both in [0, N); the move is taken as the
 * periodic minimum image of the cell difference, so a particle may cross the
 * periodic boundary.  A particle with a coordinate outside [0, N) (or NaN), or
 * whose cell changes by more than one along an axis (beyond the scheme's CFL
 * limit), is skipped and counted.  Returns that count.  grid[mu] >= 3.
 */
int64_t oracle_deposit_zigzag(const int32_t *grid, int64_t n, const float *const *pos_prev,
                              const float *const *pos, const float *q, double dt, double *J) {
    const int64_t N[3] = {grid[0], grid[1], grid[2]};
    const int64_t ncells = N[0] * N[1] * N[2];
    memset(J, 0, sizeof(double) * 3 * (size_t)ncells);
    int64_t n_invalid = 0;
    for (int64_t p = 0; p < n; ++p) {
        int ok = 1;
        int64_t base[3];        /* lower of the two cells (unwrapped) */
        int cell[2][3];         /* cell of each segment relative to base: 0 or 1 */
        double F[2][3], W[2][3], D[2][3];
        for (int mu = 0; mu < 3 && ok; ++mu) {
            double x1 = pos_prev[mu][p], x2 = pos[mu][p];
            if (!in_domain(x1, (int32_t)N[mu]) || !in_domain(x2, (int32_t)N[mu])) {
                ok = 0;
                break;
            }
            int64_t i1 = (int64_t)floor(x1), i2 = (int64_t)floor(x2);
            int64_t di = i2 - i1;  /* periodic minimum image */
            if (2 * di > N[mu]) di -= N[mu];
            if (2 * di < -N[mu]) di += N[mu];
            if (di < -1 || di > 1) {
                ok = 0;
                break;
            }
            int64_t lo = di < 0 ? di : 0;
            int a = (int)(-lo), b = (int)(di - lo);
            /* positions relative to the lower cell's low node */
            double X1 = (double)a + (x1 - (double)i1);
            double X2 = (double)b + (x2 - (double)i2);
            double hi = (double)(a > b ? a : b);
            double xr = fmin(1.0, fmax(hi, 0.5 * (X1 + X2)));
            base[mu] = i1 + lo;
            cell[0][mu] = a;
            cell[1][mu] = b;
            D[0][mu] = xr - X1;
            D[1][mu] = X2 - xr;
            F[0][mu] = (double)q[p] * D[0][mu] / dt;
            F[1][mu] = (double)q[p] * D[1][mu] / dt;
            W[0][mu] = 0.5 * (X1 + xr) - (double)a;
            W[1][mu] = 0.5 * (xr + X2) - (double)b;
        }
        if (!ok) {
            ++n_invalid;
            continue;
        }
        for (int s = 0; s < 2; ++s)
            for (int c = 0; c < 3; ++c) {
                int u = (c + 1) % 3, v = (c + 2) % 3; /* the two transverse axes */
                for (int du = 0; du < 2; ++du)
                    for (int dv = 0; dv < 2; ++dv) {
                        int64_t node[3];
                        for (int mu = 0; mu < 3; ++mu) node[mu] = base[mu] + cell[s][mu];
                        node[u] += du;
                        node[v] += dv;
                        double wu = du ? W[s][u] : 1.0 - W[s][u];
                        double wv = dv ? W[s][v] : 1.0 - W[s][v];
                        double avg = D[s][u] * D[s][v] / 12.0;
                        double w = wu * wv + (du == dv ? avg : -avg);
                        int64_t g = (mod_floor(node[2], N[2]) * N[1] + mod_floor(node[1], N[1])) * N[0] +
                                    mod_floor(node[0], N[0]);
                        J[c * ncells + g] += F[s][c] * w;
                    }
            }
    }
    return n_invalid;
}

/* ------------------------------------------------------------------------ */
/* Rotation-response tensor (Pennati & Markidis, Sec. 2.1, Eq. (5))          */
/* ------------------------------------------------------------------------ */
/*
 * alpha = (I - C(w) + w w^T) / (1 + |w|^2) with C(w) u = w x u, i.e.
 * C = [[0,-w3,w2],[w3,0,-w1],[-w2,w1,0]].  alpha is row-major [i][j].
 */
void oracle_alpha(const double *w, double *alpha) {
    double C[3][3] = {{0.0, -w[2], w[1]}, {w[2], 0.0, -w[0]}, {-w[1], w[0], 0.0}};
    double n2 = w[0] * w[0] + w[1] * w[1] + w[2] * w[2];
    for (int i = 0; i < 3; ++i)
        for (int j = 0; j < 3; ++j) {
            double I = (i == j) ? 1.0 : 0.0;
            alpha[i * 3 + j] = (I - C[i][j] + w[i] * w[j]) / (1.0 + n2);
        }
}

/* ------------------------------------------------------------------------ */
/* ECSIM block mass matrix, first-order B-splines (Sec. 2.1 Eq. (6), 3.4)    */
/* ------------------------------------------------------------------------ */
/*
 * M[g][o][i][j] = sum_p w_p alpha_p^{ij} W_pg W_pg',  g' = g + delta (mod N),
 * delta in {-1,0,1}^3, o = (dz+1)*9 + (dy+1)*3 + (dx+1).  sigma = 1.
 * grid = (Nx, Ny, Nz), each >= 3 so that the 27 offsets name distinct nodes.
 * M is double[ncells][27][3][3], overwritten.  Out-of-domain particles are
 * skipped and counted; the count is returned.
 */
int64_t oracle_mass_matrix(const int32_t *grid, int64_t n,
                           const float *const *pos, const float *wq,
                           const float *const *omega, double *M) {
    int32_t Nx = grid[0], Ny = grid[1], Nz = grid[2];
    int64_t ncells = (int64_t)Nx * Ny * Nz;
    memset(M, 0, sizeof(double) * 243 * (size_t)ncells);
    int64_t n_invalid = 0;
    for (int64_t p = 0; p < n; ++p) {
        double x[3] = {pos[0][p], pos[1][p], pos[2][p]};
        if (!in_domain(x[0], Nx) || !in_domain(x[1], Ny) || !in_domain(x[2], Nz)) {
            ++n_invalid;
            continue;
        }
        int64_t first[3];
        double wt[3][3];
        for (int mu = 0; mu < 3; ++mu) axis_support(1, x[mu], &first[mu], wt[mu]);
        double om[3] = {omega[0][p], omega[1][p], omega[2][p]};
        double alpha[9];
        oracle_alpha(om, alpha);
        double s[9];
        for (int ij = 0; ij < 9; ++ij) s[ij] = (double)wq[p] * alpha[ij];
        /* corner a = (ax, ay, az) in {0,1}^3 */
        for (int a = 0; a < 8; ++a) {
            int ax = a & 1, ay = (a >> 1) & 1, az = (a >> 2) & 1;
            double Wa = wt[0][ax] * wt[1][ay] * wt[2][az];
            int64_t g = (mod_floor(first[2] + az, Nz) * Ny + mod_floor(first[1] + ay, Ny)) * Nx
                        + mod_floor(first[0] + ax, Nx);
            for (int b = 0; b < 8; ++b) {
                int bx = b & 1, by = (b >> 1) & 1, bz = (b >> 2) & 1;
                double Wb = wt[0][bx] * wt[1][by] * wt[2][bz];
                int o = (bz - az + 1) * 9 + (by - ay + 1) * 3 + (bx - ax + 1);
                double *blk = M + ((size_t)g * 27 + (size_t)o) * 9;
                for (int ij = 0; ij < 9; ++ij) blk[ij] += s[ij] * Wa * Wb;
            }
        }
    }
    return n_invalid;
}

/* Mass matrix with second-order (TSC) B-splines (Pennati & Markidis, Sec. 2.3
 * Eq. (12) and the base-offset rule: a coordinate with fractional part < 1/2
 * uses nodes j-1..j+1, else j..j+2; Sec. 3.3: particles of a cell with the same
 * node set form a support group, up to 8 per cell; Sec. 3.4: displacements in
 * {-2..2}^3, 125 offsets).  M^{ij}_{gg'} = sum_p w_p alpha_p^{ij} W_pg W_pg',
 * stored with every offset: M[g][o][i][j], o = (dz+2)*25 + (dy+2)*5 + (dx+2)
 * for g' = g + (dx,dy,dz) (periodic), double[ncells][125][9], overwritten.
 * Every grid edge must be >= 5.  Returns the particles skipped for a
 * coordinate outside [0, N). */
int64_t oracle_mass_matrix_tsc(const int32_t *grid, int64_t n, const float *const *pos, const float *wq,
                               const float *const *omega, double *M) {
    int32_t Nx = grid[0], Ny = grid[1], Nz = grid[2];
    int64_t ncells = (int64_t)Nx * Ny * Nz;
    memset(M, 0, sizeof(double) * 1125 * (size_t)ncells);
    int64_t n_invalid = 0;
    for (int64_t p = 0; p < n; ++p) {
        double x[3] = {pos[0][p], pos[1][p], pos[2][p]};
        if (!in_domain(x[0], Nx) || !in_domain(x[1], Ny) || !in_domain(x[2], Nz)) {
            ++n_invalid;
            continue;
        }
        int64_t first[3];
        double wt[3][3];
        for (int mu = 0; mu < 3; ++mu) axis_support(2, x[mu], &first[mu], wt[mu]);
        double om[3] = {omega[0][p], omega[1][p], omega[2][p]};
        double alpha[9];
        oracle_alpha(om, alpha);
        for (int a = 0; a < 27; ++a) {
            int ax = a % 3, ay = (a / 3) % 3, az = a / 9;
            double Wa = wt[0][ax] * wt[1][ay] * wt[2][az];
            int64_t g = (mod_floor(first[2] + az, Nz) * Ny + mod_floor(first[1] + ay, Ny)) * Nx
                        + mod_floor(first[0] + ax, Nx);
            for (int b = 0; b < 27; ++b) {
                int bx = b % 3, by = (b / 3) % 3, bz = b / 9;
                double Wb = wt[0][bx] * wt[1][by] * wt[2][bz];
                int o = (bz - az + 2) * 25 + (by - ay + 2) * 5 + (bx - ax + 2);
                double *blk = M + ((size_t)g * 125 + (size_t)o) * 9;
                for (int ij = 0; ij < 9; ++ij) blk[ij] += (double)wq[p] * alpha[ij] * Wa * Wb;
            }
        }
    }
    return n_invalid;
}

/* Scalar mass matrix (Pennati & Markidis, Sec. 2.1 after Eq. (6): the scalar
 * case s_p^{ij} = q_p delta^{ij}, e.g. the MPM mass matrix, one component per
 * node pair): M_{gg'} = sum_p w_p W_pg W_pg' with CIC shapes, stored by stencil
 * offset as M[g][o], o = (dz+1)*9 + (dy+1)*3 + (dx+1) for g' = g + (dx,dy,dz)
 * (periodic).  M is double[ncells][27], overwritten.  Returns the number of
 * particles skipped for a coordinate outside [0, N). */
int64_t oracle_mass_matrix_scalar(const int32_t *grid, int64_t n, const float *const *pos,
                                  const float *w, double *M) {
    int32_t Nx = grid[0], Ny = grid[1], Nz = grid[2];
    int64_t ncells = (int64_t)Nx * Ny * Nz;
    memset(M, 0, sizeof(double) * 27 * (size_t)ncells);
    int64_t n_invalid = 0;
    for (int64_t p = 0; p < n; ++p) {
        double x[3] = {pos[0][p], pos[1][p], pos[2][p]};
        if (!in_domain(x[0], Nx) || !in_domain(x[1], Ny) || !in_domain(x[2], Nz)) {
            ++n_invalid;
            continue;
        }
        int64_t first[3];
        double wt[3][3];
        for (int mu = 0; mu < 3; ++mu) axis_support(1, x[mu], &first[mu], wt[mu]);
        for (int a = 0; a < 8; ++a) {
            int ax = a & 1, ay = (a >> 1) & 1, az = (a >> 2) & 1;
            double Wa = wt[0][ax] * wt[1][ay] * wt[2][az];
            int64_t g = (mod_floor(first[2] + az, Nz) * Ny + mod_floor(first[1] + ay, Ny)) * Nx
                        + mod_floor(first[0] + ax, Nx);
            for (int b = 0; b < 8; ++b) {
                int bx = b & 1, by = (b >> 1) & 1, bz = (b >> 2) & 1;
                double Wb = wt[0][bx] * wt[1][by] * wt[2][bz];
                int o = (bz - az + 1) * 9 + (by - ay + 1) * 3 + (bx - ax + 1);
                M[(size_t)g * 27 + (size_t)o] += (double)w[p] * Wa * Wb;
            }
        }
    }
    return n_invalid;
}

/* ------------------------------------------------------------------------ */
/* Tile key and tile_offsets ("Tiled current deposit", tile-based sort)      */
/* ------------------------------------------------------------------------ */
/*
 * ntiles per axis = ceil(N / tile); tile index of a particle = index of the
 * tile holding its cell floor(x), x fastest.  Out-of-domain particles get the
 * sentinel key ntiles_total.  offsets[0..ntiles_total] is the exclusive prefix
 * sum of the per-tile counts (offsets[ntiles_total] = number of in-domain
 * particles).  Returns ntiles_total.
 */
int64_t oracle_tile_keys(int32_t dim, const int32_t *grid, int32_t tile, int64_t n,
                         const float *const *pos, uint32_t *keys, uint32_t *offsets) {
    int64_t nt[3] = {1, 1, 1};
    for (int mu = 0; mu < dim; ++mu) nt[mu] = (grid[mu] + tile - 1) / tile;
    int64_t total = nt[0] * nt[1] * nt[2];
    for (int64_t t = 0; t <= total; ++t) offsets[t] = 0;
    for (int64_t p = 0; p < n; ++p) {
        int ok = 1;
        int64_t tc[3] = {0, 0, 0};
        for (int mu = 0; mu < dim; ++mu) {
            double x = pos[mu][p];
            if (!in_domain(x, grid[mu])) { ok = 0; break; }
            tc[mu] = (int64_t)floor(x) / tile;
        }
        uint32_t k = ok ? (uint32_t)((tc[2] * nt[1] + tc[1]) * nt[0] + tc[0]) : (uint32_t)total;
        if (keys) keys[p] = k;
        if (ok) offsets[k] += 1;
    }
    /* exclusive scan in place */
    uint32_t run = 0;
    for (int64_t t = 0; t <= total; ++t) {
        uint32_t c = offsets[t];
        offsets[t] = run;
        run += c;
    }
    return total;
}
