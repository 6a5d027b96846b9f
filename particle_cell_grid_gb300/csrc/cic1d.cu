// cic1d.cu -- 1D windowed cloud-in-cell histogram, loss and gradient.
//
// Method: "03. Compaction and scatter-add" (WEANJ examples), sections "The
// problem" and "Code".  For every step t = 1..T the particles inside a window of
// half-width h around c = t/T add a tapered weight w = (1 - |d|/h)^2 to the two
// CIC bins of g = x*nb - 1/2; the loss is ||H - target||^2, and the gradient
// dL/dx0 is seeded with dL/dH = 2 (H - target).
//
// GB300 design.  The pages launch one kernel per step (T launches) with global
// atomics and note that a stream-compaction pass before the deposit is what a
// CUDA programmer would add ("Where JAX wins / what we did not do").  Here all
// T steps run in one launch, and the compaction is done per warp, in shared
// memory, on the fly:
//   * every lane owns one particle of a 32-particle chunk and walks t = 1..T
//     with a cheap fp32 window test (the screen);
//   * the (particle, step) pairs that pass (~1% for h = 0.005) are appended to
//     a 64-entry queue private to the warp (ballot + popc, no atomics, no
//     block barrier);
//   * whenever the queue holds 32 candidates the warp takes them together, one
//     per lane, through the exact fp64 test and the deposit (or the gradient
//     gather).  So the slow fp64 path always runs with all 32 lanes busy,
//     instead of a few lanes of a diverged warp.
// Small N: one 8-CTA thread-block cluster; each CTA keeps a private histogram in
// shared memory, the CTAs meet at a cluster barrier and CTA 0 sums the eight
// histograms through distributed shared memory in a fixed order, writes H and
// reduces the loss in fp64 (one launch, no workspace).  Large N: a full grid of
// CTAs, each adding its shared histogram to H with global reductions, then a
// one-CTA loss kernel.  The gradient is a second kernel of the same shape that
// gathers 2 (H - target) at the same two bins.
//
// Precision.  In fp32, x = x0 + v*t*dt carries ~6e-8 absolute error, i.e.
// ~6e-5 of a bin after the scaling by nb = 1024, which would move CIC weights
// by more than the 1e-5 tolerance; so the window test, g and floor(g) are done
// in fp64 with individually rounded operations (the __d*_rn intrinsics are never
// contracted into FMAs), exactly as the fp64 oracle does them; the weights that
// follow from the exact d and f are fp32.  The fp32 screen uses a margin that
// provably covers its own rounding, so it never drops a pair the fp64 test
// would select, and each particle screens only the steps near its window
// crossings (about 4.5 of T = 50 here), found from the linear motion.
#include <cooperative_groups.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace pcg {
namespace {

constexpr int kCtas = 8;      // CTAs of the small-N cluster
constexpr int kThreads = 256;  // threads of every CTA here
constexpr int kWarps = kThreads / 32;
constexpr int kQueue = 64;     // candidates a warp can hold (31 left over + 32 new, rounded up)
// up to this many particles the histogram is built by the single 8-CTA
// cluster; above it by a full grid with global reductions
constexpr long long kClusterMaxN = 1ll << 14;

// Per-launch constants of the method.
struct Cic1dArgs {
    const float *x0, *v;
    long long n;
    const float *target;
    int nbins, nsteps;
    double dt, hw;
    float dt32, hw32, inv_t32;  // dt, h and 1/T rounded to fp32 for the screen
    float inv_hw32;             // 1/h for the weights
};

// c = t/T for t = 1..kTab, filled once per CTA in shared memory (longer runs
// divide per pair).
constexpr int kTab = 1024;

// fp32 screen of one (particle, step) pair.  |d32 - d64| stays below
// ~6 ulp(1 + |x0| + |v s|) (the rounding of t*dt, v*s, x0 + v s, c and the
// subtractions); the margin 2e-6 * (4 + |x0| + |v s|) is far above that, so
// every pair the fp64 test selects passes.  When h + margin reaches 0.45 the
// screen passes everything (both tests then reject |d| ~ 1/2 alike, where the
// minimum image jumps).
__device__ __forceinline__ bool cic1d_screen(const Cic1dArgs &a, float xf, float vf, int t) {
    const float tf = (float)t;
    const float vs32 = vf * (tf * a.dt32);
    float d32 = (xf + vs32) - tf * a.inv_t32;
    d32 = d32 - rintf(d32);
    const float lim = a.hw32 + 2e-6f * (4.f + fabsf(xf) + fabsf(vs32));
    return fabsf(d32) < lim || !(lim < 0.45f);
}

// One selected (particle, step) pair in fp64.
struct Pair {
    float sgn, u, w, f;  // sign of the minimum-image distance, 1 - |d|/h, taper, CIC fraction
    int b0, b1;          // the two bins
};

// Exact fp64 window test and CIC bins, the same operation sequence as the
// oracle: s = t dt, x = wrap(x0 + v s), d = minimg(x - t/T), |d| < h,
// g = x nb - 1/2, bins floor(g) and floor(g) + 1.  The weights, which decide
// nothing, are taken in fp32 from the exact d and f = g - floor(g) (fp64 runs
// at 1/64 of the fp32 rate on this part): relative error ~1e-7, far inside
// the 1e-5 tolerance.  d is a multiple of 2^-53 or zero, so its fp32 sign is
// exact.
__device__ __forceinline__ bool cic1d_select(const Cic1dArgs &a, const double *ctab, float xf, float vf, int t,
                                             Pair &o) {
    const double s = __dmul_rn((double)t, a.dt);
    const double xu = __dadd_rn((double)xf, __dmul_rn((double)vf, s));
    const double x = __dsub_rn(xu, floor(xu));
    const double c = ctab != nullptr ? ctab[t - 1] : __ddiv_rn((double)t, (double)a.nsteps);
    const double d0 = __dsub_rn(x, c);
    const double d = __dsub_rn(d0, rint(d0));
    const double ad = fabs(d);
    if (!(ad < a.hw)) return false;
    const float d32 = (float)d;
    o.sgn = d32 > 0.f ? 1.f : (d32 < 0.f ? -1.f : 0.f);
    o.u = 1.f - fabsf(d32) * a.inv_hw32;
    o.w = o.u * o.u;
    const double g = __dsub_rn(__dmul_rn(x, (double)a.nbins), 0.5);
    const double jf = floor(g);
    o.f = (float)__dsub_rn(g, jf);
    int b0 = (int)jf % a.nbins;
    if (b0 < 0) b0 += a.nbins;
    o.b0 = b0;
    o.b1 = b0 + 1 == a.nbins ? 0 : b0 + 1;
    return true;
}

// Candidate queue of one warp, in shared memory.
struct WarpQueue {
    float2 xv[kQueue];      // x0 and v of the particle
    int t[kQueue];          // step
    long long p[kQueue];    // particle index (read by the gradient only)
};

// Candidate steps of one particle.  The screen's distance before the minimum
// image is linear in t: l(t) = x0 + t a with a = v dt - 1/T, so the steps it
// can pass lie in one short run per window crossing, |l(t) - k| < L for an
// integer k.  L = h + 4e-6 (4 + |x0| + |v| T dt) exceeds the screen's limit
// plus its rounding (both at most h + 2.3e-6 (4 + ...)), and each run is
// widened by a step on both sides, so every step the screen would pass is
// generated; each generated step still goes through the screen itself.  Runs
// are visited in increasing t and never overlap, so no step repeats.  Wide
// windows, slopes under 1e-3 per step, |x0| > 1e3 or runs that would not save
// work fall back to every step 1..T.
struct StepGen {
    int t, t_end;       // next step, end of the current run
    int k, k_last, dk;  // current window index, last one, direction (+-1)
    float x, a, L;

    __device__ __forceinline__ void init(const Cic1dArgs &args, float xf, float vf, bool live) {
        const int T = args.nsteps;
        t = 1;
        t_end = live ? T : 0;
        k = k_last = 0;
        dk = 1;
        x = xf;
        a = vf * args.dt32 - args.inv_t32;
        L = args.hw32 + 4e-6f * (4.f + fabsf(xf) + fabsf(vf) * (float)T * args.dt32);
        if (!live || !(L < 0.45f) || !(fabsf(a) >= 1e-3f) || !(fabsf(xf) <= 1e3f)) return;
        const float y1 = xf + a, yT = xf + a * (float)T;
        const float kmin = floorf(fminf(y1, yT) - L) - 1.f, kmax = ceilf(fmaxf(y1, yT) + L) + 1.f;
        if (!(kmax - kmin <= (float)T * 0.25f)) return;  // the direct walk is as cheap
        dk = a > 0.f ? 1 : -1;
        k = (int)(a > 0.f ? kmin : kmax);
        k_last = (int)(a > 0.f ? kmax : kmin);
        t = 1;
        window(T);
    }
    // steps of window k, clipped to [t, T]
    __device__ __forceinline__ void window(int T) {
        float lo = ((float)k - x - L) / a, hi = ((float)k - x + L) / a;
        if (a < 0.f) {
            const float tmp = lo;
            lo = hi;
            hi = tmp;
        }
        lo = fminf(fmaxf(lo, -2.f), (float)T + 2.f);
        hi = fminf(fmaxf(hi, -2.f), (float)T + 2.f);
        const int tlo = (int)floorf(lo) - 1, thi = (int)ceilf(hi) + 1;
        if (tlo > t) t = tlo;
        t_end = thi < T ? thi : T;
    }
    // next candidate step, 0 when none is left
    __device__ __forceinline__ int next(int T) {
        while (t > t_end) {
            if (k == k_last) return 0;
            k += dk;
            window(T);
        }
        return t++;
    }
};

// The warp walks the 32-particle chunks warp_id, warp_id + nwarps, ... (lane =
// particle) over its candidate steps.  Pairs that pass the screen go to the
// warp's queue; every time it holds 32 they are handed to take(x0, v, t, p)
// together, one per lane; the last partial batch goes at the end.
// on_load(p) runs once per particle when its chunk is loaded.  The count of
// queued pairs is the same in every lane (it only changes by popc of a
// ballot), so every branch on it is warp-uniform and no block barrier is
// needed.
template <bool kNeedP, class OnLoad, class Take>
__device__ __forceinline__ void cic1d_walk(const Cic1dArgs &a, long long warp_id, long long nwarps,
                                           WarpQueue &q, OnLoad on_load, Take take) {
    const int lane = threadIdx.x & 31;
    const unsigned below = (1u << lane) - 1u;
    int count = 0;
    for (long long base = warp_id * 32; base < a.n; base += nwarps * 32) {
        const long long p = base + lane;
        const bool live = p < a.n;
        float xf = 0.f, vf = 0.f;
        if (live) {
            xf = a.x0[p];
            vf = a.v[p];
            on_load(p);
        }
        StepGen gen;
        gen.init(a, xf, vf, live);
        for (;;) {
            const int t = gen.next(a.nsteps);
            if (!__any_sync(0xffffffffu, t > 0)) break;
            const bool pass = t > 0 && cic1d_screen(a, xf, vf, t);
            const unsigned m = __ballot_sync(0xffffffffu, pass);
            if (m == 0u) continue;
            if (pass) {
                const int slot = count + __popc(m & below);
                q.xv[slot] = make_float2(xf, vf);
                q.t[slot] = t;
                if (kNeedP) q.p[slot] = p;
            }
            count += __popc(m);
            if (count >= 32) {  // take the newest 32
                count -= 32;
                __syncwarp();
                const int e = count + lane;
                take(q.xv[e].x, q.xv[e].y, q.t[e], kNeedP ? q.p[e] : 0ll);
                __syncwarp();
            }
        }
    }
    __syncwarp();
    if (lane < count) take(q.xv[lane].x, q.xv[lane].y, q.t[lane], kNeedP ? q.p[lane] : 0ll);
}

// t/T for t = 1..min(T, kTab) into the CTA's table; the caller syncs.
__device__ __forceinline__ const double *fill_ctab(const Cic1dArgs &a, double *ctab) {
    if (a.nsteps > kTab) return nullptr;
    for (int t = threadIdx.x; t < a.nsteps; t += kThreads) ctab[t] = __ddiv_rn((double)(t + 1), (double)a.nsteps);
    return ctab;
}

// Deposit of one selected pair into the CTA's shared histogram.
__device__ __forceinline__ void cic1d_deposit_pair(const Cic1dArgs &a, const double *ctab, float *hist, float xf,
                                                   float vf, int t) {
    Pair pr;
    if (!cic1d_select(a, ctab, xf, vf, t, pr)) return;
    if (!PCG_IN(pr.b0, a.nbins) || !PCG_IN(pr.b1, a.nbins)) return;
    red_shared_add_f32(&hist[pr.b0], pr.w * (1.f - pr.f));
    red_shared_add_f32(&hist[pr.b1], pr.w * pr.f);
}

// Small N: the whole histogram and the loss in one 8-CTA cluster.
__global__ void __cluster_dims__(kCtas, 1, 1) __launch_bounds__(kThreads)
    cic1d_cluster_kernel(Cic1dArgs a, float *__restrict__ H, double *__restrict__ loss) {
    extern __shared__ float hist[];  // [nbins]
    __shared__ WarpQueue queues[kWarps];
    __shared__ double red[kWarps];
    __shared__ double ctab_s[kTab];
    cg::cluster_group cluster = cg::this_cluster();
    const unsigned rank = cluster.block_rank();
    const int nbins = a.nbins;

    for (int b = threadIdx.x; b < nbins; b += kThreads) hist[b] = 0.f;
    const double *ctab = fill_ctab(a, ctab_s);
    __syncthreads();

    const int warp = threadIdx.x >> 5;
    cic1d_walk<false>(
        a, (long long)rank * kWarps + warp, (long long)kCtas * kWarps, queues[warp], [](long long) {},
        [&](float xf, float vf, int t, long long) { cic1d_deposit_pair(a, ctab, hist, xf, vf, t); });

    // all eight histograms complete and visible cluster-wide
    cluster.sync();

    if (rank == 0) {
        float *remote[kCtas];
        for (int r = 0; r < kCtas; ++r) remote[r] = cluster.map_shared_rank(hist, r);
        double acc = 0.0;
        for (int b = threadIdx.x; b < nbins; b += kThreads) {
            float sum = 0.f;
#pragma unroll
            for (int r = 0; r < kCtas; ++r) sum += remote[r][b];
            H[b] = sum;
            const double e = (double)sum - (double)a.target[b];
            acc = fma(e, e, acc);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if ((threadIdx.x & 31) == 0) red[warp] = acc;
        __syncthreads();
        if (threadIdx.x == 0) {
            double L = 0.0;
            for (int w = 0; w < kWarps; ++w) L += red[w];
            *loss = L;
        }
    }
    // keep every CTA's shared memory alive until CTA 0 has read it
    cluster.sync();
}

// Large N: every CTA builds a partial histogram and adds its non-zero bins to
// H (zeroed before the launch) with global reductions.
__global__ void __launch_bounds__(kThreads) cic1d_hist_kernel(Cic1dArgs a, float *__restrict__ H) {
    extern __shared__ float hist[];  // [nbins]
    __shared__ WarpQueue queues[kWarps];
    __shared__ double ctab_s[kTab];
    const int nbins = a.nbins;
    for (int b = threadIdx.x; b < nbins; b += kThreads) hist[b] = 0.f;
    const double *ctab = fill_ctab(a, ctab_s);
    __syncthreads();
    const int warp = threadIdx.x >> 5;
    cic1d_walk<false>(
        a, (long long)blockIdx.x * kWarps + warp, (long long)gridDim.x * kWarps, queues[warp],
        [](long long) {},
        [&](float xf, float vf, int t, long long) { cic1d_deposit_pair(a, ctab, hist, xf, vf, t); });
    __syncthreads();
    for (int b = threadIdx.x; b < nbins; b += kThreads) {
        const float h = hist[b];
        if (h != 0.f) red_add_f32(&H[b], h);
    }
}

// loss = sum_b (H_b - target_b)^2 in fp64, one CTA.
__global__ void __launch_bounds__(kThreads)
    cic1d_loss_kernel(const float *__restrict__ H, const float *__restrict__ target, int nbins,
                      double *__restrict__ loss) {
    __shared__ double red[kWarps];
    double acc = 0.0;
    for (int b = threadIdx.x; b < nbins; b += kThreads) {
        const double e = (double)H[b] - (double)target[b];
        acc = fma(e, e, acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        double L = 0.0;
        for (int w = 0; w < kWarps; ++w) L += red[w];
        *loss = L;
    }
}

// Gradient: dx0[p] = sum over the selected steps of
//   G[b0] (w' (1 - f) - w nb) + G[b1] (w' f + w nb),  G = 2 (H - target),
// with w' = dw/dd = -2 u sign(d) / h and df/dx0 = nb (the wrap, the window
// test and floor(g) are piecewise constant).  Every particle's entry is
// zeroed when its chunk is loaded; pairs of the same particle can sit in one
// batch, so they are added with fp64 atomics.
__global__ void __launch_bounds__(kThreads)
    cic1d_grad_kernel(Cic1dArgs a, const float *__restrict__ H, double *__restrict__ dx0) {
    __shared__ WarpQueue queues[kWarps];
    __shared__ double ctab_s[kTab];
    const double *ctab = fill_ctab(a, ctab_s);
    __syncthreads();
    const int warp = threadIdx.x >> 5;
    const float nb = (float)a.nbins;
    cic1d_walk<true>(
        a, (long long)blockIdx.x * kWarps + warp, (long long)gridDim.x * kWarps, queues[warp],
        [&](long long p) { dx0[p] = 0.0; },
        [&](float xf, float vf, int t, long long p) {
            Pair pr;
            if (!cic1d_select(a, ctab, xf, vf, t, pr)) return;
            if (!PCG_IN(pr.b0, a.nbins) || !PCG_IN(pr.b1, a.nbins) || !PCG_IN(p, a.n)) return;
            const float dw = -2.f * pr.u * pr.sgn * a.inv_hw32;
            const float G0 = 2.f * (H[pr.b0] - a.target[pr.b0]);
            const float G1 = 2.f * (H[pr.b1] - a.target[pr.b1]);
            atomicAdd(&dx0[p], (double)(G0 * (dw * (1.f - pr.f) - pr.w * nb) + G1 * (dw * pr.f + pr.w * nb)));
        });
}

pcg_status check_cic1d_args(const float *x0, const float *v, int64_t n, const float *target, int32_t nbins,
                            int32_t nsteps, double dt, double halfwidth, const float *H, const double *loss) {
    if (n < 0 || nbins < 1 || nbins > 16384 || nsteps < 1) return PCG_ERR_INVALID_ARG;
    if (!(halfwidth > 0.0) || !(dt == dt) || !(halfwidth < 1e300) || !(dt < 1e300 && dt > -1e300))
        return PCG_ERR_INVALID_ARG;
    if (target == nullptr || H == nullptr || loss == nullptr) return PCG_ERR_INVALID_ARG;
    if (n > 0 && (x0 == nullptr || v == nullptr)) return PCG_ERR_INVALID_ARG;
    return PCG_OK;
}

Cic1dArgs make_args(const float *x0, const float *v, int64_t n, const float *target, int32_t nbins,
                    int32_t nsteps, double dt, double halfwidth) {
    Cic1dArgs a;
    a.x0 = x0;
    a.v = v;
    a.n = (long long)n;
    a.target = target;
    a.nbins = nbins;
    a.nsteps = nsteps;
    a.dt = dt;
    a.hw = halfwidth;
    a.inv_hw32 = (float)(1.0 / halfwidth);
    a.dt32 = (float)dt;
    a.hw32 = (float)halfwidth;
    a.inv_t32 = 1.0f / (float)nsteps;
    return a;
}

// CTAs of a full grid for the large-N kernels: enough to cover the 32-particle
// chunks, at most what is resident on all SMs at once and at most max_per_sm
// per SM (2 per SM for the histogram, to flush fewer copies of H, was 1.37x
// slower at N = 10^7 than a full grid).
int full_grid(const void *kernel, size_t smem, long long n, int max_per_sm) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    if (per_sm > max_per_sm) per_sm = max_per_sm;
    const long long need = (n + kThreads - 1) / kThreads;
    const long long cap = (long long)num_sms() * per_sm;
    return (int)(need < cap ? (need < 1 ? 1 : need) : cap);
}

pcg_status cic1d_forward(const Cic1dArgs &a, float *H, double *loss, cudaStream_t s) {
    const size_t smem = (size_t)a.nbins * sizeof(float);
    // the shared histogram plus the static queues can exceed the 48 KB default
    static const bool opted_in = [] {
        const int max_dyn = 16384 * (int)sizeof(float);
        return cudaFuncSetAttribute(cic1d_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    max_dyn) == cudaSuccess &&
               cudaFuncSetAttribute(cic1d_hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    max_dyn) == cudaSuccess;
    }();
    if (!opted_in) return PCG_ERR_CUDA;
    if (a.n <= kClusterMaxN) {
        prof::Mark mk("cic1d", s);
        cic1d_cluster_kernel<<<kCtas, kThreads, smem, s>>>(a, H, loss);
        return launch_status();
    }
    prof::Mark mk("cic1d", s);
    PCG_CHECK_CUDA(cudaMemsetAsync(H, 0, (size_t)a.nbins * sizeof(float), s));
    const int grid = full_grid((const void *)cic1d_hist_kernel, smem, a.n, 8);
    cic1d_hist_kernel<<<grid, kThreads, smem, s>>>(a, H);
    PCG_CHECK_CUDA(cudaGetLastError());
    cic1d_loss_kernel<<<1, kThreads, 0, s>>>(H, a.target, a.nbins, loss);
    return launch_status();
}

}  // namespace
}  // namespace pcg

extern "C" pcg_status pcg_deposit_cic1d(const float *x0, const float *v, int64_t n,
                                        const float *target, int32_t nbins, int32_t nsteps,
                                        double dt, double halfwidth, float *H, double *loss,
                                        void *stream) {
    using namespace pcg;
    const pcg_status st = check_cic1d_args(x0, v, n, target, nbins, nsteps, dt, halfwidth, H, loss);
    if (st != PCG_OK) return st;
    return cic1d_forward(make_args(x0, v, n, target, nbins, nsteps, dt, halfwidth), H, loss, as_stream(stream));
}

extern "C" pcg_status pcg_deposit_cic1d_grad(const float *x0, const float *v, int64_t n,
                                             const float *target, int32_t nbins, int32_t nsteps,
                                             double dt, double halfwidth, float *H, double *loss,
                                             double *dx0, void *stream) {
    using namespace pcg;
    pcg_status st = check_cic1d_args(x0, v, n, target, nbins, nsteps, dt, halfwidth, H, loss);
    if (st != PCG_OK) return st;
    if (n > 0 && dx0 == nullptr) return PCG_ERR_INVALID_ARG;
    const Cic1dArgs a = make_args(x0, v, n, target, nbins, nsteps, dt, halfwidth);
    const cudaStream_t s = as_stream(stream);
    st = cic1d_forward(a, H, loss, s);
    if (st != PCG_OK || n == 0) return st;
    prof::Mark mk("cic1d_grad", s);
    const int grid = full_grid((const void *)cic1d_grad_kernel, 0, a.n, 8);
    cic1d_grad_kernel<<<grid, kThreads, 0, s>>>(a, H, dx0);
    return launch_status();
}
