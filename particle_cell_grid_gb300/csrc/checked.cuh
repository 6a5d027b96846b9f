// checked.cuh -- optional index checks of the kernels.
//
// Built with -DPCG_CHECKED (the checked library, particle_cell_grid_gb300/
// _build_checked/libpcg.so), PCG_IN(i, n) tests 0 <= i < n for the
// data-dependent indices of the kernels (from positions, offsets, counts and
// ranks) before the access they guard; a failed test adds one to a device
// counter and the access is skipped.  Nothing traps or asserts.
// pcg_bounds_check_failures() returns the count (summed over the library's
// translation units, each of which keeps its own counter) and resets it.
// Without PCG_CHECKED, PCG_IN is `true` and no check is compiled.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace pcg {

// Host registry of the per-translation-unit counter readers (api.cu).
typedef unsigned long long (*CheckReader)(void);
int check_register(CheckReader reader);

#ifdef PCG_CHECKED
namespace {
__device__ unsigned long long g_check_failures;  // this translation unit's counter

__device__ __noinline__ bool check_failed() {
    atomicAdd(&g_check_failures, 1ull);
    return false;
}

// The counter's value, then zero (host; synchronises the device).
unsigned long long check_read_reset() {
    unsigned long long v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_check_failures, sizeof(v)) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    (void)cudaMemcpyToSymbol(g_check_failures, &z, sizeof(z));
    return v;
}
const int g_check_registered = check_register(&check_read_reset);
}  // namespace
#define PCG_IN(i, n) \
    (((unsigned long long)(long long)(i) < (unsigned long long)(long long)(n)) ? true : ::pcg::check_failed())
#else
#define PCG_IN(i, n) true
#endif

}  // namespace pcg
