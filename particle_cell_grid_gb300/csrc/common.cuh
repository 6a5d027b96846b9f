// common.cuh -- shared device/host helpers of the deposit library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pcg.h"
#include "checked.cuh"
#include "profile.cuh"

#define PCG_VERSION_NUMBER 100  // 0.1.0

namespace pcg {

// SMs of the current device (152 on a full GB300: 2 dies x 76), cached per
// device; grids are sized in multiples of it and persistent grids equal it.
inline int num_sms() {
    constexpr int kMaxDev = 64;
    static int cache[kMaxDev] = {0};  // benign race: every writer stores the same value
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
        (void)cudaGetLastError();
        return 152;
    }
    if (cache[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
            (void)cudaGetLastError();
            v = 152;
        }
        cache[dev] = v;
    }
    return cache[dev];
}

inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

// Map the last CUDA error (launch configuration errors are synchronous) to a status.
inline pcg_status launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? PCG_OK : PCG_ERR_CUDA;
}

#define PCG_CHECK_CUDA(call)                          \
    do {                                              \
        if ((call) != cudaSuccess) {                  \
            (void)cudaGetLastError();                 \
            return PCG_ERR_CUDA;                      \
        }                                             \
    } while (0)

#define PCG_CHECK_LAUNCH()                            \
    do {                                              \
        pcg_status _s = ::pcg::launch_status();       \
        if (_s != PCG_OK) return _s;                  \
    } while (0)

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Periodic tile geometry shared by the sort and the tiled deposit.
struct TileGrid {
    int dim;
    int N[3];   // nodes (= cells) per axis; 1 on unused axes
    int nt[3];  // tiles per axis, ceil(N / tile)
    int tile;
    long long n_tiles;
};

inline bool make_tile_grid(int dim, const int32_t *grid, int tile, TileGrid *g) {
    if (dim != 2 && dim != 3) return false;
    if (grid == nullptr || tile < 1) return false;
    g->dim = dim;
    g->tile = tile;
    long long total = 1, cells = 1;
    for (int mu = 0; mu < 3; ++mu) {
        int N = mu < dim ? grid[mu] : 1;
        if (N < 1 || N > (1 << 20)) return false;
        g->N[mu] = N;
        g->nt[mu] = (N + tile - 1) / tile;
        total *= g->nt[mu];
        cells *= N;
    }
    if (cells >= (1ll << 31) || total + 1 >= (1ll << 31)) return false;
    g->n_tiles = total;
    return true;
}

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }

// Add `v` to a 64-bit counter once per warp (the active lanes' values summed).
__device__ __forceinline__ void warp_add_u64(unsigned long long *ctr, unsigned v) {
    unsigned mask = __activemask();
    unsigned sum = __reduce_add_sync(mask, v);
    int leader = __ffs(mask) - 1;
    if (lane_id() == leader && sum != 0 && ctr != nullptr) atomicAdd(ctr, (unsigned long long)sum);
}

// Fire-and-forget fp32 reduction into global memory (red.global.add.f32).
__device__ __forceinline__ void red_add_f32(float *addr, float v) {
    asm volatile("red.relaxed.gpu.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

// Vector reductions (sm_90+): 8- and 16-byte aligned addresses only.
__device__ __forceinline__ void red_add_v2_f32(float *addr, float a, float b) {
    asm volatile("red.relaxed.gpu.global.add.v2.f32 [%0], {%1, %2};" ::"l"(addr), "f"(a), "f"(b)
                 : "memory");
}
__device__ __forceinline__ void red_add_v4_f32(float *addr, float a, float b, float c, float d) {
    asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a),
                 "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// Ask for [p, p + bytes) to be brought into L2 (bytes a multiple of 16, p 16-byte aligned).
__device__ __forceinline__ void prefetch_l2_bulk(const void *p, unsigned bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Fire-and-forget fp32 add into shared memory (red.shared.add.f32).
__device__ __forceinline__ void red_shared_add_f32(float *addr, float v) {
    unsigned a = static_cast<unsigned>(__cvta_generic_to_shared(addr));
    asm volatile("red.shared.add.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}

__device__ __forceinline__ int wrap_index(int i, int N) {
    i %= N;
    return i < 0 ? i + N : i;
}

}  // namespace pcg

// Host-side launchers implemented in the .cu files (internal linkage across TUs).
namespace pcg {
pcg_status zero_f32(float *p, size_t count, cudaStream_t s);
}
