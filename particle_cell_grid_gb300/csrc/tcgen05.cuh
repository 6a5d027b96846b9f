// tcgen05.cuh -- inline-PTX wrappers for the 5th-generation tensor cores
// (tcgen05.*), tensor memory and mbarriers on sm_100-family GPUs (sm_103a).
//
// Shared-memory matrix descriptors describe operands in the canonical K-major
// layout without swizzling: the operand is tiled into "core matrices" of
// 8 rows x 16 bytes (128 contiguous bytes, rows 16 bytes apart); LBO is the byte
// distance between core matrices adjacent along K, SBO the distance between
// core matrices adjacent along M (or N).
#pragma once

#include <stdint.h>

namespace pcg {
namespace tc {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 64-bit shared-memory descriptor, no swizzle, sm_100 descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
    // base offset 0, LBO mode 0, layout type 0 (no swizzle)
    return d;
}

// 64-bit shared-memory descriptor for a K-major operand in the 128-byte swizzled
// layout: 8-row atoms of 8 x 128 bytes (1024 bytes, 1024-byte aligned), the 16-byte
// chunk c of row r stored at chunk c ^ (r % 8); SBO = distance between 8-row atoms.
// One MMA reads 32 bytes of K from each row, starting `saddr` bytes into the atom.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)1 << 16;  // leading byte offset: unused for swizzled K-major operands
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;  // layout type: 128-byte swizzle
    return d;
}

// Instruction descriptor for kind::tf32 / kind::f16: D fp32, A and B K-major.
// fmt: 1 = BF16 (kind::f16), 2 = TF32 (kind::tf32).
__host__ __device__ constexpr uint32_t instr_desc(uint32_t fmt, uint32_t M, uint32_t N) {
    return (1u << 4)              // D format: F32
           | (fmt << 7)           // A format
           | (fmt << 10)          // B format
           | ((N >> 3) << 17)     // N / 8
           | ((M >> 4) << 24);    // M / 16
}

// ---- tensor memory --------------------------------------------------------
// Allocate `ncols` TMEM columns (power of two >= 32); one full warp executes it.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (the tensor core reads operands through it).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]; issued by one thread.
template <bool TF32>
__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                    uint32_t idesc, bool accumulate) {
    const uint32_t acc = accumulate ? 1u : 0u;
    if (TF32) {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(acc)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(acc)
            : "memory");
    }
}

// Arrive once on `mbar` when every previously issued tcgen05.mma of this thread completes.
__device__ __forceinline__ void commit(uint64_t *mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(mbar))
                 : "memory");
}

// Warp-collective load of 8 consecutive 32-bit TMEM columns for the warp's 32 lanes.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
    uint32_t r[8];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// Warp-collective load of 8 consecutive 32-bit TMEM columns without waiting;
// the registers are valid only after tmem_wait_ld(...) on them.
__device__ __forceinline__ void tmem_ld8_async(uint32_t taddr, uint32_t *r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7])
        : "r"(taddr)
        : "memory");
}

// Warp-collective load of 4 consecutive 32-bit TMEM columns without waiting.
__device__ __forceinline__ void tmem_ld4_async(uint32_t taddr, uint32_t *r) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr)
                 : "memory");
}

// Wait for this thread's outstanding tcgen05.ld, then pin every register of `r`
// behind the wait (an empty volatile asm per register), so that no use of a
// loaded value is scheduled before the data has arrived.
template <int NR>
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[NR]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < NR; ++i) asm volatile("" : "+r"(r[i]));
}

// ---- bulk asynchronous copies (TMA engine, no tensor map) ------------------
// dst[0..bytes) += src[0..bytes) element-wise in fp32, global <- shared; both
// addresses 16-byte aligned, bytes a multiple of 16.  Completion is tracked by
// the issuing thread's bulk groups.
__device__ __forceinline__ void bulk_reduce_add_f32(float *gdst, const float *ssrc, uint32_t bytes) {
    asm volatile(
        "cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(gdst),
        "r"(smem_addr(ssrc)), "r"(bytes)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until the committed bulk groups have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Wait until the committed bulk groups have completed.
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ---- mbarrier -------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *mbar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(mbar)), "r"(count)
                 : "memory");
}

// Arrive once on `mbar` (release at CTA scope).
__device__ __forceinline__ void mbar_arrive(uint64_t *mbar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(mbar)) : "memory");
}

// Wait for the phase with the given parity to complete.  Gives up after
// `max_polls` polls and returns false (the caller records a timeout).
__device__ __forceinline__ bool mbar_wait(uint64_t *mbar, uint32_t parity, uint32_t max_polls) {
    const uint32_t a = smem_addr(mbar);
    for (uint32_t i = 0; i < max_polls; ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.b32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(a), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}

// As mbar_wait, but each poll lets the hardware suspend the thread for up to
// `hint_ns` nanoseconds until the phase completes, instead of spinning: waiting
// warps then take no issue slots from the warps doing work.  Gives up after
// `max_polls` polls (a bound of at most max_polls * hint_ns).
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t *mbar, uint32_t parity, uint32_t max_polls,
                                                uint32_t hint_ns) {
    const uint32_t a = smem_addr(mbar);
    for (uint32_t i = 0; i < max_polls; ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.b32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(a), "r"(parity), "r"(hint_ns)
            : "memory");
        if (done) return true;
    }
    return false;
}

// fp32 -> tf32 (round to nearest, ties away), kept in a 32-bit container.
__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

}  // namespace tc
}  // namespace pcg
