// api.cu -- version, status strings, stats check, the index-check counters
// and the fill kernel.
#include <mutex>

#include "common.cuh"

namespace pcg {

namespace {
std::mutex g_check_mu;
CheckReader g_check_readers[64];
int g_check_n = 0;
}  // namespace

int check_register(CheckReader reader) {
    std::lock_guard<std::mutex> lock(g_check_mu);
    if (g_check_n < 64) g_check_readers[g_check_n++] = reader;
    return g_check_n;
}

// Grid-stride zero fill; 16-byte stores on the aligned body.
__global__ void __launch_bounds__(256) zero_f32_kernel(float *__restrict__ p, size_t count) {
    size_t head = (16 - (reinterpret_cast<uintptr_t>(p) & 15)) / 4 % 4;
    if (head > count) head = count;
    size_t tid = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
    size_t stride = (size_t)gridDim.x * blockDim.x;
    if (tid < head) p[tid] = 0.f;
    float4 *q = reinterpret_cast<float4 *>(p + head);
    size_t nvec = (count - head) / 4;
    for (size_t i = tid; i < nvec; i += stride) q[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    size_t tail0 = head + nvec * 4;
    if (tid < count - tail0) p[tail0 + tid] = 0.f;
}

pcg_status zero_f32(float *p, size_t count, cudaStream_t s) {
    if (count == 0) return PCG_OK;
    size_t vec = count / 4 + 1;
    size_t blocks = (vec + 255) / 256;
    size_t cap = (size_t)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    prof::Mark mk("zero_f32", s);
    zero_f32_kernel<<<(unsigned)blocks, 256, 0, s>>>(p, count);
    return launch_status();
}

}  // namespace pcg

extern "C" int pcg_version(void) { return PCG_VERSION_NUMBER; }

extern "C" const char *pcg_status_string(int status) {
    switch (status) {
        case PCG_OK: return "ok";
        case PCG_ERR_INVALID_ARG: return "invalid argument";
        case PCG_ERR_WORKSPACE: return "workspace too small";
        case PCG_ERR_UNSUPPORTED: return "unsupported configuration";
        case PCG_ERR_CUDA: return "CUDA error";
        case PCG_ERR_TIMEOUT: return "device-side wait timed out";
        case PCG_ERR_DOMAIN: return "invalid particles or layout reported in stats";
        default: return "unknown status";
    }
}

extern "C" pcg_status pcg_stats_check(const pcg_stats *s) {
    if (s == nullptr) return PCG_ERR_INVALID_ARG;
    if (s->n_invalid != 0 || s->error_flags != 0) return PCG_ERR_DOMAIN;
    return PCG_OK;
}

extern "C" pcg_status pcg_bounds_check_failures(uint64_t *failures, int32_t *checked_build) {
    if (failures == nullptr) return PCG_ERR_INVALID_ARG;
#ifdef PCG_CHECKED
    const int32_t checked = 1;
#else
    const int32_t checked = 0;
#endif
    if (checked_build) *checked_build = checked;
    uint64_t total = 0;
    if (checked) {
        if (cudaDeviceSynchronize() != cudaSuccess) {
            (void)cudaGetLastError();
            return PCG_ERR_CUDA;
        }
        std::lock_guard<std::mutex> lock(pcg::g_check_mu);
        for (int i = 0; i < pcg::g_check_n; ++i) total += pcg::g_check_readers[i]();
    }
    *failures = total;
    return PCG_OK;
}
