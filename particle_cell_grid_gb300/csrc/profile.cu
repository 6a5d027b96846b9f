// profile.cu -- per-kernel CUDA-event timing, aggregated by kernel name.
#include <mutex>
#include <string.h>
#include <string>
#include <vector>

#include "common.cuh"
#include "profile.cuh"

namespace pcg {
namespace prof {
namespace {

struct Rec {
    const char *name;
    cudaEvent_t a, b;
    bool closed;
};

std::mutex mu;
bool on = false;
std::vector<Rec> recs;
std::vector<cudaEvent_t> pool;

cudaEvent_t take() {
    if (!pool.empty()) {
        cudaEvent_t e = pool.back();
        pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

}  // namespace

bool enabled() { return on; }

void record(const char *name, cudaStream_t s, bool start) {
    std::lock_guard<std::mutex> g(mu);
    if (start) {
        Rec r{name, take(), take(), false};
        if (r.a) cudaEventRecord(r.a, s);
        recs.push_back(r);
    } else {
        for (auto it = recs.rbegin(); it != recs.rend(); ++it) {
            if (!it->closed && it->name == name) {
                if (it->b) cudaEventRecord(it->b, s);
                it->closed = true;
                break;
            }
        }
    }
}

}  // namespace prof
}  // namespace pcg

extern "C" pcg_status pcg_profile_enable(int32_t enable) {
    std::lock_guard<std::mutex> g(pcg::prof::mu);
    pcg::prof::on = enable != 0;
    return PCG_OK;
}

extern "C" pcg_status pcg_profile_collect(int32_t max_entries, char *names, int64_t *launches,
                                          double *total_ms, int32_t *n_entries) {
    using namespace pcg::prof;
    if (max_entries < 0 || n_entries == nullptr) return PCG_ERR_INVALID_ARG;
    if (max_entries > 0 && (names == nullptr || launches == nullptr || total_ms == nullptr))
        return PCG_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(mu);
    std::vector<std::string> keys;
    std::vector<long long> cnt;
    std::vector<double> ms;
    pcg_status st = PCG_OK;
    for (Rec &r : recs) {
        float t = 0.f;
        if (!r.closed || r.a == nullptr || r.b == nullptr || cudaEventSynchronize(r.b) != cudaSuccess ||
            cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) {
            (void)cudaGetLastError();
            st = PCG_ERR_CUDA;
        } else {
            size_t k = 0;
            while (k < keys.size() && keys[k] != r.name) ++k;
            if (k == keys.size()) {
                keys.push_back(r.name);
                cnt.push_back(0);
                ms.push_back(0.0);
            }
            cnt[k] += 1;
            ms[k] += t;
        }
        if (r.a) pool.push_back(r.a);
        if (r.b) pool.push_back(r.b);
    }
    recs.clear();
    const int m = (int)keys.size() < max_entries ? (int)keys.size() : max_entries;
    for (int i = 0; i < m; ++i) {
        strncpy(names + 64 * i, keys[i].c_str(), 63);
        names[64 * i + 63] = 0;
        launches[i] = cnt[i];
        total_ms[i] = ms[i];
    }
    *n_entries = (int32_t)keys.size();
    return st;
}
