// profile.cuh -- optional per-kernel timing with CUDA events on the launching stream.
#pragma once

#include <cuda_runtime.h>

namespace pcg {
namespace prof {

bool enabled();
void record(const char *name, cudaStream_t s, bool start);

// Brackets one kernel launch: an event before it and one after it, recorded on
// the launch stream, only while profiling is enabled.
struct Mark {
    const char *name;
    cudaStream_t s;
    bool on;
    Mark(const char *n, cudaStream_t st) : name(n), s(st), on(enabled()) {
        if (on) record(name, s, true);
    }
    ~Mark() {
        if (on) record(name, s, false);
    }
};

}  // namespace prof
}  // namespace pcg
