// Kernel timing hook: CUDA events around library launches while enabled.
#pragma once
#include <cuda_runtime.h>

namespace cpr {

// Records an event pair around the enclosed launch(es) on `stream` when
// profiling is enabled; does nothing otherwise.
class ProfScope {
public:
    ProfScope(const char* name, cudaStream_t stream);
    ~ProfScope();
    ProfScope(const ProfScope&) = delete;
    ProfScope& operator=(const ProfScope&) = delete;

private:
    int slot_;
    cudaStream_t stream_;
};

}  // namespace cpr
