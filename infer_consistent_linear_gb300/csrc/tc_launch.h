// Host entry points of the TC_BF16X3 kernels (defined in tc_launch.cu).
#pragma once
#include <cuda_runtime.h>

#include "tc_fwd.cuh"

namespace cpr {
namespace tc {
struct TcDecArgs;
}
// setup must already have run on `st`; a.dvs selects the state-pass split width.
cudaError_t tc_forward(const tc::TcArgs& a, int64_t cmax, int n_seq, int H, cudaStream_t st);
cudaError_t tc_decode_step(const tc::TcDecArgs& a, int dvs, cudaStream_t st);
}  // namespace cpr
