// Batch-invariant projection GEMM (see gemm.cu).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace cpr {
namespace gemm {

struct GemmArgs {
    const __nv_bfloat16* X;   // [M, K] row-major
    const __nv_bfloat16* W;   // [K, N] row-major
    float* Y;                 // [M, N] row-major
    int M, N, K;
    int leaf_k;               // K rows per leaf: a multiple of 64 dividing K, K / leaf_k in {1, 2, 4}
    uint32_t* err;
};

}  // namespace gemm

cudaError_t gemm_launch(const gemm::GemmArgs& a, cudaStream_t st);

}  // namespace cpr
