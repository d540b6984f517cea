// SIMT_F32 kernels instantiated for io dtype __nv_bfloat16 and d_k = d_v = 64.
#include "simt_launch.cuh"

namespace cpr {
CPR_DEFINE_SIMT_OPS(simt_ops_bf16_d64, __nv_bfloat16, 64)
}  // namespace cpr
