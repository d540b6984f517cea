// SIMT_F32 kernels instantiated for io dtype __nv_bfloat16 and d_k = d_v = 128.
#include "simt_launch.cuh"

namespace cpr {
CPR_DEFINE_SIMT_OPS(simt_ops_bf16_d128, __nv_bfloat16, 128)
}  // namespace cpr
