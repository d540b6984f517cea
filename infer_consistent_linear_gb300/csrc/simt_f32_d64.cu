// SIMT_F32 kernels instantiated for io dtype float and d_k = d_v = 64.
#include "simt_launch.cuh"

namespace cpr {
CPR_DEFINE_SIMT_OPS(simt_ops_f32_d64, float, 64)
}  // namespace cpr
