// Launch sequences of the SIMT_F32 policy, instantiated once per (io dtype,
// head dim) in the simt_*.cu translation units.
#pragma once

#include "profile.h"
#include "simt_bwd.cuh"

namespace cpr {

struct LaunchCfg {
    int64_t cmax;       // chunk upper bound: n_tok / C + n_seq
    int n_seq;
    int H;
    int dv_splits;
    cudaStream_t stream;
};

namespace simt {

template <class K>
inline cudaError_t set_smem(K kernel, size_t bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <class IO, int D, int DVS>
cudaError_t launch_state_fwd(const FwdArgs& a, const LaunchCfg& L) {
    auto kern = k_state_fwd<IO, D, D, DVS>;
    const size_t sm = state_fwd_smem<IO, D, D, DVS>();
    cudaError_t e = set_smem(kern, sm);
    if (e != cudaSuccess) return e;
    const int64_t grid = (int64_t)L.n_seq * L.H * (D / DVS);
    if (grid > 0) {
        ProfScope ps("cpr_state_fwd", L.stream);
        kern<<<(unsigned)grid, 256, sm, L.stream>>>(a);
    }
    return cudaGetLastError();
}

template <class IO, int D, int DVS>
cudaError_t launch_state_bwd(const BwdArgs& a, const LaunchCfg& L) {
    auto kern = k_state_bwd<IO, D, D, DVS>;
    const size_t sm = state_bwd_smem<IO, D, D, DVS>();
    cudaError_t e = set_smem(kern, sm);
    if (e != cudaSuccess) return e;
    const int64_t grid = (int64_t)L.n_seq * L.H * (D / DVS);
    if (grid > 0) {
        ProfScope ps("cpr_state_bwd", L.stream);
        kern<<<(unsigned)grid, 256, sm, L.stream>>>(a);
    }
    return cudaGetLastError();
}

template <class IO, int D>
cudaError_t fwd(const FwdArgs& a, const LaunchCfg& L) {
    {
        auto kern = k_prep<IO, D, D>;
        const size_t sm = prep_smem<IO, D, D>();
        cudaError_t e = set_smem(kern, sm);
        if (e != cudaSuccess) return e;
        if (L.cmax > 0) {
            ProfScope ps("cpr_prep", L.stream);
            kern<<<dim3((unsigned)L.cmax, L.H), 256, sm, L.stream>>>(a);
        }
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    switch (L.dv_splits) {
        case 1: return launch_state_fwd<IO, D, D>(a, L);
        case 2: return launch_state_fwd<IO, D, D / 2>(a, L);
        case 4: return launch_state_fwd<IO, D, D / 4>(a, L);
        default: return cudaErrorInvalidValue;
    }
}

template <class IO, int D>
cudaError_t bwd(const FwdArgs& fa, const BwdArgs& ba, const LaunchCfg& L) {
    cudaError_t e = fwd<IO, D>(fa, L);  // prep (with T, Kd) + state pass storing H_n
    if (e != cudaSuccess) return e;
    switch (L.dv_splits) {
        case 1: e = launch_state_bwd<IO, D, D>(ba, L); break;
        case 2: e = launch_state_bwd<IO, D, D / 2>(ba, L); break;
        case 4: e = launch_state_bwd<IO, D, D / 4>(ba, L); break;
        default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    auto kern = k_grad_chunk<IO, D, D>;
    const size_t sm = grad_chunk_smem<IO, D, D>();
    e = set_smem(kern, sm);
    if (e != cudaSuccess) return e;
    if (L.cmax > 0) {
        ProfScope ps("cpr_grad_chunk", L.stream);
        kern<<<dim3((unsigned)L.cmax, L.H), 256, sm, L.stream>>>(ba);
    }
    return cudaGetLastError();
}

template <class IO, int D>
cudaError_t decode(const DecArgs& a, const LaunchCfg& L) {
    const int64_t grid = (int64_t)L.n_seq * L.H;
    if (grid > 0) {
        ProfScope ps("cpr_decode", L.stream);
        k_decode<IO, D, D><<<(unsigned)grid, 128, 0, L.stream>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace simt

// One table of launchers per (io dtype, head dim).
struct SimtOps {
    cudaError_t (*fwd)(const simt::FwdArgs&, const LaunchCfg&);
    cudaError_t (*bwd)(const simt::FwdArgs&, const simt::BwdArgs&, const LaunchCfg&);
    cudaError_t (*decode)(const simt::DecArgs&, const LaunchCfg&);
};

const SimtOps* simt_ops_bf16_d64();
const SimtOps* simt_ops_bf16_d128();
const SimtOps* simt_ops_f32_d64();

#define CPR_DEFINE_SIMT_OPS(NAME, IO, D)                                              \
    const SimtOps* NAME() {                                                            \
        static const SimtOps ops = {&simt::fwd<IO, D>, &simt::bwd<IO, D>,              \
                                    &simt::decode<IO, D>};                             \
        return &ops;                                                                   \
    }

}  // namespace cpr
