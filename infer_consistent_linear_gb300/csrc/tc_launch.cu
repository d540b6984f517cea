// Launch sequences of the TC_BF16X3 policy (tensor-core prep, state pass and
// decode; bf16 io, d = 128).
#include "profile.h"
#include "tc_bwd.cuh"
#include "tc_decode.cuh"
#include "tc_launch.h"

namespace cpr {

namespace {

template <class K>
cudaError_t set_smem(K kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

int sm_count() {
    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return nsm;
}

// PERSIST: the reading-B commit, one CTA per SM walking the units.
template <int DVS, bool PERSIST>
cudaError_t state(const tc::TcArgs& a, int n_seq, int H, cudaStream_t st) {
    auto kern = tc::k_tc_state<DVS, PERSIST>;
    const size_t sm = tc::StateSmem<DVS>::Total;
    cudaError_t e = set_smem(kern, sm);
    if (e != cudaSuccess) return e;
    int64_t grid = (int64_t)n_seq * H * (tc::D / DVS);
    if (PERSIST) {
        const int nsm = sm_count();
        if (nsm <= 0) return cudaErrorInvalidDevice;
        grid = grid < nsm ? grid : nsm;
    }
    if (grid > 0) {
        ProfScope ps(PERSIST ? "cpr_tc_commit_state" : "cpr_tc_state", st);
        kern<<<(unsigned)grid, tc::kStateThreads, sm, st>>>(a);
    }
    return cudaGetLastError();
}

template <int DVS>
cudaError_t cache_tiles(const tc::TcArgs& a, int n_seq, int H, cudaStream_t st) {
    const int64_t grid = (int64_t)n_seq * H;
    if (grid > 0) {
        ProfScope ps("cpr_tc_cache_tiles", st);
        tc::k_tc_cache_tiles<DVS><<<(unsigned)grid, 256, 0, st>>>(a.cache, a.co, a.chunk_off, n_seq, H);
    }
    return cudaGetLastError();
}

template <int DVS>
cudaError_t decode(const tc::TcDecArgs& a, cudaStream_t st) {
    auto kern = tc::k_tc_decode<DVS>;
    const size_t sm = tc::DecSmem::Total;
    cudaError_t e = set_smem(kern, sm);
    if (e != cudaSuccess) return e;
    // persistent: one CTA per SM walks the (sequence, head) units
    int dev = 0, nsm = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int64_t units = (int64_t)a.n_seq * a.H;
    const int64_t grid = units < nsm ? units : nsm;
    if (grid > 0) {
        ProfScope ps("cpr_tc_decode", st);
        kern<<<(unsigned)grid, tc::kDecThreads, sm, st>>>(a);
    }
    return cudaGetLastError();
}

template <int DVS>
cudaError_t state_bwd(const tc::TcBwdArgs& a, int n_seq, int H, cudaStream_t st) {
    auto kern = tc::k_tc_state_bwd<DVS>;
    const size_t sm = tc::SbSmem<DVS>::Total;
    cudaError_t e = set_smem(kern, sm);
    if (e != cudaSuccess) return e;
    const int64_t grid = (int64_t)n_seq * H * (tc::D / DVS);
    if (grid > 0) {
        ProfScope ps("cpr_tc_state_bwd", st);
        kern<<<(unsigned)grid, 256, sm, st>>>(a);
    }
    return cudaGetLastError();
}

// The timeout path of the bounded waits: one thread waits on an mbarrier that
// nothing arrives on, with a short poll limit; it records CPR_ERR_DEVICE_TIMEOUT,
// the kernel returns and the context stays usable.
__global__ void k_wait_timeout(uint32_t* err, uint32_t limit, uint32_t* ok_out) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    tc::mbar_init(&bar, 1);
    tc::mbar_init_fence();
    const bool ok = tc::mbar_wait_n(&bar, 0, err, limit);
    *ok_out = ok ? 1u : 0u;
}

}  // namespace

cudaError_t tc_wait_timeout_selftest(uint32_t* err, uint32_t limit, uint32_t* ok_out, cudaStream_t st) {
    k_wait_timeout<<<1, 32, 0, st>>>(err, limit, ok_out);
    return cudaGetLastError();
}

cudaError_t tc_forward(const tc::TcArgs& a, int64_t cmax, int n_seq, int H, cudaStream_t st) {
    cudaError_t e = set_smem(tc::k_tc_prep<false>, tc::kPrepSmem);
    if (e != cudaSuccess) return e;
    if (cmax > 0) {
        ProfScope ps("cpr_tc_prep", st);
        tc::k_tc_prep<false><<<dim3((unsigned)cmax, H), 128, tc::kPrepSmem, st>>>(a);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    switch (a.dvs) {
        case 64: e = state<64, false>(a, n_seq, H, st); break;
        case 32: e = state<32, false>(a, n_seq, H, st); break;
        default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess || !a.cache) return e;
    return a.dvs == 64 ? cache_tiles<64>(a, n_seq, H, st) : cache_tiles<32>(a, n_seq, H, st);
}

cudaError_t tc_commit(const tc::TcArgs& a, int n_seq, int H, cudaStream_t st) {
    if (!a.commit_pos || !a.commit_header) return cudaErrorInvalidValue;
    cudaError_t e = set_smem(tc::k_tc_prep<true>, tc::kPrepSmem);
    if (e != cudaSuccess) return e;
    const int nsm = sm_count();
    if (nsm <= 0) return cudaErrorInvalidDevice;
    const int64_t units = (int64_t)n_seq * H;
    const int64_t grid = units < nsm ? units : nsm;
    if (grid > 0) {
        ProfScope ps("cpr_tc_commit_prep", st);
        tc::k_tc_prep<true><<<(unsigned)grid, 128, tc::kPrepSmem, st>>>(a);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    switch (a.dvs) {
        case 64: return state<64, true>(a, n_seq, H, st);
        case 32: return state<32, true>(a, n_seq, H, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t tc_decode_step(const tc::TcDecArgs& a, int dvs, cudaStream_t st) {
    switch (dvs) {
        case 64: return decode<64>(a, st);
        case 32: return decode<32>(a, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t tc_backward(const tc::TcArgs& f, const tc::TcBwdArgs& b, int64_t cmax, int n_seq, int H,
                        cudaStream_t st, bool recompute) {
    cudaError_t e = cudaSuccess;
    if (recompute) {
        e = tc_forward(f, cmax, n_seq, H, st);
        if (e != cudaSuccess) return e;
    }
    switch (f.dvs) {
        case 64: e = state_bwd<64>(b, n_seq, H, st); break;
        case 32: e = state_bwd<32>(b, n_seq, H, st); break;
        default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    e = set_smem(tc::k_tc_grad, tc::GradSmem::Total);
    if (e != cudaSuccess) return e;
    // persistent: one CTA per SM walks the (chunk, head) items
    int dev = 0, nsm = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int64_t items = cmax * (int64_t)H;
    const int grid = (int)(items < nsm ? items : nsm);
    if (grid > 0) {
        ProfScope ps("cpr_tc_grad", st);
        tc::k_tc_grad<<<grid, 256, tc::GradSmem::Total, st>>>(b);
    }
    return cudaGetLastError();
}

}  // namespace cpr
