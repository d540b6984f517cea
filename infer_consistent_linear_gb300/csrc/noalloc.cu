// Allocation-free trainer forward (cpr_gdn_fwd_noalloc, see cpr_gdn.h).
//
// Some callers cannot call cudaMalloc where they need the forward: host
// callbacks and allocator hooks (where allocating is forbidden or would
// deadlock), or embedders with fixed memory pools.  This entry point gives
// them the forward with its scratch in a file-scope device array instead of a
// caller workspace, and then runs the ordinary cpr_gdn_fwd path unchanged.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <mutex>
#include <utility>

#include "cpr_gdn.h"

namespace cpr {
int record_error(int code, const char* fmt, ...);
}

namespace {

// The scratch.  In host code this name is only a stand-in for the device
// symbol; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[CPR_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Unique id of the calling thread's current CUDA context (0 when the driver does
// not offer the query).  A device reset destroys the context, and with it the
// module holding the scratch; the next context on that device gets another id.
unsigned long long current_context_id() {
    static const auto fns = [] {
        void* get = nullptr;
        void* id = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &get, 4000, cudaEnableDefault, &q) !=
                cudaSuccess || q != cudaDriverEntryPointSuccess)
            get = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &id, 12000, cudaEnableDefault, &q) !=
                cudaSuccess || q != cudaDriverEntryPointSuccess)
            id = nullptr;
        return std::make_pair(reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(get),
                              reinterpret_cast<PFN_cuCtxGetId_v12000>(id));
    }();
    CUcontext ctx = nullptr;
    unsigned long long cid = 0;
    if (!fns.first || !fns.second || fns.first(&ctx) != CUDA_SUCCESS || !ctx ||
        fns.second(ctx, &cid) != CUDA_SUCCESS)
        return 0;
    return cid;
}

// Device address of the scratch for the current device.  It is looked up with
// cudaGetSymbolAddress once per device -- with that device current -- and again
// whenever the device's context has changed since (after cudaDeviceReset the old
// address would point into a destroyed module).  Returns nullptr on failure.
void* scratch_for_current_device(cudaError_t* why) {
    static std::mutex mu;
    static void* addr[kMaxDevices] = {nullptr};
    static unsigned long long ctx_of[kMaxDevices] = {0};
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *why = e != cudaSuccess ? e : cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    // (the query makes the runtime create the device's context if it has none yet)
    void* p = nullptr;
    const bool fresh = addr[dev] == nullptr;
    if (fresh) {
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            *why = e != cudaSuccess ? e : cudaErrorInvalidSymbol;
            return nullptr;
        }
    }
    const unsigned long long cid = current_context_id();
    if (!fresh && cid != ctx_of[dev]) {   // a new context since the set-up: look up again
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            *why = e != cudaSuccess ? e : cudaErrorInvalidSymbol;
            return nullptr;
        }
    }
    if (p) {
        addr[dev] = p;
        ctx_of[dev] = cid;
    }
    return addr[dev];
}

}  // namespace

extern "C" int cpr_gdn_fwd_noalloc(const cpr_contract* c, const uint8_t digest[32],
                                   const void* q, const void* k, const void* v, const float* g,
                                   const float* beta, const int32_t* cu_seqlens, int n_seq,
                                   int64_t n_tok, int H, const float* h0, void* o,
                                   float* final_state, void* stream) {
    size_t need = 0;
    int rc = cpr_gdn_workspace_size(c, CPR_OP_FWD, n_seq, n_tok, H, &need);
    if (rc != CPR_OK) return rc;
    if (need > (size_t)CPR_NOALLOC_SCRATCH_BYTES)
        return cpr::record_error(CPR_ERR_WORKSPACE,
                                 "cpr_gdn_fwd_noalloc: this batch needs %zu bytes of scratch but the "
                                 "built-in scratch holds %u bytes; use cpr_gdn_fwd with a workspace "
                                 "or split the batch",
                                 need, (unsigned)CPR_NOALLOC_SCRATCH_BYTES);
    cudaError_t why = cudaSuccess;
    void* scratch = scratch_for_current_device(&why);
    if (!scratch)
        return cpr::record_error(CPR_ERR_CUDA, "cpr_gdn_fwd_noalloc: scratch address lookup failed: %s",
                                 cudaGetErrorString(why));
    return cpr_gdn_fwd(c, digest, q, k, v, g, beta, cu_seqlens, n_seq, n_tok, H, h0, o,
                       final_state, scratch, (size_t)CPR_NOALLOC_SCRATCH_BYTES, stream);
}
