// C ABI of the CPR Gated DeltaNet library: contract handling, argument and
// claim checks, workspace / cache layouts and kernel dispatch.  Declarations
// and their documentation are in include/cpr_gdn.h.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "cpr_gdn.h"
#include "profile.h"
#include "sha256.h"
#include "simt_launch.cuh"
#include "tc_decode.cuh"
#include "rec.h"
#include "gemm.h"
#include "tc_launch.h"

namespace {

// Bumped whenever any rounding-relevant detail of a kernel changes.
constexpr uint32_t kKernelBuildId = 3u;

thread_local char g_msg[512] = "";

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return code;
}

}  // namespace

namespace cpr {
// Records a message for cpr_last_error() from other translation units.
int record_error(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return code;
}
}  // namespace cpr

// Device error word: first recorded error code, 0 = none.
__device__ uint32_t g_cpr_device_error = 0u;

namespace {

uint32_t* device_error_ptr() {
    static std::mutex mu;
    static uint32_t* ptrs[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_cpr_device_error) != cudaSuccess) return nullptr;
        ptrs[dev] = static_cast<uint32_t*>(p);
    }
    return ptrs[dev];
}

size_t io_size(uint32_t dt) { return dt == CPR_DTYPE_BF16 ? 2 : 4; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

void serialize(const cpr_contract& c, uint8_t out[76]) {
    static const char tag[17] = "CPR-GDN-CONTRACT";
    std::memcpy(out, tag, 16);
    uint32_t f[15];
    f[0] = c.version; f[1] = c.chunk_size; f[2] = c.d_k; f[3] = c.d_v; f[4] = c.io_dtype;
    f[5] = c.out_dtype; f[6] = c.gate_dtype; f[7] = c.accum_dtype; f[8] = c.state_dtype;
    f[9] = c.operand_policy; f[10] = c.intra_order; f[11] = c.state_schedule;
    f[12] = c.dv_splits;
    std::memcpy(&f[13], &c.scale, 4);
    f[14] = c.kernel_build_id;
    for (int i = 0; i < 15; ++i)
        for (int b = 0; b < 4; ++b) out[16 + 4 * i + b] = (uint8_t)(f[i] >> (8 * b));
}

int check_contract(const cpr_contract* c) {
    if (!c) return fail(CPR_ERR_INVALID_ARG, "contract is NULL");
    if (c->version != CPR_CONTRACT_VERSION) return fail(CPR_ERR_UNSUPPORTED, "contract version %u", c->version);
    if (c->chunk_size != 64) return fail(CPR_ERR_UNSUPPORTED, "chunk_size %u (this build: 64)", c->chunk_size);
    if (c->d_k != c->d_v) return fail(CPR_ERR_UNSUPPORTED, "d_k != d_v");
    if (c->io_dtype == CPR_DTYPE_BF16) {
        if (c->d_k != 64 && c->d_k != 128) return fail(CPR_ERR_UNSUPPORTED, "d_k %u (bf16: 64 or 128)", c->d_k);
    } else if (c->io_dtype == CPR_DTYPE_F32) {
        if (c->d_k != 64) return fail(CPR_ERR_UNSUPPORTED, "d_k %u (fp32 io: 64)", c->d_k);
    } else {
        return fail(CPR_ERR_UNSUPPORTED, "io_dtype %u", c->io_dtype);
    }
    if (c->out_dtype != CPR_DTYPE_F32 || c->gate_dtype != CPR_DTYPE_F32 ||
        c->accum_dtype != CPR_DTYPE_F32 || c->state_dtype != CPR_DTYPE_F32)
        return fail(CPR_ERR_UNSUPPORTED, "out/gate/accum/state dtype must be F32");
    if (c->operand_policy == CPR_POLICY_TC_BF16X3) {
        if (c->io_dtype != CPR_DTYPE_BF16 || c->d_k != 128)
            return fail(CPR_ERR_UNSUPPORTED, "TC_BF16X3 needs bf16 io and d_k = d_v = 128");
        if (c->dv_splits != 2 && c->dv_splits != 4)
            return fail(CPR_ERR_UNSUPPORTED, "TC_BF16X3 needs dv_splits 2 or 4");
    } else if (c->operand_policy != CPR_POLICY_SIMT_F32) {
        return fail(CPR_ERR_UNSUPPORTED, "operand_policy %u", c->operand_policy);
    }
    if (c->intra_order == CPR_ORDER_TOKENREC_V1) {
        if (c->operand_policy != CPR_POLICY_TC_BF16X3)
            return fail(CPR_ERR_UNSUPPORTED, "intra_order TOKENREC_V1 needs the TC_BF16X3 policy");
    } else if (c->intra_order != CPR_ORDER_ROWSEQ_V1) {
        return fail(CPR_ERR_UNSUPPORTED, "intra_order %u", c->intra_order);
    }
    if (c->state_schedule != CPR_SCHED_SEQ_CHUNKS) return fail(CPR_ERR_UNSUPPORTED, "state_schedule %u", c->state_schedule);
    if (c->dv_splits != 1 && c->dv_splits != 2 && c->dv_splits != 4)
        return fail(CPR_ERR_UNSUPPORTED, "dv_splits %u (1, 2 or 4)", c->dv_splits);
    if (!std::isfinite(c->scale)) return fail(CPR_ERR_INVALID_ARG, "scale not finite");
    if (c->kernel_build_id != kKernelBuildId)
        return fail(CPR_ERR_UNSUPPORTED, "kernel_build_id %u (this build: %u)", c->kernel_build_id, kKernelBuildId);
    return CPR_OK;
}

int check_digest(const cpr_contract* c, const uint8_t* digest) {
    int rc = check_contract(c);
    if (rc) return rc;
    if (!digest) return fail(CPR_ERR_INVALID_ARG, "digest is NULL");
    uint8_t buf[76], d[32];
    serialize(*c, buf);
    cpr::sha256(buf, sizeof(buf), d);
    if (std::memcmp(d, digest, 32) != 0)
        return fail(CPR_ERR_CONTRACT_MISMATCH, "digest does not match SHA-256 of the contract");
    return CPR_OK;
}

struct WsLayout {
    size_t chunk_off, W, U, P, gam, T, Kd, Hn, dH, total;
    int64_t cmax;
};

WsLayout ws_layout(const cpr_contract& c, int op, int n_seq, int64_t n_tok, int H) {
    WsLayout w{};
    const size_t C = c.chunk_size, dk = c.d_k, dv = c.d_v;
    w.cmax = n_tok / (int64_t)C + n_seq;
    const size_t ch = (size_t)w.cmax * (size_t)H;
    size_t off = 0;
    auto add = [&](size_t& field, size_t bytes) { field = off; off = align256(off + bytes); };
    add(w.chunk_off, sizeof(int32_t) * (n_seq + 1));
    if (c.operand_policy == CPR_POLICY_TC_BF16X3) {  // per (chunk, head) operand blocks
        // (reading B's forward keeps every chunk's boundary state: the training block)
        const bool keep = op == CPR_OP_BWD || c.intra_order == CPR_ORDER_TOKENREC_V1;
        add(w.W, ch * (keep ? cpr::tc::kBlockTrain : cpr::tc::kBlock));
        w.total = off;
        return w;
    }
    add(w.W, ch * C * dk * 4);
    add(w.U, ch * C * dv * 4);
    add(w.P, ch * C * C * 4);
    add(w.gam, ch * 2 * C * 4);   // gate prefix hi, lo
    if (op == CPR_OP_BWD) {
        add(w.T, ch * C * C * 4);
        add(w.Kd, ch * C * C * 4);
        add(w.Hn, ch * dk * dv * 4);
        add(w.dH, ch * dk * dv * 4);
    }
    w.total = off;
    return w;
}

// Workspace of a reading-B decode commit: a forward of n_seq full chunks under the chunk
// form's own contract (ROWSEQ_V1).
WsLayout commit_ws(const cpr_contract& c, int n_seq, int H) {
    cpr_contract a = c;
    a.intra_order = CPR_ORDER_ROWSEQ_V1;
    return ws_layout(a, CPR_OP_FWD, n_seq, (int64_t)n_seq * (int64_t)c.chunk_size, H);
}

cpr_cache_layout cache_layout(const cpr_contract& c, int n_seq, int H) {
    cpr_cache_layout l{};
    const size_t C = c.chunk_size, dk = c.d_k, dv = c.d_v, io = io_size(c.io_dtype);
    const size_t sh = (size_t)n_seq * H;
    size_t off = 0;
    auto add = [&](size_t& field, size_t bytes) { field = off; off = align256(off + bytes); };
    add(l.header, 256);
    add(l.pos, 4 * (size_t)n_seq);
    add(l.done, 4 * (size_t)n_seq);
    add(l.state, sh * dk * dv * 4);
    add(l.k_rows, sh * C * dk * io);
    add(l.v_rows, sh * C * dv * io);
    add(l.gam_rows, sh * 2 * C * 4);   // gate prefix hi, lo
    add(l.beta_rows, sh * C * 4);
    add(l.t_rows, sh * C * C * 4);
    add(l.delta_rows, sh * C * dv * 4);
    add(l.state_tiles, sh * dk * dv * 4);   // bf16 hi + lo operand tiles of the state
    add(l.delta_tiles, sh * C * dv * 4);    // bf16 hi + lo operand tiles of the Delta rows
    if (c.intra_order == CPR_ORDER_TOKENREC_V1) {
        add(l.run, sh * dk * dv * 4);   // running in-chunk state
        // the current chunk's token rows and the chunk commit's workspace (a forward of
        // n_seq full chunks under the chunk form's own contract)
        add(l.rb_k, sh * C * dk * io);
        add(l.rb_v, sh * C * dv * io);
        add(l.rb_g, sh * C * 4);
        add(l.rb_beta, sh * C * 4);
        add(l.rb_cu, 4 * ((size_t)n_seq + 1));
        add(l.rb_ws, commit_ws(c, n_seq, H).total);
    }
    l.total_bytes = off;
    return l;
}

cpr::CacheOff to_off(const cpr_cache_layout& l) {
    return cpr::CacheOff{l.header, l.pos, l.done, l.state, l.k_rows, l.v_rows,
                         l.gam_rows, l.beta_rows, l.t_rows, l.delta_rows, l.state_tiles, l.delta_tiles};
}

const cpr::SimtOps* ops_for(const cpr_contract& c) {
    if (c.io_dtype == CPR_DTYPE_BF16) return c.d_k == 64 ? cpr::simt_ops_bf16_d64() : cpr::simt_ops_bf16_d128();
    return cpr::simt_ops_f32_d64();
}

cpr::Digest digest_words(const uint8_t* d) {
    cpr::Digest w;
    std::memcpy(w.w, d, 32);
    return w;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(CPR_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// The one -gencode target this library is compiled for (the build passes only it).
constexpr const char* kBuildArch = "sm_103a";

// Deployment identity of the current device: SHA-256 of a canonical text naming what the
// numerical policy runs on (the compiled arch, the device's compute capability and name,
// the CUDA runtime and driver versions, the kernel build).  Worked out once per device.
struct Deployment {
    bool ok = false;
    uint8_t digest[32];
    char text[512];   // the prefix, a device name of up to 255 bytes and the numbers fit
};

int deployment_of_current_device(const Deployment** out) {
    static std::mutex mu;
    static Deployment dep[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "deployment identity: no CUDA device");
    if (dev < 0 || dev >= 64) return fail(CPR_ERR_UNSUPPORTED, "device index %d", dev);
    std::lock_guard<std::mutex> lock(mu);
    Deployment& d = dep[dev];
    if (!d.ok) {
        cudaDeviceProp prop;
        e = cudaGetDeviceProperties(&prop, dev);
        if (e != cudaSuccess) return cuda_fail(e, "deployment identity: device properties");
        int rt = 0, drv = 0;
        e = cudaRuntimeGetVersion(&rt);
        if (e == cudaSuccess) e = cudaDriverGetVersion(&drv);
        if (e != cudaSuccess) return cuda_fail(e, "deployment identity: versions");
        snprintf(d.text, sizeof(d.text),
                 "CPR-GDN-DEPLOYMENT;arch=%s;cc=%d.%d;gpu=%s;cudart=%d;driver=%d;kernel_build_id=%u",
                 kBuildArch, prop.major, prop.minor, prop.name, rt, drv, kKernelBuildId);
        cpr::sha256(d.text, std::strlen(d.text), d.digest);
        d.ok = true;
    }
    *out = &d;
    return CPR_OK;
}

// Header words 10..24 of a decode cache for this contract and batch on the current device.
int header_words(const cpr_contract& c, int n_seq, int H, uint32_t out[cpr::kHdrWords]) {
    out[0] = (uint32_t)n_seq; out[1] = (uint32_t)H; out[2] = c.chunk_size; out[3] = c.d_k;
    out[4] = c.d_v; out[5] = c.operand_policy; out[6] = c.io_dtype;
    const Deployment* d = nullptr;
    const int rc = deployment_of_current_device(&d);
    if (rc) return rc;
    std::memcpy(out + 7, d->digest, 32);
    return CPR_OK;
}

#define REQ_PTR(p)                                                             \
    do {                                                                       \
        if (!(p)) return fail(CPR_ERR_INVALID_ARG, "%s is NULL", #p);          \
        if (!aligned16(p)) return fail(CPR_ERR_ALIGNMENT, "%s not 16-byte aligned", #p); \
    } while (0)
#define REQ_PTR4(p)                                                            \
    do {                                                                       \
        if (!(p)) return fail(CPR_ERR_INVALID_ARG, "%s is NULL", #p);          \
        if (reinterpret_cast<uintptr_t>(p) & 3u) return fail(CPR_ERR_ALIGNMENT, "%s not 4-byte aligned", #p); \
    } while (0)
// Outputs written with whole 32-byte sector stores.
#define REQ_PTR32(p)                                                           \
    do {                                                                       \
        if (reinterpret_cast<uintptr_t>(p) & 31u)                              \
            return fail(CPR_ERR_ALIGNMENT, "%s not 32-byte aligned", #p);      \
    } while (0)
#define OPT_PTR(p)                                                             \
    do {                                                                       \
        if ((p) && !aligned16(p)) return fail(CPR_ERR_ALIGNMENT, "%s not 16-byte aligned", #p); \
    } while (0)

int check_sizes(int n_seq, int64_t n_tok, int H) {
    if (n_seq < 0 || n_tok < 0 || H <= 0) return fail(CPR_ERR_INVALID_ARG, "n_seq/n_tok/H out of range");
    if (n_tok > INT32_MAX) return fail(CPR_ERR_INVALID_ARG, "n_tok exceeds int32 (cu_seqlens is int32)");
    if ((int64_t)n_seq * H > INT32_MAX / 4) return fail(CPR_ERR_INVALID_ARG, "n_seq * H too large");
    return CPR_OK;
}

cudaError_t launch_setup(const cpr::simt::SetupArgs& sa, cudaStream_t st) {
    cpr::ProfScope ps("cpr_setup", st);
    cpr::simt::k_setup<<<1, 256, 0, st>>>(sa);
    return cudaGetLastError();
}

// Shared by cpr_gdn_fwd and cpr_gdn_prefill: one code path, so the trainer
// forward and the engine prefill run identical kernels.
// `train`: also leave the backward's per-chunk tiles in the (CPR_OP_BWD-sized)
// workspace; the kernels and the outputs' arithmetic are the same.
int forward_impl(const cpr_contract* c, const uint8_t* digest, const void* q, const void* k,
                 const void* v, const float* g, const float* beta, const int32_t* cu, int n_seq,
                 int64_t n_tok, int H, const float* h0, void* o, float* final_state, void* cache,
                 void* ws, size_t ws_bytes, void* stream, bool train = false) {
    int rc = check_digest(c, digest);
    if (rc) return rc;
    if (train && c->operand_policy != CPR_POLICY_TC_BF16X3)
        return fail(CPR_ERR_UNSUPPORTED, "training forward: tensor-core operand policy only");
    rc = check_sizes(n_seq, n_tok, H);
    if (rc) return rc;
    REQ_PTR4(cu);
    if (n_tok > 0) {
        REQ_PTR(q); REQ_PTR(k); REQ_PTR(v); REQ_PTR4(g); REQ_PTR4(beta); REQ_PTR(o);
    }
    OPT_PTR(h0); OPT_PTR(final_state); OPT_PTR(cache);
    const WsLayout w = ws_layout(*c, train ? CPR_OP_BWD : CPR_OP_FWD, n_seq, n_tok, H);
    if (!ws || ws_bytes < w.total || (reinterpret_cast<uintptr_t>(ws) & 255u))
        return fail(CPR_ERR_WORKSPACE, "workspace needs %zu bytes, 256-byte aligned", w.total);
    uint32_t* err = device_error_ptr();
    if (!err) return fail(CPR_ERR_CUDA, "device error word unavailable");
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    const cpr_cache_layout cl = cache_layout(*c, n_seq, H);

    cpr::simt::SetupArgs sa{};
    sa.cu = cu; sa.n_seq = n_seq; sa.n_tok = n_tok;
    sa.chunk_off = reinterpret_cast<int32_t*>(wsb + w.chunk_off);
    sa.cache = static_cast<uint8_t*>(cache); sa.co = to_off(cl);
    sa.digest = digest_words(digest); sa.err = err;
    if (cache) {
        rc = header_words(*c, n_seq, H, sa.hdr);
        if (rc) return rc;
    }
    cudaError_t e = launch_setup(sa, st);
    if (e != cudaSuccess) return cuda_fail(e, "setup launch");

    if (c->operand_policy == CPR_POLICY_TC_BF16X3) {
        cpr::tc::TcArgs t{};
        t.q = static_cast<const __nv_bfloat16*>(q); t.k = static_cast<const __nv_bfloat16*>(k);
        t.v = static_cast<const __nv_bfloat16*>(v); t.g = g; t.beta = beta; t.cu = cu;
        t.chunk_off = sa.chunk_off; t.n_seq = n_seq; t.H = H; t.dvs = (int)(c->d_v / c->dv_splits);
        t.scale = c->scale; t.ws = wsb + w.W; t.train = train;
        t.blk_bytes = train ? cpr::tc::kBlockTrain : cpr::tc::kBlock;
        t.h0 = h0; t.o = static_cast<float*>(o);
        t.final_state = final_state; t.cache = static_cast<uint8_t*>(cache); t.co = to_off(cl);
        t.err = err;
        e = cpr::tc_forward(t, w.cmax, n_seq, H, st);
        if (e != cudaSuccess) return cuda_fail(e, "forward launch");
        return CPR_OK;
    }

    cpr::simt::FwdArgs a{};
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.cu = cu; a.chunk_off = sa.chunk_off;
    a.n_seq = n_seq; a.H = H; a.scale = c->scale;
    a.wsW = reinterpret_cast<float*>(wsb + w.W); a.wsU = reinterpret_cast<float*>(wsb + w.U);
    a.wsP = reinterpret_cast<float*>(wsb + w.P); a.wsGam = reinterpret_cast<float*>(wsb + w.gam);
    a.h0 = h0; a.o = o; a.final_state = final_state;
    a.cache = static_cast<uint8_t*>(cache); a.co = to_off(cl); a.err = err;
    cpr::LaunchCfg L{w.cmax, n_seq, H, (int)c->dv_splits, st};
    e = ops_for(*c)->fwd(a, L);
    if (e != cudaSuccess) return cuda_fail(e, "forward launch");
    return CPR_OK;
}

bool reading_b(const cpr_contract* c) { return c && c->intra_order == CPR_ORDER_TOKENREC_V1; }

// TOKENREC_V1 (reading B): the chunk-form forward keeps every chunk's boundary state in
// the workspace (training blocks); then each chunk's outputs by the token recurrence from
// hi + lo of that state.  `run` (with a cache) receives the in-chunk state after each
// sequence's partial last chunk.
int reading_b_forward(const cpr_contract* c, const uint8_t* digest, const void* q, const void* k,
                      const void* v, const float* g, const float* beta, const int32_t* cu_seqlens,
                      int n_seq, int64_t n_tok, int H, const float* h0, void* o, float* final_state,
                      void* cache, void* workspace, size_t workspace_bytes, void* stream) {
    const int rc = forward_impl(c, digest, q, k, v, g, beta, cu_seqlens, n_seq, n_tok, H, h0, o,
                                final_state, cache, workspace, workspace_bytes, stream, true);
    if (rc) return rc;
    const WsLayout w = ws_layout(*c, CPR_OP_BWD, n_seq, n_tok, H);
    unsigned char* wsb = static_cast<unsigned char*>(workspace);
    cpr::rec::RbArgs a{};
    a.q = static_cast<const __nv_bfloat16*>(q); a.k = static_cast<const __nv_bfloat16*>(k);
    a.v = static_cast<const __nv_bfloat16*>(v); a.g = g; a.beta = beta; a.cu = cu_seqlens;
    a.chunk_off = reinterpret_cast<const int32_t*>(wsb + w.chunk_off); a.n_seq = n_seq; a.H = H;
    a.scale = c->scale; a.ws = wsb + w.W; a.blk_bytes = cpr::tc::kBlockTrain;
    a.off_hn = cpr::tc::kOffHn; a.o = static_cast<float*>(o);
    a.run = cache ? reinterpret_cast<float*>(static_cast<uint8_t*>(cache) + cache_layout(*c, n_seq, H).run)
                  : nullptr;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    {
        cpr::ProfScope ps("cpr_reading_b", st);
        const cudaError_t e = cpr::rb_launch(a, n_tok > 0 ? w.cmax : 0, st);
        if (e != cudaSuccess) return cuda_fail(e, "reading-B launch");
    }
    if (!cache) return CPR_OK;
    // the decode steps continue from the cache: the partial last chunk's token rows, and
    // the chunk table of the commit batch (n_seq full chunks)
    const cpr_cache_layout cl = cache_layout(*c, n_seq, H);
    uint8_t* cb = static_cast<uint8_t*>(cache);
    cpr::rec::RbFillArgs f{};
    f.k = a.k; f.v = a.v; f.g = g; f.beta = beta; f.cu = cu_seqlens; f.n_seq = n_seq; f.H = H;
    f.rk = reinterpret_cast<__nv_bfloat16*>(cb + cl.rb_k); f.rv = reinterpret_cast<__nv_bfloat16*>(cb + cl.rb_v);
    f.rg = reinterpret_cast<float*>(cb + cl.rb_g); f.rbeta = reinterpret_cast<float*>(cb + cl.rb_beta);
    f.rcu = reinterpret_cast<int32_t*>(cb + cl.rb_cu);
    cudaError_t e;
    {
        cpr::ProfScope ps("cpr_reading_b_fill", st);
        e = cpr::rb_fill_launch(f, st);
    }
    if (e != cudaSuccess) return cuda_fail(e, "reading-B fill launch");
    uint32_t* err = device_error_ptr();
    if (!err) return fail(CPR_ERR_CUDA, "device error word unavailable");
    cpr::simt::SetupArgs sa{};
    sa.cu = f.rcu; sa.n_seq = n_seq; sa.n_tok = (int64_t)n_seq * c->chunk_size;
    sa.chunk_off = reinterpret_cast<int32_t*>(cb + cl.rb_ws + commit_ws(*c, n_seq, H).chunk_off);
    sa.err = err;
    e = launch_setup(sa, st);
    if (e != cudaSuccess) return cuda_fail(e, "setup launch");
    return CPR_OK;
}

// Reading B's decode step: the token recurrence on the running state (k_rb_step, which
// also appends the token's rows to the cache and moves the positions on), then the chunk
// commit -- the chunk form's prep and state pass over the buffered rows of every sequence
// whose chunk this token completed, from its fp32 chunk-start state to the next one (the
// prefill's kernels and inputs, so the prefill's bits).  The commit kernels run every step
// and return at once for the other sequences; a cache with another header is refused by
// every kernel before it reads past the header.
int reading_b_step(const cpr_contract* c, const uint8_t* digest, const void* q_t, const void* k_t,
                   const void* v_t, const float* g_t, const float* beta_t, int n_seq, int H,
                   void* cache, void* o_t, void* stream, bool no_commit) {
    int rc = check_digest(c, digest);
    if (rc) return rc;
    rc = check_sizes(n_seq, 0, H);
    if (rc) return rc;
    REQ_PTR(cache);
    if (n_seq == 0) return CPR_OK;
    REQ_PTR(q_t); REQ_PTR(k_t); REQ_PTR(v_t); REQ_PTR4(g_t); REQ_PTR4(beta_t); REQ_PTR(o_t);
    uint32_t* err = device_error_ptr();
    if (!err) return fail(CPR_ERR_CUDA, "device error word unavailable");
    const cpr_cache_layout cl = cache_layout(*c, n_seq, H);
    uint8_t* cb = static_cast<uint8_t*>(cache);
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    cpr::rec::RbStepArgs a{};
    a.header = reinterpret_cast<const uint32_t*>(cb + cl.header);
    std::memcpy(a.digest, digest, 32);
    rc = header_words(*c, n_seq, H, a.hdr);
    if (rc) return rc;
    static_assert(sizeof(a.hdr) == sizeof(uint32_t) * cpr::kHdrWords, "header words");
    a.q = static_cast<const __nv_bfloat16*>(q_t); a.k = static_cast<const __nv_bfloat16*>(k_t);
    a.v = static_cast<const __nv_bfloat16*>(v_t); a.g = g_t; a.beta = beta_t; a.n_seq = n_seq; a.H = H;
    a.scale = c->scale; a.pos = reinterpret_cast<int32_t*>(cb + cl.pos);
    a.done = reinterpret_cast<uint32_t*>(cb + cl.done);
    a.state = reinterpret_cast<const float*>(cb + cl.state); a.run = reinterpret_cast<float*>(cb + cl.run);
    a.rk = reinterpret_cast<__nv_bfloat16*>(cb + cl.rb_k); a.rv = reinterpret_cast<__nv_bfloat16*>(cb + cl.rb_v);
    a.rg = reinterpret_cast<float*>(cb + cl.rb_g); a.rbeta = reinterpret_cast<float*>(cb + cl.rb_beta);
    a.o = static_cast<float*>(o_t); a.err = err; a.no_commit = no_commit ? 1 : 0;
    cudaError_t e;
    {
        cpr::ProfScope ps("cpr_reading_b_step", st);
        e = cpr::rb_step_launch(a, st);
    }
    if (e != cudaSuccess) return cuda_fail(e, "reading-B step launch");
    if (no_commit) return CPR_OK;   // the step kernel checked the claim
    // the commit: n_seq full chunks from the token rows; only completed ones run
    const WsLayout w = commit_ws(*c, n_seq, H);
    cpr::tc::TcArgs t{};
    t.q = a.rk;   // (q is not needed for the state: these rows are finite, P goes unused)
    t.k = a.rk; t.v = a.rv; t.g = a.rg; t.beta = a.rbeta;
    t.cu = reinterpret_cast<const int32_t*>(cb + cl.rb_cu);
    t.chunk_off = reinterpret_cast<const int32_t*>(cb + cl.rb_ws + w.chunk_off);
    t.n_seq = n_seq; t.H = H; t.dvs = (int)(c->d_v / c->dv_splits); t.scale = c->scale;
    t.ws = cb + cl.rb_ws + w.W; t.blk_bytes = cpr::tc::kBlock; t.train = false;
    t.h0 = reinterpret_cast<const float*>(cb + cl.state);
    t.final_state = reinterpret_cast<float*>(cb + cl.state);   // in place (each thread its own entries)
    t.o = nullptr; t.cache = nullptr; t.err = err;
    t.commit_pos = a.pos; t.commit_header = a.header;
    std::memcpy(t.commit_words, a.digest, 32);
    std::memcpy(t.commit_words + 8, a.hdr, sizeof(a.hdr));
    e = cpr::tc_commit(t, n_seq, H, st);
    if (e != cudaSuccess) return cuda_fail(e, "reading-B commit launch");
    return CPR_OK;
}

int no_training(const cpr_contract* c) {
    return reading_b(c) ? fail(CPR_ERR_UNSUPPORTED, "intra_order TOKENREC_V1 (reading B) has no training ops")
                        : CPR_OK;
}

}  // namespace

extern "C" {

uint32_t cpr_kernel_build_id(void) { return kKernelBuildId; }

int cpr_contract_init_default(cpr_contract* c, uint32_t io_dtype, uint32_t d_k, uint32_t d_v) {
    if (!c) return fail(CPR_ERR_INVALID_ARG, "contract is NULL");
    std::memset(c, 0, sizeof(*c));
    c->version = CPR_CONTRACT_VERSION;
    c->chunk_size = 64;
    c->d_k = d_k;
    c->d_v = d_v;
    c->io_dtype = io_dtype;
    c->out_dtype = CPR_DTYPE_F32;
    c->gate_dtype = CPR_DTYPE_F32;
    c->accum_dtype = CPR_DTYPE_F32;
    c->state_dtype = CPR_DTYPE_F32;
    // the tensor-core policy wherever this build has it (bf16 io, d_k = d_v = 128), the
    // CUDA-core policy for the other shapes
    const bool tc = io_dtype == CPR_DTYPE_BF16 && d_k == 128 && d_v == 128;
    c->operand_policy = tc ? CPR_POLICY_TC_BF16X3 : CPR_POLICY_SIMT_F32;
    c->intra_order = CPR_ORDER_ROWSEQ_V1;
    c->state_schedule = CPR_SCHED_SEQ_CHUNKS;
    c->dv_splits = tc ? 2 : (d_v >= 128 ? 4 : 2);
    c->scale = 1.0f;
    c->kernel_build_id = kKernelBuildId;
    return check_contract(c);
}

int cpr_contract_serialize(const cpr_contract* c, uint8_t* out, size_t* len) {
    if (!c || !len) return fail(CPR_ERR_INVALID_ARG, "NULL argument");
    const size_t need = 76;
    const size_t have = *len;
    *len = need;
    if (out) {
        if (have < need) return fail(CPR_ERR_INVALID_ARG, "buffer too small (%zu < 76)", have);
        serialize(*c, out);
    }
    return CPR_OK;
}

int cpr_contract_digest(const cpr_contract* c, uint8_t out[32]) {
    if (!c || !out) return fail(CPR_ERR_INVALID_ARG, "NULL argument");
    uint8_t buf[76];
    serialize(*c, buf);
    cpr::sha256(buf, sizeof(buf), out);
    return CPR_OK;
}

int cpr_contract_check(const cpr_contract* c) { return check_contract(c); }

int cpr_deployment_digest(uint8_t out[32], char* text, size_t text_len) {
    if (!out) return fail(CPR_ERR_INVALID_ARG, "out is NULL");
    const Deployment* d = nullptr;
    const int rc = deployment_of_current_device(&d);
    if (rc) return rc;
    std::memcpy(out, d->digest, 32);
    if (text && text_len) {
        std::strncpy(text, d->text, text_len - 1);
        text[text_len - 1] = '\0';
    }
    return CPR_OK;
}

int cpr_sha256(const void* data, size_t len, uint8_t out[32]) {
    if ((!data && len) || !out) return fail(CPR_ERR_INVALID_ARG, "NULL argument");
    cpr::sha256(data, len, out);
    return CPR_OK;
}

int cpr_gdn_workspace_size(const cpr_contract* c, int op, int n_seq, int64_t n_tok, int H,
                           size_t* bytes) {
    int rc = check_contract(c);
    if (rc) return rc;
    if (!bytes) return fail(CPR_ERR_INVALID_ARG, "bytes is NULL");
    if (op != CPR_OP_FWD && op != CPR_OP_BWD) return fail(CPR_ERR_INVALID_ARG, "op %d", op);
    rc = check_sizes(n_seq, n_tok, H);
    if (rc) return rc;
    *bytes = ws_layout(*c, op, n_seq, n_tok, H).total;
    return CPR_OK;
}

int cpr_decode_cache_layout(const cpr_contract* c, int n_seq, int H, cpr_cache_layout* out) {
    int rc = check_contract(c);
    if (rc) return rc;
    if (!out) return fail(CPR_ERR_INVALID_ARG, "out is NULL");
    rc = check_sizes(n_seq, 0, H);
    if (rc) return rc;
    *out = cache_layout(*c, n_seq, H);
    return CPR_OK;
}

int cpr_decode_cache_bytes(const cpr_contract* c, int n_seq, int H, size_t* bytes) {
    if (!bytes) return fail(CPR_ERR_INVALID_ARG, "bytes is NULL");
    cpr_cache_layout l;
    int rc = cpr_decode_cache_layout(c, n_seq, H, &l);
    if (rc) return rc;
    *bytes = l.total_bytes;
    return CPR_OK;
}

int cpr_gdn_fwd(const cpr_contract* c, const uint8_t digest[32], const void* q, const void* k,
                const void* v, const float* g, const float* beta, const int32_t* cu_seqlens,
                int n_seq, int64_t n_tok, int H, const float* h0, void* o, float* final_state,
                void* workspace, size_t workspace_bytes, void* stream) {
    if (reading_b(c))
        return reading_b_forward(c, digest, q, k, v, g, beta, cu_seqlens, n_seq, n_tok, H, h0, o,
                                 final_state, nullptr, workspace, workspace_bytes, stream);
    return forward_impl(c, digest, q, k, v, g, beta, cu_seqlens, n_seq, n_tok, H, h0, o,
                        final_state, nullptr, workspace, workspace_bytes, stream);
}

int cpr_gdn_fwd_train(const cpr_contract* c, const uint8_t digest[32], const void* q,
                      const void* k, const void* v, const float* g, const float* beta,
                      const int32_t* cu_seqlens, int n_seq, int64_t n_tok, int H,
                      const float* h0, void* o, float* final_state, void* workspace,
                      size_t workspace_bytes, void* stream) {
    const int rc = no_training(c);
    if (rc) return rc;
    return forward_impl(c, digest, q, k, v, g, beta, cu_seqlens, n_seq, n_tok, H, h0, o,
                        final_state, nullptr, workspace, workspace_bytes, stream, true);
}

int cpr_gdn_prefill(const cpr_contract* c, const uint8_t digest[32], const void* q,
                    const void* k, const void* v, const float* g, const float* beta,
                    const int32_t* cu_seqlens, int n_seq, int64_t n_tok, int H, const float* h0,
                    void* o, float* final_state, void* cache, void* workspace,
                    size_t workspace_bytes, void* stream) {
    if (!cache) return fail(CPR_ERR_INVALID_ARG, "cache is NULL (use cpr_gdn_fwd without a cache)");
    if (reading_b(c))
        return reading_b_forward(c, digest, q, k, v, g, beta, cu_seqlens, n_seq, n_tok, H, h0, o,
                                 final_state, cache, workspace, workspace_bytes, stream);
    return forward_impl(c, digest, q, k, v, g, beta, cu_seqlens, n_seq, n_tok, H, h0, o,
                        final_state, cache, workspace, workspace_bytes, stream);
}

static int decode_impl(const cpr_contract* c, const uint8_t* digest, const void* q_t,
                       const void* k_t, const void* v_t, const float* g_t, const float* beta_t,
                       int n_seq, int H, void* cache, void* o_t, void* stream) {
    int rc = check_digest(c, digest);
    if (rc) return rc;
    rc = check_sizes(n_seq, 0, H);
    if (rc) return rc;
    REQ_PTR(cache);
    if (n_seq > 0) {
        REQ_PTR(q_t); REQ_PTR(k_t); REQ_PTR(v_t); REQ_PTR4(g_t); REQ_PTR4(beta_t); REQ_PTR(o_t);
    }
    uint32_t* err = device_error_ptr();
    if (!err) return fail(CPR_ERR_CUDA, "device error word unavailable");
    const cpr_cache_layout cl = cache_layout(*c, n_seq, H);
    if (c->operand_policy == CPR_POLICY_TC_BF16X3) {
        cpr::tc::TcDecArgs t{};
        t.q = static_cast<const __nv_bfloat16*>(q_t); t.k = static_cast<const __nv_bfloat16*>(k_t);
        t.v = static_cast<const __nv_bfloat16*>(v_t); t.g = g_t; t.beta = beta_t;
        t.n_seq = n_seq; t.H = H; t.scale = c->scale; t.cache = static_cast<uint8_t*>(cache);
        t.co = to_off(cl); t.digest = digest_words(digest);
        rc = header_words(*c, n_seq, H, t.hdr);
        if (rc) return rc;
        t.o = static_cast<float*>(o_t); t.err = err;
        const cudaError_t e = cpr::tc_decode_step(t, (int)(c->d_v / c->dv_splits),
                                                  static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(e, "decode launch");
        return CPR_OK;
    }
    cpr::simt::DecArgs a{};
    a.q = q_t; a.k = k_t; a.v = v_t; a.g = g_t; a.beta = beta_t; a.n_seq = n_seq; a.H = H;
    a.scale = c->scale; a.cache = static_cast<uint8_t*>(cache); a.co = to_off(cl);
    a.digest = digest_words(digest);
    rc = header_words(*c, n_seq, H, a.hdr);
    if (rc) return rc;
    a.o = static_cast<float*>(o_t); a.err = err;
    cpr::LaunchCfg L{0, n_seq, H, (int)c->dv_splits, static_cast<cudaStream_t>(stream)};
    const cudaError_t e = ops_for(*c)->decode(a, L);
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    return CPR_OK;
}

// `saved`: the workspace holds a training forward's tiles; skip the recompute.
static int backward_impl(const cpr_contract* c, const uint8_t* digest, const void* q, const void* k,
                  const void* v, const float* g, const float* beta, const int32_t* cu_seqlens,
                  int n_seq, int64_t n_tok, int H, const float* h0, const float* dO,
                  const float* dHT, void* dq, void* dk, void* dv, float* dg, float* dbeta,
                  float* dh0, void* workspace, size_t workspace_bytes, void* stream, bool saved) {
    int rc = check_digest(c, digest);
    if (rc) return rc;
    rc = no_training(c);
    if (rc) return rc;
    if (saved && c->operand_policy != CPR_POLICY_TC_BF16X3)
        return fail(CPR_ERR_UNSUPPORTED, "backward from saved tiles: tensor-core operand policy only");
    rc = check_sizes(n_seq, n_tok, H);
    if (rc) return rc;
    REQ_PTR4(cu_seqlens);
    if (n_seq > 0) REQ_PTR(dh0);
    if (n_tok > 0) {
        REQ_PTR(q); REQ_PTR(k); REQ_PTR(v); REQ_PTR4(g); REQ_PTR4(beta);
        REQ_PTR(dO); REQ_PTR(dq); REQ_PTR(dk); REQ_PTR(dv); REQ_PTR4(dg); REQ_PTR4(dbeta);
        if (c->operand_policy == CPR_POLICY_TC_BF16X3) {
            REQ_PTR32(dq); REQ_PTR32(dk);
        }
    }
    OPT_PTR(h0); OPT_PTR(dHT);
    const WsLayout w = ws_layout(*c, CPR_OP_BWD, n_seq, n_tok, H);
    if (!workspace || workspace_bytes < w.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(CPR_ERR_WORKSPACE, "workspace needs %zu bytes, 256-byte aligned", w.total);
    uint32_t* err = device_error_ptr();
    if (!err) return fail(CPR_ERR_CUDA, "device error word unavailable");
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* wsb = static_cast<uint8_t*>(workspace);

    cpr::simt::SetupArgs sa{};
    sa.cu = cu_seqlens; sa.n_seq = n_seq; sa.n_tok = n_tok;
    sa.chunk_off = reinterpret_cast<int32_t*>(wsb + w.chunk_off); sa.err = err;
    cudaError_t e = launch_setup(sa, st);
    if (e != cudaSuccess) return cuda_fail(e, "setup launch");

    if (c->operand_policy == CPR_POLICY_TC_BF16X3) {
        cpr::tc::TcArgs t{};
        t.q = static_cast<const __nv_bfloat16*>(q); t.k = static_cast<const __nv_bfloat16*>(k);
        t.v = static_cast<const __nv_bfloat16*>(v); t.g = g; t.beta = beta; t.cu = cu_seqlens;
        t.chunk_off = sa.chunk_off; t.n_seq = n_seq; t.H = H; t.dvs = (int)(c->d_v / c->dv_splits);
        t.scale = c->scale; t.ws = wsb + w.W; t.blk_bytes = cpr::tc::kBlockTrain; t.train = true;
        t.h0 = h0; t.o = nullptr; t.final_state = nullptr; t.cache = nullptr; t.err = err;
        cpr::tc::TcBwdArgs tb{};
        tb.q = t.q; tb.k = t.k; tb.v = t.v; tb.g = g; tb.beta = beta; tb.cu = cu_seqlens;
        tb.chunk_off = sa.chunk_off; tb.n_seq = n_seq; tb.H = H; tb.scale = c->scale; tb.ws = t.ws;
        tb.dO = dO; tb.dHT = dHT; tb.dq = static_cast<float*>(dq); tb.dk = static_cast<float*>(dk);
        tb.dv = static_cast<float*>(dv); tb.dg = dg; tb.dbeta = dbeta; tb.dh0 = dh0; tb.err = err;
        tb.nsplit = (int)c->dv_splits;
        e = cpr::tc_backward(t, tb, w.cmax, n_seq, H, st, !saved);
        if (e != cudaSuccess) return cuda_fail(e, "backward launch");
        return CPR_OK;
    }

    cpr::simt::FwdArgs fa{};
    fa.q = q; fa.k = k; fa.v = v; fa.g = g; fa.beta = beta; fa.cu = cu_seqlens;
    fa.chunk_off = sa.chunk_off; fa.n_seq = n_seq; fa.H = H; fa.scale = c->scale;
    fa.wsW = reinterpret_cast<float*>(wsb + w.W); fa.wsU = reinterpret_cast<float*>(wsb + w.U);
    fa.wsP = reinterpret_cast<float*>(wsb + w.P); fa.wsGam = reinterpret_cast<float*>(wsb + w.gam);
    fa.wsT = reinterpret_cast<float*>(wsb + w.T); fa.wsKd = reinterpret_cast<float*>(wsb + w.Kd);
    fa.wsHn = reinterpret_cast<float*>(wsb + w.Hn);
    fa.h0 = h0; fa.o = nullptr; fa.final_state = nullptr; fa.cache = nullptr; fa.err = err;

    cpr::simt::BwdArgs ba{};
    ba.q = q; ba.k = k; ba.v = v; ba.g = g; ba.beta = beta; ba.cu = cu_seqlens;
    ba.chunk_off = sa.chunk_off; ba.n_seq = n_seq; ba.H = H; ba.scale = c->scale;
    ba.dO = dO; ba.dHT = dHT;
    ba.wsW = fa.wsW; ba.wsU = fa.wsU; ba.wsP = fa.wsP; ba.wsGam = fa.wsGam; ba.wsT = fa.wsT;
    ba.wsKd = fa.wsKd; ba.wsHn = fa.wsHn; ba.wsdH = reinterpret_cast<float*>(wsb + w.dH);
    ba.dq = static_cast<float*>(dq); ba.dk = static_cast<float*>(dk); ba.dv = static_cast<float*>(dv);
    ba.dg = dg; ba.dbeta = dbeta; ba.dh0 = dh0; ba.err = err;
    cpr::LaunchCfg L{w.cmax, n_seq, H, (int)c->dv_splits, st};
    e = ops_for(*c)->bwd(fa, ba, L);
    if (e != cudaSuccess) return cuda_fail(e, "backward launch");
    return CPR_OK;
}

int cpr_gdn_bwd(const cpr_contract* c, const uint8_t digest[32], const void* q, const void* k,
                const void* v, const float* g, const float* beta, const int32_t* cu_seqlens,
                int n_seq, int64_t n_tok, int H, const float* h0, const float* dO,
                const float* dHT, void* dq, void* dk, void* dv, float* dg, float* dbeta,
                float* dh0, void* workspace, size_t workspace_bytes, void* stream) {
    return backward_impl(c, digest, q, k, v, g, beta, cu_seqlens, n_seq, n_tok, H, h0, dO, dHT,
                         dq, dk, dv, dg, dbeta, dh0, workspace, workspace_bytes, stream, false);
}

int cpr_gdn_bwd_saved(const cpr_contract* c, const uint8_t digest[32], const void* q,
                      const void* k, const void* v, const float* g, const float* beta,
                      const int32_t* cu_seqlens, int n_seq, int64_t n_tok, int H,
                      const float* h0, const float* dO, const float* dHT, void* dq, void* dk,
                      void* dv, float* dg, float* dbeta, float* dh0, void* workspace,
                      size_t workspace_bytes, void* stream) {
    return backward_impl(c, digest, q, k, v, g, beta, cu_seqlens, n_seq, n_tok, H, h0, dO, dHT,
                         dq, dk, dv, dg, dbeta, dh0, workspace, workspace_bytes, stream, true);
}

int cpr_get_device_error(uint32_t* code, int clear) {
    if (!code) return fail(CPR_ERR_INVALID_ARG, "code is NULL");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "synchronize");
    e = cudaMemcpyFromSymbol(code, g_cpr_device_error, sizeof(uint32_t));
    if (e != cudaSuccess) return cuda_fail(e, "read device error");
    if (clear) {
        const uint32_t zero = 0u;
        e = cudaMemcpyToSymbol(g_cpr_device_error, &zero, sizeof(uint32_t));
        if (e != cudaSuccess) return cuda_fail(e, "clear device error");
    }
    return CPR_OK;
}

int cpr_selftest_wait_timeout(uint32_t poll_limit, uint32_t* completed) {
    if (!completed) return fail(CPR_ERR_INVALID_ARG, "completed is NULL");
    uint32_t* err = device_error_ptr();
    if (!err) return fail(CPR_ERR_CUDA, "device error word unavailable");
    uint32_t* d_ok = nullptr;
    cudaError_t e = cudaMalloc(&d_ok, sizeof(uint32_t));
    if (e != cudaSuccess) return cuda_fail(e, "selftest alloc");
    e = cpr::tc_wait_timeout_selftest(err, poll_limit, d_ok, nullptr);
    if (e == cudaSuccess) e = cudaMemcpy(completed, d_ok, sizeof(uint32_t), cudaMemcpyDeviceToHost);
    cudaFree(d_ok);
    if (e != cudaSuccess) return cuda_fail(e, "selftest");
    return CPR_OK;
}

int cpr_gdn_decode_step(const cpr_contract* c, const uint8_t digest[32], const void* q_t,
                        const void* k_t, const void* v_t, const float* g_t, const float* beta_t,
                        int n_seq, int H, void* cache, void* o_t, void* stream) {
    if (reading_b(c))
        return reading_b_step(c, digest, q_t, k_t, v_t, g_t, beta_t, n_seq, H, cache, o_t, stream, false);
    return decode_impl(c, digest, q_t, k_t, v_t, g_t, beta_t, n_seq, H, cache, o_t, stream);
}

int cpr_gdn_decode_step_nocommit(const cpr_contract* c, const uint8_t digest[32], const void* q_t,
                                 const void* k_t, const void* v_t, const float* g_t,
                                 const float* beta_t, int n_seq, int H, void* cache, void* o_t,
                                 void* stream) {
    if (reading_b(c))
        return reading_b_step(c, digest, q_t, k_t, v_t, g_t, beta_t, n_seq, H, cache, o_t, stream, true);
    return decode_impl(c, digest, q_t, k_t, v_t, g_t, beta_t, n_seq, H, cache, o_t, stream);
}

static int rec_check(const cpr_contract* c) {
    if (!c) return fail(CPR_ERR_INVALID_ARG, "contract is NULL");
    if (c->d_k != c->d_v || (c->d_k != 64 && c->d_k != 128))
        return fail(CPR_ERR_UNSUPPORTED, "recurrent path: d_k = d_v = 64 or 128 only");
    if (c->io_dtype != CPR_DTYPE_BF16 && c->io_dtype != CPR_DTYPE_F32)
        return fail(CPR_ERR_UNSUPPORTED, "recurrent path: io dtype bf16 or fp32");
    return CPR_OK;
}

int cpr_gdn_recurrent_fwd(const cpr_contract* c, const void* q, const void* k, const void* v,
                          const float* g, const float* beta, const int32_t* cu_seqlens,
                          int n_seq, int64_t n_tok, int H, const float* h0, float* o,
                          float* final_state, void* stream) {
    int rc = rec_check(c);
    if (rc) return rc;
    rc = check_sizes(n_seq, n_tok, H);
    if (rc) return rc;
    REQ_PTR4(cu_seqlens);
    if (n_tok > 0) {
        REQ_PTR(q); REQ_PTR(k); REQ_PTR(v); REQ_PTR4(g); REQ_PTR4(beta); REQ_PTR(o);
    }
    OPT_PTR(h0); OPT_PTR(final_state);
    uint32_t* err = device_error_ptr();
    if (!err) return fail(CPR_ERR_CUDA, "device error word unavailable");
    cpr::rec::RecArgs a{};
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.cu = cu_seqlens; a.n_seq = n_seq;
    a.n_tok = n_tok; a.H = H; a.scale = c->scale; a.h0 = h0; a.final_state = final_state; a.o = o;
    a.err = err;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    cpr::ProfScope ps("cpr_rec_fwd", st);
    const cudaError_t e = cpr::rec_launch(a, (int)c->d_k, c->io_dtype == CPR_DTYPE_BF16, st);
    if (e != cudaSuccess) return cuda_fail(e, "recurrent forward launch");
    return CPR_OK;
}

int cpr_gdn_recurrent_step(const cpr_contract* c, const void* q_t, const void* k_t,
                           const void* v_t, const float* g_t, const float* beta_t, int n_seq,
                           int H, float* state, float* o_t, void* stream) {
    int rc = rec_check(c);
    if (rc) return rc;
    rc = check_sizes(n_seq, 0, H);
    if (rc) return rc;
    if (n_seq > 0) {
        REQ_PTR(q_t); REQ_PTR(k_t); REQ_PTR(v_t); REQ_PTR4(g_t); REQ_PTR4(beta_t); REQ_PTR(o_t);
        REQ_PTR(state);
    }
    uint32_t* err = device_error_ptr();
    if (!err) return fail(CPR_ERR_CUDA, "device error word unavailable");
    cpr::rec::RecArgs a{};
    a.q = q_t; a.k = k_t; a.v = v_t; a.g = g_t; a.beta = beta_t; a.cu = nullptr; a.n_seq = n_seq;
    a.n_tok = n_seq; a.H = H; a.scale = c->scale; a.state = state; a.o = o_t; a.err = err;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    cpr::ProfScope ps("cpr_rec_step", st);
    const cudaError_t e = cpr::rec_launch(a, (int)c->d_k, c->io_dtype == CPR_DTYPE_BF16, st);
    if (e != cudaSuccess) return cuda_fail(e, "recurrent step launch");
    return CPR_OK;
}

static size_t rec_bwd_ckpt_bytes(const cpr_contract* c, int n_seq, int64_t n_tok, int H) {
    return (size_t)(n_tok / cpr::rec::kRecSeg + n_seq) * (size_t)H * c->d_k * c->d_v * 4;
}

int cpr_gdn_recurrent_bwd_workspace_size(const cpr_contract* c, int n_seq, int64_t n_tok, int H,
                                         size_t* bytes) {
    int rc = rec_check(c);
    if (rc) return rc;
    rc = check_sizes(n_seq, n_tok, H);
    if (rc) return rc;
    if (!bytes) return fail(CPR_ERR_INVALID_ARG, "bytes is NULL");
    *bytes = align256(rec_bwd_ckpt_bytes(c, n_seq, n_tok, H)) +
             (size_t)n_seq * H * cpr::rec::kRecSeg * c->d_k * c->d_v * 4;
    return CPR_OK;
}

int cpr_gdn_recurrent_bwd(const cpr_contract* c, const void* q, const void* k, const void* v,
                          const float* g, const float* beta, const int32_t* cu_seqlens,
                          int n_seq, int64_t n_tok, int H, const float* h0, const float* dO,
                          const float* dHT, float* dq, float* dk, float* dv, float* dg,
                          float* dbeta, float* dh0, void* workspace, size_t workspace_bytes,
                          void* stream) {
    size_t need = 0;
    int rc = cpr_gdn_recurrent_bwd_workspace_size(c, n_seq, n_tok, H, &need);
    if (rc) return rc;
    REQ_PTR4(cu_seqlens);
    if (n_seq > 0) REQ_PTR(dh0);
    if (n_tok > 0) {
        REQ_PTR(q); REQ_PTR(k); REQ_PTR(v); REQ_PTR4(g); REQ_PTR4(beta); REQ_PTR(dO);
        REQ_PTR(dq); REQ_PTR(dk); REQ_PTR(dv); REQ_PTR4(dg); REQ_PTR4(dbeta);
    }
    OPT_PTR(h0); OPT_PTR(dHT);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(CPR_ERR_WORKSPACE, "workspace needs %zu bytes, 256-byte aligned", need);
    uint32_t* err = device_error_ptr();
    if (!err) return fail(CPR_ERR_CUDA, "device error word unavailable");
    cpr::rec::RecBwdArgs a{};
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.cu = cu_seqlens; a.n_seq = n_seq;
    a.n_tok = n_tok; a.H = H; a.scale = c->scale; a.h0 = h0; a.dO = dO; a.dHT = dHT;
    a.dq = dq; a.dk = dk; a.dv = dv; a.dg = dg; a.dbeta = dbeta; a.dh0 = dh0;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    a.ckpt = reinterpret_cast<float*>(ws);
    a.seg = reinterpret_cast<float*>(ws + align256(rec_bwd_ckpt_bytes(c, n_seq, n_tok, H)));
    a.err = err;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    cpr::ProfScope ps("cpr_rec_bwd", st);
    const cudaError_t e = cpr::rec_bwd_launch(a, (int)c->d_k, c->io_dtype == CPR_DTYPE_BF16, st);
    if (e != cudaSuccess) return cuda_fail(e, "recurrent backward launch");
    return CPR_OK;
}

int cpr_gemm_bf16(const void* X, const void* W, float* Y, int M, int N, int K, int leaf_k,
                  void* stream) {
    if (M < 0 || N <= 0 || K <= 0 || N % 128 || K % 64 || leaf_k <= 0 || leaf_k % 64 || K % leaf_k)
        return fail(CPR_ERR_INVALID_ARG, "gemm: N a multiple of 128, leaf_k a multiple of 64 dividing K");
    const int nleaf = K / leaf_k;
    if (nleaf != 1 && nleaf != 2 && nleaf != 4)
        return fail(CPR_ERR_INVALID_ARG, "gemm: K / leaf_k must be 1, 2 or 4");
    if ((int64_t)M * K > INT32_MAX * 4ll) return fail(CPR_ERR_INVALID_ARG, "gemm: M * K too large");
    if (M > 0) {
        REQ_PTR(X); REQ_PTR(W); REQ_PTR(Y); REQ_PTR32(Y);
    }
    uint32_t* err = device_error_ptr();
    if (!err) return fail(CPR_ERR_CUDA, "device error word unavailable");
    cpr::gemm::GemmArgs a{};
    a.X = static_cast<const __nv_bfloat16*>(X); a.W = static_cast<const __nv_bfloat16*>(W); a.Y = Y;
    a.M = M; a.N = N; a.K = K; a.leaf_k = leaf_k; a.err = err;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    cpr::ProfScope ps("cpr_gemm", st);
    const cudaError_t e = cpr::gemm_launch(a, st);
    if (e != cudaSuccess) return cuda_fail(e, "gemm launch");
    return CPR_OK;
}

const char* cpr_last_error(void) { return g_msg; }

}  // extern "C"
