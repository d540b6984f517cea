// The gated delta rule as a plain token recurrence, for the stage-table ablations:
// "recurrent everywhere" (cpr_gdn_recurrent_fwd over whole sequences) and the
// non-resynchronised decode of "native mixed" (cpr_gdn_recurrent_step on an fp32
// state, after a chunked prefill).  Page "IsoExec: 切换 SkyRL 中的训练器-推理不匹配",
// section "Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet" and its stage table:
// the engines' native path decodes token by token, which is what CPR replaces.
//
// Per token, with H = S^T (d_k x d_v) and a = exp(g):
//   S_t = a S_{t-1} (I - b k k^T) + b v k^T   <=>   H_t = a H + k u^T,  u = b (v - a H^T k)
//   o_t = S_t q = H_t^T (scale q)
// One CTA per (sequence, head), 2 d threads: thread (j, part) keeps column j of H for
// rows part * d/2 .. + d/2 in registers.  Every sum is one fp32 fma chain in ascending
// row order per half, the two halves added half 0 first, so the prefill and a decode
// step evaluate the same operations for a token (the two agree bit for bit); neither
// agrees bit for bit with the chunked form.
#include <cuda_bf16.h>
#include <stdint.h>

#include "common.cuh"
#include "rec.h"
#include "tc_common.cuh"

namespace cpr {
namespace rec {

__device__ __forceinline__ float ld_io(const __nv_bfloat16* p, size_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ float ld_io(const float* p, size_t i) { return p[i]; }

template <int D>
struct RecSmem {
    float kq[2][2][D];   // [buffer][k | scale q][row]
    float vv[2][D];
    float ab[2][2];      // [buffer][a | b]
    float red[2][D];     // H^T k halves
    float red2[2][D];    // H^T q halves
};

// One token: H = a H + k u^T, u = b (v - a H^T k); returns the complete o_j (valid after
// the second barrier).  `stage` runs between the two barriers (the next token's rows).
template <int D, typename Stage>
__device__ __forceinline__ float token(float (&h)[D / 2], RecSmem<D>& s, int cur, int j, int part,
                                       Stage&& stage) {
    const float* ks = s.kq[cur][0] + part * (D / 2);
    const float* qs = s.kq[cur][1] + part * (D / 2);
    float w = 0.f;
#pragma unroll
    for (int i = 0; i < D / 2; ++i) w = __fmaf_rn(h[i], ks[i], w);
    s.red[part][j] = w;
    __syncthreads();
    const float a = s.ab[cur][0], b = s.ab[cur][1];
    const float wj = __fadd_rn(s.red[0][j], s.red[1][j]);
    const float u = __fmul_rn(b, __fsub_rn(s.vv[cur][j], __fmul_rn(a, wj)));
    float o = 0.f;
#pragma unroll
    for (int i = 0; i < D / 2; ++i) {
        h[i] = __fmaf_rn(ks[i], u, __fmul_rn(a, h[i]));
        o = __fmaf_rn(h[i], qs[i], o);
    }
    s.red2[part][j] = o;
    stage();
    __syncthreads();
    return __fadd_rn(s.red2[0][j], s.red2[1][j]);
}

// Tokens t0 .. t1 - 1 of head h from the state in hr: each token's rows are loaded into
// registers while the previous token's sums run, then staged in a shared buffer.
template <int D, typename IO>
__device__ __forceinline__ void token_loop(float (&hr)[D / 2], RecSmem<D>& s, const IO* q, const IO* k,
                                           const IO* v, const float* g, const float* beta, int H, int h,
                                           float scale, int t0, int t1, float* out) {
    const int tid = threadIdx.x, j = tid % D, part = tid / D;
    float rk = 0.f, rq = 0.f, rv = 0.f, ra = 0.f, rb = 0.f;
    auto load = [&](int t) {
        if (tid < D) {
            const size_t row = ((size_t)t * H + h) * D + tid;
            rk = ld_io(k, row);
            rq = __fmul_rn(scale, ld_io(q, row));
            rv = ld_io(v, row);
        }
        if (tid == 0) {
            ra = expf(g[(size_t)t * H + h]);
            rb = beta[(size_t)t * H + h];
        }
    };
    auto store = [&](int buf) {
        if (tid < D) {
            s.kq[buf][0][tid] = rk;
            s.kq[buf][1][tid] = rq;
            s.vv[buf][tid] = rv;
        }
        if (tid == 0) {
            s.ab[buf][0] = ra;
            s.ab[buf][1] = rb;
        }
    };
    if (t0 < t1) {
        load(t0);
        store(0);
    }
    __syncthreads();
    for (int t = t0; t < t1; ++t) {
        const int cur = (t - t0) & 1;
        const bool more = t + 1 < t1;
        if (more) load(t + 1);   // lands while this token's sums run
        const float o = token<D>(hr, s, cur, j, part, [&]() { if (more) store(cur ^ 1); });
        if (part == 0) out[((size_t)t * H + h) * D + j] = o;
    }
}

template <int D, typename IO>
__global__ void __launch_bounds__(2 * D) k_rec(RecArgs a) {
    __shared__ RecSmem<D> s;
    const int tid = threadIdx.x, j = tid % D, part = tid / D;
    const int H = a.H;
    const int b = blockIdx.x / H, h = blockIdx.x % H;
    const size_t sh = (size_t)b * H + h;
    const IO* q = static_cast<const IO*>(a.q);
    const IO* k = static_cast<const IO*>(a.k);
    const IO* v = static_cast<const IO*>(a.v);
    int t0, t1;
    if (a.cu) {  // recurrent prefill over the sequence's tokens
        t0 = a.cu[b];
        t1 = a.cu[b + 1];
        if (t0 < 0 || t1 < t0 || (int64_t)t1 > a.n_tok) {
            if (tid == 0) set_error(a.err, CPR_ERR_BAD_SEQLENS);
            return;
        }
    } else {     // one decode step: token b of the step's batch
        t0 = b;
        t1 = b + 1;
    }
    // the state: column j, this thread's half of the rows
    float hr[D / 2];
    const float* hin = a.cu ? a.h0 : a.state;
#pragma unroll
    for (int i = 0; i < D / 2; ++i)
        hr[i] = hin ? hin[(sh * D + part * (D / 2) + i) * D + j] : 0.f;
    token_loop<D, IO>(hr, s, q, k, v, a.g, a.beta, H, h, a.scale, t0, t1, a.o);
    float* hout = a.cu ? a.final_state : a.state;
    if (hout) {
#pragma unroll
        for (int i = 0; i < D / 2; ++i) hout[(sh * D + part * (D / 2) + i) * D + j] = hr[i];
    }
}

// Reading B of the chunk form: each chunk's outputs from the token recurrence started at
// the chunk form's boundary state H_n.  The training forward leaves H_n in every chunk's
// workspace block as hi/lo operand tiles (K-major (d, j)); the start state is hi + lo,
// the same bits a decode cache's state tiles hold for that chunk.  One CTA per (chunk,
// head), chunks independent.
__global__ void __launch_bounds__(256) k_rb(RbArgs a) {
    constexpr int D = 128;
    __shared__ RecSmem<D> s;
    const int tid = threadIdx.x, j = tid % D, part = tid / D;
    const int total = a.chunk_off[a.n_seq];
    const int cidx = blockIdx.x, h = blockIdx.y, H = a.H;
    if (total < 0 || cidx >= total) return;
    const int b = find_seq(a.chunk_off, a.n_seq, cidx);
    const int n = cidx - a.chunk_off[b];
    const int seq0 = a.cu[b], T = a.cu[b + 1] - seq0;
    const int t0 = seq0 + n * kChunk, t1 = t0 + min(kChunk, T - n * kChunk);
    const unsigned char* hn = a.ws + ((size_t)cidx * H + h) * a.blk_bytes + a.off_hn;
    float hr[D / 2];
#pragma unroll
    for (int i = 0; i < D / 2; ++i) {
        const uint32_t off = tc::cm_off(part * (D / 2) + i, j, D);
        hr[i] = __fadd_rn(__bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(hn + off)),
                          __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(hn + 32768 + off)));
    }
    token_loop<D, __nv_bfloat16>(hr, s, a.q, a.k, a.v, a.g, a.beta, H, h, a.scale, t0, t1, a.o);
    if (a.run && t1 == seq0 + T && t1 - t0 < kChunk) {  // a decode continues this partial chunk
        float* run = a.run + ((size_t)b * H + h) * D * D;
#pragma unroll
        for (int i = 0; i < D / 2; ++i) run[(part * (D / 2) + i) * D + j] = hr[i];
    }
}

// Reading B, one decode step per (sequence, head), after the CPR decode step of the same
// tokens (which keeps the cache and commits a full chunk): at a chunk's first row the
// running state restarts from hi + lo of the cache's chunk-start state tiles -- the bits
// the reading-B prefill starts that chunk from -- otherwise it continues; one token of
// the recurrence, o from it.  A cache whose header is not this contract's (another
// digest, another shape; the CPR step has recorded the mismatch) is left untouched: its
// blob need not have the running-state section at all.
__global__ void __launch_bounds__(256) k_rb_step(RbStepArgs a) {
    constexpr int D = 128;
    __shared__ RecSmem<D> s;
    __shared__ int ok_s;
    const int tid = threadIdx.x, j = tid % D, part = tid / D;
    if (tid == 0) {
        bool ok = a.header[0] == kCacheMagic && a.header[1] == CPR_CONTRACT_VERSION;
        for (int i = 0; i < 8; ++i) ok = ok && a.header[2 + i] == a.digest[i];
        for (int i = 0; i < 7; ++i) ok = ok && a.header[10 + i] == a.hdr[i];
        ok_s = ok ? 1 : 0;
    }
    __syncthreads();
    if (!ok_s) return;
    const int H = a.H, b = blockIdx.x / H, h = blockIdx.x % H;
    const size_t sh = (size_t)b * H + h;
    const int p = (a.pos[b] + kChunk - 1) % kChunk;   // this step's row in its chunk
    float* run = a.run + sh * D * D;
    float hr[D / 2];
    if (p == 0) {
        const unsigned char* ct = a.state_tiles + sh * 65536;
        const int sp = j / a.dvs, jl = j - sp * a.dvs;
#pragma unroll
        for (int i = 0; i < D / 2; ++i) {
            const uint32_t off = (uint32_t)sp * a.dvs * 256 + tc::mn_off(jl, part * (D / 2) + i, a.dvs);
            hr[i] = __fadd_rn(__bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(ct + off)),
                              __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(ct + 32768 + off)));
        }
    } else {
#pragma unroll
        for (int i = 0; i < D / 2; ++i) hr[i] = run[(part * (D / 2) + i) * D + j];
    }
    token_loop<D, __nv_bfloat16>(hr, s, a.q, a.k, a.v, a.g, a.beta, H, h, a.scale, b, b + 1, a.o);
#pragma unroll
    for (int i = 0; i < D / 2; ++i) run[(part * (D / 2) + i) * D + j] = hr[i];
}

template <int D, typename IO>
static cudaError_t launch(const RecArgs& a, cudaStream_t st) {
    const int64_t grid = (int64_t)a.n_seq * a.H;
    if (grid > 0) k_rec<D, IO><<<(unsigned)grid, 2 * D, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace rec

cudaError_t rb_launch(const rec::RbArgs& a, int64_t cmax, cudaStream_t st) {
    if (cmax > 0 && a.H > 0) rec::k_rb<<<dim3((unsigned)cmax, (unsigned)a.H), 256, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t rb_step_launch(const rec::RbStepArgs& a, cudaStream_t st) {
    const int64_t grid = (int64_t)a.n_seq * a.H;
    if (grid > 0) rec::k_rb_step<<<(unsigned)grid, 256, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t rec_launch(const rec::RecArgs& a, int d, bool bf16, cudaStream_t st) {
    if (d == 128) return bf16 ? rec::launch<128, __nv_bfloat16>(a, st) : rec::launch<128, float>(a, st);
    if (d == 64) return bf16 ? rec::launch<64, __nv_bfloat16>(a, st) : rec::launch<64, float>(a, st);
    return cudaErrorInvalidValue;
}

}  // namespace cpr
