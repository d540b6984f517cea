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

// One token's state update, H = a H + k u^T with u = b (v - a H^T k): the two halves'
// sums H^T k combined half 0 first.  Reads the token's k, v, a, b from buffer `cur`,
// writes s.red; one barrier inside.
template <int D>
__device__ __forceinline__ void update(float (&h)[D / 2], RecSmem<D>& s, int cur, int j, int part) {
    const float* ks = s.kq[cur][0] + part * (D / 2);
    float w = 0.f;
#pragma unroll
    for (int i = 0; i < D / 2; ++i) w = __fmaf_rn(h[i], ks[i], w);
    s.red[part][j] = w;
    __syncthreads();
    const float a = s.ab[cur][0], b = s.ab[cur][1];
    const float wj = __fadd_rn(s.red[0][j], s.red[1][j]);
    const float u = __fmul_rn(b, __fsub_rn(s.vv[cur][j], __fmul_rn(a, wj)));
#pragma unroll
    for (int i = 0; i < D / 2; ++i) h[i] = __fmaf_rn(ks[i], u, __fmul_rn(a, h[i]));
}

// One token: the update, then o_j = sum_d H_t[d][j] (scale q)[d] (returned complete after
// the second barrier).  `stage` runs between the two barriers (the next token's rows).
template <int D, typename Stage>
__device__ __forceinline__ float token(float (&h)[D / 2], RecSmem<D>& s, int cur, int j, int part,
                                       Stage&& stage) {
    update<D>(h, s, cur, j, part);
    const float* qs = s.kq[cur][1] + part * (D / 2);
    float o = 0.f;
#pragma unroll
    for (int i = 0; i < D / 2; ++i) o = __fmaf_rn(h[i], qs[i], o);
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

// fp32 load and store with an L2 cache policy (createpolicy), and the policy itself.
__device__ __forceinline__ float ld_hint(const float* p, uint64_t pol) {
    float v;
    asm volatile("ld.global.L2::cache_hint.f32 %0, [%1], %2;" : "=f"(v) : "l"(p), "l"(pol));
    return v;
}
__device__ __forceinline__ void st_hint(float* p, float v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" :: "l"(p), "f"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ uint64_t l2_keep_policy(bool keep) {
    uint64_t pol;
    if (keep) asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    else asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
// A decode step's recurrent states (64 KB a (sequence, head); the native step's and reading
// B's running states) are read and written once a step, and all of them together are a
// little more than L2 holds.  Those of 3 (sequence, head) in every 8 are accessed with the
// evict-last priority, so that they can stay in L2 from one step to the next, and the others
// with evict-first.
constexpr int kRunKeepOf8 = 3;

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
    const uint64_t pol = l2_keep_policy((int)(sh % 8) < kRunKeepOf8);   // (the decode step's)
#pragma unroll
    for (int i = 0; i < D / 2; ++i) {
        hr[i] = 0.f;
        if (hin) {
            const float* src = hin + (sh * D + part * (D / 2) + i) * D + j;
            hr[i] = a.cu ? *src : ld_hint(src, pol);
        }
    }
    token_loop<D, IO>(hr, s, q, k, v, a.g, a.beta, H, h, a.scale, t0, t1, a.o);
    float* hout = a.cu ? a.final_state : a.state;
    if (hout) {
#pragma unroll
        for (int i = 0; i < D / 2; ++i) {
            float* dst = hout + (sh * D + part * (D / 2) + i) * D + j;
            if (a.cu) *dst = hr[i];
            else st_hint(dst, hr[i], pol);
        }
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

// Reading B, one decode step per (sequence, head).  Between commits a step is only the
// token recurrence: at a chunk's first row the running state restarts from hi + lo of the
// fp32 chunk-start state (split to bf16 hi, lo as the state tiles hold it: the bits the
// reading-B prefill starts that chunk from), otherwise it continues; o comes from it.
// The token's k, v, g, beta rows are appended to the cache's chunk rows, which the commit
// (the chunk form's prep and state pass over the buffered chunk, launched after this
// kernel) reads once the chunk is complete.  The last CTA moves every position on.  A
// cache whose header is not this contract's is left untouched (nothing past its header
// is read) and CPR_ERR_CONTRACT_MISMATCH is recorded.  Under the caller's no-commit claim
// every CTA reads every sequence's position: if one is C - 1 (its chunk would complete, but
// no commit follows) every CTA leaves, nothing is written and CPR_ERR_COMMIT_DUE is recorded.

__global__ void __launch_bounds__(256) k_rb_step(RbStepArgs a) {
    constexpr int D = 128;
    __shared__ RecSmem<D> s;
    __shared__ int ok_s;
    const int tid = threadIdx.x, j = tid % D, part = tid / D;
    const int H = a.H, b = blockIdx.x / H, h = blockIdx.x % H;
    if (tid < 32) {   // the header (a word per lane), then the positions once it is right
        bool ok = cache_header_ok(a.header, a.digest, a.hdr);
        bool due = false;
        if (ok && a.no_commit) {
            bool d = false;
            for (int sq = tid; sq < a.n_seq; sq += 32) d = d | (a.pos[sq] == kChunk - 1);
            due = __any_sync(0xffffffffu, d);
        }
        if (tid == 0) {
            const int p = ok ? a.pos[b] : -1;
            if (!(p >= 0 && p < kChunk)) ok = false;
            if (!ok) set_error(a.err, CPR_ERR_CONTRACT_MISMATCH);
            else if (due) set_error(a.err, CPR_ERR_COMMIT_DUE);
            ok_s = (ok && !due) ? 1 + p : 0;
        }
    }
    __syncthreads();
    if (!ok_s) return;
    const int p = ok_s - 1;   // this step's row in its chunk
    const size_t sh = (size_t)b * H + h;
    float* run = a.run + sh * D * D;
    const uint64_t pol = l2_keep_policy((int)(sh % 8) < kRunKeepOf8);
    float hr[D / 2];
    if (p == 0) {
        const float* st = a.state + sh * D * D;
#pragma unroll
        for (int i = 0; i < D / 2; ++i) {
            __nv_bfloat16 hi, lo;
            tc::split_bf16(st[(part * (D / 2) + i) * D + j], hi, lo);
            hr[i] = __fadd_rn(__bfloat162float(hi), __bfloat162float(lo));
        }
    } else {
#pragma unroll
        for (int i = 0; i < D / 2; ++i) hr[i] = ld_hint(run + (part * (D / 2) + i) * D + j, pol);
    }
    token_loop<D, __nv_bfloat16>(hr, s, a.q, a.k, a.v, a.g, a.beta, H, h, a.scale, b, b + 1, a.o);
#pragma unroll
    for (int i = 0; i < D / 2; ++i) st_hint(run + (part * (D / 2) + i) * D + j, hr[i], pol);
    const size_t row = (size_t)b * kChunk + p;   // the chunk rows' token index
    if (tid < D) {
        a.rk[(row * H + h) * D + tid] = a.k[sh * D + tid];
        a.rv[(row * H + h) * D + tid] = a.v[sh * D + tid];
    } else if (tid == D) {
        a.rg[row * H + h] = a.g[sh];
        a.rbeta[row * H + h] = a.beta[sh];
    }
    __syncthreads();
    if (tid == 0) {
        // every sequence advances one token per step: the last CTA to finish moves all the
        // positions on (every CTA read its position before its count; the commit and the
        // next step are later launches)
        __threadfence();
        const uint32_t prev = atomicAdd(a.done, 1u);
        if (prev == gridDim.x - 1) {
            for (int sq = 0; sq < a.n_seq; ++sq) a.pos[sq] = (a.pos[sq] + 1) % kChunk;
            *a.done = 0u;
            __threadfence();
        }
    }
}

// Reading B prefill with a decode cache: each sequence's partial last chunk (rows from the
// last chunk boundary to its end) into the cache's token-major chunk rows, and the commit
// batch's fixed sequence offsets b * C.  One CTA per (sequence, head).
__global__ void __launch_bounds__(128) k_rb_fill(RbFillArgs a) {
    constexpr int D = 128;
    const int H = a.H, b = blockIdx.x / H, h = blockIdx.x % H;
    const int t0 = a.cu[b], T = a.cu[b + 1] - t0;
    const int full = T - T % kChunk;
    for (int i = threadIdx.x; i < (T - full) * D; i += blockDim.x) {
        const int r = i / D, d = i % D;
        const size_t src = ((size_t)(t0 + full + r) * H + h) * D + d;
        const size_t dst = (((size_t)b * kChunk + r) * H + h) * D + d;
        a.rk[dst] = a.k[src];
        a.rv[dst] = a.v[src];
    }
    for (int r = threadIdx.x; r < T - full; r += blockDim.x) {
        a.rg[((size_t)b * kChunk + r) * H + h] = a.g[(size_t)(t0 + full + r) * H + h];
        a.rbeta[((size_t)b * kChunk + r) * H + h] = a.beta[(size_t)(t0 + full + r) * H + h];
    }
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i <= a.n_seq; i += blockDim.x) a.rcu[i] = i * kChunk;
}

// Tokens t0 .. t1 - 1 of head h through the state update only (no outputs): the same
// operations as token_loop's, so the states are the recurrent forward's bit for bit.
// pre(t) runs before token t, post(t) after it, both with the state in hr.
template <int D, typename IO, typename Pre, typename Post>
__device__ __forceinline__ void state_loop(float (&hr)[D / 2], RecSmem<D>& s, const IO* k, const IO* v,
                                           const float* g, const float* beta, int H, int h, int t0, int t1,
                                           Pre&& pre, Post&& post) {
    const int tid = threadIdx.x, j = tid % D, part = tid / D;
    float rk = 0.f, rv = 0.f, ra = 0.f, rb = 0.f;
    auto load = [&](int t) {
        if (tid < D) {
            const size_t row = ((size_t)t * H + h) * D + tid;
            rk = ld_io(k, row);
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
        if (more) load(t + 1);
        pre(t);
        update<D>(hr, s, cur, j, part);
        post(t);
        if (more) store(cur ^ 1);
        __syncthreads();
    }
}

template <int D>
struct RecBwdSmem {
    RecSmem<D> f;                  // the forward's token buffers
    float tq[2][D], tk[2][D], tv[2][D], tdo[2][D];   // backward token rows (q scaled)
    float tab[2][2];               // a, b
    float Rq[D][D + 1];            // dq partials [d][j] (rows padded: conflict-free columns)
    float Rk[D][D + 1];            // dk partials
    float ru[2][D], rs[2][D];      // halves of H_{t-1}^T k and Hhat^T k
    float wsum[3][2 * D / 32];     // per-warp partials: <Hhat, H_{t-1}>, e . sk, sk . u1
};

// Sum over the 32 lanes of a warp in a fixed tree (lane 0 gets the result).
__device__ __forceinline__ float warp_tree(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = __fadd_rn(x, __shfl_down_sync(0xffffffffu, x, o));
    return x;
}

// The backward of the token recurrence ("recurrent everywhere" training): the adjoint of
// each token update, walked from the last token to the first.  With S = H^T and its
// adjoint Shat = Hhat^T (thread (j, part): column j of H and Hhat, its half of the rows d),
// per token t (a = exp(g_t), q^ = scale q_t):
//   Shat += do_t q^^T;   dq_t = scale S_t^T do_t;   u1 = S_{t-1} k_t;  e = v_t - a u1
//   sk = Shat k_t;  dv_t = b sk;  dbeta_t = e . sk;  dk_t = b Shat^T e - a b S_{t-1}^T sk
//   dalpha = <Shat, S_{t-1}> - b sk . u1;  dg_t = a dalpha;  Shat = a (Shat - b sk k_t^T)
// and dh0 = Hhat at the end.  S_{t-1} and S_t come from a forward pass that keeps a
// checkpoint every kRecSeg tokens, each segment's states recomputed into scratch before
// it is walked back (the recurrent forward's own operations, so its states bit for bit).
// Sums over j (dq, dk and the scalars) are fixed-order reductions through shared memory
// and warp trees; deterministic and batch-invariant (one CTA per (sequence, head)).
template <int D, typename IO>
__global__ void __launch_bounds__(2 * D, 1) k_rec_bwd(RecBwdArgs a) {
    extern __shared__ __align__(16) unsigned char smraw[];
    RecBwdSmem<D>& s = *reinterpret_cast<RecBwdSmem<D>*>(smraw);
    constexpr int L = kRecSeg, NW = 2 * D / 32;
    const int tid = threadIdx.x, j = tid % D, part = tid / D, warp = tid >> 5, lane = tid & 31;
    const int H = a.H, b = blockIdx.x / H, h = blockIdx.x % H;
    const int t0 = a.cu[b], t1 = a.cu[b + 1];
    if (t0 < 0 || t1 < t0 || (int64_t)t1 > a.n_tok) {
        if (tid == 0) set_error(a.err, CPR_ERR_BAD_SEQLENS);
        return;
    }
    const IO* q = static_cast<const IO*>(a.q);
    const IO* k = static_cast<const IO*>(a.k);
    const IO* v = static_cast<const IO*>(a.v);
    const size_t sh = (size_t)b * H + h;
    const int nseg = (t1 - t0 + L - 1) / L;
    // this thread's elements of a d x d state: (part * D/2 + i, j)
    auto el = [&](int i) { return (size_t)(part * (D / 2) + i) * D + j; };
    // checkpoint c of this (sequence, head): the state before token t0 + c L
    auto ck = [&](int c) { return a.ckpt + ((size_t)(t0 / L + b + c) * H + h) * D * D; };
    float* segp = a.seg + sh * L * D * D;   // segment state i: after the segment's token i

    float hr[D / 2];
#pragma unroll
    for (int i = 0; i < D / 2; ++i) hr[i] = a.h0 ? a.h0[sh * D * D + el(i)] : 0.f;
    state_loop<D, IO>(hr, s.f, k, v, a.g, a.beta, H, h, t0, t1,
                      [&](int t) {
                          if ((t - t0) % L == 0) {
                              float* c = ck((t - t0) / L);
#pragma unroll
                              for (int i = 0; i < D / 2; ++i) c[el(i)] = hr[i];
                          }
                      },
                      [](int) {});
    float ah[D / 2];   // Hhat
#pragma unroll
    for (int i = 0; i < D / 2; ++i) ah[i] = a.dHT ? a.dHT[sh * D * D + el(i)] : 0.f;

    // the backward token rows: loaded into registers a token ahead, staged in a buffer
    float rq = 0.f, rk = 0.f, rv = 0.f, rdo = 0.f, ra = 0.f, rb = 0.f;
    auto load = [&](int t) {
        if (tid < D) {
            const size_t row = ((size_t)t * H + h) * D + tid;
            rq = __fmul_rn(a.scale, ld_io(q, row));
            rk = ld_io(k, row);
            rv = ld_io(v, row);
            rdo = a.dO[row];
        }
        if (tid == 0) {
            ra = expf(a.g[(size_t)t * H + h]);
            rb = a.beta[(size_t)t * H + h];
        }
    };
    auto store = [&](int buf) {
        if (tid < D) {
            s.tq[buf][tid] = rq;
            s.tk[buf][tid] = rk;
            s.tv[buf][tid] = rv;
            s.tdo[buf][tid] = rdo;
        }
        if (tid == 0) {
            s.tab[buf][0] = ra;
            s.tab[buf][1] = rb;
        }
    };
    for (int c = nseg - 1; c >= 0; --c) {
        const int s0 = t0 + c * L, s1 = min(t1, s0 + L);
        // the segment's states, after each of its tokens, into the scratch
        const float* cst = ck(c);
#pragma unroll
        for (int i = 0; i < D / 2; ++i) hr[i] = cst[el(i)];
        state_loop<D, IO>(hr, s.f, k, v, a.g, a.beta, H, h, s0, s1, [](int) {},
                          [&](int t) {
                              float* dst = segp + (size_t)(t - s0) * D * D;
#pragma unroll
                              for (int i = 0; i < D / 2; ++i) dst[el(i)] = hr[i];
                          });
        // hr is the state after token s1 - 1; walk the segment back
        load(s1 - 1);
        store(0);
        __syncthreads();
        for (int t = s1 - 1; t >= s0; --t) {
            const int cur = (s1 - 1 - t) & 1;
            const bool more = t > s0;
            if (more) load(t - 1);
            const float* qs = s.tq[cur] + part * (D / 2);
            const float* ks = s.tk[cur] + part * (D / 2);
            const float doj = s.tdo[cur][j];
            const float al = s.tab[cur][0], be = s.tab[cur][1];
            // Hhat += do q^^T; dq partials from S_t (in hr)
#pragma unroll
            for (int i = 0; i < D / 2; ++i) {
                ah[i] = __fmaf_rn(doj, qs[i], ah[i]);
                s.Rq[part * (D / 2) + i][j] = __fmul_rn(hr[i], doj);
            }
            // S_{t-1}: the previous token's scratch state, or the segment's checkpoint
            const float* prev = (t > s0) ? segp + (size_t)(t - 1 - s0) * D * D : cst;
#pragma unroll
            for (int i = 0; i < D / 2; ++i) hr[i] = prev[el(i)];
            float pu = 0.f, ps = 0.f, pa = 0.f;
#pragma unroll
            for (int i = 0; i < D / 2; ++i) {
                pu = __fmaf_rn(hr[i], ks[i], pu);
                ps = __fmaf_rn(ah[i], ks[i], ps);
                pa = __fmaf_rn(ah[i], hr[i], pa);
            }
            s.ru[part][j] = pu;
            s.rs[part][j] = ps;
            pa = warp_tree(pa);
            if (lane == 0) s.wsum[0][warp] = pa;
            __syncthreads();
            const size_t row = ((size_t)t * H + h) * D;
            if (tid < D) {   // dq_t[d], d = tid
                float acc = 0.f;
                for (int jj = 0; jj < D; ++jj) acc = __fadd_rn(acc, s.Rq[tid][jj]);
                a.dq[row + tid] = __fmul_rn(a.scale, acc);
            }
            const float u1 = __fadd_rn(s.ru[0][j], s.ru[1][j]);
            const float sk = __fadd_rn(s.rs[0][j], s.rs[1][j]);
            const float e = __fsub_rn(s.tv[cur][j], __fmul_rn(al, u1));
            const float c1 = __fmul_rn(be, e), c2 = __fmul_rn(__fmul_rn(al, be), sk);
#pragma unroll
            for (int i = 0; i < D / 2; ++i)
                s.Rk[part * (D / 2) + i][j] = __fmaf_rn(c1, ah[i], -__fmul_rn(c2, hr[i]));
            float pb = 0.f, pk = 0.f;
            if (part == 0) {
                a.dv[row + j] = __fmul_rn(be, sk);
                pb = __fmul_rn(e, sk);
                pk = __fmul_rn(sk, u1);
            }
            pb = warp_tree(pb);
            pk = warp_tree(pk);
            if (lane == 0) {
                s.wsum[1][warp] = pb;
                s.wsum[2][warp] = pk;
            }
            __syncthreads();
            if (tid < D) {   // dk_t[d], d = tid
                float acc = 0.f;
                for (int jj = 0; jj < D; ++jj) acc = __fadd_rn(acc, s.Rk[tid][jj]);
                a.dk[row + tid] = acc;
            }
            if (tid == 0) {
                float sb = 0.f, sa = 0.f, su = 0.f;
                for (int w = 0; w < NW; ++w) {
                    sa = __fadd_rn(sa, s.wsum[0][w]);
                    sb = __fadd_rn(sb, s.wsum[1][w]);
                    su = __fadd_rn(su, s.wsum[2][w]);
                }
                a.dbeta[(size_t)t * H + h] = sb;
                a.dg[(size_t)t * H + h] = __fmul_rn(al, __fsub_rn(sa, __fmul_rn(be, su)));
            }
            // Hhat = a (Hhat - b sk k^T)
            const float bs = __fmul_rn(be, sk);
#pragma unroll
            for (int i = 0; i < D / 2; ++i) ah[i] = __fmul_rn(al, __fmaf_rn(-bs, ks[i], ah[i]));
            if (more) store(cur ^ 1);
            __syncthreads();
        }
    }
#pragma unroll
    for (int i = 0; i < D / 2; ++i) a.dh0[sh * D * D + el(i)] = ah[i];
}

template <int D, typename IO>
static cudaError_t launch_bwd(const RecBwdArgs& a, cudaStream_t st) {
    const int64_t grid = (int64_t)a.n_seq * a.H;
    const size_t sm = sizeof(RecBwdSmem<D>);
    cudaError_t e = cudaFuncSetAttribute(k_rec_bwd<D, IO>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    if (grid > 0) k_rec_bwd<D, IO><<<(unsigned)grid, 2 * D, sm, st>>>(a);
    return cudaGetLastError();
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

cudaError_t rb_fill_launch(const rec::RbFillArgs& a, cudaStream_t st) {
    const int64_t grid = (int64_t)a.n_seq * a.H;
    if (grid > 0) rec::k_rb_fill<<<(unsigned)grid, 128, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t rec_bwd_launch(const rec::RecBwdArgs& a, int d, bool bf16, cudaStream_t st) {
    if (d == 128) return bf16 ? rec::launch_bwd<128, __nv_bfloat16>(a, st) : rec::launch_bwd<128, float>(a, st);
    if (d == 64) return bf16 ? rec::launch_bwd<64, __nv_bfloat16>(a, st) : rec::launch_bwd<64, float>(a, st);
    return cudaErrorInvalidValue;
}

cudaError_t rec_launch(const rec::RecArgs& a, int d, bool bf16, cudaStream_t st) {
    if (d == 128) return bf16 ? rec::launch<128, __nv_bfloat16>(a, st) : rec::launch<128, float>(a, st);
    if (d == 64) return bf16 ? rec::launch<64, __nv_bfloat16>(a, st) : rec::launch<64, float>(a, st);
    return cudaErrorInvalidValue;
}

}  // namespace cpr
