// CPR Gated DeltaNet forward, prefill and decode kernels: operand policy
// SIMT_F32, within-chunk orders ROWSEQ_V1.
//
// The method (page "IsoExec: 切换 SkyRL 中的训练器-推理不匹配", section
// "Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet"): the gated delta rule
// is evaluated chunk by chunk; chunk states follow each other strictly in
// order (the recurrence is primary), the work inside a chunk is parallel, and
// decode re-synchronises the state every C tokens.  The chunk form is derived
// from the recurrence (the pages name it, they do not write it).  For a
// chunk of n <= C rows with start state H (d_k x d_v):
//   gam_r = gam_{r-1} + g_r  (gam_{-1} = 0; kept as a compensated pair, gam_add),
//   G_r = exp(gam_r)
//   a_rs  = (b_r exp(gam_r - gam_s)) (k_r . k_s)            s < r
//   T     = (I + A)^-1   (unit lower triangular)
//   W'_r  = sum_{s<=r} T_rs (b_s G_s) k_s,   U_r = sum_{s<=r} T_rs b_s v_s
//   D_r   = U_r - W'_r H                                   ("Delta")
//   p_rs  = exp(gam_r - gam_s) (scale q_r . k_s)           s <= r
//   o_r   = G_r (scale q_r) H + sum_{s<=r} p_rs D_s
//   H'    = G_L H + sum_{s<=L} (exp(gam_L - gam_s) k_s) D_s^T,  L = n - 1
//
// Bitwise consistency between prefill and decode.  Every quantity of row r
// depends only on rows <= r and on H, and every one is produced by the SAME
// per-entry operation sequence in both paths: an fp32 fma chain from +0 in
// ascending index order, the scalar helpers below, and the same expf call.
// The prefill kernels run chains over whole tiles, so rows shorter than the
// tile see extra terms whose first factor is an exact +0 (T_rs for s > r,
// p_rs for s > r).  Such a term leaves the accumulator's bits unchanged: an
// fma with a zero product returns acc + (+-0), which is acc unless acc is
// -0, and a chain started at +0 never holds -0 (round-to-nearest gives +0 for
// an exact zero sum unless both addends are -0).  Inputs are finite.  The
// decode step therefore evaluates only the chains of its own row and
// reproduces the prefill's bits exactly.  All arithmetic uses the _rn
// intrinsics, which the compiler never contracts or reorders.
#pragma once

#include "common.cuh"

namespace cpr {
namespace simt {

// ---- scalar arithmetic shared by every path --------------------------------
// In-chunk gate prefix gam_r = sum_{s<=r} g_s, in token order, carried as the
// unevaluated pair hi + lo: hi is the plain fp32 running sum and lo collects the
// exact rounding error of each of its additions (Knuth's TwoSum).  Reason: after a
// strong gate (g << 0, e.g. a reset with alpha ~ 0) |gam| is large, and a single
// fp32 running sum rounds every later log-gate to the spacing of |gam| (about 1e-3
// at |gam| = 1e4), so exp(gam_r - gam_s) between two later tokens would be off by
// a relative 1e-3.  With the pair, hi_r - hi_s is exact whenever the two are
// within a factor of two (Sterbenz), and the exponent below is accurate to a few
// units in the last place of its own size.  (hi, lo) start at (0, 0) in every
// chunk; every path advances them with this one function.
__device__ __forceinline__ void gam_add(float& hi, float& lo, float g) {
    const float s = __fadd_rn(hi, g);
    const float bp = __fsub_rn(s, hi);
    const float ap = __fsub_rn(s, bp);
    const float err = __fadd_rn(__fsub_rn(hi, ap), __fsub_rn(g, bp));
    hi = s;
    lo = __fadd_rn(lo, err);
}
// gam_r - gam_s from the two pairs.
__device__ __forceinline__ float gam_diff(float hr, float lr, float hs, float ls) {
    return __fadd_rn(__fsub_rn(hr, hs), __fsub_rn(lr, ls));
}
// exp(gam_r - gam_s) (s <= r: <= 1) and exp(gam_r).
__device__ __forceinline__ float decay(float hr, float lr, float hs, float ls) {
    return expf(gam_diff(hr, lr, hs, ls));
}
__device__ __forceinline__ float gate(float hr, float lr) { return expf(__fadd_rn(hr, lr)); }
__device__ __forceinline__ float a_entry(float beta_r, float hr, float lr, float hs, float ls, float kk) {
    return __fmul_rn(__fmul_rn(beta_r, decay(hr, lr, hs, ls)), kk);
}
__device__ __forceinline__ float p_entry(float hr, float lr, float hs, float ls, float qk) {
    return __fmul_rn(decay(hr, lr, hs, ls), qk);
}
__device__ __forceinline__ float bg_entry(float beta, float hr, float lr) { return __fmul_rn(beta, gate(hr, lr)); }
__device__ __forceinline__ float qhat(float scale, float q) { return __fmul_rn(scale, q); }

// ---- tiled fma chains over shared-memory operands ----------------------------
// For every tile (m0..m0+TM-1, n0..n0+TN-1) of an M x N result:
//   acc[i][j] = init(m, n);  for kk in [k0, k1): acc = fma(A(m, kk), B(kk, n), acc)
// with [k0, k1) = krange(m0) and then epi(m0, n0, acc).  Each entry's chain is
// the ascending-index chain of its definition.
template <int TM, int TN, class FI, class FA, class FB, class FK, class FE>
__device__ __forceinline__ void tile_mm(int M, int N, FI init, FA fa, FB fb, FK krange, FE epi) {
    const int tiles_n = N / TN;
    const int ntiles = (M / TM) * tiles_n;
    for (int t = threadIdx.x; t < ntiles; t += blockDim.x) {
        const int m0 = (t / tiles_n) * TM, n0 = (t % tiles_n) * TN;
        int k0, k1;
        krange(m0, k0, k1);
        float acc[TM][TN];
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) acc[i][j] = init(m0 + i, n0 + j);
        for (int kk = k0; kk < k1; ++kk) {
            float av[TM], bv[TN];
#pragma unroll
            for (int i = 0; i < TM; ++i) av[i] = fa(m0 + i, kk);
#pragma unroll
            for (int j = 0; j < TN; ++j) bv[j] = fb(kk, n0 + j);
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = __fmaf_rn(av[i], bv[j], acc[i][j]);
        }
        epi(m0, n0, acc);
    }
}

struct Zero {
    __device__ __forceinline__ float operator()(int, int) const { return 0.f; }
};

// ---- arguments ------------------------------------------------------------------
struct FwdArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* g;
    const float* beta;
    const int32_t* cu;
    const int32_t* chunk_off;   // [n_seq + 1] in workspace
    int n_seq;
    int H;
    float scale;
    // per (chunk, head) workspace arrays
    float* wsW;     // [chunks, H, C, d_k]
    float* wsU;     // [chunks, H, C, d_v]
    float* wsP;     // [chunks, H, C, C]
    float* wsGam;   // [chunks, H, C]
    float* wsT;     // [chunks, H, C, C]  or null
    float* wsKd;    // [chunks, H, C, C]  decay(r,s) (k_r.k_s), s < r, or null
    float* wsHn;    // [chunks, H, d_k, d_v] chunk-start states, or null
    const float* h0;
    void* o;              // null: do not produce outputs
    float* final_state;   // null: not written
    uint8_t* cache;       // null: no decode cache
    CacheOff co;
    uint32_t* err;
};

// ---- setup: validate cu_seqlens, chunk table, cache header ---------------------
struct SetupArgs {
    const int32_t* cu;
    int n_seq;
    int64_t n_tok;
    int32_t* chunk_off;
    uint8_t* cache;
    CacheOff co;
    Digest digest;
    uint32_t hdr[kHdrWords];   // n_seq, H, C, d_k, d_v, policy, io dtype, deployment digest
    uint32_t* err;
};

static __global__ void k_setup(SetupArgs a) {
    __shared__ int ok_s;
    if (threadIdx.x == 0) {
        bool ok = a.cu[0] == 0 && (int64_t)a.cu[a.n_seq] == a.n_tok;
        int32_t acc = 0;
        for (int b = 0; b < a.n_seq; ++b) {
            const int32_t T = a.cu[b + 1] - a.cu[b];
            if (T < 0) ok = false;
            a.chunk_off[b] = acc;
            if (T > 0) acc += (int32_t)(((int64_t)T + kChunk - 1) / kChunk);
        }
        a.chunk_off[a.n_seq] = ok ? acc : -1;
        if (!ok) set_error(a.err, CPR_ERR_BAD_SEQLENS);
        ok_s = ok;
    }
    __syncthreads();
    if (!a.cache || !ok_s) return;
    uint32_t* hdr = reinterpret_cast<uint32_t*>(a.cache + a.co.header);
    if (threadIdx.x == 0) {
        hdr[0] = kCacheMagic;
        hdr[1] = CPR_CONTRACT_VERSION;
        for (int i = 0; i < 8; ++i) hdr[2 + i] = a.digest.w[i];
        for (int i = 0; i < kHdrWords; ++i) hdr[10 + i] = a.hdr[i];
    }
    int32_t* pos = reinterpret_cast<int32_t*>(a.cache + a.co.pos);
    uint32_t* done = reinterpret_cast<uint32_t*>(a.cache + a.co.done);
    for (int b = threadIdx.x; b < a.n_seq; b += blockDim.x) {
        pos[b] = (a.cu[b + 1] - a.cu[b]) % kChunk;
        done[b] = 0u;
    }
}

// ---- prep: per (chunk, head), everything that does not depend on H ------------
// Writes P, W', U, gam (and T, Kd) to the workspace; for the last, partial
// chunk of a sequence it also stores the rows the decode steps need in the
// cache.
template <class IO, int DK, int DV>
__global__ void __launch_bounds__(256) k_prep(FwdArgs a) {
    constexpr int C = kChunk;
    constexpr int LK = DK + 8, LV = DV + 8, LC = C + 1;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    IO* Ks = reinterpret_cast<IO*>(smem_raw);
    IO* Qs = Ks + C * LK;
    IO* Vs = Qs + C * LK;
    float* A = reinterpret_cast<float*>(Vs + C * LV);
    float* Tm = A + C * LC;
    float* gam = Tm + C * LC;   // gate prefix, hi
    float* gml = gam + C;       // gate prefix, lo
    float* bet = gml + C;
    float* bg = bet + C;

    const int total = a.chunk_off[a.n_seq];
    const int cidx = blockIdx.x, h = blockIdx.y, H = a.H;
    if (total < 0 || cidx >= total) return;
    const int b = find_seq(a.chunk_off, a.n_seq, cidx);
    const int n = cidx - a.chunk_off[b];
    const int seq0 = a.cu[b], T = a.cu[b + 1] - seq0;
    const int t0 = seq0 + n * C;
    const int nrows = min(C, T - n * C);
    const bool last = (n * C + nrows == T);
    const int tid = threadIdx.x;
    const IO* q = static_cast<const IO*>(a.q);
    const IO* k = static_cast<const IO*>(a.k);
    const IO* v = static_cast<const IO*>(a.v);

    // rows -> shared (io dtype, zero padded)
    for (int i = tid; i < C * (DK / 8); i += blockDim.x) {
        const int r = i / (DK / 8), c8 = (i % (DK / 8)) * 8;
        float kv[8], qv[8];
        if (r < nrows) {
            load8(k + ((size_t)(t0 + r) * H + h) * DK + c8, kv);
            load8(q + ((size_t)(t0 + r) * H + h) * DK + c8, qv);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) kv[e] = qv[e] = 0.f;
        }
        store8(Ks + r * LK + c8, kv);
        store8(Qs + r * LK + c8, qv);
    }
    for (int i = tid; i < C * (DV / 8); i += blockDim.x) {
        const int r = i / (DV / 8), c8 = (i % (DV / 8)) * 8;
        float vv[8];
        if (r < nrows) {
            load8(v + ((size_t)(t0 + r) * H + h) * DV + c8, vv);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) vv[e] = 0.f;
        }
        store8(Vs + r * LV + c8, vv);
    }
    if (tid < C) {
        gam[tid] = (tid < nrows) ? a.g[(size_t)(t0 + tid) * H + h] : 0.f;
        gml[tid] = 0.f;
        bet[tid] = (tid < nrows) ? a.beta[(size_t)(t0 + tid) * H + h] : 0.f;
    }
    __syncthreads();
    if (tid == 0) {  // gate prefix: serial compensated sum in token order
        float hi = 0.f, lo = 0.f;
        for (int r = 0; r < nrows; ++r) {
            gam_add(hi, lo, gam[r]);
            gam[r] = hi;
            gml[r] = lo;
        }
    }
    __syncthreads();
    if (tid < C) bg[tid] = (tid < nrows) ? bg_entry(bet[tid], gam[tid], gml[tid]) : 0.f;

    // A = strict_lower(b_r decay kk) (and Kd), P = lower(decay qk) -> workspace
    const size_t ch = (size_t)cidx * H + h;
    float* P = a.wsP + ch * C * C;
    float* Kd = a.wsKd ? a.wsKd + ch * C * C : nullptr;
    const float scale = a.scale;
    auto kr = [&](int m0, int& k0, int& k1) { k0 = 0; k1 = DK; (void)m0; };
    tile_mm<4, 4>(C, C, Zero{},
        [&](int m, int d) { return cvt(Ks[m * LK + d]); },
        [&](int d, int s) { return cvt(Ks[s * LK + d]); },
        kr,
        [&](int m0, int n0, float (&acc)[4][4]) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int r = m0 + i, s = n0 + j;
                    const bool in = (s < r && r < nrows);
                    A[r * LC + s] = in ? a_entry(bet[r], gam[r], gml[r], gam[s], gml[s], acc[i][j]) : 0.f;
                    if (Kd) Kd[r * C + s] = in ? __fmul_rn(decay(gam[r], gml[r], gam[s], gml[s]), acc[i][j]) : 0.f;
                }
        });
    tile_mm<4, 4>(C, C, Zero{},
        [&](int m, int d) { return qhat(scale, cvt(Qs[m * LK + d])); },
        [&](int d, int s) { return cvt(Ks[s * LK + d]); },
        kr,
        [&](int m0, int n0, float (&acc)[4][4]) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float out[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int r = m0 + i, s = n0 + j;
                    out[j] = (s <= r && r < nrows) ? p_entry(gam[r], gml[r], gam[s], gml[s], acc[i][j]) : 0.f;
                }
                *reinterpret_cast<float4*>(P + (m0 + i) * C + n0) = make_float4(out[0], out[1], out[2], out[3]);
            }
        });
    __syncthreads();

    // T = (I + A)^-1 by columns: T_rj = -(sum_{s=j}^{r-1} a_rs T_sj), ascending s
    if (tid < C) {
        const int j = tid;
        for (int r = 0; r < C; ++r) Tm[r * LC + j] = (r == j && r < nrows) ? 1.f : 0.f;
        for (int r = j + 1; r < nrows; ++r) {
            float acc = 0.f;
            for (int s = j; s < r; ++s) acc = __fmaf_rn(A[r * LC + s], Tm[s * LC + j], acc);
            Tm[r * LC + j] = -acc;
        }
    }
    __syncthreads();

    // W' = T diag(b G) K,  U = T diag(b) V  (chains over s ascending from 0)
    float* W = a.wsW + ch * C * DK;
    float* U = a.wsU + ch * C * DV;
    auto tri = [&](int m0, int& k0, int& k1) { k0 = 0; k1 = min(m0 + 4, nrows); };
    tile_mm<4, 4>(C, DK, Zero{},
        [&](int r, int s) { return Tm[r * LC + s]; },
        [&](int s, int d) { return __fmul_rn(bg[s], cvt(Ks[s * LK + d])); },
        tri,
        [&](int m0, int n0, float (&acc)[4][4]) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                *reinterpret_cast<float4*>(W + (m0 + i) * DK + n0) =
                    make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        });
    tile_mm<4, 4>(C, DV, Zero{},
        [&](int r, int s) { return Tm[r * LC + s]; },
        [&](int s, int j) { return __fmul_rn(bet[s], cvt(Vs[s * LV + j])); },
        tri,
        [&](int m0, int n0, float (&acc)[4][4]) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                *reinterpret_cast<float4*>(U + (m0 + i) * DV + n0) =
                    make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        });
    if (tid < C) {
        a.wsGam[ch * 2 * C + tid] = gam[tid];
        a.wsGam[ch * 2 * C + C + tid] = gml[tid];
    }
    if (a.wsT) {
        float* Tw = a.wsT + ch * C * C;
        for (int i = tid; i < C * C; i += blockDim.x) Tw[i] = Tm[(i / C) * LC + (i % C)];
    }
    // decode cache: rows of the sequence's last chunk when it is partial
    if (a.cache && last && nrows < C) {
        const size_t sh = (size_t)b * H + h;
        IO* ck = reinterpret_cast<IO*>(a.cache + a.co.k_rows) + sh * C * DK;
        IO* cv = reinterpret_cast<IO*>(a.cache + a.co.v_rows) + sh * C * DV;
        float* cg = reinterpret_cast<float*>(a.cache + a.co.gam_rows) + sh * 2 * C;
        float* cb = reinterpret_cast<float*>(a.cache + a.co.beta_rows) + sh * C;
        float* ct = reinterpret_cast<float*>(a.cache + a.co.t_rows) + sh * C * C;
        for (int i = tid; i < nrows * DK; i += blockDim.x)
            ck[i] = k[((size_t)(t0 + i / DK) * H + h) * DK + i % DK];
        for (int i = tid; i < nrows * DV; i += blockDim.x)
            cv[i] = v[((size_t)(t0 + i / DV) * H + h) * DV + i % DV];
        if (tid < nrows) {
            cg[tid] = gam[tid];
            cg[C + tid] = gml[tid];
            cb[tid] = bet[tid];
        }
        for (int i = tid; i < nrows * C; i += blockDim.x) ct[i] = Tm[(i / C) * LC + (i % C)];
    }
}

// ---- state pass: sequential over the chunks of one (sequence, head, d_v split) ---
template <class IO, int DK, int DV, int DVS>
__global__ void __launch_bounds__(256) k_state_fwd(FwdArgs a) {
    constexpr int C = kChunk;
    constexpr int LK = DK + 4, LKI = DK + 8, LS = DVS + 4, LC = C + 4;
    constexpr int NSPLIT = DV / DVS;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float* Ws = reinterpret_cast<float*>(smem_raw);   // [C][LK]   W' rows
    float* Ps = Ws + C * LK;                          // [C][LC]   p_rs
    float* Hs = Ps + C * LC;                          // [DK][LS]  state columns
    float* Ds = Hs + DK * LS;                         // [C][LS]   U, then Delta
    float* QH = Ds + C * LS;                          // [C][LS]
    float* gam = QH + C * LS;                         // [C] gate prefix, hi
    float* gml = gam + C;                             // [C] gate prefix, lo
    float* dec = gml + C;                             // [C]
    IO* Qs = reinterpret_cast<IO*>(dec + C);          // [C][LKI]
    IO* Ks = Qs + C * LKI;                            // [C][LKI]

    const int total = a.chunk_off[a.n_seq];
    if (total < 0) return;
    const int H = a.H;
    const int sp = blockIdx.x % NSPLIT;
    const int h = (blockIdx.x / NSPLIT) % H;
    const int b = blockIdx.x / (NSPLIT * H);
    const int j0 = sp * DVS;
    const int tid = threadIdx.x;
    const int seq0 = a.cu[b], T = a.cu[b + 1] - seq0;
    const int nch = a.chunk_off[b + 1] - a.chunk_off[b];
    const IO* q = static_cast<const IO*>(a.q);
    const IO* k = static_cast<const IO*>(a.k);
    float* o = static_cast<float*>(a.o);
    const size_t sh = (size_t)b * H + h;
    const float scale = a.scale;

    for (int i = tid; i < DK * DVS; i += blockDim.x) {
        const int d = i / DVS, j = i % DVS;
        Hs[d * LS + j] = a.h0 ? a.h0[(sh * DK + d) * DV + j0 + j] : 0.f;
    }
    float* cstate = a.cache ? reinterpret_cast<float*>(a.cache + a.co.state) + sh * DK * DV : nullptr;
    if (nch == 0 && cstate) {
        __syncthreads();
        for (int i = tid; i < DK * DVS; i += blockDim.x)
            cstate[(i / DVS) * DV + j0 + i % DVS] = Hs[(i / DVS) * LS + i % DVS];
    }

    for (int n = 0; n < nch; ++n) {
        const int cidx = a.chunk_off[b] + n;
        const int t0 = seq0 + n * C;
        const int nrows = min(C, T - n * C);
        const bool last = (n == nch - 1);
        const size_t ch = (size_t)cidx * H + h;
        __syncthreads();  // previous chunk fully consumed
        const float* W = a.wsW + ch * C * DK;
        for (int i = tid; i < C * DK / 4; i += blockDim.x) {
            const int r = i / (DK / 4), c4 = (i % (DK / 4)) * 4;
            *reinterpret_cast<float4*>(Ws + r * LK + c4) = *reinterpret_cast<const float4*>(W + r * DK + c4);
        }
        const float* P = a.wsP + ch * C * C;
        for (int i = tid; i < C * C / 4; i += blockDim.x) {
            const int r = i / (C / 4), c4 = (i % (C / 4)) * 4;
            *reinterpret_cast<float4*>(Ps + r * LC + c4) = *reinterpret_cast<const float4*>(P + r * C + c4);
        }
        const float* U = a.wsU + ch * C * DV;
        for (int i = tid; i < C * DVS / 4; i += blockDim.x) {
            const int r = i / (DVS / 4), c4 = (i % (DVS / 4)) * 4;
            *reinterpret_cast<float4*>(Ds + r * LS + c4) = *reinterpret_cast<const float4*>(U + r * DV + j0 + c4);
        }
        for (int i = tid; i < C * (DK / 8); i += blockDim.x) {
            const int r = i / (DK / 8), c8 = (i % (DK / 8)) * 8;
            float kv[8], qv[8];
            if (r < nrows) {
                load8(k + ((size_t)(t0 + r) * H + h) * DK + c8, kv);
                load8(q + ((size_t)(t0 + r) * H + h) * DK + c8, qv);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) kv[e] = qv[e] = 0.f;
            }
            store8(Ks + r * LKI + c8, kv);
            store8(Qs + r * LKI + c8, qv);
        }
        if (tid < C) {
            gam[tid] = a.wsGam[ch * 2 * C + tid];
            gml[tid] = a.wsGam[ch * 2 * C + C + tid];
        }
        if (a.wsHn) {  // chunk-start state (backward)
            float* Hn = a.wsHn + ch * DK * DV;
            for (int i = tid; i < DK * DVS; i += blockDim.x)
                Hn[(i / DVS) * DV + j0 + i % DVS] = Hs[(i / DVS) * LS + i % DVS];
        }
        __syncthreads();
        // Delta = U - W' H  (rows 0..C-1) and QH = (scale q) H (rows C..2C-1)
        const bool want_o = (o != nullptr);
        tile_mm<4, 4>(want_o ? 2 * C : C, DVS, Zero{},
            [&](int m, int d) { return m < C ? Ws[m * LK + d] : qhat(scale, cvt(Qs[(m - C) * LKI + d])); },
            [&](int d, int j) { return Hs[d * LS + j]; },
            [&](int m0, int& k0, int& k1) { k0 = 0; k1 = DK; (void)m0; },
            [&](int m0, int n0, float (&acc)[4][4]) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int m = m0 + i, jj = n0 + j;
                        if (m < C) Ds[m * LS + jj] = (m < nrows) ? __fsub_rn(Ds[m * LS + jj], acc[i][j]) : 0.f;
                        else QH[(m - C) * LS + jj] = acc[i][j];
                    }
            });
        __syncthreads();
        if (last && nrows < C && cstate) {  // decode cache: chunk-start state + Delta rows
            for (int i = tid; i < DK * DVS; i += blockDim.x)
                cstate[(i / DVS) * DV + j0 + i % DVS] = Hs[(i / DVS) * LS + i % DVS];
            float* cd = reinterpret_cast<float*>(a.cache + a.co.delta_rows) + sh * C * DV;
            for (int i = tid; i < nrows * DVS; i += blockDim.x)
                cd[(i / DVS) * DV + j0 + i % DVS] = Ds[(i / DVS) * LS + i % DVS];
        }
        if (want_o) {
            // o_r = G_r QH_r + sum_{s<=r} p_rs D_s
            tile_mm<2, 4>(C, DVS,
                [&](int r, int j) { return __fmul_rn(gate(gam[r], gml[r]), QH[r * LS + j]); },
                [&](int r, int s) { return Ps[r * LC + s]; },
                [&](int s, int j) { return Ds[s * LS + j]; },
                [&](int m0, int& k0, int& k1) { k0 = 0; k1 = min(m0 + 2, nrows); },
                [&](int m0, int n0, float (&acc)[2][4]) {
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const int r = m0 + i;
                        if (r < nrows)
                            *reinterpret_cast<float4*>(o + ((size_t)(t0 + r) * H + h) * DV + j0 + n0) =
                                make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
                    }
                });
        }
        // commit: H' = G_L H + sum_{s<=L} (decay(L, s) k_s) D_s^T
        const int L = nrows - 1;
        if (tid < C) dec[tid] = (tid < nrows) ? decay(gam[L], gml[L], gam[tid], gml[tid]) : 0.f;
        __syncthreads();
        const float GL = gate(gam[L], gml[L]);
        tile_mm<4, 4>(DK, DVS,
            [&](int d, int j) { return __fmul_rn(GL, Hs[d * LS + j]); },
            [&](int d, int s) { return __fmul_rn(dec[s], cvt(Ks[s * LKI + d])); },
            [&](int s, int j) { return Ds[s * LS + j]; },
            [&](int m0, int& k0, int& k1) { k0 = 0; k1 = nrows; (void)m0; },
            [&](int m0, int n0, float (&acc)[4][4]) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) Hs[(m0 + i) * LS + n0 + j] = acc[i][j];
            });
        if (last && nrows == C && cstate) {
            __syncthreads();
            for (int i = tid; i < DK * DVS; i += blockDim.x)
                cstate[(i / DVS) * DV + j0 + i % DVS] = Hs[(i / DVS) * LS + i % DVS];
        }
    }
    if (a.final_state) {
        __syncthreads();
        for (int i = tid; i < DK * DVS; i += blockDim.x)
            a.final_state[(sh * DK + i / DVS) * DV + j0 + i % DVS] = Hs[(i / DVS) * LS + i % DVS];
    }
}

template <class IO, int DK, int DV, int DVS>
constexpr size_t state_fwd_smem() {
    return sizeof(float) * ((size_t)kChunk * (DK + 4) + kChunk * (kChunk + 4) + DK * (DVS + 4) +
                            2 * kChunk * (DVS + 4) + 3 * kChunk) +
           sizeof(IO) * 2 * kChunk * (DK + 8);
}
template <class IO, int DK, int DV>
constexpr size_t prep_smem() {
    return sizeof(IO) * ((size_t)2 * kChunk * (DK + 8) + kChunk * (DV + 8)) +
           sizeof(float) * (2 * kChunk * (kChunk + 1) + 4 * kChunk);
}

// ---- decode: one token per sequence, one CTA per (sequence, head) ---------------
struct DecArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* g;
    const float* beta;
    int n_seq;
    int H;
    float scale;
    uint8_t* cache;
    CacheOff co;
    Digest digest;
    uint32_t hdr[kHdrWords];
    float* o;
    uint32_t* err;
};

template <class IO, int DK, int DV>
__global__ void __launch_bounds__(128) k_decode(DecArgs a) {
    constexpr int C = kChunk;
    __shared__ float kp[DK], qp[DK], vp[DV], Wp[DK], Up[DV], Dp[DV];
    __shared__ float arow[C], prow[C], trow[C], gams[C], gmls[C], bets[C], bgs[C];
    __shared__ int ok_s;
    const int tid = threadIdx.x;
    const int H = a.H;
    const int b = blockIdx.x / H, h = blockIdx.x % H;
    const uint32_t* hdr = reinterpret_cast<const uint32_t*>(a.cache + a.co.header);
    int32_t* pos = reinterpret_cast<int32_t*>(a.cache + a.co.pos);
    uint32_t* done = reinterpret_cast<uint32_t*>(a.cache + a.co.done);
    if (tid < 32) {   // the header (a word per lane), then the position once it is right
        bool ok = cache_header_ok(hdr, a.digest.w, a.hdr);
        if (tid == 0) {
            const int p = ok ? pos[b] : -1;
            if (!(p >= 0 && p < C)) ok = false;
            if (!ok) set_error(a.err, CPR_ERR_CONTRACT_MISMATCH);
            ok_s = ok ? 1 + p : 0;
        }
    }
    __syncthreads();
    if (!ok_s) return;
    const int p = ok_s - 1;
    const size_t sh = (size_t)b * H + h;
    const IO* ck = reinterpret_cast<const IO*>(a.cache + a.co.k_rows) + sh * C * DK;
    const IO* cv = reinterpret_cast<const IO*>(a.cache + a.co.v_rows) + sh * C * DV;
    float* cg = reinterpret_cast<float*>(a.cache + a.co.gam_rows) + sh * 2 * C;   // hi | lo
    float* cb = reinterpret_cast<float*>(a.cache + a.co.beta_rows) + sh * C;
    float* ct = reinterpret_cast<float*>(a.cache + a.co.t_rows) + sh * C * C;
    float* cd = reinterpret_cast<float*>(a.cache + a.co.delta_rows) + sh * C * DV;
    float* Hst = reinterpret_cast<float*>(a.cache + a.co.state) + sh * DK * DV;
    const IO* q = static_cast<const IO*>(a.q) + sh * DK;
    const IO* k = static_cast<const IO*>(a.k) + sh * DK;
    const IO* v = static_cast<const IO*>(a.v) + sh * DV;

    for (int d = tid; d < DK; d += blockDim.x) {
        kp[d] = cvt(k[d]);
        qp[d] = qhat(a.scale, cvt(q[d]));
    }
    for (int j = tid; j < DV; j += blockDim.x) vp[j] = cvt(v[j]);
    if (tid < p) {
        gams[tid] = cg[tid];
        gmls[tid] = cg[C + tid];
        bets[tid] = cb[tid];
    }
    if (tid == 0) {
        float hi = p > 0 ? cg[p - 1] : 0.f, lo = p > 0 ? cg[C + p - 1] : 0.f;
        gam_add(hi, lo, a.g[sh]);
        gams[p] = hi;
        gmls[p] = lo;
        bets[p] = a.beta[sh];
    }
    __syncthreads();
    if (tid <= p) bgs[tid] = bg_entry(bets[tid], gams[tid], gmls[tid]);
    const float gp = gams[p], lp = gmls[p], bp = bets[p];
    // a_ps (s < p) and p_ps (s <= p): dot chains over d ascending
    if (tid < C) {
        const int s = tid;
        if (s < p) {
            float acc = 0.f;
            for (int d = 0; d < DK; ++d) acc = __fmaf_rn(kp[d], cvt(ck[s * DK + d]), acc);
            arow[s] = a_entry(bp, gp, lp, gams[s], gmls[s], acc);
        } else {
            arow[s] = 0.f;
        }
    } else {
        const int s = tid - C;
        if (s <= p) {
            float acc = 0.f;
            for (int d = 0; d < DK; ++d)
                acc = __fmaf_rn(qp[d], s == p ? kp[d] : cvt(ck[s * DK + d]), acc);
            prow[s] = p_entry(gp, lp, gams[s], gmls[s], acc);
        }
    }
    __syncthreads();
    // T row p
    if (tid < C) {
        const int j = tid;
        float t = 0.f;
        if (j < p) {
            float acc = 0.f;
            for (int s = j; s < p; ++s) acc = __fmaf_rn(arow[s], ct[s * C + j], acc);
            t = -acc;
        } else if (j == p) {
            t = 1.f;
        }
        trow[j] = t;
    }
    __syncthreads();
    // W'_p, U_p: chains over s = 0..p
    for (int d = tid; d < DK; d += blockDim.x) {
        float acc = 0.f;
        for (int s = 0; s <= p; ++s)
            acc = __fmaf_rn(trow[s], __fmul_rn(bgs[s], s == p ? kp[d] : cvt(ck[s * DK + d])), acc);
        Wp[d] = acc;
    }
    for (int j = tid; j < DV; j += blockDim.x) {
        float acc = 0.f;
        for (int s = 0; s <= p; ++s)
            acc = __fmaf_rn(trow[s], __fmul_rn(bets[s], s == p ? vp[j] : cvt(cv[s * DV + j])), acc);
        Up[j] = acc;
    }
    __syncthreads();
    // Delta_p = U_p - W'_p H ; qh = (scale q_p) H ; o_p
    for (int j = tid; j < DV; j += blockDim.x) {
        float wh = 0.f, qh = 0.f;
        for (int d = 0; d < DK; ++d) {
            const float hv = Hst[d * DV + j];
            wh = __fmaf_rn(Wp[d], hv, wh);
            qh = __fmaf_rn(qp[d], hv, qh);
        }
        const float dp = __fsub_rn(Up[j], wh);
        Dp[j] = dp;
        float acc = __fmul_rn(gate(gp, lp), qh);
        for (int s = 0; s <= p; ++s) acc = __fmaf_rn(prow[s], s == p ? dp : cd[s * DV + j], acc);
        a.o[sh * DV + j] = acc;
    }
    __syncthreads();
    // append row p
    IO* ckw = reinterpret_cast<IO*>(a.cache + a.co.k_rows) + sh * C * DK;
    IO* cvw = reinterpret_cast<IO*>(a.cache + a.co.v_rows) + sh * C * DV;
    for (int d = tid; d < DK; d += blockDim.x) ckw[p * DK + d] = k[d];
    for (int j = tid; j < DV; j += blockDim.x) {
        cvw[p * DV + j] = v[j];
        cd[p * DV + j] = Dp[j];
    }
    if (tid < C) ct[p * C + tid] = trow[tid];
    if (tid == 0) {
        cg[p] = gp;
        cg[C + p] = lp;
        cb[p] = bp;
    }
    if (p == C - 1) {  // resynchronise: commit H_{n+1}
        __syncthreads();
        const int L = C - 1;
        if (tid < C) arow[tid] = decay(gams[L], gmls[L], gams[tid], gmls[tid]);
        __syncthreads();
        const float GL = gate(gams[L], gmls[L]);
        for (int i = tid; i < DK * DV; i += blockDim.x) {
            const int d = i / DV, j = i % DV;
            float acc = __fmul_rn(GL, Hst[d * DV + j]);
            for (int s = 0; s < C; ++s)
                acc = __fmaf_rn(__fmul_rn(arow[s], s == p ? kp[d] : cvt(ck[s * DK + d])),
                                s == p ? Dp[j] : cd[s * DV + j], acc);
            Hst[d * DV + j] = acc;
        }
    }
    // advance the sequence position once every head of the sequence is done
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const uint32_t prev = atomicAdd(&done[b], 1u);
        if (prev == (uint32_t)H - 1) {
            pos[b] = (p + 1) % C;
            done[b] = 0u;
            __threadfence();
        }
    }
}

}  // namespace simt
}  // namespace cpr
