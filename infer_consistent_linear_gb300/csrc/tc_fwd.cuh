// CPR Gated DeltaNet forward / prefill on the tensor cores: operand policy
// TC_BF16X3 (see cpr_gdn.h), bf16 io, d_k = d_v = 128, C = 64.
//
// Same chunk form as the SIMT kernels (page "IsoExec: 切换 SkyRL 中的训练器-
// 推理不匹配", section "Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet";
// the form is derived from the gated delta rule):
//   S1   = [K; Q] K^T                      (exact bf16 inputs, one MMA group)
//   a_rs = (b_r exp(gam_r - gam_s)) kk_rs       s < r
//   p_rs = exp(gam_r - gam_s) (scale qk_rs)     s <= r
//   T    = (I + A)^-1                       (fp32 column chains)
//   W'   = (T diag(b G)) K,   U = (T diag(b)) V     (split A operand: hi + lo)
//   acc4 = [W'; Q] H                        (hi*hi + hi*lo + lo*hi)
//   D    = U - acc4[rows 0..63],   qh = acc4[rows 64..127]
//   pd   = P D                              (hi*hi + hi*lo + lo*hi)
//   o_r  = G_r (scale qh_r) + pd_r
//   H'   = G_L H + K^T (diag(exp(gam_L - gam_s)) D)    (exact K, split D)
// Kernels: k_tc_prep (one CTA per chunk and head, everything independent of
// H, written to the workspace in the operand layouts the tensor core reads)
// and k_tc_state (one CTA per (sequence, head, d_v split), strictly in chunk
// order, the H-dependent part with the workspace tiles streamed in by bulk
// async copies).
#pragma once

#include "simt_fwd.cuh"
#include "tc_common.cuh"

namespace cpr {
namespace tc {

constexpr int D = 128;
constexpr int C = kChunk;

// Per (chunk, head) workspace block (bytes).
constexpr size_t kOffA4hi = 0;        // 128 x 128 bf16: rows 0..63 W'_hi, 64..127 Q
constexpr size_t kOffA4lo = 32768;    // 64 x 128 bf16: W'_lo
constexpr size_t kOffKt = 49152;      // 128 x 64 bf16: K^T (rows d, K dim s)
constexpr size_t kOffPhi = 65536;     // 64 x 64 bf16
constexpr size_t kOffPlo = 73728;     // 64 x 64 bf16
constexpr size_t kOffU = 81920;       // 64 x 128 fp32, stored [split][64][DVS]
constexpr size_t kOffGam = 114688;    // 64 fp32
constexpr size_t kBlock = 114944;

struct TcArgs {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const float* g;
    const float* beta;
    const int32_t* cu;
    const int32_t* chunk_off;
    int n_seq;
    int H;
    int dvs;              // d_v columns per state CTA
    float scale;
    unsigned char* ws;    // [chunks * H] blocks of kBlock bytes
    const float* h0;
    float* o;
    float* final_state;
    uint8_t* cache;
    CacheOff co;
    uint32_t* err;
};

// Transposes an 8 x 8 bf16 block: in[j] holds row j (8 values); writes the
// 8 rows of the transpose (row i = {in[0][i], ..., in[7][i]}) as one core matrix.
__device__ __forceinline__ void transpose8_store(const uint4 (&in)[8], unsigned char* core) {
    const __nv_bfloat16* e[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) e[j] = reinterpret_cast<const __nv_bfloat16*>(&in[j]);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        __align__(16) __nv_bfloat16 row[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) row[j] = e[j][i];
        *reinterpret_cast<uint4*>(core + 16 * i) = *reinterpret_cast<const uint4*>(row);
    }
}

__device__ __forceinline__ uint4 ld16_or_zero(const __nv_bfloat16* p, bool valid) {
    return valid ? *reinterpret_cast<const uint4*>(p) : make_uint4(0u, 0u, 0u, 0u);
}

// ---- prep: everything of a chunk that does not depend on H ------------------------
constexpr size_t kPrepSmem = 65536 + 2 * 64 * 65 * 4 + 4 * 64 * 4 + 64;

static __global__ void __launch_bounds__(128) k_tc_prep(TcArgs a) {
    extern __shared__ __align__(1024) unsigned char sm[];
    unsigned char* tKQ = sm;            // 128 x 128 bf16; later the four X tiles
    unsigned char* tKt = sm + 32768;    // 128 x 64
    unsigned char* tVt = sm + 49152;    // 128 x 64
    float* Afp = reinterpret_cast<float*>(sm + 65536);  // [64][65]
    float* Tfp = Afp + 64 * 65;
    float* gam = Tfp + 64 * 65;
    float* bet = gam + 64;
    float* bg = bet + 64;
    float* spare = bg + 64;
    uint64_t* mbar = reinterpret_cast<uint64_t*>(spare + 64);
    uint32_t* tbase = reinterpret_cast<uint32_t*>(mbar + 1);

    const int total = a.chunk_off[a.n_seq];
    const int cidx = blockIdx.x, h = blockIdx.y, H = a.H;
    if (total < 0 || cidx >= total) return;
    const int b = find_seq(a.chunk_off, a.n_seq, cidx);
    const int n = cidx - a.chunk_off[b];
    const int seq0 = a.cu[b], T = a.cu[b + 1] - seq0;
    const int t0 = seq0 + n * C;
    const int nrows = min(C, T - n * C);
    const bool last = (n * C + nrows == T);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    unsigned char* blk = a.ws + ((size_t)cidx * H + h) * kBlock;

    if (warp == 0) tmem_alloc(tbase, 256);
    if (tid == 0) {
        mbar_init(mbar, 1);
        mbar_init_fence();
    }
    // [K; Q] rows (K-major: row = token, K dim = d)
    for (int i = tid; i < 128 * (D / 8); i += 128) {
        const int r = i / (D / 8), d8 = i % (D / 8);
        const int tr = r & 63;
        const __nv_bfloat16* src = (r < 64 ? a.k : a.q) + ((size_t)(t0 + tr) * H + h) * D + d8 * 8;
        *reinterpret_cast<uint4*>(tKQ + cm_off(r, d8 * 8, D)) = ld16_or_zero(src, tr < nrows);
    }
    // K^T and V^T (rows = d, K dim = token): 8 x 8 block transposes
    for (int i = tid; i < 2 * 8 * (D / 8); i += 128) {
        const int which = i / (8 * (D / 8));
        const int s8 = (i / (D / 8)) % 8, d8 = i % (D / 8);
        const __nv_bfloat16* base = which ? a.v : a.k;
        uint4 rows[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int s = s8 * 8 + j;
            rows[j] = ld16_or_zero(base + ((size_t)(t0 + s) * H + h) * D + d8 * 8, s < nrows);
        }
        transpose8_store(rows, (which ? tVt : tKt) + cm_off(d8 * 8, s8 * 8, C));
    }
    if (tid < C) {
        gam[tid] = (tid < nrows) ? a.g[(size_t)(t0 + tid) * H + h] : 0.f;
        bet[tid] = (tid < nrows) ? a.beta[(size_t)(t0 + tid) * H + h] : 0.f;
    }
    __syncthreads();
    if (tid == 0) {  // gate prefix: serial fp32 sum in token order
        float acc = 0.f;
        for (int r = 0; r < nrows; ++r) {
            acc = __fadd_rn(acc, gam[r]);
            gam[r] = acc;
        }
    }
    fence_async_smem();
    tc_sync();
    const uint32_t tmem = *tbase;
    if (tid == 0) {
        mma_tile<128, 64, D>(tmem, tKQ, tKQ, false);  // B = rows 0..63 of [K; Q] = K
        mma_commit(mbar);
    }
    if (tid < C) bg[tid] = (tid < nrows) ? simt::bg_entry(bet[tid], gam[tid]) : 0.f;
    // Q rows and K^T go to the workspace as the state pass's operand tiles
    for (int i = tid; i < 1024; i += 128) {
        reinterpret_cast<uint4*>(blk + kOffA4hi + 16384)[i] = reinterpret_cast<const uint4*>(tKQ + 16384)[i];
        reinterpret_cast<uint4*>(blk + kOffKt)[i] = reinterpret_cast<const uint4*>(tKt)[i];
    }
    int outstanding = 0;  // mbarrier phase an in-flight MMA group will complete, or -1
    const bool ok1 = mbar_wait(mbar, 0, a.err);
    fence_after();
    if (__syncthreads_or(!ok1)) goto done;
    outstanding = -1;
    {
        // S1 epilogue: thread = TMEM lane = row (0..63: K rows, 64..127: Q rows)
        float v[32];
        const int r = tid & 63;
        for (int c0 = 0; c0 < C; c0 += 32) {
            tmem_ld32(taddr_of(tmem, warp, c0), v);
            if (tid < 64) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int s = c0 + j;
                    Afp[r * 65 + s] = (s < r && r < nrows) ? simt::a_entry(bet[r], gam[r], gam[s], v[j]) : 0.f;
                }
            } else {
#pragma unroll
                for (int j8 = 0; j8 < 4; ++j8) {
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int s = c0 + j8 * 8 + e;
                        x[e] = (s <= r && r < nrows)
                                   ? __fmul_rn(simt::decay(gam[r], gam[s]), __fmul_rn(a.scale, v[j8 * 8 + e]))
                                   : 0.f;
                    }
                    store8_split(blk + kOffPhi, blk + kOffPlo, cm_off(r, c0 + j8 * 8, C), x);
                }
            }
        }
    }
    __syncthreads();
    // T = (I + A)^-1 by columns: T_rj = -(sum_{s=j}^{r-1} a_rs T_sj), ascending s
    if (tid < C) {
        const int j = tid;
        for (int r = 0; r < C; ++r) Tfp[r * 65 + j] = (r == j && r < nrows) ? 1.f : 0.f;
        for (int r = j + 1; r < nrows; ++r) {
            float acc = 0.f;
            for (int s = j; s < r; ++s) acc = __fmaf_rn(Afp[r * 65 + s], Tfp[s * 65 + j], acc);
            Tfp[r * 65 + j] = -acc;
        }
    }
    __syncthreads();
    {
        // X1 = T diag(b G) (threads 0..63), X2 = T diag(b) (threads 64..127), split
        const int r = tid & 63, which = tid >> 6;
        unsigned char* xhi = tKQ + which * 16384;
        unsigned char* xlo = xhi + 8192;
        const float* sc = which ? bet : bg;
        for (int s8 = 0; s8 < C / 8; ++s8) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = __fmul_rn(Tfp[r * 65 + s8 * 8 + e], sc[s8 * 8 + e]);
            store8_split(xhi, xlo, cm_off(r, s8 * 8, C), x);
        }
    }
    if (a.cache && last && nrows < C) {  // decode cache: rows of the last, partial chunk
        const size_t sh = (size_t)b * H + h;
        __nv_bfloat16* ck = reinterpret_cast<__nv_bfloat16*>(a.cache + a.co.k_rows) + sh * C * D;
        __nv_bfloat16* cv = reinterpret_cast<__nv_bfloat16*>(a.cache + a.co.v_rows) + sh * C * D;
        float* cg = reinterpret_cast<float*>(a.cache + a.co.gam_rows) + sh * C;
        float* cb = reinterpret_cast<float*>(a.cache + a.co.beta_rows) + sh * C;
        float* ct = reinterpret_cast<float*>(a.cache + a.co.t_rows) + sh * C * C;
        for (int i = tid; i < nrows * (D / 8); i += 128) {
            const int r = i / (D / 8), d8 = i % (D / 8);
            const size_t src = ((size_t)(t0 + r) * H + h) * D + d8 * 8;
            *reinterpret_cast<uint4*>(ck + r * D + d8 * 8) = *reinterpret_cast<const uint4*>(a.k + src);
            *reinterpret_cast<uint4*>(cv + r * D + d8 * 8) = *reinterpret_cast<const uint4*>(a.v + src);
        }
        if (tid < nrows) {
            cg[tid] = gam[tid];
            cb[tid] = bet[tid];
        }
        for (int i = tid; i < nrows * C; i += 128) ct[i] = Tfp[(i / C) * 65 + (i % C)];
    }
    fence_async_smem();
    tc_sync();
    if (tid == 0) {
        mma_tile<64, D, C>(tmem, tKQ, tKt, false);                // W' = X1_hi K
        mma_tile<64, D, C>(tmem, tKQ + 8192, tKt, true);          //    + X1_lo K
        mma_tile<64, D, C>(tmem + 128, tKQ + 16384, tVt, false);  // U  = X2_hi V
        mma_tile<64, D, C>(tmem + 128, tKQ + 24576, tVt, true);   //    + X2_lo V
        mma_commit(mbar);
    }
    outstanding = 1;
    {
        const bool ok2 = mbar_wait(mbar, 1, a.err);
        fence_after();
        if (__syncthreads_or(!ok2)) goto done;
    }
    outstanding = -1;
    {
        // W' and U rows: M = 64 layout, row r = 16 * warp + lane for lanes < 16
        const int r = warp * 16 + lane;
        float v[32];
        for (int c0 = 0; c0 < D; c0 += 32) {
            tmem_ld32(taddr_of(tmem, warp, c0), v);
            if (lane < 16) {
#pragma unroll
                for (int j8 = 0; j8 < 4; ++j8) {
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = v[j8 * 8 + e];
                    store8_split(blk + kOffA4hi, blk + kOffA4lo, cm_off(r, c0 + j8 * 8, D), x);
                }
            }
        }
        float* U = reinterpret_cast<float*>(blk + kOffU);
        const int dvs = a.dvs;
        for (int c0 = 0; c0 < D; c0 += 32) {
            tmem_ld32(taddr_of(tmem, warp, 128 + c0), v);
            if (lane < 16) {
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    const int j = c0 + j4 * 4;
                    const int sp = j / dvs, jl = j % dvs;
                    *reinterpret_cast<float4*>(U + ((size_t)sp * 64 + r) * dvs + jl) =
                        make_float4(v[j4 * 4], v[j4 * 4 + 1], v[j4 * 4 + 2], v[j4 * 4 + 3]);
                }
            }
        }
        if (tid < C) reinterpret_cast<float*>(blk + kOffGam)[tid] = gam[tid];
    }
done:
    if (outstanding >= 0) mbar_wait(mbar, (uint32_t)outstanding, a.err);  // bounded
    tc_sync();
    if (warp == 0) tmem_dealloc(*tbase, 256);
}

// ---- state pass: one CTA per (sequence, head, d_v split), chunks in order -----------
template <int DVS>
struct StateSmem {
    static constexpr size_t A4hi = 0, A4lo = 32768, Kt = 65536, Phi = 81920, Plo = 90112;
    static constexpr size_t U = 98304;                       // 64 x DVS fp32
    static constexpr size_t Hhi = U + 64 * DVS * 4;          // DVS x 128 bf16
    static constexpr size_t Hlo = Hhi + DVS * 128 * 2;
    static constexpr size_t Dhi = Hlo + DVS * 128 * 2;       // DVS x 64 bf16
    static constexpr size_t Dlo = Dhi + DVS * 64 * 2;
    static constexpr size_t Bhi = Dlo + DVS * 64 * 2;
    static constexpr size_t Blo = Bhi + DVS * 64 * 2;
    static constexpr size_t Q = Blo + DVS * 64 * 2;          // 64 x DVS fp32
    static constexpr size_t Gam = Q + 64 * DVS * 4;          // 64 fp32 (bulk copied)
    static constexpr size_t Gm = Gam + 256, Dec = Gm + 256;
    static constexpr size_t Bar = Dec + 256;                 // 2 mbarriers + TMEM base
    static constexpr size_t Total = Bar + 64;
    static constexpr uint32_t LoadBytes = 32768 + 16384 + 16384 + 8192 + 8192 + 64 * DVS * 4 + 256;
};

template <int DVS>
__global__ void __launch_bounds__(128) k_tc_state(TcArgs a) {
    using L = StateSmem<DVS>;
    constexpr int NSPLIT = D / DVS;
    extern __shared__ __align__(1024) unsigned char sm[];
    float* sU = reinterpret_cast<float*>(sm + L::U);
    float* sQ = reinterpret_cast<float*>(sm + L::Q);
    float* gam = reinterpret_cast<float*>(sm + L::Gam);
    float* Gm = reinterpret_cast<float*>(sm + L::Gm);
    float* dec = reinterpret_cast<float*>(sm + L::Dec);
    uint64_t* bar_mma = reinterpret_cast<uint64_t*>(sm + L::Bar);
    uint64_t* bar_ld = bar_mma + 1;
    uint32_t* tbase = reinterpret_cast<uint32_t*>(bar_mma + 2);

    const int total = a.chunk_off[a.n_seq];
    if (total < 0) return;
    const int H = a.H;
    const int sp = blockIdx.x % NSPLIT;
    const int h = (blockIdx.x / NSPLIT) % H;
    const int b = blockIdx.x / (NSPLIT * H);
    const int j0 = sp * DVS;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int seq0 = a.cu[b], T = a.cu[b + 1] - seq0;
    const int nch = a.chunk_off[b + 1] - a.chunk_off[b];
    const size_t sh = (size_t)b * H + h;
    float* cstate = a.cache ? reinterpret_cast<float*>(a.cache + a.co.state) + sh * D * D : nullptr;

    if (warp == 0) tmem_alloc(tbase, 256);
    if (tid == 0) {
        mbar_init(bar_mma, 1);
        mbar_init(bar_ld, 1);
        mbar_init_fence();
    }
    for (int i = tid; i < 1024; i += 128)  // rows 64..127 of the W'_lo operand stay zero
        reinterpret_cast<uint4*>(sm + L::A4lo + 16384)[i] = make_uint4(0u, 0u, 0u, 0u);
    // state columns j0..j0+DVS of row d = tid, fp32, kept in registers
    float Hreg[DVS];
    const int d = tid;
#pragma unroll
    for (int j = 0; j < DVS; ++j) Hreg[j] = a.h0 ? a.h0[(sh * D + d) * D + j0 + j] : 0.f;
#pragma unroll
    for (int j = 0; j < DVS; ++j) {
        __nv_bfloat16 hi, lo;
        split_bf16(Hreg[j], hi, lo);
        *reinterpret_cast<__nv_bfloat16*>(sm + L::Hhi + cm_off(j, d, D)) = hi;
        *reinterpret_cast<__nv_bfloat16*>(sm + L::Hlo + cm_off(j, d, D)) = lo;
    }
    if (nch == 0 && cstate) {
#pragma unroll
        for (int j = 0; j < DVS; ++j) cstate[d * D + j0 + j] = Hreg[j];
    }
    fence_async_smem();
    tc_sync();
    const uint32_t tmem = *tbase;
    const uint32_t acc4 = tmem, acc5 = tmem + DVS, acc6 = tmem + 2 * DVS;
    uint32_t ph_mma = 0, ph_ld = 0;
    bool pending = false, failed = false, mma_out = false;

    auto issue_loads = [&](int n) {
        const unsigned char* blk = a.ws + ((size_t)(a.chunk_off[b] + n) * H + h) * kBlock;
        mbar_expect_tx(bar_ld, L::LoadBytes);
        bulk_g2s(sm + L::A4hi, blk + kOffA4hi, 32768, bar_ld);
        bulk_g2s(sm + L::A4lo, blk + kOffA4lo, 16384, bar_ld);
        bulk_g2s(sm + L::Kt, blk + kOffKt, 16384, bar_ld);
        bulk_g2s(sm + L::Phi, blk + kOffPhi, 8192, bar_ld);
        bulk_g2s(sm + L::Plo, blk + kOffPlo, 8192, bar_ld);
        bulk_g2s(sm + L::U, blk + kOffU + (size_t)sp * 64 * DVS * 4, 64 * DVS * 4, bar_ld);
        bulk_g2s(sm + L::Gam, blk + kOffGam, 256, bar_ld);
    };
    if (nch > 0) {
        if (tid == 0) issue_loads(0);
        pending = true;
    }

    for (int n = 0; n < nch; ++n) {
        const int t0 = seq0 + n * C;
        const int nrows = min(C, T - n * C);
        const int Lr = nrows - 1;
        const bool last = (n == nch - 1);
        bool ok = mbar_wait(bar_ld, ph_ld, a.err);
        pending = !ok;
        if (__syncthreads_or(!ok)) { failed = true; break; }
        ph_ld ^= 1u;
        if (tid < C) {
            Gm[tid] = (tid < nrows) ? simt::gate(gam[tid]) : 0.f;
            dec[tid] = (tid < nrows) ? simt::decay(gam[Lr], gam[tid]) : 0.f;
        }
        const float GL = simt::gate(gam[Lr]);
        if (tid == 0) {
            mma_tile<128, DVS, D>(acc4, sm + L::A4hi, sm + L::Hhi, false);
            mma_tile<128, DVS, D>(acc4, sm + L::A4hi, sm + L::Hlo, true);
            mma_tile<128, DVS, D>(acc4, sm + L::A4lo, sm + L::Hhi, true);
            mma_commit(bar_mma);
        }
        mma_out = true;
        ok = mbar_wait(bar_mma, ph_mma, a.err);
        fence_after();
        if (__syncthreads_or(!ok)) { failed = true; break; }
        ph_mma ^= 1u;
        mma_out = false;
        {
            // rows 0..63: Delta = U - W'H ; rows 64..127: qh
            const int r = tid;
            float v[32];
#pragma unroll
            for (int c0 = 0; c0 < DVS; c0 += 32) {
                tmem_ld32(taddr_of(acc4, warp, c0), v);
                if (r < 64) {
                    const bool in = r < nrows;
                    float* cd = (a.cache && last && nrows < C && in)
                                    ? reinterpret_cast<float*>(a.cache + a.co.delta_rows) + (sh * C + r) * D + j0
                                    : nullptr;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int jj = c0 + j;
                        const float dl = in ? __fsub_rn(sU[r * DVS + jj], v[j]) : 0.f;
                        __nv_bfloat16 hi, lo;
                        split_bf16(dl, hi, lo);
                        *reinterpret_cast<__nv_bfloat16*>(sm + L::Dhi + cm_off(jj, r, C)) = hi;
                        *reinterpret_cast<__nv_bfloat16*>(sm + L::Dlo + cm_off(jj, r, C)) = lo;
                        split_bf16(__fmul_rn(dec[r], dl), hi, lo);
                        *reinterpret_cast<__nv_bfloat16*>(sm + L::Bhi + cm_off(jj, r, C)) = hi;
                        *reinterpret_cast<__nv_bfloat16*>(sm + L::Blo + cm_off(jj, r, C)) = lo;
                        if (cd) cd[jj] = dl;
                    }
                } else {
                    const int rr = r - 64;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        sQ[rr * DVS + c0 + j] = __fmul_rn(Gm[rr], __fmul_rn(a.scale, v[j]));
                }
            }
            if (cstate && last && nrows < C) {
#pragma unroll
                for (int j = 0; j < DVS; ++j) cstate[d * D + j0 + j] = Hreg[j];
            }
        }
        fence_async_smem();
        tc_sync();
        if (tid == 0) {
            mma_tile<64, DVS, C>(acc5, sm + L::Phi, sm + L::Dhi, false);
            mma_tile<64, DVS, C>(acc5, sm + L::Phi, sm + L::Dlo, true);
            mma_tile<64, DVS, C>(acc5, sm + L::Plo, sm + L::Dhi, true);
            mma_tile<128, DVS, C>(acc6, sm + L::Kt, sm + L::Bhi, false);
            mma_tile<128, DVS, C>(acc6, sm + L::Kt, sm + L::Blo, true);
            mma_commit(bar_mma);
        }
        mma_out = true;
        ok = mbar_wait(bar_mma, ph_mma, a.err);
        fence_after();
        if (__syncthreads_or(!ok)) { failed = true; break; }
        ph_mma ^= 1u;
        mma_out = false;
        if (tid == 0 && n + 1 < nch) {  // every operand tile of chunk n has been consumed
            fence_async_smem();
            issue_loads(n + 1);
        }
        pending = (n + 1 < nch);
        {
            float v[32];
            // o rows: M = 64 accumulator, row r = 16 * warp + lane for lanes < 16
            const int r = warp * 16 + lane;
#pragma unroll
            for (int c0 = 0; c0 < DVS; c0 += 32) {
                tmem_ld32(taddr_of(acc5, warp, c0), v);
                if (lane < 16 && r < nrows) {
                    float* orow = a.o + ((size_t)(t0 + r) * H + h) * D + j0 + c0;
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        float4 x;
                        x.x = __fadd_rn(sQ[r * DVS + c0 + 4 * j4 + 0], v[4 * j4 + 0]);
                        x.y = __fadd_rn(sQ[r * DVS + c0 + 4 * j4 + 1], v[4 * j4 + 1]);
                        x.z = __fadd_rn(sQ[r * DVS + c0 + 4 * j4 + 2], v[4 * j4 + 2]);
                        x.w = __fadd_rn(sQ[r * DVS + c0 + 4 * j4 + 3], v[4 * j4 + 3]);
                        if (a.o) *reinterpret_cast<float4*>(orow + 4 * j4) = x;
                    }
                }
            }
            // H' = G_L H + K^T (dec . Delta): row d = tid
#pragma unroll
            for (int c0 = 0; c0 < DVS; c0 += 32) {
                tmem_ld32(taddr_of(acc6, warp, c0), v);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float hn = __fadd_rn(__fmul_rn(GL, Hreg[c0 + j]), v[j]);
                    Hreg[c0 + j] = hn;
                    __nv_bfloat16 hi, lo;
                    split_bf16(hn, hi, lo);
                    *reinterpret_cast<__nv_bfloat16*>(sm + L::Hhi + cm_off(c0 + j, d, D)) = hi;
                    *reinterpret_cast<__nv_bfloat16*>(sm + L::Hlo + cm_off(c0 + j, d, D)) = lo;
                }
            }
            if (cstate && last && nrows == C) {
#pragma unroll
                for (int j = 0; j < DVS; ++j) cstate[d * D + j0 + j] = Hreg[j];
            }
        }
        fence_async_smem();
        tc_sync();
    }
    if (!failed && a.final_state) {
#pragma unroll
        for (int j = 0; j < DVS; ++j) a.final_state[(sh * D + d) * D + j0 + j] = Hreg[j];
    }
    if (failed) {
        // let in-flight copies and MMAs finish (bounded) before TMEM is released
        if (pending) mbar_wait(bar_ld, ph_ld, a.err);
        if (mma_out) mbar_wait(bar_mma, ph_mma, a.err);
    }
    tc_sync();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

}  // namespace tc
}  // namespace cpr
