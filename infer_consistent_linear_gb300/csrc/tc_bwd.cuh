// CPR Gated DeltaNet backward on the tensor cores (operand policy TC_BF16X3).
//
// The backward of the forward chunk form (derived here; the pages give the
// trainer forward+backward stage only as a timing, page "IsoExec: 切换 SkyRL
// 中的训练器-推理不匹配", section "Chunkwise-Parallel Recurrent (CPR) Gated
// DeltaNet", stage table).  Per chunk, with start state H, dH' = dL/dH_{n+1},
// E_rs = exp(gam_r - gam_s), dec_s = E_Ls, bg_s = b_s G_s, R = diag(b)(V - diag(G) K H)
// (so that Delta = T R):
//   dDelta = P^T dO + diag(dec) (K dH')
//   dR     = T^T dDelta
//   dH     = G_L dH' + Q^T diag(G scale) dO - K^T diag(bg) dR        (previous chunk's dH')
//   dP_rs  =  dO_r . Delta_s  (s <= r),   dA_rs = -dR_r . Delta_s  (s < r)
//   dq     = scale (diag(G) dO H^T + (E . dP) K)
//   dk     = -diag(bg) dR H^T + diag(dec) Delta dH'^T + (E . dP)^T Q^ + (G2 + G2^T) K,
//            G2_rs = b_r E_rs dA_rs
//   dv     = diag(b) dR
//   db_r   = dR_r . v_r - G_r k_r . (dR H^T)_r + sum_{s<r} dA_rs E_rs kk_rs
//   dgam_r = G_r (q^_r . (dO H^T)_r - b_r k_r . (dR H^T)_r) + rowE_r - colE_r - e_r
//            (+ G_L <dH', H> + sum_{s<L} e_s at r = L),
//            e_s = dec_s k_s . (Delta dH'^T)_s,  t_rs = dP_rs P_rs + b_r dA_rs E_rs kk_rs,
//            rowE_r = sum_{s<r} t_rs,  colE_s = sum_{r>s} t_rs
//   dg_s   = sum_{r=s}^{L} dgam_r
// Kernels: k_tc_state_bwd (one CTA per (sequence, head, d_v split), chunks in
// reverse order: the dH chain; stores dH' and dR per chunk) and k_tc_grad (one
// CTA per chunk and head, all d_v columns: every per-token gradient).  The
// training forward (k_tc_prep, k_tc_state with `train`) leaves T, H_n and Delta
// in each chunk's workspace block; every fp32 x fp32 product is three bf16 MMA
// passes (hi hi, hi lo, lo hi), fp32 x exact-bf16 two.  No bitwise coupling to
// another path: deterministic (fixed orders, no atomics) and batch-invariant
// (one CTA per chunk or per sequence).
#pragma once

#include "tc_fwd.cuh"

namespace cpr {
namespace tc {

struct TcBwdArgs {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const float* g;
    const float* beta;
    const int32_t* cu;
    const int32_t* chunk_off;
    int n_seq;
    int H;
    float scale;
    unsigned char* ws;    // kBlockTrain blocks from the training forward
    const float* dO;
    const float* dHT;
    float* dq;
    float* dk;
    float* dv;
    float* dg;
    float* dbeta;
    float* dh0;
    int nsplit;           // d_v splits of the reverse state pass (2 or 4)
    uint32_t* err;
};

// Sum over the 32 lanes of a warp in a fixed tree (lane 0 gets the result).
__device__ __forceinline__ float warp_sum_tree(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = __fadd_rn(x, __shfl_down_sync(0xffffffffu, x, o));
    return x;
}

// ---- reverse state pass ---------------------------------------------------------------
template <int DVS>
struct SbSmem {
    static constexpr size_t Phi = 0, Plo = 8192;             // P, K-major (r, s); read as P^T
    static constexpr size_t Thi = 16384, Tlo = 24576;        // T, K-major (r, j); read as T^T
    static constexpr size_t KQ0 = 32768, KQ1 = 65536;        // [K | Q] K-major, two buffers
    static constexpr size_t dHhi = 98304;                    // dH', MN-major (j, d)
    static constexpr size_t dHlo = dHhi + DVS * 128 * 2;
    static constexpr size_t B1hi = dHlo + DVS * 128 * 2;     // dO, then dDelta: MN-major (j, t)
    static constexpr size_t B1lo = B1hi + DVS * 64 * 2;
    static constexpr size_t B2hi = B1lo + DVS * 64 * 2;      // G scale dO, then -bg dR
    static constexpr size_t B2lo = B2hi + DVS * 64 * 2;
    static constexpr size_t Vec = B2lo + DVS * 64 * 2;      // gam (hi, lo), Gm, dec, bg (64 fp32
                                                             // each), 8 warp sums
    static constexpr size_t Bar = Vec + 6 * 256;             // 5 mbarriers + TMEM base
    static constexpr size_t Total = Bar + 64;
};

// 256 threads: warp w reads TMEM lane quarter w % 4, the two warps of a
// quarter one half of the DVS columns each.
template <int DVS>
__global__ void __launch_bounds__(256, 1) k_tc_state_bwd(TcBwdArgs a) {
    using L = SbSmem<DVS>;
    constexpr int NSPLIT = D / DVS;
    constexpr int HALF = DVS / 2;
    extern __shared__ __align__(1024) unsigned char sm[];
    float* gam = reinterpret_cast<float*>(sm + L::Vec);   // gate prefix hi, then lo
    float* gml = gam + 64;
    float* Gm = gml + 64;
    float* dec = Gm + 64;
    float* bgv = dec + 64;
    float* red = bgv + 64;
    uint64_t* bar_mma = reinterpret_cast<uint64_t*>(sm + L::Bar);
    uint64_t* bar_P = bar_mma + 1;
    uint64_t* bar_T = bar_mma + 2;
    uint64_t* bar_KQ = bar_mma + 3;  // two
    uint32_t* tbase = reinterpret_cast<uint32_t*>(bar_mma + 5);

    const int total = a.chunk_off[a.n_seq];
    if (total < 0) return;
    const int H = a.H;
    const int sp = blockIdx.x % NSPLIT;
    const int h = (blockIdx.x / NSPLIT) % H;
    const int b = blockIdx.x / (NSPLIT * H);
    const int j0 = sp * DVS;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, cb = (warp >> 2) * HALF;
    const int seq0 = a.cu[b], T = a.cu[b + 1] - seq0;
    const int coff = a.chunk_off[b];
    const int nch = a.chunk_off[b + 1] - coff;
    const size_t sh = (size_t)b * H + h;
    auto blk_of = [&](int n) { return a.ws + ((size_t)(coff + n) * H + h) * kBlockTrain; };

    if (warp == 0) tmem_alloc(tbase, 256);
    if (tid == 0) {
        for (int i = 0; i < 5; ++i) mbar_init(bar_mma + i, 1);
        mbar_init_fence();
    }
    // dL/dH of the last chunk's end state, row d, columns j0 + cb .. + HALF
    float dHreg[HALF];
    const int d = quarter * 32 + lane;
#pragma unroll
    for (int j4 = 0; j4 < HALF / 4; ++j4) {
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (a.dHT) x = *reinterpret_cast<const float4*>(a.dHT + (sh * D + d) * D + j0 + cb + 4 * j4);
        dHreg[4 * j4] = x.x; dHreg[4 * j4 + 1] = x.y; dHreg[4 * j4 + 2] = x.z; dHreg[4 * j4 + 3] = x.w;
    }
    // dH' as the B operand of K dH'; also chunk nn's dH' tiles for k_tc_grad
    auto put_dh = [&](int nn) {
        unsigned char* g = (nn >= 0) ? blk_of(nn) + kOffdH : nullptr;
#pragma unroll
        for (int j8 = 0; j8 < HALF / 8; ++j8) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = dHreg[j8 * 8 + e];
            uint4 hi, lo;
            split8(x, hi, lo);
            const int jj = cb + j8 * 8;
            *reinterpret_cast<uint4*>(sm + L::dHhi + mn_off(jj, d, DVS)) = hi;
            *reinterpret_cast<uint4*>(sm + L::dHlo + mn_off(jj, d, DVS)) = lo;
            if (g) {
                *reinterpret_cast<uint4*>(g + cm_off(d, j0 + jj, D)) = hi;
                *reinterpret_cast<uint4*>(g + 32768 + cm_off(d, j0 + jj, D)) = lo;
            }
        }
    };
    auto issue_P = [&](int n) {
        const unsigned char* blk = blk_of(n);
        mbar_expect_tx(bar_P, 16384 + 512);
        bulk_g2s(sm + L::Phi, blk + kOffPhi, 16384, bar_P);
        bulk_g2s(gam, blk + kOffGam, 512, bar_P);
    };
    auto issue_T = [&](int n) {
        mbar_expect_tx(bar_T, 16384);
        bulk_g2s(sm + L::Thi, blk_of(n) + kOffT, 16384, bar_T);
    };
    auto issue_KQ = [&](int n) {
        const unsigned char* blk = blk_of(n);
        unsigned char* dst = sm + ((n & 1) ? L::KQ1 : L::KQ0);
        uint64_t* bar = bar_KQ + (n & 1);
        mbar_expect_tx(bar, 32768);
        bulk_g2s(dst, blk + kOffKmn, 16384, bar);
        bulk_g2s(dst + 16384, blk + kOffA4hi + 16384, 16384, bar);
    };
    // this thread's slice of chunk n's dO rows (token rr, 8-column groups j8 of its part),
    // loaded into registers one chunk ahead; rows past the end are zero
    constexpr int NJ8 = DVS / 32;                     // 8-column groups per thread
    const int rr = tid & 63, part = tid >> 6;
    // (the loads read a valid row unconditionally; rows past the end are masked where
    // the values are used, so that nothing waits on the loads where they are issued)
    float4 dOpre[2 * NJ8];
    auto load_dO = [&](int n) {
        const int t0 = seq0 + n * C;
        const bool in = rr < min(C, T - n * C);
        const float4* src = reinterpret_cast<const float4*>(a.dO + ((size_t)(t0 + (in ? rr : 0)) * H + h) * D + j0);
#pragma unroll
        for (int q = 0; q < NJ8; ++q) {
            const int j8 = part * NJ8 + q;
            dOpre[2 * q] = src[2 * j8];
            dOpre[2 * q + 1] = src[2 * j8 + 1];
        }
    };
    auto beta_of = [&](int n) {
        const int t0 = seq0 + n * C, nrows = min(C, T - n * C);
        return a.beta[(size_t)(t0 + (tid < nrows ? tid : 0)) * H + h];
    };

    // this thread's part of H_n (row d, its columns) for <dH', H_n>, loaded a chunk ahead
    uint4 hn[HALF / 4];
    auto load_hn = [&](int n) {
        const unsigned char* g = blk_of(n) + kOffHn;
#pragma unroll
        for (int j8 = 0; j8 < HALF / 8; ++j8) {
            const uint32_t off = cm_off(d, j0 + cb + j8 * 8, D);
            hn[2 * j8] = *reinterpret_cast<const uint4*>(g + off);
            hn[2 * j8 + 1] = *reinterpret_cast<const uint4*>(g + 32768 + off);
        }
    };
    if (nch > 0) load_hn(nch - 1);
    put_dh(nch - 1);
    float bcur = 0.f;
    if (nch > 0) {
        if (tid == 0) {
            issue_P(nch - 1);
            issue_T(nch - 1);
            issue_KQ(nch - 1);
            if (nch > 1) issue_KQ(nch - 2);
        }
        load_dO(nch - 1);
        bcur = beta_of(nch - 1);
    }
    fence_async_smem();
    tc_sync();
    const uint32_t tmem = *tbase;
    const uint32_t tD1 = tmem, tD2 = tmem + DVS, tR = tmem + 2 * DVS, tH = tmem + 3 * DVS;
    uint32_t ph_mma = 0, ph_P = 0, ph_T = 0, ph_KQ[2] = {0u, 0u};
    bool pendP = nch > 0, pendT = nch > 0, pendKQ[2] = {nch > 0, nch > 1}, mma_out = false;
    if (nch > 0 && ((nch - 1) & 1)) { pendKQ[0] = nch > 1; pendKQ[1] = true; }
    bool failed = false;
    const float scale = a.scale;
    // M = 64 accumulator rows: lanes 0..15 of each lane quarter
    const int r64 = quarter * 16 + lane;

    for (int it = 0; it < nch; ++it) {
        const int n = nch - 1 - it;
        const int nrows = min(C, T - n * C);
        const int Lr = nrows - 1;
        const int cur = n & 1;
        unsigned char* KQ = sm + (cur ? L::KQ1 : L::KQ0);
        bool ok = mbar_wait(bar_P, ph_P, a.err);
        if (__syncthreads_or(!ok)) { failed = true; break; }
        ph_P ^= 1u;
        pendP = false;
        {
            // token row rr, a quarter of the columns per thread: dO (B1) and G scale dO
            // (B2) rows, MN-major (j, t); dO also to the workspace (K-major (r, j)) and
            // beta (split 0) for k_tc_grad
            unsigned char* gdo = blk_of(n) + kOffdO;
            bcur = (tid < nrows) ? bcur : 0.f;
            if (sp == 0 && tid < C) reinterpret_cast<float*>(blk_of(n) + kOffBet)[tid] = bcur;
            const bool in = rr < nrows;
            const float gr = gam[rr], lr = gml[rr];
            const float Gr = in ? simt::gate(gr, lr) : 0.f;
            if (part == 0) {
                Gm[rr] = Gr;
                dec[rr] = in ? simt::decay(gam[Lr], gml[Lr], gr, lr) : 0.f;
                bgv[rr] = in ? simt::bg_entry(bcur, gr, lr) : 0.f;
            }
            const float gs = __fmul_rn(Gr, scale);
#pragma unroll
            for (int q = 0; q < NJ8; ++q) {
                const int j8 = part * NJ8 + q;
                const float4 u0 = dOpre[2 * q], u1 = dOpre[2 * q + 1];
                float x[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = in ? x[e] : 0.f;
                float y[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) y[e] = __fmul_rn(gs, x[e]);
                uint4 hi, lo;
                split8(x, hi, lo);
                *reinterpret_cast<uint4*>(sm + L::B1hi + mn_off(j8 * 8, rr, DVS)) = hi;
                *reinterpret_cast<uint4*>(sm + L::B1lo + mn_off(j8 * 8, rr, DVS)) = lo;
                *reinterpret_cast<uint4*>(gdo + cm_off(rr, j0 + j8 * 8, D)) = hi;
                *reinterpret_cast<uint4*>(gdo + 16384 + cm_off(rr, j0 + j8 * 8, D)) = lo;
                store8_split(sm + L::B2hi, sm + L::B2lo, mn_off(j8 * 8, rr, DVS), y);
            }
        }
        const float GL = simt::gate(gam[Lr], gml[Lr]);
        fence_async_smem();
        ok = mbar_wait(bar_KQ + cur, ph_KQ[cur], a.err);
        fence_after();
        if (__syncthreads_or(!ok)) { failed = true; break; }
        ph_KQ[cur] ^= 1u;
        pendKQ[cur] = false;
        if (tid == 0) {
            mma_tile_mj<64, DVS, C, true, true>(tD1, sm + L::Phi, sm + L::B1hi, false);   // P^T dO
            mma_tile_mj<64, DVS, C, true, true>(tD1, sm + L::Phi, sm + L::B1lo, true);
            mma_tile_mj<64, DVS, C, true, true>(tD1, sm + L::Plo, sm + L::B1hi, true);
            mma_tile_mj<64, DVS, D, false, true>(tD2, KQ, sm + L::dHhi, false);            // K dH'
            mma_tile_mj<64, DVS, D, false, true>(tD2, KQ, sm + L::dHlo, true);
            mma_tile_mj<128, DVS, C, true, true>(tH, KQ + 16384, sm + L::B2hi, false);     // Q^T G scale dO
            mma_tile_mj<128, DVS, C, true, true>(tH, KQ + 16384, sm + L::B2lo, true);
            mma_commit(bar_mma);
        }
        mma_out = true;
        {
            // <dH', H_n> over this thread's columns (dH' = dHreg, still chunk n's) while the
            // MMAs run, then a fixed tree over the warp.  The next chunk's dO slice, beta
            // and H_n are loaded here, just after a proxy fence: a fence.proxy.async waits
            // for this thread's global loads in flight, and the next one is a phase away.
            float acc = 0.f;
#pragma unroll
            for (int j8 = 0; j8 < HALF / 8; ++j8) {
                float hv[8];
                join8(hn[2 * j8], hn[2 * j8 + 1], hv);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc = __fmaf_rn(dHreg[j8 * 8 + e], hv[e], acc);
            }
            acc = warp_sum_tree(acc);
            if (lane == 0) red[warp] = acc;
            if (n > 0) {
                load_dO(n - 1);
                bcur = beta_of(n - 1);
                load_hn(n - 1);
            }
        }
        ok = mbar_wait(bar_mma, ph_mma, a.err);
        fence_after();
        if (__syncthreads_or(!ok)) { failed = true; break; }
        ph_mma ^= 1u;
        mma_out = false;
        if (tid == 0 && n > 0) {  // P and gam of chunk n are consumed
            fence_async_smem();
            issue_P(n - 1);
        }
        pendP = n > 0;
        {
            // dDelta = P^T dO + dec . (K dH') -> B1 (MN-major (j, t)), this thread's columns
            float v1[32], v2[32];
            tmem_ld32x2(taddr_of(tD1, warp, cb), v1, taddr_of(tD2, warp, cb), v2);
            if (lane < 16) {
                const float dr = dec[r64];
#pragma unroll
                for (int j8 = 0; j8 < HALF / 8; ++j8) {
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = __fmaf_rn(dr, v2[j8 * 8 + e], v1[j8 * 8 + e]);
                    store8_split(sm + L::B1hi, sm + L::B1lo, mn_off(cb + j8 * 8, r64, DVS), x);
                }
            }
        }
        fence_async_smem();
        tc_sync();
        if (tid == 0) {  // this split's share of <dH', H_n>, warps in order
            float s = 0.f;
            for (int w = 0; w < 8; ++w) s = __fadd_rn(s, red[w]);
            reinterpret_cast<float*>(blk_of(n) + kOffHdot)[sp] = s;
        }
        ok = mbar_wait(bar_T, ph_T, a.err);
        if (__syncthreads_or(!ok)) { failed = true; break; }
        ph_T ^= 1u;
        pendT = false;
        if (tid == 0) {
            mma_tile_mj<64, DVS, C, true, true>(tR, sm + L::Thi, sm + L::B1hi, false);    // T^T dDelta
            mma_tile_mj<64, DVS, C, true, true>(tR, sm + L::Thi, sm + L::B1lo, true);
            mma_tile_mj<64, DVS, C, true, true>(tR, sm + L::Tlo, sm + L::B1hi, true);
            mma_commit(bar_mma);
        }
        mma_out = true;
        ok = mbar_wait(bar_mma, ph_mma, a.err);
        fence_after();
        if (__syncthreads_or(!ok)) { failed = true; break; }
        ph_mma ^= 1u;
        mma_out = false;
        if (tid == 0 && n > 0) {
            fence_async_smem();
            issue_T(n - 1);
        }
        pendT = n > 0;
        {
            // dR rows: to the workspace (K-major (r, j) hi/lo) and -bg . dR -> B2
            unsigned char* gdr = blk_of(n) + kOffdR;
            float v1[32];
            tmem_ld32(taddr_of(tR, warp, cb), v1);
            if (lane < 16) {
                const float nb = -bgv[r64];
#pragma unroll
                for (int j8 = 0; j8 < HALF / 8; ++j8) {
                    float x[8], y[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        x[e] = v1[j8 * 8 + e];
                        y[e] = __fmul_rn(nb, x[e]);
                    }
                    uint4 hi, lo;
                    split8(x, hi, lo);
                    const int jj = cb + j8 * 8;
                    *reinterpret_cast<uint4*>(gdr + cm_off(r64, j0 + jj, D)) = hi;
                    *reinterpret_cast<uint4*>(gdr + 16384 + cm_off(r64, j0 + jj, D)) = lo;
                    store8_split(sm + L::B2hi, sm + L::B2lo, mn_off(jj, r64, DVS), y);
                }
            }
        }
        fence_async_smem();
        tc_sync();
        if (tid == 0) {
            mma_tile_mj<128, DVS, C, true, true>(tH, KQ, sm + L::B2hi, true);   // += K^T (-bg dR)
            mma_tile_mj<128, DVS, C, true, true>(tH, KQ, sm + L::B2lo, true);
            mma_commit(bar_mma);
        }
        mma_out = true;
        ok = mbar_wait(bar_mma, ph_mma, a.err);
        fence_after();
        if (__syncthreads_or(!ok)) { failed = true; break; }
        ph_mma ^= 1u;
        mma_out = false;
        if (tid == 0 && n >= 2) {  // K and Q of chunk n are consumed: chunk n - 2 takes the buffer
            fence_async_smem();
            issue_KQ(n - 2);
        }
        if (n >= 2) pendKQ[cur] = true;
        {
            // dH = G_L dH' + acc, row d, this thread's columns
            float v1[32];
            tmem_ld32(taddr_of(tH, warp, cb), v1);
#pragma unroll
            for (int j = 0; j < HALF; ++j) dHreg[j] = __fmaf_rn(GL, dHreg[j], v1[j]);
            put_dh(n - 1);
        }
        fence_async_smem();
        tc_sync();
    }
    if (!failed) {
#pragma unroll
        for (int j4 = 0; j4 < HALF / 4; ++j4)
            *reinterpret_cast<float4*>(a.dh0 + (sh * D + d) * D + j0 + cb + 4 * j4) =
                make_float4(dHreg[4 * j4], dHreg[4 * j4 + 1], dHreg[4 * j4 + 2], dHreg[4 * j4 + 3]);
    } else {
        // let in-flight copies and MMAs finish (bounded) before TMEM is released
        if (pendP) mbar_wait(bar_P, ph_P, a.err);
        if (pendT) mbar_wait(bar_T, ph_T, a.err);
        if (pendKQ[0]) mbar_wait(bar_KQ, ph_KQ[0], a.err);
        if (pendKQ[1]) mbar_wait(bar_KQ + 1, ph_KQ[1], a.err);
        if (mma_out) mbar_wait(bar_mma, ph_mma, a.err);
    }
    tc_sync();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// ---- per-chunk gradients -------------------------------------------------------------------
// 256 threads.  Accumulator row L (TMEM lane L) is read by warps L / 32 and
// L / 32 + 4, each taking half of the columns.  Rows 0..63 ("top") carry the
// dO / Q-side quantities of token r = L, rows 64..127 ("bottom") the dR /
// K-side ones of token r = L - 64.
struct GradSmem {
    static constexpr size_t QK = 0;            // [Q | K] K-major: Q rows 0..63, K rows 64..127
    static constexpr size_t Rhi = 32768;       // [dO | dR | Delta] K-major 192 x 128, hi
    static constexpr size_t Rlo = 81920;       // lo
    static constexpr size_t Bt = 131072;       // H_n, then dH': K-major (d, j), hi then lo
    static constexpr size_t Scr = 196608;      // 64 x 65 fp32: t_rs
    static constexpr size_t Vec = Scr + 64 * 65 * 4;
    static constexpr int kVec = 22;            // 64-float vectors
    static constexpr size_t Bar = Vec + kVec * 256;   // 2 mbarriers + TMEM base
    static constexpr size_t Total = Bar + 64;
};

static __global__ void __launch_bounds__(256, 1) k_tc_grad(TcBwdArgs a) {
    using L = GradSmem;
    extern __shared__ __align__(1024) unsigned char sm[];
    unsigned char* QK = sm + L::QK;
    unsigned char* Rhi = sm + L::Rhi;
    unsigned char* Rlo = sm + L::Rlo;
    unsigned char* Bt = sm + L::Bt;
    float* scr = reinterpret_cast<float*>(sm + L::Scr);
    float* vec = reinterpret_cast<float*>(sm + L::Vec);
    // [2][64] vectors hold the two column halves' partial sums of a row
    float *gam = vec, *Gm = vec + 64, *bet = vec + 128, *bgv = vec + 192, *dec = vec + 256,
          *qh = vec + 320, *kh = vec + 448, *rowA = vec + 576, *rowB = vec + 704, *dbA = vec + 832,
          *dRv = vec + 960, *colE = vec + 1024, *eL = vec + 1088, *dgam = vec + 1216,
          *red = vec + 1280,   // red: the d_v splits' shares of <dH', H_n>
          *gml = vec + 1288;   // gate prefix, lo; 1352 floats in all
    uint64_t* bar_in = reinterpret_cast<uint64_t*>(sm + L::Bar);   // Q, K, dR, Delta, gam
    uint64_t* bar_hn = bar_in + 1;                                   // H_n
    uint64_t* bar_dh = bar_in + 2;                                   // dH'
    uint64_t* bar_mma = bar_in + 3;
    uint32_t* tbase = reinterpret_cast<uint32_t*>(bar_in + 4);

    const int total = a.chunk_off[a.n_seq];
    if (total < 0) return;
    const int H = a.H;
    const int nwork = total * H;           // (chunk, head) items, chunk-major
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, hf = warp >> 2;
    const int row = quarter * 32 + lane;       // accumulator row / TMEM lane
    const bool top = row < 64;
    const int r = row & 63;                    // token row of the chunk
    const float scale = a.scale;
    auto blk_of = [&](int w) { return a.ws + (size_t)w * kBlockTrain; };   // w = cidx * H + h
    auto issue_in = [&](int w) {
        const unsigned char* blk = blk_of(w);
        mbar_expect_tx(bar_in, 8 * 16384 + 3 * 256 + 16);
        bulk_g2s(Rhi, blk + kOffdO, 16384, bar_in);              // dO rows, split
        bulk_g2s(Rlo, blk + kOffdO + 16384, 16384, bar_in);
        bulk_g2s(QK, blk + kOffA4hi + 16384, 16384, bar_in);     // Q rows
        bulk_g2s(QK + 16384, blk + kOffKmn, 16384, bar_in);      // K rows
        bulk_g2s(Rhi + 16384, blk + kOffdR, 16384, bar_in);
        bulk_g2s(Rlo + 16384, blk + kOffdR + 16384, 16384, bar_in);
        bulk_g2s(Rhi + 32768, blk + kOffDl, 16384, bar_in);
        bulk_g2s(Rlo + 32768, blk + kOffDl + 16384, 16384, bar_in);
        bulk_g2s(gam, blk + kOffGam, 256, bar_in);               // gate prefix hi, lo
        bulk_g2s(gml, blk + kOffGam + 256, 256, bar_in);
        bulk_g2s(red, blk + kOffHdot, 16, bar_in);               // the splits' <dH', H_n>
        bulk_g2s(bet, blk + kOffBet, 256, bar_in);
    };
    auto issue_hn = [&](int w) {
        mbar_expect_tx(bar_hn, 65536);
        bulk_g2s(Bt, blk_of(w) + kOffHn, 65536, bar_hn);
    };

    if (warp == 0) tmem_alloc(tbase, 512);
    if (tid == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(bar_in + i, 1);
        mbar_init_fence();
        if ((int)blockIdx.x < nwork) {
            issue_in(blockIdx.x);
            issue_hn(blockIdx.x);
        }
    }
    tc_sync();
    const uint32_t tmem = *tbase;
    const uint32_t tX1 = 0, tG = 128, tS1 = 192, tX2 = 256, tdq = 384, tdk = 128;
    uint32_t ph_mma = 0;
    bool pend_in = (int)blockIdx.x < nwork, pend_hn = pend_in, pend_dh = false, mma_out = false;
    uint32_t ph_in = 0, ph_hn = 0;  // parity the pending input / H_n copy completes
    bool failed = false;
    int it = 0;                    // this CTA's item count: the load barriers' phase parity
    float bloc[32];                // bottom rows: b_r dA_rs Kd_rs for this thread's columns

    // an item's sequence, its chunk within it, the sequence's first token and length: a
    // chain of dependent loads, taken for the next item while this one's first MMA group runs
    int nx_b = -1, nx_n = 0, nx_seq0 = 0, nx_T = 0;
    auto locate = [&](int w) {
        const int cidx = w / H;
        nx_b = find_seq(a.chunk_off, a.n_seq, cidx);
        nx_n = cidx - a.chunk_off[nx_b];
        nx_seq0 = a.cu[nx_b];
        nx_T = a.cu[nx_b + 1] - nx_seq0;
    };
    for (int w = blockIdx.x; w < nwork; w += gridDim.x, ++it) {
    const uint32_t ph = (uint32_t)(it & 1);
    const int wn = w + (int)gridDim.x;         // the next item of this CTA
    const int h = w % H;
    if (nx_b < 0) locate(w);                   // the CTA's first item
    const int n = nx_n, seq0 = nx_seq0, T = nx_T;
    nx_b = -1;
    const int t0 = seq0 + n * C;
    const int nrows = min(C, T - n * C);
    const int Lr = nrows - 1;
    const unsigned char* blk = blk_of(w);
    tc_sync();   // the previous item's TMEM reads and shared-memory use are over
    {
        const bool ok = mbar_wait(bar_in, ph, a.err) && mbar_wait(bar_hn, ph, a.err);
        fence_async_smem();
        tc_sync();
        if (__syncthreads_or(!ok)) { failed = true; break; }
    }
    pend_in = pend_hn = false;
    if (tid < C) {
        const bool in = tid < nrows;
        const float gr = gam[tid], lr = gml[tid];
        Gm[tid] = in ? simt::gate(gr, lr) : 0.f;
        dec[tid] = in ? simt::decay(gam[Lr], gml[Lr], gr, lr) : 0.f;
        bgv[tid] = in ? simt::bg_entry(bet[tid], gr, lr) : 0.f;
    }
    if (tid == 0) {
        mma_tile<128, 64, D>(tmem + tS1, QK, QK + 16384, false);            // [Q; K] K^T
        mma_tile<128, 128, D>(tmem + tX1, Rhi, Bt, false);                  // [dO; dR] H^T
        mma_tile<128, 128, D>(tmem + tX1, Rhi, Bt + 32768, true);
        mma_tile<128, 128, D>(tmem + tX1, Rlo, Bt, true);
        mma_tile<128, 64, D>(tmem + tG, Rhi, Rhi + 32768, false);           // [dO; dR] Delta^T
        mma_tile<128, 64, D>(tmem + tG, Rhi, Rlo + 32768, true);
        mma_tile<128, 64, D>(tmem + tG, Rlo, Rhi + 32768, true);
        mma_commit(bar_mma);
    }
    mma_out = true;
    {
        // dv = b dR and dR . v while the first MMA group runs (dR, beta and the v rows are
        // all in): a warp per row, 16-byte pieces side by side, the v rows loaded first
        const int w4 = warp, c4 = lane * 4;
        uint2 vrow[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int rr = w4 + 8 * k;
            vrow[k] = (rr < nrows) ? *reinterpret_cast<const uint2*>(a.v + ((size_t)(t0 + rr) * H + h) * D + c4)
                                   : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int rr = w4 + 8 * k;
            if (rr >= nrows) break;
            const uint32_t off = cm_off(rr, c4, D);
            const uint2 hi = *reinterpret_cast<const uint2*>(Rhi + 16384 + off);
            const uint2 lo = *reinterpret_cast<const uint2*>(Rlo + 16384 + off);
            const __nv_bfloat16* hh = reinterpret_cast<const __nv_bfloat16*>(&hi);
            const __nv_bfloat16* ll = reinterpret_cast<const __nv_bfloat16*>(&lo);
            const size_t g = ((size_t)(t0 + rr) * H + h) * D + c4;
            const __nv_bfloat16* vb = reinterpret_cast<const __nv_bfloat16*>(&vrow[k]);
            const float brr = bet[rr];
            float x[4], sdot = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                x[e] = __fadd_rn(__bfloat162float(hh[e]), __bfloat162float(ll[e]));
                sdot = __fmaf_rn(x[e], __bfloat162float(vb[e]), sdot);
            }
            *reinterpret_cast<float4*>(a.dv + g) =
                make_float4(__fmul_rn(brr, x[0]), __fmul_rn(brr, x[1]), __fmul_rn(brr, x[2]), __fmul_rn(brr, x[3]));
            sdot = warp_sum_tree(sdot);
            if (lane == 0) dRv[rr] = sdot;
        }
    }
    if (wn < nwork) locate(wn);
    {
        const bool ok = mbar_wait(bar_mma, ph_mma, a.err);
        fence_after();
        if (__syncthreads_or(!ok)) { failed = true; break; }
    }
    ph_mma ^= 1u;
    mma_out = false;
    if (tid == 0) {  // H_n is consumed: dH' takes its place
        fence_async_smem();
        mbar_expect_tx(bar_dh, 65536);
        bulk_g2s(Bt, blk + kOffdH, 65536, bar_dh);
    }
    pend_dh = true;
    {
        // ---- phase A: one pass over this thread's 32 columns s of the row
        const int s0 = hf * 32;
        const float gr = gam[r], lr = gml[r], br = bet[r];
        float v1[32], v2[32];
        tmem_ld32x2(taddr_of(tmem + tS1, warp, s0), v1, taddr_of(tmem + tG, warp, s0), v2);
        float sa = 0.f, sb = 0.f;
#pragma unroll
        for (int j8 = 0; j8 < 4; ++j8) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int s = s0 + j8 * 8 + e, j = j8 * 8 + e;
                if (top) {
                    const bool in = s <= r && r < nrows;
                    const float E = in ? simt::decay(gr, lr, gam[s], gml[s]) : 0.f;
                    const float P = __fmul_rn(E, __fmul_rn(scale, v1[j]));
                    const float dP = in ? v2[j] : 0.f;
                    const float t = (s < r) ? __fmul_rn(dP, P) : 0.f;
                    scr[r * 65 + s] = t;
                    sa = __fadd_rn(sa, t);
                    x[e] = __fmul_rn(E, dP);                        // G1 = E . dP
                } else {
                    const bool in = s < r && r < nrows;
                    const float E = in ? simt::decay(gr, lr, gam[s], gml[s]) : 0.f;
                    const float Kd = __fmul_rn(E, v1[j]);
                    const float dA = in ? -v2[j] : 0.f;
                    sa = __fmaf_rn(dA, Kd, sa);                      // dbA part
                    bloc[j] = __fmul_rn(__fmul_rn(br, dA), Kd);
                    sb = __fadd_rn(sb, bloc[j]);                     // rowB part
                    x[e] = __fmul_rn(__fmul_rn(br, E), dA);         // G2 = b E dA
                }
            }
            // [G1; G2] K-major 128 x 64 tile: G1 in rows 0..63, G2 in rows 64..127
            store8_split(Rhi, Rlo, cm_off(row, s0 + j8 * 8, C), x);
        }
        // q^_r . (dO H^T)_r (top) or k_r . (dR H^T)_r (bottom), this thread's 64 columns
        const unsigned char* qrow = QK + (top ? 0 : 16384);
        float acc = 0.f;
        for (int c = 0; c < 2; ++c) {
            const int c0 = hf * 64 + c * 32;
            tmem_ld32(taddr_of(tmem + tX1, warp, c0), v1);
#pragma unroll
            for (int j8 = 0; j8 < 4; ++j8) {
                float qv[8];
                bf16x8_to_f32(*reinterpret_cast<const uint4*>(qrow + cm_off(r, c0 + j8 * 8, D)), qv);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    acc = __fmaf_rn(top ? __fmul_rn(scale, qv[e]) : qv[e], v1[j8 * 8 + e], acc);
            }
        }
        if (top) {
            rowA[hf * 64 + r] = sa;
            qh[hf * 64 + r] = acc;
        } else {
            dbA[hf * 64 + r] = sa;
            rowB[hf * 64 + r] = sb;
            kh[hf * 64 + r] = acc;
        }
    }
    __syncthreads();
    if (!top) {  // t_rs = dP_rs P_rs (written above) + b_r dA_rs Kd_rs
        const int s0 = hf * 32;
#pragma unroll
        for (int j = 0; j < 32; ++j) scr[r * 65 + s0 + j] = __fadd_rn(scr[r * 65 + s0 + j], bloc[j]);
    }
    __syncthreads();
    if (tid < C) {  // column sums colE_s = sum_{r > s} t_rs, ascending r (16 loads, then their adds)
        const int s = tid;
        float acc = 0.f;
#pragma unroll
        for (int r0 = 0; r0 < C; r0 += 16) {
            float v[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = scr[(r0 + e) * 65 + s];
#pragma unroll
            for (int e = 0; e < 16; ++e)
                if (r0 + e > s && r0 + e < nrows) acc = __fadd_rn(acc, v[e]);
        }
        colE[s] = acc;
    }
    {
        // dH' has arrived: X2 = [dR; Delta] dH'^T (rows 64.. are Delta dH'^T)
        const bool ok = mbar_wait(bar_dh, ph, a.err);
        if (__syncthreads_or(!ok)) { failed = true; break; }
    }
    pend_dh = false;
    if (tid == 0) {
        mma_tile<128, 128, D>(tmem + tX2, Rhi + 16384, Bt, false);
        mma_tile<128, 128, D>(tmem + tX2, Rhi + 16384, Bt + 32768, true);
        mma_tile<128, 128, D>(tmem + tX2, Rlo + 16384, Bt, true);
        mma_commit(bar_mma);
    }
    mma_out = true;
    {
        const bool ok = mbar_wait(bar_mma, ph_mma, a.err);
        fence_after();
        if (__syncthreads_or(!ok)) { failed = true; break; }
    }
    ph_mma ^= 1u;
    mma_out = false;
    if (tid == 0 && wn < nwork) {  // dH' is consumed: the next item's H_n goes to Bt already
        fence_async_smem();
        issue_hn(wn);
    }
    pend_hn = wn < nwork;
    ph_hn = ph ^ 1u;
    {
        // ---- phase E: MN-major A tiles (mn = 64 + s, k = r) of (scale G1)^T and G2^T from
        // the [G1; G2] tile's rows, interleaved in the dR / Delta space (free now: X2 is done);
        // e_s = dec_s k_s . (Delta dH'^T)_s
        unsigned char* mhi = Rhi + 16384 + (top ? 0 : 1024);
        unsigned char* mlo = Rlo + 16384 + (top ? 0 : 1024);
#pragma unroll
        for (int s8 = hf * 4; s8 < hf * 4 + 4; ++s8) {
            float x[8];
            join8(*reinterpret_cast<const uint4*>(Rhi + cm_off(row, s8 * 8, C)),
                  *reinterpret_cast<const uint4*>(Rlo + cm_off(row, s8 * 8, C)), x);
            if (top) {
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = __fmul_rn(scale, x[e]);
            }
            store8_split(mhi, mlo, mn_off(64 + s8 * 8, r, 128), x);
        }
        float v1[32], acc = 0.f;
        for (int c = 0; c < 2; ++c) {
            const int c0 = hf * 64 + c * 32;
            tmem_ld32(taddr_of(tmem + tX2, warp, c0), v1);
            if (!top) {
#pragma unroll
                for (int j8 = 0; j8 < 4; ++j8) {
                    float kv[8];
                    bf16x8_to_f32(*reinterpret_cast<const uint4*>(QK + 16384 + cm_off(r, c0 + j8 * 8, D)), kv);
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc = __fmaf_rn(kv[e], v1[j8 * 8 + e], acc);
                }
            }
        }
        if (!top) eL[hf * 64 + r] = acc;
    }
    fence_async_smem();
    tc_sync();
    if (tid == 0) {
        // interleaved MN-major tiles: (scale G1)^T at +0, G2^T at +1 KB (its garbage halves
        // lie on the other tile's rows, which no read of this accumulator uses)
        mma_tile_mj<128, 128, C, false, true>(tmem + tdq, Rhi, QK + 16384, false);          // [G1; G2] K
        mma_tile_mj<128, 128, C, false, true>(tmem + tdq, Rlo, QK + 16384, true);
        mma_tile_mj<128, 128, C, true, true>(tmem + tdk, Rhi + 16384, QK, false);           // (s G1)^T Q
        mma_tile_mj<128, 128, C, true, true>(tmem + tdk, Rlo + 16384, QK, true);
        mma_tile_mj<128, 128, C, true, true>(tmem + tdk, Rhi + 16384 + 1024, QK + 16384, true);  // G2^T K
        mma_tile_mj<128, 128, C, true, true>(tmem + tdk, Rlo + 16384 + 1024, QK + 16384, true);
        mma_commit(bar_mma);
    }
    mma_out = true;
    if (tid < C) {  // gate and beta gradients of row r = tid
        const int rr = tid;
        const float kr = __fadd_rn(kh[rr], kh[64 + rr]);
        const float qr = __fadd_rn(qh[rr], qh[64 + rr]);
        const float e_r = (rr < Lr) ? __fmul_rn(dec[rr], __fadd_rn(eL[rr], eL[64 + rr])) : 0.f;
        dgam[rr] = e_r;   // e_s, read by row L below after the barrier
        const float dG = __fsub_rn(qr, __fmul_rn(bet[rr], kr));
        const float dbR = __fsub_rn(dRv[rr], __fmul_rn(Gm[rr], kr));
        const float rowE = __fadd_rn(__fadd_rn(rowA[rr], rowA[64 + rr]), __fadd_rn(rowB[rr], rowB[64 + rr]));
        float dgr = __fsub_rn(__fadd_rn(__fmul_rn(Gm[rr], dG), rowE), colE[rr]);
        dgr = __fsub_rn(dgr, e_r);
        if (rr < nrows)
            a.dbeta[(size_t)(t0 + rr) * H + h] = __fadd_rn(dbR, __fadd_rn(dbA[rr], dbA[64 + rr]));
        eL[rr] = dgr;     // this row's dgam before the row-L terms
    }
    __syncthreads();
    if (tid < C) {
        const int rr = tid;
        float dgr = eL[rr];
        if (rr == Lr) {
            float sumL = 0.f, rs = 0.f;
#pragma unroll
            for (int s0 = 0; s0 < C; s0 += 16) {   // ascending s (16 loads, then their adds)
                float v[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) v[e] = dgam[s0 + e];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    if (s0 + e < Lr) sumL = __fadd_rn(sumL, v[e]);
            }
            for (int w = 0; w < a.nsplit; ++w) rs = __fadd_rn(rs, red[w]);
            dgr = __fadd_rn(dgr, __fadd_rn(__fmul_rn(Gm[Lr], rs), sumL));
        }
        colE[rr] = (rr < nrows) ? dgr : 0.f;   // dgam_r
    }
    __syncthreads();
    if (tid < nrows) {  // dg_s = sum_{r=s}^{L} dgam_r, from the last row down (16 loads, then their adds)
        float acc = 0.f;
#pragma unroll
        for (int r0 = C - 1; r0 >= 0; r0 -= 16) {
            float v[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = colE[r0 - e];
#pragma unroll
            for (int e = 0; e < 16; ++e)
                if (r0 - e <= Lr && r0 - e >= tid) acc = __fadd_rn(acc, v[e]);
        }
        a.dg[(size_t)(t0 + tid) * H + h] = acc;
    }
    {
        const bool ok = mbar_wait(bar_mma, ph_mma, a.err);
        fence_after();
        if (__syncthreads_or(!ok)) { failed = true; break; }
    }
    ph_mma ^= 1u;
    mma_out = false;
    if (tid == 0 && wn < nwork) {  // Q, K, the R tiles and gam are consumed: next item's inputs
        fence_async_smem();
        issue_in(wn);
    }
    pend_in = wn < nwork;
    ph_in = ph ^ 1u;
    {
        // dq rows (top), dk rows (bottom); this thread's 64 columns
        const bool in = r < nrows;
        float x1[32], y[32], z[32], w2[32];
        float* out = (top ? a.dq : a.dk) + ((size_t)(t0 + r) * H + h) * D;
        const float gr = Gm[r], nb = -bgv[r], dr = dec[r];
        for (int c = 0; c < 2; ++c) {
            const int c0 = hf * 64 + c * 32;
            tmem_ld32x4(taddr_of(tmem + tX1, warp, c0), x1, taddr_of(tmem + tdq, warp, c0), y,
                        taddr_of(tmem + tX2, warp, c0), z, taddr_of(tmem + tdk, warp, c0), w2);
            if (in) {   // whole 32-byte sectors: one row per lane
#pragma unroll
                for (int j8 = 0; j8 < 4; ++j8) {
                    float o8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int j = 8 * j8 + e;
                        // bottom: -bg X1 + dec X2 + (s G1)^T Q + G2^T K + G2 K (the last from tdq)
                        o8[e] = top ? __fmul_rn(scale, __fmaf_rn(gr, x1[j], y[j]))
                                    : __fadd_rn(__fadd_rn(__fmaf_rn(nb, x1[j], __fmul_rn(dr, z[j])), w2[j]), y[j]);
                    }
                    st_global_v8(out + c0 + 8 * j8, o8);
                }
            }
        }
    }
    }  // items
    if (failed) {   // let in-flight copies and MMAs finish (bounded) before TMEM is released
        if (pend_dh) mbar_wait(bar_dh, (uint32_t)(it & 1), a.err);
        if (mma_out) mbar_wait(bar_mma, ph_mma, a.err);
        if (pend_in) mbar_wait(bar_in, ph_in, a.err);
        if (pend_hn) mbar_wait(bar_hn, ph_hn, a.err);
    }
    tc_sync();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace tc
}  // namespace cpr
