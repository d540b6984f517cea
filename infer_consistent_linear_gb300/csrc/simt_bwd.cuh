// CPR Gated DeltaNet backward kernels, operand policy SIMT_F32.
//
// The backward of the chunk form used by the forward kernels (derived here
// from that form; the pages give the trainer forward+backward stage only as
// a timing).  Per chunk, with start state H, dH' = dL/dH_{n+1}, dO rows,
// E_rs = exp(gam_r - gam_s), kt_s = E_Ls k_s, bg_s = b_s G_s:
//   dD     = P^T dO + kt dH'                       (dL/dDelta)
//   dR     = T^T dD                                 (Delta = T R, R = diag(b)(V - diag(G) K H))
//   dA_rs  = -dR_r . D_s                 s < r
//   dP_rs  =  dO_r . D_s                 s <= r
//   dH     = G_L dH' + sum_r G_r q^_r dO_r^T - sum_r bg_r k_r dR_r^T
//   dv_r   = b_r dR_r
//   db_r   = dR_r . (v_r - G_r K H_r) + sum_{s<r} dA_rs E_rs kk_rs
//   dq^_r  = G_r H dO_r + sum_{s<=r} E_rs dP_rs k_s,            dq = scale dq^
//   dk_s   = -bg_s H dR_s + E_Ls dH' D_s + sum_{r>=s} E_rs dP_rs q^_r
//            + sum_{r>s} b_r E_rs dA_rs k_r + sum_{r<s} b_s E_sr dA_sr k_r
//   dgam_r = G_r dG_r + sum_{s<r} dE_rs E_rs - sum_{r'>r} dE_r'r E_r'r (+ the H' terms)
//     dG_r  = -b_r dR_r . KH_r + dO_r . QH_r,  dE_rs E_rs = dP_rs P_rs + b_r dA_rs E_rs kk_rs
//     H' terms: dgam_L += G_L <dH', H> + sum_{s<L} e_s,  dgam_s -= e_s,
//               e_s = E_Ls k_s . (dH' D_s)
//   dg_s   = sum_{r=s}^{L} dgam_r
// The backward has no bitwise coupling to another path; it is deterministic
// (every sum has a fixed order, no atomics) and batch-invariant (one CTA per
// chunk or per sequence, independent of the batch).
#pragma once

#include "simt_fwd.cuh"

namespace cpr {
namespace simt {

struct BwdArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* g;
    const float* beta;
    const int32_t* cu;
    const int32_t* chunk_off;
    int n_seq;
    int H;
    float scale;
    const float* dO;
    const float* dHT;
    // workspace (written by the forward-side kernels)
    const float* wsW;
    const float* wsU;
    const float* wsP;
    const float* wsGam;
    const float* wsT;
    const float* wsKd;
    const float* wsHn;
    float* wsdH;     // [chunks, H, d_k, d_v]: dL/d(end state) of every chunk
    // outputs
    float* dq;
    float* dk;
    float* dv;
    float* dg;
    float* dbeta;
    float* dh0;
    uint32_t* err;
};

// ---- reverse state pass: dL/dH_n for every chunk boundary ---------------------
template <class IO, int DK, int DV, int DVS>
__global__ void __launch_bounds__(256) k_state_bwd(BwdArgs a) {
    constexpr int C = kChunk;
    constexpr int LC = C + 4, LS = DVS + 4, LKI = DK + 8;
    constexpr int NSPLIT = DV / DVS;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float* Ps = reinterpret_cast<float*>(smem_raw);  // [C][LC]
    float* Ts = Ps + C * LC;                         // [C][LC]
    float* dOs = Ts + C * LC;                        // [C][LS]
    float* dD = dOs + C * LS;                        // [C][LS]
    float* dR = dD + C * LS;                         // [C][LS]
    float* dHs = dR + C * LS;                        // [DK][LS]
    float* Gm = dHs + DK * LS;                       // [C]
    float* bg = Gm + C;                              // [C]
    float* dec = bg + C;                             // [C]
    IO* Qs = reinterpret_cast<IO*>(dec + C);         // [C][LKI]
    IO* Ks = Qs + C * LKI;                           // [C][LKI]

    const int total = a.chunk_off[a.n_seq];
    if (total < 0) return;
    const int H = a.H;
    const int sp = blockIdx.x % NSPLIT;
    const int h = (blockIdx.x / NSPLIT) % H;
    const int b = blockIdx.x / (NSPLIT * H);
    const int j0 = sp * DVS, tid = threadIdx.x;
    const int seq0 = a.cu[b], T = a.cu[b + 1] - seq0;
    const int nch = a.chunk_off[b + 1] - a.chunk_off[b];
    const size_t sh = (size_t)b * H + h;
    const IO* q = static_cast<const IO*>(a.q);
    const IO* k = static_cast<const IO*>(a.k);
    const float scale = a.scale;

    for (int i = tid; i < DK * DVS; i += blockDim.x) {
        const int d = i / DVS, j = i % DVS;
        dHs[d * LS + j] = a.dHT ? a.dHT[(sh * DK + d) * DV + j0 + j] : 0.f;
    }
    for (int n = nch - 1; n >= 0; --n) {
        const int cidx = a.chunk_off[b] + n;
        const int t0 = seq0 + n * C;
        const int nrows = min(C, T - n * C);
        const int L = nrows - 1;
        const size_t ch = (size_t)cidx * H + h;
        __syncthreads();
        float* dHw = a.wsdH + ch * DK * DV;
        for (int i = tid; i < DK * DVS; i += blockDim.x)
            dHw[(i / DVS) * DV + j0 + i % DVS] = dHs[(i / DVS) * LS + i % DVS];
        const float* P = a.wsP + ch * C * C;
        const float* Tg = a.wsT + ch * C * C;
        for (int i = tid; i < C * C / 4; i += blockDim.x) {
            const int r = i / (C / 4), c4 = (i % (C / 4)) * 4;
            *reinterpret_cast<float4*>(Ps + r * LC + c4) = *reinterpret_cast<const float4*>(P + r * C + c4);
            *reinterpret_cast<float4*>(Ts + r * LC + c4) = *reinterpret_cast<const float4*>(Tg + r * C + c4);
        }
        for (int i = tid; i < C * DVS; i += blockDim.x) {
            const int r = i / DVS, j = i % DVS;
            dOs[r * LS + j] = (r < nrows) ? a.dO[((size_t)(t0 + r) * H + h) * DV + j0 + j] : 0.f;
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
            const float* gw = a.wsGam + ch * 2 * C;   // gate prefix hi | lo
            const bool in = tid < nrows;
            const float gr = gw[tid], lr = gw[C + tid];
            Gm[tid] = in ? gate(gr, lr) : 0.f;
            bg[tid] = in ? bg_entry(a.beta[(size_t)(t0 + tid) * H + h], gr, lr) : 0.f;
            dec[tid] = in ? decay(gw[L], gw[C + L], gr, lr) : 0.f;
        }
        __syncthreads();
        // dD = P^T dO + kt dH'
        tile_mm<4, 4>(C, DVS, Zero{},
            [&](int s, int x) { return x < C ? Ps[x * LC + s] : __fmul_rn(dec[s], cvt(Ks[s * LKI + x - C])); },
            [&](int x, int j) { return x < C ? dOs[x * LS + j] : dHs[(x - C) * LS + j]; },
            [&](int m0, int& k0, int& k1) { k0 = m0; k1 = C + DK; },
            [&](int m0, int n0, float (&acc)[4][4]) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) dD[(m0 + i) * LS + n0 + j] = acc[i][j];
            });
        __syncthreads();
        // dR = T^T dD
        tile_mm<4, 4>(C, DVS, Zero{},
            [&](int s, int r) { return Ts[r * LC + s]; },
            [&](int r, int j) { return dD[r * LS + j]; },
            [&](int m0, int& k0, int& k1) { k0 = m0; k1 = nrows; },
            [&](int m0, int n0, float (&acc)[4][4]) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) dR[(m0 + i) * LS + n0 + j] = acc[i][j];
            });
        __syncthreads();
        // dH = G_L dH' + sum_r G_r q^_r dO_r^T - sum_r bg_r k_r dR_r^T
        const float GL = Gm[L];
        tile_mm<4, 4>(DK, DVS,
            [&](int d, int j) { return __fmul_rn(GL, dHs[d * LS + j]); },
            [&](int d, int x) {
                return x < C ? __fmul_rn(Gm[x], qhat(scale, cvt(Qs[x * LKI + d])))
                             : -__fmul_rn(bg[x - C], cvt(Ks[(x - C) * LKI + d]));
            },
            [&](int x, int j) { return x < C ? dOs[x * LS + j] : dR[(x - C) * LS + j]; },
            [&](int m0, int& k0, int& k1) { k0 = 0; k1 = 2 * C; (void)m0; },
            [&](int m0, int n0, float (&acc)[4][4]) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) dHs[(m0 + i) * LS + n0 + j] = acc[i][j];
            });
    }
    __syncthreads();
    for (int i = tid; i < DK * DVS; i += blockDim.x)
        a.dh0[(sh * DK + i / DVS) * DV + j0 + i % DVS] = dHs[(i / DVS) * LS + i % DVS];
}

template <class IO, int DK, int DV, int DVS>
constexpr size_t state_bwd_smem() {
    return sizeof(float) * ((size_t)2 * kChunk * (kChunk + 4) + 3 * kChunk * (DVS + 4) +
                            DK * (DVS + 4) + 3 * kChunk) +
           sizeof(IO) * 2 * kChunk * (DK + 8);
}

// ---- per-chunk gradients (chunk-parallel) ------------------------------------
template <class IO, int DK, int DV>
__global__ void __launch_bounds__(256) k_grad_chunk(BwdArgs a) {
    constexpr int C = kChunk;
    constexpr int LKI = DK + 8, LVI = DV + 8, LV = DV + 4, LC = C + 1;
    constexpr int NJT = DV / 4;  // column tiles of width 4
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float* dOs = reinterpret_cast<float*>(smem_raw);  // [C][LV]
    float* Dl = dOs + C * LV;                         // [C][LV]  Delta
    float* dR = Dl + C * LV;                          // [C][LV]
    float* G1 = dR + C * LV;                          // [C][LC]  dP, then E*dP
    float* G2 = G1 + C * LC;                          // [C][LC]  dA, then b E dA
    float* part1 = G2 + C * LC;                       // [C][NJT]
    float* part2 = part1 + C * NJT;                   // [C][NJT]
    float* gam = part2 + C * NJT;                     // [C] gate prefix, hi
    float* gml = gam + C;                             // [C] gate prefix, lo
    float* Gm = gml + C;
    float* bet = Gm + C;
    float* bg = bet + C;
    float* decL = bg + C;
    float* dgam = decL + C;                           // [C]
    float* eL = dgam + C;                             // [C]
    float* red = eL + C;                              // [256]
    IO* Ks = reinterpret_cast<IO*>(red + 256);        // [C][LKI]
    IO* Qs = Ks + C * LKI;                            // [C][LKI]
    IO* Vs = Qs + C * LKI;                            // [C][LVI]
    float* dDtmp = G1;  // dD lives in the G1/G2 region (C*DV <= 2*C*LC) until dR exists

    const int total = a.chunk_off[a.n_seq];
    const int cidx = blockIdx.x, h = blockIdx.y, H = a.H;
    if (total < 0 || cidx >= total) return;
    const int b = find_seq(a.chunk_off, a.n_seq, cidx);
    const int n = cidx - a.chunk_off[b];
    const int seq0 = a.cu[b], T = a.cu[b + 1] - seq0;
    const int t0 = seq0 + n * C;
    const int nrows = min(C, T - n * C);
    const int L = nrows - 1;
    const int tid = threadIdx.x;
    const size_t ch = (size_t)cidx * H + h;
    const IO* q = static_cast<const IO*>(a.q);
    const IO* k = static_cast<const IO*>(a.k);
    const IO* v = static_cast<const IO*>(a.v);
    const float scale = a.scale;
    const float* Hn = a.wsHn + ch * DK * DV;
    const float* dHn = a.wsdH + ch * DK * DV;
    const float* Wg = a.wsW + ch * C * DK;
    const float* Ug = a.wsU + ch * C * DV;
    const float* Pg = a.wsP + ch * C * C;
    const float* Tg = a.wsT + ch * C * C;
    const float* Kdg = a.wsKd + ch * C * C;

    // ---- P1: loads
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
    for (int i = tid; i < C * (DV / 8); i += blockDim.x) {
        const int r = i / (DV / 8), c8 = (i % (DV / 8)) * 8;
        float vv[8];
        if (r < nrows) {
            load8(v + ((size_t)(t0 + r) * H + h) * DV + c8, vv);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) vv[e] = 0.f;
        }
        store8(Vs + r * LVI + c8, vv);
    }
    for (int i = tid; i < C * DV / 4; i += blockDim.x) {
        const int r = i / (DV / 4), c4 = (i % (DV / 4)) * 4;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < nrows) x = *reinterpret_cast<const float4*>(a.dO + ((size_t)(t0 + r) * H + h) * DV + c4);
        *reinterpret_cast<float4*>(dOs + r * LV + c4) = x;
    }
    if (tid < C) {
        const bool in = tid < nrows;
        const float* gw = a.wsGam + ch * 2 * C;   // gate prefix hi | lo
        const float gr = gw[tid], lr = gw[C + tid];
        const float br = in ? a.beta[(size_t)(t0 + tid) * H + h] : 0.f;
        gam[tid] = gr;
        gml[tid] = lr;
        Gm[tid] = in ? gate(gr, lr) : 0.f;
        bet[tid] = br;
        bg[tid] = in ? bg_entry(br, gr, lr) : 0.f;
        decL[tid] = in ? decay(gw[L], gw[C + L], gr, lr) : 0.f;
    }
    __syncthreads();
    // ---- P2: Delta = U - W' H (the forward's chains)
    tile_mm<4, 4>(C, DV, Zero{},
        [&](int r, int d) { return Wg[r * DK + d]; },
        [&](int d, int j) { return Hn[d * DV + j]; },
        [&](int m0, int& k0, int& k1) { k0 = 0; k1 = DK; (void)m0; },
        [&](int m0, int n0, float (&acc)[4][4]) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int r = m0 + i;
                    Dl[r * LV + n0 + j] = (r < nrows) ? __fsub_rn(Ug[r * DV + n0 + j], acc[i][j]) : 0.f;
                }
        });
    // ---- P3: dD = P^T dO + kt dH'
    tile_mm<4, 4>(C, DV, Zero{},
        [&](int s, int x) { return x < C ? Pg[x * C + s] : __fmul_rn(decL[s], cvt(Ks[s * LKI + x - C])); },
        [&](int x, int j) { return x < C ? dOs[x * LV + j] : dHn[(x - C) * DV + j]; },
        [&](int m0, int& k0, int& k1) { k0 = m0; k1 = C + DK; },
        [&](int m0, int n0, float (&acc)[4][4]) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) dDtmp[(m0 + i) * DV + n0 + j] = acc[i][j];
        });
    __syncthreads();
    // ---- P4: dR = T^T dD
    tile_mm<4, 4>(C, DV, Zero{},
        [&](int s, int r) { return Tg[r * C + s]; },
        [&](int r, int j) { return dDtmp[r * DV + j]; },
        [&](int m0, int& k0, int& k1) { k0 = m0; k1 = nrows; },
        [&](int m0, int n0, float (&acc)[4][4]) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) dR[(m0 + i) * LV + n0 + j] = acc[i][j];
        });
    __syncthreads();
    // ---- P5: row partials of dR_r . KH_r and dO_r . QH_r (4-column tiles)
    tile_mm<4, 4>(2 * C, DV, Zero{},
        [&](int m, int d) { return m < C ? cvt(Ks[m * LKI + d]) : qhat(scale, cvt(Qs[(m - C) * LKI + d])); },
        [&](int d, int j) { return Hn[d * DV + j]; },
        [&](int m0, int& k0, int& k1) { k0 = 0; k1 = DK; (void)m0; },
        [&](int m0, int n0, float (&acc)[4][4]) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int m = m0 + i;
                float s = 0.f;
                if (m < C) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) s = __fmaf_rn(dR[m * LV + n0 + j], acc[i][j], s);
                    part1[m * NJT + n0 / 4] = s;
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) s = __fmaf_rn(dOs[(m - C) * LV + n0 + j], acc[i][j], s);
                    part2[(m - C) * NJT + n0 / 4] = s;
                }
            }
        });
    // ---- P6: dP = dO D^T (s <= r), dA = -dR D^T (s < r)
    tile_mm<4, 4>(2 * C, C, Zero{},
        [&](int m, int j) { return m < C ? dOs[m * LV + j] : dR[(m - C) * LV + j]; },
        [&](int j, int s) { return Dl[s * LV + j]; },
        [&](int m0, int& k0, int& k1) { k0 = 0; k1 = DV; (void)m0; },
        [&](int m0, int n0, float (&acc)[4][4]) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int m = m0 + i, s = n0 + j;
                    if (m < C) G1[m * LC + s] = (s <= m && m < nrows) ? acc[i][j] : 0.f;
                    else G2[(m - C) * LC + s] = (s < m - C && m - C < nrows) ? -acc[i][j] : 0.f;
                }
        });
    __syncthreads();
    // ---- P7: per-row scalars (dG_r, db_r, dE row sums) and dE column sums
    float rowE = 0.f, colE = 0.f, dG = 0.f, dbR = 0.f, dbA = 0.f;
    if (tid < C) {
        const int r = tid;
        float dRKH = 0.f, dOQH = 0.f, dRv = 0.f;
        for (int t = 0; t < NJT; ++t) {
            dRKH = __fadd_rn(dRKH, part1[r * NJT + t]);
            dOQH = __fadd_rn(dOQH, part2[r * NJT + t]);
        }
        for (int j = 0; j < DV; ++j) dRv = __fmaf_rn(dR[r * LV + j], cvt(Vs[r * LVI + j]), dRv);
        dG = __fsub_rn(dOQH, __fmul_rn(bet[r], dRKH));
        dbR = __fsub_rn(dRv, __fmul_rn(Gm[r], dRKH));
        for (int s = 0; s < r; ++s) {
            const float kd = Kdg[r * C + s];
            const float da = G2[r * LC + s];
            dbA = __fmaf_rn(da, kd, dbA);
            rowE = __fmaf_rn(G1[r * LC + s], Pg[r * C + s], rowE);
            rowE = __fmaf_rn(__fmul_rn(bet[r], da), kd, rowE);
        }
    } else if (tid < 2 * C) {
        const int s = tid - C;
        for (int r = s + 1; r < nrows; ++r) {
            colE = __fmaf_rn(G1[r * LC + s], Pg[r * C + s], colE);
            colE = __fmaf_rn(__fmul_rn(bet[r], G2[r * LC + s]), Kdg[r * C + s], colE);
        }
    }
    // ---- P8: e_s = E_Ls k_s . (dH' D_s) partials, <dH', H>
    __syncthreads();  // part1 reused below
    tile_mm<4, 4>(C, DV, Zero{},
        [&](int s, int d) { return cvt(Ks[s * LKI + d]); },
        [&](int d, int j) { return dHn[d * DV + j]; },
        [&](int m0, int& k0, int& k1) { k0 = 0; k1 = DK; (void)m0; },
        [&](int m0, int n0, float (&acc)[4][4]) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int s = m0 + i;
                float x = 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j) x = __fmaf_rn(Dl[s * LV + n0 + j], acc[i][j], x);
                part1[s * NJT + n0 / 4] = x;
            }
        });
    {
        float acc = 0.f;
        for (int i = tid; i < DK * DV; i += blockDim.x) acc = __fmaf_rn(dHn[i], Hn[i], acc);
        red[tid] = acc;
    }
    __syncthreads();
    if (tid < C) {
        float x = 0.f;
        for (int t = 0; t < NJT; ++t) x = __fadd_rn(x, part1[tid * NJT + t]);
        eL[tid] = (tid < L) ? __fmul_rn(decL[tid], x) : 0.f;
    }
    if (tid == 0) {  // fixed-order sum of the 256 partials
        float acc = 0.f;
        for (int i = 0; i < 256; ++i) acc = __fadd_rn(acc, red[i]);
        red[0] = acc;
    }
    if (tid >= C && tid < 2 * C) dgam[tid - C] = colE;
    __syncthreads();
    if (tid < C) {
        const int r = tid;
        float dgr = __fsub_rn(__fadd_rn(__fmul_rn(Gm[r], dG), rowE), dgam[r]);
        dgr = __fsub_rn(dgr, eL[r]);
        if (r == L) {
            float sumL = 0.f;
            for (int s = 0; s < L; ++s) sumL = __fadd_rn(sumL, eL[s]);
            dgr = __fadd_rn(dgr, __fadd_rn(__fmul_rn(Gm[L], red[0]), sumL));
        }
        if (r < nrows) a.dbeta[(size_t)(t0 + r) * H + h] = __fadd_rn(dbR, dbA);
        part2[r] = (r < nrows) ? dgr : 0.f;
    }
    __syncthreads();
    if (tid < nrows) {  // dg_s = sum_{r=s}^{L} dgam_r, from the last row down
        float acc = 0.f;
        for (int r = L; r >= tid; --r) acc = __fadd_rn(acc, part2[r]);
        a.dg[(size_t)(t0 + tid) * H + h] = acc;
    }
    // ---- P9: G1 <- E dP (s <= r), G2 <- b_r E dA (s < r)
    for (int i = tid; i < C * C; i += blockDim.x) {
        const int r = i / C, s = i % C;
        if (r < nrows && s <= r) {
            const float e = decay(gam[r], gml[r], gam[s], gml[s]);
            G1[r * LC + s] = __fmul_rn(e, G1[r * LC + s]);
            G2[r * LC + s] = (s < r) ? __fmul_rn(__fmul_rn(bet[r], e), G2[r * LC + s]) : 0.f;
        }
    }
    for (int i = tid; i < nrows * DV; i += blockDim.x) {  // dv = b dR
        const int r = i / DV, j = i % DV;
        a.dv[((size_t)(t0 + r) * H + h) * DV + j] = __fmul_rn(bet[r], dR[r * LV + j]);
    }
    __syncthreads();
    // ---- P10: dq = scale (G_r H dO_r + sum_{s<=r} E dP_rs k_s)
    tile_mm<4, 4>(C, DK, Zero{},
        [&](int r, int x) { return x < DV ? __fmul_rn(Gm[r], dOs[r * LV + x]) : G1[r * LC + x - DV]; },
        [&](int x, int d) { return x < DV ? Hn[d * DV + x] : cvt(Ks[(x - DV) * LKI + d]); },
        [&](int m0, int& k0, int& k1) { k0 = 0; k1 = DV + min(m0 + 4, nrows); },
        [&](int m0, int n0, float (&acc)[4][4]) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = m0 + i;
                if (r < nrows)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        a.dq[((size_t)(t0 + r) * H + h) * DK + n0 + j] = __fmul_rn(scale, acc[i][j]);
            }
        });
    // ---- P11: dk
    tile_mm<4, 4>(C, DK, Zero{},
        [&](int s, int x) {
            if (x < DV) return -__fmul_rn(bg[s], dR[s * LV + x]);
            if (x < 2 * DV) return __fmul_rn(decL[s], Dl[s * LV + x - DV]);
            if (x < 2 * DV + C) return G1[(x - 2 * DV) * LC + s];
            const int r = x - 2 * DV - C;
            return __fadd_rn(G2[r * LC + s], G2[s * LC + r]);
        },
        [&](int x, int d) {
            if (x < DV) return Hn[d * DV + x];
            if (x < 2 * DV) return dHn[d * DV + x - DV];
            if (x < 2 * DV + C) return qhat(scale, cvt(Qs[(x - 2 * DV) * LKI + d]));
            return cvt(Ks[(x - 2 * DV - C) * LKI + d]);
        },
        [&](int m0, int& k0, int& k1) { k0 = 0; k1 = 2 * DV + 2 * C; (void)m0; },
        [&](int m0, int n0, float (&acc)[4][4]) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int s = m0 + i;
                if (s < nrows)
#pragma unroll
                    for (int j = 0; j < 4; ++j) a.dk[((size_t)(t0 + s) * H + h) * DK + n0 + j] = acc[i][j];
            }
        });
}

template <class IO, int DK, int DV>
constexpr size_t grad_chunk_smem() {
    return sizeof(float) * ((size_t)3 * kChunk * (DV + 4) + 2 * kChunk * (kChunk + 1) +
                            2 * kChunk * (DV / 4) + 8 * kChunk + 256) +
           sizeof(IO) * ((size_t)2 * kChunk * (DK + 8) + kChunk * (DV + 8));
}

}  // namespace simt
}  // namespace cpr
