// CPR Gated DeltaNet decode step on the tensor cores (policy TC_BF16X3).
//
// Per (sequence, head) unit: for the new row p of the current chunk it
// re-issues exactly the MMA instructions of the prefill kernels (k_tc_prep,
// k_tc_state): same shapes, same operand tiles, layouts and row positions,
// same k-step and hi/lo pass order, with the rows of the chunk that do not
// exist yet set to zero.  An output row of an MMA depends only on its own A
// row and on B, and zero rows of B only meet zero entries of the row's A (T
// and P are lower triangular), so row p gets the prefill's bits.  The fp32
// parts (gate prefix, exponentials, T row, epilogues) are the same operation
// sequences as the prefill's.  When the chunk fills (p = C - 1) the step
// commits the next chunk-start state with the prefill's commit MMAs: the
// resynchronisation every C tokens (page "IsoExec: 切换 SkyRL 中的训练器-
// 推理不匹配", section "Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet").
#pragma once

#include "tc_fwd.cuh"

namespace cpr {
namespace tc {

struct DecSmem {
    static constexpr size_t Hhi = 0, Hlo = 32768;   // state tiles, per split MN-major DVS (j) x 128 (d)
    static constexpr size_t Kmn = 65536;             // K tile, MN-major 128 (d) x 64 (token)
    static constexpr size_t R1 = 81920;              // 64 KB right after Kmn, reused by phase
    static constexpr size_t Vt = R1 + 65536;         // V tile, MN-major 128 (d) x 64 (token)
    static constexpr size_t F = Vt + 16384;          // fp32 scratch
    static constexpr int fGam = 0, fBet = 64, fBg = 128, fArow = 192, fProw = 256, fTrow = 320,
                         fDec = 384, fWp = 448, fUp = 576, fDp = 704, fQs = 832, fRow = 960,
                         fRow2 = 1088, fGml = 1216, fEnd = 1280;
    static constexpr size_t Dt = F + 5120;           // Delta tiles: hi (16 KB) | lo (16 KB), per split
                                                     // MN-major DVS (j) x 64 (token); at a commit the
                                                     // fp32 Delta rows
    static constexpr size_t Tt = Dt + 32768;         // the cached T rows, fp32 [C][C] (rows < p valid)
    static constexpr size_t Bar = Tt + C * C * 4;    // 4 mbarriers + TMEM base
    static constexpr size_t Total = Bar + 64;
};

struct TcDecArgs {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
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

// A bulk copy (as bulk_g2s) with an L2 eviction-priority hint, a cache policy from
// l2_policy: data read once per step can leave L2 before the data every step reads again.
__device__ __forceinline__ void bulk_g2s_hint(void* dst_smem, const void* src, uint32_t bytes, uint64_t* mbar,
                                              uint64_t policy) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
                 :: "r"(smem_u32(dst_smem)), "l"(src), "r"(bytes), "r"(smem_u32(mbar)), "l"(policy) : "memory");
}
template <bool LAST>
__device__ __forceinline__ uint64_t l2_policy() {
    uint64_t pol;
    if (LAST) asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    else asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 16 KB of zeros (never written) that fill the rows of a decode operand tile past the
// unit's position: a bulk copy of it hits L2, where the cache's own zero rows cost HBM reads.
static __device__ __align__(128) unsigned char kZeroTile[16384];

// After a prefill that writes a decode cache: the chunk-start state and the current
// chunk's Delta rows (rows >= pos zero) as the decode's hi/lo operand tiles, per split
// MN-major (split sp at sp * DVS * 256 / 128 bytes, lo tiles 32 KB / 16 KB after hi) --
// split8 of the fp32 values the state pass left in the cache, so the decode reads the
// same bits it would compute itself.  The K and V rows of the current chunk are kept
// as operand tiles (row r at cm_off(r, ., D), written by the prefill for r < pos); their
// rows >= pos are zeroed here.  One CTA per (sequence, head).
template <int DVS>
__global__ void __launch_bounds__(256) k_tc_cache_tiles(uint8_t* cache, CacheOff co, const int32_t* chunk_off,
                                                        int n_seq, int H) {
    if (chunk_off[n_seq] < 0) return;   // rejected cu_seqlens: the prefill wrote nothing
    const size_t sh = blockIdx.x;
    const int b = (int)(sh / H);
    const int p = reinterpret_cast<const int32_t*>(cache + co.pos)[b];
    const float* Hs = reinterpret_cast<const float*>(cache + co.state) + sh * D * D;
    const float* Dr = reinterpret_cast<const float*>(cache + co.delta_rows) + sh * C * D;
    unsigned char* ct = cache + co.state_tiles + sh * 65536;
    unsigned char* cdt = cache + co.delta_tiles + sh * 32768;
    unsigned char* ckt = cache + co.k_rows + sh * C * D * 2;
    unsigned char* cvt = cache + co.v_rows + sh * C * D * 2;
    for (int i = threadIdx.x; i < (C - p) * (D / 8); i += blockDim.x) {
        const uint32_t off = cm_off(p + i / (D / 8), (i % (D / 8)) * 8, D);
        *reinterpret_cast<uint4*>(ckt + off) = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(cvt + off) = make_uint4(0u, 0u, 0u, 0u);
    }
    for (int i = threadIdx.x; i < (D + C) * (D / 8); i += blockDim.x) {
        const bool st = i < D * (D / 8);
        const int rr = (st ? i : i - D * (D / 8)) / (D / 8), j8 = i % (D / 8);
        float x[8];
        if (st || rr < p) {
            const float4* src = reinterpret_cast<const float4*>((st ? Hs : Dr) + (size_t)rr * D + j8 * 8);
            const float4 u0 = src[0], u1 = src[1];
            x[0] = u0.x; x[1] = u0.y; x[2] = u0.z; x[3] = u0.w;
            x[4] = u1.x; x[5] = u1.y; x[6] = u1.z; x[7] = u1.w;
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = 0.f;
        }
        uint4 hi, lo;
        split8(x, hi, lo);
        if (st) {
            const uint32_t off = mn_off(j8 * 8, rr, D);
            *reinterpret_cast<uint4*>(ct + off) = hi;
            *reinterpret_cast<uint4*>(ct + 32768 + off) = lo;
        } else {
            const uint32_t off = mn_off(j8 * 8, rr, D);
            *reinterpret_cast<uint4*>(cdt + off) = hi;
            *reinterpret_cast<uint4*>(cdt + 16384 + off) = lo;
        }
    }
}

// One thread's 128 loaded columns into a 16-byte aligned row of shared memory.
__device__ __forceinline__ void store_row128(float* dst, const float (&v)[128]) {
#pragma unroll
    for (int j = 0; j < 128; j += 4)
        *reinterpret_cast<float4*>(dst + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
}

// Persistent: a CTA per SM walks the (sequence, head) units of the step.  While
// unit u runs, the next unit's operands arrive by bulk copies into buffers u no
// longer needs: K and V tiles once the X MMA has read them, the state tiles once
// A4 has, the Delta prefix once P Delta has (after the commit MMA when u commits),
// and the new token's q, k, v pieces and gate rows into registers.
// A unit needs one row of each chunk-form product (row p, and the q row p), so the
// products the prefill takes as M = 128 groups ([K; Q] K^T and [W'; Q] H) run here as
// M = 64 groups over an A tile that holds just the two rows (p and p ^ 32): an output
// element's bits do not depend on the instruction's M or N, nor on which row it sits in.
// 160 threads: warps 0..3 do the unit's operand and epilogue work, warp 4 only issues the
// MMA groups (about 56 cycles an instruction, during which the issuing warp does nothing else)
// and the bulk copies.
constexpr int kDecThreads = 160, kDecIssuer = 128;

template <int DVS>
__global__ void __launch_bounds__(kDecThreads, 1) k_tc_decode(TcDecArgs a) {
    using S = DecSmem;
    extern __shared__ __align__(1024) unsigned char sm[];
    float* F = reinterpret_cast<float*>(sm + S::F);
    float *gams = F + S::fGam, *bets = F + S::fBet, *bgs = F + S::fBg, *arow = F + S::fArow,
          *prow = F + S::fProw, *trow = F + S::fTrow, *decs = F + S::fDec, *Wp = F + S::fWp,
          *Up = F + S::fUp, *Dp = F + S::fDp, *Qs = F + S::fQs, *row1 = F + S::fRow,
          *row2 = F + S::fRow2, *gmls = F + S::fGml;
    uint64_t* mbar = reinterpret_cast<uint64_t*>(sm + S::Bar);   // MMA groups
    uint64_t* bar_H = mbar + 1;                                   // state tiles
    uint64_t* bar_D = mbar + 2;                                   // Delta tiles; fp32 Delta rows
    uint64_t* bar_KV = mbar + 3;                                  // K and V tiles
    uint32_t* tbase = reinterpret_cast<uint32_t*>(mbar + 4);
    float* stage = reinterpret_cast<float*>(sm + S::Dt);   // fp32 Delta rows at a commit
    unsigned char* R1 = sm + S::R1;
    __shared__ int ok_s;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H;
    const int nunit = a.n_seq * H;
    const uint32_t* hdr = reinterpret_cast<const uint32_t*>(a.cache + a.co.header);
    int32_t* pos = reinterpret_cast<int32_t*>(a.cache + a.co.pos);
    uint32_t* done = reinterpret_cast<uint32_t*>(a.cache + a.co.done);
    if (warp == 0) {
        // the cache header, a word per lane (words 0..9 + kHdrWords), and only once it is
        // the expected one the position of every unit this CTA takes, a unit per lane
        bool ok = cache_header_ok(hdr, a.digest.w, a.hdr);
        if (ok) {
            bool okp = true;
            for (int u = blockIdx.x + lane * (int)gridDim.x; u < nunit; u += 32 * (int)gridDim.x) {
                const int p = pos[u / H];
                okp = okp & (p >= 0) & (p < C);
            }
            ok = __all_sync(0xffffffffu, okp);
        }
        if (lane == 0) {
            if (!ok) set_error(a.err, CPR_ERR_CONTRACT_MISMATCH);
            ok_s = ok ? 1 : 0;
        }
    }
    __syncthreads();
    if (!ok_s || (int)blockIdx.x >= nunit) return;

    // unit u = sequence u / H, head u % H = row u of every [n_seq, H, ...] section
    auto k_tile = [&](int u) { return a.cache + a.co.k_rows + (size_t)u * C * D * 2; };
    auto v_tile = [&](int u) { return a.cache + a.co.v_rows + (size_t)u * C * D * 2; };
    // Of the K, V and Delta tiles and the T rows only the rows below the unit's position pu
    // hold data: the copies take the 8-row groups that contain them (2 KB each in every
    // tile) and the T rows below pu.  The rest of each tile, zero in the cache, is copied
    // from kZeroTile instead, which every CTA reads and so stays in L2.
    const uint64_t pol_keep = l2_policy<true>();
    auto tile_g2s = [&](unsigned char* dst, const unsigned char* src, uint32_t head, uint64_t* bar) {
        if (head) bulk_g2s_hint(dst, src, head, bar, pol_keep);
        if (head < 16384u) bulk_g2s(dst + head, kZeroTile, 16384u - head, bar);
    };
    auto issue_KV = [&](int u, int pu) {   // K and V tiles and the T rows
        const uint32_t kv = (uint32_t)((pu + 7) >> 3) * 2048u, tr = (uint32_t)pu * C * 4;
        mbar_expect_tx(bar_KV, 2 * 16384u + tr);
        tile_g2s(sm + S::Kmn, k_tile(u), kv, bar_KV);
        tile_g2s(sm + S::Vt, v_tile(u), kv, bar_KV);
        if (tr) bulk_g2s_hint(sm + S::Tt, a.cache + a.co.t_rows + (size_t)u * C * C * 4, tr, bar_KV, pol_keep);
    };
    // The state tiles (64 KB a unit, 134 MB a step on 2048 units) stream through L2 with the
    // evict-first priority, and the chunk's K, V, Delta and T rows, which every step of the
    // chunk reads again, are read with evict-last, so that they can stay in L2 from one step
    // to the next.
    const uint64_t pol_stream = l2_policy<false>();
    auto issue_H = [&](int u) {
        mbar_expect_tx(bar_H, 65536);
        bulk_g2s_hint(sm + S::Hhi, a.cache + a.co.state_tiles + (size_t)u * 65536, 65536, bar_H, pol_stream);
    };
    auto issue_D = [&](int u, int pu) {  // the Delta hi and lo tiles
        const uint32_t dt = (uint32_t)((pu + 7) >> 3) * 2048u;
        const unsigned char* src = a.cache + a.co.delta_tiles + (size_t)u * 32768;
        mbar_expect_tx(bar_D, 2 * 16384u);
        tile_g2s(sm + S::Dt, src, dt, bar_D);
        tile_g2s(sm + S::Dt + 16384, src + 16384, dt, bar_D);
    };
    // the new token's q (threads 0..15), k (16..31), v (32..47) pieces and the cached
    // gate / beta rows, into registers (the n* set is the next unit's, loaded while this
    // one runs); every load reads valid memory, masks apply at use
    uint4 rowreg = make_uint4(0u, 0u, 0u, 0u), nrowreg = rowreg;
    float cgv = 0.f, clv = 0.f, cbv = 0.f, gprev = 0.f, lprev = 0.f, gnew = 0.f, bnew = 0.f;
    float ncgv = 0.f, nclv = 0.f, ncbv = 0.f, ngprev = 0.f, nlprev = 0.f, ngnew = 0.f, nbnew = 0.f;
    auto load_rows = [&](int u, int p) {
        if (tid < 48) {
            const __nv_bfloat16* src = (tid < 16 ? a.q : tid < 32 ? a.k : a.v) + (size_t)u * D + (tid & 15) * 8;
            nrowreg = *reinterpret_cast<const uint4*>(src);
        }
        const float* cg = reinterpret_cast<const float*>(a.cache + a.co.gam_rows) + (size_t)u * 2 * C;
        const float* cb = reinterpret_cast<const float*>(a.cache + a.co.beta_rows) + (size_t)u * C;
        ncgv = cg[tid & (C - 1)];
        nclv = cg[C + (tid & (C - 1))];
        ncbv = cb[tid & (C - 1)];
        ngprev = cg[p > 0 ? p - 1 : 0];
        nlprev = cg[C + (p > 0 ? p - 1 : 0)];
        ngnew = a.g[u];
        nbnew = a.beta[u];
    };
    auto take_rows = [&]() {
        rowreg = nrowreg;
        cgv = ncgv; clv = nclv; cbv = ncbv; gprev = ngprev; lprev = nlprev; gnew = ngnew; bnew = nbnew;
    };

    if (warp == 0) tmem_alloc(tbase, 256);
    int p = pos[blockIdx.x / H];
    if (tid == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(mbar + i, 1);
        mbar_init_fence();
        issue_KV(blockIdx.x, p);
        issue_H(blockIdx.x);
        issue_D(blockIdx.x, p);
    }
    load_rows(blockIdx.x, p);
    take_rows();
    tc_sync();
    const uint32_t tmem = *tbase;
    uint32_t ph_mma = 0, ph_H = 0, ph_D = 0, ph_KV = 0;
    bool pend_KV = true, pend_H = true, pend_D = true, mma_out = false;
    bool ok = true;
    auto mma_wait = [&]() {
        const bool w = mbar_wait(mbar, ph_mma, a.err);
        fence_after();
        if (w) {
            ph_mma ^= 1u;
            mma_out = false;
        }
        return !__syncthreads_or(!w);
    };

    for (int u = blockIdx.x; u < nunit; u += gridDim.x) {
    const size_t sh = (size_t)u;
    const int un = u + (int)gridDim.x;
    const bool has_next = un < nunit;
    int pn = 0;   // the next unit's position, read once the S1 MMA is on its way
    __nv_bfloat16* ck = reinterpret_cast<__nv_bfloat16*>(k_tile(u));
    __nv_bfloat16* cv = reinterpret_cast<__nv_bfloat16*>(v_tile(u));
    float* cg = reinterpret_cast<float*>(a.cache + a.co.gam_rows) + sh * 2 * C;   // hi | lo
    float* cb = reinterpret_cast<float*>(a.cache + a.co.beta_rows) + sh * C;
    float* ct = reinterpret_cast<float*>(a.cache + a.co.t_rows) + sh * C * C;
    float* cd = reinterpret_cast<float*>(a.cache + a.co.delta_rows) + sh * C * D;
    float* Hst = reinterpret_cast<float*>(a.cache + a.co.state) + sh * D * D;
    unsigned char* cst = a.cache + a.co.state_tiles + sh * 65536;     // state hi | lo tiles
    unsigned char* cdt = a.cache + a.co.delta_tiles + sh * 32768;     // Delta hi | lo tiles
    // once this unit's K and V tiles have landed (each thread waits itself): row p from the
    // new token; the S1 operand (R1's first 16 KB) takes k_p as row p and q_p as row p ^ 32
    // (its other rows reach only accumulator rows never read)
    const bool wkv = mbar_wait(bar_KV, ph_KV, a.err);
    if (wkv) {
        ph_KV ^= 1u;
        pend_KV = false;
        if (tid < 16) {
            *reinterpret_cast<uint4*>(R1 + cm_off(p ^ 32, tid * 8, D)) = rowreg;
        } else if (tid < 32) {
            *reinterpret_cast<uint4*>(sm + S::Kmn + cm_off(p, (tid - 16) * 8, D)) = rowreg;
            *reinterpret_cast<uint4*>(R1 + cm_off(p, (tid - 16) * 8, D)) = rowreg;
        } else if (tid < 48) {
            *reinterpret_cast<uint4*>(sm + S::Vt + cm_off(p, (tid - 32) * 8, D)) = rowreg;
        }
    }
    if (tid < p) {
        gams[tid] = cgv;
        gmls[tid] = clv;
        bets[tid] = cbv;
    }
    if (tid == 0) {
        float hi = p > 0 ? gprev : 0.f, lo = p > 0 ? lprev : 0.f;
        simt::gam_add(hi, lo, gnew);
        gams[p] = hi;
        gmls[p] = lo;
        bets[p] = bnew;
    }
    fence_async_smem();
    fence_before();
    if (__syncthreads_or(!wkv)) { ok = false; break; }
    fence_after();
    if (has_next) pn = pos[un / H];
    if (tid == kDecIssuer) {
        mma_tile<64, 64, D>(tmem, R1, sm + S::Kmn, false);
        mma_commit(mbar);
    }
    mma_out = true;
    if (tid <= p) bgs[tid] = simt::bg_entry(bets[tid], gams[tid], gmls[tid]);
    // while S1 runs: the exponentials of row p's A and P entries and Gamma_p (the factors
    // a_entry, p_entry and the state scaling take, in their order)
    const float Gp = simt::gate(gams[p], gmls[p]);
    float Eps = 0.f, bEps = 0.f;
    if (tid < C) {
        Eps = simt::decay(gams[p], gmls[p], gams[tid], gmls[tid]);
        bEps = __fmul_rn(bets[p], Eps);
    }
    if (!mma_wait()) { ok = false; break; }
    if (warp == (p >> 4) || warp == ((p ^ 32) >> 4)) {   // the lane quarters of rows p, p ^ 32
        float v0[32], v1[32];
        tmem_ld32x2(taddr_of(tmem, warp, 0), v0, taddr_of(tmem, warp, 32), v1);
        float* dst = tid == lane_m64(p) ? row1 : tid == lane_m64(p ^ 32) ? row2 : nullptr;
        if (dst) {
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                *reinterpret_cast<float4*>(dst + j) = make_float4(v0[j], v0[j + 1], v0[j + 2], v0[j + 3]);
                *reinterpret_cast<float4*>(dst + 32 + j) = make_float4(v1[j], v1[j + 1], v1[j + 2], v1[j + 3]);
            }
        }
    }
    __syncthreads();
    if (tid < C) {
        const int s = tid;
        arow[s] = (s < p) ? __fmul_rn(bEps, row1[s]) : 0.f;
        prow[s] = (s <= p) ? __fmul_rn(Eps, __fmul_rn(a.scale, row2[s])) : 0.f;
    }
    // X tiles (R1 + 0 .. 32 KB, row p only) and the T row
    __syncthreads();
    if (tid < C) {  // T row p: T_pj = -(sum_{s=j}^{p-1} a_ps T_sj), ascending s (cached rows s < p)
        const int j = tid;
        const float* Tt = reinterpret_cast<const float*>(sm + S::Tt);
        float acc = 0.f;
        for (int s0 = 0; s0 < p; s0 += 16) {   // 16 rows' loads first, then their fma chain
            float tv[16], av[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {      // (rows >= p hold stale values, never selected)
                tv[e] = Tt[(s0 + e) * C + j];
                av[e] = arow[s0 + e];
            }
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int s = s0 + e;
                const float f = __fmaf_rn(av[e], tv[e], acc);
                if (s >= j && s < p) acc = f;
            }
        }
        const float tj = (j < p) ? -acc : (j == p ? 1.f : 0.f);
        trow[j] = tj;
        // X row p, entry j: T_pj (b_j Gamma_j) and T_pj b_j, split hi + lo
        const uint32_t off = cm_off(p, j, C);
        __nv_bfloat16 hi, lo;
        split_bf16(j <= p ? __fmul_rn(tj, bgs[j]) : 0.f, hi, lo);
        *reinterpret_cast<__nv_bfloat16*>(R1 + off) = hi;
        *reinterpret_cast<__nv_bfloat16*>(R1 + 8192 + off) = lo;
        split_bf16(j <= p ? __fmul_rn(tj, bets[j]) : 0.f, hi, lo);
        *reinterpret_cast<__nv_bfloat16*>(R1 + 16384 + off) = hi;
        *reinterpret_cast<__nv_bfloat16*>(R1 + 24576 + off) = lo;
    } else if (tid < C + C / 8) {  // P row p (R1 + 48 KB: hi, + 56 KB: lo), for P Delta
        const int s8 = tid - C;
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = prow[s8 * 8 + e];
        store8_split(R1 + 49152, R1 + 57344, cm_off(p, s8 * 8, C), x);
    }
    fence_async_smem();
    tc_sync();
    if (tid == kDecIssuer) {
        mma_tile_mj<64, D, C, false, true>(tmem, R1, sm + S::Kmn, false);
        mma_tile_mj<64, D, C, false, true>(tmem, R1 + 8192, sm + S::Kmn, true);
        mma_tile_mj<64, D, C, false, true>(tmem + 128, R1 + 16384, sm + S::Vt, false);
        mma_tile_mj<64, D, C, false, true>(tmem + 128, R1 + 24576, sm + S::Vt, true);
        mma_commit(mbar);
    }
    mma_out = true;
    if (!mma_wait()) { ok = false; break; }
    if (tid == kDecIssuer && has_next && p != C - 1) {  // K and V are consumed (a committing unit still
        fence_async_smem();                    // needs K): the next unit's tiles
        issue_KV(un, pn);
    }
    if (has_next && p != C - 1) pend_KV = true;
    if (warp == (p >> 4)) {   // M = 64: row p is lane p % 16 of lane quarter p / 16
        const bool mine = lane == (p & 15);
        float v[128];
        tmem_ld128(taddr_of(tmem, warp, 0), v);
        if (mine) store_row128(Wp, v);
        tmem_ld128(taddr_of(tmem, warp, D), v);
        if (mine) store_row128(Up, v);
    }
    // A4 tiles, M = 64 (R1: hi at +0, lo at +32 KB): row p = W'_p, row p ^ 32 = q_p
    __syncthreads();
    if (tid < 16) {  // q_p has no lo part: that row of the lo tile is zero, as in the prefill
        *reinterpret_cast<uint4*>(R1 + cm_off(p ^ 32, tid * 8, D)) = rowreg;
        *reinterpret_cast<uint4*>(R1 + 32768 + cm_off(p ^ 32, tid * 8, D)) = make_uint4(0u, 0u, 0u, 0u);
    } else if (tid < 32) {
        const int d8 = tid - 16;
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = Wp[d8 * 8 + e];
        store8_split(R1, R1 + 32768, cm_off(p, d8 * 8, D), x);
    }
    fence_async_smem();
    {
        // the state tiles and the Delta tiles have landed (row p is written below, and rows
        // past it only meet zero P entries)
        const bool wh = mbar_wait(bar_H, ph_H, a.err);
        const bool wd = mbar_wait(bar_D, ph_D, a.err);
        if (wh) {
            ph_H ^= 1u;
            pend_H = false;
        }
        if (wd) {
            ph_D ^= 1u;
            pend_D = false;
        }
        fence_before();
        if (__syncthreads_or(!(wh && wd))) { ok = false; break; }
        fence_after();
    }
    if (tid == kDecIssuer) {
        mma_tile_mj<64, D, D, false, true>(tmem, R1, sm + S::Hhi, false);
        mma_tile_mj<64, D, D, false, true>(tmem, R1, sm + S::Hlo, true);
        mma_tile_mj<64, D, D, false, true>(tmem, R1 + 32768, sm + S::Hhi, true);
        mma_commit(mbar);
    }
    mma_out = true;
    if (has_next) load_rows(un, pn);   // the next unit's token rows land while A4 runs
    if (!mma_wait()) { ok = false; break; }
    if (tid == kDecIssuer && has_next) {  // the state tiles are consumed: the next unit's
        fence_async_smem();
        issue_H(un);
    }
    if (has_next) pend_H = true;
    if (warp == (p >> 4) || warp == ((p ^ 32) >> 4)) {   // the lane quarters of rows p, p ^ 32
        float v[128];
        tmem_ld128(taddr_of(tmem, warp, 0), v);
        if (tid == lane_m64(p)) store_row128(row1, v);
        else if (tid == lane_m64(p ^ 32)) store_row128(row2, v);
    }
    __syncthreads();
    if (tid < D) {  // Delta row p, and its entry j in the Delta tiles, split hi + lo
        const int j = tid;
        const float dj = __fsub_rn(Up[j], row1[j]);
        Dp[j] = dj;
        Qs[j] = __fmul_rn(Gp, __fmul_rn(a.scale, row2[j]));
        __nv_bfloat16 hi, lo;
        split_bf16(dj, hi, lo);
        const uint32_t off = mn_off(j, p, D);
        *reinterpret_cast<__nv_bfloat16*>(sm + S::Dt + off) = hi;
        *reinterpret_cast<__nv_bfloat16*>(sm + S::Dt + 16384 + off) = lo;
    }
    fence_async_smem();
    tc_sync();
    if (tid == kDecIssuer) {
        mma_tile_mj<64, D, C, false, true>(tmem + 128, R1 + 49152, sm + S::Dt, false);
        mma_tile_mj<64, D, C, false, true>(tmem + 128, R1 + 49152, sm + S::Dt + 16384, true);
        mma_tile_mj<64, D, C, false, true>(tmem + 128, R1 + 57344, sm + S::Dt, true);
        mma_commit(mbar);
    }
    mma_out = true;
    if (tid < D / 8) {  // the cache's copy of Delta row p, while P Delta runs
        const int j8 = tid;
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = Dp[j8 * 8 + e];
        uint4 hi, lo;
        split8(x, hi, lo);
        const uint32_t off = mn_off(j8 * 8, p, D);
        *reinterpret_cast<uint4*>(cdt + off) = hi;
        *reinterpret_cast<uint4*>(cdt + 16384 + off) = lo;
    }
    if (!mma_wait()) { ok = false; break; }
    if (tid == kDecIssuer && has_next && p != C - 1) {  // the Delta tiles are consumed: the next unit's
        fence_async_smem();                    // (a committing unit stages its rows there first)
        issue_D(un, pn);
    }
    if (has_next && p != C - 1) pend_D = true;
    if (warp == (p >> 4)) {
        float v[128];
        tmem_ld128(taddr_of(tmem, warp, 128), v);
        if (lane == (p & 15)) store_row128(row1, v);
    }
    __syncthreads();
    if (tid < D) a.o[sh * D + tid] = __fadd_rn(Qs[tid], row1[tid]);
    {
        // append row p to the cache (k and v as rows of their operand tiles; a committing
        // step clears those tiles for the next chunk instead)
        if (p != C - 1) {
            if (tid >= 16 && tid < 32)
                *reinterpret_cast<uint4*>(reinterpret_cast<unsigned char*>(ck) + cm_off(p, (tid - 16) * 8, D)) = rowreg;
            else if (tid >= 32 && tid < 48)
                *reinterpret_cast<uint4*>(reinterpret_cast<unsigned char*>(cv) + cm_off(p, (tid - 32) * 8, D)) = rowreg;
        }
        if (tid < D) cd[(size_t)p * D + tid] = Dp[tid];
        if (tid < C) ct[p * C + tid] = trow[tid];
        if (tid == 0) {
            cg[p] = gams[p];
            cg[C + p] = gmls[p];
            cb[p] = bets[p];
        }
    }
    if (p == C - 1) {  // resynchronise: commit the next chunk-start state
        const int Lr = C - 1;
        if (tid == kDecIssuer) {  // the chunk's other fp32 Delta rows (the Delta tiles are consumed)
            fence_async_smem();
            mbar_expect_tx(bar_D, (uint32_t)p * D * 4);
            bulk_g2s(stage, cd, (uint32_t)p * D * 4, bar_D);
        }
        pend_D = true;
        if (tid < C) decs[tid] = simt::decay(gams[Lr], gmls[Lr], gams[tid], gmls[tid]);
        {
            const bool wd = mbar_wait(bar_D, ph_D, a.err);
            if (wd) {
                ph_D ^= 1u;
                pend_D = false;
            }
            if (__syncthreads_or(!wd)) { ok = false; break; }
        }
        if (tid < C) {
            const int s = tid;
            const float ds = decs[s];
#pragma unroll 4
            for (int jj = 0; jj < D / 8; ++jj) {
                const int j8 = (jj + s) & (D / 8 - 1);
                float x[8];
                if (s < p) {
                    const float4 x0 = *reinterpret_cast<const float4*>(stage + s * D + j8 * 8);
                    const float4 x1 = *reinterpret_cast<const float4*>(stage + s * D + j8 * 8 + 4);
                    x[0] = x0.x; x[1] = x0.y; x[2] = x0.z; x[3] = x0.w;
                    x[4] = x1.x; x[5] = x1.y; x[6] = x1.z; x[7] = x1.w;
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = Dp[j8 * 8 + e];
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = __fmul_rn(ds, x[e]);
                store8_split(R1 + 16384, R1 + 32768, mn_off(j8 * 8, s, D), x);
            }
        }
        fence_async_smem();
        tc_sync();
        if (tid == kDecIssuer) {
            mma_tile_mj<128, D, C, true, true>(tmem, sm + S::Kmn, R1 + 16384, false);
            mma_tile_mj<128, D, C, true, true>(tmem, sm + S::Kmn, R1 + 32768, true);
            mma_commit(mbar);
        }
        mma_out = true;
        if (!mma_wait()) { ok = false; break; }
        if (tid == kDecIssuer && has_next) {  // K and the staged rows are consumed: the next unit's
            fence_async_smem();      // K, V and Delta tiles
            issue_KV(un, pn);
            issue_D(un, pn);
        }
        if (has_next) pend_KV = pend_D = true;
        const float GL = simt::gate(gams[Lr], gmls[Lr]);
        float v[32];
        const int d = tid;
        for (int c0 = 0; c0 < D && tid < D; c0 += 32) {
            tmem_ld32(taddr_of(tmem, warp, c0), v);
#pragma unroll
            for (int j8 = 0; j8 < 4; ++j8) {
                float4* hp = reinterpret_cast<float4*>(Hst + (size_t)d * D + c0 + 8 * j8);
                const float4 h0 = hp[0], h1 = hp[1];
                const float hv[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = __fadd_rn(__fmul_rn(GL, hv[e]), v[8 * j8 + e]);
                hp[0] = make_float4(x[0], x[1], x[2], x[3]);
                hp[1] = make_float4(x[4], x[5], x[6], x[7]);
                // and the operand tiles the next steps load
                uint4 hi, lo;
                split8(x, hi, lo);
                const uint32_t off = mn_off(c0 + 8 * j8, d, D);
                *reinterpret_cast<uint4*>(cst + off) = hi;
                *reinterpret_cast<uint4*>(cst + 32768 + off) = lo;
            }
        }
        for (int i = tid; i < C * D / 8; i += kDecThreads) {  // the next chunk starts with no K, V, Delta rows
            reinterpret_cast<uint4*>(ck)[i] = make_uint4(0u, 0u, 0u, 0u);
            reinterpret_cast<uint4*>(cv)[i] = make_uint4(0u, 0u, 0u, 0u);
        }
        for (int i = tid; i < 32768 / 16; i += kDecThreads) reinterpret_cast<uint4*>(cdt)[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
    p = pn;
    take_rows();
    }  // units
    if (ok && warp == 0) {
        // every sequence advances one token per step: the last CTA to finish moves all the
        // positions on (warp 0, a sequence per lane).  Every CTA read the positions of its
        // units before its count, and the next step is a later launch.
        uint32_t prev = 0;
        if (lane == 0) prev = atomicAdd(&done[0], 1u);
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (prev == gridDim.x - 1) {
            for (int sq = lane; sq < a.n_seq; sq += 32) pos[sq] = (pos[sq] + 1) % C;
            __syncwarp();
            if (lane == 0) done[0] = 0u;
            __threadfence();
        }
    }
    if (!ok) {  // let this CTA's copies and MMAs in flight finish (bounded) before TMEM goes
        if (pend_KV) mbar_wait(bar_KV, ph_KV, a.err);
        if (pend_H) mbar_wait(bar_H, ph_H, a.err);
        if (pend_D) mbar_wait(bar_D, ph_D, a.err);
        if (mma_out) mbar_wait(mbar, ph_mma, a.err);
    }
    tc_sync();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

}  // namespace tc
}  // namespace cpr
