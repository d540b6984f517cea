// CPR Gated DeltaNet forward / prefill on the tensor cores: operand policy
// TC_BF16X3 (see cpr_gdn.h), bf16 io, d_k = d_v = 128, C = 64.
//
// Same chunk form as the SIMT kernels (page "IsoExec: 切换 SkyRL 中的训练器-
// 推理不匹配", section "Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet";
// the form is derived from the gated delta rule):
//   S1   = [K; Q] K^T                      (exact bf16 inputs, one MMA group)
//   gam  = in-chunk prefix of g (compensated pair, simt::gam_add)
//   a_rs = (b_r exp(gam_r - gam_s)) kk_rs       s < r
//   p_rs = exp(gam_r - gam_s) (scale qk_rs)     s <= r
//   T    = (I + A)^-1                       (fp32, T_rj = -sum_{s=j}^{r-1} a_rs T_sj, ascending s)
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
// async copies).  Token rows (k, v, a row of H or of Delta) feed MN-major
// operand tiles directly, so no kernel transposes anything.
#pragma once

#include "simt_fwd.cuh"
#include "tc_common.cuh"

namespace cpr {
namespace tc {

constexpr int D = 128;
constexpr int C = kChunk;

// Per (chunk, head) workspace block (bytes).
constexpr size_t kOffA4hi = 0;        // 128 x 128 bf16 K-major: rows 0..63 W'_hi, 64..127 Q
constexpr size_t kOffA4lo = 32768;    // 64 x 128 bf16 K-major: W'_lo
constexpr size_t kOffKmn = 49152;     // K as an MN-major 128 (d) x 64 (token) tile
constexpr size_t kOffPhi = 65536;     // 64 x 64 bf16 K-major
constexpr size_t kOffPlo = 73728;     // 64 x 64 bf16 K-major
constexpr size_t kOffU = 81920;       // 64 x 128 fp32, [split][DVS/4][64 rows] float4 groups
constexpr size_t kOffGam = 114688;    // gate prefix: 64 fp32 hi, then 64 fp32 lo
constexpr size_t kBlock = 115200;
// Training blocks (the backward) append, all as hi/lo bf16 tile pairs in the
// K-major core-matrix layout the backward kernels read with bulk copies:
constexpr size_t kOffT = kBlock;               // T, 64 x 64 (r, j): hi, lo (8 KB each)
constexpr size_t kOffHn = kOffT + 16384;       // chunk-start state H_n, 128 x 128 (d, j): hi, lo
constexpr size_t kOffDl = kOffHn + 65536;      // Delta, 64 x 128 (s, j): hi, lo
constexpr size_t kOffdH = kOffDl + 32768;      // dL/dH_{n+1}, 128 x 128 (d, j): hi, lo
constexpr size_t kOffdR = kOffdH + 65536;      // dL/dR, 64 x 128 (r, j): hi, lo
constexpr size_t kOffHdot = kOffdR + 32768;    // <dH', H_n> over each d_v split's columns (fp32 x 4)
constexpr size_t kOffBet = kOffHdot + 256;     // beta of the chunk's rows (fp32 x 64, 0 past the end)
constexpr size_t kOffdO = kOffBet + 256;       // dO, 64 x 128 (r, j): hi, lo (rows past the end 0)
constexpr size_t kBlockTrain = kOffdO + 32768;

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
    unsigned char* ws;    // [chunks * H] blocks of blk_bytes bytes
    size_t blk_bytes;     // kBlock (forward) or kBlockTrain (recompute for the backward)
    bool train;           // also write T, H_n and Delta tiles for the backward
    const float* h0;
    float* o;
    float* final_state;
    uint8_t* cache;
    CacheOff co;
    uint32_t* err;
    // Reading-B decode commit (null otherwise): the batch is one full chunk per sequence
    // (chunk b = sequence b), buffered in a decode cache; only the chunks of sequences
    // whose position `commit_pos[b]` is 0 after this step's token (the chunk is complete)
    // run, and only when the cache header carries the magic, version and these words
    // (contract digest, then n_seq, H, C, d_k, d_v, policy, io dtype, deployment digest).
    // The header is checked before anything else of the cache is read.
    const int32_t* commit_pos;
    const uint32_t* commit_header;
    uint32_t commit_words[8 + kHdrWords];
};

// True when a commit-mode CTA's cache header is not the one TcArgs names (nothing of the
// cache past its header may then be read).  Warp 0 compares a word per lane; the verdict
// reaches every thread of the CTA through shared memory (a CTA barrier inside).
__device__ __forceinline__ bool commit_header_bad(const TcArgs& a) {
    __shared__ int bad_s;
    if (threadIdx.x < 32) {
        const int i = threadIdx.x;
        bool ok = true;
        if (i == 0) ok = a.commit_header[0] == kCacheMagic;
        else if (i == 1) ok = a.commit_header[1] == CPR_CONTRACT_VERSION;
        else if (i < 2 + 8 + kHdrWords) ok = a.commit_header[i] == a.commit_words[i - 2];
        const bool all_ok = __all_sync(0xffffffffu, ok);
        if (i == 0) bad_s = all_ok ? 0 : 1;
    }
    __syncthreads();
    return bad_s != 0;
}

__device__ __forceinline__ uint4 ld16_or_zero(const __nv_bfloat16* p, bool valid) {
    return valid ? *reinterpret_cast<const uint4*>(p) : make_uint4(0u, 0u, 0u, 0u);
}

// T = (I + A)^-1 by the column wavefront: T_rj = -(sum_{s=j}^{r-1} a_rs T_sj), each
// row's sum one fma chain in ascending s (the chain a decode step evaluates for its own
// row).  Step t adds a_rt T_tj to every row r > t of column j.  Two threads per column
// (lanes 2j and 2j + 1) keep the running sums of the even and odd rows in registers; the
// owner of row t hands its final value to the partner with a shuffle.  At2 holds A
// transposed with the rows of each parity together, the odd half rotated by 16 so that
// the two halves' float4 groups fall in different banks:
// At2[s * 64 + at2_pos(r)] = a_rs.  Writes T rows < nrows of column j to Tout[r * ldT + j]
// (rows >= nrows get 0).  128 threads.
__device__ __forceinline__ int at2_pos(int r) { return (r & 1) * 32 + (((r >> 1) + (r & 1) * 16) & 31); }
__device__ __forceinline__ void t_solve_pairs(const float* At2, float* Tout, int ldT, int nrows) {
    const int j = threadIdx.x >> 1, p = threadIdx.x & 1;
    float acc[C / 2];
#pragma unroll
    for (int i = 0; i < C / 2; ++i) acc[i] = 0.f;
#pragma unroll
    for (int t = 0; t < C; ++t) {
        const float mine = -acc[t >> 1];
        const float other = __shfl_xor_sync(0xffffffffu, mine, 1);
        const float fin = ((t & 1) == p) ? mine : other;
        const float Tt = (t < j) ? 0.f : (t == j ? 1.f : fin);
        if ((t & 1) == p) Tout[t * ldT + j] = (t < nrows) ? Tt : 0.f;
        if (t >= j) {
            const float* arow = At2 + t * C + p * (C / 2);
#pragma unroll
            for (int i4 = t / 8; i4 < C / 8; ++i4) {   // i >= t / 2 - 1 covers every row > t
                const float4 a4 = *reinterpret_cast<const float4*>(arow + 4 * ((i4 + 4 * p) & 7));
                const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = 4 * i4 + e;
                    if (2 * i + 1 > t && 2 * i + p > t) acc[i] = __fmaf_rn(av[e], Tt, acc[i]);
                }
            }
        }
    }
}

// ---- prep: everything of a chunk that does not depend on H ------------------------
// Shared memory (65 KB, three CTAs per SM): [K; Q] K-major (32 KB; the K rows double
// as the MN-major d x token K tile, the two layouts being byte-identical), V MN-major
// (16 KB), the fp32 T buffer (E table, then T, then the X2 tiles), gate vectors.  A^T
// and then the X1 tiles take the Q rows' space once the S1 MMA has read it.  The 256
// TMEM columns are allocated once the copies are in flight: with three CTAs per SM
// the third one's allocation waits for another CTA to finish, but its loads do not.
// (W' and then U in the same 128 columns, so that all three hold theirs at once,
// measured slower: 224 -> 231 us on the Prefill workload.)
constexpr size_t kPrepOffVmn = 32768, kPrepOffT = 49152, kPrepOffVec = kPrepOffT + 64 * 65 * 4;
constexpr size_t kPrepSmem = kPrepOffVec + 4 * 64 * 4 + 64;

// PERSIST (the reading-B decode commit): a CTA walks the (chunk, head) units blockIdx.x,
// + gridDim.x, ... and runs only the chunks of sequences that completed one
// (TcArgs::commit_pos); otherwise a CTA runs chunk blockIdx.x of head blockIdx.y.
template <bool PERSIST>
__global__ void __launch_bounds__(128, 3) k_tc_prep(TcArgs a) {
    extern __shared__ __align__(1024) unsigned char sm[];
    unsigned char* tKQ = sm;                       // [K; Q] 128 x 128 K-major; Q rows later A^T, X1
    unsigned char* tKmn = sm;                      // the K rows read as an MN-major 128 (d) x 64 tile
    unsigned char* tVmn = sm + kPrepOffVmn;        // V, MN-major
    float* At = reinterpret_cast<float*>(sm + 16384);        // [64][64], a_rs at s * 64 + (r & 1) * 32 + r / 2
    float* Tfp = reinterpret_cast<float*>(sm + kPrepOffT);   // [64][65]
    float* gam = reinterpret_cast<float*>(sm + kPrepOffVec);   // gate prefix hi, then lo (gml)
    float* gml = gam + 64;
    float* bet = gml + 64;
    float* bg = bet + 64;
    uint64_t* mbar = reinterpret_cast<uint64_t*>(bg + 64);
    uint32_t* tbase = reinterpret_cast<uint32_t*>(mbar + 1);

    if (PERSIST && commit_header_bad(a)) return;
    const int total = a.chunk_off[a.n_seq];
    const int H = a.H;
    if (total < 0) return;
    const int nunits = PERSIST ? a.n_seq * H : 0;
    if (PERSIST) {   // most steps commit nothing: leave at once
        bool any = false;
        for (int u = blockIdx.x + (int)threadIdx.x * (int)gridDim.x; u < nunits; u += 128 * (int)gridDim.x)
            any = any || (u / H < total && a.commit_pos[u / H] == 0);
        if (!__syncthreads_or(any)) return;
    }
    __shared__ uint32_t act[4];   // PERSIST: which of a round of 128 units run, a bit each
    for (int unit = blockIdx.x, k = 0; PERSIST ? unit < nunits : unit == (int)blockIdx.x;
         unit += gridDim.x, ++k) {
    if (PERSIST) {   // commit batch: chunk b is sequence b
        if ((k & 127) == 0) {   // one thread looks up each position of the next round
            const int u = unit + (int)threadIdx.x * (int)gridDim.x;
            const bool on = u < nunits && u / H < total && a.commit_pos[u / H] == 0;
            const uint32_t m = __ballot_sync(0xffffffffu, on);
            __syncthreads();   // the previous round's bits are read
            if ((threadIdx.x & 31) == 0) act[threadIdx.x >> 5] = m;
            __syncthreads();
        }
        if (!((act[(k & 127) >> 5] >> (k & 31)) & 1u)) continue;
    }
    const int cidx = PERSIST ? unit / H : (int)blockIdx.x, h = PERSIST ? unit % H : (int)blockIdx.y;
    if (cidx >= total) break;
    const int b = find_seq(a.chunk_off, a.n_seq, cidx);
    const int n = cidx - a.chunk_off[b];
    const int seq0 = a.cu[b], T = a.cu[b + 1] - seq0;
    const int t0 = seq0 + n * C;
    const int nrows = min(C, T - n * C);
    const bool last = (n * C + nrows == T);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    unsigned char* blk = a.ws + ((size_t)cidx * H + h) * a.blk_bytes;

    if (tid == 0) {
        mbar_init(mbar, 1);
        mbar_init_fence();
    }
    // [K; Q] rows (K-major) and V token rows (MN-major): all copies in flight at
    // once, rows past the chunk's end zero-filled
    for (int i = tid; i < 64 * (D / 8); i += 128) {
        const int tr = i / (D / 8), d8 = i % (D / 8);
        const bool in = tr < nrows;
        const size_t src = in ? ((size_t)(t0 + tr) * H + h) * D + d8 * 8 : 0;
        cp_async16(tKQ + cm_off(tr, d8 * 8, D), a.k + src, in);
        cp_async16(tKQ + cm_off(64 + tr, d8 * 8, D), a.q + src, in);
        cp_async16(tVmn + mn_off(d8 * 8, tr, D), a.v + src, in);
    }
    if (tid < C) bet[tid] = (tid < nrows) ? a.beta[(size_t)(t0 + tid) * H + h] : 0.f;
    if (warp == 3) {  // gate prefix while the copies land: serial compensated sum in token order
        for (int r = lane; r < C; r += 32) {
            gam[r] = (r < nrows) ? a.g[(size_t)(t0 + r) * H + h] : 0.f;
            gml[r] = 0.f;
        }
        __syncwarp();
        if (lane == 0) {
            float hi = 0.f, lo = 0.f;
            for (int r = 0; r < nrows; ++r) {
                simt::gam_add(hi, lo, gam[r]);
                gam[r] = hi;
                gml[r] = lo;
            }
        }
    }
    if (warp == 0) {   // while the copies land
        if (PERSIST) tmem_alloc_keep(tbase, 256);
        else tmem_alloc(tbase, 256);
    }
    cp_async_wait_all();
    __syncthreads();
    fence_async_smem();
    tc_sync();
    const uint32_t tmem = *tbase;
    bool held = true;      // the TMEM columns, released before the last bulk stores
    int outstanding = 0;   // mbarrier phase an in-flight MMA group will complete, or -1
    if (tid == 0) {
        mma_tile<128, 64, D>(tmem, tKQ, tKQ, false);  // B = rows 0..63 of [K; Q] = K
        mma_commit(mbar);
        // Q rows and K go to the workspace as the later kernels' operand tiles
        bulk_s2g(blk + kOffA4hi + 16384, tKQ + 16384, 16384);
        bulk_s2g(blk + kOffKmn, tKmn, 16384);
        bulk_commit();
    }
    if (tid < C) bg[tid] = (tid < nrows) ? simt::bg_entry(bet[tid], gam[tid], gml[tid]) : 0.f;
    // E_rs = exp(gam_r - gam_s), s <= r, once per pair, spread evenly over the threads while
    // the S1 MMA runs (rows p and 63 - p together hold 65 entries), into the T buffer
    for (int i = tid; i < 32 * (C + 1); i += 128) {
        const int pr = i / (C + 1), k = i % (C + 1);
        const int r = (k <= pr) ? pr : C - 1 - pr, s_ = (k <= pr) ? k : k - pr - 1;
        Tfp[r * 65 + s_] = simt::decay(gam[r], gml[r], gam[s_], gml[s_]);
    }
    {
        const bool ok1 = mbar_wait(mbar, 0, a.err);
        fence_after();
        if (tid == 0) bulk_wait_read();  // the Q rows' space takes A^T next
        if (__syncthreads_or(!ok1)) goto done;
    }
    outstanding = -1;
    {
        // S1 epilogue: thread = TMEM lane = row (0..63: K rows -> A, 64..127: Q rows -> P)
        float v[32];
        const int r = tid & 63;
        for (int c0 = 0; c0 < C; c0 += 32) {
            tmem_ld32(taddr_of(tmem, warp, c0), v);
            if (tid < 64) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {   // a_rs = (b_r E_rs) kk_rs, as a_entry
                    const int s = c0 + j;
                    At[s * C + at2_pos(r)] =
                        (s < r && r < nrows) ? __fmul_rn(__fmul_rn(bet[r], Tfp[r * 65 + s]), v[j]) : 0.f;
                }
            } else {
#pragma unroll
                for (int j8 = 0; j8 < 4; ++j8) {
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int s = c0 + j8 * 8 + e;
                        x[e] = (s <= r && r < nrows)
                                   ? __fmul_rn(Tfp[r * 65 + s], __fmul_rn(a.scale, v[j8 * 8 + e]))
                                   : 0.f;
                    }
                    store8_split(blk + kOffPhi, blk + kOffPlo, cm_off(r, c0 + j8 * 8, C), x);
                }
            }
        }
    }
    __syncthreads();
    t_solve_pairs(At, Tfp, 65, nrows);
    __syncthreads();
    if (a.cache && last && nrows < C) {  // decode cache: T rows of the last, partial chunk
        float* ct = reinterpret_cast<float*>(a.cache + a.co.t_rows) + ((size_t)b * H + h) * C * C;
        for (int i = tid; i < nrows * C; i += 128) ct[i] = Tfp[(i / C) * 65 + (i % C)];
    }
    {
        // X1 = T diag(b G) (threads 0..63, into the Q rows' space), X2 = T diag(b)
        // (threads 64..127, over the T buffer once every row of T is in registers), split
        const int r = tid & 63, which = tid >> 6;
        float trow[C];
#pragma unroll
        for (int s = 0; s < C; ++s) trow[s] = Tfp[r * 65 + s];
        __syncthreads();
        unsigned char* xhi = which ? reinterpret_cast<unsigned char*>(Tfp) : tKQ + 16384;
        unsigned char* xlo = xhi + 8192;
        const float* sc = which ? bet : bg;
#pragma unroll
        for (int s8 = 0; s8 < C / 8; ++s8) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = __fmul_rn(trow[s8 * 8 + e], sc[s8 * 8 + e]);
            store8_split(xhi, xlo, cm_off(r, s8 * 8, C), x);
        }
        if (a.train && which == 0) {  // T itself, for dR = T^T dDelta in the backward
#pragma unroll
            for (int s8 = 0; s8 < C / 8; ++s8) {
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = trow[s8 * 8 + e];
                store8_split(blk + kOffT, blk + kOffT + 8192, cm_off(r, s8 * 8, C), x);
            }
        }
    }
    if (a.cache && last && nrows < C) {  // decode cache: the other rows of the last, partial chunk
        const size_t sh = (size_t)b * H + h;
        __nv_bfloat16* ck = reinterpret_cast<__nv_bfloat16*>(a.cache + a.co.k_rows) + sh * C * D;
        __nv_bfloat16* cv = reinterpret_cast<__nv_bfloat16*>(a.cache + a.co.v_rows) + sh * C * D;
        float* cg = reinterpret_cast<float*>(a.cache + a.co.gam_rows) + sh * 2 * C;   // hi | lo
        float* cb = reinterpret_cast<float*>(a.cache + a.co.beta_rows) + sh * C;
        for (int i = tid; i < nrows * (D / 8); i += 128) {  // as rows of the decode's operand tiles
            const int r = i / (D / 8), d8 = i % (D / 8);
            const size_t src = ((size_t)(t0 + r) * H + h) * D + d8 * 8;
            const uint32_t off = cm_off(r, d8 * 8, D);
            *reinterpret_cast<uint4*>(reinterpret_cast<unsigned char*>(ck) + off) =
                *reinterpret_cast<const uint4*>(a.k + src);
            *reinterpret_cast<uint4*>(reinterpret_cast<unsigned char*>(cv) + off) =
                *reinterpret_cast<const uint4*>(a.v + src);
        }
        if (tid < nrows) {
            cg[tid] = gam[tid];
            cg[C + tid] = gml[tid];
            cb[tid] = bet[tid];
        }
    }
    fence_async_smem();
    tc_sync();
    if (tid == 0) {
        unsigned char* x2 = reinterpret_cast<unsigned char*>(Tfp);
        mma_tile_mj<64, D, C, false, true>(tmem, tKQ + 16384, tKmn, false);        // W' = X1_hi K
        mma_tile_mj<64, D, C, false, true>(tmem, tKQ + 24576, tKmn, true);         //    + X1_lo K
        mma_tile_mj<64, D, C, false, true>(tmem + 128, x2, tVmn, false);           // U  = X2_hi V
        mma_tile_mj<64, D, C, false, true>(tmem + 128, x2 + 8192, tVmn, true);     //    + X2_lo V
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
        // W' and U rows (M = 64 layout, row r = 16 * warp + lane for lanes < 16) are
        // staged in the now free operand space in their workspace layouts, then
        // bulk-stored: W' hi, lo over the [K; Q] tile, U over the V tile and the T buffer
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
                    store8_split(tKQ, tKQ + 16384, cm_off(r, c0 + j8 * 8, D), x);
                }
            }
        }
        float* U = reinterpret_cast<float*>(tVmn);
        const int dvs = a.dvs, dsh = __ffs(dvs) - 1;   // dvs is a power of two
        for (int c0 = 0; c0 < D; c0 += 32) {
            tmem_ld32(taddr_of(tmem, warp, 128 + c0), v);
            if (lane < 16) {
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    const int j = c0 + j4 * 4;
                    const int sp = j >> dsh, jl = j & (dvs - 1);
                    *reinterpret_cast<float4*>(U + (((size_t)sp * (dvs / 4) + jl / 4) * 64 + r) * 4) =
                        make_float4(v[j4 * 4], v[j4 * 4 + 1], v[j4 * 4 + 2], v[j4 * 4 + 3]);
                }
            }
        }
        fence_async_smem();
        tc_sync();
        if (warp == 0) tmem_dealloc(tmem, 256);
        held = false;
        if (tid == 0) {
            bulk_s2g(blk + kOffA4hi, tKQ, 16384);
            bulk_s2g(blk + kOffA4lo, tKQ + 16384, 16384);
            bulk_s2g(blk + kOffU, tVmn, 32768);
            bulk_s2g(blk + kOffGam, gam, 512);
            bulk_commit();
        }
    }
done:
    if (outstanding >= 0) mbar_wait(mbar, (uint32_t)outstanding, a.err);  // bounded
    if (tid == 0) bulk_wait_read();  // shared memory stays until the bulk stores have read it
    tc_sync();
    if (warp == 0 && held) tmem_dealloc(tmem, 256);
    }  // units
}

// OR over the predicates of `count` threads meeting at hardware barrier `id` (a
// __syncthreads_or for a subset of the CTA's warps).
__device__ __forceinline__ bool bar_or(int id, int count, bool pred) {
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
                 "barrier.cta.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r) : "r"((uint32_t)pred), "r"(id), "r"(count) : "memory");
    return r != 0;
}

// ---- state pass: one CTA per (sequence, head, d_v split), chunks in order -----------
// 288 threads: warps 0..7 do the operand and epilogue work (warp w reads TMEM lane
// quarter w % 4; the two warps of a quarter take one half of the DVS columns each);
// warp 8 only issues the MMA groups, so that issuing (about 56 cycles an instruction
// at N = 64) and epilogue work do not queue behind each other on one warp.  Barriers:
// three CTA-wide ones per chunk (chunk start, Delta tiles written, and the next chunk's
// start), the others only among warps 0..7 (hardware barrier 1).  Per chunk the dependent chain is
// A4 MMA -> Delta epilogue -> H' MMA -> H' epilogue; the output rows of chunk n
// (P Delta and the Q H rows) are read while chunk n + 1's A4 MMA runs, from
// double-buffered accumulators.
template <int DVS>
struct StateSmem {
    static constexpr size_t A4hi = 0, A4lo = 32768, Kmn = 65536, Phi = 81920, Plo = 90112;
    static constexpr size_t U = 98304;                       // 64 x DVS fp32, [DVS/4][64] float4
    static constexpr size_t Hhi = U + 64 * DVS * 4;          // H as MN-major DVS (j) x 128 (d)
    static constexpr size_t Hlo = Hhi + DVS * 128 * 2;
    static constexpr size_t Dhi = Hlo + DVS * 128 * 2;       // Delta, MN-major DVS (j) x 64 (token)
    static constexpr size_t Dlo = Dhi + DVS * 64 * 2;
    static constexpr size_t Bhi = Dlo + DVS * 64 * 2;        // decay * Delta, same layout
    static constexpr size_t Blo = Bhi + DVS * 64 * 2;
    static constexpr size_t Q = Blo + DVS * 64 * 2;          // 64 x DVS fp32, [DVS/4][64] float4
    static constexpr size_t Gam = Q + 64 * DVS * 4;          // 64 fp32 hi, 64 lo (bulk copied)
    static constexpr size_t Gm = Gam + 512, Dec = Gm + 256;
    static constexpr size_t Ost = Dec + 256;                 // output rows, 64 x (DVS + 4) fp32
    static constexpr size_t Bar = Ost + 64 * (DVS + 4) * 4;  // 5 mbarriers + TMEM base
    static constexpr size_t Total = Bar + 64;
    static constexpr uint32_t LoadA = 32768 + 16384 + 512;   // A4 tiles + gam
    static constexpr uint32_t LoadB = 16384 + 64 * DVS * 4;  // K, U
    static constexpr uint32_t LoadP = 16384;                 // P hi, lo
    static constexpr uint32_t TmemCols = 5 * DVS > 256 ? 512 : 256;
};

constexpr int kStateThreads = 288, kStateIssuer = 256;

// PERSIST (the reading-B decode commit): a CTA walks the units blockIdx.x, + gridDim.x,
// ... and runs only those whose sequence completed a chunk (TcArgs::commit_pos); TMEM,
// the mbarriers and their phases carry over from unit to unit.  Otherwise a CTA runs
// unit blockIdx.x, the (sequence, head, d_v split) it is launched for.
template <int DVS, bool PERSIST>
__global__ void __launch_bounds__(kStateThreads, 1) k_tc_state(TcArgs a) {
    using L = StateSmem<DVS>;
    constexpr int NSPLIT = D / DVS;
    constexpr int HALF = DVS / 2;  // columns per thread
    extern __shared__ __align__(1024) unsigned char sm[];
    float* sU = reinterpret_cast<float*>(sm + L::U);
    float* sQ = reinterpret_cast<float*>(sm + L::Q);
    float* gam = reinterpret_cast<float*>(sm + L::Gam);   // gate prefix hi, then lo
    float* gml = gam + 64;
    float* Gm = reinterpret_cast<float*>(sm + L::Gm);
    float* dec = reinterpret_cast<float*>(sm + L::Dec);
    uint64_t* bar_mma = reinterpret_cast<uint64_t*>(sm + L::Bar);   // A4 and H' groups
    uint64_t* bar_pd = bar_mma + 1;                                   // P Delta groups
    uint64_t* bar_ldA = bar_mma + 2;
    uint64_t* bar_ldB = bar_mma + 3;
    uint64_t* bar_ldP = bar_mma + 4;
    uint32_t* tbase = reinterpret_cast<uint32_t*>(bar_mma + 5);

    if (PERSIST && commit_header_bad(a)) return;
    const int total = a.chunk_off[a.n_seq];
    if (total < 0) return;
    const int H = a.H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool epi = warp < 8;                  // warp 8 issues the MMAs
    const int quarter = warp & 3, half = (warp >> 2) & 1;
    const int cb = half * HALF;                 // this thread's first column (within the split)
    const int d = quarter * 32 + lane;          // this thread's state row
    if (PERSIST) {   // most steps commit nothing: leave before taking TMEM
        bool any = false;
        for (int u = blockIdx.x + tid * (int)gridDim.x; u < a.n_seq * H * NSPLIT; u += kStateThreads * (int)gridDim.x)
            any = any || a.commit_pos[u / (NSPLIT * H)] == 0;
        if (!__syncthreads_or(any)) return;
    }

    if (warp == 0) tmem_alloc(tbase, L::TmemCols);
    if (tid == 0) {
        for (int i = 0; i < 5; ++i) mbar_init(bar_mma + i, 1);
        mbar_init_fence();
    }
    for (int i = tid; i < 1024; i += kStateThreads)  // rows 64..127 of the W'_lo operand stay zero
        reinterpret_cast<uint4*>(sm + L::A4lo + 16384)[i] = make_uint4(0u, 0u, 0u, 0u);
    uint32_t ph_mma = 0, ph_pd = 0, ph_ldA = 0, ph_ldB = 0, ph_ldP = 0;
    bool pendA = false, pendB = false, pendP = false, failed = false, mma_out = false, pd_out = false;
    // the issuing thread's operand descriptors (k-step 0), once: its tiles never move
    const uint64_t dA4hi = tile_desc<128, D, false>(sm + L::A4hi), dA4lo = tile_desc<128, D, false>(sm + L::A4lo);
    const uint64_t dHhi = tile_desc<DVS, D, true>(sm + L::Hhi), dHlo = tile_desc<DVS, D, true>(sm + L::Hlo);
    const uint64_t dKmn = tile_desc<128, C, true>(sm + L::Kmn);
    const uint64_t dBhi = tile_desc<DVS, C, true>(sm + L::Bhi), dBlo = tile_desc<DVS, C, true>(sm + L::Blo);
    const uint64_t dPhi = tile_desc<64, C, false>(sm + L::Phi), dPlo = tile_desc<64, C, false>(sm + L::Plo);
    const uint64_t dDhi = tile_desc<DVS, C, true>(sm + L::Dhi), dDlo = tile_desc<DVS, C, true>(sm + L::Dlo);
    auto run_unit = [&](int unit) {
    const int b = unit / (NSPLIT * H);
    const int sp = unit % NSPLIT;
    const int h = (unit / NSPLIT) % H;
    const int j0 = sp * DVS;
    const int seq0 = a.cu[b], T = a.cu[b + 1] - seq0;
    const int nch = a.chunk_off[b + 1] - a.chunk_off[b];
    const size_t sh = (size_t)b * H + h;
    float* cstate = a.cache ? reinterpret_cast<float*>(a.cache + a.co.state) + sh * D * D : nullptr;

    // state row d = 32 quarter + lane, columns j0 + cb .. + HALF, fp32 in registers
    float Hreg[HALF];
#pragma unroll
    for (int j4 = 0; j4 < HALF / 4; ++j4) {
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (a.h0 && epi) x = *reinterpret_cast<const float4*>(a.h0 + (sh * D + d) * D + j0 + cb + 4 * j4);
        Hreg[4 * j4] = x.x; Hreg[4 * j4 + 1] = x.y; Hreg[4 * j4 + 2] = x.z; Hreg[4 * j4 + 3] = x.w;
    }
    const int coff = a.chunk_off[b];
    auto blk_of = [&](int n) { return a.ws + ((size_t)(coff + n) * H + h) * a.blk_bytes; };
    // H as the B operand of the next chunk; for training also chunk nn's start
    // state as K-major (d, j) hi/lo tiles in its workspace block
    auto put_h = [&](int nn) {
        unsigned char* g = (a.train && nn < nch) ? blk_of(nn) + kOffHn : nullptr;
#pragma unroll
        for (int j8 = 0; j8 < HALF / 8; ++j8) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = Hreg[j8 * 8 + e];
            uint4 hi, lo;
            split8(x, hi, lo);
            const int jj = cb + j8 * 8;
            *reinterpret_cast<uint4*>(sm + L::Hhi + mn_off(jj, d, DVS)) = hi;
            *reinterpret_cast<uint4*>(sm + L::Hlo + mn_off(jj, d, DVS)) = lo;
            if (g) {
                *reinterpret_cast<uint4*>(g + cm_off(d, j0 + jj, D)) = hi;
                *reinterpret_cast<uint4*>(g + 32768 + cm_off(d, j0 + jj, D)) = lo;
            }
        }
    };
    auto put_state = [&](float* dst) {
#pragma unroll
        for (int j4 = 0; j4 < HALF / 4; ++j4)
            *reinterpret_cast<float4*>(dst + (size_t)d * D + j0 + cb + 4 * j4) =
                make_float4(Hreg[4 * j4], Hreg[4 * j4 + 1], Hreg[4 * j4 + 2], Hreg[4 * j4 + 3]);
    };
    if (epi) {
        put_h(0);
        if (nch == 0 && cstate) put_state(cstate);
    }
    fence_async_smem();
    tc_sync();
    const uint32_t tmem = *tbase;
    auto acc4 = [&](int n) { return tmem + (uint32_t)((n & 1) * DVS); };
    auto acc5 = [&](int n) { return tmem + (uint32_t)((2 + (n & 1)) * DVS); };
    const uint32_t acc6 = tmem + 4 * DVS;

    auto issue_A = [&](int n) {
        const unsigned char* blk = blk_of(n);
        mbar_expect_tx(bar_ldA, L::LoadA);
        bulk_g2s(sm + L::A4hi, blk + kOffA4hi, 32768, bar_ldA);
        bulk_g2s(sm + L::A4lo, blk + kOffA4lo, 16384, bar_ldA);
        bulk_g2s(sm + L::Gam, blk + kOffGam, 512, bar_ldA);
    };
    auto issue_B = [&](int n) {
        const unsigned char* blk = blk_of(n);
        mbar_expect_tx(bar_ldB, L::LoadB);
        bulk_g2s(sm + L::Kmn, blk + kOffKmn, 16384, bar_ldB);
        bulk_g2s(sm + L::U, blk + kOffU + (size_t)sp * 64 * DVS * 4, 64 * DVS * 4, bar_ldB);
    };
    auto issue_P = [&](int n) {
        mbar_expect_tx(bar_ldP, L::LoadP);
        bulk_g2s(sm + L::Phi, blk_of(n) + kOffPhi, 16384, bar_ldP);
    };
    // output rows of chunk m: o_r = G_r (scale qh_r) + (P Delta)_r, staged in Ost (rows
    // padded to DVS + 4 floats: conflict-free writes).  o_copy (the 128 threads of lane
    // quarters 2 and 3, idle while the Delta epilogue runs) stores them, whole rows per
    // warp instruction.
    float* ost = reinterpret_cast<float*>(sm + L::Ost);
    auto o_copy = [&](int m) {
        if (!a.o) return;
        constexpr int R4 = DVS / 4;   // float4 per row
        const int t0 = seq0 + m * C, nrows = min(C, T - m * C);
        const int lt = ((warp & 3) - 2) * 64 + (warp >> 2) * 32 + lane;  // 0..127 over warps 2, 3, 6, 7
#pragma unroll
        for (int i = 0; i < 64 * R4 / 128; ++i) {
            const int idx = i * 128 + lt, r = idx / R4, c4 = idx % R4;
            if (r < nrows)
                *reinterpret_cast<float4*>(a.o + ((size_t)(t0 + r) * H + h) * D + j0 + 4 * c4) =
                    *reinterpret_cast<const float4*>(ost + r * (DVS + 4) + 4 * c4);
        }
    };
    // chunk n's Q H rows (accumulator rows 64..127, lane quarters 2 and 3) -> sQ, scaled
    // by G_r: taken while quarters 0 and 1 run the Delta epilogue
    auto qh_to_sq = [&](int n) {
        float v[32];
        tmem_ld32(taddr_of(acc4(n), warp, cb), v);
        const int rr = d - 64;
        const float gr = Gm[rr];
#pragma unroll
        for (int j4 = 0; j4 < HALF / 4; ++j4)
            reinterpret_cast<float4*>(sQ)[(cb / 4 + j4) * 64 + rr] =
                make_float4(__fmul_rn(gr, __fmul_rn(a.scale, v[4 * j4])),
                            __fmul_rn(gr, __fmul_rn(a.scale, v[4 * j4 + 1])),
                            __fmul_rn(gr, __fmul_rn(a.scale, v[4 * j4 + 2])),
                            __fmul_rn(gr, __fmul_rn(a.scale, v[4 * j4 + 3])));
    };
    // (each thread waits for P Delta itself; a failed wait reaches the other threads at the
    // next barrier)
    auto o_epilogue = [&](int m) -> bool {
        const bool w = mbar_wait(bar_pd, ph_pd, a.err);
        fence_after();
        if (!w) return false;
        ph_pd ^= 1u;
        pd_out = false;
        if (tid == 0 && m + 1 < nch) {  // P of chunk m is consumed
            fence_async_smem();
            issue_P(m + 1);
        }
        pendP = (m + 1 < nch);
        const int nrows = min(C, T - m * C);
        float v[32];
        tmem_ld32(taddr_of(acc5(m), warp, cb), v);  // M = 64: row 16 quarter + lane, lanes < 16
        const int r = quarter * 16 + lane;
        if (lane < 16 && r < nrows && a.o) {
            float* orow = ost + r * (DVS + 4) + cb;
#pragma unroll
            for (int j4 = 0; j4 < HALF / 4; ++j4) {
                const float4 q4 = reinterpret_cast<const float4*>(sQ)[(cb / 4 + j4) * 64 + r];
                *reinterpret_cast<float4*>(orow + 4 * j4) =
                    make_float4(__fadd_rn(q4.x, v[4 * j4]), __fadd_rn(q4.y, v[4 * j4 + 1]),
                                __fadd_rn(q4.z, v[4 * j4 + 2]), __fadd_rn(q4.w, v[4 * j4 + 3]));
            }
        }
        return true;
    };
    if (nch > 0) {
        if (tid == 0) {
            issue_A(0);
            issue_B(0);
            issue_P(0);
        }
        pendA = pendB = pendP = true;
    }

    bool carry = true;   // the previous H' epilogue's consensus among warps 0..7
    for (int n = 0; n < nch; ++n) {
        const int nrows = min(C, T - n * C);
        const int Lr = nrows - 1;
        const bool last = (n == nch - 1);
        // [all] the A4 tiles have landed; the H tiles put_h wrote are visible
        bool ok = mbar_wait(bar_ldA, ph_ldA, a.err);
        fence_before();
        if (__syncthreads_or(!(ok && carry))) { failed = true; break; }
        fence_after();
        ph_ldA ^= 1u;
        pendA = false;
        bool okg = true;   // this phase's consensus among warps 0..7
        float GL = 0.f;    // G_L, read before issue_A(n + 1) replaces gam
        if (tid == kStateIssuer) {
            mma_tile_d<128, DVS, D, false, true>(acc4(n), dA4hi, dHhi, false);
            mma_tile_d<128, DVS, D, false, true>(acc4(n), dA4hi, dHlo, true);
            mma_tile_d<128, DVS, D, false, true>(acc4(n), dA4lo, dHhi, true);
            mma_commit(bar_mma);
        }
        mma_out = true;
        ok = mbar_wait(bar_ldB, ph_ldB, a.err);   // K and U (every thread tracks the phase)
        if (ok) {
            ph_ldB ^= 1u;
            pendB = false;
        }
        if (epi) {
            const bool okpd = n == 0 || o_epilogue(n - 1);
            if (tid < C) {
                Gm[tid] = (tid < nrows) ? simt::gate(gam[tid], gml[tid]) : 0.f;
                dec[tid] = (tid < nrows) ? simt::decay(gam[Lr], gml[Lr], gam[tid], gml[tid]) : 0.f;
            }
            GL = simt::gate(gam[Lr], gml[Lr]);
            okg = !bar_or(1, 256, !(ok && okpd));
            if (okg) {
                ok = mbar_wait(bar_mma, ph_mma, a.err);
                fence_after();
                okg = !bar_or(1, 256, !ok);
            }
            if (okg) {
                ph_mma ^= 1u;
                mma_out = false;
                if (tid == 0 && n + 1 < nch) {  // the A4 operand tiles and gam of chunk n are consumed
                    fence_async_smem();
                    issue_A(n + 1);
                }
                pendA = (n + 1 < nch);
                if (quarter < 2) {
                    // rows 0..63: Delta = U - W'H, columns cb .. cb + HALF
                    const int r = d;
                    float v[32];
                    tmem_ld32(taddr_of(acc4(n), warp, cb), v);
                    const bool in = r < nrows;
                    float* cd = (a.cache && last && nrows < C && in)
                                    ? reinterpret_cast<float*>(a.cache + a.co.delta_rows) + (sh * C + r) * D + j0 + cb
                                    : nullptr;
                    const float dr = dec[r];
#pragma unroll
                    for (int j8 = 0; j8 < HALF / 8; ++j8) {
                        float x[8], y[8];
                        const int jj = cb + j8 * 8;
                        const float4 u0 = reinterpret_cast<const float4*>(sU)[(jj / 4) * 64 + r];
                        const float4 u1 = reinterpret_cast<const float4*>(sU)[(jj / 4 + 1) * 64 + r];
                        const float uu[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            x[e] = in ? __fsub_rn(uu[e], v[j8 * 8 + e]) : 0.f;
                            y[e] = __fmul_rn(dr, x[e]);
                        }
                        uint4 hi, lo;
                        split8(x, hi, lo);
                        *reinterpret_cast<uint4*>(sm + L::Dhi + mn_off(jj, r, DVS)) = hi;
                        *reinterpret_cast<uint4*>(sm + L::Dlo + mn_off(jj, r, DVS)) = lo;
                        if (a.train) {  // Delta rows for the backward, K-major (s, j)
                            unsigned char* g = blk_of(n) + kOffDl + cm_off(r, j0 + jj, D);
                            *reinterpret_cast<uint4*>(g) = hi;
                            *reinterpret_cast<uint4*>(g + 16384) = lo;
                        }
                        store8_split(sm + L::Bhi, sm + L::Blo, mn_off(jj, r, DVS), y);
                        if (cd) {
                            *reinterpret_cast<float4*>(cd + j8 * 8) = make_float4(x[0], x[1], x[2], x[3]);
                            *reinterpret_cast<float4*>(cd + j8 * 8 + 4) = make_float4(x[4], x[5], x[6], x[7]);
                        }
                    }
                } else {
                    if (n > 0) o_copy(n - 1);   // staged by o_epilogue(n - 1), barriers ago
                    qh_to_sq(n);
                }
                if (cstate && last && nrows < C) put_state(cstate);
            }
        } else {
            okg = ok;
        }
        // [all] the Delta tiles are written and the P tiles have landed
        fence_async_smem();
        ok = okg && mbar_wait(bar_ldP, ph_ldP, a.err);
        fence_before();
        if (__syncthreads_or(!ok)) { failed = true; break; }
        fence_after();
        ph_ldP ^= 1u;
        pendP = false;
        if (tid == kStateIssuer) {
            mma_tile_d<128, DVS, C, true, true>(acc6, dKmn, dBhi, false);   // H' part
            mma_tile_d<128, DVS, C, true, true>(acc6, dKmn, dBlo, true);
            mma_commit(bar_mma);
            mma_tile_d<64, DVS, C, false, true>(acc5(n), dPhi, dDhi, false);  // P Delta
            mma_tile_d<64, DVS, C, false, true>(acc5(n), dPhi, dDlo, true);
            mma_tile_d<64, DVS, C, false, true>(acc5(n), dPlo, dDhi, true);
            mma_commit(bar_pd);
        }
        mma_out = true;
        pd_out = true;
        carry = true;
        if (epi) {
            ok = mbar_wait(bar_mma, ph_mma, a.err);
            fence_after();
            carry = !bar_or(1, 256, !ok);
            if (carry) {
                ph_mma ^= 1u;
                mma_out = false;
                if (tid == 0 && n + 1 < nch) {  // K and U of chunk n are consumed
                    fence_async_smem();
                    issue_B(n + 1);
                }
                pendB = (n + 1 < nch);
                {
                    // H' = G_L H + K^T (dec . Delta): row d, columns cb .. cb + HALF
                    float v[32];
                    tmem_ld32(taddr_of(acc6, warp, cb), v);
#pragma unroll
                    for (int j = 0; j < HALF; ++j) Hreg[j] = __fadd_rn(__fmul_rn(GL, Hreg[j]), v[j]);
                    put_h(n + 1);
                    if (cstate && last && nrows == C) put_state(cstate);
                }
            }
        }
        fence_async_smem();
    }
    if (!failed && nch > 0) {   // (failed is the same in every thread here)
        const bool okl = !epi || o_epilogue(nch - 1);
        if (__syncthreads_or(!(okl && carry))) failed = true;
        else if (epi && quarter >= 2) o_copy(nch - 1);
    }
    if (!failed && a.final_state && epi) put_state(a.final_state + sh * D * D);
    };  // run_unit
    if (PERSIST) {
        // rounds of kStateThreads units of this CTA: one thread looks up each unit's
        // position, a bit per unit says which run
        __shared__ uint32_t act[kStateThreads / 32];
        const int nunits = a.n_seq * H * NSPLIT;
        for (int r0 = blockIdx.x; r0 < nunits && !failed; r0 += kStateThreads * gridDim.x) {
            const int u = r0 + tid * (int)gridDim.x;
            const bool on = u < nunits && a.commit_pos[u / (NSPLIT * H)] == 0;
            const uint32_t m = __ballot_sync(0xffffffffu, on);
            if (lane == 0) act[warp] = m;
            __syncthreads();
            for (int t = 0; t < kStateThreads && !failed; ++t)
                if ((act[t >> 5] >> (t & 31)) & 1u) run_unit(r0 + t * (int)gridDim.x);
            __syncthreads();   // act is rewritten for the next round
        }
    } else {
        run_unit(blockIdx.x);
    }
    if (failed && epi) {
        // let in-flight copies and MMAs finish (bounded) before TMEM is released
        if (pendA) mbar_wait(bar_ldA, ph_ldA, a.err);
        if (pendB) mbar_wait(bar_ldB, ph_ldB, a.err);
        if (pendP) mbar_wait(bar_ldP, ph_ldP, a.err);
        if (mma_out) mbar_wait(bar_mma, ph_mma, a.err);
        if (pd_out) mbar_wait(bar_pd, ph_pd, a.err);
    }
    tc_sync();
    if (warp == 0) tmem_dealloc(*tbase, L::TmemCols);
}

}  // namespace tc
}  // namespace cpr
