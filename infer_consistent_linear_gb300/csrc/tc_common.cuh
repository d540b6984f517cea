// sm_103a tensor-core building blocks (inline PTX): TMEM allocation, tcgen05.mma
// (kind::f16, bf16 operands, fp32 accumulation), commit to mbarrier, TMEM loads,
// bulk async copies, and the shared-memory operand layout they use.
//
// Operand layout ("core-matrix K-major, no swizzle"): an R x K bf16 tile is a
// grid of 8-row x 8-element (8 x 16 B) core matrices stored row-group-major:
// core matrix (rg, kg) at byte ((rg * K/8) + kg) * 128, row i of it at +16 i.
// In the shared-memory descriptor the leading byte offset (LBO) is the stride
// between core matrices adjacent along K (128 B) and the stride byte offset
// (SBO) the stride between 8-row groups (K/8 * 128 B).  One MMA instruction
// consumes K = 16 (two core matrices along K); the next k-step starts 256 B
// further.  Accumulator rows: M = 128 -> TMEM lane r; M = 64 -> lane
// (r / 16) * 32 + r % 16 (16 rows in each warp's lane quarter).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "common.cuh"

namespace cpr {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// Byte offset of element (r, k) in an R x K core-matrix K-major bf16 tile.
__host__ __device__ __forceinline__ uint32_t cm_off(int r, int k, int K) {
    return (uint32_t)((((r >> 3) * (K >> 3)) + (k >> 3)) * 128 + (r & 7) * 16 + (k & 7) * 2);
}

// TMEM lane holding accumulator row r for an M = 64 MMA.
__device__ __forceinline__ int lane_m64(int r) { return ((r >> 4) << 5) + (r & 15); }

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, int K) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((128u >> 4) & 0x3FFFu) << 16;                  // LBO: along K
    d |= (uint64_t)((((uint32_t)K >> 3) * 128u >> 4) & 0x3FFFu) << 32;  // SBO: along M/N
    d |= (uint64_t)1 << 46;                                          // descriptor version
    return d;
}

// kind::f16 instruction descriptor: D f32, A and B bf16, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ---- TMEM --------------------------------------------------------------------
// Whole-warp operations.
// The CTA's only allocation (it gives up the permit to allocate again); blocks until
// the columns are free.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(dst_smem)), "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
// As tmem_alloc, keeping the permit: for a CTA that allocates once per work unit.
__device__ __forceinline__ void tmem_alloc_keep(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(dst_smem)), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Makes this thread's generic-proxy shared-memory writes visible to the async
// proxy (tensor core, bulk copies).
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// CTA barrier that also orders tcgen05 operations around it.
__device__ __forceinline__ void tc_sync() {
    fence_before();
    __syncthreads();
    fence_after();
}

// ---- MMA -----------------------------------------------------------------------
// D[tmem] (+)= A[smem] * B[smem]^T over K = 16 (one instruction).
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// Issues the k-steps of A (M x K) * B (N x K)^T into d_tmem in ascending K
// order; accumulates onto the existing D when `accumulate` is set.
template <int M, int N, int K>
__device__ __forceinline__ void mma_tile(uint32_t d_tmem, const void* a_tile, const void* b_tile,
                                         bool accumulate) {
    constexpr uint32_t idesc = idesc_bf16(M, N);
    const uint32_t a0 = smem_u32(a_tile), b0 = smem_u32(b_tile);
#pragma unroll
    for (int ks = 0; ks < K / 16; ++ks) {
        mma_bf16(d_tmem, smem_desc(a0 + ks * 256, K), smem_desc(b0 + ks * 256, K), idesc,
                 (accumulate || ks > 0) ? 1u : 0u);
    }
}

// MN-major ("transposed") tiles: an MN x K bf16 tile stored as core matrices
// of 8 K-rows x 8 MN-elements (16 B per K-row), MN-groups contiguous:
// element (mn, k) at ((k / 8) * (MN / 8) + mn / 8) * 128 + (k % 8) * 16 + (mn % 8) * 2.
// Descriptor: LBO = K-direction core-matrix stride ((MN/8) * 128 B), SBO = 128 B;
// one k-step (K = 16) advances the start by 2 * LBO.  A row of the source
// matrix with MN contiguous (e.g. a token's k or v, a row of H) is stored with
// 16-byte vector writes.  Results are bit-identical to the K-major layout.
__host__ __device__ __forceinline__ uint32_t mn_off(int mn, int k, int MN) {
    return (uint32_t)((((k >> 3) * (MN >> 3)) + (mn >> 3)) * 128 + (k & 7) * 16 + (mn & 7) * 2);
}

__device__ __forceinline__ uint64_t smem_desc_mn(uint32_t saddr, int MN) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((((uint32_t)MN >> 3) * 128u >> 4) & 0x3FFFu) << 16;  // LBO: along K
    d |= (uint64_t)((128u >> 4) & 0x3FFFu) << 32;                        // SBO: along MN
    d |= (uint64_t)1 << 46;
    return d;
}

__host__ __device__ constexpr uint32_t idesc_bf16_major(int M, int N, bool a_mn, bool b_mn) {
    return idesc_bf16(M, N) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16);
}

// As mma_tile, with each operand either K-major (false) or MN-major (true).
template <int M, int N, int K, bool AMN, bool BMN>
__device__ __forceinline__ void mma_tile_mj(uint32_t d_tmem, const void* a_tile, const void* b_tile,
                                            bool accumulate) {
    constexpr uint32_t idesc = idesc_bf16_major(M, N, AMN, BMN);
    const uint32_t a0 = smem_u32(a_tile), b0 = smem_u32(b_tile);
#pragma unroll
    for (int ks = 0; ks < K / 16; ++ks) {
        const uint64_t da = AMN ? smem_desc_mn(a0 + ks * 2 * (M / 8) * 128, M) : smem_desc(a0 + ks * 256, K);
        const uint64_t db = BMN ? smem_desc_mn(b0 + ks * 2 * (N / 8) * 128, N) : smem_desc(b0 + ks * 256, K);
        mma_bf16(d_tmem, da, db, idesc, (accumulate || ks > 0) ? 1u : 0u);
    }
}

// Descriptor of the k-step-0 sub-tile of an operand tile: K-major (smem_desc) or
// MN-major (smem_desc_mn).  The k-steps of mma_tile_d add a constant to its address field.
template <int MN, int K, bool MJ>
__device__ __forceinline__ uint64_t tile_desc(const void* tile) {
    return MJ ? smem_desc_mn(smem_u32(tile), MN) : smem_desc(smem_u32(tile), K);
}

// As mma_tile_mj, from precomputed k-step-0 descriptors (tile_desc): the same
// instructions with the same operands, for an issuing thread that reuses its tiles.
template <int M, int N, int K, bool AMN, bool BMN>
__device__ __forceinline__ void mma_tile_d(uint32_t d_tmem, uint64_t da, uint64_t db, bool accumulate) {
    constexpr uint32_t idesc = idesc_bf16_major(M, N, AMN, BMN);
    constexpr uint64_t astep = AMN ? (2 * (M / 8) * 128) >> 4 : 256 >> 4;
    constexpr uint64_t bstep = BMN ? (2 * (N / 8) * 128) >> 4 : 256 >> 4;
#pragma unroll
    for (int ks = 0; ks < K / 16; ++ks)
        mma_bf16(d_tmem, da + ks * astep, db + ks * bstep, idesc, (accumulate || ks > 0) ? 1u : 0u);
}

// Arrives on `mbar` once every MMA issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t* mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(smem_u32(mbar)) : "memory");
}

// ---- mbarrier ----------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* mbar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(mbar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* mbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_u32(mbar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ uint32_t mbar_try_wait(uint64_t* mbar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_u32(mbar)), "r"(parity) : "memory");
    return ok;
}
// Bounded wait for the phase with the given parity.  Returns false (and
// records CPR_ERR_DEVICE_TIMEOUT) if it does not complete within `limit` polls.
__device__ __forceinline__ bool mbar_wait_n(uint64_t* mbar, uint32_t parity, uint32_t* err, uint32_t limit) {
    for (uint32_t it = 0; it < limit; ++it)
        if (mbar_try_wait(mbar, parity)) return true;
    set_error(err, CPR_ERR_DEVICE_TIMEOUT);
    return false;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* mbar, uint32_t parity, uint32_t* err) {
    return mbar_wait_n(mbar, parity, err, 1u << 22);
}

// ---- bulk async copy (global -> shared), completion on an mbarrier ----------------
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src, uint32_t bytes, uint64_t* mbar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(smem_u32(dst_smem)), "l"(src), "r"(bytes), "r"(smem_u32(mbar)) : "memory");
}

// ---- bulk async copy (shared -> global), completion tracked by bulk groups ----------------
// Both addresses 16-byte aligned, bytes a multiple of 16.  The writes to shared memory that
// produced the source must be made visible to the async proxy first (fence_async_smem).
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src_smem, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 :: "l"(dst), "r"(smem_u32(src_smem)), "r"(bytes) : "memory");
}
// One 32-byte global store (a whole sector): p must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8(float* p, const float (&x)[8]) {
    asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                 :: "l"(p), "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]),
                    "f"(x[7]) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until every committed bulk store of this thread has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// ---- 16-byte asynchronous copies (global -> shared), zero-filled when !valid ----------
__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                 :: "r"(smem_u32(dst_smem)), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// ---- TMEM -> registers ---------------------------------------------------------------
// 32 consecutive columns of this warp's lane quarter: thread i gets lane (32w + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
                   "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
                   "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
                   "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 128 consecutive columns of this warp's lane quarter in one load (thread i gets lane
// 32w + i); the wait is part of the same statement, so no use of v precedes it.
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, float (&v)[128]) {
    uint32_t r[128];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x128.b32 {"
                 "%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
                 "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
                 "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,"
                 "%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,"
                 "%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,"
                 "%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,"
                 "%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127"
                 "}, [%128];\n\ttcgen05.wait::ld.sync.aligned;"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
                   "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
                   "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
                   "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]),
                   "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]),
                   "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
                   "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]),
                   "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]),
                   "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]),
                   "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]),
                   "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]),
                   "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]),
                   "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]),
                   "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]),
                   "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]),
                   "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]),
                   "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]),
                   "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]),
                   "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]),
                   "=r"(r[126]), "=r"(r[127])
                 : "r"(taddr)
                 : "memory");
#pragma unroll
    for (int i = 0; i < 128; ++i) v[i] = __uint_as_float(r[i]);
}

// Several 32-column loads (any lanes' quarter, any columns) under one wait: as tmem_ld32
// each, without a wait between them.
__device__ __forceinline__ void tmem_ld32x2(uint32_t t0, float (&v0)[32], uint32_t t1, float (&v1)[32]) {
    uint32_t r0[32], r1[32];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {"
                 "%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
                 "tcgen05.ld.sync.aligned.32x32b.x32.b32 {"
                 "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
                 "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
                 "tcgen05.wait::ld.sync.aligned;"
                 : "=r"(r0[0]), "=r"(r0[1]), "=r"(r0[2]), "=r"(r0[3]), "=r"(r0[4]), "=r"(r0[5]),
                   "=r"(r0[6]), "=r"(r0[7]), "=r"(r0[8]), "=r"(r0[9]), "=r"(r0[10]), "=r"(r0[11]),
                   "=r"(r0[12]), "=r"(r0[13]), "=r"(r0[14]), "=r"(r0[15]), "=r"(r0[16]), "=r"(r0[17]),
                   "=r"(r0[18]), "=r"(r0[19]), "=r"(r0[20]), "=r"(r0[21]), "=r"(r0[22]), "=r"(r0[23]),
                   "=r"(r0[24]), "=r"(r0[25]), "=r"(r0[26]), "=r"(r0[27]), "=r"(r0[28]), "=r"(r0[29]),
                   "=r"(r0[30]), "=r"(r0[31]), "=r"(r1[0]), "=r"(r1[1]), "=r"(r1[2]), "=r"(r1[3]),
                   "=r"(r1[4]), "=r"(r1[5]), "=r"(r1[6]), "=r"(r1[7]), "=r"(r1[8]), "=r"(r1[9]),
                   "=r"(r1[10]), "=r"(r1[11]), "=r"(r1[12]), "=r"(r1[13]), "=r"(r1[14]), "=r"(r1[15]),
                   "=r"(r1[16]), "=r"(r1[17]), "=r"(r1[18]), "=r"(r1[19]), "=r"(r1[20]), "=r"(r1[21]),
                   "=r"(r1[22]), "=r"(r1[23]), "=r"(r1[24]), "=r"(r1[25]), "=r"(r1[26]), "=r"(r1[27]),
                   "=r"(r1[28]), "=r"(r1[29]), "=r"(r1[30]), "=r"(r1[31])
                 : "r"(t0), "r"(t1)
                 : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v0[i] = __uint_as_float(r0[i]);
#pragma unroll
    for (int i = 0; i < 32; ++i) v1[i] = __uint_as_float(r1[i]);
}
__device__ __forceinline__ void tmem_ld32x4(uint32_t t0, float (&v0)[32], uint32_t t1, float (&v1)[32],
                                            uint32_t t2, float (&v2)[32], uint32_t t3, float (&v3)[32]) {
    uint32_t r0[32], r1[32], r2[32], r3[32];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {"
                 "%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%128];\n\t"
                 "tcgen05.ld.sync.aligned.32x32b.x32.b32 {"
                 "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
                 "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%129];\n\t"
                 "tcgen05.ld.sync.aligned.32x32b.x32.b32 {"
                 "%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,"
                 "%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95}, [%130];\n\t"
                 "tcgen05.ld.sync.aligned.32x32b.x32.b32 {"
                 "%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,"
                 "%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%131];\n\t"
                 "tcgen05.wait::ld.sync.aligned;"
                 : "=r"(r0[0]), "=r"(r0[1]), "=r"(r0[2]), "=r"(r0[3]), "=r"(r0[4]), "=r"(r0[5]),
                   "=r"(r0[6]), "=r"(r0[7]), "=r"(r0[8]), "=r"(r0[9]), "=r"(r0[10]), "=r"(r0[11]),
                   "=r"(r0[12]), "=r"(r0[13]), "=r"(r0[14]), "=r"(r0[15]), "=r"(r0[16]), "=r"(r0[17]),
                   "=r"(r0[18]), "=r"(r0[19]), "=r"(r0[20]), "=r"(r0[21]), "=r"(r0[22]), "=r"(r0[23]),
                   "=r"(r0[24]), "=r"(r0[25]), "=r"(r0[26]), "=r"(r0[27]), "=r"(r0[28]), "=r"(r0[29]),
                   "=r"(r0[30]), "=r"(r0[31]), "=r"(r1[0]), "=r"(r1[1]), "=r"(r1[2]), "=r"(r1[3]),
                   "=r"(r1[4]), "=r"(r1[5]), "=r"(r1[6]), "=r"(r1[7]), "=r"(r1[8]), "=r"(r1[9]),
                   "=r"(r1[10]), "=r"(r1[11]), "=r"(r1[12]), "=r"(r1[13]), "=r"(r1[14]), "=r"(r1[15]),
                   "=r"(r1[16]), "=r"(r1[17]), "=r"(r1[18]), "=r"(r1[19]), "=r"(r1[20]), "=r"(r1[21]),
                   "=r"(r1[22]), "=r"(r1[23]), "=r"(r1[24]), "=r"(r1[25]), "=r"(r1[26]), "=r"(r1[27]),
                   "=r"(r1[28]), "=r"(r1[29]), "=r"(r1[30]), "=r"(r1[31]), "=r"(r2[0]), "=r"(r2[1]),
                   "=r"(r2[2]), "=r"(r2[3]), "=r"(r2[4]), "=r"(r2[5]), "=r"(r2[6]), "=r"(r2[7]),
                   "=r"(r2[8]), "=r"(r2[9]), "=r"(r2[10]), "=r"(r2[11]), "=r"(r2[12]), "=r"(r2[13]),
                   "=r"(r2[14]), "=r"(r2[15]), "=r"(r2[16]), "=r"(r2[17]), "=r"(r2[18]), "=r"(r2[19]),
                   "=r"(r2[20]), "=r"(r2[21]), "=r"(r2[22]), "=r"(r2[23]), "=r"(r2[24]), "=r"(r2[25]),
                   "=r"(r2[26]), "=r"(r2[27]), "=r"(r2[28]), "=r"(r2[29]), "=r"(r2[30]), "=r"(r2[31]),
                   "=r"(r3[0]), "=r"(r3[1]), "=r"(r3[2]), "=r"(r3[3]), "=r"(r3[4]), "=r"(r3[5]),
                   "=r"(r3[6]), "=r"(r3[7]), "=r"(r3[8]), "=r"(r3[9]), "=r"(r3[10]), "=r"(r3[11]),
                   "=r"(r3[12]), "=r"(r3[13]), "=r"(r3[14]), "=r"(r3[15]), "=r"(r3[16]), "=r"(r3[17]),
                   "=r"(r3[18]), "=r"(r3[19]), "=r"(r3[20]), "=r"(r3[21]), "=r"(r3[22]), "=r"(r3[23]),
                   "=r"(r3[24]), "=r"(r3[25]), "=r"(r3[26]), "=r"(r3[27]), "=r"(r3[28]), "=r"(r3[29]),
                   "=r"(r3[30]), "=r"(r3[31])
                 : "r"(t0), "r"(t1), "r"(t2), "r"(t3)
                 : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v0[i] = __uint_as_float(r0[i]);
#pragma unroll
    for (int i = 0; i < 32; ++i) v1[i] = __uint_as_float(r1[i]);
#pragma unroll
    for (int i = 0; i < 32; ++i) v2[i] = __uint_as_float(r2[i]);
#pragma unroll
    for (int i = 0; i < 32; ++i) v3[i] = __uint_as_float(r3[i]);
}

// TMEM address of (warp's lane quarter, column c).
__device__ __forceinline__ uint32_t taddr_of(uint32_t base, int warp, int col) {
    return base + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)col;
}

// ---- bf16 hi/lo split -------------------------------------------------------------------
// x ~= hi + lo with hi = bf16(x), lo = bf16(x - hi); x - hi is exact in fp32.
__device__ __forceinline__ void split_bf16(float x, __nv_bfloat16& hi, __nv_bfloat16& lo) {
    hi = __float2bfloat16_rn(x);
    lo = __float2bfloat16_rn(__fsub_rn(x, __bfloat162float(hi)));
}

// Splits 8 fp32 values into packed hi and lo bf16 vectors (the split of
// split_bf16, two values per conversion: both round to nearest even, so the
// bits are the same).
__device__ __forceinline__ void split8(const float (&x)[8], uint4& hi, uint4& lo) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 hb = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
        const float2 hf = __bfloat1622float2(hb);
        const __nv_bfloat162 lb = __floats2bfloat162_rn(__fsub_rn(x[2 * i], hf.x), __fsub_rn(x[2 * i + 1], hf.y));
        h[i] = *reinterpret_cast<const uint32_t*>(&hb);
        l[i] = *reinterpret_cast<const uint32_t*>(&lb);
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// Stores 8 fp32 values (consecutive along K) as one 16-byte core-matrix row,
// split into hi and lo tiles at the same offset.
__device__ __forceinline__ void store8_split(unsigned char* hi_tile, unsigned char* lo_tile,
                                             uint32_t off, const float (&x)[8]) {
    uint4 hi, lo;
    split8(x, hi, lo);
    *reinterpret_cast<uint4*>(hi_tile + off) = hi;
    *reinterpret_cast<uint4*>(lo_tile + off) = lo;
}

// Packed hi/lo vectors back to 8 fp32 values (hi + lo).
__device__ __forceinline__ void join8(const uint4& hi, const uint4& lo, float (&x)[8]) {
    const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&hi);
    const __nv_bfloat16* l = reinterpret_cast<const __nv_bfloat16*>(&lo);
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = __fadd_rn(__bfloat162float(h[i]), __bfloat162float(l[i]));
}

// 8 bf16 values (16 bytes) to fp32.
__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&x)[8]) {
    const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&v);
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = __bfloat162float(h[i]);
}

}  // namespace tc
}  // namespace cpr
