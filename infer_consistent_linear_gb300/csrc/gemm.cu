// Batch-invariant projection GEMM Y = X W (bf16 X [M, K], W [K, N], fp32 Y [M, N]) with a
// fixed split of K into contiguous leaves: the projections that feed CPR must not change
// a token's bits with the batch it is in (page "IsoExec: 切换 SkyRL 中的训练器-推理不匹配",
// batch-invariant kernels; the q/k/v/gate projections in front of the CPR layer).
//
// One CTA per 128 x 128 tile of Y, 128 threads.  Leaf l (K rows [l*leaf_k, (l+1)*leaf_k))
// accumulates into its own 128 TMEM columns with tcgen05 MMAs (M = 128, N = 128, K = 16)
// in ascending k; the epilogue adds the leaves in a fixed pairwise tree ((P0 + P1) +
// (P2 + P3)).  Nothing in a row's arithmetic depends on M, on the other rows or on the
// tile the row falls in, so a token's output is the same in any batch.  Operands reach
// shared memory through a 4-stage cp.async pipeline (X rows K-major, W rows MN-major,
// no transposes); a stage is refilled once the MMAs that read it have committed.
#include <cuda_bf16.h>
#include <stdint.h>

#include "gemm.h"
#include "tc_common.cuh"

namespace cpr {
namespace gemm {

constexpr int BM = 128, BN = 128, BK = 64, STAGES = 4;
constexpr uint32_t kStage = BM * BK * 2 + BN * BK * 2;   // 32 KB: A tile | B tile
constexpr size_t kSmem = STAGES * kStage + 64;

__global__ void __launch_bounds__(128, 1) k_gemm(GemmArgs a) {
    extern __shared__ __align__(1024) unsigned char sm[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + STAGES * kStage);   // one per stage
    uint32_t* tbase = reinterpret_cast<uint32_t*>(bar + STAGES);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    const int nkb = a.K / BK, kb_leaf = a.leaf_k / BK, nleaf = a.K / a.leaf_k;
    const __nv_bfloat16* X = a.X;
    const __nv_bfloat16* W = a.W;

    if (warp == 0) tc::tmem_alloc(tbase, 512);
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) tc::mbar_init(bar + s, 1);
        tc::mbar_init_fence();
    }
    // k-block kb into stage s: A rows m0.. (zero past M), K-major; B rows kb*64.., MN-major
    auto load = [&](int kb, int s) {
        unsigned char* At = sm + s * kStage;
        unsigned char* Bt = At + BM * BK * 2;
        const int k0 = kb * BK;
        for (int i = tid; i < BM * (BK / 8); i += 128) {
            const int r = i / (BK / 8), c8 = i % (BK / 8);
            const bool in = m0 + r < a.M;
            const __nv_bfloat16* src = X + (size_t)(in ? m0 + r : 0) * a.K + k0 + c8 * 8;
            tc::cp_async16(At + tc::cm_off(r, c8 * 8, BK), src, in);
        }
        for (int i = tid; i < BK * (BN / 8); i += 128) {
            const int kr = i / (BN / 8), c8 = i % (BN / 8);
            const __nv_bfloat16* src = W + (size_t)(k0 + kr) * a.N + n0 + c8 * 8;
            tc::cp_async16(Bt + tc::mn_off(c8 * 8, kr, BN), src, true);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    for (int s = 0; s < STAGES - 1; ++s) {
        if (s < nkb) load(s, s);
        else asm volatile("cp.async.commit_group;" ::: "memory");
    }
    tc::tc_sync();
    const uint32_t tmem = *tbase;
    uint32_t ph[STAGES] = {};
    bool pend[STAGES] = {};
    bool ok = true;
    for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % STAGES;
        asm volatile("cp.async.wait_group %0;" :: "n"(STAGES - 2) : "memory");
        tc::fence_async_smem();
        tc::tc_sync();
        if (tid == 0) {
            const int leaf = kb / kb_leaf;
            const bool first = (kb % kb_leaf) == 0;
            tc::mma_tile_mj<BM, BN, BK, false, true>(tmem + leaf * BN, sm + s * kStage,
                                                     sm + s * kStage + BM * BK * 2, !first);
            tc::mma_commit(bar + s);
        }
        pend[s] = true;
        // refill the stage k-block kb - 1 used, once its MMAs are done
        const int kn = kb + STAGES - 1, sn = kn % STAGES;
        if (kb >= 1 && pend[sn]) {
            ok = tc::mbar_wait(bar + sn, ph[sn], a.err) && ok;
            ph[sn] ^= 1u;
            pend[sn] = false;
        }
        if (__syncthreads_or(!ok)) break;
        if (kn < nkb) load(kn, sn);
        else asm volatile("cp.async.commit_group;" ::: "memory");
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    for (int s = 0; s < STAGES; ++s)   // the last MMAs (bounded)
        if (pend[s]) {
            ok = tc::mbar_wait(bar + s, ph[s], a.err) && ok;
            ph[s] ^= 1u;
        }
    tc::fence_after();
    ok = !__syncthreads_or(!ok);
    if (ok) {
        // epilogue: row m0 + 32 warp + lane, 32 columns at a time, leaves in a fixed tree
        const int r = warp * 32 + (tid & 31);
        const bool in = m0 + r < a.M;
        float* yrow = a.Y + (size_t)(in ? m0 + r : 0) * a.N + n0;
        for (int c0 = 0; c0 < BN; c0 += 32) {
            float p0[32], p1[32];
            tc::tmem_ld32(tc::taddr_of(tmem, warp, c0), p0);
            if (nleaf >= 2) {
                tc::tmem_ld32(tc::taddr_of(tmem + BN, warp, c0), p1);
#pragma unroll
                for (int j = 0; j < 32; ++j) p0[j] = __fadd_rn(p0[j], p1[j]);
            }
            if (nleaf == 4) {
                float p2[32];
                tc::tmem_ld32(tc::taddr_of(tmem + 2 * BN, warp, c0), p1);
                tc::tmem_ld32(tc::taddr_of(tmem + 3 * BN, warp, c0), p2);
#pragma unroll
                for (int j = 0; j < 32; ++j) p0[j] = __fadd_rn(p0[j], __fadd_rn(p1[j], p2[j]));
            }
            if (in) {
#pragma unroll
                for (int j8 = 0; j8 < 4; ++j8) {
                    float o8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) o8[e] = p0[8 * j8 + e];
                    tc::st_global_v8(yrow + c0 + 8 * j8, o8);
                }
            }
        }
    }
    tc::tc_sync();
    if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

}  // namespace gemm

cudaError_t gemm_launch(const gemm::GemmArgs& a, cudaStream_t st) {
    if (a.M == 0) return cudaSuccess;
    // per call (the attribute belongs to the current device), as the other launchers do
    const cudaError_t e = cudaFuncSetAttribute(gemm::k_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)gemm::kSmem);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)(a.N / gemm::BN), (unsigned)((a.M + gemm::BM - 1) / gemm::BM));
    gemm::k_gemm<<<grid, 128, gemm::kSmem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace cpr
