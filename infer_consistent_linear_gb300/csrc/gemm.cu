// Batch-invariant projection GEMM Y = X W (bf16 X [M, K], W [K, N], fp32 Y [M, N]) with a
// fixed split of K into contiguous leaves: the projections that feed CPR must not change
// a token's bits with the batch it is in (page "IsoExec: 切换 SkyRL 中的训练器-推理不匹配",
// batch-invariant kernels; the fixed leaf tree of its tensor-parallel section).
//
// Arithmetic (what fixes a row's bits): leaf l covers K rows [l * leaf_k, (l + 1) * leaf_k)
// and is accumulated in fp32 by tcgen05 MMAs (M = 128, N = 256, K = 16) in ascending k;
// the leaves are added in the fixed tree (P0 + P1) + (P2 + P3).  Nothing in a row's
// arithmetic depends on M, on the other rows or on the tile the row falls in, so a
// token's output is the same in any batch.
//
// Schedule: persistent CTAs (one per SM) walk 128 x 256 output tiles.  320 threads in
// three roles:
//   warp 0      TMA producer: per k-block one 128 x 64 box of X and up to four 64 x 64
//               boxes of W, 128-byte swizzled, into a 4-stage ring (48 KB a stage);
//   warp 1      MMA issuer: leaves in pairs, leaf 2p into TMEM columns 0..255 and leaf
//               2p + 1 into 256..511; each stage is released by a commit once its MMAs
//               are done, each pair by a commit to the epilogue;
//   warps 2..9  epilogue: two warps per TMEM lane quarter, 128 columns each; they add a
//               pair's two leaves (P0 + P1, kept in registers, then P2 + P3), hand the
//               columns back, and store finished rows as whole 32-byte sectors.
// The MMA issuer waits only for the epilogue to have read a pair, so one tile's stores
// overlap the next tile's MMAs.  Every wait is bounded; a wait that runs out records
// CPR_ERR_DEVICE_TIMEOUT and its role stops, copies and MMAs in flight are waited for
// (bounded) and TMEM is released.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "gemm.h"
#include "tc_common.cuh"

namespace cpr {
namespace gemm {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int kThreads = 320;
constexpr uint32_t kABytes = BM * BK * 2;                   // X box: 128 rows of 128 bytes
constexpr uint32_t kBBox = BK * 64 * 2;                     // W box: 64 k-rows x 64 columns
constexpr uint32_t kStage = kABytes + (BN / 64) * kBBox;    // 48 KB
constexpr size_t kSmem = 1024 + (size_t)STAGES * kStage + 256;   // + alignment slack, barriers

// Shared-memory matrix descriptor for a 128-byte-swizzled operand (8 rows of 128 bytes per
// swizzle atom).  K-major (X rows): SBO = 1024 B between 8-row groups, LBO unused; one
// K = 16 step advances the start by 32 B inside the atom.  MN-major (W rows, N
// contiguous): LBO = stride between 64-column atoms, SBO = 1024 B between 8-k-row groups;
// one K = 16 step advances the start by 2048 B.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;   // descriptor version
    d |= (uint64_t)2 << 61;   // 128-byte swizzle
    return d;
}

// 2-D TMA tile load (x = innermost element coordinate, y = row), completion on mbar.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* mbar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        :: "r"(tc::smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y),
           "r"(tc::smem_u32(mbar))
        : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* mbar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(tc::smem_u32(mbar)) : "memory");
}

// 16 consecutive TMEM columns of this warp's lane quarter.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__global__ void __launch_bounds__(kThreads, 1)
k_gemm(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap mw, GemmArgs a) {
    extern __shared__ unsigned char sm_raw[];
    // 128-byte swizzle atoms want 1024-byte aligned tiles
    unsigned char* sm = sm_raw + ((1024u - (tc::smem_u32(sm_raw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + STAGES * kStage);   // stage loaded
    uint64_t* empty = full + STAGES;                                      // stage consumed
    uint64_t* tfull = empty + STAGES;                                     // leaf pair in TMEM
    uint64_t* tempty = tfull + 1;                                         // leaf pair read
    uint32_t* tbase = reinterpret_cast<uint32_t*>(tempty + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_nt = (a.N + BN - 1) / BN;
    const int tiles = ((a.M + BM - 1) / BM) * n_nt;
    const int nkb = a.K / BK, kb_leaf = a.leaf_k / BK, nleaf = a.K / a.leaf_k;
    const int npair = nleaf == 4 ? 2 : 1;
    const int per_pair = nleaf == 1 ? 1 : 2;

    if (warp == 1) tc::tmem_alloc(tbase, 512);
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            tc::mbar_init(full + s, 1);
            tc::mbar_init(empty + s, 1);
        }
        tc::mbar_init(tfull, 1);
        tc::mbar_init(tempty, 8);   // one arrival per epilogue warp
        tc::mbar_init_fence();
    }
    tc::tc_sync();
    const uint32_t tmem = *tbase;

    if (warp == 0) {
        if (lane == 0) {
            uint32_t it = 0;   // k-blocks issued by this CTA
            bool ok = true;
            for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
                const int m0 = (t / n_nt) * BM, n0 = (t % n_nt) * BN;
                const int nbox = min(BN, a.N - n0) / 64;   // boxes past N are not loaded
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const uint32_t s = it % STAGES;
                    if (it >= STAGES && !(ok = tc::mbar_wait(empty + s, ((it / STAGES) - 1) & 1u, a.err))) break;
                    unsigned char* st = sm + s * kStage;
                    tc::mbar_expect_tx(full + s, kABytes + nbox * kBBox);
                    tma_load_2d(st, &mx, kb * BK, m0, full + s);
                    for (int i = 0; i < nbox; ++i)
                        tma_load_2d(st + kABytes + i * kBBox, &mw, n0 + 64 * i, kb * BK, full + s);
                }
            }
            // the last loads land before the CTA exits (bounded)
            for (uint32_t j = it > STAGES ? it - STAGES : 0; j < it; ++j)
                tc::mbar_wait(full + j % STAGES, (j / STAGES) & 1u, a.err);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_bf16_major(BM, BN, false, true);
            uint32_t it = 0, g = 0;   // k-blocks consumed, leaf pairs issued
            bool ok = true;
            for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
                for (int p = 0; p < npair && ok; ++p, ++g) {
                    if (g >= 1 && !(ok = tc::mbar_wait(tempty, (g - 1) & 1u, a.err))) break;
                    tc::fence_after();
                    for (int l = 0; l < per_pair && ok; ++l) {
                        const uint32_t d = tmem + (uint32_t)(l * BN);
                        const int kb0 = (p * 2 + l) * kb_leaf;
                        for (int kb = kb0; kb < kb0 + kb_leaf; ++kb, ++it) {
                            const uint32_t s = it % STAGES;
                            if (!(ok = tc::mbar_wait(full + s, (it / STAGES) & 1u, a.err))) break;
                            tc::fence_after();
                            const uint32_t a0 = tc::smem_u32(sm + s * kStage), b0 = a0 + kABytes;
#pragma unroll
                            for (int ks = 0; ks < BK / 16; ++ks)
                                tc::mma_bf16(d, desc_sw128(a0 + ks * 32, 16, 1024),
                                             desc_sw128(b0 + ks * 2048, kBBox, 1024), idesc,
                                             (kb > kb0 || ks > 0) ? 1u : 0u);
                            tc::mma_commit(empty + s);
                        }
                    }
                    if (ok) tc::mma_commit(tfull);
                }
            }
            // the last MMAs complete before TMEM is released (bounded)
            if (it > 0) tc::mbar_wait(empty + (it - 1) % STAGES, ((it - 1) / STAGES) & 1u, a.err);
        }
    } else {
        const int q = warp & 3, half = (warp - 2) >> 2;
        const int r = q * 32 + lane;
        const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(half * 128);
        uint32_t g = 0;
        bool ok = true;
        float acc[128];
        // one leaf pair: its two leaves added, onto acc unless it is the tile's first pair
        auto drain = [&](bool first) -> bool {
            if (!tc::mbar_wait(tfull, g & 1u, a.err)) return false;
            ++g;
            tc::fence_after();
#pragma unroll
            for (int c = 0; c < 128; c += 16) {
                float u[16];
                tmem_ld16(tq + c, u);
                if (per_pair == 2) {
                    float w[16];
                    tmem_ld16(tq + BN + c, w);
#pragma unroll
                    for (int j = 0; j < 16; ++j) u[j] = __fadd_rn(u[j], w[j]);
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) acc[c + j] = first ? u[j] : __fadd_rn(acc[c + j], u[j]);
            }
            tc::fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty);
            return true;
        };
        for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
            const int m0 = (t / n_nt) * BM, n0 = (t % n_nt) * BN;
            ok = drain(true);
            if (ok && npair == 2) ok = drain(false);
            if (!ok) break;
            if (m0 + r < a.M && n0 + half * 128 < a.N) {
                float* y = a.Y + (size_t)(m0 + r) * a.N + n0 + half * 128;
#pragma unroll
                for (int j8 = 0; j8 < 16; ++j8) {
                    float o8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) o8[e] = acc[8 * j8 + e];
                    tc::st_global_v8(y + 8 * j8, o8);
                }
            }
        }
    }
    tc::tc_sync();
    if (warp == 1) tc::tmem_dealloc(tmem, 512);
}

// cuTensorMapEncodeTiled from the driver, through the runtime (no link against libcuda).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// Row-major bf16 [rows, cols] as a 2-D tensor map with a (64 columns, box_rows) box,
// 128-byte swizzle, zero fill past the edges.
bool encode(CUtensorMap* m, const void* base, int rows, int cols, int box_rows) {
    const PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dim[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t stride[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
    const cuuint32_t estride[2] = {1u, 1u};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dim, stride, box, estride,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace gemm

cudaError_t gemm_launch(const gemm::GemmArgs& a, cudaStream_t st) {
    if (a.M == 0) return cudaSuccess;
    if (!gemm::encode_fn()) return cudaErrorNotSupported;   // the driver has no tensor-map encoder
    CUtensorMap mx, mw;
    if (!gemm::encode(&mx, a.X, a.M, a.K, gemm::BM) || !gemm::encode(&mw, a.W, a.K, a.N, gemm::BK))
        return cudaErrorInvalidValue;
    // per call (the attribute belongs to the current device), as the other launchers do
    cudaError_t e = cudaFuncSetAttribute(gemm::k_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)gemm::kSmem);
    if (e != cudaSuccess) return e;
    int dev = 0, nsm = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int64_t tiles = (int64_t)((a.M + gemm::BM - 1) / gemm::BM) * ((a.N + gemm::BN - 1) / gemm::BN);
    const int grid = (int)(tiles < nsm ? tiles : nsm);
    gemm::k_gemm<<<grid, gemm::kThreads, gemm::kSmem, st>>>(mx, mw, a);
    return cudaGetLastError();
}

}  // namespace cpr
