// Shared device helpers of the CPR Gated DeltaNet kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "cpr_gdn.h"

namespace cpr {

constexpr int kChunk = 64;  // C of this build

// ---- io conversion (bf16 -> fp32 is exact) ---------------------------------
__device__ __forceinline__ float cvt(float x) { return x; }
__device__ __forceinline__ float cvt(__nv_bfloat16 x) { return __bfloat162float(x); }

// Converts 8 consecutive io elements (16-byte aligned for bf16, 32-byte for
// fp32) to fp32.
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float out[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        out[2 * i] = f.x;
        out[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ void load8(const float* p, float out[8]) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
    out[4] = b.x; out[5] = b.y; out[6] = b.z; out[7] = b.w;
}
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float in[8]) {
    uint4 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(in[2 * i], in[2 * i + 1]);
    *reinterpret_cast<uint4*>(p) = u;
}
__device__ __forceinline__ void store8(float* p, const float in[8]) {
    *reinterpret_cast<float4*>(p) = make_float4(in[0], in[1], in[2], in[3]);
    *reinterpret_cast<float4*>(p + 4) = make_float4(in[4], in[5], in[6], in[7]);
}

// ---- device error word -----------------------------------------------------
// First error wins; kernels skip their work after recording one.
__device__ __forceinline__ void set_error(uint32_t* err, uint32_t code) {
    if (err) atomicCAS(err, 0u, code);
}

// ---- chunk table -------------------------------------------------------------
// chunk_off[b] = number of chunks of sequences < b; chunk_off[n_seq] = total
// (or -1 when cu_seqlens failed validation).  Returns the sequence owning
// global chunk `c` (0 <= c < total).
__device__ __forceinline__ int find_seq(const int32_t* chunk_off, int n_seq, int c) {
    int lo = 0, hi = n_seq - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (chunk_off[mid] <= c) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// ---- decode cache section offsets (bytes) ------------------------------------
struct CacheOff {
    size_t header, pos, done, state, k_rows, v_rows, gam_rows, beta_rows, t_rows, delta_rows,
        state_tiles, delta_tiles;
};

struct Digest {
    uint32_t w[8];
};

// Header words (uint32): [0] magic, [1] version, [2..9] contract digest, [10] n_seq,
// [11] H, [12] C, [13] d_k, [14] d_v, [15] operand policy, [16] io dtype, [17..24] the
// deployment digest of the process that wrote the cache (cpr_deployment_digest).
constexpr uint32_t kCacheMagic = 0x43505243u;
constexpr int kHdrWords = 15;   // header words 10..24, after the contract digest

// Whether a decode cache's header words 0 .. 9 + kHdrWords are the expected ones: the
// magic, the contract version, `digest` and then `words`.  Called by all 32 lanes of a
// warp, a word per lane (the loads are independent); every lane gets the verdict.
__device__ __forceinline__ bool cache_header_ok(const uint32_t* hdr, const uint32_t* digest,
                                                const uint32_t* words) {
    const int lane = threadIdx.x & 31;
    bool ok = true;
    if (lane == 0) ok = hdr[0] == kCacheMagic;
    else if (lane == 1) ok = hdr[1] == CPR_CONTRACT_VERSION;
    else if (lane < 10) ok = hdr[lane] == digest[lane - 2];
    else if (lane < 10 + kHdrWords) ok = hdr[lane] == words[lane - 10];
    return __all_sync(0xffffffffu, ok);
}

}  // namespace cpr
