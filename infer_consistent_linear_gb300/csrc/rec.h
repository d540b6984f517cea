// Token-recurrence kernels for the stage-table ablations (see rec.cu).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace cpr {
namespace rec {

struct RecArgs {
    const void* q;            // io dtype [n_tok, H, d]
    const void* k;
    const void* v;
    const float* g;           // [n_tok, H]
    const float* beta;
    const int32_t* cu;        // sequences for the prefill; null for a decode step
    int n_seq;
    int64_t n_tok;
    int H;
    float scale;
    const float* h0;          // prefill: initial state or null (zeros)
    float* state;             // decode: the state, read and written in place
    float* final_state;       // prefill: final state or null
    float* o;                 // fp32 [n_tok, H, d]
    uint32_t* err;
};

// Backward of the token recurrence (cpr_gdn_recurrent_bwd).  States are recomputed from
// checkpoints every kRecSeg tokens; each segment's states go to a per-(sequence, head)
// scratch before the segment is walked back.
constexpr int kRecSeg = 16;

struct RecBwdArgs {
    const void* q;            // io dtype [n_tok, H, d]
    const void* k;
    const void* v;
    const float* g;           // [n_tok, H]
    const float* beta;
    const int32_t* cu;
    int n_seq;
    int64_t n_tok;
    int H;
    float scale;
    const float* h0;          // or null (zeros)
    const float* dO;          // fp32 [n_tok, H, d]
    const float* dHT;         // or null (zeros)
    float* dq;                // fp32 [n_tok, H, d]
    float* dk;
    float* dv;
    float* dg;                // fp32 [n_tok, H]
    float* dbeta;
    float* dh0;               // fp32 [n_seq, H, d, d]
    float* ckpt;              // [(n_tok / kRecSeg + n_seq) * H] states of d * d fp32
    float* seg;               // [n_seq * H * kRecSeg] states of d * d fp32
    uint32_t* err;
};

struct RbArgs {               // reading B (d = 128, bf16 io)
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const float* g;
    const float* beta;
    const int32_t* cu;
    const int32_t* chunk_off;   // the training forward's chunk table
    int n_seq;
    int H;
    float scale;
    const unsigned char* ws;    // its per-(chunk, head) blocks
    size_t blk_bytes;
    size_t off_hn;              // H_n hi/lo tiles within a block
    float* o;
    float* run;                 // or null: the in-chunk state after a sequence's partial last chunk
};

struct RbStepArgs {           // reading B decode step (d = 128, bf16 io)
    const uint32_t* header;   // the cache's header words
    uint32_t digest[8];       // the contract's digest and header words the cache must carry
    uint32_t hdr[15];         // (kHdrWords of common.cuh)
    const __nv_bfloat16* q;   // [n_seq, H, d]
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const float* g;
    const float* beta;
    int n_seq;
    int H;
    float scale;
    int32_t* pos;             // the cache's positions (moved on by this step)
    uint32_t* done;           // the cache's step counter (one word)
    const float* state;       // the cache's chunk-start states, fp32 [n_seq, H, d, d]
    float* run;               // [n_seq, H, d, d] running in-chunk states
    __nv_bfloat16* rk;        // the current chunk's token rows, token-major [n_seq * C, H, d]
    __nv_bfloat16* rv;
    float* rg;                // [n_seq * C, H]
    float* rbeta;
    float* o;
    uint32_t* err;
    int no_commit;            // the caller's claim that no sequence completes its chunk now
};

struct RbFillArgs {           // reading B prefill: the partial last chunk's rows into a cache
    const __nv_bfloat16* k;   // the prefill's token tensors
    const __nv_bfloat16* v;
    const float* g;
    const float* beta;
    const int32_t* cu;
    int n_seq;
    int H;
    __nv_bfloat16* rk;        // as RbStepArgs
    __nv_bfloat16* rv;
    float* rg;
    float* rbeta;
    int32_t* rcu;             // [n_seq + 1]: b * C, the commit batch's sequence offsets
};

}  // namespace rec

// d in {64, 128}; io bf16 or fp32.
cudaError_t rec_launch(const rec::RecArgs& a, int d, bool bf16, cudaStream_t st);
cudaError_t rec_bwd_launch(const rec::RecBwdArgs& a, int d, bool bf16, cudaStream_t st);
// grid (chunk slots, H)
cudaError_t rb_launch(const rec::RbArgs& a, int64_t cmax, cudaStream_t st);
cudaError_t rb_step_launch(const rec::RbStepArgs& a, cudaStream_t st);
cudaError_t rb_fill_launch(const rec::RbFillArgs& a, cudaStream_t st);

}  // namespace cpr
