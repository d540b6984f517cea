/*
 * cpr_gdn.h -- C ABI of the Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet
 * library for sm_103a (GB300).
 *
 * What the library computes.  Per (sequence, head) the gated delta rule
 *     S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *     o_t = S_t (scale q_t),       alpha_t = exp(g_t),
 * with S_t of size d_v x d_k.  Source: page "IsoExec: 切换 SkyRL 中的训练器-
 * 推理不匹配", section "Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet"
 * (Gated DeltaNet; the recurrence is primary, parallelised across chunks of
 * C tokens, and decode resynchronises the hidden state every C tokens), and
 * the same page's "Bitwise Exact" row of its CPR table: trainer forward,
 * rollout prefill and rollout decode must give identical bits.
 *
 * Execution contract.  Every call carries a cpr_contract and the SHA-256
 * digest of its canonical serialisation.  The contract pins every choice
 * that affects rounding (chunk size, dtypes, operand policy, reduction
 * orders, chunk-to-state schedule, kernel build); the digest lets separate
 * processes (trainer, rollout engine) prove they run the same numerical
 * policy.  Source: page "IsoExec: bitpontos végrehajtással csökkentené az
 * RL-rendszerek eltéréseit", section "Szerződés és közös modell" (contract
 * fixing implementation, accumulation dtype, boundary dtype, reduction
 * decomposition; SHA-256 digests), and page "IsoExec: 切换 SkyRL 中的训练器-
 * 推理不匹配", section "合约结构与强制执行" (cases x regions, composition,
 * claims, identities).  This library is one region with the cases
 * trainer_fwd (cpr_gdn_fwd), engine_prefill (cpr_gdn_prefill) and decode
 * (cpr_gdn_decode_step), plus the trainer backward (cpr_gdn_bwd).
 *
 * Layouts (all row-major, contiguous, token-major as a projection writes):
 *     q, k          [n_tok, H, d_k]        io dtype
 *     v             [n_tok, H, d_v]        io dtype
 *     o             [n_tok, H, d_v]        out dtype (fp32)
 *     g, beta       [n_tok, H]             fp32  (log-gate g <= 0; beta in (0,1))
 *     h0, final     [n_seq, H, d_k, d_v]   fp32  (H = S^T, "state")
 *     cu_seqlens    [n_seq + 1]            int32, cu[0] = 0, non-decreasing,
 *                                          cu[n_seq] = n_tok (device memory)
 *     decode tokens [n_seq, H, d]          one token per sequence per step
 * Chunks restart at every sequence start; the last chunk of a sequence may
 * be partial.
 *
 * Conventions.
 *   - All pointers to tensors are DEVICE pointers owned by the caller; the
 *     library never allocates or frees device memory and never synchronises
 *     the host (except the functions that say so).
 *   - Every compute call is asynchronous on `stream` (a cudaStream_t passed
 *     as void*; NULL = legacy default stream).
 *   - Tensor pointers must be 16-byte aligned, except the per-token scalar
 *     tensors (g, beta, dg, dbeta) and cu_seqlens, which need 4 bytes, and
 *     the outputs written in whole 32-byte sectors, which need 32 bytes: dq
 *     and dk under CPR_POLICY_TC_BF16X3, and Y of cpr_gemm_bf16
 *     (CPR_ERR_ALIGNMENT).  Token tensors may be NULL when n_tok == 0.
 *   - Host-side checks return an error code immediately and launch nothing.
 *     Checks that need device data (cu_seqlens validity, the digest stored in
 *     a decode cache) run on the device: on failure the kernels skip their
 *     work and record the code in a device error word read by
 *     cpr_get_device_error.  Nothing traps.
 *   - cpr_last_error() returns a thread-local message for the last failure.
 */
#ifndef CPR_GDN_H
#define CPR_GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------- */
#define CPR_OK                     0
#define CPR_ERR_INVALID_ARG        1  /* null/negative/inconsistent argument  */
#define CPR_ERR_UNSUPPORTED        2  /* valid contract this build cannot run */
#define CPR_ERR_ALIGNMENT          3  /* pointer not aligned as required      */
#define CPR_ERR_CONTRACT_MISMATCH  4  /* digest != SHA-256(contract), or a
                                         decode cache made under another
                                         contract (device-side)              */
#define CPR_ERR_UNALIGNED          5  /* a prefill that does not start on a
                                         chunk boundary                      */
#define CPR_ERR_CUDA               6  /* a CUDA runtime call failed           */
#define CPR_ERR_WORKSPACE          7  /* workspace null or too small          */
#define CPR_ERR_BAD_SEQLENS        8  /* cu_seqlens invalid (device-side)     */
#define CPR_ERR_DEVICE_TIMEOUT     9  /* a bounded device-side wait expired;
                                         the kernel gave up (device-side)     */
#define CPR_ERR_COMMIT_DUE        10  /* a no-commit decode step while some
                                         sequence completes its chunk
                                         (device-side; nothing written)       */

/* ---- contract --------------------------------------------------------- */
#define CPR_CONTRACT_VERSION 1u

#define CPR_DTYPE_F32  1u
#define CPR_DTYPE_BF16 2u

/* operand_policy: how the within-chunk contractions are evaluated.
 * SIMT_F32: every product and sum is an fp32 CUDA-core operation (fma
 * chains in the order fixed by intra_order); io values are widened exactly. */
#define CPR_POLICY_SIMT_F32 1u
/* TC_BF16X3: every within-chunk contraction is a 5th-generation tensor-core
 * MMA (tcgen05, kind::f16, fp32 accumulation).  bf16 inputs (q, k, v) enter
 * exactly; every fp32 operand x is split into bf16 hi = bf16(x) and
 * lo = bf16(x - hi) and a product of two split operands is the fixed
 * sequence hi*hi + hi*lo + lo*hi (one exact operand: hi + lo).  Gate prefix,
 * exponentials, the triangular solve and all epilogues are fp32 CUDA-core
 * operations.  Decode re-issues the same MMA instructions (same shapes, same
 * row positions) on the zero-padded partial chunk.  This build: bf16 io,
 * d_k = d_v = 128, dv_splits 2 or 4. */
#define CPR_POLICY_TC_BF16X3 2u

/* intra_order: id of the fixed within-chunk reduction orders.
 * ROWSEQ_V1: gate prefix = serial fp32 sum in token order; every dot product
 * an fma chain in ascending index order from +0; triangular solve by rows
 * with the inner sums ascending.                                           */
#define CPR_ORDER_ROWSEQ_V1 1u
/* TOKENREC_V1 (reading B of the pages' CPR wording): chunk-boundary states as
 * ROWSEQ_V1 computes them; every output of a chunk comes from the plain token
 * recurrence (H = a H + k u^T, u = b (v - a H^T k), o = H^T (scale q); fp32
 * fma chains in ascending row order per half of the rows, halves added in
 * order) started from hi + lo of the chunk's boundary-state operand tiles.
 * TC_BF16X3 only; forward, prefill and decode (no training ops).  Its decode
 * cache adds the running in-chunk state (cpr_cache_layout.run).  Page "IsoExec:
 * 切换 SkyRL 中的训练器-推理不匹配", section "Chunkwise-Parallel Recurrent (CPR)
 * Gated DeltaNet": the recurrence is primary and the state is resynchronised
 * every C tokens. */
#define CPR_ORDER_TOKENREC_V1 2u

/* state_schedule: how chunk states are produced.
 * SEQ_CHUNKS: H_{n+1} = f(H_n, chunk n) strictly in chunk order; d_v may be
 * split across independent CTAs (columns of H evolve independently).       */
#define CPR_SCHED_SEQ_CHUNKS 1u

typedef struct cpr_contract {
    uint32_t version;          /* CPR_CONTRACT_VERSION                          */
    uint32_t chunk_size;       /* C; this build: 64                             */
    uint32_t d_k;              /* this build: 64 or 128 (fp32 io: 64)           */
    uint32_t d_v;              /* this build: equal to d_k                      */
    uint32_t io_dtype;         /* q, k, v: CPR_DTYPE_BF16 or CPR_DTYPE_F32      */
    uint32_t out_dtype;        /* o, dq, dk, dv: CPR_DTYPE_F32                  */
    uint32_t gate_dtype;       /* g, beta, dg, dbeta: CPR_DTYPE_F32             */
    uint32_t accum_dtype;      /* CPR_DTYPE_F32                                 */
    uint32_t state_dtype;      /* chunk-boundary ("boundary dtype"): F32        */
    uint32_t operand_policy;   /* CPR_POLICY_*                                  */
    uint32_t intra_order;      /* CPR_ORDER_*                                   */
    uint32_t state_schedule;   /* CPR_SCHED_*                                   */
    uint32_t dv_splits;        /* CTAs per (seq, head) in the state pass: 1,2,4 */
    float    scale;            /* multiplies q; finite                          */
    uint32_t kernel_build_id;  /* must equal cpr_kernel_build_id()              */
} cpr_contract;

/* Identifier of this build's kernel arithmetic.  Bumped whenever any
 * rounding-relevant detail of a kernel changes. */
uint32_t cpr_kernel_build_id(void);

/* Fill *c with this build's default contract for the given io dtype and head
 * dims: C = 64, fp32 out/state/accumulation, ROWSEQ_V1, SEQ_CHUNKS, scale = 1;
 * operand policy TC_BF16X3 with dv_splits = 2 for bf16 io at d_k = d_v = 128
 * (the shape the tensor-core kernels cover), else SIMT_F32 with dv_splits = 4
 * for d_v = 128 and 2 below. */
int cpr_contract_init_default(cpr_contract* c, uint32_t io_dtype, uint32_t d_k, uint32_t d_v);

/* Canonical serialisation: the 16-byte tag "CPR-GDN-CONTRACT" followed by
 * the 15 fields in declaration order, each as 4 little-endian bytes (scale
 * as its IEEE-754 bit pattern) -- 76 bytes.  Writes the byte count to *len
 * and, if out != NULL and *len was large enough on entry, the bytes. */
int cpr_contract_serialize(const cpr_contract* c, uint8_t* out, size_t* len);

/* SHA-256 (FIPS 180-4) of the canonical serialisation: the contract's
 * numerical_policy identity. */
int cpr_contract_digest(const cpr_contract* c, uint8_t out[32]);

/* CPR_OK if this build can execute the contract, else INVALID_ARG or
 * UNSUPPORTED with a message in cpr_last_error(). */
int cpr_contract_check(const cpr_contract* c);

/* Plain SHA-256 of a byte string (exposed so callers and tests can check the
 * implementation against other SHA-256 implementations). */
int cpr_sha256(const void* data, size_t len, uint8_t out[32]);

/* Deployment identity (page "IsoExec: 切换 SkyRL 中的训练器-推理不匹配", section
 * "合约结构与强制执行": the contract's identities are SHA-256 digests, one of them over
 * the deployment the numerical policy runs on).  SHA-256 of the canonical text
 *   CPR-GDN-DEPLOYMENT;arch=sm_103a;cc=<major>.<minor>;gpu=<device name>;
 *   cudart=<runtime version>;driver=<driver version>;kernel_build_id=<id>
 * (one line, no spaces added) for the CURRENT device.  A decode cache carries the
 * deployment digest of the process that wrote it (header words 17..24); a decode
 * step on another deployment -- another build of this library, GPU model, CUDA
 * runtime or driver -- refuses it on the device like a foreign contract
 * (CPR_ERR_CONTRACT_MISMATCH recorded, nothing written).  Writes the digest to out
 * and, when text != NULL, the canonical text (truncated to text_len - 1 bytes,
 * NUL-terminated).  CPR_ERR_CUDA when no CUDA device is usable. */
int cpr_deployment_digest(uint8_t out[32], char* text, size_t text_len);

/* ---- workspace and decode cache sizes --------------------------------- */
#define CPR_OP_FWD 1   /* cpr_gdn_fwd and cpr_gdn_prefill */
#define CPR_OP_BWD 2   /* cpr_gdn_bwd, cpr_gdn_fwd_train, cpr_gdn_bwd_saved */

/* Bytes of device workspace an op needs for a batch with n_seq sequences and
 * n_tok tokens in total (an upper bound valid for any split of n_tok). */
int cpr_gdn_workspace_size(const cpr_contract* c, int op, int n_seq, int64_t n_tok, int H,
                           size_t* bytes);

/* Decode cache: one caller-owned device blob per batch of n_seq sequences.
 * It holds, per sequence, the position inside the current chunk and, per
 * (sequence, head), the chunk-start state H_n plus the rows of the current
 * partial chunk that the next decode steps need.  Sections (byte offsets
 * from the blob start, each 256-byte aligned) are reported by
 * cpr_decode_cache_layout. */
typedef struct cpr_cache_layout {
    size_t total_bytes;
    size_t header;      /* 256 B: magic, version, digest[32], n_seq, H, C, d_k, d_v */
    size_t pos;         /* int32  [n_seq]            tokens in the current chunk   */
    size_t done;        /* uint32 [n_seq]            internal step counter (zero)  */
    size_t state;       /* fp32   [n_seq, H, d_k, d_v] chunk-start state H_n      */
    size_t k_rows;      /* io     [n_seq, H, C, d_k]; tensor-core contracts keep each
                           (sequence, head) block as an operand tile: element (r, i) at
                           byte ((r/8)(d_k/8) + i/8) * 128 + (r%8) * 16 + (i%8) * 2, rows at
                           or past the position zero                              */
    size_t v_rows;      /* io     [n_seq, H, C, d_v]; same tile form as k_rows        */
    size_t gam_rows;    /* fp32   [n_seq, H, 2, C]   in-chunk gate prefix hi, lo   */
    size_t beta_rows;   /* fp32   [n_seq, H, C]                                    */
    size_t t_rows;      /* fp32   [n_seq, H, C, C]   rows of (I + A)^-1            */
    size_t delta_rows;  /* fp32   [n_seq, H, C, d_v] rows of Delta                 */
    size_t state_tiles; /* bf16   [n_seq, H] x 64 KB: H_n as hi/lo tensor-core operand
                           tiles (tensor-core contracts; the fp32 copy stays authoritative) */
    size_t delta_tiles; /* bf16   [n_seq, H] x 32 KB: the Delta rows as hi/lo operand tiles */
    size_t run;         /* fp32   [n_seq, H, d_k, d_v] running in-chunk state (TOKENREC_V1
                           contracts; 0 and absent otherwise)                     */
    /* TOKENREC_V1 contracts only (0 and absent otherwise): the current chunk's token rows,
       token-major (row b * C + r of sequence b), which the decode step appends to and the
       chunk commit reads, and the commit's own scratch: */
    size_t rb_k;        /* io     [n_seq * C, H, d_k]                              */
    size_t rb_v;        /* io     [n_seq * C, H, d_v]                              */
    size_t rb_g;        /* fp32   [n_seq * C, H]                                   */
    size_t rb_beta;     /* fp32   [n_seq * C, H]                                   */
    size_t rb_cu;       /* int32  [n_seq + 1]  b * C                               */
    size_t rb_ws;       /* the forward workspace of a batch of n_seq full chunks   */
} cpr_cache_layout;

int cpr_decode_cache_layout(const cpr_contract* c, int n_seq, int H, cpr_cache_layout* out);
int cpr_decode_cache_bytes(const cpr_contract* c, int n_seq, int H, size_t* bytes);

/* ---- compute entry points ---------------------------------------------- */

/* Trainer forward (case trainer_fwd).  h0 and final_state may be NULL (h0 =
 * zeros; final state not written).  o is required.  workspace: at least
 * cpr_gdn_workspace_size(c, CPR_OP_FWD, ...) bytes, 256-byte aligned.
 * Under intra_order TOKENREC_V1 (reading B) the chunk-form forward keeps every
 * chunk's boundary state in the workspace and each chunk's o is then the
 * token recurrence from it (chunks independent); the final state is the chunk
 * form's. */
int cpr_gdn_fwd(const cpr_contract* c, const uint8_t digest[32],
                const void* q, const void* k, const void* v, const float* g, const float* beta,
                const int32_t* cu_seqlens, int n_seq, int64_t n_tok, int H,
                const float* h0, void* o, float* final_state,
                void* workspace, size_t workspace_bytes, void* stream);

/* Rollout prefill (case engine_prefill): the same arithmetic as cpr_gdn_fwd
 * and, with the required cache, also initialises a decode cache (header with
 * the digest, per-sequence position, the chunk-start state of each
 * sequence's last chunk and that chunk's rows), so decoding continues exactly
 * where the prefill stopped.  Every sequence starts on a chunk boundary (h0
 * is the state at that boundary); a caller that continues a sequence from a
 * cache whose position is not 0 must decode up to the boundary first.  Under
 * TOKENREC_V1 the cache also receives the in-chunk state after each
 * sequence's partial last chunk (cpr_cache_layout.run). */
int cpr_gdn_prefill(const cpr_contract* c, const uint8_t digest[32],
                    const void* q, const void* k, const void* v, const float* g,
                    const float* beta, const int32_t* cu_seqlens, int n_seq, int64_t n_tok,
                    int H, const float* h0, void* o, float* final_state, void* cache,
                    void* workspace, size_t workspace_bytes, void* stream);

/* One decode step (case decode) for n_seq sequences, one token each:
 * q_t, k_t [n_seq, H, d_k], v_t [n_seq, H, d_v] (io dtype), g_t, beta_t
 * [n_seq, H] fp32, o_t [n_seq, H, d_v] (out dtype).  Uses the same per-row
 * arithmetic as the prefill's chunk kernels, so o_t and every committed
 * chunk-boundary state equal a one-shot prefill's bits.  When a chunk fills,
 * the step commits H_{n+1} into the cache (the resynchronisation every C
 * tokens).  The cache's stored digest is checked on the device; on mismatch
 * nothing is written and CPR_ERR_CONTRACT_MISMATCH is recorded.  Under
 * TOKENREC_V1 the same step keeps the cache, then one token of the recurrence
 * advances the running in-chunk state (restarted at a chunk's first row from
 * hi + lo of the cache's chunk-start state tiles) and gives o_t: bit-identical
 * to cpr_gdn_fwd over the same tokens under that contract. */
int cpr_gdn_decode_step(const cpr_contract* c, const uint8_t digest[32],
                        const void* q_t, const void* k_t, const void* v_t, const float* g_t,
                        const float* beta_t, int n_seq, int H, void* cache, void* o_t,
                        void* stream);

/* cpr_gdn_decode_step for a step in which the caller knows that no sequence
 * completes its chunk (no sequence's position is C - 1 before the step; the
 * caller knows its sequences' lengths).  Under TOKENREC_V1 the chunk-form
 * commit is then not launched at all, which leaves the token recurrence's step
 * alone in C - 1 of every C steps.  The claim is checked on the device against
 * every sequence's position: if some sequence would complete its chunk, nothing
 * is written, no position moves, and CPR_ERR_COMMIT_DUE is recorded.  Under
 * reading A (whose step commits inside its own kernel) it is
 * cpr_gdn_decode_step.  Same arguments, results and bits as
 * cpr_gdn_decode_step. */
int cpr_gdn_decode_step_nocommit(const cpr_contract* c, const uint8_t digest[32],
                                 const void* q_t, const void* k_t, const void* v_t,
                                 const float* g_t, const float* beta_t, int n_seq, int H,
                                 void* cache, void* o_t, void* stream);

/* Trainer backward of cpr_gdn_fwd for the loss  <dO, o> + <dHT, final>.
 * dHT and h0 may be NULL (zeros).  Outputs dq, dk [n_tok,H,d_k], dv
 * [n_tok,H,d_v] (out dtype), dg, dbeta [n_tok,H] fp32, dh0 [n_seq,H,d_k,d_v]
 * fp32 are all required.  workspace: cpr_gdn_workspace_size(c, CPR_OP_BWD). */
int cpr_gdn_bwd(const cpr_contract* c, const uint8_t digest[32],
                const void* q, const void* k, const void* v, const float* g, const float* beta,
                const int32_t* cu_seqlens, int n_seq, int64_t n_tok, int H,
                const float* h0, const float* dO, const float* dHT,
                void* dq, void* dk, void* dv, float* dg, float* dbeta, float* dh0,
                void* workspace, size_t workspace_bytes, void* stream);

/* Training forward: the outputs of cpr_gdn_fwd (same arithmetic, same bits)
 * and, in the workspace, the per-chunk tiles the backward reads (chunk-start
 * states, Delta, (I + A)^-1 and the operand tiles), so that
 * cpr_gdn_bwd_saved need not recompute the forward -- the trainer's
 * forward-then-backward step of the stage table (page "IsoExec: 切换 SkyRL
 * 中的训练器-推理不匹配", section "Chunkwise-Parallel Recurrent (CPR) Gated
 * DeltaNet", "Trainer Fwd+Bwd").  workspace: cpr_gdn_workspace_size(c,
 * CPR_OP_BWD, ...) bytes, 256-byte aligned, owned by the caller until the
 * matching cpr_gdn_bwd_saved has run.  CPR_POLICY_TC_BF16X3 contracts only
 * (CPR_ERR_UNSUPPORTED otherwise).  The training ops (this one, cpr_gdn_bwd,
 * cpr_gdn_bwd_saved) refuse intra_order TOKENREC_V1 with CPR_ERR_UNSUPPORTED. */
int cpr_gdn_fwd_train(const cpr_contract* c, const uint8_t digest[32],
                      const void* q, const void* k, const void* v, const float* g,
                      const float* beta, const int32_t* cu_seqlens, int n_seq, int64_t n_tok,
                      int H, const float* h0, void* o, float* final_state,
                      void* workspace, size_t workspace_bytes, void* stream);

/* Backward from a training forward's workspace: the same arguments and
 * results as cpr_gdn_bwd, but the forward is not recomputed; `workspace`
 * must be the one cpr_gdn_fwd_train filled for the same contract, inputs and
 * h0, unchanged since (the library cannot check this).  Results are
 * bit-identical to cpr_gdn_bwd's.  CPR_POLICY_TC_BF16X3 contracts only. */
int cpr_gdn_bwd_saved(const cpr_contract* c, const uint8_t digest[32],
                      const void* q, const void* k, const void* v, const float* g,
                      const float* beta, const int32_t* cu_seqlens, int n_seq, int64_t n_tok,
                      int H, const float* h0, const float* dO, const float* dHT,
                      void* dq, void* dk, void* dv, float* dg, float* dbeta, float* dh0,
                      void* workspace, size_t workspace_bytes, void* stream);

/* Allocation-free trainer forward.  The pages have no counterpart for this
 * entry point: it exists for callers that cannot allocate device memory at
 * the point of the call -- for example code running inside a host callback or
 * a custom allocator hook, where cudaMalloc is forbidden or would deadlock, or
 * embedders whose memory pools are fixed at start-up and have no room for a
 * per-call workspace.
 *
 * Same arguments and result bits as cpr_gdn_fwd minus the workspace: the
 * scratch lives in a fixed device array of CPR_NOALLOC_SCRATCH_BYTES inside
 * this library (every GPU that loads the library holds it until the process
 * exits).  A batch whose forward workspace (cpr_gdn_workspace_size with
 * CPR_OP_FWD) exceeds that size is rejected with CPR_ERR_WORKSPACE before
 * anything is launched.  The first call on a device looks up the array's
 * device address with that device current; make that first call before any
 * stream capture.  The address is kept per device and looked up again when the
 * device's context has changed since (cudaDeviceReset destroys the context and
 * the module that holds the array), so the first call after a reset is again a
 * first call in this sense.  All calls share the one array and it keeps the last
 * call's contents (the forward writes every scratch word before reading it,
 * so nothing needs clearing); calls that overlap on the GPU -- on two streams,
 * or from two host threads -- race on it and must be serialised by the
 * caller.  Allocates nothing (no cudaMalloc / cudaFree). */
#define CPR_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
int cpr_gdn_fwd_noalloc(const cpr_contract* c, const uint8_t digest[32],
                        const void* q, const void* k, const void* v, const float* g,
                        const float* beta, const int32_t* cu_seqlens, int n_seq, int64_t n_tok,
                        int H, const float* h0, void* o, float* final_state, void* stream);

/* ---- kernel timing ------------------------------------------------------ */

/* Per-kernel timing collected with CUDA events recorded on the launching
 * stream around every kernel this library launches between
 * cpr_profile_begin and cpr_profile_end (process-wide).  Recording adds one
 * event pair per launch; results are per kernel name. */
typedef struct cpr_kernel_time {
    char name[40];
    uint32_t launches;
    double total_ms;
} cpr_kernel_time;

/* Starts recording (discarding earlier records). */
int cpr_profile_begin(void);

/* Stops recording, SYNCHRONISES the device, and writes up to max_entries
 * per-kernel totals to out (*n_entries = number of distinct kernels). */
int cpr_profile_end(cpr_kernel_time* out, int max_entries, int* n_entries);

/* ---- errors ------------------------------------------------------------ */

/* Reads (and, if clear != 0, resets) the device error word of the current
 * device.  SYNCHRONISES the device.  *code = CPR_OK if no kernel recorded an
 * error since the last clear. */
int cpr_get_device_error(uint32_t* code, int clear);

/* Thread-local message describing the last non-OK return on this thread. */
const char* cpr_last_error(void);

/* Test support for the device-side failure path.  Every wait of the kernels on
 * an mbarrier (an async copy or MMA completing) polls at most a fixed number of
 * times; on expiry the kernel records CPR_ERR_DEVICE_TIMEOUT in the device error
 * word, lets its own copies and MMAs finish (bounded), frees its tensor memory
 * and returns.  This call runs that path for real: one thread waits, with
 * `poll_limit` polls, on an mbarrier nothing arrives on.  It allocates 4 bytes of
 * device memory, synchronises the device, and sets *completed to 0 when the
 * wait ran out (the expected result); CPR_ERR_DEVICE_TIMEOUT is then readable
 * with cpr_get_device_error. */
int cpr_selftest_wait_timeout(uint32_t poll_limit, uint32_t* completed);

/* ---- stage-table ablations (outside the CPR guarantee) -------------------
 * The gated delta rule run as a plain token recurrence, the engines' native
 * decode that CPR replaces (page "IsoExec: 切换 SkyRL 中的训练器-推理不匹配",
 * section "Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet", stage table:
 * "native mixed" = chunked prefill + token-recurrent decode without
 * resynchronisation; "recurrent everywhere").  Per token, with H = S^T:
 * H_t = a H + k u^T, u = b (v - a H^T k), a = exp(g), o_t = H_t^T (scale q),
 * every sum an fp32 fma chain in a fixed order, so the two calls below agree
 * bit for bit with each other; they do not agree bit for bit with the chunked
 * path (which is the point of the comparison).  No digest: these calls make
 * no cross-path promise.  The contract gives d_k = d_v (64 or 128), the io
 * dtype (bf16 or fp32) and scale.  Pointers: device, 16-byte aligned (g and
 * beta 4-byte); layouts as cpr_gdn_fwd; o is fp32.  Errors: CPR_ERR_INVALID_ARG,
 * CPR_ERR_ALIGNMENT, CPR_ERR_UNSUPPORTED (d_k != d_v or d not 64/128), and
 * CPR_ERR_BAD_SEQLENS on the device word for a sequence outside [0, n_tok]. */

/* Token recurrence over whole sequences ("recurrent everywhere"): o for every
 * token and, if final_state is not NULL, the final state.  h0 may be NULL. */
int cpr_gdn_recurrent_fwd(const cpr_contract* c, const void* q, const void* k, const void* v,
                          const float* g, const float* beta, const int32_t* cu_seqlens,
                          int n_seq, int64_t n_tok, int H, const float* h0, float* o,
                          float* final_state, void* stream);

/* One token per sequence on an fp32 state [n_seq, H, d_k, d_v] updated in
 * place (the native decode step); q_t..beta_t as cpr_gdn_decode_step. */
int cpr_gdn_recurrent_step(const cpr_contract* c, const void* q_t, const void* k_t,
                           const void* v_t, const float* g_t, const float* beta_t, int n_seq,
                           int H, float* state, float* o_t, void* stream);

/* Backward of cpr_gdn_recurrent_fwd ("recurrent everywhere" training): the adjoint
 * of each token update, walked from the last token back (the reverse recurrence:
 * Shat += do q^T, dq = scale S_t^T do, e = v - a S_{t-1} k, sk = Shat k, dv = b sk,
 * dbeta = e . sk, dk = b Shat^T e - a b S_{t-1}^T sk, dg = a (<Shat, S_{t-1}> - b sk .
 * S_{t-1} k), Shat = a (Shat - b sk k^T); dh0 = the final Shat^T).  S_{t-1} and S_t are
 * the recurrent forward's states bit for bit, recomputed from checkpoints the call
 * keeps every 16 tokens in `workspace` (cpr_gdn_recurrent_bwd_workspace_size bytes,
 * 256-byte aligned, caller-owned).  h0, dHT may be NULL (zeros).  dO and every
 * gradient are fp32 in the layouts of cpr_gdn_bwd; deterministic, one CTA per
 * (sequence, head).  Errors as cpr_gdn_recurrent_fwd, plus CPR_ERR_WORKSPACE. */
int cpr_gdn_recurrent_bwd_workspace_size(const cpr_contract* c, int n_seq, int64_t n_tok, int H,
                                         size_t* bytes);
int cpr_gdn_recurrent_bwd(const cpr_contract* c, const void* q, const void* k, const void* v,
                          const float* g, const float* beta, const int32_t* cu_seqlens,
                          int n_seq, int64_t n_tok, int H, const float* h0, const float* dO,
                          const float* dHT, float* dq, float* dk, float* dv, float* dg,
                          float* dbeta, float* dh0, void* workspace, size_t workspace_bytes,
                          void* stream);

/* ---- batch-invariant projection GEMM ------------------------------------
 * Y = X W for the projections that feed the CPR layer (page "IsoExec: 切换
 * SkyRL 中的训练器-推理不匹配": batch-invariant kernels for everything around
 * the layer, so a token's inputs do not change with its batch).  X bf16 [M, K],
 * W bf16 [K, N], Y fp32 [M, N], all row-major, device, X and W 16-byte and
 * Y 32-byte aligned.  K is split into K / leaf_k contiguous leaves (leaf_k a
 * multiple of 64; 1, 2 or 4 leaves); each leaf is accumulated in fp32 by
 * tensor-core MMAs in ascending
 * k and the leaves are added in the fixed tree (P0 + P1) + (P2 + P3).  A row's
 * result depends only on that row of X, on W and on leaf_k: it is the same for
 * any M and any batch the row sits in.  N must be a multiple of 128.  Errors:
 * CPR_ERR_INVALID_ARG (shapes, leaf_k, NULL), CPR_ERR_ALIGNMENT; a bounded
 * device wait that runs out records CPR_ERR_DEVICE_TIMEOUT. */
int cpr_gemm_bf16(const void* X, const void* W, float* Y, int M, int N, int K, int leaf_k,
                  void* stream);

#ifdef __cplusplus
}
#endif
#endif /* CPR_GDN_H */
