/*
 * kda.h -- C ABI of libkda, the GB300 (sm_103a) forward pass of Kimi Delta
 * Attention (KDA).
 *
 * What the library computes (cited by page title and section):
 *   "Kimi K3" article, lshu.cn/news/263999, §四: per head, a d_k x d_v state
 *       S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,
 *   with a per-key-channel decay alpha_t = exp(log_alpha_t) in (0,1]^{d_k};
 *   §二.1: the read o_t = S_t^T q_t (after token t's update, no 1/sqrt(d) scale);
 *   §三: the delta-rule reading of the same update (predict from the decayed
 *   state, write beta times the error);
 *   §六: the chunkwise evaluation (recurrent between chunks, WY form inside).
 *   "Kimi K3 混合线性注意力", hubwiz.com, §3: the state is 128 x 128 per head
 *   and independent of the sequence length; §5: state snapshots at fixed token
 *   intervals make a long run restartable and its prefixes reusable.
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *     never allocates, frees or keeps a pointer after the call returns.
 *   - Layouts are row-major and token-major:
 *       q, k        [.., H, d_k]   (in_dtype: KDA_BF16 or KDA_F32)
 *       v           [.., H, d_v]   (in_dtype)
 *       log_alpha   [.., H, d_k]   float32, <= 0 (-inf allowed in the forward calls:
 *                                  alpha = 0; the backward wants finite values)
 *       beta        [.., H]        float32
 *       state       [.., H, d_k, d_v] float32, row i = key channel i
 *       out         [.., H, d_v]   (out_dtype)
 *     where ".." is [B, T] for the batched prefill, [T_total] for packed
 *     sequences and [B] for decode.
 *   - Supported sizes: d_k = d_v = 128.  chunk = 64 (tensor-core chunked
 *     path) or chunk = 1 (token-serial path).  Anything else returns
 *     KDA_ERR_UNSUPPORTED.
 *   - Alignment (KDA_ERR_MISALIGNED otherwise): q, k, v, log_alpha, out and
 *     every state/snapshot pointer of the prefill calls 16 bytes (tensor-map
 *     loads); the state of both decode calls 16 bytes; beta 4 bytes; cu_seqlens
 *     and snap_offsets 8 bytes; the other decode operands their element size.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream).  A return of KDA_OK means the work was enqueued.
 *     Faults found inside a kernel (a bounded wait that ran out, a state-pool
 *     slot out of range) are recorded in a device status word, never by a
 *     trap; read them with kda_get_device_status().
 *   - No C++ exception crosses this boundary.  Results are bit-reproducible
 *     from run to run on the same GPU.
 *   - Numerics of the chunk = 64 path: tensor-core products take fp16 operands
 *     with fp32 accumulation; the state and every carry are fp32.  Decay
 *     factors are taken relative to the log-decay after a chunk's first 32
 *     tokens, which keeps every fp16 operand within 2^10 of its undecayed
 *     value while, in every 64-token chunk, the summed log_alpha of tokens
 *     1..31 and of tokens 32..63 are each >= -10 ln 2 (about -6.9) per key
 *     channel.  That covers gates down to a mean of about -0.2 per token.  A
 *     (sequence, head) with any chunk beyond that bound is marked by the kernel
 *     and recomputed within the same call by a second pass of the same kernel,
 *     in which each chunk within the bound goes through the same products (bit
 *     for bit) and each chunk beyond it applies its tokens one at a time in
 *     fp32 (exact for any alpha).  So every log_alpha <= 0 is supported,
 *     including -inf (alpha = 0); only the speed of such units differs, and
 *     since a chunk's path depends on its own gates only, runs resumed at chunk
 *     boundaries and snapshots stay bit-exact.  The chunked backward recomputes
 *     units beyond its fp32 bound (-80 per half-chunk) with the token-serial
 *     backward.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types of q/k/v (in_dtype) and of out (out_dtype). */
typedef enum { KDA_BF16 = 0, KDA_F32 = 1 } kda_dtype;

/* Return codes of every entry point. */
typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1, /* null required pointer, negative size, bad enum */
    KDA_ERR_UNSUPPORTED = 2, /* d_k, d_v or chunk outside the supported set */
    KDA_ERR_MISALIGNED = 3,  /* a pointer is not 16-byte aligned */
    KDA_ERR_CUDA = 4,        /* a CUDA runtime/driver call or a launch failed */
    KDA_ERR_TIMEOUT = 5,     /* device status: a bounded wait inside a kernel expired */
    KDA_ERR_WORKSPACE = 6,   /* workspace missing or smaller than kda_workspace_size() */
    KDA_STATUS_GATE_RANGE = 7, /* no longer raised: units whose gates leave the chunked kernels' range are
                                  recomputed exactly within the same call (the code is kept for the ABI) */
    KDA_STATUS_SLOT_RANGE = 8, /* device status: a state-pool slot index outside [-1, pool_slots) was skipped */
    KDA_ERR_SCRATCH_TOO_SMALL = 9 /* the problem needs more than the library's static scratch (kda_bwd_noalloc) */
} kda_status;

/* Operation selector of kda_workspace_size(). */
typedef enum { KDA_OP_CHUNK = 0, KDA_OP_VARLEN = 1, KDA_OP_DECODE = 2, KDA_OP_BWD = 3, KDA_OP_CHUNK_BWD = 4 } kda_op;

/* Layout of log_alpha for kda_varlen_fwd_pool: one value per key channel (KDA), one per head
   (Gated DeltaNet), or none (DeltaNet, log_alpha NULL).  See kda_gdn_chunk_fwd. */
typedef enum { KDA_GATE_CHANNEL = 0, KDA_GATE_HEAD = 1, KDA_GATE_NONE = 2 } kda_gate;

/*
 * Batched prefill: B independent sequences of T tokens, H heads each.
 * "Kimi K3" article (lshu.cn/news/263999) §四 recurrence, evaluated chunkwise
 * as in §六.
 *   q, k        [B, T, H, dk]  in_dtype
 *   v           [B, T, H, dv]  in_dtype
 *   log_alpha   [B, T, H, dk]  float32
 *   beta        [B, T, H]      float32
 *   init_state  [B, H, dk, dv] float32, or NULL for a zero initial state
 *   out         [B, T, H, dv]  out_dtype, o_t = S_t^T q_t
 *   final_state [B, H, dk, dv] float32, or NULL if not wanted
 *   workspace   device scratch of at least kda_workspace_size(KDA_OP_CHUNK, ...)
 *               bytes, 16-byte aligned (chunk = 64: one int per (sequence, head),
 *               rounded up to 256 bytes, marking the units the exact pass
 *               recomputes, then 256 bytes of counters with which the CTAs of a
 *               launch with fewer (sequence, head) units than SMs claim their
 *               units; chunk = 1: 0 bytes, may be NULL); contents need no
 *               initialisation and are not preserved.
 * B, T or H equal to 0 is valid (nothing to compute; with T = 0 the final
 * state is the initial state).  init_state may alias final_state.
 */
int kda_chunk_fwd(const void* q, const void* k, const void* v, const float* log_alpha, const float* beta,
                  const float* init_state, void* out, float* final_state, int B, int64_t T, int H, int dk,
                  int dv, int chunk, int in_dtype, int out_dtype, void* workspace, size_t ws_bytes,
                  void* stream);

/*
 * Packed variable-length prefill with state snapshots ("Kimi K3 混合线性注意力",
 * hubwiz.com, §5: restartable checkpoints of the recurrent state).
 *   q, k, v, log_alpha, beta, out : token-major over T_total packed tokens,
 *               shapes as in kda_chunk_fwd with [B, T] replaced by [T_total].
 *   cu_seqlens  device int64 [N+1], cu_seqlens[0] = 0, non-decreasing,
 *               cu_seqlens[N] = T_total; sequence s is tokens
 *               [cu_seqlens[s], cu_seqlens[s+1]).
 *   init_states [N, H, dk, dv] float32, or NULL for zero initial states.
 *   final_states[N, H, dk, dv] float32 (required).
 *   snapshot_interval  0 for none, else a positive multiple of `chunk`:
 *               snapshot m (m = 1 .. floor(len_s / interval)) of sequence s is
 *               the state right after its token m * interval (counted from the
 *               sequence start) and is stored at
 *               snapshots[snap_offsets[s] + m - 1][H][dk][dv].  When len_s is a
 *               multiple of the interval, the last snapshot equals the final
 *               state bit for bit.
 *   snap_offsets device int64 [N+1] from kda_snapshot_offsets() (copied to the
 *               device by the caller); NULL when snapshot_interval = 0.
 *   snapshots   float32 [snap_offsets[N], H, dk, dv]; NULL when no snapshot (a NULL
 *               array with snapshot positions present stores nothing).
 * Chunks are aligned to each sequence's first token; each sequence's result
 * is bit-identical to running that sequence alone through this function.
 */
int kda_varlen_fwd(const void* q, const void* k, const void* v, const float* log_alpha, const float* beta,
                   const int64_t* cu_seqlens, int N, int64_t T_total, int H, int dk, int dv, int chunk,
                   const float* init_states, float* final_states, int64_t snapshot_interval,
                   const int64_t* snap_offsets, float* snapshots, void* out, int in_dtype, int out_dtype,
                   void* workspace, size_t ws_bytes, void* stream);

/*
 * One decode step for B sessions (one new token each), state updated in place:
 * "Kimi K3" article §四 applied once; the state is read once and written once.
 *   q, k [B, H, dk] in_dtype;  v [B, H, dv] in_dtype;
 *   log_alpha [B, H, dk] float32;  beta [B, H] float32;
 *   state [B, H, dk, dv] float32, read and overwritten;
 *   out [B, H, dv] out_dtype.
 */
int kda_decode_step(const void* q, const void* k, const void* v, const float* log_alpha, const float* beta,
                    float* state, void* out, int B, int H, int dk, int dv, int in_dtype, int out_dtype,
                    void* stream);

/*
 * kda_decode_step with the state STORED in bf16 (halving the state bytes each
 * step moves; the state is the whole memory of a session, "Kimi K3 混合线性注意力",
 * hubwiz.com, §3, so its storage precision is a serving choice).  Arguments as
 * for kda_decode_step except
 *   state [B, H, dk, dv] bf16 (raw 16-bit storage), read and overwritten.
 * Each element is widened exactly to fp32, the whole step runs in fp32, o_t is
 * read from the updated state BEFORE rounding, and the new state is then stored
 * rounded to nearest-even bf16.
 */
int kda_decode_step_bf16state(const void* q, const void* k, const void* v, const float* log_alpha,
                              const float* beta, void* state, void* out, int B, int H, int dk, int dv,
                              int in_dtype, int out_dtype, void* stream);

/*
 * The same three operations with a coarser gate.  "Kimi K3" article, §四: Gated
 * DeltaNet decays the whole state of a head by ONE scalar alpha_t per token,
 *     S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,
 * which KDA refines into one alpha per key channel; with a scalar, decaying
 * before or after the delta step is the same operator.  §三: with no gate at
 * all (alpha_t = 1) the update is the plain delta rule (DeltaNet).
 *   log_alpha  float32 with ONE value per (token, head): [B, T, H] for
 *              kda_gdn_chunk_fwd, [T_total, H] for kda_gdn_varlen_fwd, [B, H] for
 *              kda_gdn_decode_step; 4-byte aligned; finite and <= 0.
 *              NULL selects DeltaNet (alpha = 1 everywhere).
 * Every other argument, the layouts, the snapshot rules, the results' bit-exact
 * reproducibility and the error codes are those of kda_chunk_fwd,
 * kda_varlen_fwd and kda_decode_step.  The chunked path's gate bound, and the
 * exact recomputation of the units beyond it, apply to the scalar gate in the same way.
 */
int kda_gdn_chunk_fwd(const void* q, const void* k, const void* v, const float* log_alpha, const float* beta,
                      const float* init_state, void* out, float* final_state, int B, int64_t T, int H, int dk,
                      int dv, int chunk, int in_dtype, int out_dtype, void* workspace, size_t ws_bytes,
                      void* stream);
int kda_gdn_varlen_fwd(const void* q, const void* k, const void* v, const float* log_alpha, const float* beta,
                       const int64_t* cu_seqlens, int N, int64_t T_total, int H, int dk, int dv, int chunk,
                       const float* init_states, float* final_states, int64_t snapshot_interval,
                       const int64_t* snap_offsets, float* snapshots, void* out, int in_dtype, int out_dtype,
                       void* workspace, size_t ws_bytes, void* stream);
int kda_gdn_decode_step(const void* q, const void* k, const void* v, const float* log_alpha, const float* beta,
                        float* state, void* out, int B, int H, int dk, int dv, int in_dtype, int out_dtype,
                        void* stream);
/* kda_gdn_decode_step with the state stored in bf16, as in kda_decode_step_bf16state. */
int kda_gdn_decode_step_bf16state(const void* q, const void* k, const void* v, const float* log_alpha,
                                  const float* beta, void* state, void* out, int B, int H, int dk, int dv,
                                  int in_dtype, int out_dtype, void* stream);

/*
 * Packed variable-length prefill over a caller-owned STATE POOL, for prefix reuse in
 * serving ("Kimi K3 混合线性注意力", hubwiz.com, §5: restartable state snapshots at a
 * fixed token interval; a prompt that shares a prefix resumes from the nearest snapshot
 * instead of recomputing it, with the snapshot block size decoupled from the
 * granularity of prefix matching).  Arguments as for kda_varlen_fwd, except:
 *   gate        kda_gate: the layout of log_alpha ([T_total, H, dk], [T_total, H] or NULL).
 *   pool        [pool_slots, H, dk, dv] of pool_dtype, 16-byte aligned; slot i holds the
 *               states of all H heads at one position of one sequence.
 *   pool_dtype  KDA_F32, or KDA_BF16 for a pool that stores states in bf16 ([hubwiz] §3
 *               sizes the state in bf16): initial states are widened exactly to fp32 and
 *               snapshots are the fp32 states rounded to nearest-even bf16, which halves
 *               the pool's memory; the arithmetic stays fp32.
 *   init_slots  device int64 [N] or NULL: sequence s starts from slot init_slots[s]
 *               (-1: zero state).  NULL: every sequence starts from zeros.
 *   snap_slots  device int64 [snap_offsets[N]]: snapshot m of sequence s (as in
 *               kda_varlen_fwd) is stored into slot snap_slots[snap_offsets[s] + m - 1];
 *               -1 means "not stored" (for example because that prefix is already in
 *               the pool).  NULL stores no snapshot (as when there are none to store).
 * final_states stays a dense [N, H, dk, dv] array.  Snapshot slots written by one call
 * must be distinct, and no slot written by a call may be an initial-state slot of the
 * same call.  A slot index outside [-1, pool_slots) is not dereferenced: the state is
 * taken as zero, or the snapshot is dropped, and KDA_STATUS_SLOT_RANGE is raised in the
 * device status word.  Results are bit-identical to kda_varlen_fwd (or
 * kda_gdn_varlen_fwd) with the same states gathered into packed fp32 arrays (a bf16
 * pool: the widened states in, the snapshots rounded out); with
 * kda_snapshot_lookup, a resumed sequence reproduces the unsplit run bit for bit.
 */
int kda_varlen_fwd_pool(const void* q, const void* k, const void* v, const float* log_alpha, int gate,
                        const float* beta, const int64_t* cu_seqlens, int N, int64_t T_total, int H, int dk, int dv,
                        int chunk, void* pool, int64_t pool_slots, int pool_dtype, const int64_t* init_slots,
                        int64_t snapshot_interval, const int64_t* snap_offsets, const int64_t* snap_slots,
                        float* final_states, void* out, int in_dtype, int out_dtype, void* workspace,
                        size_t ws_bytes, void* stream);

/*
 * Gradients for training ("Kimi Linear 最多砍掉 75% KV Cache", ai.concitech.org: the
 * chunkwise kernel serves training; the pages give no backward).  For the loss
 *     L = sum_t <d_out_t, o_t> + sum_s <d_final_states_s, S_final_s>
 * through the recurrence of kda_chunk_fwd (gate layout `gate`, as in kda_varlen_fwd_pool),
 * returns dL/dq, dL/dk, dL/dv, dL/dlog_alpha, dL/dbeta and dL/dinit_states, each in the
 * layout of its input, in float32.  Derived as the reverse mode of the per-token step.
 *   cu_seqlens  NULL: N sequences of T tokens each, batched [N, T, H, ..] layout;
 *               else device int64 [N+1] of packed sequences and T = T_total.
 *   init_states [N, H, dk, dv] float32 or NULL (zeros); d_final_states likewise (no
 *               loss on the final state); d_init_states may be NULL (not returned).
 *   d_out       [.., H, dv] float32.  q, k, v in in_dtype; everything else float32.
 *   dlog_alpha  [.., H, dk] (KDA_GATE_CHANNEL), [.., H] (KDA_GATE_HEAD), NULL (KDA_GATE_NONE).
 *   workspace   device, kda_workspace_size(KDA_OP_BWD, N, T_total, H, dk, dv, 64) bytes,
 *               16-byte aligned: a state checkpoint every 64 tokens of every head, and
 *               a small per-(sequence, head) recomputation area.
 * Evaluated token by token in fp32 (the state and its gradient of each (sequence,
 * head) stay in one CTA's registers), with states recomputed from the checkpoints;
 * deterministic.  Alignment: 16 bytes for the state arrays and the workspace, element
 * size for the rest.
 */
int kda_bwd(const void* q, const void* k, const void* v, const float* log_alpha, int gate, const float* beta,
            const float* init_states, const float* d_out, const float* d_final_states, const int64_t* cu_seqlens,
            int N, int64_t T, int H, int dk, int dv, float* dq, float* dk_out, float* dv_out, float* dlog_alpha,
            float* dbeta, float* d_init_states, int in_dtype, void* workspace, size_t ws_bytes, void* stream);

/*
 * kda_bwd evaluated in chunks.  Same arguments, loss and results as kda_bwd, plus `chunk`:
 *   chunk = 64  the chunked reverse mode of the §六.2 WY form ("Kimi K3" article,
 *               lshu.cn/news/263999): the chunk-local products and all input gradients
 *               run chunk-parallel as GEMMs on shared-memory tiles; only the
 *               chunk-to-chunk state and state-gradient recurrences (two dependent
 *               products per chunk) are serial per (sequence, head): one CTA per unit
 *               with the products on tcgen05 and TMEM accumulators, or, when the units
 *               fill at most a quarter of the SMs, warp-level products with each unit's
 *               value columns split over 4 CTAs.  Every product runs on the tensor
 *               cores with each fp32 operand split into bf16 hi + lo (three products,
 *               fp32 accumulation: about 16 significant bits per operand); every
 *               element-wise step is fp32; deterministic for a given device and shape.  Each chunk factors its decays about its 32nd row, which
 *               stays in fp32 range while every half-chunk's summed log-decay is >= -80;
 *               a (sequence, head) with a chunk beyond that is recomputed in the same
 *               call by the token-serial backward (chunk = 1), so every finite gate is
 *               supported.
 *               q, k, v and d_out must be 16-byte aligned (KDA_ERR_MISALIGNED otherwise).
 *   chunk = 1   the token-serial evaluation of kda_bwd (no gate limit).
 *   workspace   device, kda_workspace_size(KDA_OP_CHUNK_BWD, N, T_total, H, dk, dv, chunk)
 *               bytes, 16-byte aligned.  For chunk = 64 it holds every chunk's local
 *               products, state and state gradient: about 5.2 KB per (token, head)
 *               (about 5.4 GB at N=4, T=8192, H=32), and at least the token-serial
 *               backward's workspace, which the recomputation reuses.
 * Returns KDA_ERR_UNSUPPORTED for any other chunk.
 */
int kda_chunk_bwd(const void* q, const void* k, const void* v, const float* log_alpha, int gate, const float* beta,
                  const float* init_states, const float* d_out, const float* d_final_states,
                  const int64_t* cu_seqlens, int N, int64_t T, int H, int dk, int dv, int chunk, float* dq,
                  float* dk_out, float* dv_out, float* dlog_alpha, float* dbeta, float* d_init_states, int in_dtype,
                  void* workspace, size_t ws_bytes, void* stream);

/*
 * kda_bwd without a caller workspace: the scratch is a static device array inside the
 * library, KDA_NOALLOC_SCRATCH_BYTES bytes per device.  Under lazy module loading
 * (CUDA_MODULE_LOADING=LAZY, the default) it is reserved on a device when this entry point
 * is first used there, and that first call should come before any stream capture; with
 * CUDA_MODULE_LOADING=EAGER every context that loads the library reserves it at creation.
 * Its address is looked up on every call (so it stays valid across cudaDeviceReset).
 * Nothing is allocated per call.  Arguments as for kda_bwd minus workspace and ws_bytes.  Returns
 * KDA_ERR_SCRATCH_TOO_SMALL, without launching anything, when
 * kda_workspace_size(KDA_OP_BWD, N, T_total, H, dk, dv, 64) exceeds the static scratch.
 * Calls on one device share that scratch: at most one may be in flight per device
 * (issue them on one stream, or synchronise between them).
 */
#define KDA_NOALLOC_SCRATCH_BYTES ((size_t)128 << 20)
int kda_bwd_noalloc(const void* q, const void* k, const void* v, const float* log_alpha, int gate, const float* beta,
                    const float* init_states, const float* d_out, const float* d_final_states,
                    const int64_t* cu_seqlens, int N, int64_t T, int H, int dk, int dv, float* dq, float* dk_out,
                    float* dv_out, float* dlog_alpha, float* dbeta, float* d_init_states, int in_dtype, void* stream);

/*
 * kda_chunk_fwd (chunk = 64) on HOST buffers, streamed: the sequence is cut into segments
 * of segment_tokens tokens (a multiple of 64; 0 selects 4096), and each segment's
 * host-to-device copy, kernel and device-to-host copy run on three streams (two created
 * for the call, plus `stream` for the kernels), so that the copies of one segment overlap
 * the work on its neighbours.  Segments start at chunk boundaries, where a resumed run
 * reproduces the unsplit one bit for bit: the results equal kda_chunk_fwd's.
 *   q, k, v, log_alpha, beta, out: HOST pointers in kda_chunk_fwd's [B, T, H, ..] layouts;
 *               page-locked memory is needed for the copies to overlap (pageable memory
 *               works, serialised).  Must stay valid and unmodified until `stream` has
 *               passed the call.
 *   init_state  DEVICE [B, H, dk, dv] float32 or NULL (zeros), 16-byte aligned.
 *   final_state HOST [B, H, dk, dv] float32 or NULL.
 *   workspace   DEVICE, at least kda_host_fwd_workspace_size(...) bytes, 16-byte aligned:
 *               two segments of staging and two states.
 * The call returns once everything is enqueued; it is complete when `stream` reaches it.
 */
int kda_chunk_fwd_host(const void* q, const void* k, const void* v, const float* log_alpha, const float* beta,
                       const float* init_state, void* out, float* final_state, int B, int64_t T, int H, int dk,
                       int dv, int in_dtype, int out_dtype, int64_t segment_tokens, void* workspace, size_t ws_bytes,
                       void* stream);
size_t kda_host_fwd_workspace_size(int B, int H, int dk, int dv, int64_t segment_tokens, int in_dtype,
                                   int out_dtype);

/* Number of snapshots of a sequence: floor(seqlen / interval); 0 if interval <= 0 or seqlen < 0. */
int64_t kda_snapshot_count(int64_t seqlen, int64_t interval);

/*
 * Host helper: exclusive prefix sum of kda_snapshot_count over the N sequences
 * given by HOST cu_seqlens [N+1]; writes HOST offsets [N+1] (offsets[N] = total).
 * Returns KDA_ERR_INVALID_ARG on null pointers, N < 0, a negative interval or
 * decreasing cu_seqlens.
 */
int kda_snapshot_offsets(const int64_t* cu_seqlens_host, int N, int64_t interval, int64_t* offsets_host);

/*
 * Host helper for resuming a sequence from its snapshots (the prefix-cache use of
 * state snapshots, "Kimi K3 混合线性注意力", hubwiz.com, §5): the latest snapshot of
 * sequence `seq` that covers at most `prefix_len` of its tokens.  `offsets_host`
 * [N+1] is the output of kda_snapshot_offsets for the same `interval`.  Returns the
 * snapshot's index into the packed snapshot array and writes the tokens it covers
 * (m * interval) to *covered_host; a run resumed from it continues at that token
 * (kda_chunk_fwd / kda_varlen_fwd with the snapshot as initial state reproduce the
 * unsplit run bit for bit).  Returns -1 with *covered_host = 0 when the prefix is
 * shorter than one interval (resume from the sequence's initial state), -2 on
 * invalid arguments (null pointers, seq outside [0, N), interval <= 0, prefix_len < 0).
 */
int64_t kda_snapshot_lookup(const int64_t* offsets_host, int N, int seq, int64_t interval, int64_t prefix_len,
                            int64_t* covered_host);

/*
 * Bytes of device workspace the call `op` needs for these sizes (T = T_total
 * and B = N for KDA_OP_VARLEN).  0 means the workspace may be NULL.
 */
size_t kda_workspace_size(int op, int B, int64_t T, int H, int dk, int dv, int chunk);

/*
 * Diagnostic of the failure detection every kernel relies on: launches one CTA that waits,
 * with the library's bounded mbarrier wait, on a barrier nothing arrives at.  After the
 * wait's deadline (about 2 s) the kernel records KDA_ERR_TIMEOUT in the device status word
 * and returns; no trap, and the context stays usable.  Read the result with
 * kda_get_device_status().  Returns KDA_OK once the kernel is enqueued.
 */
int kda_selftest_bounded_wait(void* stream);

/* Static, human-readable name of a kda_status value. */
const char* kda_status_string(int status);

/*
 * Waits for `stream`, then reads and clears the device status word of the
 * current device: KDA_OK, KDA_ERR_TIMEOUT or KDA_STATUS_SLOT_RANGE (the first fault
 * recorded since the last read).  Returns KDA_ERR_CUDA if the read fails.
 */
int kda_get_device_status(void* stream);

#ifdef __cplusplus
}
#endif
#endif /* KDA_H_ */
