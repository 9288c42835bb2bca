/*
 * kda.h -- C ABI of libkda.so: Kimi Delta Attention (KDA) on one GB300 (sm_103a).
 *
 * The operation (per head h of every sequence) is defined on the dev.to page
 * "Kimi K3 Architecture: Scaling 2.8T Parameters for Long-Context Multimodal
 * MoE", section "The Sequence Bottleneck: Hybrid KDA and Gated MLA":
 *   gate   g_t = g_min * Sigmoid(exp(A_h) * z_t),  g_min = -5,  alpha_t = exp(g_t)
 *   state  S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *   output o_t = S_t^T q_t
 * with a fixed-size dk x dv fp32 state per (sequence, head) (also "Kimi K3 -
 * Sparsity Mechanics...", section 2, "Temporal Sequence (KDA)").  The same
 * section of the dev.to page bounds the cumulative log-decay of every 16-token
 * tile to (-80, 0), which is what lets the chunked form run on bf16 tiles.
 *
 * Conventions shared by every entry point
 *  - Layout "THD": token-major packed tensors [T_tot, H, D], D contiguous.
 *    q, k, z: D = dk; v and o: D = dv; beta: [T_tot, H].
 *  - States are fp32 [N, H, dk, dv], row-major: S[n][h][i][j], i the key
 *    channel (dk), j the value channel (dv).
 *  - dtype selects the storage type of q, k, v, z, beta and o: KDA_F32 or
 *    KDA_BF16.  A_log ([H], the per-head A^h) and all states are fp32.
 *    Arithmetic is fp32 (bf16 tensor-core operands where a kernel says so).
 *  - q must arrive already normalised and scaled; the library applies no
 *    scale and no normalisation.  beta must already lie in (0, 1).
 *  - Every pointer except `stream` is a DEVICE pointer.  The caller owns and
 *    allocates every buffer, including the workspace; the library allocates
 *    no device memory and keeps no per-call state.
 *  - Pointers to q, k, v, z, o and states must be 16-byte aligned.
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL means
 *    the legacy default stream).  Argument errors are returned synchronously
 *    and nothing is launched.  Errors found on the device (a non-finite or
 *    out-of-range cumulative decay, inconsistent cu_seqlens, a bounded wait
 *    that expired) are recorded in a status word at the start of the
 *    workspace; read it with kda_query_status.  The first error recorded wins.
 *  - Supported head sizes: dk, dv in {32, 64, 128}.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kda_status {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, aliasing, small workspace */
    KDA_ERR_UNSUPPORTED = 2, /* head size or dtype this library does not build */
    KDA_ERR_DECAY_RANGE = 3, /* a 16-token cumulative log-decay not finite or outside [-80, 0] */
    KDA_ERR_TIMEOUT = 4,     /* a bounded device-side wait expired */
    KDA_ERR_CUDA = 5,        /* a CUDA runtime call failed */
    KDA_ERR_SEQLENS = 6      /* cu_seqlens not 0-based, decreasing, or not ending at T_tot */
} kda_status;

typedef enum kda_dtype { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype;

/* Version of this ABI (bumped on any signature change). */
int32_t kda_abi_version(void);

/* Human-readable name of a status code (static storage, never NULL). */
const char *kda_status_string(int32_t status);

/*
 * Bytes of workspace kda_chunk_fwd needs for this problem size.  The
 * workspace holds the status word, the chunk plan of the packed sequences
 * and the intermediates of the chunked form; its contents need no
 * initialisation and are overwritten by every call.  Returns 0 for
 * arguments kda_chunk_fwd would reject.  On the tensor-core path the size
 * includes the segment-parallel schedule's buffers when kda_chunk_fwd would pick
 * that schedule on the current device (see kda_chunk_fwd).
 */
size_t kda_chunk_fwd_workspace_size(int64_t total_tokens, int32_t num_seqs, int32_t H,
                                    int32_t dk, int32_t dv, int32_t dtype);

/*
 * Chunked prefill over packed variable-length sequences.
 *
 * Computes, for every sequence n = 0..num_seqs-1 (tokens cu_seqlens[n] ..
 * cu_seqlens[n+1]-1) and head h, the recurrence in the file header starting
 * from initial_state[n][h] (zeros when initial_state is NULL); writes o for
 * every token and, when final_state is not NULL, the state after the
 * sequence's last token.  An empty sequence leaves its state unchanged.
 * Internally the sequence is cut into chunks that start at the sequence's
 * first token; the intra-chunk part runs as dense products over 16-token
 * tiles (the chunkwise-parallel form of the dev.to page, section "The
 * Sequence Bottleneck").  The result equals the token-by-token recurrence
 * up to rounding.  On the tensor-core path, when a few long sequences would
 * leave most SMs idle (num_seqs x H x (4 + 8 (s - 1)) 32-column chain CTAs for s
 * segments fit one wave of the device's SMs, with >= 64 chunks per segment of the
 * average sequence, s >= 2), the call runs the segment-parallel schedule of
 * kda_chunk_fwd_segmented with the largest such s <= 16, provided the workspace
 * holds its buffers (the size query includes them); otherwise the plain schedule.
 *
 * Work is enqueued on `stream` and returns without synchronising.  On the
 * tensor-core path (bf16, dk = dv = 128) a problem with more than one window
 * of chunk records also runs kernels on streams the library owns (created on
 * first use per device, kept for the life of the process): they start after
 * everything enqueued on `stream` before the call, and `stream` waits for them
 * before anything enqueued after it, so to the caller the call behaves as work
 * on `stream` alone.  Calls from several host threads are serialised while
 * they enqueue.
 *
 *   q, k, z       [total_tokens, H, dk]  dtype
 *   v             [total_tokens, H, dv]  dtype
 *   beta          [total_tokens, H]      dtype
 *   A_log         [H]                    fp32
 *   cu_seqlens    [num_seqs + 1]         int32, device; 0 = cu[0] <= ... <= cu[num_seqs] = total_tokens
 *   initial_state [num_seqs, H, dk, dv]  fp32 or NULL
 *   final_state   [num_seqs, H, dk, dv]  fp32 or NULL; may alias initial_state (in-place update)
 *   o             [total_tokens, H, dv]  dtype; must not alias any input
 *   workspace     >= kda_chunk_fwd_workspace_size(...) bytes, 256-byte aligned
 * Limits: total_tokens < 2^31 on the tensor-core path (KDA_ERR_INVALID_ARG otherwise).
 * Device-found errors: KDA_ERR_SEQLENS (nothing computed for the offending
 * sequence), KDA_ERR_DECAY_RANGE (outputs of that chunk are not meaningful),
 * KDA_ERR_TIMEOUT.
 */
kda_status kda_chunk_fwd(const void *q, const void *k, const void *v, const void *z,
                         const void *beta, const float *A_log, const int32_t *cu_seqlens,
                         int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t dk,
                         int32_t dv, int32_t dtype, const float *initial_state,
                         float *final_state, void *o, void *workspace, size_t workspace_bytes,
                         void *stream);

/*
 * Segment-parallel prefill: kda_chunk_fwd for a few long sequences.  The pages'
 * KDA context parallelism (dev.to page "Kimi K3 Architecture...", section
 * "Infrastructure and Training/Inference Mechanics": per-rank state maps merged
 * by a prefix scan) applied inside one GPU, to segments of each sequence.
 *
 * On the tensor-core path (bf16, dk = dv = 128), within each window of chunk
 * records every sequence's chunks are cut into s = min(segments, chunks)
 * near-equal consecutive segments.  A first pass walks segment 0 from the
 * sequence's state (writing its outputs) while every later segment k walks from
 * [I | 0] with [0 | U~], giving its affine map S_end = M_k S_start + B_k
 * (M_k is dk x dk: the state's evolution with V = 0).  A scan composes the maps
 * into each later segment's start state (fp32), and a second pass walks the later
 * segments from those states, writing their outputs and the final state.  The
 * sequential depth per window falls from L chunks to about 2 L / s, at the price
 * of (dk + dv) / dv times the chain work on later segments; it pays off when
 * sequences x heads leave most SMs idle.  The windows run one after the other on
 * `stream` alone.  segments == 1, or any call off the tensor-core path, is the
 * plain schedule.  Results equal the plain schedule's up to rounding (the later
 * segments' start states go through the composed maps).  kda_chunk_fwd picks this
 * schedule by itself for the shapes where it pays; this entry fixes the count.
 *
 * Arguments are those of kda_chunk_fwd, plus:
 *   segments      1 ..= 64
 *   workspace     >= kda_chunk_fwd_segmented_workspace_size(..., segments) bytes,
 *                 256-byte aligned (adds num_seqs x H x segments x dk x (dk + 2 dv)
 *                 fp32 on the tensor-core path)
 * Errors: those of kda_chunk_fwd; KDA_ERR_INVALID_ARG for segments outside 1 ..= 64.
 */
size_t kda_chunk_fwd_segmented_workspace_size(int64_t total_tokens, int32_t num_seqs, int32_t H,
                                              int32_t dk, int32_t dv, int32_t dtype,
                                              int32_t segments);
kda_status kda_chunk_fwd_segmented(const void *q, const void *k, const void *v, const void *z,
                                   const void *beta, const float *A_log,
                                   const int32_t *cu_seqlens, int32_t num_seqs,
                                   int64_t total_tokens, int32_t H, int32_t dk, int32_t dv,
                                   int32_t dtype, const float *initial_state, float *final_state,
                                   void *o, int32_t segments, void *workspace,
                                   size_t workspace_bytes, void *stream);

/*
 * kda_chunk_fwd with per-kernel timing: identical arguments and results, plus
 * `events`, an array of n_events caller-created cudaEvent_t handles (created
 * with timing enabled).  The call brackets its j-th kernel with events[2j]
 * (before) and events[2j+1] (after), both recorded on the stream that kernel is
 * launched on, for as many kernels as fit, and writes the number of events
 * recorded to *n_recorded (host pointer).  The kernels of one call on the
 * tensor-core path are, in launch order: the chunk plan (which also clears the
 * status word and writes the final state of sequences that own no chunk), then
 * one (prep, chain) pair per window of chunk records; on
 * the CUDA-core path, one chunked kernel.  Used by the benchmark to time the
 * dominant kernel on its own launch stream.
 */
kda_status kda_chunk_fwd_profiled(const void *q, const void *k, const void *v, const void *z,
                                  const void *beta, const float *A_log,
                                  const int32_t *cu_seqlens, int32_t num_seqs,
                                  int64_t total_tokens, int32_t H, int32_t dk, int32_t dv,
                                  int32_t dtype, const float *initial_state, float *final_state,
                                  void *o, void *workspace, size_t workspace_bytes, void *stream,
                                  void *const *events, int32_t n_events, int32_t *n_recorded);

/*
 * Size of the scratch array behind kda_chunk_fwd_noalloc: 32 MiB, held on
 * every GPU that loads this library until the process exits.
 */
#define KDA_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * kda_chunk_fwd for callers that cannot allocate device memory.  (The pages
 * have no counterpart: this is an interface convenience, not part of the
 * method.)
 *
 * Who needs it: code that is handed its input and output buffers and nothing
 * else -- a plug-in inside a host application that owns every device
 * allocation, or a serving loop that must not call cudaMalloc after start-up
 * (cudaMalloc synchronises the device and can fail under memory pressure).
 * Such callers cannot supply kda_chunk_fwd's workspace.  This entry runs the
 * same kernels with the same results, and takes its scratch (status word,
 * chunk plan, running state, chunk records) from a fixed array of
 * KDA_NOALLOC_SCRATCH_BYTES owned by the library.  It calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *
 * Arguments are those of kda_chunk_fwd without the workspace, plus:
 *   status_out  NULL, or a device buffer of >= 16 bytes (16-byte aligned)
 *               that receives the call's status word when the call's work
 *               completes; read it with kda_query_status(status_out, ...).
 * Limits: the problem must fit the array.  On the tensor-core path (bf16,
 * dk = dv = 128) the chunk plan ((num_seqs + 1) int32), the running state
 * (num_seqs * H * 64 KiB, only when final_state is NULL) and at least one
 * chunk record per head (H * 74,240 bytes) must fit in 32 MiB; larger
 * problems are rejected with KDA_ERR_INVALID_ARG before anything is launched.
 * Fewer records fit than in a caller-sized workspace, so long inputs run in
 * more, smaller windows.
 * On the CUDA-core path (fp32, or other head sizes) only the status word and
 * the chunk plan live in the array.
 * Set-up: every call looks up the array's device address on the current
 * device with cudaGetSymbolAddress (no allocation, nothing cached, so the
 * library stays usable after a cudaDeviceReset); the first call on a device
 * also loads the library's device code there, so make it before any stream
 * capture.
 * Concurrency: every call uses the same array, which keeps the previous
 * call's contents (each call clears what it needs).  Calls whose work can
 * overlap on the GPU -- on different streams, or from threads that do not
 * order their launches -- race on the array and must be serialised.
 */
kda_status kda_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const void *z,
                                 const void *beta, const float *A_log,
                                 const int32_t *cu_seqlens, int32_t num_seqs,
                                 int64_t total_tokens, int32_t H, int32_t dk, int32_t dv,
                                 int32_t dtype, const float *initial_state, float *final_state,
                                 void *o, void *status_out, void *stream);

/*
 * Test hook for failure detection (the pages have no counterpart).  The next
 * tensor-core kda_chunk_fwd / kda_chunk_fwd_segmented call of this process
 * (bf16, dk = dv = 128) gives every bounded wait of its chain kernels the
 * limit `wait_ns` (nanoseconds, > 0; the default is one second) and leaves out
 * the first chunk-record load of chain CTA `skip_cta` (-1: none).  That CTA's
 * wait for the record then expires: the call reports KDA_ERR_TIMEOUT through
 * the status word (info: the CTA's work item), the CTA stops after letting
 * every copy and product it issued finish, and the library stays usable for
 * the next call.  Returns KDA_ERR_INVALID_ARG for wait_ns <= 0.  Which call
 * picks the setting up is not defined between threads; meant for tests only.
 */
kda_status kda_test_chain_fault(int64_t wait_ns, int32_t skip_cta);

/* Bytes of workspace kda_decode_step needs (the status word only). */
size_t kda_decode_workspace_size(void);

/*
 * One decode step: every one of N sequences advances by exactly one token
 * against its resident state, which is updated in place (the constant-size
 * state of "Kimi K3 - Sparsity Mechanics...", section 2 "Temporal Sequence
 * (KDA)", "constant decoding memory"; the update of the dev.to page).
 *
 *   q, k, z  [N, H, dk]  dtype       v  [N, H, dv]  dtype      beta [N, H] dtype
 *   A_log    [H] fp32
 *   state    [N, H, dk, dv] fp32, read and written in place
 *   o        [N, H, dv]  dtype
 *   workspace >= kda_decode_workspace_size() bytes
 * The state is streamed once from HBM and written once; the step is
 * memory-bound.  Device-found errors: none beyond KDA_ERR_CUDA (a non-finite
 * gate propagates into the state and output as in the definition).
 */
kda_status kda_decode_step(const void *q, const void *k, const void *v, const void *z,
                           const void *beta, const float *A_log, float *state, void *o,
                           int32_t N, int32_t H, int32_t dk, int32_t dv, int32_t dtype,
                           void *workspace, size_t workspace_bytes, void *stream);

/*
 * kda_decode_step against a pool of states: sequence n advances the state in
 * slot state_idx[n] of state_pool, which is updated in place.  This is the
 * KDA half of the serving engine's paged hybrid cache, where fixed-size KDA
 * states live in pooled memory (dev.to page, section "Infrastructure and
 * Training/Inference Mechanics", "Serving Engine").
 *
 *   state_pool [P, H, dk, dv] fp32          state_idx [N] int32, device, values in [0, P)
 *   other arguments as kda_decode_step (q, k, z, v, beta, o are per sequence n)
 * The N indices must be distinct (two sequences sharing a slot race).  An
 * index outside [0, P) is recorded as KDA_ERR_INVALID_ARG in the status word
 * (info = the sequence) and that sequence is skipped.
 */
kda_status kda_decode_step_indexed(const void *q, const void *k, const void *v, const void *z,
                                   const void *beta, const float *A_log, float *state_pool,
                                   const int32_t *state_idx, int32_t P, void *o, int32_t N,
                                   int32_t H, int32_t dk, int32_t dv, int32_t dtype,
                                   void *workspace, size_t workspace_bytes, void *stream);

/*
 * The gate on its own: g = -5 Sigmoid(exp(A_h) z) per channel and its
 * inclusive cumulative sum restarted every `chunk` tokens (chunks start at
 * each sequence's first token), written as fp32 [total_tokens, H, dk].
 * Also range-checks every 16-token tile prefix sum against [-80, 0]
 * (dev.to page, section "The Sequence Bottleneck", the bound after the gate
 * equation) and records KDA_ERR_DECAY_RANGE on a violation.  `chunk` must
 * be a positive multiple of 16.  kda_chunk_fwd fuses the same computation
 * into its own kernels; this entry exposes it for inspection.
 * gate_mode 0 is the lower-bounded gate above; gate_mode 1 evaluates the
 * unbounded baseline the page says it replaces, g = -Softplus(exp(A_h) z),
 * with the same range check, for an A/B of the bound (the chunked forward
 * accepts only the bounded gate).
 * Workspace: >= kda_chunk_fwd_workspace_size(total_tokens, num_seqs, H, dk, dk, dtype).
 */
kda_status kda_gate_cumsum(const void *z, const float *A_log, const int32_t *cu_seqlens,
                           int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t dk,
                           int32_t dtype, int32_t chunk, int32_t gate_mode, float *g_cumsum,
                           void *workspace, size_t workspace_bytes, void *stream);

/*
 * Waits for `stream`, then returns the status recorded in `workspace` by the
 * last call that used it (KDA_OK if none).  When `info` is not NULL it
 * receives a detail of the first error: the flat token*H+head index of a
 * decay-range violation, the sequence index of a cu_seqlens error, or the
 * site of an expired wait.
 */
kda_status kda_query_status(const void *workspace, void *stream, int64_t *info);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
