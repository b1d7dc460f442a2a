/*
 * libkda -- Kimi Delta Attention (KDA) on one GB300 (sm_103a): packed prefill,
 * decode, ReplaySSM replay, state-pool operations, input preprocessing and the
 * short convolution, and the backward of the prefill.
 *
 * What is computed.  The KDA paragraph of "Kimi K3 on Fireworks: Fast RL at
 * frontier scale" (kernels section) describes KDA as linear attention that
 * updates a compact, fixed-size recurrent state per head with channel-wise
 * gating, trained in chunk-parallel form.  The pages print no equation; this
 * library implements the gated delta rule with per-channel decay, for each
 * (sequence, head) with state S in R^{dk x dv}:
 *
 *     S <- Diag(exp(g_t)) S                    (decay of the dk rows)
 *     S <- S - beta_t k_t (k_t^T S) + beta_t k_t v_t^T
 *     o_t = S^T (scale * q_t)                  (output after the update)
 *
 * The same page's speculative-decoding paragraph (ReplaySSM) keeps the
 * recurrent state consistent after rejected draft tokens by replaying the
 * accepted tokens' update inputs from a committed checkpoint: kda_replay.
 *
 * Conventions shared by every call
 * --------------------------------
 * - All tensor arguments are DEVICE pointers to caller-owned memory (the
 *   state-pool offload / restore calls also take page-locked host memory).  The
 *   library never allocates or frees device memory; its scratch is the caller's
 *   workspace (kda_chunk_fwd_noalloc: one fixed array of its own).
 * - Token-major packed layouts, C-contiguous:
 *     q, k, g  [T, H, dk]     v, o [T, H, dv]     beta [T, H]
 *   of dtype `kda_dtype` (bf16 or fp32; o uses the same dtype as the inputs).
 *   States are always fp32, [.., H, dk, dv] with dv contiguous.
 * - g holds log-gates (alpha = exp(g) in [0, 1]); g = -inf erases the state.
 * - dk and dv must each be 64 or 128 (KDA_ERR_UNSUPPORTED otherwise).
 * - Pointers must be 16-byte aligned (beta: element-aligned; each call's
 *   section names its exceptions).
 * - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call is
 *   asynchronous on `stream`; none synchronizes except kda_device_status.
 * - Errors the host can see (NULL pointers, bad sizes, dtype, alignment, small
 *   workspace) return immediately and launch nothing.  Errors only the device
 *   can see (bad cu_seqlens / cu_accept, slot out of range, gate range, a
 *   bounded wait that gave up) are OR-ed into a status word in the workspace;
 *   read it with kda_device_status.  Each call clears that word first.  A
 *   work item that detects a device error skips its work and writes nothing.
 *   No call aborts, prints or traps.
 * - Results are deterministic: fixed reduction order, no floating-point
 *   atomics; the same sequence gives the same bits whatever else is batched
 *   with it.
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
    KDA_ERR_INVALID_ARGUMENT = 1, /* NULL pointer, negative size, misaligned pointer          */
    KDA_ERR_UNSUPPORTED = 2,      /* dk/dv not in {64,128}, unknown dtype                     */
    KDA_ERR_WORKSPACE = 3,        /* workspace NULL or smaller than required                  */
    KDA_ERR_CUDA = 4,             /* a CUDA runtime call or launch failed                     */
    KDA_ERR_GATE_RANGE = 5,       /* device: a chunk decays below 2^-100 and the workspace has
                                     no room to recompute its chain (see kda_chunk_fwd)       */
    KDA_ERR_TIMEOUT = 6,          /* device: a bounded wait gave up                           */
    KDA_ERR_BAD_SEQLENS = 7,      /* device: cu_seqlens / cu_accept not a valid partition     */
    KDA_ERR_BAD_SLOT = 8          /* device: slot index outside [0, num_slots)                */
} kda_status;

typedef enum kda_dtype {
    KDA_BF16 = 0, /* q, k, v, g, beta and o are bfloat16 */
    KDA_F32 = 1   /* q, k, v, g, beta and o are float32  */
} kda_dtype;

/* Bytes at the start of every workspace: the device status word and padding. */
#define KDA_WS_HEADER_BYTES 256

/*
 * Workspace for kda_chunk_fwd, in bytes: the size with which every path of the
 * call is available.  Returns 0 for invalid arguments.
 *
 * The minimum is smaller.  With final_state != NULL, KDA_WS_HEADER_BYTES
 * suffice; with final_state == NULL the chunked path needs a staging copy of
 * every (sequence, head) state (N*H*dk*dv*4 bytes after the header) to hand the
 * state from the chunked kernel to the partial-chunk kernel.
 *
 * T-segment split: when dk = dv = 128, N*H <= 48 and T_total >= 4096, a batch
 * has too few (sequence, head) chains to occupy the GPU, and kda_chunk_fwd cuts
 * the full chunks of every sequence in two at a chunk boundary and runs the
 * halves concurrently: segment 1 from a zero state and, with v = 0, from the
 * identity (its transition), then merges the results exactly (the recurrence is
 * affine in the state) -- the context-parallel hand-over of a long sequence's
 * state described in "Kimi K3 on Fireworks: Fast RL at frontier scale", done
 * within one GPU.  It needs 3*N*H*dk*dv*4 + T_total*H*dv*2 bytes after the
 * header, which this function then includes; with a smaller (but sufficient)
 * workspace the call runs unsplit.  Results agree within floating-point
 * rounding either way.
 *
 * Launch order: when a batch has more (sequence, head) chains than one wave of
 * chunked-kernel CTAs (N*H > 152, 2 <= N <= 8192, cu_seqlens given), the call
 * ranks the sequences by length on the device and starts the longest chains
 * first, which shortens the tail of a variable-length batch.  It needs N int32
 * (rounded up to 16 bytes) after the staging states, which this function then
 * includes; the results are bit-identical with or without it.  With it, chunked-kernel
 * CTAs are launched only for the first floor(T_total / 64) sequences of that order
 * (the others have no full chunk), which keeps a batch of short sequences (a
 * speculative verify step) from paying for thousands of empty CTAs.
 *
 * Strong decay: the chunked kernel factors each chunk's decay through prefix
 * products and needs every channel's product over a 64-token chunk to stay at or
 * above 2^-100.  With N*H bytes (rounded up to 16) after everything above, which
 * this function includes, a (sequence, head) chain that leaves that range is
 * flagged and recomputed from its initial state by the token-sequential kernel,
 * which takes any gate (g = -inf included); without that room the call reports
 * KDA_ERR_GATE_RANGE instead.
 */
size_t kda_chunk_fwd_workspace_size(int N, int64_t T_total, int H, int dk, int dv);

/*
 * Packed variable-length prefill (the chunk-parallel training/prefill form).
 *
 *   q, k, g      [T_total, H, dk]   dtype
 *   v            [T_total, H, dv]   dtype
 *   beta         [T_total, H]       dtype
 *   init_state   [N, H, dk, dv] fp32, or NULL for zeros
 *   cu_seqlens   [N+1] int32 on the device, cu[0] = 0, non-decreasing,
 *                cu[N] = T_total; sequence n is tokens [cu[n], cu[n+1]).
 *                NULL means N sequences of equal length T_total / N.
 *   scale        multiplies q (pass 1/sqrt(dk) for raw queries)
 *   o            [T_total, H, dv]   dtype (written for every token)
 *   final_state  [N, H, dk, dv] fp32, or NULL (not written).  May alias
 *                init_state (in-place update).
 *   workspace    >= kda_chunk_fwd_workspace_size() bytes (see above), device.
 *
 * Full 64-token chunks run through the chunked WY kernel (bf16; dk and dv each
 * 64 or 128: the kernel's tiles are 128 wide and a 64-wide head arrives with
 * zero channels and columns, which leave the result unchanged);
 * the last len % 64 tokens of each sequence, sequences shorter than 64, and
 * fp32 inputs run through the token-sequential kernel,
 * which is the same routine kda_decode_step and kda_replay use: a 1-token
 * sequence here gives the same bits as kda_decode_step on the same state.
 * An empty sequence copies init_state to final_state.  A chain whose chunk
 * decays below the chunked kernel's range is recomputed token by token (see
 * kda_chunk_fwd_workspace_size), so any gate values are accepted.
 */
kda_status kda_chunk_fwd(const void *q, const void *k, const void *v, const void *g, const void *beta,
                         kda_dtype dtype, const float *init_state, const int32_t *cu_seqlens, int N,
                         int64_t T_total, int H, int dk, int dv, float scale, void *o, float *final_state,
                         void *workspace, size_t ws_bytes, void *stream);

/*
 * Optional input preprocessing, fused into the kernels (the kda_*_prep calls):
 * callers that hold raw projections pass them as they are and skip a separate
 * normalisation pass over q, k, g and beta.  The pages do not define KDA's
 * input maps; the common ones for delta-rule attention are provided, each
 * behind its own flag:
 *   KDA_PREP_L2NORM_Q     q_t <- q_t / sqrt(sum_i q_{t,i}^2 + l2_eps)   per (token, head)
 *   KDA_PREP_L2NORM_K     k_t <- k_t / sqrt(sum_i k_{t,i}^2 + l2_eps)
 *   KDA_PREP_SIGMOID_GATE g holds raw gates x: the log-gate is logsigmoid(x), so the
 *                         decay is alpha = sigmoid(x) (0 only where fp32 underflows,
 *                         below about x = -88)
 *   KDA_PREP_SIGMOID_BETA beta <- sigmoid(beta)
 * scale still multiplies q after the normalisation.  Unknown flags or a
 * negative / non-finite l2_eps return KDA_ERR_INVALID_ARGUMENT.  With prep = 0
 * the _prep calls are exactly the plain ones.
 */
#define KDA_PREP_L2NORM_Q 1u
#define KDA_PREP_L2NORM_K 2u
#define KDA_PREP_SIGMOID_GATE 4u
#define KDA_PREP_SIGMOID_BETA 8u

kda_status kda_chunk_fwd_prep(const void *q, const void *k, const void *v, const void *g, const void *beta,
                              kda_dtype dtype, const float *init_state, const int32_t *cu_seqlens, int N,
                              int64_t T_total, int H, int dk, int dv, float scale, uint32_t prep, float l2_eps,
                              void *o, float *final_state, void *workspace, size_t ws_bytes, void *stream);

/*
 * One decode token per sequence on a slot-indexed state pool (in place).
 *
 *   q, k, g      [N, H, dk]   dtype;  v [N, H, dv];  beta [N, H]
 *   state_pool   [num_slots, H, dk, dv] fp32, read and written in place
 *   slots        [N] int32 device, or NULL for slot n = n (needs N <= num_slots).
 *                Two sequences must not name the same slot.
 *   o            [N, H, dv]   dtype
 *   workspace    >= KDA_WS_HEADER_BYTES bytes (status word)
 */
kda_status kda_decode_step(const void *q, const void *k, const void *v, const void *g, const void *beta,
                           kda_dtype dtype, float *state_pool, int64_t num_slots, const int32_t *slots,
                           int N, int H, int dk, int dv, float scale, void *o, void *workspace,
                           size_t ws_bytes, void *stream);

/* kda_decode_step with input preprocessing (see kda_chunk_fwd_prep). */
kda_status kda_decode_step_prep(const void *q, const void *k, const void *v, const void *g, const void *beta,
                                kda_dtype dtype, float *state_pool, int64_t num_slots, const int32_t *slots,
                                int N, int H, int dk, int dv, float scale, uint32_t prep, float l2_eps, void *o,
                                void *workspace, size_t ws_bytes, void *stream);

/*
 * ReplaySSM-style rollback: apply each sequence's accepted tokens to its
 * committed state, in place, without producing outputs.  Equivalent to
 * kda_chunk_fwd over the accepted tokens with init_state = final_state =
 * the committed state (bit for bit).
 *
 *   state_pool   [num_slots, H, dk, dv] fp32, in place
 *   slots        [N] int32 device, or NULL for slot n = n
 *   k, g         [A_total, H, dk] dtype;  v [A_total, H, dv];  beta [A_total, H]
 *   cu_accept    [N+1] int32 device; sequence n's accepted tokens are
 *                [cu_accept[n], cu_accept[n+1]) (0 tokens leaves the state)
 *   workspace    >= KDA_WS_HEADER_BYTES bytes (status word)
 */
kda_status kda_replay(float *state_pool, int64_t num_slots, const int32_t *slots, const void *k,
                      const void *v, const void *g, const void *beta, kda_dtype dtype,
                      const int32_t *cu_accept, int N, int64_t A_total, int H, int dk, int dv,
                      void *workspace, size_t ws_bytes, void *stream);

/*
 * State-pool operations for rollout caching.  In RL rollouts many trajectories
 * branch from a shared prompt, and each branch continues from its own copy of
 * the prompt's recurrent state; the states of inactive trajectories are kept
 * in host memory and brought back when the trajectory resumes ("Kimi K3 on
 * Fireworks: Fast RL at frontier scale": the rollout paragraph on MLA / KDA
 * histories that stay consistent as trajectories branch from shared prompts,
 * and the serverless-training paragraph on moving reusable KV and KDA states to
 * host memory and loading inactive snapshots asynchronously).
 *
 * A slot's state is the whole [H, dk, dv] fp32 block of the pool,
 * state_pool[slot] (H*dk*dv*4 bytes).  Slot arrays are int32 DEVICE arrays of
 * length n.  A slot outside [0, num_slots) sets KDA_ERR_BAD_SLOT in the status
 * word and that item copies nothing.  Copies are exact (bit for bit).
 * workspace: >= KDA_WS_HEADER_BYTES bytes (status word).
 */

/* Fork: state_pool[dst_slots[i]] = state_pool[src_slots[i]] for i < n.  No
 * destination may appear twice or be the source of another item (the items
 * run concurrently); src == dst copies a state onto itself. */
kda_status kda_state_fork(float *state_pool, int64_t num_slots, const int32_t *src_slots, const int32_t *dst_slots,
                          int n, int H, int dk, int dv, void *workspace, size_t ws_bytes, void *stream);

/* Offload: host_states[i] = state_pool[slots[i]] (slots NULL: slot i), for i < n.
 * host_states: [n, H, dk, dv] fp32 in page-locked host memory that the device
 * can address (cudaHostAlloc / cudaHostRegister with mapping; with unified
 * addressing every page-locked allocation is), 16-byte aligned; otherwise
 * KDA_ERR_INVALID_ARGUMENT.  The kernel writes the host memory directly;
 * synchronize `stream` before reading it on the host. */
kda_status kda_state_offload(const float *state_pool, int64_t num_slots, const int32_t *slots, int n, int H, int dk,
                             int dv, float *host_states, void *workspace, size_t ws_bytes, void *stream);

/* Restore: state_pool[slots[i]] = host_states[i] (slots NULL: slot i), for i < n;
 * host_states as for kda_state_offload.  No slot may appear twice. */
kda_status kda_state_restore(float *state_pool, int64_t num_slots, const int32_t *slots, int n, int H, int dk,
                             int dv, const float *host_states, void *workspace, size_t ws_bytes, void *stream);

/* kda_replay with input preprocessing (see kda_chunk_fwd_prep; KDA_PREP_L2NORM_Q has
 * no effect, replay reads no q).  Bit for bit the final state of
 * kda_chunk_fwd_prep over the accepted tokens with the same flags. */
kda_status kda_replay_prep(float *state_pool, int64_t num_slots, const int32_t *slots, const void *k,
                           const void *v, const void *g, const void *beta, kda_dtype dtype,
                           const int32_t *cu_accept, int N, int64_t A_total, int H, int dk, int dv, uint32_t prep,
                           float l2_eps, void *workspace, size_t ws_bytes, void *stream);

/*
 * Backward of kda_chunk_fwd (training): the gradients of a loss with respect to
 * q, k, v, g (the log-gates), beta and the initial states, given its gradients
 * with respect to o (d_o [T_total, H, dv]) and to the final states
 * (d_final_state [N, H, dk, dv] fp32, or NULL = zero).  The KDA paragraph of
 * "Kimi K3 on Fireworks: Fast RL at frontier scale" quotes a backward kernel but
 * no formula; this is the reverse mode of the same recurrence, evaluated on the
 * 64-token chunked form in four launches: a forward pass stores the state at
 * every chunk start in the workspace; every (chunk, head) computes its
 * chunk-local terms in parallel; one CTA per (sequence, head, block of state
 * columns) carries the state gradient back through the chunks; every (chunk,
 * head) then computes its gradients in parallel.  The matrix products run on the
 * tensor cores in tf32 with fp32 accumulation.  Gates whose 64-token decay falls
 * below the chunked form's range are not recomputed token by token here (the
 * forward call does that): the backward reports KDA_ERR_GATE_RANGE instead.
 *
 * Inputs as for kda_chunk_fwd (same dtype, layouts, cu_seqlens, init_state,
 * scale).  Outputs, all in the input dtype: d_q, d_k, d_g [T_total, H, dk],
 * d_v [T_total, H, dv], d_beta [T_total, H]; d_init_state [N, H, dk, dv] fp32 or
 * NULL.  Every output element is written (they need no clearing).
 * Workspace: at least kda_chunk_bwd_workspace_size(N, T_total, H, dk, dv) bytes,
 * 16-byte aligned, owned by the caller, not read back.  Errors as for
 * kda_chunk_fwd: KDA_ERR_UNSUPPORTED (dtype, dk, dv), KDA_ERR_INVALID_ARGUMENT
 * (NULL or misaligned pointers, N not dividing T_total without cu_seqlens),
 * KDA_ERR_WORKSPACE; invalid cu_seqlens and a chunk decay below 2^-100 are
 * reported through kda_device_status (KDA_ERR_BAD_SEQLENS, KDA_ERR_GATE_RANGE).
 */
size_t kda_chunk_bwd_workspace_size(int N, int64_t T_total, int H, int dk, int dv);

kda_status kda_chunk_bwd(const void *q, const void *k, const void *v, const void *g, const void *beta,
                         kda_dtype dtype, const float *init_state, const int32_t *cu_seqlens, int N,
                         int64_t T_total, int H, int dk, int dv, float scale, const void *d_o,
                         const float *d_final_state, void *d_q, void *d_k, void *d_v, void *d_g, void *d_beta,
                         float *d_init_state, void *workspace, size_t ws_bytes, void *stream);

/* kda_chunk_bwd for a forward taken with kda_chunk_fwd_prep: the inputs are the raw
 * ones given to the forward, with the same prep flags and l2_eps, and the gradients
 * are taken with respect to those raw inputs (carried back through the L2
 * normalisation, alpha = sigmoid(x_g) and beta = sigmoid(x_beta)).  prep = 0 is
 * kda_chunk_bwd. */
kda_status kda_chunk_bwd_prep(const void *q, const void *k, const void *v, const void *g, const void *beta,
                              kda_dtype dtype, const float *init_state, const int32_t *cu_seqlens, int N,
                              int64_t T_total, int H, int dk, int dv, float scale, uint32_t prep, float l2_eps,
                              const void *d_o, const float *d_final_state, void *d_q, void *d_k, void *d_v,
                              void *d_g, void *d_beta, float *d_init_state, void *workspace, size_t ws_bytes,
                              void *stream);

/*
 * Short convolution of the input projections, with its state carried across calls
 * (the disaggregated-serving paragraph of "Kimi K3 on Fireworks: Fast RL at
 * frontier scale" lists KDA's convolution state beside its recurrent state; the
 * pages define neither).  The reading implemented: a depthwise causal convolution
 * of width KDA_CONV_WIDTH over the tokens of each sequence, one weight vector per
 * channel, then SiLU:
 *   pre_t[c] = sum_{i=0}^{3} w[h][c][i] x_{t-3+i}[c],   y_t[c] = pre / (1 + exp(-pre)),
 * applied to q, k and v before everything else (the _prep flags act on its output).
 * Channels of a head are packed (q 0..dk-1 | k dk..2dk-1 | v 2dk..2dk+dv-1):
 *   conv_weight [H, 2dk+dv, KDA_CONV_WIDTH] fp32;
 *   a convolution state [KDA_CONV_WIDTH-1, H, 2dk+dv] fp32 per sequence holds its
 *   previous raw inputs, oldest first (zeros for a new sequence).
 *
 * kda_conv_fwd: the prefill form.  q, k, v [T_total, H, d] raw -> q_out, k_out,
 * v_out (same dtype and layout, not overlapping the inputs, since a block's window
 * reads the raw rows before it; then call kda_chunk_fwd(_prep) on them);
 * conv_state_in / conv_state_out [N, 3, H, 2dk+dv] (either NULL = zeros / not
 * written; they may be the same buffer).
 * kda_decode_step_conv / kda_replay_conv: the decode and replay forms, the
 * convolution fused into the token-sequential kernel; conv_pool [num_slots, 3, H,
 * 2dk+dv] is indexed by the same slots as state_pool and advanced in place.  Replay
 * takes q too: the accepted tokens' q advances the convolution state.
 * conv_width must be KDA_CONV_WIDTH (else KDA_ERR_UNSUPPORTED); other errors as
 * for the calls without convolution.
 */
#define KDA_CONV_WIDTH 4

kda_status kda_conv_fwd(const void *q, const void *k, const void *v, kda_dtype dtype, const float *conv_weight,
                        int conv_width, const float *conv_state_in, const int32_t *cu_seqlens, int N, int64_t T_total,
                        int H, int dk, int dv, void *q_out, void *k_out, void *v_out, float *conv_state_out,
                        void *workspace, size_t ws_bytes, void *stream);

kda_status kda_decode_step_conv(const void *q, const void *k, const void *v, const void *g, const void *beta,
                                kda_dtype dtype, float *state_pool, int64_t num_slots, const int32_t *slots,
                                int N, int H, int dk, int dv, float scale, const float *conv_weight,
                                int conv_width, float *conv_pool, uint32_t prep, float l2_eps, void *o,
                                void *workspace, size_t ws_bytes, void *stream);

kda_status kda_replay_conv(float *state_pool, int64_t num_slots, const int32_t *slots, const void *q, const void *k,
                           const void *v, const void *g, const void *beta, kda_dtype dtype,
                           const int32_t *cu_accept, int N, int64_t A_total, int H, int dk, int dv,
                           const float *conv_weight, int conv_width, float *conv_pool, uint32_t prep, float l2_eps,
                           void *workspace, size_t ws_bytes, void *stream);

/*
 * Synchronizes `stream`, then reads the device status word of `workspace`
 * (errors from the last call that used it).  Returns KDA_OK or the first of
 * BAD_SEQLENS, BAD_SLOT, GATE_RANGE, TIMEOUT that was raised; KDA_ERR_CUDA if
 * the synchronization or the copy failed.
 */
kda_status kda_device_status(const void *workspace, void *stream);

/* Size of the library-owned scratch behind kda_chunk_fwd_noalloc: the status
 * header plus staging room for 128 states of 128 x 128 fp32 (8 MiB). */
#define KDA_NOALLOC_WORKSPACE_BYTES ((size_t)KDA_WS_HEADER_BYTES + (size_t)8 * 1024 * 1024)

/*
 * kda_chunk_fwd for callers that cannot allocate device memory.  The pages
 * have no counterpart to this call: it exists for hosts that plan every device
 * byte themselves and give plug-in kernels no workspace hook, and for
 * latency-critical loops where a cudaMalloc (which can synchronize the device)
 * is not allowed.  It computes exactly what kda_chunk_fwd computes, with the
 * same arguments minus the workspace, and calls no allocator.
 *
 * Scratch: one array of KDA_NOALLOC_WORKSPACE_BYTES in the library's own
 * device memory; every GPU that loads libkda holds it until the process exits.
 * - Each call made outside stream capture looks up the array's device
 *   address on the current device; a call made during capture reuses the
 *   address last looked up there, so make the first call on a device before
 *   any stream capture (it returns KDA_ERR_CUDA otherwise).
 * - Every call shares the array: calls that could run at the same time on the
 *   GPU (other streams, other host threads on the same device) race on it and
 *   must be serialized by the caller.  The status word is cleared by each call.
 * - With final_state != NULL the size limit below does not apply and any
 *   batch is accepted.  With final_state == NULL the states are staged in the
 *   array, so N*H*dk*dv*4 must not exceed 8 MiB; larger requests return
 *   KDA_ERR_WORKSPACE and launch nothing.
 * - The call hands the whole array to kda_chunk_fwd as its workspace, so
 *   whatever of that call's optional buffers fit (the T-segment split's
 *   buffers, the launch order) are placed in the array too; overlapping calls
 *   race on all of it, not only on the status word and staged states.
 *
 *   status_workspace  optional out: receives the array's device address, which
 *                     kda_device_status() accepts to read this call's status.
 */
kda_status kda_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const void *g, const void *beta,
                                 kda_dtype dtype, const float *init_state, const int32_t *cu_seqlens, int N,
                                 int64_t T_total, int H, int dk, int dv, float scale, void *o, float *final_state,
                                 const void **status_workspace, void *stream);

/*
 * 1 if kda_chunk_fwd runs its full 64-token chunks on the tensor-core (tcgen05)
 * kernel for this shape and dtype, 0 if every token goes through the
 * token-sequential kernel.  Pure query; touches no device.
 */
int kda_chunk_fwd_uses_tensor_cores(int dk, int dv, kda_dtype dtype);

/* Static, human-readable name of a status code. */
const char *kda_status_string(kda_status status);

/* Library version: major*10000 + minor*100 + patch. */
int kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
