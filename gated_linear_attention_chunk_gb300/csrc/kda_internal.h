// Internal declarations shared by the host launcher and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

// Device-side error bits OR-ed into the workspace status word.
enum DeviceError : uint32_t {
    DEV_ERR_SEQLENS = 1u,  // cu_seqlens / cu_accept not a valid partition
    DEV_ERR_SLOT = 2u,     // slot outside [0, num_slots)
    DEV_ERR_GATE = 4u,     // a chunk's cumulative decay left the supported range
    DEV_ERR_TIMEOUT = 8u,  // a bounded wait gave up
};

enum SeqMode : int {
    SEQ_MODE_PREFILL = 0,  // tokens [cu[n], cu[n+1]) of a packed prefill
    SEQ_MODE_DECODE = 1,   // token n, state in a slot-indexed pool
    SEQ_MODE_REPLAY = 2,   // tokens [cu[n], cu[n+1]) onto a pool state, no output
};

// Arguments of the token-sequential kernel.  One CTA per (sequence, head).
// Input preprocessing flags (the same values as KDA_PREP_* in kda.h).
constexpr int PREP_L2NORM_Q = 1, PREP_L2NORM_K = 2, PREP_SIGMOID_GATE = 4, PREP_SIGMOID_BETA = 8;

struct SeqParams {
    const void *q, *k, *v, *g, *beta;
    void *o;                    // may be null (replay)
    int N, H;
    float scale;
    int mode;                   // SeqMode
    const int32_t *cu;          // cu_seqlens / cu_accept (prefill: may be null)
    int64_t T_total;            // total packed tokens (validation)
    int64_t seq_len_fixed;      // prefill with cu == null: every sequence has this length
    int chunk_skip;             // prefill: 1 = the first 64*floor(len/64) tokens were done by the chunked kernel
    const float *state_in;      // prefill: init_state or null; decode/replay: pool
    float *state_out;           // prefill: final_state or null; decode/replay: pool
    const float *chunk_state;   // prefill with chunk_skip: states left by the chunked kernel
    const int32_t *slots;       // decode/replay: slot map or null
    int64_t num_slots;
    uint32_t *status;           // device status word
    int prep;                   // input preprocessing flags (PREP_*), 0 = inputs used as given
    float prep_eps;             // epsilon of the L2 normalisation
    // prefill only, or null: the state at the start of every 64-token chunk of sequence n
    // goes to slot (ckpt_base(n) + c) * H + h, ckpt_base(n) = floor(first token / 64) + n
    float *ckpt;
    // prefill with chunk_skip, or null: per (sequence, head), 1 when the chunked kernel met a
    // chunk it cannot factor (decay below its range); such a chain is recomputed here from its
    // initial state, token by token, over the whole sequence
    const uint8_t *fallback;
    // decode / replay only, or null: short convolution of q, k, v (width kConvW, then SiLU)
    // before everything else, weights [H, 2dk + dv, kConvW], states [slots, kConvW - 1, H,
    // 2dk + dv] indexed like the recurrent pool and updated in place
    const float *conv_w;
    float *conv_state;
};

// Width of the short convolution of the input projections (kda_conv.cu).
constexpr int kConvW = 4;

// Prefill form of the short convolution: q, k, v -> q_out, k_out, v_out (same dtype),
// state_in / state_out [N, kConvW - 1, H, 2dk + dv] fp32 (either may be null; they may be
// the same buffer).
struct ConvParams {
    const void *q, *k, *v;
    void *q_out, *k_out, *v_out;
    const float *weight;        // [H, 2dk + dv, kConvW]
    const float *state_in;
    float *state_out;
    const int32_t *cu;
    int64_t T_total, seq_len_fixed;
    int N, H, dk, dv;
    uint32_t *status;
};
cudaError_t launch_conv(const ConvParams &p, int dtype, cudaStream_t stream);

// First checkpoint slot of a sequence starting at token `bos` (sequence index n): the
// ranges [base, base + ceil(len / 64)) of consecutive sequences do not overlap, and
// floor(T_total / 64) + N + 1 slots cover every sequence.
__host__ __device__ inline int64_t ckpt_base(int64_t bos, int64_t n) { return bos / 64 + n; }

// T-segment merge after a split chunked launch (kda_merge.cu): o on segment-1 tokens
// += S1^T o_phi, then state <- phi state + psi.  o, o_phi: [T, H, 128] bf16.
struct MergeParams {
    void *o;
    const void *o_phi;
    float *state;               // S1 on entry, final full-chunk state on exit
    const float *phi, *psi;
    const int32_t *cu;
    int64_t T_total, seq_len_fixed;
    int N, H;
    uint32_t *status;           // device status word (wait timeouts)
};
cudaError_t launch_merge(const MergeParams &p, cudaStream_t stream);

// dtype: 0 = bf16, 1 = fp32 (kda_dtype).  Returns the launch error.
cudaError_t launch_seq(const SeqParams &p, int dk, int dv, int dtype, cudaStream_t stream);

// Backward of the packed prefill (kda_bwd.cu), in three launches after the forward pass
// that leaves the chunk-start states in `ckpt` (slot ckpt_base(bos, n) + c for chunk c;
// slot 0 of each sequence is not read, the initial state is): (A) chunk-local work of
// every chunk, (B) the reverse chain of state gradients per (sequence, head), (C) the
// gradients of every chunk.  A and C run on `ctas` persistent CTAs with their own
// scratch; `rec` holds bwd_record_floats per (slot, head).
struct BwdParams {
    const void *q, *k, *v, *g, *beta, *d_o;
    const float *init_state;    // may be null (zero)
    const float *d_final;       // may be null (zero)
    void *dq, *dk, *dv, *dg, *dbeta;
    float *d_init;              // may be null
    const float *ckpt;
    float *rec;                 // per (slot, head) records
    float *scratch;             // per persistent CTA: bwd_scratch_floats; then per chain: 2 states
    int ctas;                   // persistent CTAs of phases A and C
    int64_t nslots;             // checkpoint / record slots: floor(T_total / 64) + N + 1
    const int32_t *cu;
    int64_t T_total, seq_len_fixed;
    int N, H;
    float scale;
    uint32_t *status;
    int prep;                   // input preprocessing of the forward (PREP_*): gradients are then taken
    float prep_eps;             // with respect to the raw inputs
};
size_t bwd_scratch_floats(int dk, int dv);
size_t bwd_record_floats(int dk, int dv);
cudaError_t launch_bwd(const BwdParams &p, int dk, int dv, int dtype, cudaStream_t stream);

// Arguments of the chunked (64-token WY, tcgen05) kernel: bf16, dk = dv = 128.
struct ChunkParams {
    const void *q, *k, *v, *g, *beta;
    void *o;
    int N, H;
    // head dims, each 64 or 128 (0 is taken as 128): q, k, g rows have dk channels, v and o
    // rows dv columns, the states are dk x dv; the kernel works at 128 x 128 with the missing
    // channels and columns zero (TMA fills them), which leaves the result unchanged
    int dk, dv;
    float scale;
    const int32_t *cu;          // may be null: equal lengths seq_len_fixed
    int64_t T_total;
    int64_t seq_len_fixed;
    const float *init_state;    // may be null (zeros)
    float *state_out;           // final_state or staging (never null)
    uint32_t *status;
    // T-segment split (see tseg_plan): 0 = off.  With it, state_out receives the state at
    // the cut, phi / psi the segment-1 transition and zero-start state, o_phi [T, H, 128]
    // bf16 the transition run's outputs.
    int split;
    float *phi, *psi;
    void *o_phi;
    int prep;                   // input preprocessing flags (PREP_*)
    float prep_eps;
    // or null: the state after every full chunk c goes to checkpoint slot
    // (ckpt_base(bos, n) + c + 1) * H + h (needs split == 0); o may then be null
    float *ckpt;
    // or null: launch order of the sequences (a permutation of 0..N-1, longest first), so
    // that a batch of more chains than one wave of CTAs starts its longest chains first
    // (needs split == 0)
    const int32_t *order;
    // or null: per (sequence, head) flag set (instead of the gate-range error) when a chunk's
    // decay leaves the range the factored form supports; the partial-chunk kernel then
    // recomputes the chain token by token
    uint8_t *fallback;
    // with an order: CTAs are launched for the first n_active ranks only (sequences with a full
    // chunk rank first, and at most T_total / 64 of them exist; 0 launches none)
    int n_active;
};
// order[rank] = n, sequences ranked by full chunks (descending, ties by index).
cudaError_t launch_order(const int32_t *cu, int N, int32_t *order, cudaStream_t stream);

// True when the chunked tensor-core kernel is compiled in and supports the shape.
bool chunk_tc_supported(int dk, int dv, int dtype);
cudaError_t launch_chunk_tc(const ChunkParams &p, cudaStream_t stream);

}  // namespace kda
