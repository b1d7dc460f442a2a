// C-ABI entry points of libkda: argument validation, workspace layout and
// kernel launches.  Declared and documented in include/kda.h.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"
#include "kda_internal.h"

namespace {

constexpr int kVersion = 10000;  // 1.0.0

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned_to(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
bool dim_ok(int d) { return d == 64 || d == 128; }
bool dtype_ok(kda_dtype t) { return t == KDA_BF16 || t == KDA_F32; }
size_t elem_size(kda_dtype t) { return t == KDA_BF16 ? 2 : 4; }

// Known preprocessing flags only, and a finite non-negative epsilon.
bool prep_ok(uint32_t prep, float eps) {
    const uint32_t known = KDA_PREP_L2NORM_Q | KDA_PREP_L2NORM_K | KDA_PREP_SIGMOID_GATE | KDA_PREP_SIGMOID_BETA;
    return (prep & ~known) == 0 && eps >= 0.f && eps < 3.0e38f;
}

size_t staging_offset() { return KDA_WS_HEADER_BYTES; }

// Launch order (longest sequences first) for batches of more (sequence, head) chains than
// one wave of chunked-kernel CTAs (one per SM; 152 on GB300): N int32 after the staging
// states, when the workspace has room for them.
constexpr int64_t kWaveChains = 152;
constexpr int kOrderMaxSeqs = 8192;
bool order_shape(int N, int H) {
    return N >= 2 && N <= kOrderMaxSeqs && static_cast<int64_t>(N) * H > kWaveChains;
}
size_t order_offset(int N, int H, int dk, int dv) {
    return staging_offset() + static_cast<size_t>(N) * H * dk * dv * sizeof(float);
}
size_t order_bytes(int N) { return (static_cast<size_t>(N) * sizeof(int32_t) + 15) & ~static_cast<size_t>(15); }

size_t state_bytes(int N, int H, int dk, int dv) {
    return static_cast<size_t>(N) * static_cast<size_t>(H) * dk * dv * sizeof(float);
}

// T-segment split (see kda_chunk_fwd_workspace_size in kda.h): used for batches of at
// most kSplitMaxPairs (sequence, head) chains, which would leave most SMs idle.
constexpr int64_t kSplitMaxPairs = 48;
constexpr int64_t kSplitMinTokens = 4096;

bool split_shape(int N, int64_t T_total, int H, int dk, int dv) {
    return dk == 128 && dv == 128 && N > 0 && static_cast<int64_t>(N) * H <= kSplitMaxPairs &&
           T_total >= kSplitMinTokens;
}

// Workspace of a split call: header | staging states | phi | psi | o_phi (bf16 [T, H, dv]).
size_t split_workspace(int N, int64_t T_total, int H, int dk, int dv) {
    return staging_offset() + 3 * state_bytes(N, H, dk, dv) + static_cast<size_t>(T_total) * H * dv * 2;
}

// Strong-decay fallback: one byte per (sequence, head) chain, after everything else the call
// uses, when the workspace has room for it.  A chain whose chunk decays below the factored
// form's range is then flagged by the chunked kernel and recomputed token by token.
size_t align16(size_t x) { return (x + 15) & ~static_cast<size_t>(15); }
size_t fallback_bytes(int N, int H) { return align16(static_cast<size_t>(N) * static_cast<size_t>(H)); }

// Clears the status word at the start of the workspace (asynchronously on the stream).
kda_status clear_status(void *workspace, cudaStream_t s) {
    if (cudaMemsetAsync(workspace, 0, sizeof(uint32_t), s) != cudaSuccess) return KDA_ERR_CUDA;
    return KDA_OK;
}

}  // namespace

extern "C" {

size_t kda_chunk_fwd_workspace_size(int N, int64_t T_total, int H, int dk, int dv) {
    if (N < 0 || T_total < 0 || H <= 0 || !dim_ok(dk) || !dim_ok(dv)) return 0;
    size_t used = staging_offset() + state_bytes(N, H, dk, dv);
    if (split_shape(N, T_total, H, dk, dv))
        used = split_workspace(N, T_total, H, dk, dv);
    else if (order_shape(N, H))
        used = order_offset(N, H, dk, dv) + order_bytes(N);
    return align16(used) + fallback_bytes(N, H);
}

kda_status kda_chunk_fwd_prep(const void *q, const void *k, const void *v, const void *g, const void *beta,
                              kda_dtype dtype, const float *init_state, const int32_t *cu_seqlens, int N,
                              int64_t T_total, int H, int dk, int dv, float scale, uint32_t prep, float l2_eps,
                              void *o, float *final_state, void *workspace, size_t ws_bytes, void *stream) {
    if (!dtype_ok(dtype) || !dim_ok(dk) || !dim_ok(dv)) return KDA_ERR_UNSUPPORTED;
    if (!prep_ok(prep, l2_eps)) return KDA_ERR_INVALID_ARGUMENT;
    if (N < 0 || T_total < 0 || H <= 0) return KDA_ERR_INVALID_ARGUMENT;
    if (!workspace || !aligned16(workspace)) return KDA_ERR_WORKSPACE;
    if (ws_bytes < KDA_WS_HEADER_BYTES) return KDA_ERR_WORKSPACE;
    if (!final_state && ws_bytes < staging_offset() + state_bytes(N, H, dk, dv)) return KDA_ERR_WORKSPACE;
    if (T_total > 0) {
        if (!q || !k || !v || !g || !beta || !o) return KDA_ERR_INVALID_ARGUMENT;
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(o))
            return KDA_ERR_INVALID_ARGUMENT;
        if (!aligned_to(beta, elem_size(dtype))) return KDA_ERR_INVALID_ARGUMENT;
    }
    if ((init_state && !aligned16(init_state)) || (final_state && !aligned16(final_state)))
        return KDA_ERR_INVALID_ARGUMENT;
    if (!cu_seqlens && N > 0 && (T_total % N) != 0) return KDA_ERR_INVALID_ARGUMENT;
    if (!cu_seqlens && N == 0 && T_total != 0) return KDA_ERR_INVALID_ARGUMENT;
    if (cu_seqlens && !aligned_to(cu_seqlens, 4)) return KDA_ERR_INVALID_ARGUMENT;
    if (!cu_seqlens && N == 0 && T_total == 0) { /* nothing */ }

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    kda_status st = clear_status(workspace, s);
    if (st != KDA_OK) return st;
    if (N == 0) return KDA_OK;

    uint32_t *status = static_cast<uint32_t *>(workspace);
    const int64_t fixed_len = cu_seqlens ? 0 : T_total / N;
    // the tensor-core kernel addresses tokens with 32-bit TMA coordinates
    const bool use_tc = kda::chunk_tc_supported(dk, dv, static_cast<int>(dtype)) && T_total <= 0x7fffffffLL;
    float *chunk_state = final_state
                             ? final_state
                             : reinterpret_cast<float *>(static_cast<char *>(workspace) + staging_offset());

    uint8_t *fallback = nullptr;
    if (use_tc) {
        const bool split = split_shape(N, T_total, H, dk, dv) && ws_bytes >= split_workspace(N, T_total, H, dk, dv);
        const bool ordered = !split && cu_seqlens && order_shape(N, H) &&
                             ws_bytes >= order_offset(N, H, dk, dv) + order_bytes(N);
        size_t used = KDA_WS_HEADER_BYTES + (final_state ? 0 : state_bytes(N, H, dk, dv));
        if (split) used = split_workspace(N, T_total, H, dk, dv);
        if (ordered) used = order_offset(N, H, dk, dv) + order_bytes(N);
        if (ws_bytes >= align16(used) + fallback_bytes(N, H)) {
            fallback = reinterpret_cast<uint8_t *>(static_cast<char *>(workspace) + align16(used));
            if (cudaMemsetAsync(fallback, 0, static_cast<size_t>(N) * H, s) != cudaSuccess) return KDA_ERR_CUDA;
        }
        kda::ChunkParams cp{};
        cp.q = q; cp.k = k; cp.v = v; cp.g = g; cp.beta = beta; cp.o = o;
        cp.N = N; cp.H = H; cp.dk = dk; cp.dv = dv; cp.scale = scale;
        cp.cu = cu_seqlens; cp.T_total = T_total; cp.seq_len_fixed = fixed_len;
        cp.init_state = init_state; cp.state_out = chunk_state; cp.status = status;
        cp.prep = static_cast<int>(prep); cp.prep_eps = l2_eps;
        cp.fallback = fallback;
        if (ordered) {
            int32_t *order = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + order_offset(N, H, dk, dv));
            if (kda::launch_order(cu_seqlens, N, order, s) != cudaSuccess) return KDA_ERR_CUDA;
            cp.order = order;
            // Sequences with a full chunk rank first and at most T_total / 64 of them exist, so the
            // CTAs of later ranks would find nothing to do (a batch of short verify sequences).
            cp.n_active = static_cast<int>(T_total / 64 < N ? T_total / 64 : N);
        }
        if (split) {
            char *base = static_cast<char *>(workspace) + staging_offset() + state_bytes(N, H, dk, dv);
            cp.split = 1;
            cp.phi = reinterpret_cast<float *>(base);
            cp.psi = reinterpret_cast<float *>(base + state_bytes(N, H, dk, dv));
            cp.o_phi = base + 2 * state_bytes(N, H, dk, dv);
        }
        if (kda::launch_chunk_tc(cp, s) != cudaSuccess) return KDA_ERR_CUDA;
        if (split) {
            kda::MergeParams mp{};
            mp.o = o; mp.o_phi = cp.o_phi; mp.state = chunk_state; mp.phi = cp.phi; mp.psi = cp.psi;
            mp.cu = cu_seqlens; mp.T_total = T_total; mp.seq_len_fixed = fixed_len; mp.N = N; mp.H = H;
            mp.status = status;
            if (kda::launch_merge(mp, s) != cudaSuccess) return KDA_ERR_CUDA;
        }
    }

    kda::SeqParams sp{};
    sp.q = q; sp.k = k; sp.v = v; sp.g = g; sp.beta = beta; sp.o = o;
    sp.N = N; sp.H = H; sp.scale = scale;
    sp.mode = kda::SEQ_MODE_PREFILL;
    sp.cu = cu_seqlens; sp.T_total = T_total; sp.seq_len_fixed = fixed_len;
    sp.chunk_skip = use_tc ? 1 : 0;
    sp.state_in = init_state; sp.state_out = final_state; sp.chunk_state = chunk_state;
    sp.slots = nullptr; sp.num_slots = 0; sp.status = status;
    sp.prep = static_cast<int>(prep); sp.prep_eps = l2_eps;
    sp.fallback = fallback;
    if (kda::launch_seq(sp, dk, dv, static_cast<int>(dtype), s) != cudaSuccess) return KDA_ERR_CUDA;
    return KDA_OK;
}

kda_status kda_chunk_fwd(const void *q, const void *k, const void *v, const void *g, const void *beta,
                         kda_dtype dtype, const float *init_state, const int32_t *cu_seqlens, int N,
                         int64_t T_total, int H, int dk, int dv, float scale, void *o, float *final_state,
                         void *workspace, size_t ws_bytes, void *stream) {
    return kda_chunk_fwd_prep(q, k, v, g, beta, dtype, init_state, cu_seqlens, N, T_total, H, dk, dv, scale, 0u,
                              0.f, o, final_state, workspace, ws_bytes, stream);
}

static kda_status decode_impl(const void *q, const void *k, const void *v, const void *g, const void *beta,
                              kda_dtype dtype, float *state_pool, int64_t num_slots, const int32_t *slots, int N,
                              int H, int dk, int dv, float scale, uint32_t prep, float l2_eps, const float *conv_w,
                              float *conv_pool, void *o, void *workspace, size_t ws_bytes, void *stream) {
    if (!dtype_ok(dtype) || !dim_ok(dk) || !dim_ok(dv)) return KDA_ERR_UNSUPPORTED;
    if (!prep_ok(prep, l2_eps)) return KDA_ERR_INVALID_ARGUMENT;
    if (conv_w && (!conv_pool || !aligned_to(conv_w, 4) || !aligned_to(conv_pool, 4)))
        return KDA_ERR_INVALID_ARGUMENT;
    if (N < 0 || H <= 0 || num_slots < 0) return KDA_ERR_INVALID_ARGUMENT;
    if (!workspace || !aligned16(workspace) || ws_bytes < KDA_WS_HEADER_BYTES) return KDA_ERR_WORKSPACE;
    if (N > 0) {
        if (!q || !k || !v || !g || !beta || !o || !state_pool) return KDA_ERR_INVALID_ARGUMENT;
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(o) ||
            !aligned16(state_pool))
            return KDA_ERR_INVALID_ARGUMENT;
        if (!aligned_to(beta, elem_size(dtype))) return KDA_ERR_INVALID_ARGUMENT;
        if (slots && !aligned_to(slots, 4)) return KDA_ERR_INVALID_ARGUMENT;
        if (!slots && N > num_slots) return KDA_ERR_INVALID_ARGUMENT;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    kda_status st = clear_status(workspace, s);
    if (st != KDA_OK || N == 0) return st;

    kda::SeqParams sp{};
    sp.q = q; sp.k = k; sp.v = v; sp.g = g; sp.beta = beta; sp.o = o;
    sp.N = N; sp.H = H; sp.scale = scale;
    sp.mode = kda::SEQ_MODE_DECODE;
    sp.cu = nullptr; sp.T_total = N; sp.seq_len_fixed = 1; sp.chunk_skip = 0;
    sp.state_in = state_pool; sp.state_out = state_pool; sp.chunk_state = nullptr;
    sp.slots = slots; sp.num_slots = num_slots; sp.status = static_cast<uint32_t *>(workspace);
    sp.prep = static_cast<int>(prep); sp.prep_eps = l2_eps;
    sp.conv_w = conv_w; sp.conv_state = conv_pool;
    if (kda::launch_seq(sp, dk, dv, static_cast<int>(dtype), s) != cudaSuccess) return KDA_ERR_CUDA;
    return KDA_OK;
}

kda_status kda_decode_step_prep(const void *q, const void *k, const void *v, const void *g, const void *beta,
                                kda_dtype dtype, float *state_pool, int64_t num_slots, const int32_t *slots,
                                int N, int H, int dk, int dv, float scale, uint32_t prep, float l2_eps, void *o,
                                void *workspace, size_t ws_bytes, void *stream) {
    return decode_impl(q, k, v, g, beta, dtype, state_pool, num_slots, slots, N, H, dk, dv, scale, prep, l2_eps,
                       nullptr, nullptr, o, workspace, ws_bytes, stream);
}

kda_status kda_decode_step_conv(const void *q, const void *k, const void *v, const void *g, const void *beta,
                                kda_dtype dtype, float *state_pool, int64_t num_slots, const int32_t *slots,
                                int N, int H, int dk, int dv, float scale, const float *conv_weight,
                                int conv_width, float *conv_pool, uint32_t prep, float l2_eps, void *o,
                                void *workspace, size_t ws_bytes, void *stream) {
    if (conv_width != KDA_CONV_WIDTH) return KDA_ERR_UNSUPPORTED;
    if (!conv_weight || !conv_pool) return KDA_ERR_INVALID_ARGUMENT;
    return decode_impl(q, k, v, g, beta, dtype, state_pool, num_slots, slots, N, H, dk, dv, scale, prep, l2_eps,
                       conv_weight, conv_pool, o, workspace, ws_bytes, stream);
}

kda_status kda_decode_step(const void *q, const void *k, const void *v, const void *g, const void *beta,
                           kda_dtype dtype, float *state_pool, int64_t num_slots, const int32_t *slots,
                           int N, int H, int dk, int dv, float scale, void *o, void *workspace,
                           size_t ws_bytes, void *stream) {
    return kda_decode_step_prep(q, k, v, g, beta, dtype, state_pool, num_slots, slots, N, H, dk, dv, scale, 0u, 0.f,
                                o, workspace, ws_bytes, stream);
}

static kda_status replay_impl(float *state_pool, int64_t num_slots, const int32_t *slots, const void *q,
                              const void *k, const void *v, const void *g, const void *beta, kda_dtype dtype,
                              const int32_t *cu_accept, int N, int64_t A_total, int H, int dk, int dv,
                              uint32_t prep, float l2_eps, const float *conv_w, float *conv_pool, void *workspace,
                              size_t ws_bytes, void *stream) {
    if (!dtype_ok(dtype) || !dim_ok(dk) || !dim_ok(dv)) return KDA_ERR_UNSUPPORTED;
    if (!prep_ok(prep, l2_eps)) return KDA_ERR_INVALID_ARGUMENT;
    if (conv_w && (!conv_pool || !aligned_to(conv_w, 4) || !aligned_to(conv_pool, 4)))
        return KDA_ERR_INVALID_ARGUMENT;
    if (conv_w && A_total > 0 && (!q || !aligned16(q))) return KDA_ERR_INVALID_ARGUMENT;
    if (N < 0 || A_total < 0 || H <= 0 || num_slots < 0) return KDA_ERR_INVALID_ARGUMENT;
    if (!workspace || !aligned16(workspace) || ws_bytes < KDA_WS_HEADER_BYTES) return KDA_ERR_WORKSPACE;
    if (N > 0) {
        if (!state_pool || !cu_accept) return KDA_ERR_INVALID_ARGUMENT;
        if (!aligned16(state_pool) || !aligned_to(cu_accept, 4)) return KDA_ERR_INVALID_ARGUMENT;
        if (slots && !aligned_to(slots, 4)) return KDA_ERR_INVALID_ARGUMENT;
        if (!slots && N > num_slots) return KDA_ERR_INVALID_ARGUMENT;
    }
    if (A_total > 0) {
        if (!k || !v || !g || !beta) return KDA_ERR_INVALID_ARGUMENT;
        if (!aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned_to(beta, elem_size(dtype)))
            return KDA_ERR_INVALID_ARGUMENT;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    kda_status st = clear_status(workspace, s);
    if (st != KDA_OK || N == 0) return st;

    kda::SeqParams sp{};
    sp.q = conv_w ? q : nullptr; sp.k = k; sp.v = v; sp.g = g; sp.beta = beta; sp.o = nullptr;
    sp.N = N; sp.H = H; sp.scale = 1.0f;
    sp.mode = kda::SEQ_MODE_REPLAY;
    sp.cu = cu_accept; sp.T_total = A_total; sp.seq_len_fixed = 0; sp.chunk_skip = 0;
    sp.state_in = state_pool; sp.state_out = state_pool; sp.chunk_state = nullptr;
    sp.slots = slots; sp.num_slots = num_slots; sp.status = static_cast<uint32_t *>(workspace);
    sp.prep = static_cast<int>(prep & ~static_cast<uint32_t>(KDA_PREP_L2NORM_Q)); sp.prep_eps = l2_eps;  // no q in replay
    sp.conv_w = conv_w; sp.conv_state = conv_pool;  // q only advances the convolution state
    if (kda::launch_seq(sp, dk, dv, static_cast<int>(dtype), s) != cudaSuccess) return KDA_ERR_CUDA;
    return KDA_OK;
}

kda_status kda_replay_prep(float *state_pool, int64_t num_slots, const int32_t *slots, const void *k,
                           const void *v, const void *g, const void *beta, kda_dtype dtype,
                           const int32_t *cu_accept, int N, int64_t A_total, int H, int dk, int dv, uint32_t prep,
                           float l2_eps, void *workspace, size_t ws_bytes, void *stream) {
    return replay_impl(state_pool, num_slots, slots, nullptr, k, v, g, beta, dtype, cu_accept, N, A_total, H, dk, dv,
                       prep, l2_eps, nullptr, nullptr, workspace, ws_bytes, stream);
}

kda_status kda_replay_conv(float *state_pool, int64_t num_slots, const int32_t *slots, const void *q, const void *k,
                           const void *v, const void *g, const void *beta, kda_dtype dtype,
                           const int32_t *cu_accept, int N, int64_t A_total, int H, int dk, int dv,
                           const float *conv_weight, int conv_width, float *conv_pool, uint32_t prep, float l2_eps,
                           void *workspace, size_t ws_bytes, void *stream) {
    if (conv_width != KDA_CONV_WIDTH) return KDA_ERR_UNSUPPORTED;
    if (!conv_weight || !conv_pool) return KDA_ERR_INVALID_ARGUMENT;
    return replay_impl(state_pool, num_slots, slots, q, k, v, g, beta, dtype, cu_accept, N, A_total, H, dk, dv, prep,
                       l2_eps, conv_weight, conv_pool, workspace, ws_bytes, stream);
}

kda_status kda_conv_fwd(const void *q, const void *k, const void *v, kda_dtype dtype, const float *conv_weight,
                        int conv_width, const float *conv_state_in, const int32_t *cu_seqlens, int N, int64_t T_total,
                        int H, int dk, int dv, void *q_out, void *k_out, void *v_out, float *conv_state_out,
                        void *workspace, size_t ws_bytes, void *stream) {
    if (!dtype_ok(dtype) || !dim_ok(dk) || !dim_ok(dv) || conv_width != KDA_CONV_WIDTH) return KDA_ERR_UNSUPPORTED;
    if (N < 0 || T_total < 0 || H <= 0) return KDA_ERR_INVALID_ARGUMENT;
    if (!workspace || !aligned16(workspace) || ws_bytes < KDA_WS_HEADER_BYTES) return KDA_ERR_WORKSPACE;
    if (!conv_weight || !aligned_to(conv_weight, 4)) return KDA_ERR_INVALID_ARGUMENT;
    if (T_total > 0) {
        if (!q || !k || !v || !q_out || !k_out || !v_out) return KDA_ERR_INVALID_ARGUMENT;
        for (const void *ptr : {q, k, v, static_cast<const void *>(q_out), static_cast<const void *>(k_out),
                                static_cast<const void *>(v_out)})
            if (!aligned16(ptr)) return KDA_ERR_INVALID_ARGUMENT;  // 16-byte vector accesses
    }
    if ((conv_state_in && !aligned_to(conv_state_in, 4)) || (conv_state_out && !aligned_to(conv_state_out, 4)))
        return KDA_ERR_INVALID_ARGUMENT;
    if (!cu_seqlens && N > 0 && (T_total % N) != 0) return KDA_ERR_INVALID_ARGUMENT;
    if (!cu_seqlens && N == 0 && T_total != 0) return KDA_ERR_INVALID_ARGUMENT;
    if (cu_seqlens && !aligned_to(cu_seqlens, 4)) return KDA_ERR_INVALID_ARGUMENT;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    kda_status st = clear_status(workspace, s);
    if (st != KDA_OK || N == 0) return st;
    kda::ConvParams cp{};
    cp.q = q; cp.k = k; cp.v = v; cp.q_out = q_out; cp.k_out = k_out; cp.v_out = v_out;
    cp.weight = conv_weight; cp.state_in = conv_state_in; cp.state_out = conv_state_out;
    cp.cu = cu_seqlens; cp.T_total = T_total; cp.seq_len_fixed = cu_seqlens ? 0 : T_total / N;
    cp.N = N; cp.H = H; cp.dk = dk; cp.dv = dv; cp.status = static_cast<uint32_t *>(workspace);
    if (kda::launch_conv(cp, static_cast<int>(dtype), s) != cudaSuccess) return KDA_ERR_CUDA;
    return KDA_OK;
}

kda_status kda_replay(float *state_pool, int64_t num_slots, const int32_t *slots, const void *k,
                      const void *v, const void *g, const void *beta, kda_dtype dtype,
                      const int32_t *cu_accept, int N, int64_t A_total, int H, int dk, int dv,
                      void *workspace, size_t ws_bytes, void *stream) {
    return kda_replay_prep(state_pool, num_slots, slots, k, v, g, beta, dtype, cu_accept, N, A_total, H, dk, dv, 0u,
                           0.f, workspace, ws_bytes, stream);
}

// Backward workspace: header | checkpoints | records (both nslots x H) | staging states
// (N x H) | persistent-CTA scratch (kBwdMaxCtas) | two states per (sequence, head).
constexpr int kBwdMaxCtas = 320;  // two per SM

static int64_t bwd_slots(int N, int64_t T_total) { return T_total / 64 + N + 1; }

static size_t bwd_layout(int N, int64_t T_total, int H, int dk, int dv, size_t *ckpt_off, size_t *rec_off,
                         size_t *stage_off, size_t *scratch_off) {
    const size_t st = static_cast<size_t>(dk) * dv * sizeof(float);
    const size_t slots = static_cast<size_t>(bwd_slots(N, T_total)) * H;
    size_t off = KDA_WS_HEADER_BYTES;
    *ckpt_off = off;
    off += slots * st;
    *rec_off = off;
    off += slots * kda::bwd_record_floats(dk, dv) * sizeof(float);
    *stage_off = off;
    off += static_cast<size_t>(N) * H * st;
    *scratch_off = off;
    off += static_cast<size_t>(kBwdMaxCtas) * kda::bwd_scratch_floats(dk, dv) * sizeof(float) +
           static_cast<size_t>(N) * H * 2 * st;
    return off;
}

size_t kda_chunk_bwd_workspace_size(int N, int64_t T_total, int H, int dk, int dv) {
    if (N < 0 || T_total < 0 || H <= 0 || !dim_ok(dk) || !dim_ok(dv)) return 0;
    size_t a, b, c, d;
    return bwd_layout(N, T_total, H, dk, dv, &a, &b, &c, &d);
}

kda_status kda_chunk_bwd_prep(const void *q, const void *k, const void *v, const void *g, const void *beta,
                              kda_dtype dtype, const float *init_state, const int32_t *cu_seqlens, int N,
                              int64_t T_total, int H, int dk, int dv, float scale, uint32_t prep, float l2_eps,
                              const void *d_o, const float *d_final_state, void *dq, void *dk_out, void *dv_out,
                              void *dg, void *dbeta, float *d_init_state, void *workspace, size_t ws_bytes,
                              void *stream) {
    if (!dtype_ok(dtype) || !dim_ok(dk) || !dim_ok(dv)) return KDA_ERR_UNSUPPORTED;
    if (!prep_ok(prep, l2_eps)) return KDA_ERR_INVALID_ARGUMENT;
    if (N < 0 || T_total < 0 || H <= 0) return KDA_ERR_INVALID_ARGUMENT;
    if (!workspace || !aligned16(workspace)) return KDA_ERR_WORKSPACE;
    if (ws_bytes < kda_chunk_bwd_workspace_size(N, T_total, H, dk, dv)) return KDA_ERR_WORKSPACE;
    const size_t es = elem_size(dtype);
    if (T_total > 0) {
        if (!q || !k || !v || !g || !beta || !d_o || !dq || !dk_out || !dv_out || !dg || !dbeta)
            return KDA_ERR_INVALID_ARGUMENT;
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g)) return KDA_ERR_INVALID_ARGUMENT;
        for (const void *ptr : {beta, d_o, static_cast<const void *>(dq), static_cast<const void *>(dk_out),
                                static_cast<const void *>(dv_out), static_cast<const void *>(dg),
                                static_cast<const void *>(dbeta)})
            if (!aligned_to(ptr, es)) return KDA_ERR_INVALID_ARGUMENT;
    }
    if ((init_state && !aligned16(init_state)) || (d_final_state && !aligned_to(d_final_state, 4)) ||
        (d_init_state && !aligned_to(d_init_state, 4)))
        return KDA_ERR_INVALID_ARGUMENT;
    if (!cu_seqlens && N > 0 && (T_total % N) != 0) return KDA_ERR_INVALID_ARGUMENT;
    if (!cu_seqlens && N == 0 && T_total != 0) return KDA_ERR_INVALID_ARGUMENT;
    if (cu_seqlens && !aligned_to(cu_seqlens, 4)) return KDA_ERR_INVALID_ARGUMENT;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    kda_status st = clear_status(workspace, s);
    if (st != KDA_OK) return st;
    if (N == 0) return KDA_OK;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return KDA_ERR_CUDA;
    uint32_t *status = static_cast<uint32_t *>(workspace);
    size_t ckpt_off, rec_off, stage_off, scratch_off;
    bwd_layout(N, T_total, H, dk, dv, &ckpt_off, &rec_off, &stage_off, &scratch_off);
    char *ws = static_cast<char *>(workspace);
    float *ckpt = reinterpret_cast<float *>(ws + ckpt_off);
    const int64_t fixed_len = cu_seqlens ? 0 : T_total / N;

    // forward pass leaving the chunk-start states: the tensor-core kernel (no outputs) where
    // it serves the shape, else the token-sequential kernel
    if (kda::chunk_tc_supported(dk, dv, static_cast<int>(dtype)) && T_total <= 0x7fffffffLL) {
        kda::ChunkParams cp{};
        cp.q = q; cp.k = k; cp.v = v; cp.g = g; cp.beta = beta; cp.o = nullptr;
        cp.N = N; cp.H = H; cp.dk = dk; cp.dv = dv; cp.scale = scale; cp.cu = cu_seqlens; cp.T_total = T_total;
        cp.seq_len_fixed = fixed_len; cp.init_state = init_state;
        cp.state_out = reinterpret_cast<float *>(ws + stage_off); cp.status = status; cp.split = 0;
        cp.ckpt = ckpt; cp.prep = static_cast<int>(prep); cp.prep_eps = l2_eps;
        if (kda::launch_chunk_tc(cp, s) != cudaSuccess) return KDA_ERR_CUDA;
    } else {
        kda::SeqParams sp{};
        sp.q = q; sp.k = k; sp.v = v; sp.g = g; sp.beta = beta; sp.o = nullptr;
        sp.N = N; sp.H = H; sp.scale = scale; sp.mode = kda::SEQ_MODE_PREFILL;
        sp.cu = cu_seqlens; sp.T_total = T_total; sp.seq_len_fixed = fixed_len; sp.chunk_skip = 0;
        sp.state_in = init_state; sp.state_out = nullptr; sp.chunk_state = nullptr;
        sp.slots = nullptr; sp.num_slots = 0; sp.status = status; sp.ckpt = ckpt;
        sp.prep = static_cast<int>(prep); sp.prep_eps = l2_eps;
        if (kda::launch_seq(sp, dk, dv, static_cast<int>(dtype), s) != cudaSuccess) return KDA_ERR_CUDA;
    }

    kda::BwdParams bp{};
    bp.q = q; bp.k = k; bp.v = v; bp.g = g; bp.beta = beta; bp.d_o = d_o;
    bp.init_state = init_state; bp.d_final = d_final_state;
    bp.dq = dq; bp.dk = dk_out; bp.dv = dv_out; bp.dg = dg; bp.dbeta = dbeta; bp.d_init = d_init_state;
    bp.ckpt = ckpt; bp.rec = reinterpret_cast<float *>(ws + rec_off);
    bp.scratch = reinterpret_cast<float *>(ws + scratch_off);
    bp.ctas = 2 * sms < kBwdMaxCtas ? 2 * sms : kBwdMaxCtas;
    bp.nslots = bwd_slots(N, T_total);
    bp.cu = cu_seqlens; bp.T_total = T_total; bp.seq_len_fixed = fixed_len;
    bp.N = N; bp.H = H; bp.scale = scale; bp.status = status;
    bp.prep = static_cast<int>(prep); bp.prep_eps = l2_eps;
    if (kda::launch_bwd(bp, dk, dv, static_cast<int>(dtype), s) != cudaSuccess) return KDA_ERR_CUDA;
    return KDA_OK;
}

kda_status kda_chunk_bwd(const void *q, const void *k, const void *v, const void *g, const void *beta,
                         kda_dtype dtype, const float *init_state, const int32_t *cu_seqlens, int N,
                         int64_t T_total, int H, int dk, int dv, float scale, const void *d_o,
                         const float *d_final_state, void *dq, void *dk_out, void *dv_out, void *dg, void *dbeta,
                         float *d_init_state, void *workspace, size_t ws_bytes, void *stream) {
    return kda_chunk_bwd_prep(q, k, v, g, beta, dtype, init_state, cu_seqlens, N, T_total, H, dk, dv, scale, 0u, 0.f,
                              d_o, d_final_state, dq, dk_out, dv_out, dg, dbeta, d_init_state, workspace, ws_bytes,
                              stream);
}

kda_status kda_device_status(const void *workspace, void *stream) {
    if (!workspace) return KDA_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return KDA_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return KDA_ERR_CUDA;
    if (word & kda::DEV_ERR_SEQLENS) return KDA_ERR_BAD_SEQLENS;
    if (word & kda::DEV_ERR_SLOT) return KDA_ERR_BAD_SLOT;
    if (word & kda::DEV_ERR_GATE) return KDA_ERR_GATE_RANGE;
    if (word & kda::DEV_ERR_TIMEOUT) return KDA_ERR_TIMEOUT;
    return KDA_OK;
}

int kda_chunk_fwd_uses_tensor_cores(int dk, int dv, kda_dtype dtype) {
    if (!dtype_ok(dtype) || !dim_ok(dk) || !dim_ok(dv)) return 0;
    return kda::chunk_tc_supported(dk, dv, static_cast<int>(dtype)) ? 1 : 0;
}

const char *kda_status_string(kda_status status) {
    switch (status) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARGUMENT: return "KDA_ERR_INVALID_ARGUMENT";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
        case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
        case KDA_ERR_GATE_RANGE: return "KDA_ERR_GATE_RANGE";
        case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT";
        case KDA_ERR_BAD_SEQLENS: return "KDA_ERR_BAD_SEQLENS";
        case KDA_ERR_BAD_SLOT: return "KDA_ERR_BAD_SLOT";
    }
    return "KDA_ERR_UNKNOWN";
}

int kda_version(void) { return kVersion; }

}  // extern "C"
