// Short causal convolution of the input projections q, k, v before the KDA
// recurrence, with the convolution state carried across calls.  "Kimi K3 on
// Fireworks: Fast RL at frontier scale" (disaggregated-serving paragraph) says a
// handoff must move KDA's recurrent and convolution state; the pages define
// neither the convolution nor its width.  The reading implemented: a depthwise
// causal 1-D convolution of width kConvW = 4 over the tokens of each sequence,
// one weight vector per channel, followed by SiLU:
//
//   pre_t[c] = sum_{i=0}^{3} w[h][c][i] x_{t-3+i}[c],   y_t[c] = pre / (1 + exp(-pre))
//
// with the channels of a head packed as (q 0..dk-1 | k dk..2dk-1 | v 2dk..2dk+dv-1),
// tokens before a sequence's first taken from its state (the 3 previous inputs,
// oldest first), and the new state = the last 3 inputs of (state ++ tokens).
//
// This file is the prefill form (two launches: outputs, then states); decode and
// replay apply the same convolution token by token inside the token-sequential
// kernel.  Every sum runs in the order i = 0..3 with round-to-nearest intrinsics.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float ld_in(const float *p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ld_in(const __nv_bfloat16 *p, int64_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void st_out(float *p, int64_t i, float x) { p[i] = x; }
__device__ __forceinline__ void st_out(__nv_bfloat16 *p, int64_t i, float x) { p[i] = __float2bfloat16_rn(x); }

// Sequence of token t: the largest n with first token <= t.
__device__ __forceinline__ int seq_of(const ConvParams &p, int64_t t) {
    if (!p.cu) return static_cast<int>(t / p.seq_len_fixed);
    int lo = 0, hi = p.N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.cu[mid] <= t) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ bool seq_bounds(const ConvParams &p, int n, int64_t &bos, int64_t &eos) {
    if (p.cu) {
        bos = p.cu[n];
        eos = p.cu[n + 1];
        bool ok = (bos >= 0) && (bos <= eos) && (eos <= p.T_total);
        if (n == 0 && bos != 0) ok = false;
        if (n == p.N - 1 && eos != p.T_total) ok = false;
        return ok;
    }
    bos = static_cast<int64_t>(n) * p.seq_len_fixed;
    eos = bos + p.seq_len_fixed;
    return true;
}

// Raw input of packed channel c (q | k | v) of token `src` of head h, or the state's
// entry `back` positions before the first token (1 <= back <= 3).
template <typename Tin>
__device__ __forceinline__ float conv_input(const ConvParams &p, int64_t src, int64_t bos, int n, int h, int c,
                                            int Ct) {
    const int64_t H = p.H;
    if (src >= bos) {
        if (c < p.dk) return ld_in(static_cast<const Tin *>(p.q), (src * H + h) * p.dk + c);
        if (c < 2 * p.dk) return ld_in(static_cast<const Tin *>(p.k), (src * H + h) * p.dk + c - p.dk);
        return ld_in(static_cast<const Tin *>(p.v), (src * H + h) * p.dv + c - 2 * p.dk);
    }
    if (!p.state_in) return 0.f;
    const int64_t back = bos - src;
    return p.state_in[((static_cast<int64_t>(n) * (kConvW - 1) + (kConvW - 1 - back)) * H + h) * Ct + c];
}

// One thread per (token, head, packed channel).
template <typename Tin>
__global__ void __launch_bounds__(kThreads) conv_out_kernel(ConvParams p) {
    const int Ct = 2 * p.dk + p.dv;
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    if (idx >= p.T_total * p.H * Ct) return;
    const int c = static_cast<int>(idx % Ct);
    const int h = static_cast<int>((idx / Ct) % p.H);
    const int64_t t = idx / (static_cast<int64_t>(Ct) * p.H);
    const int n = seq_of(p, t);
    int64_t bos, eos;
    if (!seq_bounds(p, n, bos, eos) || t < bos || t >= eos) {
        if (c == 0 && h == 0) atomicOr(p.status, DEV_ERR_SEQLENS);
        return;
    }
    const float *w = p.weight + (static_cast<int64_t>(h) * Ct + c) * kConvW;
    float pre = 0.f;
#pragma unroll
    for (int i = 0; i < kConvW; ++i) pre = __fmaf_rn(w[i], conv_input<Tin>(p, t - (kConvW - 1) + i, bos, n, h, c, Ct), pre);
    const float y = __fdiv_rn(pre, __fadd_rn(1.f, expf(-pre)));
    const int64_t H = p.H;
    if (c < p.dk) st_out(static_cast<Tin *>(p.q_out), (t * H + h) * p.dk + c, y);
    else if (c < 2 * p.dk) st_out(static_cast<Tin *>(p.k_out), (t * H + h) * p.dk + c - p.dk, y);
    else st_out(static_cast<Tin *>(p.v_out), (t * H + h) * p.dv + c - 2 * p.dk, y);
}

// One thread per (sequence, head, packed channel): the new state, slots in increasing
// order (slot j reads old slot j + len, so an in-place update is safe).
template <typename Tin>
__global__ void __launch_bounds__(kThreads) conv_state_kernel(ConvParams p) {
    const int Ct = 2 * p.dk + p.dv;
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    if (idx >= static_cast<int64_t>(p.N) * p.H * Ct) return;
    const int c = static_cast<int>(idx % Ct);
    const int h = static_cast<int>((idx / Ct) % p.H);
    const int n = static_cast<int>(idx / (static_cast<int64_t>(Ct) * p.H));
    int64_t bos, eos;
    if (!seq_bounds(p, n, bos, eos)) return;  // reported by the output kernel
    const int64_t H = p.H;
    for (int j = 0; j < kConvW - 1; ++j) {
        const float x = conv_input<Tin>(p, eos - (kConvW - 1) + j, bos, n, h, c, Ct);
        p.state_out[((static_cast<int64_t>(n) * (kConvW - 1) + j) * H + h) * Ct + c] = x;
    }
}

template <typename Tin>
cudaError_t launch_typed(const ConvParams &p, cudaStream_t s) {
    const int64_t Ct = 2 * p.dk + p.dv;
    const int64_t n_out = p.T_total * p.H * Ct, n_state = static_cast<int64_t>(p.N) * p.H * Ct;
    const int64_t b_out = (n_out + kThreads - 1) / kThreads, b_state = (n_state + kThreads - 1) / kThreads;
    if (b_out > 0x7fffffffLL || b_state > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (b_out > 0) conv_out_kernel<Tin><<<static_cast<unsigned>(b_out), kThreads, 0, s>>>(p);
    if (p.state_out && b_state > 0) conv_state_kernel<Tin><<<static_cast<unsigned>(b_state), kThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_conv(const ConvParams &p, int dtype, cudaStream_t stream) {
    if (dtype == 0) return launch_typed<__nv_bfloat16>(p, stream);
    return launch_typed<float>(p, stream);
}

}  // namespace kda
