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
// kernel.  Every sum runs in the order i = 0..3 with round-to-nearest intrinsics; the
// prefill form takes SiLU with the fast exp / divide intrinsics (its outputs are rounded
// to the input dtype), the fused form with correctly rounded ones.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float ld_in(const float *p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ld_in(const __nv_bfloat16 *p, int64_t i) { return __bfloat162float(p[i]); }

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

// Raw rows of 4 channels, kept undecoded until they are used (bf16: 8 bytes, fp32: 16).
template <typename Tin>
struct Raw4;
template <>
struct Raw4<__nv_bfloat16> {
    uint2 u;
    __device__ __forceinline__ void load(const __nv_bfloat16 *p) { u = *reinterpret_cast<const uint2 *>(p); }
    __device__ __forceinline__ void get(float (&x)[4]) const {
        x[0] = __uint_as_float(u.x << 16);
        x[1] = __uint_as_float(u.x & 0xffff0000u);
        x[2] = __uint_as_float(u.y << 16);
        x[3] = __uint_as_float(u.y & 0xffff0000u);
    }
};
template <>
struct Raw4<float> {
    float4 a;
    __device__ __forceinline__ void load(const float *p) { a = *reinterpret_cast<const float4 *>(p); }
    __device__ __forceinline__ void get(float (&x)[4]) const {
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    }
};
__device__ __forceinline__ void ld4f(const float *p, float (&x)[4]) {
    const float4 a = *reinterpret_cast<const float4 *>(p);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
}
__device__ __forceinline__ void ld4f(const __nv_bfloat16 *p, float (&x)[4]) {
    Raw4<__nv_bfloat16> r;
    r.load(p);
    r.get(x);
}
__device__ __forceinline__ void st4(float *p, const float (&y)[4]) {
    *reinterpret_cast<float4 *>(p) = make_float4(y[0], y[1], y[2], y[3]);
}
__device__ __forceinline__ void st4(__nv_bfloat16 *p, const float (&y)[4]) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(y[0], y[1]), b = __floats2bfloat162_rn(y[2], y[3]);
    *reinterpret_cast<uint2 *>(p) = make_uint2(*reinterpret_cast<const uint32_t *>(&a), *reinterpret_cast<const uint32_t *>(&b));
}

// A thread owns 4 consecutive channels (all in one of q, k, v) of one head and slides the
// width-4 window down a block of kConvBlock tokens, so every input is loaded once (a warp
// reads 256 contiguous bytes of bf16 per token).  The rows are loaded 16 tokens at a time
// before any is used, so a batch costs one memory latency instead of one per token, and few
// enough registers stay live that two CTAs fit on an SM.  The window restarts from the
// sequence's state where a sequence begins inside the block.  Grid: token blocks x groups of
// kConvThreads (head, channel group) pairs.
constexpr int kConvBlock = 64;
constexpr int kConvThreads = 256;
constexpr int kConvCh = 4;  // channels per thread

template <typename Tin>
__global__ void __launch_bounds__(kConvThreads, 2) conv_out_kernel(ConvParams p) {
    constexpr int kBatch = 16;
    static_assert(kConvBlock % kBatch == 0, "batch");
    const int Ct = 2 * p.dk + p.dv, G = Ct / kConvCh;
    const int u = static_cast<int>(blockIdx.y) * kConvThreads + threadIdx.x;
    if (u >= p.H * G) return;
    const int h = u / G, c0 = (u % G) * kConvCh;
    const int64_t H = p.H;
    // which tensor the group lies in, its channel offset there and row length
    const Tin *X;
    Tin *Y;
    int cx, d;
    if (c0 < p.dk) { X = static_cast<const Tin *>(p.q); Y = static_cast<Tin *>(p.q_out); cx = c0; d = p.dk; }
    else if (c0 < 2 * p.dk) { X = static_cast<const Tin *>(p.k); Y = static_cast<Tin *>(p.k_out); cx = c0 - p.dk; d = p.dk; }
    else { X = static_cast<const Tin *>(p.v); Y = static_cast<Tin *>(p.v_out); cx = c0 - 2 * p.dk; d = p.dv; }
    float w[kConvCh][kConvW];
#pragma unroll
    for (int e = 0; e < kConvCh; ++e)
#pragma unroll
        for (int i = 0; i < kConvW; ++i) w[e][i] = p.weight[(static_cast<int64_t>(h) * Ct + c0 + e) * kConvW + i];
    const int64_t t_begin = static_cast<int64_t>(blockIdx.x) * kConvBlock;
    const int64_t t_end = t_begin + kConvBlock < p.T_total ? t_begin + kConvBlock : p.T_total;
    int n = seq_of(p, t_begin);
    int64_t bos, eos;
    if (!seq_bounds(p, n, bos, eos)) {
        if (u == 0) atomicOr(p.status, DEV_ERR_SEQLENS);
        return;
    }
    float hw[kConvW - 1][kConvCh];  // the window: inputs t-3, t-2, t-1
    auto window_at = [&](int64_t t) {
#pragma unroll
        for (int j = 0; j < kConvW - 1; ++j) {
            const int64_t src = t - (kConvW - 1) + j;
            if (src >= bos) {
                ld4f(X + (src * H + h) * d + cx, hw[j]);
            } else if (p.state_in) {
                const int64_t back = bos - src;
                const float *sp = p.state_in + ((static_cast<int64_t>(n) * (kConvW - 1) + (kConvW - 1 - back)) * H + h) * Ct + c0;
#pragma unroll
                for (int e = 0; e < kConvCh; ++e) hw[j][e] = sp[e];
            } else {
#pragma unroll
                for (int e = 0; e < kConvCh; ++e) hw[j][e] = 0.f;
            }
        }
    };
    window_at(t_begin);
    for (int64_t tb = t_begin; tb < t_end; tb += kBatch) {
        Raw4<Tin> r[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b)
            if (tb + b < t_end) r[b].load(X + ((tb + b) * H + h) * d + cx);
        // the next batch's rows into L2 while this one is computed (no registers held)
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int64_t tn = tb + kBatch + b;
            if (tn < t_end) asm volatile("prefetch.global.L2 [%0];" ::"l"(X + (tn * H + h) * d + cx));
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int64_t t = tb + b;
            if (t >= t_end) break;
            if (t >= eos) {  // the next sequence (skipping empty ones) starts here
                while (n + 1 < p.N && t >= eos) {
                    ++n;
                    if (!seq_bounds(p, n, bos, eos)) {
                        if (u == 0) atomicOr(p.status, DEV_ERR_SEQLENS);
                        return;
                    }
                }
                window_at(t);
            }
            float x[kConvCh], y[kConvCh];
            r[b].get(x);
#pragma unroll
            for (int e = 0; e < kConvCh; ++e) {
                float pre = __fmaf_rn(w[e][0], hw[0][e], 0.f);
                pre = __fmaf_rn(w[e][1], hw[1][e], pre);
                pre = __fmaf_rn(w[e][2], hw[2][e], pre);
                pre = __fmaf_rn(w[e][3], x[e], pre);
                y[e] = __fdividef(pre, 1.f + __expf(-pre));  // SiLU (fast intrinsics; the outputs are rounded to Tin)
                hw[0][e] = hw[1][e];
                hw[1][e] = hw[2][e];
                hw[2][e] = x[e];
            }
            st4(Y + (t * H + h) * d + cx, y);
        }
    }
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
    const int64_t n_state = static_cast<int64_t>(p.N) * p.H * Ct;
    const int64_t b_out = (p.T_total + kConvBlock - 1) / kConvBlock, b_state = (n_state + kThreads - 1) / kThreads;
    const int64_t b_grp = (static_cast<int64_t>(p.H) * (Ct / kConvCh) + kConvThreads - 1) / kConvThreads;
    if (b_out > 0x7fffffffLL || b_state > 0x7fffffffLL || b_grp > 65535) return cudaErrorInvalidConfiguration;
    if (b_out > 0)
        conv_out_kernel<Tin><<<dim3(static_cast<unsigned>(b_out), static_cast<unsigned>(b_grp)), kConvThreads, 0, s>>>(p);
    if (p.state_out && b_state > 0) conv_state_kernel<Tin><<<static_cast<unsigned>(b_state), kThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_conv(const ConvParams &p, int dtype, cudaStream_t stream) {
    if (dtype == 0) return launch_typed<__nv_bfloat16>(p, stream);
    return launch_typed<float>(p, stream);
}

}  // namespace kda
