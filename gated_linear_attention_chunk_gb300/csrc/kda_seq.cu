// Token-sequential KDA kernel: decode, ReplaySSM replay, and the partial-chunk
// tail of the packed prefill.
//
// Per (sequence, head) the gated delta rule with per-channel decay is stepped
// one token at a time on an fp32 state held in registers ("Kimi K3 on
// Fireworks: Fast RL at frontier scale", KDA paragraph: compact recurrent state
// with channel-wise gating; speculative-decoding paragraph: replay of accepted
// tokens from a committed checkpoint).  For token t with alpha = exp(g_t):
//
//     S' = Diag(alpha) S
//     y  = S'^T k,  z = S'^T (scale q),  qk = (scale q) . k
//     u  = beta (v - y)
//     S  = S' + k u^T
//     o  = z + qk u            (= S^T (scale q), the output after the update)
//
// Computing z and qk from the decayed state lets one reduction pass serve both
// the delta step and the output, so each token costs one __syncthreads.
//
// Layout: the dv columns of S follow independent recurrences (y, u and the update
// of column j involve column j only), so a CTA owns one block of 32 columns of
// one (sequence, head): 128 threads, a thread holding dk/16 rows x 4 consecutive
// columns (float4, 128-bit loads/stores).  Four column blocks per state give the
// SM many small CTAs, whose state loads overlap the other CTAs' token steps.
// Reductions over dk run in a fixed order (rows in order inside a thread, then
// the four row groups of a warp as (0+1)+(2+3), then warps 0..3 in order), and
// every floating-point step of the recurrence uses an explicit round-to-nearest
// intrinsic.  The optional preprocessing's sigmoid, SiLU and inverse row norm use the
// fast exp, divide and reciprocal-square-root intrinsics (deterministic, a few ulp; they
// sit on the token path, and the IEEE-rounded forms cost replay with the fused
// convolution 18% of its bandwidth).
// Every caller of this routine -- decode, replay and the prefill tail -- runs the
// same code, so it produces the same bits for the same state and tokens.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kSeqThreads = 128;
constexpr int kSeqWarps = kSeqThreads / 32;
constexpr int kColBlock = 32;  // state columns per CTA

__device__ __forceinline__ float ld_in(const float *p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ld_in(const __nv_bfloat16 *p, int64_t i) { return __bfloat162float(p[i]); }

__device__ __forceinline__ void st_out4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ void st_out4(__nv_bfloat16 *p, float4 v) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 packed;
    packed.x = *reinterpret_cast<uint32_t *>(&lo);
    packed.y = *reinterpret_cast<uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(p) = packed;
}

// float4 arithmetic as two packed f32x2 instructions each (per-lane IEEE round to
// nearest, so the bits equal four scalar __fmaf_rn / __fadd_rn / __fmul_rn)
__device__ __forceinline__ uint64_t f2u(float x, float y) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(x), "f"(y));
    return d;
}
__device__ __forceinline__ float2 u2f(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(f2u(a.x, a.y)), "l"(f2u(b.x, b.y)), "l"(f2u(c.x, c.y)));
    return u2f(d);
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2u(a.x, a.y)), "l"(f2u(b.x, b.y)));
    return u2f(d);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2u(a.x, a.y)), "l"(f2u(b.x, b.y)));
    return u2f(d);
}
__device__ __forceinline__ float4 f4_fma(float a, float4 b, float4 c) {
    const float2 aa = make_float2(a, a);
    const float2 lo = fma2(aa, make_float2(b.x, b.y), make_float2(c.x, c.y));
    const float2 hi = fma2(aa, make_float2(b.z, b.w), make_float2(c.z, c.w));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}
__device__ __forceinline__ float4 f4_add(float4 a, float4 b) {
    const float2 lo = add2(make_float2(a.x, a.y), make_float2(b.x, b.y));
    const float2 hi = add2(make_float2(a.z, a.w), make_float2(b.z, b.w));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}
__device__ __forceinline__ float4 f4_scale(float4 a, float s) {
    const float2 ss = make_float2(s, s);
    const float2 lo = mul2(make_float2(a.x, a.y), ss);
    const float2 hi = mul2(make_float2(a.z, a.w), ss);
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}
__device__ __forceinline__ float4 f4_shfl_xor(float4 a, int m) {
    return make_float4(__shfl_xor_sync(0xffffffffu, a.x, m), __shfl_xor_sync(0xffffffffu, a.y, m),
                       __shfl_xor_sync(0xffffffffu, a.z, m), __shfl_xor_sync(0xffffffffu, a.w, m));
}

// PREP: the extended instance -- it applies the input preprocessing of p.prep and
// writes the chunk-start checkpoints of p.ckpt (the other one carries none of that code).
// Six CTAs per SM, except the instances that preprocess and write o (decode with the fused
// convolution or flags, the preprocessed prefill tail): they carry more live values and ran
// faster with five CTAs' worth of registers each (decode with the convolution: 5274 against
// 4924 GB/s), while the replay instances ran slower with fewer CTAs.
template <int DK, int DV, typename Tin, bool WRITE_O, bool PREP>
__global__ void __launch_bounds__(kSeqThreads, (PREP && WRITE_O) ? 5 : 6) kda_seq_kernel(SeqParams p) {
    constexpr int CB = kColBlock;         // columns of this CTA
    constexpr int NCB = DV / CB;          // column blocks per state
    constexpr int LPR = CB / 4;           // lanes per state row (8)
    constexpr int RPW = 32 / LPR;         // rows per warp per step (4)
    constexpr int RPS = kSeqWarps * RPW;  // rows per step (16)
    constexpr int NS = DK / RPS;          // rows per thread
    static_assert(LPR * RPW == 32 && RPW == 4 && NS * RPS == DK && NCB * CB == DV, "thread layout");

    __shared__ float tok_a[3][DK], tok_k[3][DK], tok_q[3][DK];
    __shared__ __align__(16) float tok_v[3][CB];
    __shared__ float tok_b[3];
    __shared__ float4 red_y[2][kSeqWarps][LPR], red_z[2][kSeqWarps][LPR];
    __shared__ float red_qk[2][kSeqWarps];
    __shared__ float red_nk[3][kSeqWarps], red_nq[3][kSeqWarps];  // per-warp sums of k^2, q^2 of a staged token

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cg = lane % LPR, rsub = lane / LPR;
    const int row0 = warp * RPW + rsub;
    const int64_t pair = blockIdx.x / NCB;
    const int cb = static_cast<int>(blockIdx.x % NCB), col0 = cb * CB;
    const int n = static_cast<int>(pair / p.H), h = static_cast<int>(pair % p.H);
    const int64_t H = p.H;

    // ---- resolve the token range and the state source/destination
    int64_t t0, t1;
    const float *src;
    float *dst;
    float *cst = nullptr;  // this sequence's short-convolution state (decode / replay with conv_w)
    if (p.mode == SEQ_MODE_DECODE) {
        t0 = n;
        t1 = n + 1;
    } else if (p.cu) {
        t0 = p.cu[n];
        t1 = p.cu[n + 1];
        bool ok = (t0 >= 0) && (t0 <= t1) && (t1 <= p.T_total);
        if (n == 0 && t0 != 0) ok = false;
        if (n == p.N - 1 && t1 != p.T_total) ok = false;
        if (!ok) {
            if (tid == 0 && h == 0 && cb == 0) atomicOr(p.status, DEV_ERR_SEQLENS);
            return;
        }
    } else {
        t0 = static_cast<int64_t>(n) * p.seq_len_fixed;
        t1 = t0 + p.seq_len_fixed;
    }
    if (p.mode == SEQ_MODE_PREFILL) {
        const int64_t len = t1 - t0;
        const bool redo = p.fallback && p.fallback[pair];  // the chunked kernel gave this chain up
        const int64_t nfull = (p.chunk_skip && !redo) ? len / 64 : 0;
        if (nfull > 0) {
            if (len % 64 == 0) return;  // the chunked kernel already left the final state
            src = p.chunk_state + pair * DK * DV;
            t0 += 64 * nfull;
        } else {
            src = p.state_in ? p.state_in + pair * DK * DV : nullptr;
        }
        dst = p.state_out ? p.state_out + pair * DK * DV : nullptr;
    } else {
        const int64_t slot = p.slots ? static_cast<int64_t>(p.slots[n]) : static_cast<int64_t>(n);
        if (slot < 0 || slot >= p.num_slots) {
            if (tid == 0 && h == 0 && cb == 0) atomicOr(p.status, DEV_ERR_SLOT);
            return;
        }
        src = p.state_in + (slot * H + h) * DK * DV;
        dst = p.state_out + (slot * H + h) * DK * DV;
        if constexpr (PREP) {
            if (p.conv_w) cst = p.conv_state + slot * (kConvW - 1) * H * (2 * DK + DV);
        }
    }

    const Tin *Q = static_cast<const Tin *>(p.q);
    const Tin *K = static_cast<const Tin *>(p.k);
    const Tin *V = static_cast<const Tin *>(p.v);
    const Tin *G = static_cast<const Tin *>(p.g);
    const Tin *B = static_cast<const Tin *>(p.beta);

    // ---- state into registers (128-bit loads; a warp reads whole rows)
    float4 S[NS];
#pragma unroll
    for (int s = 0; s < NS; ++s) {
        const int row = s * RPS + row0;
        S[s] = src ? *reinterpret_cast<const float4 *>(src + row * DV + col0 + 4 * cg) : make_float4(0.f, 0.f, 0.f, 0.f);
    }

    // Token staging: threads [0, DK) hold alpha/k/q of one channel, threads
    // [0, CB) also one value column of this block, the last thread beta.
    auto load_raw = [&](int64_t t, float &rg, float &rk, float &rq, float &rv, float &rb) {
        if (tid < DK) {
            const int64_t base = (t * H + h) * DK + tid;
            rg = ld_in(G, base);
            rk = ld_in(K, base);
            if (WRITE_O || (PREP && cst)) rq = ld_in(Q, base);
        }
        if (tid < CB) rv = ld_in(V, (t * H + h) * DV + col0 + tid);
        if (tid == kSeqThreads - 1) rb = ld_in(B, t * H + h);
    };
    // Optional preprocessing (p.prep): alpha = sigmoid(x_g) instead of exp(g), beta =
    // sigmoid(x_beta), and k / q rows divided by sqrt(sum of squares + eps); the row sums
    // are reduced here per warp (a xor butterfly gives every lane the same bits) and the
    // inverse norms are applied where k and q are read.
    // Short convolution (extended instance, decode / replay with conv_w): each thread keeps
    // its channel's last kConvW - 1 raw inputs and the kConvW weights in registers; the sum
    // runs oldest first with round-to-nearest multiply-adds, then SiLU (fast intrinsics).
    constexpr int Ct = 2 * DK + DV;
    float hq[kConvW - 1], hk[kConvW - 1], hv[kConvW - 1], wq[kConvW], wk[kConvW], wv[kConvW];
    if constexpr (PREP) {
        if (cst) {
#pragma unroll
            for (int j = 0; j < kConvW - 1; ++j) {
                const float *row = cst + (static_cast<int64_t>(j) * H + h) * Ct;
                hq[j] = tid < DK ? row[tid] : 0.f;
                hk[j] = tid < DK ? row[DK + tid] : 0.f;
                hv[j] = tid < CB ? row[2 * DK + col0 + tid] : 0.f;
            }
            const float *wrow = p.conv_w + static_cast<int64_t>(h) * Ct * kConvW;
#pragma unroll
            for (int i = 0; i < kConvW; ++i) {
                wq[i] = tid < DK ? wrow[tid * kConvW + i] : 0.f;
                wk[i] = tid < DK ? wrow[(DK + tid) * kConvW + i] : 0.f;
                wv[i] = tid < CB ? wrow[(2 * DK + col0 + tid) * kConvW + i] : 0.f;
            }
        }
    }
    auto conv_step = [&](float (&hist)[kConvW - 1], const float (&w)[kConvW], float x) {
        float pre = 0.f;
#pragma unroll
        for (int i = 0; i < kConvW - 1; ++i) pre = __fmaf_rn(w[i], hist[i], pre);
        pre = __fmaf_rn(w[kConvW - 1], x, pre);
#pragma unroll
        for (int i = 0; i < kConvW - 2; ++i) hist[i] = hist[i + 1];
        hist[kConvW - 2] = x;
        return __fdividef(pre, 1.f + __expf(-pre));
    };
    auto stage = [&](int buf, float rg, float rk, float rq, float rv, float rb) {
        if constexpr (PREP) {
            if (cst) {
                if (tid < DK) {
                    rq = conv_step(hq, wq, rq);
                    rk = conv_step(hk, wk, rk);
                }
                if (tid < CB) rv = conv_step(hv, wv, rv);
            }
        }
        if (tid < DK) {
            tok_a[buf][tid] = (PREP && (p.prep & PREP_SIGMOID_GATE)) ? __fdividef(1.f, 1.f + __expf(-rg)) : expf(rg);
            tok_k[buf][tid] = rk;
            if (WRITE_O) tok_q[buf][tid] = __fmul_rn(rq, p.scale);
        }
        if (tid < CB) tok_v[buf][tid] = rv;
        if (tid == kSeqThreads - 1)
            tok_b[buf] = (PREP && (p.prep & PREP_SIGMOID_BETA)) ? __fdividef(1.f, 1.f + __expf(-rb)) : rb;
        if constexpr (PREP) {
            if (p.prep & (PREP_L2NORM_K | PREP_L2NORM_Q)) {
                float sk = __fmul_rn(rk, rk), sq = __fmul_rn(rq, rq);  // 0 beyond dk
#pragma unroll
                for (int m = 16; m >= 1; m >>= 1) {
                    sk = __fadd_rn(sk, __shfl_xor_sync(0xffffffffu, sk, m));
                    sq = __fadd_rn(sq, __shfl_xor_sync(0xffffffffu, sq, m));
                }
                if (lane == 0) {
                    red_nk[buf][warp] = sk;
                    red_nq[buf][warp] = sq;
                }
            }
        }
    };
    // inverse L2 norm of a staged row from the warps' partial sums (warps in order), or 1
    auto inv_norm = [&](const float (&part)[kSeqWarps], int flag) {
        if (!PREP || !(p.prep & flag)) return 1.f;
        float t = part[0];
#pragma unroll
        for (int w = 1; w < kSeqWarps; ++w) t = __fadd_rn(t, part[w]);
        return rsqrtf(__fadd_rn(t, p.prep_eps));
    };

    // Warm L2 with the next three tokens' rows (fire and forget): in a multi-token call
    // (replay, prefill tail) each token's load would otherwise be a full memory round
    // trip between two dependent token steps.
    for (int64_t t = t0 + 1; t < t1 && t < t0 + 4; ++t) {
        if (tid < DK) {
            const int64_t base = (t * H + h) * DK + tid;
            asm volatile("prefetch.L2 [%0];" ::"l"(G + base));
            asm volatile("prefetch.L2 [%0];" ::"l"(K + base));
            if (WRITE_O) asm volatile("prefetch.L2 [%0];" ::"l"(Q + base));
        }
        if (tid < CB) asm volatile("prefetch.L2 [%0];" ::"l"(V + (t * H + h) * DV + col0 + tid));
        if (tid == kSeqThreads - 1) asm volatile("prefetch.L2 [%0];" ::"l"(B + t * H + h));
    }
    if (t0 < t1) {
        float rg = 0.f, rk = 0.f, rq = 0.f, rv = 0.f, rb = 0.f;
        load_raw(t0, rg, rk, rq, rv, rb);
        stage(0, rg, rk, rq, rv, rb);
    }
    __syncthreads();

    int64_t ck = 0;  // checkpoint slot of the chunk that starts at t0 (backward's forward pass)
    if constexpr (PREP) {
        if (p.ckpt) ck = (ckpt_base(t0, n) * H + h) * DK * DV + col0 + 4 * cg;
    }
    int it = 0;
    for (int64_t t = t0; t < t1; ++t, ++it) {
        const int b = it % 3, r = it & 1;
        if constexpr (PREP) {
            if (p.ckpt && (it & 63) == 0) {  // state before the first token of each chunk
                float *dstc = p.ckpt + ck + static_cast<int64_t>(it >> 6) * H * DK * DV;
#pragma unroll
                for (int s = 0; s < NS; ++s) *reinterpret_cast<float4 *>(dstc + (s * RPS + row0) * DV) = S[s];
            }
        }
        const bool has_next = (t + 1 < t1);
        float ng = 0.f, nk = 0.f, nq = 0.f, nv = 0.f, nb = 0.f;
        if (has_next) load_raw(t + 1, ng, nk, nq, nv, nb);

        // decay, then partial reductions over this thread's rows (rows in order)
        const float kn = inv_norm(red_nk[b], PREP_L2NORM_K);
        const float qn = WRITE_O ? inv_norm(red_nq[b], PREP_L2NORM_Q) : 1.f;
        float4 py = make_float4(0.f, 0.f, 0.f, 0.f), pz = py;
        float pqk = 0.f;
#pragma unroll
        for (int s = 0; s < NS; ++s) {
            const int row = s * RPS + row0;
            const float a = tok_a[b][row], kk = PREP ? __fmul_rn(tok_k[b][row], kn) : tok_k[b][row];
            S[s] = f4_scale(S[s], a);
            py = f4_fma(kk, S[s], py);
            if (WRITE_O) {
                const float qq = PREP ? __fmul_rn(tok_q[b][row], qn) : tok_q[b][row];
                pz = f4_fma(qq, S[s], pz);
                pqk = __fmaf_rn(qq, kk, pqk);
            }
        }
        // combine the warp's four row groups as (0 + 1) + (2 + 3); a + b == b + a exactly,
        // so every lane of a column ends with the same bits
        py = f4_add(py, f4_shfl_xor(py, LPR));
        py = f4_add(py, f4_shfl_xor(py, 2 * LPR));
        if (WRITE_O) {
            pz = f4_add(pz, f4_shfl_xor(pz, LPR));
            pz = f4_add(pz, f4_shfl_xor(pz, 2 * LPR));
            pqk = __fadd_rn(pqk, __shfl_xor_sync(0xffffffffu, pqk, LPR));
            pqk = __fadd_rn(pqk, __shfl_xor_sync(0xffffffffu, pqk, 2 * LPR));
        }
        if (rsub == 0) {
            red_y[r][warp][cg] = py;
            if (WRITE_O) red_z[r][warp][cg] = pz;
        }
        if (WRITE_O && lane == 0) red_qk[r][warp] = pqk;
        if (has_next) stage((it + 1) % 3, ng, nk, nq, nv, nb);
        __syncthreads();

        // every thread reduces the warps' partials for its columns, warps in order
        float4 y = red_y[r][0][cg];
#pragma unroll
        for (int w = 1; w < kSeqWarps; ++w) y = f4_add(y, red_y[r][w][cg]);
        const float4 vv = *reinterpret_cast<const float4 *>(&tok_v[b][4 * cg]);
        const float bt = tok_b[b];
        const float4 u = make_float4(__fmul_rn(bt, __fsub_rn(vv.x, y.x)), __fmul_rn(bt, __fsub_rn(vv.y, y.y)),
                                     __fmul_rn(bt, __fsub_rn(vv.z, y.z)), __fmul_rn(bt, __fsub_rn(vv.w, y.w)));
#pragma unroll
        for (int s = 0; s < NS; ++s) {
            const float kk = tok_k[b][s * RPS + row0];
            S[s] = f4_fma(PREP ? __fmul_rn(kk, kn) : kk, u, S[s]);
        }

        if (WRITE_O && warp == 0 && rsub == 0) {
            float4 z = red_z[r][0][cg];
            float qk = red_qk[r][0];
#pragma unroll
            for (int w = 1; w < kSeqWarps; ++w) {
                z = f4_add(z, red_z[r][w][cg]);
                qk = __fadd_rn(qk, red_qk[r][w]);
            }
            const float4 o = f4_fma(qk, u, z);
            st_out4(static_cast<Tin *>(p.o) + (t * H + h) * DV + col0 + 4 * cg, o);
        }
    }

    if constexpr (PREP) {  // the advanced convolution state (q, k once per head; v per column block)
        if (cst) {
#pragma unroll
            for (int j = 0; j < kConvW - 1; ++j) {
                float *row = cst + (static_cast<int64_t>(j) * H + h) * Ct;
                if (tid < DK && cb == 0) {
                    row[tid] = hq[j];
                    row[DK + tid] = hk[j];
                }
                if (tid < CB) row[2 * DK + col0 + tid] = hv[j];
            }
        }
    }
    if (dst) {
#pragma unroll
        for (int s = 0; s < NS; ++s) {
            const int row = s * RPS + row0;
            *reinterpret_cast<float4 *>(dst + row * DV + col0 + 4 * cg) = S[s];
        }
    }
}

template <int DK, int DV, typename Tin>
cudaError_t launch_typed(const SeqParams &p, cudaStream_t stream) {
    const int64_t blocks = static_cast<int64_t>(p.N) * p.H * (DV / kColBlock);
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const dim3 grid(static_cast<unsigned>(blocks));
    if (p.o) {
        if (p.prep || p.ckpt || p.conv_w)
            kda_seq_kernel<DK, DV, Tin, true, true><<<grid, kSeqThreads, 0, stream>>>(p);
        else
            kda_seq_kernel<DK, DV, Tin, true, false><<<grid, kSeqThreads, 0, stream>>>(p);
    } else {
        if (p.prep || p.ckpt || p.conv_w)
            kda_seq_kernel<DK, DV, Tin, false, true><<<grid, kSeqThreads, 0, stream>>>(p);
        else
            kda_seq_kernel<DK, DV, Tin, false, false><<<grid, kSeqThreads, 0, stream>>>(p);
    }
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_dims(const SeqParams &p, int dk, int dv, cudaStream_t stream) {
    if (dk == 128 && dv == 128) return launch_typed<128, 128, Tin>(p, stream);
    if (dk == 64 && dv == 64) return launch_typed<64, 64, Tin>(p, stream);
    if (dk == 128 && dv == 64) return launch_typed<128, 64, Tin>(p, stream);
    if (dk == 64 && dv == 128) return launch_typed<64, 128, Tin>(p, stream);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_seq(const SeqParams &p, int dk, int dv, int dtype, cudaStream_t stream) {
    if (dtype == 0) return launch_dims<__nv_bfloat16>(p, dk, dv, stream);
    return launch_dims<float>(p, dk, dv, stream);
}

}  // namespace kda
