// Backward of the KDA prefill: gradients of a loss with respect to q, k, v, the
// log-gates g, beta and the initial states, given its gradients with respect to
// the outputs o and the final states.  The KDA paragraph of "Kimi K3 on
// Fireworks: Fast RL at frontier scale" quotes a backward kernel (its speedup
// over FLA) but no formula; this is the reverse mode of the chunked (WY) form of
// the forward.
//
// Per (sequence, head) and 64-token chunk with start state S (from the forward
// pass's checkpoints), in-chunk prefix products A_r of alpha = exp(g) and
// A_C = A_64, Kbar = K*A, Ktil = K/A, Khat = Ktil*A_C, Qbar = scale Q*A:
//
//   M = Diag(beta) strictly-lower(Kbar Ktil^T),  T = (I + M)^-1,  T' = T Diag(beta)
//   R = V - Kbar S,  U = T' R,  P = lower(Qbar Ktil^T)
//   O = Qbar S + P U,   S_next = Diag(A_C) S + Khat^T U
//
// and, given dO and dS_next (the gradient of the chunk's end state):
//
//   dU = Khat dS_next + P^T dO            dP = lower(dO U^T)
//   dR = T'^T dU  (= dV)                  dT' = dU R^T
//   dQbar = dO S^T + dP Ktil              dKhat = U dS_next^T
//   dKbar = -dR S^T + dMr Ktil            dKtil = dP^T Qbar + dMr^T Kbar
//   dT = dT' Diag(beta),  dM = strictly-lower(-T^T dT T^T),  dMr = Diag(beta) dM
//   dbeta_j = sum_i dT'_ij T_ij + sum_{k<j} dM_jk (Kbar Ktil^T)_jk
//   dS = Diag(A_C) dS_next + Qbar^T dO - Kbar^T dR        (the next chunk back's dS_next)
//   dK = dKbar*A + dKtil/A + dKhat*A_C/A,  dQ = scale dQbar*A
//   dlogA_r = dKbar*Kbar - dKtil*Ktil + dQbar*Qbar - dKhat*Khat
//   dlogA_C = sum_j dS_next*A_C*S + sum_r dKhat*Khat,   dg_s = sum_{r >= s} dlogA_r + dlogA_C
//
// A partial last chunk is padded with zero tokens (k = q = v = g = beta = dO = 0),
// which change neither the state nor any gradient.
//
// Only dS runs through the chunks in sequence, and it needs only
// dR = G dS_next + F with G = T'^T Khat and F = T'^T P^T dO, and
// dS = Diag(A_C) dS_next + E - Kbar^T dR with E = Qbar^T dO.  So the backward is
// three launches, like the forward's split into chunk-local work and a chain:
//   (A) every (chunk, head), in parallel: T, Kbar, G, F, E, A_C into its record;
//   (B) every (sequence, head): the chain of dS, two small products per chunk,
//       leaving dS_next and dR in the records;
//   (C) every (chunk, head), in parallel: all the gradients of the chunk.
// A and C run on two persistent CTAs per SM, each with its own scratch.  Every
// product runs on the tcgen05 tensor cores (kda_tc_gemm.cuh: tf32 operands staged
// from the global scratch and records into swizzled shared-memory tiles, fp32
// accumulation in TMEM), in the order and with the masks the equations above give.
// The work between products is a string of round trips through L2 and DRAM, so every
// CTA-wide loop issues all of its loads before its first store, and the chain
// prefetches the next chunk's records into L2 while it works on the current one.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_internal.h"
#include "kda_tc_gemm.cuh"

namespace kda {
namespace {

constexpr int kBT = 256;  // threads per CTA
constexpr int kC = 64;    // chunk length
constexpr int kPad = kC + 1;
constexpr float kMinDecay = 7.888609052210118e-31f;  // 2^-100, the forward's gate range

__device__ __forceinline__ float ld_in(const float *p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ld_in(const __nv_bfloat16 *p, int64_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void st_out(float *p, int64_t i, float x) { p[i] = x; }
__device__ __forceinline__ void st_out(__nv_bfloat16 *p, int64_t i, float x) { p[i] = __float2bfloat16_rn(x); }

// Eight consecutive inputs p[i .. i + 7] as floats: one or two 16-byte loads when `vec` (the
// address is 16-byte aligned), else element by element.
__device__ __forceinline__ void ld8(const __nv_bfloat16 *p, int64_t i, bool vec, float *x) {
    if (vec) {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p + i));
        const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const float2 f = __bfloat1622float2(b[t]);
            x[2 * t] = f.x;
            x[2 * t + 1] = f.y;
        }
    } else {
#pragma unroll
        for (int t = 0; t < 8; ++t) x[t] = __bfloat162float(p[i + t]);
    }
}
__device__ __forceinline__ void ld8(const float *p, int64_t i, bool vec, float *x) {
    if (vec) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(p + i)), b = __ldg(reinterpret_cast<const float4 *>(p + i + 4));
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    } else {
#pragma unroll
        for (int t = 0; t < 8; ++t) x[t] = p[i + t];
    }
}
__device__ __forceinline__ void st4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ float4 ld4(const float *p) { return __ldcg(reinterpret_cast<const float4 *>(p)); }

// dst[r * ldd + j] = src[r * lds + j] for r < R, j < NC (global memory, 16-byte aligned rows,
// NC a multiple of 4); all loads are issued before the first store.
template <int R, int NC>
__device__ __forceinline__ void cta_copy(float *dst, int ldd, const float *src, int lds) {
    constexpr int kVec = R * NC / 4, kIt = (kVec + kBT - 1) / kBT;
    float4 v[kIt];
#pragma unroll
    for (int it = 0; it < kIt; ++it) {
        const int e = threadIdx.x + it * kBT;
        if (kVec % kBT == 0 || e < kVec)
            v[it] = __ldcg(reinterpret_cast<const float4 *>(src + (e / (NC / 4)) * lds + (e % (NC / 4)) * 4));
    }
#pragma unroll
    for (int it = 0; it < kIt; ++it) {
        const int e = threadIdx.x + it * kBT;
        if (kVec % kBT == 0 || e < kVec) *reinterpret_cast<float4 *>(dst + (e / (NC / 4)) * ldd + (e % (NC / 4)) * 4) = v[it];
    }
}

// dst[r * NC + j] = f(r, j, src[r * NC + j]) over an R x NC tile in global memory (dst may be
// src: every element is read and written by the same thread); loads first, then stores.
template <int R, int NC, typename F>
__device__ __forceinline__ void cta_map(float *dst, const float *src, F f) {
    constexpr int kVec = R * NC / 4, kIt = kVec / kBT;
    static_assert(kVec % kBT == 0, "tile");
    float4 v[kIt];
#pragma unroll
    for (int it = 0; it < kIt; ++it) v[it] = ld4(src + (threadIdx.x + it * kBT) * 4);
#pragma unroll
    for (int it = 0; it < kIt; ++it) {
        const int e = (threadIdx.x + it * kBT) * 4, r = e / NC, j = e % NC;
        st4(dst + e, make_float4(f(r, j, v[it].x), f(r, j + 1, v[it].y), f(r, j + 2, v[it].z), f(r, j + 3, v[it].w)));
    }
}

// The CTA's tensor-core product context: the operand tiles in dynamic shared memory (aligned to
// 1024 bytes), 128 TMEM columns for the accumulator (allocated by warp 0) and one mbarrier.
__device__ tcg::Ctx tc_setup(uint8_t *dyn, uint64_t *bar, uint32_t *s_tmem, uint32_t *status) {
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dyn) + 1023) & ~uintptr_t(1023));
    if (threadIdx.x < 32) {
        ptx::tmem_alloc(s_tmem, 128);
        ptx::tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        ptx::mbar_init(bar, 1);
        ptx::fence_mbar_init();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    return tcg::Ctx{base, base + tcg::kTileA, bar, *s_tmem, 0u, status, DEV_ERR_TIMEOUT};
}
__device__ void tc_teardown(const tcg::Ctx &cx) {
    ptx::tc_fence_before();
    __syncthreads();
    if (threadIdx.x < 32) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(cx.tmem, 128);
    }
}

// Record of one (chunk slot, head), in floats.  Phase A writes F into the dR slot and E into
// its own slot; the chain accumulates dR = F + G dS_next and E - Kbar^T dR onto them in place
// and writes dS_next.
template <int DK, int DV>
struct Rec {
    static constexpr int64_t kT = 0, kKb = kT + kC * kC, kG = kKb + kC * DK, kdR = kG + kC * DK,
                             kE = kdR + kC * DV, kdSn = kE + DK * DV, kAC = kdSn + DK * DV, kTotal = kAC + DK;
};
// Scratch of one persistent CTA, in floats.
template <int DK, int DV>
struct Scr {
    // Kbar and Qbar are adjacent (one 128-row operand for [M; P]), as are M and P; V is loaded
    // into R's slot, where R = V - Kbar S accumulates
    static constexpr int64_t kA = 0, kKb = kA + kC * DK, kQb = kKb + kC * DK, kKt = kQb + kC * DK,
                             kKh = kKt + kC * DK, kdQb = kKh + kC * DK, kdKb = kdQb + kC * DK,
                             kdKt = kdKb + kC * DK, kdKh = kdKt + kC * DK, kR = kdKh + kC * DK, kdO = kR + kC * DV,
                             kV = kR, kU = kdO + kC * DV, kdU = kU + kC * DV, kY = kdU + kC * DV,
                             kMr = kY + kC * DV, kP = kMr + kC * kC, kTp = kP + kC * kC,
                             kdP = kTp + kC * kC, kdTp = kdP + kC * kC, kX = kdTp + kC * kC, kdM = kX + kC * kC,
                             kTotal = kdM + kC * kC;
};

// Shared memory of the A and C kernels besides the tensor-core tiles: the gate tile, or the two
// 64 x 64 matrices of the inverse, or the gate-gradient tile (never live at once).
template <int DK>
struct SmemBuf {
    static constexpr int kFloats = kC * DK > 2 * kC * kPad ? kC * DK : 2 * kC * kPad;
};

// Token range of sequence n; false (and the status bit) for an invalid partition.
__device__ __forceinline__ bool seq_range(const BwdParams &p, int n, int64_t &bos, int64_t &eos) {
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

// The sequence and chunk of checkpoint slot `slot`: the largest n whose first slot
// ckpt_base(bos_n, n) is <= slot (first slots increase with n).  False for a slot no
// chunk uses, or an invalid partition (reported by the chain kernel).
__device__ bool slot_chunk(const BwdParams &p, int64_t slot, int &n, int &c, int64_t &bos, int64_t &eos) {
    int lo = 0, hi = p.N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        const int64_t b = p.cu ? static_cast<int64_t>(p.cu[mid]) : static_cast<int64_t>(mid) * p.seq_len_fixed;
        if (ckpt_base(b, mid) <= slot) lo = mid;
        else hi = mid - 1;
    }
    n = lo;
    if (!seq_range(p, n, bos, eos)) return false;
    const int64_t cc = slot - ckpt_base(bos, n);
    const int64_t nch = (eos - bos + kC - 1) / kC;
    if (cc < 0 || cc >= nch) return false;
    c = static_cast<int>(cc);
    return true;
}

// Prefetches the rows [0, rows) x [0, row_bytes) of a matrix with row stride `ld_bytes` into
// L2, one 128-byte line per thread and round.
__device__ __forceinline__ void prefetch_rows(const void *base, int rows, int row_bytes, int64_t ld_bytes) {
    const int lines = row_bytes / 128;
    for (int e = threadIdx.x; e < rows * lines; e += kBT) {
        const char *a = static_cast<const char *>(base) + (e / lines) * ld_bytes + (e % lines) * 128;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
    }
}

// Prefetches into L2 what (chunk, head) item `item` will read: its rows of q, k, g, v and dO,
// and with `records` also its chunk-start state (a checkpoint, or the initial state) and the
// parts of its record the gradient phase reads (T, dR, dS_next).  Items past the end, or of
// an invalid partition, prefetch nothing.
template <int DK, int DV, typename Tin>
__device__ void prefetch_item(const BwdParams &p, int64_t item, bool records) {
    if (item >= p.nslots * p.H) return;
    const int64_t slot = item / p.H;
    const int h = static_cast<int>(item % p.H);
    int n, c;
    int64_t bos, eos;
    if (!slot_chunk(p, slot, n, c, bos, eos)) return;
    const int64_t t0 = bos + static_cast<int64_t>(c) * kC;
    const int Lc = static_cast<int>(eos - t0 < kC ? eos - t0 : kC);
    const int64_t H = p.H, es = sizeof(Tin);
    const char *q = static_cast<const char *>(p.q), *k = static_cast<const char *>(p.k);
    const char *g = static_cast<const char *>(p.g), *v = static_cast<const char *>(p.v);
    const char *d_o = static_cast<const char *>(p.d_o);
    const int64_t rk = (t0 * H + h) * DK * es, rv = (t0 * H + h) * DV * es;
    prefetch_rows(q + rk, Lc, DK * es, H * DK * es);
    prefetch_rows(k + rk, Lc, DK * es, H * DK * es);
    prefetch_rows(g + rk, Lc, DK * es, H * DK * es);
    prefetch_rows(v + rv, Lc, DV * es, H * DV * es);
    prefetch_rows(d_o + rv, Lc, DV * es, H * DV * es);  // (dO may be unaligned: a row's last line can be missed)
    if (!records) return;
    using RC = Rec<DK, DV>;
    const float *rec = p.rec + item * RC::kTotal;
    prefetch_rows(rec + RC::kT, 1, kC * kC * 4, 0);
    prefetch_rows(rec + RC::kdR, 1, kC * DV * 4, 0);
    prefetch_rows(rec + RC::kdSn, 1, DK * DV * 4, 0);
    const float *Sc = c > 0 ? p.ckpt + (slot * H + h) * DK * DV
                            : (p.init_state ? p.init_state + (static_cast<int64_t>(n) * H + h) * DK * DV : nullptr);
    if (Sc) prefetch_rows(Sc, 1, DK * DV * 4, 0);
}

// Chunk inputs of (t0, Lc, h) into the CTA scratch: A, Kbar, Ktil, Khat, Qbar (C x DK),
// V (optional) and dO (C x DV), beta and A_C into shared memory.  With preprocessing
// (p.prep) the raw inputs are mapped as the forward maps them: alpha = sigmoid(x_g),
// beta = sigmoid(x_beta), k and q rows scaled by their inverse L2 norms (s_rk, s_rq; 1
// when the flag is off).
template <int DK, int DV, typename Tin>
__device__ void load_chunk(const BwdParams &p, int64_t t0, int Lc, int h, float *W, bool want_v, float *s_buf,
                           float *s_beta, float *s_ac, float *s_rk, float *s_rq) {
    using S = Scr<DK, DV>;
    const int tid = threadIdx.x;
    const int64_t H = p.H;
    const Tin *G = static_cast<const Tin *>(p.g), *K = static_cast<const Tin *>(p.k);
    const Tin *Q = static_cast<const Tin *>(p.q), *V = static_cast<const Tin *>(p.v);
    const Tin *B = static_cast<const Tin *>(p.beta), *DO = static_cast<const Tin *>(p.d_o);
    // gate tile into shared memory, eight channels per load (q, k, v, g are 16-byte aligned and
    // every row starts at a multiple of eight elements)
    {
        constexpr int kG = kC * DK / 8, kIt = kG / kBT;
        static_assert(kG % kBT == 0, "gate tile");
        float x[kIt][8];
#pragma unroll
        for (int it = 0; it < kIt; ++it) {
            const int e = tid + it * kBT, r = e / (DK / 8), i = (e % (DK / 8)) * 8;
            if (r < Lc) ld8(G, ((t0 + r) * H + h) * DK + i, true, x[it]);
            else
#pragma unroll
                for (int t = 0; t < 8; ++t) x[it][t] = 0.f;
        }
#pragma unroll
        for (int it = 0; it < kIt; ++it) {
            const int e = tid + it * kBT, r = e / (DK / 8), i = (e % (DK / 8)) * 8;
            *reinterpret_cast<float4 *>(s_buf + r * DK + i) = make_float4(x[it][0], x[it][1], x[it][2], x[it][3]);
            *reinterpret_cast<float4 *>(s_buf + r * DK + i + 4) = make_float4(x[it][4], x[it][5], x[it][6], x[it][7]);
        }
    }
    if (tid < kC) {
        float b = tid < Lc ? ld_in(B, (t0 + tid) * H + h) : 0.f;
        if ((p.prep & PREP_SIGMOID_BETA) && tid < Lc) b = 1.f / (1.f + expf(-b));
        s_beta[tid] = b;
    }
    if (tid >= 128 && tid < 128 + 2 * kC) {  // inverse row norms of k (rows 0-63) and q (rows 64-127)
        const int r = (tid - 128) % kC;
        const bool is_q = tid - 128 >= kC;
        const int flag = is_q ? PREP_L2NORM_Q : PREP_L2NORM_K;
        float inv = 1.f;
        if ((p.prep & flag) && r < Lc) {
            const Tin *X = is_q ? static_cast<const Tin *>(p.q) : static_cast<const Tin *>(p.k);
            float ss = 0.f;
#pragma unroll 8
            for (int i = 0; i < DK; ++i) {
                const float x = ld_in(X, ((t0 + r) * H + h) * DK + i);
                ss = fmaf(x, x, ss);
            }
            inv = rsqrtf(ss + p.prep_eps);
        }
        (is_q ? s_rq : s_rk)[r] = inv;
    }
    __syncthreads();
    // in-chunk prefix products A_r of alpha, in place of the gate tile (and into the scratch)
    if (tid < DK) {
        const bool sig = (p.prep & PREP_SIGMOID_GATE) != 0;
        float a = 1.f;
        for (int r = 0; r < kC; ++r) {
            const float x = s_buf[r * DK + tid];
            if (r < Lc) a *= sig ? 1.f / (1.f + expf(-x)) : expf(x);  // padding rows: alpha = 1
            s_buf[r * DK + tid] = a;
            W[S::kA + r * DK + tid] = a;
        }
        s_ac[tid] = a;
    }
    __syncthreads();
    const float sc = p.scale;
    {
        constexpr int kG = kC * DK / 8, kIt = kG / kBT;
        float kx[kIt][8], qx[kIt][8];
#pragma unroll
        for (int it = 0; it < kIt; ++it) {
            const int e = tid + it * kBT, r = e / (DK / 8), i = (e % (DK / 8)) * 8;
            if (r < Lc) {
                ld8(K, ((t0 + r) * H + h) * DK + i, true, kx[it]);
                ld8(Q, ((t0 + r) * H + h) * DK + i, true, qx[it]);
            } else {
#pragma unroll
                for (int t = 0; t < 8; ++t) kx[it][t] = qx[it][t] = 0.f;
            }
        }
#pragma unroll
        for (int it = 0; it < kIt; ++it) {
            const int e = tid + it * kBT, r = e / (DK / 8), i = (e % (DK / 8)) * 8;
            const float rk = s_rk[r], rq = s_rq[r];
            float kb[8], kt[8], kh[8], qb[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const float a = s_buf[r * DK + i + t], kk = kx[it][t] * rk, qq = qx[it][t] * rq;
                kb[t] = kk * a;
                kt[t] = kk / a;
                kh[t] = (kk / a) * s_ac[i + t];
                qb[t] = sc * qq * a;
            }
            const int o = r * DK + i;
            st4(W + S::kKb + o, make_float4(kb[0], kb[1], kb[2], kb[3]));
            st4(W + S::kKb + o + 4, make_float4(kb[4], kb[5], kb[6], kb[7]));
            st4(W + S::kKt + o, make_float4(kt[0], kt[1], kt[2], kt[3]));
            st4(W + S::kKt + o + 4, make_float4(kt[4], kt[5], kt[6], kt[7]));
            st4(W + S::kKh + o, make_float4(kh[0], kh[1], kh[2], kh[3]));
            st4(W + S::kKh + o + 4, make_float4(kh[4], kh[5], kh[6], kh[7]));
            st4(W + S::kQb + o, make_float4(qb[0], qb[1], qb[2], qb[3]));
            st4(W + S::kQb + o + 4, make_float4(qb[4], qb[5], qb[6], qb[7]));
        }
    }
    {
        constexpr int kG = kC * DV / 8, kIt = kG / kBT;
        static_assert(kG % kBT == 0, "value tile");
        const bool vec_do = (reinterpret_cast<uintptr_t>(DO) & 15u) == 0;
        float vx[kIt][8], dx[kIt][8];
#pragma unroll
        for (int it = 0; it < kIt; ++it) {
            const int e = tid + it * kBT, r = e / (DV / 8), j = (e % (DV / 8)) * 8;
            if (r < Lc) {
                if (want_v) ld8(V, ((t0 + r) * H + h) * DV + j, true, vx[it]);
                ld8(DO, ((t0 + r) * H + h) * DV + j, vec_do, dx[it]);
            } else {
#pragma unroll
                for (int t = 0; t < 8; ++t) vx[it][t] = dx[it][t] = 0.f;
            }
        }
#pragma unroll
        for (int it = 0; it < kIt; ++it) {
            const int e = tid + it * kBT, r = e / (DV / 8), j = (e % (DV / 8)) * 8;
            const int o = r * DV + j;
            if (want_v) {
                st4(W + S::kV + o, make_float4(vx[it][0], vx[it][1], vx[it][2], vx[it][3]));
                st4(W + S::kV + o + 4, make_float4(vx[it][4], vx[it][5], vx[it][6], vx[it][7]));
            }
            st4(W + S::kdO + o, make_float4(dx[it][0], dx[it][1], dx[it][2], dx[it][3]));
            st4(W + S::kdO + o + 4, make_float4(dx[it][4], dx[it][5], dx[it][6], dx[it][7]));
        }
    }
    __syncthreads();
}

// T = (I + M)^-1 for M = Diag(beta) strictly-lower(Mr) (64 x 64, unit lower triangular), by
// blocks: the four 16 x 16 diagonal blocks by forward substitution down each column (four
// threads per column split each sum; a column never leaves its warp), then twice the block
// rule for a lower-triangular inverse, [[A, 0], [C, D]]^-1 = [[A^-1, 0], [-D^-1 C A^-1, D^-1]],
// from 16 to 32 and from 32 to 64 rows.  Writes T (row stride 64) to `Tout` and T Diag(beta)
// to `Tp_out` (if not null).
__device__ void tri_inverse(const float *Mr, const float *s_beta, float *s_buf, float *Tout, float *Tp_out) {
    const int tid = threadIdx.x;
    float *sM = s_buf, *sT = s_buf + kC * kPad;
    static_assert(kBT == 256 && kC == 64, "block layout");
    {
        constexpr int kIt = kC * kC / 4 / kBT;
        float4 v[kIt];
#pragma unroll
        for (int it = 0; it < kIt; ++it) v[it] = ld4(Mr + (tid + it * kBT) * 4);
#pragma unroll
        for (int it = 0; it < kIt; ++it) {
            const int e = (tid + it * kBT) * 4, i = e / kC, j = e % kC;
            const float b = s_beta[i];
            const float m[4] = {v[it].x, v[it].y, v[it].z, v[it].w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                sM[i * kPad + j + t] = i > j + t ? b * m[t] : 0.f;
                sT[i * kPad + j + t] = i == j + t ? 1.f : 0.f;
            }
        }
    }
    __syncthreads();
    {  // diagonal blocks: block b = tid / 64 (two warps), column jl = (tid / 4) % 16, part = tid % 4
        const int b = tid >> 6, jl = (tid >> 2) & 15, part = tid & 3, j = b * 16 + jl;
        for (int il = 1; il < 16; ++il) {
            const int i = b * 16 + il;
            float acc = 0.f;
            if (il > jl)
                for (int k = j + part; k < i; k += 4) acc = fmaf(sM[i * kPad + k], sT[k * kPad + j], acc);
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            if (part == 0 && il > jl) sT[i * kPad + j] = -acc;
            __syncwarp();
        }
    }
    __syncthreads();
    {  // 16 -> 32: in each 32-row block (o = 0, 32), C = M[o+16.., o..], A^-1 = T[o.., o..], D^-1 = T[o+16.., o+16..]
        const int o = (tid >> 7) * 32, t = tid & 127, r = t >> 3, c = (t & 7) * 2;
        float y0 = 0.f, y1 = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const float m = sM[(o + 16 + r) * kPad + o + k];
            y0 = fmaf(m, sT[(o + k) * kPad + o + c], y0);
            y1 = fmaf(m, sT[(o + k) * kPad + o + c + 1], y1);
        }
        sT[(o + 16 + r) * kPad + o + c] = y0;  // C A^-1, in place of the (zero) lower-left block
        sT[(o + 16 + r) * kPad + o + c + 1] = y1;
        __syncthreads();
        float z0 = 0.f, z1 = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const float d = sT[(o + 16 + r) * kPad + o + 16 + k];
            z0 = fmaf(d, sT[(o + 16 + k) * kPad + o + c], z0);
            z1 = fmaf(d, sT[(o + 16 + k) * kPad + o + c + 1], z1);
        }
        __syncthreads();
        sT[(o + 16 + r) * kPad + o + c] = -z0;
        sT[(o + 16 + r) * kPad + o + c + 1] = -z1;
    }
    __syncthreads();
    {  // 32 -> 64: C = M[32.., ..32], A^-1 = T[..32, ..32], D^-1 = T[32.., 32..]; four columns per thread
        const int r = tid >> 3, c = (tid & 7) * 4;
        float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
        for (int k = 0; k < 32; ++k) {
            const float m = sM[(32 + r) * kPad + k];
#pragma unroll
            for (int t = 0; t < 4; ++t) y[t] = fmaf(m, sT[k * kPad + c + t], y[t]);
        }
#pragma unroll
        for (int t = 0; t < 4; ++t) sT[(32 + r) * kPad + c + t] = y[t];
        __syncthreads();
        float z[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
        for (int k = 0; k < 32; ++k) {
            const float d = sT[(32 + r) * kPad + 32 + k];
#pragma unroll
            for (int t = 0; t < 4; ++t) z[t] = fmaf(d, sT[(32 + k) * kPad + c + t], z[t]);
        }
        __syncthreads();
#pragma unroll
        for (int t = 0; t < 4; ++t) sT[(32 + r) * kPad + c + t] = -z[t];
    }
    __syncthreads();
    for (int e = tid; e < kC * kC; e += kBT) {
        const float t = sT[(e / kC) * kPad + e % kC];
        Tout[e] = t;
        if (Tp_out) Tp_out[e] = t * s_beta[e % kC];
    }
    __syncthreads();
}

// ---------------------------------------------------------------------------- phase A
template <int DK, int DV, typename Tin>
__global__ void __launch_bounds__(kBT, 2) kda_bwd_chunk_kernel(BwdParams p) {
    using S = Scr<DK, DV>;
    using RC = Rec<DK, DV>;
    __shared__ __align__(16) float s_buf[SmemBuf<DK>::kFloats];
    __shared__ float s_beta[kC], s_ac[DK], s_rk[kC], s_rq[kC];
    extern __shared__ uint8_t bwd_dyn[];
    __shared__ uint64_t s_bar;
    __shared__ uint32_t s_tmem;
    tcg::Ctx cx = tc_setup(bwd_dyn, &s_bar, &s_tmem, p.status);
    float *W = p.scratch + static_cast<int64_t>(blockIdx.x) * S::kTotal;
    const int64_t items = p.nslots * p.H;
    for (int64_t item = blockIdx.x; item < items; item += gridDim.x) {
        const int64_t slot = item / p.H;
        const int h = static_cast<int>(item % p.H);
        int n, c;
        int64_t bos, eos;
        if (!slot_chunk(p, slot, n, c, bos, eos)) continue;  // uniform across the CTA
        const int64_t t0 = bos + static_cast<int64_t>(c) * kC;
        const int Lc = static_cast<int>(eos - t0 < kC ? eos - t0 : kC);
        float *rec = p.rec + item * RC::kTotal;
        load_chunk<DK, DV, Tin>(p, t0, Lc, h, W, false, s_buf, s_beta, s_ac, s_rk, s_rq);
        prefetch_item<DK, DV, Tin>(p, item + gridDim.x, false);
        if (threadIdx.x < DK) {
            rec[RC::kAC + threadIdx.x] = s_ac[threadIdx.x];
            if (!(s_ac[threadIdx.x] >= kMinDecay)) atomicOr(p.status, DEV_ERR_GATE);
        }
        cta_copy<kC, DK>(rec + RC::kKb, DK, W + S::kKb, DK);
        // [Mr; P] = [Kbar; Qbar] Ktil^T in one product, P's rows masked to the lower triangle
        tcg::gemm<2 * kC, kC, DK, false, true, kBT>(cx, W + S::kMr, kC, W + S::kKb, DK, W + S::kKt, DK, 1.f, false, 3);
        tri_inverse(W + S::kMr, s_beta, s_buf, rec + RC::kT, W + S::kTp);
        // G = T'^T Khat, F = T'^T (P^T dO), E = Qbar^T dO
        tcg::gemm<kC, DK, kC, true, false, kBT>(cx, rec + RC::kG, DK, W + S::kTp, kC, W + S::kKh, DK, 1.f, false, 0);
        tcg::gemm<kC, DV, kC, true, false, kBT>(cx, W + S::kY, DV, W + S::kP, kC, W + S::kdO, DV, 1.f, false, 0);
        tcg::gemm<kC, DV, kC, true, false, kBT>(cx, rec + RC::kdR, DV, W + S::kTp, kC, W + S::kY, DV, 1.f, false, 0);
        tcg::gemm<DK, DV, kC, true, false, kBT>(cx, rec + RC::kE, DV, W + S::kQb, DK, W + S::kdO, DV, 1.f, false, 0);
    }
    tc_teardown(cx);
}

// ---------------------------------------------------------------------------- phase B
// The columns of dS follow independent recurrences (dR and the update of column j read
// column j only), so each (sequence, head) chain is split into DV / kCB CTAs of kCB columns
// (32 when that still fits the resident CTAs, else 64).  While one chunk is processed the
// records of the next one back are prefetched into L2.


template <int DK, int DV>
__device__ __forceinline__ void prefetch_chain_record(const float *rec, int col0, int kCB) {
    using RC = Rec<DK, DV>;
    prefetch_rows(rec + RC::kG, 1, kC * DK * 4, 0);
    prefetch_rows(rec + RC::kKb, 1, kC * DK * 4, 0);
    prefetch_rows(rec + RC::kdR + col0, kC, kCB * 4, DV * 4);
    prefetch_rows(rec + RC::kE + col0, DK, kCB * 4, DV * 4);
    prefetch_rows(rec + RC::kAC, 1, DK * 4, 0);
}

template <int DK, int DV, int kCB>
__global__ void __launch_bounds__(kBT, 2) kda_bwd_chain_kernel(BwdParams p) {
    using S = Scr<DK, DV>;
    using RC = Rec<DK, DV>;
    constexpr int kBlocks = DV / kCB;
    const int tid = threadIdx.x;
    const int64_t pair = blockIdx.x / kBlocks;
    const int col0 = static_cast<int>(blockIdx.x % kBlocks) * kCB;
    const int n = static_cast<int>(pair / p.H), h = static_cast<int>(pair % p.H);
    int64_t bos, eos;
    if (!seq_range(p, n, bos, eos)) {
        if (tid == 0 && h == 0 && col0 == 0) atomicOr(p.status, DEV_ERR_SEQLENS);
        return;
    }
    extern __shared__ uint8_t bwd_dyn[];
    __shared__ uint64_t s_bar;
    __shared__ uint32_t s_tmem;
    tcg::Ctx cx = tc_setup(bwd_dyn, &s_bar, &s_tmem, p.status);
    // this CTA's columns of the chain's DK x DV state dS (row stride DV)
    float *dS = p.scratch + static_cast<int64_t>(p.ctas) * S::kTotal + pair * 2 * DK * DV + col0;
    const int nch = static_cast<int>((eos - bos + kC - 1) / kC);
    const int64_t base = ckpt_base(bos, n);
    auto rec_of = [&](int c) { return p.rec + ((base + c) * p.H + h) * RC::kTotal; };
    if (nch > 0) prefetch_chain_record<DK, DV>(rec_of(nch - 1), col0, kCB);
    for (int e = tid; e < DK * kCB; e += kBT) {
        const int i = e / kCB, j = e % kCB;
        const float x = p.d_final ? p.d_final[pair * DK * DV + i * DV + col0 + j] : 0.f;
        dS[i * DV + j] = x;
        if (nch > 0) rec_of(nch - 1)[RC::kdSn + i * DV + col0 + j] = x;  // dS_next of the last chunk
    }
    __syncthreads();
    for (int c = nch - 1; c >= 0; --c) {
        float *rec = rec_of(c);
        if (c > 0) prefetch_chain_record<DK, DV>(rec_of(c - 1), col0, kCB);
        // dR = F + G dS_next (onto F in the dR slot);  E' = E - Kbar^T dR (onto E);
        // dS = Diag(A_C) dS_next + E', which is also the dS_next of chunk c - 1
        tcg::gemm<kC, kCB, DK, false, false, kBT>(cx, rec + RC::kdR + col0, DV, rec + RC::kG, DK, dS, DV, 1.f, true, 0);
        tcg::gemm<DK, kCB, kC, true, false, kBT>(cx, rec + RC::kE + col0, DV, rec + RC::kKb, DK, rec + RC::kdR + col0,
                                                 DV, -1.f, true, 0);
        {
            constexpr int kVec = DK * kCB / 4, kIt = kVec / kBT;
            static_assert(kVec % kBT == 0, "chain block");
            float4 a[kIt], b[kIt];
            float ac[kIt];
#pragma unroll
            for (int it = 0; it < kIt; ++it) {
                const int e = tid + it * kBT, i = e / (kCB / 4), j = (e % (kCB / 4)) * 4;
                a[it] = __ldcg(reinterpret_cast<const float4 *>(dS + i * DV + j));
                b[it] = __ldcg(reinterpret_cast<const float4 *>(rec + RC::kE + col0 + i * DV + j));
                ac[it] = __ldcg(rec + RC::kAC + i);
            }
            float *prev = c > 0 ? rec_of(c - 1) + RC::kdSn + col0 : nullptr;
#pragma unroll
            for (int it = 0; it < kIt; ++it) {
                const int e = tid + it * kBT, i = e / (kCB / 4), j = (e % (kCB / 4)) * 4;
                const float4 r = make_float4(fmaf(ac[it], a[it].x, b[it].x), fmaf(ac[it], a[it].y, b[it].y),
                                             fmaf(ac[it], a[it].z, b[it].z), fmaf(ac[it], a[it].w, b[it].w));
                *reinterpret_cast<float4 *>(dS + i * DV + j) = r;
                if (prev) *reinterpret_cast<float4 *>(prev + i * DV + j) = r;
            }
        }
        __syncthreads();
    }
    if (p.d_init)
        for (int e = tid; e < DK * kCB; e += kBT) {
            const int i = e / kCB, j = e % kCB;
            p.d_init[pair * DK * DV + i * DV + col0 + j] = dS[i * DV + j];
        }
    tc_teardown(cx);
}

// ---------------------------------------------------------------------------- phase C
template <int DK, int DV, typename Tin>
__global__ void __launch_bounds__(kBT, 2) kda_bwd_grad_kernel(BwdParams p) {
    using S = Scr<DK, DV>;
    using RC = Rec<DK, DV>;
    __shared__ __align__(16) float s_buf[SmemBuf<DK>::kFloats];
    __shared__ float s_beta[kC], s_dbeta[kC], s_ac[DK], s_red[kBT], s_rk[kC], s_rq[kC], s_rowdot[DK];
    extern __shared__ uint8_t bwd_dyn[];
    __shared__ uint64_t s_bar;
    __shared__ uint32_t s_tmem;
    tcg::Ctx cx = tc_setup(bwd_dyn, &s_bar, &s_tmem, p.status);
    const int tid = threadIdx.x;
    float *W = p.scratch + static_cast<int64_t>(blockIdx.x) * S::kTotal;
    const int64_t H = p.H;
    Tin *DQ = static_cast<Tin *>(p.dq), *DK_ = static_cast<Tin *>(p.dk), *DV_ = static_cast<Tin *>(p.dv);
    Tin *DG = static_cast<Tin *>(p.dg), *DB = static_cast<Tin *>(p.dbeta);
    const float sc = p.scale;
    const int64_t items = p.nslots * p.H;
    for (int64_t item = blockIdx.x; item < items; item += gridDim.x) {
        const int64_t slot = item / p.H;
        const int h = static_cast<int>(item % p.H);
        int n, c;
        int64_t bos, eos;
        if (!slot_chunk(p, slot, n, c, bos, eos)) continue;
        const int64_t t0 = bos + static_cast<int64_t>(c) * kC;
        const int Lc = static_cast<int>(eos - t0 < kC ? eos - t0 : kC);
        const float *rec = p.rec + item * RC::kTotal;
        const int64_t pair = static_cast<int64_t>(n) * H + h;
        // the chunk's start state: the initial state for the first chunk, else a checkpoint
        const float *Sc = c > 0 ? p.ckpt + (slot * H + h) * DK * DV
                                : (p.init_state ? p.init_state + pair * DK * DV : nullptr);
        const float *dSx = rec + RC::kdSn, *dR = rec + RC::kdR, *T = rec + RC::kT;
        float *A_ = W + S::kA, *Kb = W + S::kKb, *Kt = W + S::kKt, *Kh = W + S::kKh, *Qb = W + S::kQb;
        float *dQb = W + S::kdQb, *dKb = W + S::kdKb, *dKt = W + S::kdKt, *dKh = W + S::kdKh;
        float *dOs = W + S::kdO, *R = W + S::kR, *U = W + S::kU, *dU = W + S::kdU;
        float *Mr = W + S::kMr, *P = W + S::kP, *Tp = W + S::kTp, *dP = W + S::kdP;
        float *dTp = W + S::kdTp, *X = W + S::kX, *dM = W + S::kdM;

        if (item == blockIdx.x) prefetch_item<DK, DV, Tin>(p, item, true);  // later items: one item ahead
        load_chunk<DK, DV, Tin>(p, t0, Lc, h, W, true, s_buf, s_beta, s_ac, s_rk, s_rq);
        tcg::gemm<2 * kC, kC, DK, false, true, kBT>(cx, Mr, kC, Kb, DK, Kt, DK, 1.f, false, 3);  // [Mr; P]
        cta_map<kC, kC>(Tp, T, [&](int, int j, float x) { return x * s_beta[j]; });
        __syncthreads();
        // forward quantities of the chunk: R = V - Kbar S, U = T' R
        if (Sc) tcg::gemm<kC, DV, DK, false, false, kBT>(cx, R, DV, Kb, DK, Sc, DV, -1.f, true, 0);
        tcg::gemm<kC, DV, kC, false, false, kBT>(cx, U, DV, Tp, kC, R, DV, 1.f, false, 0);
        // reverse
        tcg::gemm<kC, DV, DK, false, false, kBT>(cx, dU, DV, Kh, DK, dSx, DV, 1.f, false, 0);
        tcg::gemm<kC, DV, kC, true, false, kBT>(cx, dU, DV, P, kC, dOs, DV, 1.f, true, 0);
        tcg::gemm<kC, kC, DV, false, true, kBT>(cx, dP, kC, dOs, DV, U, DV, 1.f, false, 1);
        tcg::gemm<kC, kC, DV, false, true, kBT>(cx, dTp, kC, dU, DV, R, DV, 1.f, false, 0);
        tcg::gemm<kC, DK, kC, false, false, kBT>(cx, dQb, DK, dP, kC, Kt, DK, 1.f, false, 0);
        if (Sc) tcg::gemm<kC, DK, DV, false, true, kBT>(cx, dQb, DK, dOs, DV, Sc, DV, 1.f, true, 0);
        tcg::gemm<kC, DK, DV, false, true, kBT>(cx, dKh, DK, U, DV, dSx, DV, 1.f, false, 0);
        if (Sc)
            tcg::gemm<kC, DK, DV, false, true, kBT>(cx, dKb, DK, dR, DV, Sc, DV, -1.f, false, 0);
        else
            for (int e = tid; e < kC * DK; e += kBT) dKb[e] = 0.f;
        tcg::gemm<kC, DK, kC, true, false, kBT>(cx, dKt, DK, dP, kC, Qb, DK, 1.f, false, 0);
        // beta through T' = T Diag(beta) (column sums over 4 row quarters); dT = dT' Diag(beta)
        {
            const int j = tid & 63, qr = tid >> 6;
            float acc = 0.f;
            for (int i = qr * 16; i < qr * 16 + 16; ++i) acc = fmaf(dTp[i * kC + j], T[i * kC + j], acc);
            s_red[tid] = acc;
        }
        __syncthreads();
        if (tid < kC) s_dbeta[tid] = (s_red[tid] + s_red[tid + 64]) + (s_red[tid + 128] + s_red[tid + 192]);
        cta_map<kC, kC>(dTp, dTp, [&](int, int j, float x) { return x * s_beta[j]; });
        __syncthreads();
        // through the inverse: dM = strictly-lower(-T^T dT T^T)
        tcg::gemm<kC, kC, kC, true, false, kBT>(cx, X, kC, T, kC, dTp, kC, 1.f, false, 0);
        tcg::gemm<kC, kC, kC, false, true, kBT>(cx, dM, kC, X, kC, T, kC, -1.f, false, 2);
        // through M = Diag(beta) strictly-lower(Kbar Ktil^T): row sums, four threads per row
        {
            const int i = tid >> 2, part = tid & 3;
            float acc = 0.f;
            for (int j = part; j < i; j += 4) acc = fmaf(dM[i * kC + j], Mr[i * kC + j], acc);
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            if (part == 0) s_dbeta[i] += acc;
        }
        __syncthreads();
        cta_map<kC, kC>(dM, dM, [&](int i, int, float x) { return x * s_beta[i]; });
        __syncthreads();
        tcg::gemm<kC, DK, kC, false, false, kBT>(cx, dKb, DK, dM, kC, Kt, DK, 1.f, true, 0);
        tcg::gemm<kC, DK, kC, true, false, kBT>(cx, dKt, DK, dM, kC, Kb, DK, 1.f, true, 0);
        prefetch_item<DK, DV, Tin>(p, item + gridDim.x, true);
        // gate gradients: dlogA_C = A_C sum_j dS_next S + sum_r dKhat Khat.  The row sums of
        // dS_next * S take one warp per group of rows, lanes across the columns (four rows'
        // loads in flight); the column sums of dKhat * Khat one thread per column and part.
        {
            constexpr int kWarps = kBT / 32, kRows = DK / kWarps, kPer = DV / 32;
            static_assert(kRows % 4 == 0 && (kPer == 4 || kPer == 2), "row sums");
            const int warp = tid >> 5, lane = tid & 31;
#pragma unroll 1
            for (int r0 = 0; r0 < kRows; r0 += 4) {
                float part[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int row = warp * kRows + r0 + u;
                    part[u] = 0.f;
                    if (Sc) {
                        const float *x = dSx + row * DV + lane * kPer, *y = Sc + row * DV + lane * kPer;
                        if (kPer == 4) {
                            const float4 a = ld4(x), b = ld4(y);
                            part[u] = fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
                        } else {
                            const float2 a = __ldcg(reinterpret_cast<const float2 *>(x));
                            const float2 b = __ldcg(reinterpret_cast<const float2 *>(y));
                            part[u] = fmaf(a.x, b.x, a.y * b.y);
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) part[u] += __shfl_xor_sync(0xffffffffu, part[u], o);
                    if (lane == 0) s_rowdot[warp * kRows + r0 + u] = part[u] * s_ac[warp * kRows + r0 + u];
                }
            }
            constexpr int kGroups = kBT / DK;
            const int i = tid % DK, grp = tid / DK;
            float acc = 0.f;
            for (int r = grp; r < kC; r += kGroups) acc = fmaf(dKh[r * DK + i], Kh[r * DK + i], acc);
            s_red[tid] = acc;
        }
        __syncthreads();
        // per element: dK, dQ and dlogA_r (into shared memory for the reverse sums); four
        // elements per thread and round, two rounds' loads in flight
        const bool norms = (p.prep & (PREP_L2NORM_K | PREP_L2NORM_Q)) != 0;
        {
            constexpr int kVec = kC * DK / 4, kRounds = kVec / kBT, kB = 2;
            static_assert(kRounds % kB == 0, "rounds");
#pragma unroll 1
            for (int rb = 0; rb < kRounds; rb += kB) {
                float4 a[kB], kb[kB], kt[kB], kh[kB], qb[kB], dkb[kB], dkt[kB], dkh[kB], dqb[kB];
#pragma unroll
                for (int u = 0; u < kB; ++u) {
                    const int e = (tid + (rb + u) * kBT) * 4;
                    a[u] = ld4(A_ + e); kb[u] = ld4(Kb + e); kt[u] = ld4(Kt + e); kh[u] = ld4(Kh + e);
                    qb[u] = ld4(Qb + e); dkb[u] = ld4(dKb + e); dkt[u] = ld4(dKt + e); dkh[u] = ld4(dKh + e);
                    dqb[u] = ld4(dQb + e);
                }
#pragma unroll
                for (int u = 0; u < kB; ++u) {
                    const int e = (tid + (rb + u) * kBT) * 4, r = e / DK, i = e % DK;
                    const float *pa = &a[u].x, *pkb = &kb[u].x, *pkt = &kt[u].x, *pkh = &kh[u].x, *pqb = &qb[u].x;
                    const float *pdkb = &dkb[u].x, *pdkt = &dkt[u].x, *pdkh = &dkh[u].x, *pdqb = &dqb[u].x;
                    float gk[4], gq[4];
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const float ra = 1.f / pa[t];
                        gk[t] = pdkb[t] * pa[t] + pdkt[t] * ra + pdkh[t] * (s_ac[i + t] * ra);
                        gq[t] = sc * pdqb[t] * pa[t];
                        s_buf[e + t] = pdkb[t] * pkb[t] - pdkt[t] * pkt[t] + pdqb[t] * pqb[t] - pdkh[t] * pkh[t];
                    }
                    if (norms) {  // gradients of the normalised rows, carried back below
                        st4(dKb + e, make_float4(gk[0], gk[1], gk[2], gk[3]));
                        st4(dQb + e, make_float4(gq[0], gq[1], gq[2], gq[3]));
                    } else if (r < Lc) {
                        const int64_t o = ((t0 + r) * H + h) * DK + i;
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            st_out(DK_, o + t, gk[t]);
                            st_out(DQ, o + t, gq[t]);
                        }
                    }
                }
            }
        }
        {
            constexpr int kVec = kC * DV / 4, kIt = kVec / kBT;
            float4 d[kIt];
#pragma unroll
            for (int it = 0; it < kIt; ++it) d[it] = ld4(dR + (tid + it * kBT) * 4);
#pragma unroll
            for (int it = 0; it < kIt; ++it) {
                const int e = (tid + it * kBT) * 4, r = e / DV, j = e % DV;
                if (r < Lc) {
                    const int64_t o = ((t0 + r) * H + h) * DV + j;
                    st_out(DV_, o, d[it].x);
                    st_out(DV_, o + 1, d[it].y);
                    st_out(DV_, o + 2, d[it].z);
                    st_out(DV_, o + 3, d[it].w);
                }
            }
        }
        __syncthreads();
        if (tid < DK) {  // dg_s = dlogA_C + sum_{r >= s} dlogA_r (raw gate x: times 1 - sigmoid(x))
            const bool sig = (p.prep & PREP_SIGMOID_GATE) != 0;
            const Tin *G = static_cast<const Tin *>(p.g);
            float acc = s_rowdot[tid];
            for (int gi = 0; gi < kBT / DK; ++gi) acc += s_red[tid + gi * DK];
            for (int r = kC - 1; r >= 0; --r) {
                acc += s_buf[r * DK + tid];
                if (r < Lc) {
                    const int64_t o = ((t0 + r) * H + h) * DK + tid;
                    st_out(DG, o, sig ? acc * (1.f - 1.f / (1.f + expf(-ld_in(G, o)))) : acc);
                }
            }
        }
        if (tid < Lc) {
            const float b = s_beta[tid];
            st_out(DB, (t0 + tid) * H + h, (p.prep & PREP_SIGMOID_BETA) ? s_dbeta[tid] * b * (1.f - b) : s_dbeta[tid]);
        }
        if (norms && tid >= 128 && tid < 128 + 2 * kC) {
            // dx = r (dxn - xn (xn . dxn)) with xn = r x, per row of k (rows 0-63) or q (64-127)
            const int r = (tid - 128) % kC;
            const bool is_q = tid - 128 >= kC;
            if (r < Lc) {
                const Tin *X = is_q ? static_cast<const Tin *>(p.q) : static_cast<const Tin *>(p.k);
                const float *gx = (is_q ? dQb : dKb) + r * DK;
                const bool on = (p.prep & (is_q ? PREP_L2NORM_Q : PREP_L2NORM_K)) != 0;
                const float inv = is_q ? s_rq[r] : s_rk[r];
                const int64_t o = ((t0 + r) * H + h) * DK;
                float dot = 0.f;
                if (on) {
#pragma unroll 8
                    for (int i = 0; i < DK; ++i) dot = fmaf(ld_in(X, o + i) * inv, gx[i], dot);
                }
#pragma unroll 8
                for (int i = 0; i < DK; ++i) {
                    const float out = on ? inv * (gx[i] - ld_in(X, o + i) * inv * dot) : gx[i];
                    st_out(is_q ? DQ : DK_, o + i, out);
                }
            }
        }
        __syncthreads();
    }
    tc_teardown(cx);
}

template <int DK, int DV, typename Tin>
cudaError_t launch_typed(const BwdParams &p, cudaStream_t stream) {
    const int64_t chains = static_cast<int64_t>(p.N) * p.H;
    if (chains <= 0) return cudaSuccess;
    if (chains > 0x7fffffffLL || p.ctas <= 0) return cudaErrorInvalidConfiguration;
    // the tensor-core operand tiles are dynamic shared memory (a per-device function attribute,
    // set on every launch)
    const int dyn = static_cast<int>(tcg::kSmemBytes);
    // chain blocks of 32 columns while they fit the resident CTAs (two per SM), else 64
    const bool narrow = DV >= 64 && chains * (DV / 32) <= p.ctas;
    const void *chain_fn = narrow ? reinterpret_cast<const void *>(kda_bwd_chain_kernel<DK, DV, 32>)
                                  : reinterpret_cast<const void *>(kda_bwd_chain_kernel<DK, DV, 64>);
    for (const void *fn : {reinterpret_cast<const void *>(kda_bwd_chunk_kernel<DK, DV, Tin>), chain_fn,
                           reinterpret_cast<const void *>(kda_bwd_grad_kernel<DK, DV, Tin>)}) {
        const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
        if (e != cudaSuccess) return e;
    }
    kda_bwd_chunk_kernel<DK, DV, Tin><<<p.ctas, kBT, dyn, stream>>>(p);
    if (narrow)
        kda_bwd_chain_kernel<DK, DV, 32><<<static_cast<unsigned>(chains * (DV / 32)), kBT, dyn, stream>>>(p);
    else
        kda_bwd_chain_kernel<DK, DV, 64><<<static_cast<unsigned>(chains * (DV / 64)), kBT, dyn, stream>>>(p);
    kda_bwd_grad_kernel<DK, DV, Tin><<<p.ctas, kBT, dyn, stream>>>(p);
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_dims(const BwdParams &p, int dk, int dv, cudaStream_t stream) {
    if (dk == 128 && dv == 128) return launch_typed<128, 128, Tin>(p, stream);
    if (dk == 64 && dv == 64) return launch_typed<64, 64, Tin>(p, stream);
    if (dk == 128 && dv == 64) return launch_typed<128, 64, Tin>(p, stream);
    if (dk == 64 && dv == 128) return launch_typed<64, 128, Tin>(p, stream);
    return cudaErrorInvalidValue;
}

template <template <int, int> class L>
size_t dims_floats(int dk, int dv) {
    if (dk == 128 && dv == 128) return static_cast<size_t>(L<128, 128>::kTotal);
    if (dk == 64 && dv == 64) return static_cast<size_t>(L<64, 64>::kTotal);
    if (dk == 128 && dv == 64) return static_cast<size_t>(L<128, 64>::kTotal);
    if (dk == 64 && dv == 128) return static_cast<size_t>(L<64, 128>::kTotal);
    return 0;
}

}  // namespace

size_t bwd_scratch_floats(int dk, int dv) { return dims_floats<Scr>(dk, dv); }
size_t bwd_record_floats(int dk, int dv) { return dims_floats<Rec>(dk, dv); }

cudaError_t launch_bwd(const BwdParams &p, int dk, int dv, int dtype, cudaStream_t stream) {
    if (dtype == 0) return launch_dims<__nv_bfloat16>(p, dk, dv, stream);
    return launch_dims<float>(p, dk, dv, stream);
}

}  // namespace kda
