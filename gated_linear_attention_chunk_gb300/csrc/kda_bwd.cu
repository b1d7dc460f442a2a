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
// product is a CTA-wide fp32 matrix product over global (L2-resident) operands,
// staged through shared memory in 16-deep slices with the next slice fetched
// into registers while the current one is multiplied.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_internal.h"

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

// C (M x N, row stride ldc) = alpha op(A) op(B), or += when `acc`.  op(A) is M x K: A is
// stored M x K (row stride lda), or K x M when TA.  op(B) is K x N: B is stored K x N, or
// N x K when TB.  mask 1 keeps entries i >= j, mask 2 entries i > j (the others become 0,
// or stay unchanged when accumulating).  All threads of the CTA take part; ends with a
// barrier, so the result is visible to the whole CTA.
template <int M, int N, int K, bool TA, bool TB>
__device__ void cta_gemm(float *C, int ldc, const float *A, int lda, const float *B, int ldb, float alpha, bool acc,
                         int mask, float *sm) {
    static_assert(M % 16 == 0 && N % 16 == 0 && K % 16 == 0 && M <= 128 && N <= 128, "shape");
    static_assert((16 * M) % kBT == 0 && (16 * N) % kBT == 0, "slice split");
    constexpr int MB = M / 16, NB = N / 16, PA = M + 4, PB = N + 4, EA = 16 * M / kBT, EB = 16 * N / kBT;
    float *As = sm;            // [16][PA]: op(A) slice, k-major
    float *Bs = sm + 16 * PA;  // [16][PB]
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    float ra[EA], rb[EB];
    auto fetch = [&](int k0) {
#pragma unroll
        for (int u = 0; u < EA; ++u) {
            const int e = tid + u * kBT;
            ra[u] = TA ? A[(k0 + e / M) * lda + e % M] : A[(e >> 4) * lda + k0 + (e & 15)];
        }
#pragma unroll
        for (int u = 0; u < EB; ++u) {
            const int e = tid + u * kBT;
            rb[u] = TB ? B[(e >> 4) * ldb + k0 + (e & 15)] : B[(k0 + e / N) * ldb + e % N];
        }
    };
    auto stash = [&]() {
#pragma unroll
        for (int u = 0; u < EA; ++u) {
            const int e = tid + u * kBT;
            if (TA)
                As[(e / M) * PA + e % M] = ra[u];
            else
                As[(e & 15) * PA + (e >> 4)] = ra[u];
        }
#pragma unroll
        for (int u = 0; u < EB; ++u) {
            const int e = tid + u * kBT;
            if (TB)
                Bs[(e & 15) * PB + (e >> 4)] = rb[u];
            else
                Bs[(e / N) * PB + e % N] = rb[u];
        }
    };
    float c[MB][NB];
#pragma unroll
    for (int x = 0; x < MB; ++x)
#pragma unroll
        for (int y = 0; y < NB; ++y) c[x][y] = 0.f;
    fetch(0);
    for (int k0 = 0; k0 < K; k0 += 16) {
        stash();
        __syncthreads();
        if (k0 + 16 < K) fetch(k0 + 16);  // in flight while this slice is multiplied
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            float a[MB], b[NB];
#pragma unroll
            for (int x = 0; x < MB; ++x) a[x] = As[kk * PA + ty + 16 * x];
#pragma unroll
            for (int y = 0; y < NB; ++y) b[y] = Bs[kk * PB + tx + 16 * y];
#pragma unroll
            for (int x = 0; x < MB; ++x)
#pragma unroll
                for (int y = 0; y < NB; ++y) c[x][y] = fmaf(a[x], b[y], c[x][y]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int x = 0; x < MB; ++x)
#pragma unroll
        for (int y = 0; y < NB; ++y) {
            const int i = ty + 16 * x, j = tx + 16 * y;
            const bool keep = mask == 0 || (mask == 1 ? i >= j : i > j);
            float *o = C + i * ldc + j;
            if (acc) {
                if (keep) *o += alpha * c[x][y];
            } else {
                *o = keep ? alpha * c[x][y] : 0.f;
            }
        }
    __syncthreads();
}

__device__ __forceinline__ void cta_copy(float *dst, const float *src, int n) {
    for (int e = threadIdx.x; e < n; e += kBT) dst[e] = src[e];
}

// Record of one (chunk slot, head), in floats.
template <int DK, int DV>
struct Rec {
    static constexpr int64_t kT = 0, kKb = kT + kC * kC, kG = kKb + kC * DK, kF = kG + kC * DK, kdR = kF + kC * DV,
                             kE = kdR + kC * DV, kdSn = kE + DK * DV, kAC = kdSn + DK * DV, kTotal = kAC + DK;
};
// Scratch of one persistent CTA, in floats.
template <int DK, int DV>
struct Scr {
    static constexpr int64_t kA = 0, kKb = kA + kC * DK, kKt = kKb + kC * DK, kKh = kKt + kC * DK,
                             kQb = kKh + kC * DK, kdQb = kQb + kC * DK, kdKb = kdQb + kC * DK,
                             kdKt = kdKb + kC * DK, kdKh = kdKt + kC * DK, kV = kdKh + kC * DK, kdO = kV + kC * DV,
                             kR = kdO + kC * DV, kU = kR + kC * DV, kdU = kU + kC * DV, kY = kdU + kC * DV,
                             kMr = kY + kC * DV, kPr = kMr + kC * kC, kP = kPr + kC * kC, kTp = kP + kC * kC,
                             kdP = kTp + kC * kC, kdTp = kdP + kC * kC, kX = kdTp + kC * kC, kdM = kX + kC * kC,
                             kTotal = kdM + kC * kC;
};

// Shared memory of the A and C kernels: the matrix-product slices, or the gate tile /
// the two 64 x 64 matrices of the inverse / the gate-gradient tile (never live at once).
template <int DK>
struct SmemBuf {
    static constexpr int kGemm = 16 * (128 + 4 + 128 + 4);
    static constexpr int kTile = kC * DK > 2 * kC * kPad ? kC * DK : 2 * kC * kPad;
    static constexpr int kFloats = kGemm > kTile ? kGemm : kTile;
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
    for (int e = tid; e < kC * DK; e += kBT) {
        const int r = e / DK, i = e % DK;
        s_buf[e] = r < Lc ? ld_in(G, ((t0 + r) * H + h) * DK + i) : 0.f;
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
    if (tid < DK) {
        const bool sig = (p.prep & PREP_SIGMOID_GATE) != 0;
        float a = 1.f;
        for (int r = 0; r < kC; ++r) {
            const float x = s_buf[r * DK + tid];
            if (r < Lc) a *= sig ? 1.f / (1.f + expf(-x)) : expf(x);  // padding rows: alpha = 1
            W[S::kA + r * DK + tid] = a;
        }
        s_ac[tid] = a;
    }
    __syncthreads();
    const float sc = p.scale;
    for (int e = tid; e < kC * DK; e += kBT) {
        const int r = e / DK, i = e % DK;
        const bool ok = r < Lc;
        const float kk = ok ? ld_in(K, ((t0 + r) * H + h) * DK + i) * s_rk[r] : 0.f;
        const float qq = ok ? ld_in(Q, ((t0 + r) * H + h) * DK + i) * s_rq[r] : 0.f;
        const float a = W[S::kA + e];
        W[S::kKb + e] = kk * a;
        W[S::kKt + e] = kk / a;
        W[S::kKh + e] = (kk / a) * s_ac[i];
        W[S::kQb + e] = sc * qq * a;
    }
    for (int e = tid; e < kC * DV; e += kBT) {
        const int r = e / DV, j = e % DV;
        const bool ok = r < Lc;
        if (want_v) W[S::kV + e] = ok ? ld_in(V, ((t0 + r) * H + h) * DV + j) : 0.f;
        W[S::kdO + e] = ok ? ld_in(DO, ((t0 + r) * H + h) * DV + j) : 0.f;
    }
    __syncthreads();
}

// T = (I + M)^-1 for M = Diag(beta) strictly-lower(Mr) (64 x 64), by forward
// substitution down each column: T_ij = -sum_{j <= k < i} M_ik T_kj.  Four threads per
// column split each sum and combine it with two shuffles; a column never leaves its
// warp, so the warp's own barrier orders its rows.  Writes T (row stride 64) to `Tout`.
__device__ void tri_inverse(const float *Mr, const float *s_beta, float *s_buf, float *Tout) {
    const int tid = threadIdx.x;
    float *sM = s_buf, *sT = s_buf + kC * kPad;
    for (int e = tid; e < kC * kC; e += kBT) {
        const int i = e / kC, j = e % kC;
        sM[i * kPad + j] = i > j ? s_beta[i] * Mr[e] : 0.f;
    }
    const int j = tid >> 2, part = tid & 3;
    for (int i = part; i < kC; i += 4) sT[i * kPad + j] = (i == j) ? 1.f : 0.f;
    __syncthreads();
    for (int i = 1; i < kC; ++i) {
        float acc = 0.f;
        if (i > j)
            for (int k = j + part; k < i; k += 4) acc = fmaf(sM[i * kPad + k], sT[k * kPad + j], acc);
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        if (part == 0 && i > j) sT[i * kPad + j] = -acc;
        __syncwarp();
    }
    __syncthreads();
    for (int e = tid; e < kC * kC; e += kBT) Tout[e] = sT[(e / kC) * kPad + e % kC];
    __syncthreads();
}

// ---------------------------------------------------------------------------- phase A
template <int DK, int DV, typename Tin>
__global__ void __launch_bounds__(kBT, 2) kda_bwd_chunk_kernel(BwdParams p) {
    using S = Scr<DK, DV>;
    using RC = Rec<DK, DV>;
    __shared__ __align__(16) float s_buf[SmemBuf<DK>::kFloats];
    __shared__ float s_beta[kC], s_ac[DK], s_rk[kC], s_rq[kC];
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
        if (threadIdx.x < DK) {
            rec[RC::kAC + threadIdx.x] = s_ac[threadIdx.x];
            if (!(s_ac[threadIdx.x] >= kMinDecay)) atomicOr(p.status, DEV_ERR_GATE);
        }
        cta_copy(rec + RC::kKb, W + S::kKb, kC * DK);
        cta_gemm<kC, kC, DK, false, true>(W + S::kMr, kC, W + S::kKb, DK, W + S::kKt, DK, 1.f, false, 0, s_buf);
        cta_gemm<kC, kC, DK, false, true>(W + S::kPr, kC, W + S::kQb, DK, W + S::kKt, DK, 1.f, false, 0, s_buf);
        tri_inverse(W + S::kMr, s_beta, s_buf, rec + RC::kT);
        for (int e = threadIdx.x; e < kC * kC; e += kBT) {
            const int i = e / kC, j = e % kC;
            W[S::kTp + e] = rec[RC::kT + e] * s_beta[j];
            W[S::kP + e] = i >= j ? W[S::kPr + e] : 0.f;
        }
        __syncthreads();
        // G = T'^T Khat, F = T'^T (P^T dO), E = Qbar^T dO
        cta_gemm<kC, DK, kC, true, false>(rec + RC::kG, DK, W + S::kTp, kC, W + S::kKh, DK, 1.f, false, 0, s_buf);
        cta_gemm<kC, DV, kC, true, false>(W + S::kY, DV, W + S::kP, kC, W + S::kdO, DV, 1.f, false, 0, s_buf);
        cta_gemm<kC, DV, kC, true, false>(rec + RC::kF, DV, W + S::kTp, kC, W + S::kY, DV, 1.f, false, 0, s_buf);
        cta_gemm<DK, DV, kC, true, false>(rec + RC::kE, DV, W + S::kQb, DK, W + S::kdO, DV, 1.f, false, 0, s_buf);
    }
}

// ---------------------------------------------------------------------------- phase B
// The columns of dS follow independent recurrences (dR and the update of column j read
// column j only), so each (sequence, head) chain is split into DV / kChainCols CTAs.
constexpr int kChainCols = 32;

template <int DK, int DV>
__global__ void __launch_bounds__(kBT, 1) kda_bwd_chain_kernel(BwdParams p) {
    using S = Scr<DK, DV>;
    using RC = Rec<DK, DV>;
    constexpr int kCB = kChainCols, kBlocks = DV / kCB;
    __shared__ __align__(16) float s_buf[SmemBuf<DK>::kFloats];
    const int tid = threadIdx.x;
    const int64_t pair = blockIdx.x / kBlocks;
    const int col0 = static_cast<int>(blockIdx.x % kBlocks) * kCB;
    const int n = static_cast<int>(pair / p.H), h = static_cast<int>(pair % p.H);
    int64_t bos, eos;
    if (!seq_range(p, n, bos, eos)) {
        if (tid == 0 && h == 0 && col0 == 0) atomicOr(p.status, DEV_ERR_SEQLENS);
        return;
    }
    // this CTA's columns of the chain's two DK x DV states (row stride DV)
    float *dS = p.scratch + static_cast<int64_t>(p.ctas) * S::kTotal + pair * 2 * DK * DV + col0;
    float *dSn = dS + DK * DV;
    for (int e = tid; e < DK * kCB; e += kBT) {
        const int i = e / kCB, j = e % kCB;
        dS[i * DV + j] = p.d_final ? p.d_final[pair * DK * DV + i * DV + col0 + j] : 0.f;
    }
    __syncthreads();
    const int nch = static_cast<int>((eos - bos + kC - 1) / kC);
    const int64_t base = ckpt_base(bos, n);
    for (int c = nch - 1; c >= 0; --c) {
        float *rec = p.rec + ((base + c) * p.H + h) * RC::kTotal;
        for (int e = tid; e < DK * kCB; e += kBT) {
            const int i = e / kCB, j = e % kCB;
            rec[RC::kdSn + i * DV + col0 + j] = dS[i * DV + j];
            dSn[i * DV + j] = rec[RC::kE + i * DV + col0 + j];
        }
        for (int e = tid; e < kC * kCB; e += kBT) {
            const int r = e / kCB, j = e % kCB;
            rec[RC::kdR + r * DV + col0 + j] = rec[RC::kF + r * DV + col0 + j];
        }
        __syncthreads();
        // dR = G dS_next + F;  dS = Diag(A_C) dS_next + E - Kbar^T dR   (this CTA's columns)
        cta_gemm<kC, kCB, DK, false, false>(rec + RC::kdR + col0, DV, rec + RC::kG, DK, dS, DV, 1.f, true, 0, s_buf);
        cta_gemm<DK, kCB, kC, true, false>(dSn, DV, rec + RC::kKb, DK, rec + RC::kdR + col0, DV, -1.f, true, 0,
                                            s_buf);
        for (int e = tid; e < DK * kCB; e += kBT) {
            const int i = e / kCB, j = e % kCB;
            dS[i * DV + j] = fmaf(rec[RC::kAC + i], dS[i * DV + j], dSn[i * DV + j]);
        }
        __syncthreads();
    }
    if (p.d_init)
        for (int e = tid; e < DK * kCB; e += kBT) {
            const int i = e / kCB, j = e % kCB;
            p.d_init[pair * DK * DV + i * DV + col0 + j] = dS[i * DV + j];
        }
}

// ---------------------------------------------------------------------------- phase C
template <int DK, int DV, typename Tin>
__global__ void __launch_bounds__(kBT, 2) kda_bwd_grad_kernel(BwdParams p) {
    using S = Scr<DK, DV>;
    using RC = Rec<DK, DV>;
    __shared__ __align__(16) float s_buf[SmemBuf<DK>::kFloats];
    __shared__ float s_beta[kC], s_dbeta[kC], s_ac[DK], s_red[kBT], s_rk[kC], s_rq[kC];
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
        float *Vs = W + S::kV, *dOs = W + S::kdO, *R = W + S::kR, *U = W + S::kU, *dU = W + S::kdU;
        float *Mr = W + S::kMr, *Pr = W + S::kPr, *P = W + S::kP, *Tp = W + S::kTp, *dP = W + S::kdP;
        float *dTp = W + S::kdTp, *X = W + S::kX, *dM = W + S::kdM;

        load_chunk<DK, DV, Tin>(p, t0, Lc, h, W, true, s_buf, s_beta, s_ac, s_rk, s_rq);
        cta_gemm<kC, kC, DK, false, true>(Mr, kC, Kb, DK, Kt, DK, 1.f, false, 0, s_buf);
        cta_gemm<kC, kC, DK, false, true>(Pr, kC, Qb, DK, Kt, DK, 1.f, false, 0, s_buf);
        for (int e = tid; e < kC * kC; e += kBT) {
            const int i = e / kC, j = e % kC;
            Tp[e] = T[e] * s_beta[j];
            P[e] = i >= j ? Pr[e] : 0.f;
        }
        cta_copy(R, Vs, kC * DV);
        __syncthreads();
        // forward quantities of the chunk: R = V - Kbar S, U = T' R
        if (Sc) cta_gemm<kC, DV, DK, false, false>(R, DV, Kb, DK, Sc, DV, -1.f, true, 0, s_buf);
        cta_gemm<kC, DV, kC, false, false>(U, DV, Tp, kC, R, DV, 1.f, false, 0, s_buf);
        // reverse
        cta_gemm<kC, DV, DK, false, false>(dU, DV, Kh, DK, dSx, DV, 1.f, false, 0, s_buf);
        cta_gemm<kC, DV, kC, true, false>(dU, DV, P, kC, dOs, DV, 1.f, true, 0, s_buf);
        cta_gemm<kC, kC, DV, false, true>(dP, kC, dOs, DV, U, DV, 1.f, false, 1, s_buf);
        cta_gemm<kC, kC, DV, false, true>(dTp, kC, dU, DV, R, DV, 1.f, false, 0, s_buf);
        cta_gemm<kC, DK, kC, false, false>(dQb, DK, dP, kC, Kt, DK, 1.f, false, 0, s_buf);
        if (Sc) cta_gemm<kC, DK, DV, false, true>(dQb, DK, dOs, DV, Sc, DV, 1.f, true, 0, s_buf);
        cta_gemm<kC, DK, DV, false, true>(dKh, DK, U, DV, dSx, DV, 1.f, false, 0, s_buf);
        if (Sc)
            cta_gemm<kC, DK, DV, false, true>(dKb, DK, dR, DV, Sc, DV, -1.f, false, 0, s_buf);
        else
            for (int e = tid; e < kC * DK; e += kBT) dKb[e] = 0.f;
        cta_gemm<kC, DK, kC, true, false>(dKt, DK, dP, kC, Qb, DK, 1.f, false, 0, s_buf);
        // beta through T' = T Diag(beta) (column sums over 4 row quarters); dT = dT' Diag(beta)
        {
            const int j = tid & 63, qr = tid >> 6;
            float acc = 0.f;
            for (int i = qr * 16; i < qr * 16 + 16; ++i) acc = fmaf(dTp[i * kC + j], T[i * kC + j], acc);
            s_red[tid] = acc;
        }
        __syncthreads();
        if (tid < kC) s_dbeta[tid] = (s_red[tid] + s_red[tid + 64]) + (s_red[tid + 128] + s_red[tid + 192]);
        for (int e = tid; e < kC * kC; e += kBT) dTp[e] *= s_beta[e % kC];
        __syncthreads();
        // through the inverse: dM = strictly-lower(-T^T dT T^T)
        cta_gemm<kC, kC, kC, true, false>(X, kC, T, kC, dTp, kC, 1.f, false, 0, s_buf);
        cta_gemm<kC, kC, kC, false, true>(dM, kC, X, kC, T, kC, -1.f, false, 2, s_buf);
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
        for (int e = tid; e < kC * kC; e += kBT) dM[e] *= s_beta[e / kC];
        __syncthreads();
        cta_gemm<kC, DK, kC, false, false>(dKb, DK, dM, kC, Kt, DK, 1.f, true, 0, s_buf);
        cta_gemm<kC, DK, kC, true, false>(dKt, DK, dM, kC, Kb, DK, 1.f, true, 0, s_buf);
        // gate gradients: dlogA_C = A_C sum_j dS_next S + sum_r dKhat Khat
        {
            constexpr int kGroups = kBT / DK;
            const int i = tid % DK, grp = tid / DK;
            float acc = 0.f;
            if (Sc)
                for (int j = grp; j < DV; j += kGroups) acc = fmaf(dSx[i * DV + j], Sc[i * DV + j], acc);
            acc *= s_ac[i];
            for (int r = grp; r < kC; r += kGroups) acc = fmaf(dKh[r * DK + i], Kh[r * DK + i], acc);
            s_red[tid] = acc;
        }
        __syncthreads();
        // per element: dK, dQ and dlogA_r (into shared memory for the reverse sums)
        const bool norms = (p.prep & (PREP_L2NORM_K | PREP_L2NORM_Q)) != 0;
        for (int e = tid; e < kC * DK; e += kBT) {
            const int r = e / DK, i = e % DK;
            const float a = A_[e];
            const float gk = dKb[e] * a + dKt[e] / a + dKh[e] * (s_ac[i] / a);
            const float gq = sc * dQb[e] * a;
            s_buf[e] = dKb[e] * Kb[e] - dKt[e] * Kt[e] + dQb[e] * Qb[e] - dKh[e] * Kh[e];
            if (norms) {  // gradients of the normalised rows, carried back below
                dKb[e] = gk;
                dQb[e] = gq;
            } else if (r < Lc) {
                const int64_t o = ((t0 + r) * H + h) * DK + i;
                st_out(DK_, o, gk);
                st_out(DQ, o, gq);
            }
        }
        for (int e = tid; e < kC * DV; e += kBT) {
            const int r = e / DV, j = e % DV;
            if (r < Lc) st_out(DV_, ((t0 + r) * H + h) * DV + j, dR[e]);
        }
        __syncthreads();
        if (tid < DK) {  // dg_s = dlogA_C + sum_{r >= s} dlogA_r (raw gate x: times 1 - sigmoid(x))
            const bool sig = (p.prep & PREP_SIGMOID_GATE) != 0;
            const Tin *G = static_cast<const Tin *>(p.g);
            float acc = 0.f;
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
}

template <int DK, int DV, typename Tin>
cudaError_t launch_typed(const BwdParams &p, cudaStream_t stream) {
    const int64_t chains = static_cast<int64_t>(p.N) * p.H;
    if (chains <= 0) return cudaSuccess;
    if (chains > 0x7fffffffLL || p.ctas <= 0) return cudaErrorInvalidConfiguration;
    kda_bwd_chunk_kernel<DK, DV, Tin><<<p.ctas, kBT, 0, stream>>>(p);
    kda_bwd_chain_kernel<DK, DV><<<static_cast<unsigned>(chains * (DV / kChainCols)), kBT, 0, stream>>>(p);
    kda_bwd_grad_kernel<DK, DV, Tin><<<p.ctas, kBT, 0, stream>>>(p);
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
