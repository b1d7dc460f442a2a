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
// One CTA of 256 threads per (sequence, head) takes the chunks last to first;
// every product is a small fp32 matrix product over the chain's scratch in global
// memory (it stays in L2), staged through shared memory in 16-deep slices.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kBT = 256;  // threads per CTA
constexpr int kC = 64;    // chunk length

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
    constexpr int MB = M / 16, NB = N / 16, PA = M + 4, PB = N + 4;
    float *As = sm;            // [16][PA]: op(A) slice, k-major
    float *Bs = sm + 16 * PA;  // [16][PB]
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    float c[MB][NB];
#pragma unroll
    for (int x = 0; x < MB; ++x)
#pragma unroll
        for (int y = 0; y < NB; ++y) c[x][y] = 0.f;
    for (int k0 = 0; k0 < K; k0 += 16) {
        for (int e = tid; e < 16 * M; e += kBT) {
            if (TA) {
                const int kk = e / M, i = e % M;
                As[kk * PA + i] = A[(k0 + kk) * lda + i];
            } else {
                const int i = e >> 4, kk = e & 15;
                As[kk * PA + i] = A[i * lda + k0 + kk];
            }
        }
        for (int e = tid; e < 16 * N; e += kBT) {
            if (!TB) {
                const int kk = e / N, j = e % N;
                Bs[kk * PB + j] = B[(k0 + kk) * ldb + j];
            } else {
                const int j = e >> 4, kk = e & 15;
                Bs[kk * PB + j] = B[j * ldb + k0 + kk];
            }
        }
        __syncthreads();
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

// Scratch of one chain, in floats.
template <int DK, int DV>
struct Scratch {
    static constexpr int64_t kA = 0, kKb = kA + kC * DK, kKt = kKb + kC * DK, kKh = kKt + kC * DK,
                             kQb = kKh + kC * DK, kdQb = kQb + kC * DK, kdKb = kdQb + kC * DK,
                             kdKt = kdKb + kC * DK, kdKh = kdKt + kC * DK, kV = kdKh + kC * DK,
                             kdO = kV + kC * DV, kR = kdO + kC * DV, kU = kR + kC * DV, kdU = kU + kC * DV,
                             kdR = kdU + kC * DV, kMr = kdR + kC * DV, kPr = kMr + kC * kC, kP = kPr + kC * kC,
                             kT = kP + kC * kC, kTp = kT + kC * kC, kdP = kTp + kC * kC, kdTp = kdP + kC * kC,
                             kX = kdTp + kC * kC, kdM = kX + kC * kC, kdS = kdM + kC * kC, kdSn = kdS + DK * DV,
                             kTotal = kdSn + DK * DV;
};

template <int DK, int DV, typename Tin>
__global__ void __launch_bounds__(kBT, 1) kda_bwd_kernel(BwdParams p) {
    using SC = Scratch<DK, DV>;
    constexpr int kPad = kC + 1;
    // shared: the matrix-product slices, or the gate tile / the two 64 x 64 matrices of
    // the inverse (never live at the same time)
    constexpr int kGemmFloats = 16 * (128 + 4 + 128 + 4);
    constexpr int kUnion = (kC * DK > 2 * kC * kPad ? kC * DK : 2 * kC * kPad);
    __shared__ __align__(16) float s_buf[kGemmFloats > kUnion ? kGemmFloats : kUnion];
    __shared__ float s_beta[kC], s_dbeta[kC], s_ac[DK], s_dlac[DK];

    const int tid = threadIdx.x;
    const int64_t pair = blockIdx.x;
    const int n = static_cast<int>(pair / p.H), h = static_cast<int>(pair % p.H);
    const int64_t H = p.H;
    int64_t bos, eos;
    if (p.cu) {
        bos = p.cu[n];
        eos = p.cu[n + 1];
        bool ok = (bos >= 0) && (bos <= eos) && (eos <= p.T_total);
        if (n == 0 && bos != 0) ok = false;
        if (n == p.N - 1 && eos != p.T_total) ok = false;
        if (!ok) {
            if (tid == 0 && h == 0) atomicOr(p.status, DEV_ERR_SEQLENS);
            return;
        }
    } else {
        bos = static_cast<int64_t>(n) * p.seq_len_fixed;
        eos = bos + p.seq_len_fixed;
    }
    const Tin *Q = static_cast<const Tin *>(p.q), *K = static_cast<const Tin *>(p.k);
    const Tin *V = static_cast<const Tin *>(p.v), *G = static_cast<const Tin *>(p.g);
    const Tin *B = static_cast<const Tin *>(p.beta), *DO = static_cast<const Tin *>(p.d_o);
    Tin *DQ = static_cast<Tin *>(p.dq), *DK_ = static_cast<Tin *>(p.dk), *DV_ = static_cast<Tin *>(p.dv);
    Tin *DG = static_cast<Tin *>(p.dg), *DB = static_cast<Tin *>(p.dbeta);

    float *W = p.scratch + pair * SC::kTotal;
    float *A_ = W + SC::kA, *Kb = W + SC::kKb, *Kt = W + SC::kKt, *Kh = W + SC::kKh, *Qb = W + SC::kQb;
    float *dQb = W + SC::kdQb, *dKb = W + SC::kdKb, *dKt = W + SC::kdKt, *dKh = W + SC::kdKh;
    float *Vs = W + SC::kV, *dOs = W + SC::kdO, *R = W + SC::kR, *U = W + SC::kU, *dU = W + SC::kdU;
    float *dR = W + SC::kdR, *Mr = W + SC::kMr, *Pr = W + SC::kPr, *P = W + SC::kP, *T = W + SC::kT;
    float *Tp = W + SC::kTp, *dP = W + SC::kdP, *dTp = W + SC::kdTp, *X = W + SC::kX, *dM = W + SC::kdM;
    float *dS = W + SC::kdS, *dSn = W + SC::kdSn;

    for (int e = tid; e < DK * DV; e += kBT) dS[e] = p.d_final ? p.d_final[pair * DK * DV + e] : 0.f;
    __syncthreads();

    const int64_t len = eos - bos;
    const int nch = static_cast<int>((len + kC - 1) / kC);
    const int64_t ck0 = ckpt_base(bos, n);
    const float sc = p.scale;
    for (int c = nch - 1; c >= 0; --c) {
        const int64_t t0 = bos + static_cast<int64_t>(c) * kC;
        const int Lc = static_cast<int>(eos - t0 < kC ? eos - t0 : kC);
        const float *S = p.ckpt + ((ck0 + c) * H + h) * DK * DV;

        // ---- chunk inputs: gates into shared memory, prefix products per channel
        for (int e = tid; e < kC * DK; e += kBT) {
            const int r = e / DK, i = e % DK;
            s_buf[e] = r < Lc ? ld_in(G, ((t0 + r) * H + h) * DK + i) : 0.f;
        }
        if (tid < kC) s_beta[tid] = tid < Lc ? ld_in(B, (t0 + tid) * H + h) : 0.f;
        __syncthreads();
        if (tid < DK) {
            float a = 1.f;
            for (int r = 0; r < kC; ++r) {
                a *= expf(s_buf[r * DK + tid]);
                A_[r * DK + tid] = a;
            }
            s_ac[tid] = a;
            if (!(a >= 7.888609052210118e-31f)) atomicOr(p.status, DEV_ERR_GATE);  // 2^-100, as in the forward
        }
        __syncthreads();
        for (int e = tid; e < kC * DK; e += kBT) {
            const int r = e / DK, i = e % DK;
            const bool ok = r < Lc;
            const float kk = ok ? ld_in(K, ((t0 + r) * H + h) * DK + i) : 0.f;
            const float qq = ok ? ld_in(Q, ((t0 + r) * H + h) * DK + i) : 0.f;
            const float a = A_[e];
            Kb[e] = kk * a;
            Kt[e] = kk / a;
            Kh[e] = (kk / a) * s_ac[i];
            Qb[e] = sc * qq * a;
        }
        for (int e = tid; e < kC * DV; e += kBT) {
            const int r = e / DV, j = e % DV;
            const bool ok = r < Lc;
            Vs[e] = ok ? ld_in(V, ((t0 + r) * H + h) * DV + j) : 0.f;
            dOs[e] = ok ? ld_in(DO, ((t0 + r) * H + h) * DV + j) : 0.f;
        }
        __syncthreads();

        // ---- Gram matrices, T = (I + M)^-1, T' and P
        cta_gemm<kC, kC, DK, false, true>(Mr, kC, Kb, DK, Kt, DK, 1.f, false, 0, s_buf);
        cta_gemm<kC, kC, DK, false, true>(Pr, kC, Qb, DK, Kt, DK, 1.f, false, 0, s_buf);
        {
            float *sM = s_buf, *sT = s_buf + kC * kPad;
            for (int e = tid; e < kC * kC; e += kBT) {
                const int i = e / kC, j = e % kC;
                sM[i * kPad + j] = i > j ? s_beta[i] * Mr[e] : 0.f;
                P[e] = i >= j ? Pr[e] : 0.f;
            }
            __syncthreads();
            if (tid < kC) {  // column j by forward substitution: T_ij = -sum_{j <= k < i} M_ik T_kj
                const int j = tid;
                for (int i = 0; i < j; ++i) sT[i * kPad + j] = 0.f;
                sT[j * kPad + j] = 1.f;
                for (int i = j + 1; i < kC; ++i) {
                    float acc = 0.f;
                    for (int k = j; k < i; ++k) acc = fmaf(sM[i * kPad + k], sT[k * kPad + j], acc);
                    sT[i * kPad + j] = -acc;
                }
            }
            __syncthreads();
            for (int e = tid; e < kC * kC; e += kBT) {
                const int i = e / kC, j = e % kC;
                const float t = sT[i * kPad + j];
                T[e] = t;
                Tp[e] = t * s_beta[j];
            }
            for (int e = tid; e < kC * DV; e += kBT) R[e] = Vs[e];
            __syncthreads();
        }
        // ---- forward quantities of the chunk: R = V - Kbar S, U = T' R
        cta_gemm<kC, DV, DK, false, false>(R, DV, Kb, DK, S, DV, -1.f, true, 0, s_buf);
        cta_gemm<kC, DV, kC, false, false>(U, DV, Tp, kC, R, DV, 1.f, false, 0, s_buf);
        // ---- reverse
        cta_gemm<kC, DV, DK, false, false>(dU, DV, Kh, DK, dS, DV, 1.f, false, 0, s_buf);
        cta_gemm<kC, DV, kC, true, false>(dU, DV, P, kC, dOs, DV, 1.f, true, 0, s_buf);
        cta_gemm<kC, kC, DV, false, true>(dP, kC, dOs, DV, U, DV, 1.f, false, 1, s_buf);
        cta_gemm<kC, DV, kC, true, false>(dR, DV, Tp, kC, dU, DV, 1.f, false, 0, s_buf);
        cta_gemm<kC, kC, DV, false, true>(dTp, kC, dU, DV, R, DV, 1.f, false, 0, s_buf);
        cta_gemm<kC, DK, DV, false, true>(dQb, DK, dOs, DV, S, DV, 1.f, false, 0, s_buf);
        cta_gemm<kC, DK, kC, false, false>(dQb, DK, dP, kC, Kt, DK, 1.f, true, 0, s_buf);
        cta_gemm<kC, DK, DV, false, true>(dKh, DK, U, DV, dS, DV, 1.f, false, 0, s_buf);
        cta_gemm<kC, DK, DV, false, true>(dKb, DK, dR, DV, S, DV, -1.f, false, 0, s_buf);
        cta_gemm<kC, DK, kC, true, false>(dKt, DK, dP, kC, Qb, DK, 1.f, false, 0, s_buf);
        // beta through T' = T Diag(beta); then dT = dT' Diag(beta) in place
        if (tid < kC) {
            float acc = 0.f;
            for (int i = 0; i < kC; ++i) acc = fmaf(dTp[i * kC + tid], T[i * kC + tid], acc);
            s_dbeta[tid] = acc;
        }
        __syncthreads();
        for (int e = tid; e < kC * kC; e += kBT) dTp[e] *= s_beta[e % kC];
        __syncthreads();
        // through the inverse: dM = strictly-lower(-T^T dT T^T)
        cta_gemm<kC, kC, kC, true, false>(X, kC, T, kC, dTp, kC, 1.f, false, 0, s_buf);
        cta_gemm<kC, kC, kC, false, true>(dM, kC, X, kC, T, kC, -1.f, false, 2, s_buf);
        // through M = Diag(beta) strictly-lower(Kbar Ktil^T)
        if (tid < kC) {
            float acc = 0.f;
            for (int j = 0; j < tid; ++j) acc = fmaf(dM[tid * kC + j], Mr[tid * kC + j], acc);
            s_dbeta[tid] += acc;
        }
        __syncthreads();
        for (int e = tid; e < kC * kC; e += kBT) dM[e] *= s_beta[e / kC];
        __syncthreads();
        cta_gemm<kC, DK, kC, false, false>(dKb, DK, dM, kC, Kt, DK, 1.f, true, 0, s_buf);
        cta_gemm<kC, DK, kC, true, false>(dKt, DK, dM, kC, Kb, DK, 1.f, true, 0, s_buf);
        // ---- gate gradients
        if (tid < DK) {
            float acc = 0.f;
            for (int j = 0; j < DV; ++j) acc = fmaf(dS[tid * DV + j], S[tid * DV + j], acc);
            acc *= s_ac[tid];
            for (int r = 0; r < kC; ++r) acc = fmaf(dKh[r * DK + tid], Kh[r * DK + tid], acc);
            s_dlac[tid] = acc;
        }
        __syncthreads();  // Khat is overwritten below
        for (int e = tid; e < kC * DK; e += kBT) {
            const int r = e / DK, i = e % DK;
            const float a = A_[e];
            const float gk = dKb[e] * a + dKt[e] / a + dKh[e] * (s_ac[i] / a);
            const float gq = sc * dQb[e] * a;
            const float dla = dKb[e] * Kb[e] - dKt[e] * Kt[e] + dQb[e] * Qb[e] - dKh[e] * Kh[e];
            Kh[e] = dla;  // Khat is not read again in this chunk
            if (r < Lc) {
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
        if (tid < DK) {  // dg_s = dlogA_C + sum_{r >= s} dlogA_r
            float acc = s_dlac[tid];
            for (int r = kC - 1; r >= 0; --r) {
                acc += Kh[r * DK + tid];
                if (r < Lc) st_out(DG, ((t0 + r) * H + h) * DK + tid, acc);
            }
        }
        if (tid < Lc) st_out(DB, (t0 + tid) * H + h, s_dbeta[tid]);
        // ---- gradient of the chunk's start state
        cta_gemm<DK, DV, kC, true, false>(dSn, DV, Qb, DK, dOs, DV, 1.f, false, 0, s_buf);
        cta_gemm<DK, DV, kC, true, false>(dSn, DV, Kb, DK, dR, DV, -1.f, true, 0, s_buf);
        for (int e = tid; e < DK * DV; e += kBT) dS[e] = fmaf(s_ac[e / DV], dS[e], dSn[e]);
        __syncthreads();
    }
    if (p.d_init)
        for (int e = tid; e < DK * DV; e += kBT) p.d_init[pair * DK * DV + e] = dS[e];
}

template <int DK, int DV, typename Tin>
cudaError_t launch_typed(const BwdParams &p, cudaStream_t stream) {
    const int64_t blocks = static_cast<int64_t>(p.N) * p.H;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kda_bwd_kernel<DK, DV, Tin><<<static_cast<unsigned>(blocks), kBT, 0, stream>>>(p);
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

}  // namespace

size_t bwd_scratch_floats(int dk, int dv) {
    if (dk == 128 && dv == 128) return static_cast<size_t>(Scratch<128, 128>::kTotal);
    if (dk == 64 && dv == 64) return static_cast<size_t>(Scratch<64, 64>::kTotal);
    if (dk == 128 && dv == 64) return static_cast<size_t>(Scratch<128, 64>::kTotal);
    if (dk == 64 && dv == 128) return static_cast<size_t>(Scratch<64, 128>::kTotal);
    return 0;
}

cudaError_t launch_bwd(const BwdParams &p, int dk, int dv, int dtype, cudaStream_t stream) {
    if (dtype == 0) return launch_dims<__nv_bfloat16>(p, dk, dv, stream);
    return launch_dims<float>(p, dk, dv, stream);
}

}  // namespace kda
