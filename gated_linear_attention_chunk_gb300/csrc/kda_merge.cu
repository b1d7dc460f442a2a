// T-segment merge for the chunked prefill.
//
// When a batch has too few (sequence, head) chains to occupy the GPU, the full
// chunks of every sequence are cut in two at a chunk boundary and the chunked
// kernel runs three independent roles per chain (see kda_chunk_tc.cu): segment 0
// from the initial state, which leaves S1, the state at the cut; segment 1 from a
// zero state, which leaves Psi and writes the zero-start outputs o0_t; and segment
// 1 from the identity with v = 0, which leaves the segment's transition Phi and
// writes Phi_t^T (scale q_t).  The recurrence is affine in the state
// (S_t = A_t S_{t-1} + B_t, with A_t = (I - beta_t k_t k_t^T) Diag(alpha_t) acting
// on the dk rows), which is what makes the split exact ("Kimi K3 on Fireworks:
// Fast RL at frontier scale", context-parallel paragraph: a long sequence's state
// is handed across segments):
//
//     o_t     = o0_t + S1^T (Phi_t^T scale q_t)     for t in segment 1
//     S_final = Phi S1 + Psi
//
// merge_o_kernel applies the first line (a [tokens x 128] x [128 x 128] product per
// chain, on the tensor cores with tf32 operands and fp32 accumulation), and
// merge_state_kernel the second (fp32), after it, since it overwrites S1.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kD = 128;
constexpr int kC = 64;
constexpr int kTB = 128;          // segment-1 tokens per step of merge_o_kernel
constexpr int kLdS = kD + 8;      // smem row stride (floats) of S1: conflict-free B fragments
constexpr int kLdY = kD + 8;      // smem row stride (bf16) of the y rows: conflict-free A fragments
constexpr int kMergeThreads = 256;

// Segment 1 of sequence n: tokens [b1, e1) (whole chunks).  False if it is empty
// or the sequence bounds are invalid (the chunked kernel reports those).
__device__ bool segment1(const MergeParams &p, int n, int64_t &b1, int64_t &e1) {
    int64_t bos, eos;
    if (p.cu) {
        bos = p.cu[n];
        eos = p.cu[n + 1];
        if (!(bos >= 0 && bos <= eos && eos <= p.T_total)) return false;
    } else {
        bos = static_cast<int64_t>(n) * p.seq_len_fixed;
        eos = bos + p.seq_len_fixed;
    }
    const int64_t nfull = (eos - bos) / kC;
    const int64_t n0 = (nfull + 1) / 2;
    b1 = bos + kC * n0;
    e1 = bos + kC * nfull;
    return e1 > b1;
}

__device__ __forceinline__ float to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// c += a b for one m16n8k8 tile (tf32 operands as fp32 bit patterns, fp32 accumulate).
__device__ __forceinline__ void mma_tf32(float (&c)[4], float a0, float a1, float a2, float a3, float b0, float b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(__float_as_uint(a0)), "r"(__float_as_uint(a1)), "r"(__float_as_uint(a2)), "r"(__float_as_uint(a3)),
          "r"(__float_as_uint(b0)), "r"(__float_as_uint(b1)));
}

// Grid: pairs x parts.  CTA (pair, part) loads S1 once and corrects its share of the
// chain's segment-1 tokens, 128 at a time: o_t += S1^T y_t with y_t = Phi_t^T scale q_t.
__global__ void __launch_bounds__(kMergeThreads, 2) merge_o_kernel(MergeParams p, int parts) {
    extern __shared__ float msm[];
    float *Ss = msm;                                                        // S1 [channel i][value j], tf32
    uint16_t *Ys = reinterpret_cast<uint16_t *>(msm + kD * kLdS);          // y rows [token][channel], bf16
    const int64_t pair = blockIdx.x / parts;
    const int part = static_cast<int>(blockIdx.x % parts);
    const int n = static_cast<int>(pair / p.H), h = static_cast<int>(pair % p.H);
    const int64_t H = p.H;
    int64_t b1, e1;
    if (!segment1(p, n, b1, e1)) return;
    const int64_t nblk = (e1 - b1 + kTB - 1) / kTB;
    const int64_t per = (nblk + parts - 1) / parts;
    const int64_t blk0 = part * per, blk1 = (blk0 + per < nblk) ? blk0 + per : nblk;
    if (blk0 >= blk1) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, tq = lane & 3, r0 = 16 * warp;

    const float *S1 = p.state + pair * kD * kD;
    for (int i = tid; i < kD * kD / 4; i += kMergeThreads) {
        const int r = i / (kD / 4), c4 = i % (kD / 4);
        const float4 v = reinterpret_cast<const float4 *>(S1)[i];
        float *d = Ss + r * kLdS + 4 * c4;
        d[0] = to_tf32(v.x);
        d[1] = to_tf32(v.y);
        d[2] = to_tf32(v.z);
        d[3] = to_tf32(v.w);
    }
    const __nv_bfloat16 *Y = static_cast<const __nv_bfloat16 *>(p.o_phi);
    __nv_bfloat16 *O = static_cast<__nv_bfloat16 *>(p.o);
    auto yv = [&](int r, int c) { return __uint_as_float(static_cast<uint32_t>(Ys[r * kLdY + c]) << 16); };
    for (int64_t blk = blk0; blk < blk1; ++blk) {
        const int64_t t_begin = b1 + blk * kTB;
        const int ntok = static_cast<int>(e1 - t_begin < kTB ? e1 - t_begin : kTB);  // 64 or 128
        __syncthreads();  // the previous block's y rows are no longer read (and S1 is staged)
        {
            // all of this thread's loads first, then the stores (one memory round trip)
            constexpr int kPer = kTB * (kD / 8) / kMergeThreads;
            uint4 yv4[kPer];
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
                const int i = tid + u * kMergeThreads, r = i / (kD / 8), c8 = i % (kD / 8);
                if (r < ntok) yv4[u] = *reinterpret_cast<const uint4 *>(Y + ((t_begin + r) * H + h) * kD + 8 * c8);
            }
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
                const int i = tid + u * kMergeThreads, r = i / (kD / 8), c8 = i % (kD / 8);
                if (r < ntok) *reinterpret_cast<uint4 *>(Ys + r * kLdY + 8 * c8) = yv4[u];
            }
        }
        __syncthreads();
        if (r0 >= ntok) continue;
        // warp: tokens [r0, r0 + 16) x all 128 value columns; fragment row gq, column tq
        float acc[16][4];
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll 2
        for (int k0 = 0; k0 < kD; k0 += 8) {
            const float a0 = yv(r0 + gq, k0 + tq), a1 = yv(r0 + gq + 8, k0 + tq);  // bf16 is exact in tf32
            const float a2 = yv(r0 + gq, k0 + tq + 4), a3 = yv(r0 + gq + 8, k0 + tq + 4);
#pragma unroll
            for (int nt = 0; nt < 16; ++nt)
                mma_tf32(acc[nt], a0, a1, a2, a3, Ss[(k0 + tq) * kLdS + 8 * nt + gq],
                         Ss[(k0 + tq + 4) * kLdS + 8 * nt + gq]);
        }
        // o (bf16) += acc, rounded once; all 32 loads are issued before the first store
        __nv_bfloat162 *orow[2];
#pragma unroll
        for (int hr = 0; hr < 2; ++hr)
            orow[hr] = reinterpret_cast<__nv_bfloat162 *>(O + ((t_begin + r0 + gq + 8 * hr) * H + h) * kD + 2 * tq);
        __nv_bfloat162 ov[16][2];
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            ov[nt][0] = orow[0][4 * nt];
            ov[nt][1] = orow[1][4 * nt];
        }
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const float2 o0 = __bfloat1622float2(ov[nt][hr]);
                orow[hr][4 * nt] = __floats2bfloat162_rn(o0.x + acc[nt][2 * hr], o0.y + acc[nt][2 * hr + 1]);
            }
        }
    }
}

// One CTA per chain: state <- Phi state + Psi (state holds S1 on entry).
__global__ void __launch_bounds__(kMergeThreads) merge_state_kernel(MergeParams p) {
    extern __shared__ float msm[];
    float *Ss = msm;              // S1 [m][j]
    float *Ps = msm + kD * kLdS;  // Phi [i][m]
    const int64_t pair = blockIdx.x;
    const int n = static_cast<int>(pair / p.H);
    int64_t b1, e1;
    if (!segment1(p, n, b1, e1)) return;  // no segment 1: the state at the cut is final
    float *S = p.state + pair * kD * kD;
    const float *Phi = p.phi + pair * kD * kD, *Psi = p.psi + pair * kD * kD;
    const int tid = threadIdx.x;
    for (int i = tid; i < kD * kD / 4; i += kMergeThreads) {
        const int r = i / (kD / 4), c4 = i % (kD / 4);
        *reinterpret_cast<float4 *>(Ss + r * kLdS + 4 * c4) = reinterpret_cast<const float4 *>(S)[i];
        *reinterpret_cast<float4 *>(Ps + r * kLdS + 4 * c4) = reinterpret_cast<const float4 *>(Phi)[i];
    }
    __syncthreads();
    // thread: rows warp + 8 a (a < 16), columns 4 (lane) .. 4 (lane) + 3
    const int i0 = tid >> 5, j0 = 4 * (tid & 31);
    float acc[16][4];
#pragma unroll
    for (int a = 0; a < 16; ++a) acc[a][0] = acc[a][1] = acc[a][2] = acc[a][3] = 0.f;
    for (int m = 0; m < kD; ++m) {
        const float4 sv = *reinterpret_cast<const float4 *>(Ss + m * kLdS + j0);
#pragma unroll
        for (int a = 0; a < 16; ++a) {
            const float ph = Ps[(i0 + 8 * a) * kLdS + m];
            acc[a][0] = fmaf(ph, sv.x, acc[a][0]);
            acc[a][1] = fmaf(ph, sv.y, acc[a][1]);
            acc[a][2] = fmaf(ph, sv.z, acc[a][2]);
            acc[a][3] = fmaf(ph, sv.w, acc[a][3]);
        }
    }
    float4 ps[16];  // all loads before the first store
#pragma unroll
    for (int a = 0; a < 16; ++a) ps[a] = *reinterpret_cast<const float4 *>(Psi + (i0 + 8 * a) * kD + j0);
#pragma unroll
    for (int a = 0; a < 16; ++a)
        *reinterpret_cast<float4 *>(S + (i0 + 8 * a) * kD + j0) =
            make_float4(acc[a][0] + ps[a].x, acc[a][1] + ps[a].y, acc[a][2] + ps[a].z, acc[a][3] + ps[a].w);
}

}  // namespace

cudaError_t launch_merge(const MergeParams &p, cudaStream_t stream) {
    const int64_t pairs = static_cast<int64_t>(p.N) * p.H;
    if (pairs <= 0) return cudaSuccess;
    // CTAs per chain: about two per SM over the whole grid
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaErrorInvalidValue;
    const int parts = static_cast<int>((2 * static_cast<int64_t>(sms) + pairs - 1) / pairs);
    const size_t smem_o = static_cast<size_t>(kD * kLdS) * sizeof(float) + static_cast<size_t>(kTB * kLdY) * 2;
    const size_t smem_s = static_cast<size_t>(2 * kD * kLdS) * sizeof(float);
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(merge_o_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem_o));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(merge_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(smem_s));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int64_t grid_o = pairs * parts;
    if (grid_o > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    merge_o_kernel<<<static_cast<unsigned>(grid_o), kMergeThreads, smem_o, stream>>>(p, parts);
    merge_state_kernel<<<static_cast<unsigned>(pairs), kMergeThreads, smem_s, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
