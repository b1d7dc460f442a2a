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
// merge_o_kernel applies the first line: per chain a [tokens x 128] x [128 x 128]
// product on tcgen05 (y tiles by TMA, S1 split into bf16 high and low parts so the
// product keeps ~16 mantissa bits, fp32 accumulation in TMEM), added to o with one
// bf16 rounding; merge_state_kernel the second (fp32), after it, since it overwrites S1.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "kda_internal.h"
#include "sm100_ptx.cuh"

namespace kda {
namespace {

constexpr int kD = 128;
constexpr int kC = 64;
constexpr int kTB = 128;          // segment-1 tokens per step of merge_o_kernel
constexpr int kLdS = kD + 8;      // smem row stride (floats) of S1: conflict-free B fragments
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

using namespace ptx;

constexpr int kMoThreads = 128;                  // one thread per token row of a block
constexpr uint32_t kYTile = 32768;               // 128 tokens x 128 channels bf16 (two 64-channel halves)
constexpr uint32_t kSTile = 32768;               // 128 x 128 bf16, MN-major (two 64-column halves)
constexpr uint32_t kMoSmem = 2 * kYTile + 2 * kSTile + 1024;
constexpr uint64_t kMoWaitNs = 1000000000ull;

// byte offset of 16-bit element (row, col) in a 128-byte-row tile with the 128B swizzle
__device__ __forceinline__ uint32_t swz128(int row, int col) {
    return static_cast<uint32_t>(row * 128 + ((((col >> 3) ^ (row & 7)) << 4) | ((col & 7) << 1)));
}

struct MoParams {
    CUtensorMap tm_y;  // o_phi [T, H, 128] bf16, boxes of 64 channels x 128 tokens
    MergeParams m;
    int parts;
};

// Grid: pairs x parts.  CTA (pair, part) stages S1 once and corrects its share of the
// chain's segment-1 tokens, 128 per block: o_t += S1^T y_t with y_t = Phi_t^T scale q_t.
// Thread 0 issues the TMA loads and the MMAs, one block ahead of the epilogue.
__global__ void __launch_bounds__(kMoThreads, 1) merge_o_kernel(const __grid_constant__ MoParams P) {
    extern __shared__ uint8_t mo_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(mo_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t bar_y[2], bar_d[2];
    __shared__ uint32_t s_tmem;
    __shared__ int s_stop;
    const MergeParams &p = P.m;
    const int64_t pair = blockIdx.x / P.parts;
    const int part = static_cast<int>(blockIdx.x % P.parts);
    const int n = static_cast<int>(pair / p.H), h = static_cast<int>(pair % p.H);
    const int64_t H = p.H;
    int64_t b1, e1;
    if (!segment1(p, n, b1, e1)) return;
    const int64_t nblk = (e1 - b1 + kTB - 1) / kTB;
    const int64_t per = (nblk + P.parts - 1) / P.parts;
    const int64_t blk0 = part * per, blk1 = (blk0 + per < nblk) ? blk0 + per : nblk;
    if (blk0 >= blk1) return;
    const int nb = static_cast<int>(blk1 - blk0);
    const int tid = threadIdx.x, warp = tid >> 5;

    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bar_y[b], 1);
            mbar_init(&bar_d[b], 1);
        }
        s_stop = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&s_tmem, 256);
        tmem_relinquish();
    }
    // S1 = hi + lo in bf16, MN-major (row = channel k, 128 bytes = 64 value columns per half)
    uint8_t *Shi = sm + 2 * kYTile, *Slo = Shi + kSTile;
    const float *S1 = p.state + pair * kD * kD;
    for (int i = tid; i < kD * kD; i += kMoThreads) {
        const int k = i >> 7, j = i & 127;
        const float x = S1[i];
        const __nv_bfloat16 hi = __float2bfloat16_rn(x);
        const __nv_bfloat16 lo = __float2bfloat16_rn(x - __bfloat162float(hi));
        const uint32_t off = (j >> 6) * 16384 + swz128(k, j & 63);
        *reinterpret_cast<__nv_bfloat16 *>(Shi + off) = hi;
        *reinterpret_cast<__nv_bfloat16 *>(Slo + off) = lo;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const uint32_t sbase = smem_u32(sm);
    const uint32_t idesc = idesc_bf16(128, 128, false, true);

    // thread 0: TMA of block i's y rows into buffer i & 1, and block i's 16 MMAs into D[i & 1]
    auto load_y = [&](int i) {
        uint8_t *dst = sm + (i & 1) * kYTile;
        const int t = static_cast<int>(b1 + (blk0 + i) * kTB);
        mbar_arrive_expect_tx(&bar_y[i & 1], kYTile);
        tma_load_3d(dst, &P.tm_y, 0, h, t, &bar_y[i & 1]);
        tma_load_3d(dst + 16384, &P.tm_y, 64, h, t, &bar_y[i & 1]);
    };
    auto issue = [&](int i) -> bool {
        if (!mbar_wait(&bar_y[i & 1], (i >> 1) & 1, globaltimer_ns() + kMoWaitNs)) return false;
        tc_fence_after();
        const uint64_t dA = sdesc_sw128(sbase + (i & 1) * kYTile, 16, 1024);        // y rows, K-major
        const uint64_t dH = sdesc_sw128(sbase + 2 * kYTile, 16384, 1024);          // S1 high, MN-major
        const uint64_t dL = sdesc_sw128(sbase + 2 * kYTile + kSTile, 16384, 1024); // S1 low
        const uint32_t tD = tmem + 128 * (i & 1);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
            mma_bf16_ss(tD, dA + (((ks >> 2) * 16384 + (ks & 3) * 32) >> 4), dH + ((ks * 2048) >> 4), idesc,
                        ks > 0 ? 1u : 0u);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
            mma_bf16_ss(tD, dA + (((ks >> 2) * 16384 + (ks & 3) * 32) >> 4), dL + ((ks * 2048) >> 4), idesc, 1u);
        mma_commit(&bar_d[i & 1]);
        return true;
    };
    if (tid == 0) {
        load_y(0);
        if (nb > 1) load_y(1);
        if (!issue(0)) {
            s_stop = 1;
            atomicOr(p.status, DEV_ERR_TIMEOUT);
        }
    }
    __syncthreads();

    __nv_bfloat16 *O = static_cast<__nv_bfloat16 *>(p.o);
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    // this thread's o row of block i (orow), and of block i + 1 (onext), read one block ahead so
    // that the read's latency overlaps the current block's products and epilogue
    uint4 orow[16], onext[16];
    {
        const int64_t t = b1 + blk0 * kTB + tid;
        if (t < e1) {
            const __nv_bfloat16 *op = O + (t * H + h) * kD;
#pragma unroll
            for (int c = 0; c < 16; ++c) orow[c] = reinterpret_cast<const uint4 *>(op)[c];
        }
    }
    int i = 0;
    for (; i < nb && !*reinterpret_cast<volatile int *>(&s_stop); ++i) {  // read after the block's barrier
        if (tid == 0) {
            bool ok = true;
            if (i + 1 < nb) {
                // buffer i & 1 is free once block i's products are done; then block i+2 may land there
                ok = mbar_wait(&bar_d[i & 1], (i >> 1) & 1, globaltimer_ns() + kMoWaitNs);
                if (ok && i + 2 < nb) load_y(i + 2);
                if (ok) ok = issue(i + 1);
            }
            if (!ok) {
                s_stop = 1;
                atomicOr(p.status, DEV_ERR_TIMEOUT);
            }
        }
        if (i + 1 < nb) {
            const int64_t t = b1 + (blk0 + i + 1) * kTB + tid;
            if (t < e1) {
                const __nv_bfloat16 *op = O + (t * H + h) * kD;
#pragma unroll
                for (int c = 0; c < 16; ++c) onext[c] = reinterpret_cast<const uint4 *>(op)[c];
            }
        }
        // every thread: block i's accumulator row -> o row (this thread's token)
        const bool got = mbar_wait(&bar_d[i & 1], (i >> 1) & 1, globaltimer_ns() + kMoWaitNs);
        if (!got) {
            s_stop = 1;
            atomicOr(p.status, DEV_ERR_TIMEOUT);
        }
        tc_fence_after();
        const int64_t t_begin = b1 + (blk0 + i) * kTB;
        const bool mine = got && (t_begin + tid < e1);
        __nv_bfloat16 *op = O + ((t_begin + tid) * H + h) * kD;
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) {
            uint32_t a[32];
            tmem_ld16(tmem + lane_base + 128 * (i & 1) + 32 * cb, *reinterpret_cast<uint32_t(*)[16]>(&a[0]));
            tmem_ld16(tmem + lane_base + 128 * (i & 1) + 32 * cb + 16, *reinterpret_cast<uint32_t(*)[16]>(&a[16]));
            tmem_ld_wait();
            if (mine) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t *w = reinterpret_cast<uint32_t *>(&orow[4 * cb + c]);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 o0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[e]));
                        const __nv_bfloat162 r = __floats2bfloat162_rn(o0.x + __uint_as_float(a[8 * c + 2 * e]),
                                                                       o0.y + __uint_as_float(a[8 * c + 2 * e + 1]));
                        w[e] = *reinterpret_cast<const uint32_t *>(&r);
                    }
                }
            }
        }
        if (mine) {
#pragma unroll
            for (int c = 0; c < 16; ++c) reinterpret_cast<uint4 *>(op)[c] = orow[c];
        }
#pragma unroll
        for (int c = 0; c < 16; ++c) orow[c] = onext[c];
        tc_fence_before();
        __syncthreads();
    }
    // drain: every MMA and TMA copy issued has completed before the TMEM and smem go away
    if (tid == 0) {
        const uint64_t dl = globaltimer_ns() + kMoWaitNs;
        for (int k = i; k < nb && k <= i + 1; ++k) {
            mbar_wait(&bar_d[k & 1], (k >> 1) & 1, dl);
        }
        for (int k = i; k < nb && k <= i + 2; ++k) mbar_wait(&bar_y[k & 1], (k >> 1) & 1, dl);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
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

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *ptr = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

}  // namespace

cudaError_t launch_merge(const MergeParams &p, cudaStream_t stream) {
    const int64_t pairs = static_cast<int64_t>(p.N) * p.H;
    if (pairs <= 0) return cudaSuccess;
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaErrorInvalidValue;
    MoParams mo{};
    mo.m = p;
    mo.parts = static_cast<int>(sms / pairs > 1 ? sms / pairs : 1);  // about one CTA per SM
    auto enc = tensor_map_encoder();
    if (!enc) return cudaErrorInvalidValue;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(p.H), static_cast<cuuint64_t>(p.T_total)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD) * 2, static_cast<cuuint64_t>(p.H) * kD * 2};
    cuuint32_t box[3] = {64, 1, kTB};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&mo.tm_y, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(p.o_phi), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const size_t smem_s = static_cast<size_t>(2 * kD * kLdS) * sizeof(float);
    // The dynamic shared-memory limit is a function attribute of the device that is current
    // when it is set, so it is set on every launch (a host-side call that allocates nothing).
    cudaError_t e = cudaFuncSetAttribute(merge_o_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kMoSmem));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(merge_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem_s));
    if (e != cudaSuccess) return e;
    const int64_t grid_o = pairs * mo.parts;
    if (grid_o > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    merge_o_kernel<<<static_cast<unsigned>(grid_o), kMoThreads, kMoSmem, stream>>>(mo);
    merge_state_kernel<<<static_cast<unsigned>(pairs), kMergeThreads, smem_s, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
