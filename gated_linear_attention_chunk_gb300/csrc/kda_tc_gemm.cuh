// CTA-wide matrix products on the tcgen05 tensor cores (kind::tf32, fp32 accumulation in TMEM),
// for the backward's small products (M, N <= 128, K in {64, 128}) whose operands and results sit
// in global memory (the chain's scratch and records; read through L2, so a CTA's own earlier
// stores are seen after a barrier).
//
//   C (M x N, row stride ldc) = alpha op(A) op(B), or += when `acc`, with the optional triangular
//   masks (1 keeps entries i >= j, 2 entries i > j, 3 rows i < 64 whole and rows i >= 64 where
//   i - 64 >= j: two stacked 64-row results, the second lower-triangular).
//
// op(A) is staged as a 128-row, K-major tile with the 128-byte swizzle (rows M .. 127 are not
// written: their results are never read), op(B) as an N-row K-major tile (row n holds column n of
// op(B)); 64 columns of K at a time, so a product with K = 128 takes two passes that accumulate
// in TMEM.  One thread issues the MMAs (K = 8 per instruction) and commits them to an mbarrier;
// every thread waits (bounded), then the accumulator is read back by TMEM lane = row.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sm100_ptx.cuh"

namespace kda {
namespace tcg {

using namespace ptx;

constexpr int kKPass = 64;                     // K columns staged per pass
constexpr uint32_t kTileA = 128 * kKPass * 4;  // 32 KB: 128 rows x 64 fp32 (two 128-byte atoms per row)
constexpr uint32_t kTileB = 128 * kKPass * 4;  // 32 KB: up to 128 rows
constexpr uint32_t kSmemBytes = kTileA + kTileB + 1024;  // plus room to align to 1024 bytes

// Instruction descriptor, kind::tf32: D f32, A and B tf32 (format 2), both K-major, M = 128.
__host__ __device__ constexpr uint32_t idesc_tf32(int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(128 >> 4) << 24);
}

__device__ __forceinline__ void mma_tf32_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

// Byte offset of fp32 element (row r, column k < 64) in a K-major, 128-byte-swizzled tile whose
// two 32-column atoms are `rows` x 128 bytes each.
__device__ __forceinline__ uint32_t tile_off(int r, int k, int rows) {
    const int atom = k >> 5, kk = k & 31;
    return static_cast<uint32_t>(atom * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 +
                                 ((((kk >> 2) ^ (r & 7)) << 4) | ((kk & 3) << 2)));
}

struct Ctx {
    uint8_t *tile_a, *tile_b;  // 1024-byte aligned shared memory
    uint64_t *bar;             // mbarrier, count 1
    uint32_t tmem;             // 128 TMEM columns
    uint32_t phase;            // parity of the next completion
    uint32_t *status;          // device status word (a wait that gave up sets the timeout bit)
    uint32_t timeout_bit;
};

// Stages rows [0, R) x columns [k0, k0 + 64) of X into `tile` as a K-major tile of `rows` rows:
// element (r, k) = X[r * ldr + k * ldk] (ldk == 1: row-major source, read 16 bytes at a time;
// ldr == 1: column-major source).  Every thread issues all of its loads before its first store,
// so a tile costs one memory latency rather than one per loop trip.
template <int R, int kThreads>
__device__ __forceinline__ void stage(uint8_t *tile, int rows, const float *X, int ldr, int ldk, int k0) {
    constexpr int kVec = R * (kKPass / 4);  // float4 loads per tile
    constexpr int kIt = (kVec + kThreads - 1) / kThreads;
    const int tid = threadIdx.x;
    float4 v[kIt];
    if (ldk == 1) {
#pragma unroll
        for (int it = 0; it < kIt; ++it) {
            const int e = tid + it * kThreads;
            if (kVec % kThreads == 0 || e < kVec) {
                const int r = e / (kKPass / 4), k4 = (e % (kKPass / 4)) * 4;
                v[it] = __ldcg(reinterpret_cast<const float4 *>(X + static_cast<int64_t>(r) * ldr + k0 + k4));
            }
        }
#pragma unroll
        for (int it = 0; it < kIt; ++it) {
            const int e = tid + it * kThreads;
            if (kVec % kThreads == 0 || e < kVec) {
                const int r = e / (kKPass / 4), k4 = (e % (kKPass / 4)) * 4;
                *reinterpret_cast<float4 *>(tile + tile_off(r, k4, rows)) = v[it];
            }
        }
    } else {
#pragma unroll
        for (int it = 0; it < kIt; ++it) {
            const int e = tid + it * kThreads;
            if (kVec % kThreads == 0 || e < kVec) {
                const int k = e / (R / 4), r4 = (e % (R / 4)) * 4;
                v[it] = __ldcg(reinterpret_cast<const float4 *>(X + static_cast<int64_t>(k0 + k) * ldk + r4));
            }
        }
#pragma unroll
        for (int it = 0; it < kIt; ++it) {
            const int e = tid + it * kThreads;
            if (kVec % kThreads == 0 || e < kVec) {
                const int k = e / (R / 4), r4 = (e % (R / 4)) * 4;
                *reinterpret_cast<float *>(tile + tile_off(r4 + 0, k, rows)) = v[it].x;
                *reinterpret_cast<float *>(tile + tile_off(r4 + 1, k, rows)) = v[it].y;
                *reinterpret_cast<float *>(tile + tile_off(r4 + 2, k, rows)) = v[it].z;
                *reinterpret_cast<float *>(tile + tile_off(r4 + 3, k, rows)) = v[it].w;
            }
        }
    }
}

// The product described at the top of this file.  Every thread of the CTA calls it (kThreads of
// them, a multiple of 128); it ends with a barrier, so C is visible to the whole CTA.  A, B and C
// are 16-byte aligned with leading dimensions that are multiples of 4 floats.  Returns
// false when the wait for the tensor cores gave up (the status word records it).
template <int M, int N, int K, bool TA, bool TB, int kThreads>
__device__ bool gemm(Ctx &cx, float *C, int ldc, const float *A, int lda, const float *B, int ldb, float alpha,
                     bool acc, int mask) {
    static_assert(M % 16 == 0 && M <= 128 && N % 16 == 0 && N >= 16 && N <= 128, "shape");
    static_assert(K % kKPass == 0, "K");
    static_assert(kThreads % 128 == 0, "threads");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    bool ok = true;
    for (int k0 = 0; k0 < K; k0 += kKPass) {
        // op(A)[m][k] = TA ? A[k][m] : A[m][k];  op(B)[k][n] = TB ? B[n][k] : B[k][n]
        stage<M, kThreads>(cx.tile_a, 128, A, TA ? 1 : lda, TA ? lda : 1, k0);
        stage<N, kThreads>(cx.tile_b, N, B, TB ? ldb : 1, TB ? 1 : ldb, k0);
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t a = smem_u32(cx.tile_a), b = smem_u32(cx.tile_b);
#pragma unroll
            for (int ks = 0; ks < kKPass / 8; ++ks) {
                const int atom = ks >> 2, kin = ks & 3;
                const uint64_t da = sdesc_sw128(a + atom * 128 * 128, 16, 1024) + ((kin * 32) >> 4);
                const uint64_t db = sdesc_sw128(b + atom * N * 128, 16, 1024) + ((kin * 32) >> 4);
                mma_tf32_ss(cx.tmem, da, db, idesc_tf32(N), (k0 > 0 || ks > 0) ? 1u : 0u);
            }
            mma_commit(cx.bar);
        }
        const bool done = mbar_wait(cx.bar, cx.phase, globaltimer_ns() + 1000000000ull);
        cx.phase ^= 1u;
        if (!done) {
            ok = false;
            if (tid == 0) atomicOr(cx.status, cx.timeout_bit);
        }
        tc_fence_after();
    }
    // read back: warp w covers TMEM lanes 32 (w % 4) .. + 31 (rows) and one part of the columns,
    // 32 columns per round (two TMEM loads, one wait, the old values loaded together)
    constexpr int kGroups = kThreads / 128, kCols = N / kGroups;
    static_assert(kCols % 16 == 0, "columns per warp group");
    const int m = (warp & 3) * 32 + lane, c0 = (warp >> 2) * kCols;
    if (ok && (warp & 3) * 32 < M) {
#pragma unroll
        for (int cc = c0; cc < c0 + kCols; cc += 32) {
            constexpr int kW = kCols >= 32 ? 32 : kCols;
            uint32_t v[kW / 16][16];
            const uint32_t taddr = cx.tmem + ((static_cast<uint32_t>((warp & 3) * 32)) << 16) + cc;
#pragma unroll
            for (int q = 0; q < kW / 16; ++q) tmem_ld16(taddr + 16 * q, v[q]);
            tmem_ld_wait();
            if (m < M) {
                float *o = C + static_cast<int64_t>(m) * ldc + cc;
                float d[kW];
#pragma unroll
                for (int e = 0; e < kW; ++e) {
                    const int n = cc + e;
                    const bool keep = mask == 0 || (mask == 1 ? m >= n : mask == 2 ? m > n : (m < 64 || m - 64 >= n));
                    d[e] = keep ? alpha * __uint_as_float(v[e >> 4][e & 15]) : 0.f;
                }
                if (acc) {
                    float old[kW];
#pragma unroll
                    for (int e = 0; e < kW; e += 4) *reinterpret_cast<float4 *>(old + e) = __ldcg(reinterpret_cast<const float4 *>(o + e));
#pragma unroll
                    for (int e = 0; e < kW; ++e) d[e] += old[e];
                }
#pragma unroll
                for (int e = 0; e < kW; e += 4) *reinterpret_cast<float4 *>(o + e) = *reinterpret_cast<const float4 *>(d + e);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    return ok;
}

}  // namespace tcg
}  // namespace kda
