// State-pool operations for rollout caching: fork (slot to slot), offload (slots to
// pinned host memory) and restore (pinned host memory to slots).
//
// RL rollouts branch many trajectories from shared prompts, and each branch needs
// its own copy of the prompt's recurrent state; states of inactive trajectories
// are kept in host memory and brought back when they resume ("Kimi K3 on
// Fireworks: Fast RL at frontier scale": the rollout paragraph on KV / KDA caches
// that stay consistent as trajectories branch, and the serverless-training
// paragraph on moving reusable KV and KDA states to host memory and loading
// inactive snapshots asynchronously).
//
// All three are one kernel: copy n whole per-slot states (H x dk x dv fp32 each)
// from (src, src_slot[i]) to (dst, dst_slot[i]), with a NULL slot array meaning
// index i.  The host buffer of offload / restore is written or read by the kernel
// itself through its device mapping, so no staging copy is made.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kPoolThreads = 256;
constexpr int kPoolUnroll = 4;  // float4 loads in flight per thread before its stores

// Grid: n items x blocks_per_item.  Each CTA copies its share of one item.
__global__ void __launch_bounds__(kPoolThreads) copy_slots_kernel(const float *src, const int32_t *src_slots,
                                                                  int64_t src_num, float *dst,
                                                                  const int32_t *dst_slots, int64_t dst_num,
                                                                  int64_t per_slot, int blocks_per_item,
                                                                  uint32_t *status) {
    const int64_t item = blockIdx.x / blocks_per_item;
    const int part = static_cast<int>(blockIdx.x % blocks_per_item);
    const int64_t s = src_slots ? static_cast<int64_t>(src_slots[item]) : item;
    const int64_t d = dst_slots ? static_cast<int64_t>(dst_slots[item]) : item;
    if (s < 0 || s >= src_num || d < 0 || d >= dst_num) {
        if (threadIdx.x == 0 && part == 0) atomicOr(status, DEV_ERR_SLOT);
        return;
    }
    const float4 *from = reinterpret_cast<const float4 *>(src + s * per_slot);
    float4 *to = reinterpret_cast<float4 *>(dst + d * per_slot);
    const int64_t n4 = per_slot / 4;
    const int64_t stride = static_cast<int64_t>(blocks_per_item) * kPoolThreads * kPoolUnroll;
    for (int64_t base = (static_cast<int64_t>(part) * kPoolThreads * kPoolUnroll) + threadIdx.x; base < n4;
         base += stride) {
        float4 v[kPoolUnroll];
#pragma unroll
        for (int u = 0; u < kPoolUnroll; ++u) {
            const int64_t i = base + static_cast<int64_t>(u) * kPoolThreads;
            if (i < n4) v[u] = from[i];
        }
#pragma unroll
        for (int u = 0; u < kPoolUnroll; ++u) {
            const int64_t i = base + static_cast<int64_t>(u) * kPoolThreads;
            if (i < n4) to[i] = v[u];
        }
    }
}

bool dim_ok(int d) { return d == 64 || d == 128; }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kda_status launch_copy(const float *src, const int32_t *src_slots, int64_t src_num, float *dst,
                       const int32_t *dst_slots, int64_t dst_num, int n, int64_t per_slot, void *workspace,
                       cudaStream_t s) {
    if (cudaMemsetAsync(workspace, 0, sizeof(uint32_t), s) != cudaSuccess) return KDA_ERR_CUDA;
    if (n == 0) return KDA_OK;
    // about four CTAs per item for large states, at least one
    const int64_t per_cta = static_cast<int64_t>(kPoolThreads) * kPoolUnroll * 4;
    int bpi = static_cast<int>((per_slot + per_cta * 4 - 1) / (per_cta * 4));
    if (bpi < 1) bpi = 1;
    if (bpi > 64) bpi = 64;
    const int64_t grid = static_cast<int64_t>(n) * bpi;
    if (grid > 0x7fffffffLL) return KDA_ERR_INVALID_ARGUMENT;
    copy_slots_kernel<<<static_cast<unsigned>(grid), kPoolThreads, 0, s>>>(
        src, src_slots, src_num, dst, dst_slots, dst_num, per_slot, bpi, static_cast<uint32_t *>(workspace));
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

// Device address of page-locked, device-mapped host memory (NULL if it is not).
const void *mapped_host(const void *host) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, host) != cudaSuccess) {
        cudaGetLastError();  // clear the error state of an unregistered pointer
        return nullptr;
    }
    if (a.type != cudaMemoryTypeHost || !a.devicePointer) return nullptr;
    return a.devicePointer;
}

kda_status check_common(int64_t num_slots, int n, int H, int dk, int dv, void *workspace, size_t ws_bytes) {
    if (!dim_ok(dk) || !dim_ok(dv)) return KDA_ERR_UNSUPPORTED;
    if (num_slots < 0 || n < 0 || H <= 0) return KDA_ERR_INVALID_ARGUMENT;
    if (!workspace || !aligned16(workspace) || ws_bytes < KDA_WS_HEADER_BYTES) return KDA_ERR_WORKSPACE;
    return KDA_OK;
}

}  // namespace
}  // namespace kda

extern "C" {

kda_status kda_state_fork(float *state_pool, int64_t num_slots, const int32_t *src_slots, const int32_t *dst_slots,
                          int n, int H, int dk, int dv, void *workspace, size_t ws_bytes, void *stream) {
    kda_status st = kda::check_common(num_slots, n, H, dk, dv, workspace, ws_bytes);
    if (st != KDA_OK) return st;
    if (n > 0 && (!state_pool || !src_slots || !dst_slots || !kda::aligned16(state_pool)))
        return KDA_ERR_INVALID_ARGUMENT;
    const int64_t per_slot = static_cast<int64_t>(H) * dk * dv;
    return kda::launch_copy(state_pool, src_slots, num_slots, state_pool, dst_slots, num_slots, n, per_slot, workspace,
                            static_cast<cudaStream_t>(stream));
}

kda_status kda_state_offload(const float *state_pool, int64_t num_slots, const int32_t *slots, int n, int H, int dk,
                             int dv, float *host_states, void *workspace, size_t ws_bytes, void *stream) {
    kda_status st = kda::check_common(num_slots, n, H, dk, dv, workspace, ws_bytes);
    if (st != KDA_OK) return st;
    if (n == 0) return kda::launch_copy(nullptr, nullptr, 0, nullptr, nullptr, 0, 0, 0, workspace,
                                        static_cast<cudaStream_t>(stream));
    if (!state_pool || !host_states || !kda::aligned16(state_pool) || !kda::aligned16(host_states))
        return KDA_ERR_INVALID_ARGUMENT;
    float *dst = static_cast<float *>(const_cast<void *>(kda::mapped_host(host_states)));
    if (!dst) return KDA_ERR_INVALID_ARGUMENT;  // not page-locked / mapped host memory
    const int64_t per_slot = static_cast<int64_t>(H) * dk * dv;
    return kda::launch_copy(state_pool, slots, num_slots, dst, nullptr, n, n, per_slot, workspace,
                            static_cast<cudaStream_t>(stream));
}

kda_status kda_state_restore(float *state_pool, int64_t num_slots, const int32_t *slots, int n, int H, int dk,
                             int dv, const float *host_states, void *workspace, size_t ws_bytes, void *stream) {
    kda_status st = kda::check_common(num_slots, n, H, dk, dv, workspace, ws_bytes);
    if (st != KDA_OK) return st;
    if (n == 0) return kda::launch_copy(nullptr, nullptr, 0, nullptr, nullptr, 0, 0, 0, workspace,
                                        static_cast<cudaStream_t>(stream));
    if (!state_pool || !host_states || !kda::aligned16(state_pool) || !kda::aligned16(host_states))
        return KDA_ERR_INVALID_ARGUMENT;
    const float *src = static_cast<const float *>(kda::mapped_host(host_states));
    if (!src) return KDA_ERR_INVALID_ARGUMENT;
    const int64_t per_slot = static_cast<int64_t>(H) * dk * dv;
    return kda::launch_copy(src, nullptr, n, state_pool, slots, num_slots, n, per_slot, workspace,
                            static_cast<cudaStream_t>(stream));
}

}  // extern "C"
