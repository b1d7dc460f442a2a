// kda_chunk_fwd_noalloc: kda_chunk_fwd for callers that cannot allocate device memory.
//
// kda_chunk_fwd needs a workspace: a status word, and (when final_state is NULL)
// a staging copy of the states that the chunked kernel hands to the
// partial-chunk kernel.  Some callers have no way to provide one -- a host
// framework that plans every device byte up front and gives plug-in kernels no
// workspace hook, or a latency-critical loop where a cudaMalloc (which can
// synchronize the whole device) is not allowed.  This entry point uses a
// fixed-size scratch array that lives in the library's own device memory
// instead, and calls no allocator at all.
//
// The array is a file-scope __device__ variable, so every GPU that loads this
// library keeps it (kStaticWorkspaceBytes) until the process exits.  In host
// code its name is only a host-side stand-in; its device address is looked up
// with cudaGetSymbolAddress, with the caller's device current.  The lookup is
// repeated on every call made outside stream capture (it is cheap and
// allocates nothing), so a reset device or another context never sees a stale
// address; during capture the address last looked up on that device is used,
// which is why the first call on a device must come before any capture.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/kda.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = KDA_NOALLOC_WORKSPACE_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

std::mutex g_mutex;
void *g_device_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.
kda_status static_workspace(cudaStream_t stream, void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_UNSUPPORTED;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return KDA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (cap == cudaStreamCaptureStatusNone) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_workspace) != cudaSuccess || !ptr) return KDA_ERR_CUDA;
        g_device_ptr[dev] = ptr;
    }
    if (!g_device_ptr[dev]) return KDA_ERR_CUDA;  // first call on this device made during capture
    *out = g_device_ptr[dev];
    return KDA_OK;
}

}  // namespace

extern "C" kda_status kda_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const void *g,
                                            const void *beta, kda_dtype dtype, const float *init_state,
                                            const int32_t *cu_seqlens, int N, int64_t T_total, int H, int dk,
                                            int dv, float scale, void *o, float *final_state,
                                            const void **status_workspace, void *stream) {
    // Same checks as kda_chunk_fwd, so oversized requests fail before any CUDA call.
    if (!(dtype == KDA_BF16 || dtype == KDA_F32) || !(dk == 64 || dk == 128) || !(dv == 64 || dv == 128))
        return KDA_ERR_UNSUPPORTED;
    if (N < 0 || T_total < 0 || H <= 0) return KDA_ERR_INVALID_ARGUMENT;
    // the minimum workspace (the status header, plus the staging states without final_state);
    // kda_chunk_fwd uses the split path only if the scratch also holds its buffers
    const size_t states = static_cast<size_t>(N) * static_cast<size_t>(H) * dk * dv * sizeof(float);
    const size_t need = KDA_WS_HEADER_BYTES + (final_state ? 0 : states);
    if (need > kStaticWorkspaceBytes) return KDA_ERR_WORKSPACE;
    void *ws = nullptr;
    const kda_status st = static_workspace(static_cast<cudaStream_t>(stream), &ws);
    if (st != KDA_OK) return st;
    if (status_workspace) *status_workspace = ws;
    // kda_chunk_fwd clears the status word first; the staging area is written before it is read.
    return kda_chunk_fwd(q, k, v, g, beta, dtype, init_state, cu_seqlens, N, T_total, H, dk, dv, scale, o,
                         final_state, ws, kStaticWorkspaceBytes, stream);
}
