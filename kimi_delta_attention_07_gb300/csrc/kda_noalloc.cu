// kda_chunk_fwd_noalloc: the chunked forward without a caller-provided
// workspace, for callers that cannot allocate device memory.
//
// Some hosts hand a kernel library nothing but its input and output buffers:
// plugin interfaces of inference servers that own every byte of device memory
// through their own pool, or code on a latency-critical path where a
// cudaMalloc (which can synchronise the whole device) is not allowed.  This
// entry point serves them from a fixed scratch array that is part of the
// library image itself, so nothing is allocated at call time.
//
// The scratch array is a file-scope __device__ variable: every GPU on which
// the library's device code is loaded holds it (KDA_NOALLOC_WORKSPACE_BYTES)
// until the process exits.  Host code cannot use the array's name as a
// device address, so its address is looked up once per device with
// cudaGetSymbolAddress, on the first call made with that device current.
#include <mutex>

#include "kda_internal.cuh"

namespace {

constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_ws[KDA_NOALLOC_WORKSPACE_BYTES];

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once per device).
int noalloc_workspace(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return KDA_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_ws) != cudaSuccess || !p) {
            cudaGetLastError();
            return KDA_ERR_CUDA;
        }
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return KDA_OK;
}

}  // namespace

extern "C" int kda_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const float *g,
                                     const float *beta, const float *initial_state,
                                     float *final_state, const int32_t *state_indices,
                                     int64_t n_slots, void *o, const int32_t *cu_seqlens,
                                     int n_seqs, int64_t total_tokens, int H, int K, int V,
                                     float scale, int dtype, int flags, void *stream) {
    // Sizes that are invalid for kda_chunk_fwd (need == 0) fall through to its
    // own validation; valid sizes beyond the fixed array are refused here.
    const size_t need = kda_chunk_workspace_bytes(total_tokens, n_seqs, H, K, V, dtype, flags);
    if (need > (size_t)KDA_NOALLOC_WORKSPACE_BYTES) return KDA_ERR_WORKSPACE;
    void *ws = nullptr;
    const int st = noalloc_workspace(&ws);
    if (st != KDA_OK) return st;
    // Every byte of the workspace that the kernels read is written earlier in
    // the same call (index, then per-chunk records), so the previous call's
    // contents need no clearing.
    return kda_chunk_fwd(q, k, v, g, beta, initial_state, final_state, state_indices, n_slots, o,
                         cu_seqlens, n_seqs, total_tokens, H, K, V, scale, dtype, flags, ws,
                         (size_t)KDA_NOALLOC_WORKSPACE_BYTES, stream);
}
