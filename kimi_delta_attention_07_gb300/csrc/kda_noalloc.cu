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
// device address, so its address is looked up with cudaGetSymbolAddress on
// the first call made with a device current, and again whenever the current
// CUDA context differs from the one the address was taken in (after a
// cudaDeviceReset the device gets a new primary context, and the old address
// would be stale).
#include <cuda.h>  // CUcontext (the query is fetched through the runtime)
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_internal.cuh"

namespace {

constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_ws[KDA_NOALLOC_WORKSPACE_BYTES];

struct NoallocSlot {
    CUcontext ctx;  // the context the address was taken in
    void *ptr;
};
std::mutex g_noalloc_mu;
NoallocSlot g_noalloc[kMaxDevices] = {};

PFN_cuCtxGetCurrent_v4000 ctx_query() {
    static std::once_flag once;
    static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuCtxGetCurrent_v4000)p;
        cudaGetLastError();
    });
    return fn;
}

// Device address of the scratch array in the current device's context.
int noalloc_workspace(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return KDA_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_UNSUPPORTED;
    auto query = ctx_query();
    if (!query) return KDA_ERR_CUDA;
    // A thread on which the runtime has not yet made the device's context
    // current sees no context here; the symbol lookup below makes it current.
    CUcontext ctx = nullptr;
    if (query(&ctx) != CUDA_SUCCESS) return KDA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    NoallocSlot &slot = g_noalloc[dev];
    if (!slot.ptr || !ctx || slot.ctx != ctx) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_ws) != cudaSuccess || !p) {
            cudaGetLastError();
            return KDA_ERR_CUDA;
        }
        if (query(&ctx) != CUDA_SUCCESS || !ctx) return KDA_ERR_CUDA;
        slot.ctx = ctx;
        slot.ptr = p;
    }
    *out = slot.ptr;
    return KDA_OK;
}

}  // namespace

extern "C" int kda_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const float *g,
                                     const float *beta, const float *initial_state,
                                     float *final_state, const int32_t *state_indices,
                                     int64_t n_slots, void *o, const int32_t *cu_seqlens,
                                     int n_seqs, int64_t total_tokens, int H, int K, int V,
                                     float scale, int dtype, int flags, void *stream) {
    // This is the forward from activated g and beta: a gate flag would only
    // size the workspace for the fp32 path's activated-gate copy, which this
    // call never makes, so it is dropped before the size check.
    flags &= ~KDA_CHUNK_GATED;
    // Sizes that are invalid for kda_chunk_fwd (need == 0) fall through to its
    // own validation; valid sizes beyond the fixed array are refused here.
    const size_t need = kda_chunk_workspace_bytes(total_tokens, n_seqs, H, K, V, dtype, flags);
    if (need > (size_t)KDA_NOALLOC_WORKSPACE_BYTES) return KDA_ERR_WORKSPACE;
    void *ws = nullptr;
    const int st = noalloc_workspace(&ws);
    if (st != KDA_OK) return st;
    // Every byte of the workspace that the kernels read is written earlier in
    // the same call (status word and index, then per-chunk records), so the
    // previous call's contents need no clearing.
    return kda_chunk_fwd(q, k, v, g, beta, initial_state, final_state, state_indices, n_slots, o,
                         cu_seqlens, n_seqs, total_tokens, H, K, V, scale, dtype, flags, ws,
                         (size_t)KDA_NOALLOC_WORKSPACE_BYTES, stream);
}
