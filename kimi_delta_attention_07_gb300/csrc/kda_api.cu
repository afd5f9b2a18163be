// C ABI of libkda: argument validation and kernel sequencing.
#include <string.h>

#include "kda_internal.cuh"

using namespace kda;

namespace {

inline bool valid_dtype(int dt) { return dt == KDA_F32 || dt == KDA_BF16; }

inline size_t elem_bytes(int dt) { return dt == KDA_BF16 ? 2 : 4; }

inline bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

// The chunk path a call takes: the tensor-core path for bf16 inputs unless
// the precise path is requested.
inline bool use_tensor_cores(int dtype, int flags) {
    return dtype == KDA_BF16 && !(flags & KDA_CHUNK_PRECISE);
}

inline size_t record_bytes(int dtype, int flags) {
    return use_tensor_cores(dtype, flags) ? (size_t)TcRec::bytes : F32Rec::bytes;
}

}  // namespace

extern "C" {

const char *kda_status_string(int status) {
    switch (status) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG: invalid argument";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED: only K = V = 128 is built";
        case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE: workspace missing, too small or misaligned";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA: a CUDA call or kernel launch failed";
        case KDA_ERR_DEVICE_TIMEOUT:
            return "KDA_ERR_DEVICE_TIMEOUT: a bounded device-side wait gave up; outputs are incomplete";
        default: return "KDA: unknown status";
    }
}

int kda_status_from_workspace_flags(int flags) {
    if (flags & KDA_WS_TIMEOUT) return KDA_ERR_DEVICE_TIMEOUT;
    if (flags & (KDA_WS_BAD_SEQLENS | KDA_WS_BAD_SLOT)) return KDA_ERR_INVALID_ARG;
    return KDA_OK;
}

int kda_version(void) { return 100; }

size_t kda_chunk_workspace_bytes(int64_t total_tokens, int n_seqs, int H, int K, int V,
                                 int dtype, int flags) {
    if (total_tokens < 0 || n_seqs <= 0 || H <= 0 || K != kHeadDim || V != kHeadDim ||
        !valid_dtype(dtype))
        return 0;
    const WsLayout L = ws_layout(total_tokens, n_seqs, H, record_bytes(dtype, flags));
    // a gated call on the fp32 path also holds the activated g and beta
    if ((flags & KDA_CHUNK_GATED) && !use_tensor_cores(dtype, flags))
        return ws_gate(L, total_tokens, H).total;
    return L.total;
}

}  // extern "C"

namespace {

enum Phase { kIntra = 1, kScan = 2, kBoth = 3 };

// epilogue arguments: out_gate rows as aligned as o's vector loads, weight
// rows 16-byte aligned, a positive finite eps
bool epi_ok(const EpiArgs *epi, int dtype) {
    if (!epi || !epi->out_gate) return true;
    return epi->weight && aligned(epi->weight, 16) &&
           aligned(epi->out_gate, dtype == KDA_BF16 ? 8 : 16) && isfinite(epi->eps) &&
           epi->eps > 0.0f;
}

// gate == nullptr: g and beta are the activated fp32 inputs; otherwise g and
// beta are unused and the model's raw gates (*gate) are activated in-kernel.
int chunk_call(int phase, const void *q, const void *k, const void *v, const float *g,
               const float *beta, const GateArgs *gate, const EpiArgs *epi,
               const float *initial_state,
               float *final_state, const int32_t *state_indices, int64_t n_slots, void *o,
               const int32_t *cu_seqlens, int n_seqs, int64_t total_tokens, int H, int K, int V,
               float scale, int dtype, int flags, void *workspace, size_t workspace_bytes,
               void *stream) {
    if (!valid_dtype(dtype) || n_seqs <= 0 || H <= 0 || K <= 0 || V <= 0 || total_tokens < 0 ||
        total_tokens > INT32_MAX ||
        (flags & ~(KDA_CHUNK_PRECISE | KDA_CHUNK_SCAN_WIDE | KDA_CHUNK_SCAN_SPLIT |
                   KDA_CHUNK_GATED)) ||
        ((flags & KDA_CHUNK_SCAN_WIDE) && (flags & KDA_CHUNK_SCAN_SPLIT)))
        return KDA_ERR_INVALID_ARG;
    flags = gate ? (flags | KDA_CHUNK_GATED) : (flags & ~KDA_CHUNK_GATED);
    if (K != kHeadDim || V != kHeadDim) return KDA_ERR_UNSUPPORTED;
    if (gate) {
        if (!gate->a_log || !gate->dt_bias || !aligned(gate->dt_bias, 16) ||
            (gate->use_lower_bound && !isfinite(gate->lower_bound)))
            return KDA_ERR_INVALID_ARG;
        if (total_tokens > 0 &&
            (!gate->raw_gate || !gate->raw_beta ||
             !aligned(gate->raw_gate, use_tensor_cores(dtype, flags) ? 16 : 4 * elem_bytes(dtype)) ||
             !aligned(gate->raw_beta, elem_bytes(dtype))))
            return KDA_ERR_INVALID_ARG;
        g = nullptr;
        beta = nullptr;
    } else if (total_tokens > 0 && (!g || !beta)) {
        return KDA_ERR_INVALID_ARG;
    }
    if (total_tokens > 0 && (!q || !k || !v || !o)) return KDA_ERR_INVALID_ARG;
    if (!epi_ok(epi, dtype)) return KDA_ERR_INVALID_ARG;
    if (!cu_seqlens && total_tokens % n_seqs != 0) return KDA_ERR_INVALID_ARG;
    if (state_indices && n_slots <= 0) return KDA_ERR_INVALID_ARG;
    if (!state_indices && n_slots < 0) return KDA_ERR_INVALID_ARG;
    // vector loads need 16-byte (fp32) / 8-byte (bf16) aligned rows; the
    // tensor-core path moves rows with 16-byte bulk copies and vector stores
    const size_t ea = use_tensor_cores(dtype, flags) ? 16 : 4 * elem_bytes(dtype);
    if ((q && !aligned(q, ea)) || (k && !aligned(k, ea)) || (v && !aligned(v, ea)) ||
        (o && !aligned(o, ea)) || (g && !aligned(g, 16)) || (beta && !aligned(beta, 4)) ||
        (initial_state && !aligned(initial_state, 16)) || (final_state && !aligned(final_state, 16)))
        return KDA_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256)) return KDA_ERR_WORKSPACE;
    const size_t need = kda_chunk_workspace_bytes(total_tokens, n_seqs, H, K, V, dtype, flags);
    if (workspace_bytes < need) return KDA_ERR_WORKSPACE;
    if (!isfinite(scale)) return KDA_ERR_INVALID_ARG;

    cudaStream_t s = (cudaStream_t)stream;
    cudaGetLastError();  // clear a stale error so the checks below see only ours
    cudaError_t e = cudaSuccess;
    const bool tc = use_tensor_cores(dtype, flags);
    // tensor-core path, whole forward: the split scan goes first and runs
    // alongside the prep, record by record (scan_ctas of its CTAs; 0 = it runs
    // after the prep)
    int scan_ctas = 0;
    if (phase & kIntra) {
        e = launch_chunk_index(cu_seqlens, n_seqs, total_tokens, H, state_indices, n_slots,
                               workspace, s);
        if (e == cudaSuccess && tc && (phase & kScan))
            scan_ctas = launch_chunk_scan_tc_ahead(initial_state, final_state, state_indices, o, n_seqs,
                                                   total_tokens, H, flags, epi, workspace, s, &e);
        if (e == cudaSuccess && gate && !tc) {  // fp32 path: activate into the workspace
            const WsGate W = ws_gate(ws_layout(total_tokens, n_seqs, H, record_bytes(dtype, flags)),
                                     total_tokens, H);
            float *g_act = ws_at<float>(workspace, W.g_off);
            float *beta_act = ws_at<float>(workspace, W.beta_off);
            e = launch_gate_activation(*gate, dtype, total_tokens, H, g_act, beta_act, s);
            g = g_act;
            beta = beta_act;
        }
        if (e == cudaSuccess)
            e = tc ? launch_chunk_prep_tc(q, k, v, g, beta, gate, n_seqs, total_tokens, H, scale,
                                          scan_ctas, workspace, s)
                   : launch_chunk_prep_f32(q, k, v, g, beta, dtype, n_seqs, total_tokens, H,
                                           scale, workspace, s);
    }
    bool epi_applied = false;
    if (e == cudaSuccess && (phase & kScan) && !scan_ctas)
        e = tc ? launch_chunk_scan_tc(initial_state, final_state, state_indices, o, n_seqs,
                                      total_tokens, H, flags, epi, &epi_applied, workspace, s)
               : launch_chunk_scan_f32(initial_state, final_state, state_indices, o, dtype,
                                       n_seqs, total_tokens, H, workspace, s);
    if (e == cudaSuccess && (phase & kScan) && epi && epi->out_gate && !epi_applied)
        e = launch_output_gate_norm(o, *epi, total_tokens * H, dtype, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

}  // namespace

extern "C" {

#define KDA_CHUNK_ARGS                                                                        \
    const void *q, const void *k, const void *v, const float *g, const float *beta,           \
        const float *initial_state, float *final_state, const int32_t *state_indices,          \
        int64_t n_slots, void *o, const int32_t *cu_seqlens, int n_seqs, int64_t total_tokens, \
        int H, int K, int V, float scale, int dtype, int flags, void *workspace,               \
        size_t workspace_bytes, void *stream
#define KDA_CHUNK_PASS                                                                       \
    q, k, v, g, beta, nullptr, nullptr, initial_state, final_state, state_indices, n_slots, o,\
        cu_seqlens,                                                                           \
        n_seqs, total_tokens, H, K, V, scale, dtype, flags, workspace, workspace_bytes, stream

int kda_chunk_fwd(KDA_CHUNK_ARGS) { return chunk_call(kBoth, KDA_CHUNK_PASS); }
int kda_chunk_intra(KDA_CHUNK_ARGS) { return chunk_call(kIntra, KDA_CHUNK_PASS); }
int kda_chunk_scan(KDA_CHUNK_ARGS) { return chunk_call(kScan, KDA_CHUNK_PASS); }

int kda_chunk_fwd_gated(const void *q, const void *k, const void *v, const void *raw_gate,
                        const void *raw_beta, const float *a_log, const float *dt_bias,
                        float lower_bound, int use_lower_bound, const void *out_gate,
                        const float *norm_weight, float norm_eps, const float *initial_state,
                        float *final_state, const int32_t *state_indices, int64_t n_slots,
                        void *o, const int32_t *cu_seqlens, int n_seqs, int64_t total_tokens,
                        int H, int K, int V, float scale, int dtype, int flags, void *workspace,
                        size_t workspace_bytes, void *stream) {
    const GateArgs gate{raw_gate, raw_beta, a_log, dt_bias, lower_bound, use_lower_bound != 0};
    const EpiArgs epi{out_gate, norm_weight, norm_eps};
    return chunk_call(kBoth, q, k, v, nullptr, nullptr, &gate, &epi, initial_state, final_state,
                      state_indices, n_slots, o, cu_seqlens, n_seqs, total_tokens, H, K, V, scale,
                      dtype, flags, workspace, workspace_bytes, stream);
}

int kda_workspace_status(const void *workspace, int *flags_out, void *stream) {
    if (!workspace || !flags_out) return KDA_ERR_INVALID_ARG;
    int32_t st = 0;
    cudaError_t e = cudaMemcpyAsync(&st, workspace, sizeof(st), cudaMemcpyDeviceToHost,
                                    (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return KDA_ERR_CUDA;
    }
    *flags_out = st;
    return kda_status_from_workspace_flags(st);
}

namespace {
int step_call(const void *q, const void *k, const void *v, const float *g, const float *beta,
              const GateArgs *gate, const EpiArgs *epi, float *state_pool,
              const int32_t *state_indices, const int32_t *num_accepted, int S,
              int64_t n_slots, void *o, int N, int H, int K, int V, float scale, int dtype,
              void *stream) {
    if (!valid_dtype(dtype) || N < 0 || S < 1 || H <= 0 || K <= 0 || V <= 0 || n_slots < 0)
        return KDA_ERR_INVALID_ARG;
    if (K != kHeadDim || V != kHeadDim) return KDA_ERR_UNSUPPORTED;
    if (N == 0) return KDA_OK;
    if (S > 1 && !state_indices) return KDA_ERR_INVALID_ARG;  // per-token slots are required
    if ((int64_t)N * S * H > INT32_MAX) return KDA_ERR_INVALID_ARG;
    if (gate) {
        if (!gate->raw_gate || !gate->raw_beta || !gate->a_log || !gate->dt_bias ||
            !aligned(gate->raw_gate, 4 * elem_bytes(dtype)) ||
            !aligned(gate->raw_beta, elem_bytes(dtype)) || !aligned(gate->dt_bias, 16) ||
            (gate->use_lower_bound && !isfinite(gate->lower_bound)))
            return KDA_ERR_INVALID_ARG;
        g = nullptr;
        beta = nullptr;
    } else if (!g || !beta || !aligned(g, 16) || !aligned(beta, 4)) {
        return KDA_ERR_INVALID_ARG;
    }
    if (!q || !k || !v || !state_pool || !o) return KDA_ERR_INVALID_ARG;
    if (!epi_ok(epi, dtype)) return KDA_ERR_INVALID_ARG;
    if (!state_indices && n_slots < N) return KDA_ERR_INVALID_ARG;
    if ((int64_t)N * H > INT32_MAX) return KDA_ERR_INVALID_ARG;
    const size_t ea = 4 * elem_bytes(dtype);
    if (!aligned(q, ea) || !aligned(k, ea) || !aligned(v, ea) || !aligned(o, elem_bytes(dtype)) ||
        !aligned(state_pool, 16))
        return KDA_ERR_INVALID_ARG;
    if (!isfinite(scale)) return KDA_ERR_INVALID_ARG;
    cudaGetLastError();
    const cudaError_t e = launch_recurrent_step(q, k, v, g, beta, gate, epi, state_pool,
                                                state_indices, num_accepted, n_slots, o, N, S, H,
                                                scale, dtype, (cudaStream_t)stream);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return KDA_ERR_CUDA;
    }
    return KDA_OK;
}
}  // namespace

int kda_recurrent_step(const void *q, const void *k, const void *v, const float *g,
                       const float *beta, float *state_pool, const int32_t *state_indices,
                       int64_t n_slots, void *o, int N, int H, int K, int V, float scale,
                       int dtype, void *stream) {
    return step_call(q, k, v, g, beta, nullptr, nullptr, state_pool, state_indices, nullptr, 1,
                     n_slots, o, N, H, K, V, scale, dtype, stream);
}

int kda_recurrent_multi_step(const void *q, const void *k, const void *v, const float *g,
                             const float *beta, float *state_pool, const int32_t *state_indices,
                             const int32_t *num_accepted, int64_t n_slots, void *o, int N, int S,
                             int H, int K, int V, float scale, int dtype, void *stream) {
    return step_call(q, k, v, g, beta, nullptr, nullptr, state_pool, state_indices, num_accepted,
                     S, n_slots, o, N, H, K, V, scale, dtype, stream);
}

int kda_recurrent_step_gated(const void *q, const void *k, const void *v, const void *raw_gate,
                             const void *raw_beta, const float *a_log, const float *dt_bias,
                             float lower_bound, int use_lower_bound, const void *out_gate,
                             const float *norm_weight, float norm_eps, float *state_pool,
                             const int32_t *state_indices, int64_t n_slots, void *o, int N,
                             int H, int K, int V, float scale, int dtype, void *stream) {
    const GateArgs gate{raw_gate, raw_beta, a_log, dt_bias, lower_bound, use_lower_bound != 0};
    const EpiArgs epi{out_gate, norm_weight, norm_eps};
    return step_call(q, k, v, nullptr, nullptr, &gate, &epi, state_pool, state_indices, nullptr, 1,
                     n_slots, o, N, H, K, V, scale, dtype, stream);
}

int kda_recurrent_multi_step_gated(const void *q, const void *k, const void *v,
                                   const void *raw_gate, const void *raw_beta, const float *a_log,
                                   const float *dt_bias, float lower_bound, int use_lower_bound,
                                   const void *out_gate, const float *norm_weight, float norm_eps,
                                   float *state_pool, const int32_t *state_indices,
                                   const int32_t *num_accepted, int64_t n_slots, void *o, int N,
                                   int S, int H, int K, int V, float scale, int dtype, void *stream) {
    const GateArgs gate{raw_gate, raw_beta, a_log, dt_bias, lower_bound, use_lower_bound != 0};
    const EpiArgs epi{out_gate, norm_weight, norm_eps};
    return step_call(q, k, v, nullptr, nullptr, &gate, &epi, state_pool, state_indices, num_accepted,
                     S, n_slots, o, N, H, K, V, scale, dtype, stream);
}

int kda_short_conv_fwd(const void *x, const void *weight, void *y, const int32_t *cu_seqlens,
                       int n_seqs, int64_t total_tokens, int D, int ks, int activation,
                       const void *initial_states, void *final_states,
                       const int32_t *state_indices, int64_t n_slots, int dtype, void *stream) {
    if (!valid_dtype(dtype) || n_seqs <= 0 || total_tokens < 0 || D <= 0 || D % 8 != 0 ||
        ks < 2 || ks > 8 || (activation != KDA_CONV_NONE && activation != KDA_CONV_SILU))
        return KDA_ERR_INVALID_ARG;
    if (!cu_seqlens && total_tokens % n_seqs != 0) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!x || !weight || !y)) return KDA_ERR_INVALID_ARG;
    if (state_indices ? n_slots <= 0 : n_slots < 0) return KDA_ERR_INVALID_ARG;
    const int64_t slots = state_indices ? n_slots : n_seqs;
    const size_t ea = 8 * elem_bytes(dtype) >= 16 ? 16 : 8 * elem_bytes(dtype);
    if ((x && !aligned(x, ea)) || (weight && !aligned(weight, ea)) || (y && !aligned(y, ea)) ||
        (initial_states && !aligned(initial_states, ea)) || (final_states && !aligned(final_states, ea)))
        return KDA_ERR_INVALID_ARG;
    cudaGetLastError();
    const cudaError_t e = launch_short_conv_prefill(x, weight, y, cu_seqlens, n_seqs, total_tokens,
                                                    D, ks, activation, initial_states, final_states,
                                                    state_indices, slots, dtype,
                                                    (cudaStream_t)stream);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

int kda_short_conv_update(const void *x, const void *weight, void *y, void *state_pool,
                          const int32_t *state_indices, int64_t n_slots, int N, int D, int ks,
                          int activation, int dtype, void *stream) {
    if (!valid_dtype(dtype) || N < 0 || D <= 0 || D % 8 != 0 || ks < 2 || ks > 8 ||
        n_slots < 0 || (activation != KDA_CONV_NONE && activation != KDA_CONV_SILU))
        return KDA_ERR_INVALID_ARG;
    if (N == 0) return KDA_OK;
    if (!x || !weight || !y || !state_pool) return KDA_ERR_INVALID_ARG;
    if (!state_indices && n_slots < N) return KDA_ERR_INVALID_ARG;
    const size_t ea = 8 * elem_bytes(dtype) >= 16 ? 16 : 8 * elem_bytes(dtype);
    if (!aligned(x, ea) || !aligned(weight, ea) || !aligned(y, ea) || !aligned(state_pool, ea))
        return KDA_ERR_INVALID_ARG;
    cudaGetLastError();
    const cudaError_t e = launch_short_conv_update(x, weight, y, state_pool, state_indices, n_slots,
                                                   N, D, ks, activation, dtype,
                                                   (cudaStream_t)stream);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

int kda_short_conv_multi_update(const void *x, const void *weight, void *y, void *state_pool,
                                const int32_t *state_indices, const int32_t *num_accepted,
                                int64_t n_slots, int N, int S, int D, int ks, int activation,
                                int dtype, void *stream) {
    if (!valid_dtype(dtype) || N < 0 || S < 1 || D <= 0 || D % 8 != 0 || ks < 2 || ks > 8 ||
        n_slots <= 0 || (activation != KDA_CONV_NONE && activation != KDA_CONV_SILU))
        return KDA_ERR_INVALID_ARG;
    if (N == 0) return KDA_OK;
    if (!x || !weight || !y || !state_pool || !state_indices) return KDA_ERR_INVALID_ARG;
    const size_t ea = 8 * elem_bytes(dtype) >= 16 ? 16 : 8 * elem_bytes(dtype);
    if (!aligned(x, ea) || !aligned(weight, ea) || !aligned(y, ea) || !aligned(state_pool, ea))
        return KDA_ERR_INVALID_ARG;
    cudaGetLastError();
    const cudaError_t e = launch_short_conv_multi_update(x, weight, y, state_pool, state_indices,
                                                         num_accepted, n_slots, N, S, D, ks,
                                                         activation, dtype, (cudaStream_t)stream);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

int kda_output_gate_norm(void *o, const void *gate, const float *weight, float eps,
                         int64_t rows, int V, int dtype, void *stream) {
    if (!valid_dtype(dtype) || rows < 0 || V <= 0) return KDA_ERR_INVALID_ARG;
    if (V != kHeadDim) return KDA_ERR_UNSUPPORTED;
    if (rows == 0) return KDA_OK;
    const EpiArgs epi{gate, weight, eps};
    if (!o || !gate || !aligned(o, dtype == KDA_BF16 ? 8 : 16) || !epi_ok(&epi, dtype))
        return KDA_ERR_INVALID_ARG;
    cudaGetLastError();
    const cudaError_t e = launch_output_gate_norm(o, epi, rows, dtype, (cudaStream_t)stream);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

}  // extern "C"
