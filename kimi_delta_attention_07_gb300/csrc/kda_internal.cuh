// Internal helpers and the workspace layout shared by the libkda kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

constexpr int kChunk = KDA_CHUNK;  // 64 tokens per chunk
constexpr int kHeadDim = 128;      // K = V = 128 is what is built

// ---- element access -------------------------------------------------------

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Four consecutive elements starting at p (p 8-byte aligned for bf16,
// 16-byte aligned for fp32).
__device__ __forceinline__ float4 load4(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16 *p) {
    const uint2 raw = *reinterpret_cast<const uint2 *>(p);
    const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162 *>(&raw.x);
    const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162 *>(&raw.y);
    const float2 a = __bfloat1622float2(lo), b = __bfloat1622float2(hi);
    return make_float4(a.x, a.y, b.x, b.y);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// ---- workspace layout -----------------------------------------------------
//
//   [0, 256)      status word (int32, StatusBits), deferred-item count, and the
//                 counters of the tensor-core path (items handed out by the prep,
//                 scan CTAs finished, strong-decay prep CTAs finished, prep CTAs
//                 finished), int32 each
//   [256, ...)    seq_start[N] int32 (-1 = sequence skipped), seq_len[N] int32,
//                 chunk_off[N+1] int32 (exclusive prefix sum of chunks per seq)
//   aligned(16)   deferred (chunk, head) items, int32 [max chunks * H]
//                 (tensor-core path: the items handed to the strong-decay prep)
//   aligned(16)   ready flags, int32 [max chunks * H]: record written (cleared by
//                 the chunk index, raised by the prep that writes the record)
//   aligned(256)  per-(chunk, head) records, index chunk * H + head
//
// The record contents depend on the chunk path (fp32 CUDA-core path or bf16
// tensor-core path); each path defines its record size.

enum StatusBits : int {
    kBadSeqlens = KDA_WS_BAD_SEQLENS,
    kBadSlot = KDA_WS_BAD_SLOT,
    kStatusTimeout = KDA_WS_TIMEOUT,
    kExactDecay = KDA_WS_EXACT_DECAY,
    kStrongDecay = KDA_WS_STRONG_DECAY
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline int64_t max_chunks(int64_t total_tokens, int n_seqs) {
    // Sum over sequences of ceil(len / 64) <= floor(T / 64) + N.
    return total_tokens / kChunk + n_seqs;
}

// Row sums of squares exchanged between the four value-column CTAs of a
// (sequence, head) when the split scan applies the output epilogue itself: a
// ring of kEpiRing chunks x 4 CTAs x 64 rows of tagged 8-byte words per
// (sequence, head), for at most kEpiPairs pairs.
constexpr int kEpiPairs = 64;
constexpr int kEpiRing = 4;

struct WsLayout {
    size_t status_off, defer_count_off, item_ctr_off, scan_done_off, strong_done_off, prep_done_off,
        seq_start_off, seq_len_off, chunk_off_off, seq_order_off, epi_part_off, defer_off,
        ready_off, records_off, record_bytes, total;
};

__host__ __device__ inline WsLayout ws_layout(int64_t total_tokens, int n_seqs, int H,
                                              size_t record_bytes) {
    WsLayout L;
    const size_t arr = align_up(sizeof(int32_t) * (size_t)(n_seqs + 1), 16);
    L.status_off = 0;
    L.defer_count_off = 4;
    L.item_ctr_off = 8;
    L.scan_done_off = 12;
    L.strong_done_off = 16;
    L.prep_done_off = 20;
    L.seq_start_off = 256;
    L.seq_len_off = L.seq_start_off + arr;
    L.chunk_off_off = L.seq_len_off + arr;
    L.seq_order_off = L.chunk_off_off + arr;  // int32 [n_seqs]: sequences by decreasing length
    L.epi_part_off = align_up(L.seq_order_off + arr, 256);  // u64 [kEpiPairs][kEpiRing][4][64]
    L.defer_off = L.epi_part_off + sizeof(uint64_t) * kEpiPairs * kEpiRing * 4 * kChunk;
    const size_t items = (size_t)max_chunks(total_tokens, n_seqs) * (size_t)H;
    L.ready_off = align_up(L.defer_off + sizeof(int32_t) * items, 16);
    L.records_off = align_up(L.ready_off + sizeof(int32_t) * items, 256);
    L.record_bytes = record_bytes;
    L.total = L.records_off + items * record_bytes;
    return L;
}

template <typename P>
__host__ __device__ inline P *ws_at(void *ws, size_t off) {
    return reinterpret_cast<P *>(reinterpret_cast<char *>(ws) + off);
}

// fp32 CUDA-core path: per (chunk, head) record, all fp32
//   W [64][K], U [64][V], QG [64][K], KD [64][K], A [64][64], gC [K]
struct F32Rec {
    static constexpr size_t W = 0;
    static constexpr size_t U = W + kChunk * kHeadDim;
    static constexpr size_t QG = U + kChunk * kHeadDim;
    static constexpr size_t KD = QG + kChunk * kHeadDim;
    static constexpr size_t A = KD + kChunk * kHeadDim;
    static constexpr size_t GC = A + kChunk * kChunk;
    static constexpr size_t floats = GC + kHeadDim;
    static constexpr size_t bytes = floats * sizeof(float);
};

// bf16 tensor-core path: per (chunk, head) record.  WQ | KD | A | gC is the
// scan's shared-memory image of the chunk, in the 128-byte-swizzled K-major
// operand layout; U follows, split in four 32-column blocks so that the scan
// CTA of value block vb copies its 4 KB piece with one bulk copy.
//   WQ  [128 rows][128 K] bf16: rows 0..63 W, rows 64..127 QG        32 KB
//   KD  [64 chunk rows][128 key] bf16, MN-major SW128 (two 64-key
//       blocks of 64 rows x 128 B): the A operand KD^T of the state update 16 KB
//   A   [64][64] bf16: causal scores (directly after KDT)             8 KB
//   gC  [128] fp32: exp(G_last)
//   U   [4 value blocks][64 rows][32] bf16; the four 16-byte chunks   16 KB
//       of row i rotated: chunk c at position c ^ ((i / 2) % 4)
struct TcRec {
    static constexpr uint32_t WQ = 0;
    static constexpr uint32_t KD = 32768;
    static constexpr uint32_t A = KD + 16384;
    static constexpr uint32_t GC = A + 8192;
    static constexpr uint32_t U = GC + 512;
    static constexpr uint32_t UBLK = 64 * 32 * 2;  // one 32-column block of U
    static constexpr uint32_t bytes = 74752;       // U + 16384, rounded up to 1024
};
static_assert(TcRec::U + 4 * TcRec::UBLK <= TcRec::bytes, "TcRec layout");

// Programmatic dependent launch.  A kernel launched with launch_dependent()
// may be scheduled while the previous kernel on its stream is finishing; it
// calls griddep_wait() before its first global-memory access, which returns
// once that kernel has completed and its writes are visible (a no-op for a
// kernel launched normally).  griddep_launch_dependents() lets the next such
// kernel be scheduled before this one exits.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// The same for a grid whose CTAs wait on one another: a cooperative launch,
// which fails rather than start a grid that cannot be resident at once.
// Where programmatic serialization cannot be combined with it, the launch is
// repeated as a plain cooperative one.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent_coop(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                  cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
    if (e != cudaSuccess) {
        cudaGetLastError();
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
    }
    return e;
}

// SM count of the current device (cached per device; host only)
inline int sm_count() {
    static int count[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!count[dev]) {
        int c = 0;
        cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev);
        count[dev] = c > 0 ? c : 148;
    }
    return count[dev];
}

// ---- gate activation (the model's gate, computed in-kernel) ----------------
// x = raw_gate + dt_bias[h][k];  g = lower_bound * sigmoid(exp(a_log[h]) x)
// with a lower bound, else -exp(a_log[h]) softplus(x);  beta = sigmoid(raw_beta).
struct GateArgs {
    const void *raw_gate;  // [T, H, K] in the q dtype
    const void *raw_beta;  // [T, H] in the q dtype
    const float *a_log;    // [H]
    const float *dt_bias;  // [H, K]
    float lower_bound;
    int use_lower_bound;
};

// g from x = raw + bias, with gscale = exp(a_log[h])
__device__ __forceinline__ float gate_decay(float x, float gscale, float lower_bound,
                                            bool use_lower_bound) {
    if (use_lower_bound) return lower_bound / (1.0f + expf(-gscale * x));
    return -gscale * (fmaxf(x, 0.0f) + log1pf(expf(-fabsf(x))));
}
__device__ __forceinline__ float gate_beta(float raw) { return 1.0f / (1.0f + expf(-raw)); }

// Output epilogue: o / sqrt(mean(o^2) + eps) * weight * sigmoid(gate) per row.
struct EpiArgs {
    const void *out_gate;  // [rows, V] in the o dtype; nullptr = no epilogue
    const float *weight;   // [V]
    float eps;
};

// Workspace of a gated call on the fp32 path: activated g [T, H, K] and beta
// [T, H] (fp32) after the records.
struct WsGate {
    size_t g_off, beta_off, total;
};
__host__ __device__ inline WsGate ws_gate(const WsLayout &L, int64_t total_tokens, int H) {
    WsGate W;
    W.g_off = align_up(L.total, 256);
    W.beta_off = align_up(W.g_off + (size_t)total_tokens * H * kHeadDim * sizeof(float), 256);
    W.total = W.beta_off + (size_t)total_tokens * H * sizeof(float);
    return W;
}

// ---- launchers (return cudaGetLastError() of the launch) ------------------

// Also clears the ready flags and the counters of the tensor-core path.
cudaError_t launch_chunk_index(const int32_t *cu_seqlens, int n_seqs, int64_t total_tokens, int H,
                               const int32_t *state_indices, int64_t n_slots, void *workspace,
                               cudaStream_t stream);

cudaError_t launch_chunk_prep_f32(const void *q, const void *k, const void *v, const float *g,
                                  const float *beta, int dtype, int n_seqs, int64_t total_tokens,
                                  int H, float scale, void *workspace, cudaStream_t stream);

cudaError_t launch_chunk_scan_f32(const float *initial_state, float *final_state,
                                  const int32_t *state_indices, void *o, int dtype, int n_seqs,
                                  int64_t total_tokens, int H, void *workspace,
                                  cudaStream_t stream);

// gate == nullptr: g, beta are activated fp32; otherwise g, beta are unused
// and the raw gates of *gate are activated on chip.  scan_ctas > 0: the split
// scan (that many CTAs) was launched just before and runs alongside, waiting
// for each record's ready flag; the prep then does not wait for the kernel
// before it, and the strong-decay prep's last CTA waits for the scan to finish
// (so that whatever follows on the stream sees the scan complete).
cudaError_t launch_chunk_prep_tc(const void *q, const void *k, const void *v, const float *g,
                                 const float *beta, const GateArgs *gate, int n_seqs,
                                 int64_t total_tokens, int H, float scale, int scan_ctas,
                                 void *workspace, cudaStream_t stream);

// The strong-decay prep of the tensor-core path: the (chunk, head) items that
// chunk_prep_tc deferred (listed in the workspace), with per-16-token decay
// references.  Launched right after launch_chunk_prep_tc, same arguments.
// prep_ctas: the grid of the prep before it (with a scan running alongside,
// this grid waits for that many prep CTAs to finish instead of waiting for
// the kernel before it, which would wait for the scan as well).
cudaError_t launch_chunk_prep_tc_strong(const void *q, const void *k, const void *v,
                                        const float *g, const float *beta, const GateArgs *gate,
                                        int n_seqs, int64_t total_tokens, int H, float scale,
                                        int scan_ctas, int prep_ctas, void *workspace,
                                        cudaStream_t stream);

// Load every kernel that a forward with the scan running alongside the prep
// launches, once per device: a kernel loaded lazily while the scan waits for
// the prep could wait for the running scan itself.
void preload_chunk_tc_kernels();
void preload_chunk_tc_strong_kernels();
void preload_chunk_index_kernel();
void preload_output_gate_norm_kernels();

// Activated g and beta of a gated call into fp32 buffers (the fp32 path).
cudaError_t launch_gate_activation(const GateArgs &gate, int dtype, int64_t total_tokens, int H,
                                   float *g_out, float *beta_out, cudaStream_t stream);

// epi (may be nullptr): the output epilogue, applied in the scan where the
// layout allows it (*epi_applied then true; otherwise the caller runs
// launch_output_gate_norm after it).
cudaError_t launch_chunk_scan_tc(const float *initial_state, float *final_state,
                                 const int32_t *state_indices, void *o, int n_seqs,
                                 int64_t total_tokens, int H, int flags, const EpiArgs *epi,
                                 bool *epi_applied, void *workspace, cudaStream_t stream);

// The split scan launched BEFORE the prep, to run alongside it: cooperatively
// (every CTA resident, at most one per SM, leaving room for a prep CTA beside
// each and for the strong-decay prep on the SMs left over).  Returns the
// number of scan CTAs launched, 0 if this layout does not apply (the wide scan
// is wanted, the epilogue would be fused, or the grid does not fit); a launch
// error is returned in *err.
int launch_chunk_scan_tc_ahead(const float *initial_state, float *final_state,
                               const int32_t *state_indices, void *o, int n_seqs,
                               int64_t total_tokens, int H, int flags, const EpiArgs *epi,
                               void *workspace, cudaStream_t stream, cudaError_t *err);

// Block-wide helper used by the chunk kernels: find the sequence that owns
// global chunk `c` (largest n with chunk_off[n] <= c; chunk_off non-decreasing).
__device__ __forceinline__ int owner_of_chunk(const int32_t *chunk_off, int n_seqs, int c) {
    int lo = 0, hi = n_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (chunk_off[mid] <= c) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// gate == nullptr: g, beta are activated fp32; otherwise raw gates (*gate).
// epi == nullptr (or epi->out_gate == nullptr): plain o; otherwise the output
// epilogue is applied in the step.
// S tokens per sequence (q/k/g/v/o [N, S, H, *], beta [N, S, H]); the state
// after token t goes to slot state_indices[n S + t], the initial state comes
// from slot state_indices[n S + num_accepted[n] - 1] (num_accepted == nullptr:
// token 0's slot; state_indices == nullptr with S == 1: slot n).
// Short causal convolution (x, weight, y, states all in `dtype`).
cudaError_t launch_short_conv_prefill(const void *x, const void *weight, void *y,
                                      const int32_t *cu_seqlens, int n_seqs, int64_t total_tokens,
                                      int D, int ks, int activation, const void *initial_states,
                                      void *final_states, const int32_t *state_indices,
                                      int64_t n_slots, int dtype, cudaStream_t stream);
cudaError_t launch_short_conv_update(const void *x, const void *weight, void *y, void *pool,
                                     const int32_t *state_indices, int64_t n_slots, int N, int D,
                                     int ks, int activation, int dtype, cudaStream_t stream);
cudaError_t launch_short_conv_multi_update(const void *x, const void *weight, void *y, void *pool,
                                           const int32_t *state_indices, const int32_t *num_accepted,
                                           int64_t n_slots, int N, int S, int D, int ks, int activation,
                                           int dtype, cudaStream_t stream);

cudaError_t launch_recurrent_step(const void *q, const void *k, const void *v, const float *g,
                                  const float *beta, const GateArgs *gate, const EpiArgs *epi,
                                  float *pool, const int32_t *state_indices,
                                  const int32_t *num_accepted, int64_t n_slots, void *o, int N,
                                  int S, int H, float scale, int dtype, cudaStream_t stream);

// The output epilogue in place on o [rows, 128].
cudaError_t launch_output_gate_norm(void *o, const EpiArgs &epi, int64_t rows, int dtype,
                                    cudaStream_t stream);

}  // namespace kda
