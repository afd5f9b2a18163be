// Sequence / chunk index of a packed (varlen) batch, built on the device.
//
// The per-request loop of the Ascend model file (_prefill_flash_kda /
// _prefill_torch_kda slice every request by its boundaries and pad it to a
// multiple of the chunk) becomes one table: for every sequence its first
// token and length, and the exclusive prefix sum of ceil(len / 64) so that a
// global chunk id maps to (sequence, chunk within sequence).  The host never
// reads cu_seqlens; bad entries are detected here, their sequences skipped,
// and a status bit raised in the workspace.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kIndexThreads = 1024;
constexpr int kMaxSortedSeqs = 256;  // beyond this, sequences keep their order

__global__ void __launch_bounds__(kIndexThreads)
    chunk_index_kernel(const int32_t *__restrict__ cu_seqlens, int n_seqs, int64_t total_tokens,
                       int H, const int32_t *__restrict__ state_indices, int64_t n_slots,
                       void *workspace, WsLayout L) {
    // the previous kernel of the stream (e.g. the previous forward's scan, or
    // its strong-decay prep, which finishes only after a scan running beside it)
    // is complete before anything is written; the next kernel may be scheduled
    // now, and waits for this grid to finish
    griddep_wait();
    griddep_launch_dependents();
    int32_t *seq_start = ws_at<int32_t>(workspace, L.seq_start_off);
    int32_t *seq_len = ws_at<int32_t>(workspace, L.seq_len_off);
    int32_t *chunk_off = ws_at<int32_t>(workspace, L.chunk_off_off);
    __shared__ int warp_tot[kIndexThreads / 32];
    __shared__ int status_s;
    if (threadIdx.x == 0) status_s = 0;
    __syncthreads();

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int carry = 0;  // chunks of all previous tiles
    for (int base = 0; base < n_seqs; base += kIndexThreads) {
        const int n = base + threadIdx.x;
        int cnt = 0;
        if (n < n_seqs) {
            int64_t s, e;
            if (cu_seqlens) {
                s = cu_seqlens[n];
                e = cu_seqlens[n + 1];
            } else {
                const int64_t len = total_tokens / n_seqs;
                s = (int64_t)n * len;
                e = s + len;
            }
            int start = -1, len = 0;
            if (s < 0 || e < s || e > total_tokens) {
                atomicOr(&status_s, kBadSeqlens);
            } else if (state_indices &&
                       (state_indices[n] < 0 || (int64_t)state_indices[n] >= n_slots)) {
                atomicOr(&status_s, kBadSlot);
            } else {
                start = (int)s;
                len = (int)(e - s);
                cnt = (len + kChunk - 1) / kChunk;
            }
            seq_start[n] = start;
            seq_len[n] = len;
        }
        // block-wide exclusive scan of cnt
        int x = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_tot[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int w = warp_tot[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            warp_tot[lane] = w;  // inclusive over warps
        }
        __syncthreads();
        const int before = (warp ? warp_tot[warp - 1] : 0) + x - cnt;
        if (n < n_seqs) chunk_off[n] = carry + before;
        carry += warp_tot[kIndexThreads / 32 - 1];
        __syncthreads();
    }
    // sequences by decreasing length (ties: lower index first), so that a
    // scan grid walking this order starts its longest chains first; the
    // quadratic count runs for batches of up to kMaxSortedSeqs sequences
    int32_t *order = ws_at<int32_t>(workspace, L.seq_order_off);
    __shared__ int len_s[kMaxSortedSeqs];
    __syncthreads();  // seq_len of every sequence is written
    const bool sorted = n_seqs <= kMaxSortedSeqs;
    if (sorted)
        for (int n = threadIdx.x; n < n_seqs; n += kIndexThreads) len_s[n] = seq_len[n];
    __syncthreads();
    for (int n = threadIdx.x; n < n_seqs; n += kIndexThreads) {
        int rank = n;
        if (sorted) {
            const int ln = len_s[n];
            rank = 0;
            for (int m = 0; m < n_seqs; ++m) {
                const int lm = len_s[m];
                rank += (lm > ln) || (lm == ln && m < n);
            }
        }
        order[rank] = n;
    }
    // no (chunk, head) record of this call is written yet
    {
        const int64_t n_items = (int64_t)carry * H;
        int4 *ready4 = ws_at<int4>(workspace, L.ready_off);
        for (int64_t i = threadIdx.x; i < n_items / 4; i += kIndexThreads) ready4[i] = make_int4(0, 0, 0, 0);
        int32_t *ready = ws_at<int32_t>(workspace, L.ready_off);
        for (int64_t i = n_items / 4 * 4 + threadIdx.x; i < n_items; i += kIndexThreads) ready[i] = 0;
    }
    if (threadIdx.x == 0) {
        chunk_off[n_seqs] = carry;
        *ws_at<int32_t>(workspace, L.status_off) = status_s;
        *ws_at<int32_t>(workspace, L.defer_count_off) = 0;  // no item deferred yet
        *ws_at<int32_t>(workspace, L.item_ctr_off) = 0;     // no item handed out yet
        *ws_at<int32_t>(workspace, L.scan_done_off) = 0;
        *ws_at<int32_t>(workspace, L.strong_done_off) = 0;
        *ws_at<int32_t>(workspace, L.prep_done_off) = 0;
    }
}

}  // namespace

void preload_chunk_index_kernel() {
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, chunk_index_kernel) != cudaSuccess) cudaGetLastError();
}

cudaError_t launch_chunk_index(const int32_t *cu_seqlens, int n_seqs, int64_t total_tokens, int H,
                               const int32_t *state_indices, int64_t n_slots, void *workspace,
                               cudaStream_t stream) {
    const WsLayout L = ws_layout(total_tokens, n_seqs, H, 0);
    const cudaError_t e = launch_dependent(chunk_index_kernel, dim3(1), dim3(kIndexThreads), 0, stream,
                                           cu_seqlens, n_seqs, total_tokens, H, state_indices,
                                           n_slots, workspace, L);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace kda
