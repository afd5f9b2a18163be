/*
 * kda.h -- C ABI of libkda, the GB300 (sm_103a) Kimi Delta Attention core.
 *
 * Kimi Delta Attention (KDA) is a gated DeltaNet whose decay is per key
 * channel (nnterp "kimi_linear" page, paragraph defining Kimi Delta
 * Attention).  Per (sequence, head), with q and k L2-normalised inside the
 * library (eps 1e-6 added to the sum of squares, inside the root; Ascend
 * model file, _l2_normalize) and an fp32 K x V state S:
 *
 *     S   <- diag(exp(g_t)) S                      decay each key channel
 *     S   <- S + beta_t k_t (v_t - S^T k_t)^T      delta-rule write
 *     o_t  = scale * S^T q_t                       read-out, updated state
 *
 * Two forms are exported, as on that page: a chunked form for prompts
 * (kda_chunk_fwd, chunk 64; Ascend model file, _torch_chunk_kda and
 * _prefill_flash_kda / _prefill_torch_kda for the per-request loop) and a
 * token step for decode on a pooled state (kda_recurrent_step; Ascend model
 * file, _decode_fused_kda / _decode_gdr).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Pointers are DEVICE pointers unless stated.  All tensors are dense,
 * row-major (C order), without padding.  Nothing is allocated: the caller
 * owns every buffer, including the chunk workspace.  Nothing is kept
 * between calls.  Work is enqueued on `stream` (a cudaStream_t passed as
 * void*; NULL = the legacy default stream) and the call returns without
 * synchronising; the host never reads device memory.
 *
 * Layouts (T = tokens, H = heads, K = key dim, V = value dim, N = sequences):
 *   q, k, g : [T, H, K]     v, o : [T, H, V]     beta : [T, H]
 *   states  : [N, H, V, K]  fp32, key dim contiguous.  This is the transpose
 *             of the mathematical K x V state, the orientation the model
 *             file's recurrent-state cache uses.
 * Element types: q, k, v and o are all `dtype` (kda_dtype); g, beta and the
 * states are always fp32.  g is the log-decay (<= 0 for a contraction; any
 * finite value is accepted, but on the bf16 tensor-core chunk path positive
 * values are supported only while their sum over 16 tokens stays below 40),
 * beta is the already-activated write strength.
 * The supported head dims are K = V = 128.
 *
 * Alignment: row pointers must be 16-byte aligned for fp32 tensors and for
 * bf16 tensors on the tensor-core chunk path, 8-byte aligned for other bf16
 * uses; the workspace 256-byte aligned.  (Tensors from cudaMalloc or
 * PyTorch's allocator always are.)
 *
 * Errors: arguments are validated before anything is enqueued; a failing
 * call returns a kda_status other than KDA_OK and enqueues nothing.  A
 * failed kernel launch returns KDA_ERR_CUDA (the CUDA error is cleared).
 * Errors that only the device can see (bad cu_seqlens, a slot index out of
 * range, a bounded wait that gave up) never cause an out-of-bounds access;
 * they are reported as stated per entry point (the chunked forward: the
 * KDA_WS_* bits of its workspace status word).
 *
 * Pending CUDA errors: before launching, every entry point reads and thereby
 * clears the calling thread's pending (non-sticky) CUDA runtime error with
 * cudaGetLastError(), so that a failed launch of its own is not mistaken for
 * an earlier one.  A caller that needs its own pending error must read it
 * (cudaGetLastError / cudaPeekAtLastError) before calling into libkda.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad dtype, ... */
    KDA_ERR_UNSUPPORTED = 2, /* valid request outside what is built (K, V != 128) */
    KDA_ERR_WORKSPACE = 3,   /* workspace NULL, too small or misaligned */
    KDA_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed */
    KDA_ERR_DEVICE_TIMEOUT = 5 /* a bounded device-side wait gave up (see KDA_WS_TIMEOUT) */
} kda_status;

typedef enum {
    KDA_F32 = 0,  /* q, k, v, o in fp32 */
    KDA_BF16 = 1  /* q, k, v, o in bf16 */
} kda_dtype;

/* kda_chunk_fwd flags */
#define KDA_CHUNK_PRECISE 1    /* fp32 CUDA-core chunk path also for bf16 inputs */
#define KDA_CHUNK_SCAN_WIDE 2  /* tensor-core path: one scan CTA per (sequence, head) */
#define KDA_CHUNK_SCAN_SPLIT 4 /* tensor-core path: four scan CTAs per (sequence, head) */
#define KDA_CHUNK_GATED 8      /* kda_chunk_workspace_bytes only: size for kda_chunk_fwd_gated */

/* Chunk length of the chunked form (Ascend model file, _KDA_CHUNK_SIZE). */
#define KDA_CHUNK 64

/* Human-readable name of a kda_status value (static string, never NULL). */
const char *kda_status_string(int status);

/* ABI version of this library: 100 * major + minor. */
int kda_version(void);

/*
 * Bytes of device workspace kda_chunk_fwd needs for these sizes (0 on
 * invalid sizes).  The workspace holds the sequence/chunk index and the
 * per-chunk intra-chunk products handed from the intra-chunk kernel to the
 * state-scan kernel.  It must be 256-byte aligned.
 */
size_t kda_chunk_workspace_bytes(int64_t total_tokens, int n_seqs, int H, int K, int V,
                                 int dtype, int flags);

/*
 * Chunked KDA forward over N packed sequences (prefill).
 *
 *   q, k        [T, H, K] dtype     v [T, H, V] dtype     g [T, H, K] fp32
 *   beta        [T, H] fp32
 *   o           [T, H, V] dtype     (output, written for every real token)
 *   cu_seqlens  device int32 [N+1], non-decreasing, cu_seqlens[0] = 0,
 *               cu_seqlens[N] = T; sequence n owns tokens [cu[n], cu[n+1]).
 *               NULL = N sequences of equal length T / N (N must divide T),
 *               i.e. a dense [B, T/B, H, *] batch.
 *   state_indices  NULL: initial_state and final_state are [N, H, V, K].
 *               Otherwise device int32 [N], distinct values in [0, n_slots):
 *               initial_state / final_state are pools [n_slots, H, V, K] and
 *               sequence n reads its initial state from, and writes its
 *               final state to, slot state_indices[n] (the hand-off of a
 *               prefill's final state into the decode state pool; model
 *               file, update_mamba_cache).
 *   initial_state  NULL = zero initial states.
 *   final_state    NULL = final states are not written.  May alias
 *               initial_state (each slot is read before it is written).
 *   scale       multiplies the normalised query (the model uses 1/sqrt(K)).
 *   dtype       kda_dtype of q, k, v, o.
 *   flags       0 or KDA_CHUNK_PRECISE.  Without it, bf16 inputs take
 *               the tensor-core path (bf16 operands, fp32 accumulation,
 *               fp32 state); fp32 inputs always take the fp32 path.  On the
 *               tensor-core path the state scan runs either as four CTAs per
 *               (sequence, head), 32 value columns each, or as one CTA per
 *               (sequence, head); by default the first when all of them fit
 *               in one wave on the device, else the second.
 *               KDA_CHUNK_SCAN_SPLIT / KDA_CHUNK_SCAN_WIDE force one (not
 *               both; ignored on the fp32 path).  Results agree within
 *               rounding of the summation order.  In kda_chunk_fwd the
 *               four-CTA scan, when its CTAs number at most the SM count
 *               less 8, is launched before the intra-chunk phase and runs
 *               alongside it (cooperatively, one CTA per SM beside one prep
 *               CTA), waiting for each (chunk, head) record as it is
 *               written; the results are those of the two phases run one
 *               after the other, bit for bit.  Chunks that need the
 *               strong-decay path (KDA_WS_STRONG_DECAY) are then redone
 *               only on the SMs that host no scan CTA, so a call where most
 *               chunks need it runs several times slower than with
 *               KDA_CHUNK_SCAN_WIDE or the two phases called separately.
 *               The scan waits for each record for at most ~2 s: work on
 *               other streams that holds the GPU's SMs that long makes the
 *               call report KDA_WS_TIMEOUT.
 *   workspace   device, 256-byte aligned, kda_chunk_workspace_bytes(...)
 *               bytes; its contents are scratch and may be anything.
 *
 * A zero-length sequence hands back its initial state (or zeros) as its
 * final state.  Device-side argument errors (cu_seqlens decreasing, out of
 * [0, T], or a slot index out of range) skip the offending sequence
 * (nothing of it is read or written) and set a KDA_WS_* bit that
 * kda_workspace_status() reports.
 */
int kda_chunk_fwd(const void *q, const void *k, const void *v, const float *g,
                  const float *beta, const float *initial_state, float *final_state,
                  const int32_t *state_indices, int64_t n_slots, void *o,
                  const int32_t *cu_seqlens, int n_seqs, int64_t total_tokens, int H, int K,
                  int V, float scale, int dtype, int flags, void *workspace,
                  size_t workspace_bytes, void *stream);

/*
 * The two phases of kda_chunk_fwd, for callers that schedule or time them
 * separately.  kda_chunk_fwd(args) == kda_chunk_intra(args) followed, on the
 * same stream and with the same workspace, by kda_chunk_scan(args).
 *
 * kda_chunk_intra: builds the sequence/chunk index from cu_seqlens (and
 *   checks state_indices), then computes, for every (chunk, head), the
 *   intra-chunk products -- L2 norms, cumulative log-decay, the UT transform
 *   (I + L)^-1 diag(beta) by forward substitution, the WY products W and U,
 *   the causal scores -- into the workspace.  Reads q, k, v, g, beta.
 * kda_chunk_scan: the sequential inter-chunk state pass; reads the
 *   workspace and the initial states, writes o and the final states.
 * Both take exactly the arguments of kda_chunk_fwd and validate them the
 * same way; q, k, v, g, beta are not read by the scan and o, states are not
 * touched by the intra phase.
 */
int kda_chunk_intra(const void *q, const void *k, const void *v, const float *g,
                    const float *beta, const float *initial_state, float *final_state,
                    const int32_t *state_indices, int64_t n_slots, void *o,
                    const int32_t *cu_seqlens, int n_seqs, int64_t total_tokens, int H, int K,
                    int V, float scale, int dtype, int flags, void *workspace,
                    size_t workspace_bytes, void *stream);
int kda_chunk_scan(const void *q, const void *k, const void *v, const float *g,
                   const float *beta, const float *initial_state, float *final_state,
                   const int32_t *state_indices, int64_t n_slots, void *o,
                   const int32_t *cu_seqlens, int n_seqs, int64_t total_tokens, int H, int K,
                   int V, float scale, int dtype, int flags, void *workspace,
                   size_t workspace_bytes, void *stream);

/*
 * Workspace status word: the first int32 of a chunk workspace, rewritten by
 * every kda_chunk_fwd / kda_chunk_intra that uses it and OR-ed into by the
 * kernels of that call.
 */
#define KDA_WS_BAD_SEQLENS 1 /* cu_seqlens decreasing or outside [0, T]: those sequences skipped */
#define KDA_WS_BAD_SLOT 2    /* a state_indices entry outside [0, n_slots): that sequence skipped */
#define KDA_WS_TIMEOUT 4     /* a bounded wait of a kernel (a copy or an MMA that never
                                completed, or a record of the intra-chunk phase that a scan
                                running alongside it never saw written, ~2 s) gave up: the
                                CTA left its remaining chunks unwritten and exited; outputs of
                                that call are incomplete */
#define KDA_WS_EXACT_DECAY 8 /* informational, not an error: on the tensor-core path some
                                16-token block decayed by more than 75 in a key channel (per-token
                                decays below about -5) and its diagonal 16 x 16 scores were
                                computed with exact pairwise exponentials */
#define KDA_WS_STRONG_DECAY 16 /* informational, not an error: on the tensor-core path some
                                  (chunk, head) had |G_r - G_31| > 80 in a key channel (G the
                                  cumulative log-decay inside the chunk) and was computed by the
                                  strong-decay prep, with per-16-token decay references */

/*
 * The kda_status that a workspace status word stands for:
 * KDA_ERR_DEVICE_TIMEOUT if KDA_WS_TIMEOUT is set, else KDA_ERR_INVALID_ARG
 * if KDA_WS_BAD_SEQLENS or KDA_WS_BAD_SLOT is set, else KDA_OK (the
 * informational KDA_WS_EXACT_DECAY and KDA_WS_STRONG_DECAY are not errors).
 * Pure host function.
 */
int kda_status_from_workspace_flags(int flags);

/*
 * Status word of the last kda_chunk_fwd that used this workspace
 * (KDA_WS_* bits, 0 = none) into *flags_out.  Synchronises `stream` and
 * copies 4 bytes to the host.  Returns KDA_ERR_CUDA if that copy fails,
 * KDA_ERR_INVALID_ARG for NULL arguments, and otherwise
 * kda_status_from_workspace_flags(*flags_out): KDA_ERR_DEVICE_TIMEOUT after
 * a bounded device-side wait gave up (the mirror of the model's own
 * raise-on-bad-input convention for errors only the device can see).
 */
int kda_workspace_status(const void *workspace, int *flags_out, void *stream);

/*
 * One decode token for each of N sequences, on a pooled state, in place
 * (model file, _decode_gdr / _decode_fused_kda with one token per sequence).
 *
 *   q, k, g     [N, H, K] (q, k dtype; g fp32)   v [N, H, V] dtype
 *   beta        [N, H] fp32
 *   state_pool  [n_slots, H, V, K] fp32, read and updated in place
 *   state_indices  device int32 [N], distinct slots; NULL = slot n for
 *               sequence n (then n_slots >= N).  A slot outside
 *               [0, n_slots) leaves the pool untouched and writes NaN to
 *               that sequence's o rows.
 *   o           [N, H, V] dtype
 *
 * The state is streamed once from HBM and written back once; N = 0 is a
 * no-op.
 */
int kda_recurrent_step(const void *q, const void *k, const void *v, const float *g,
                       const float *beta, float *state_pool, const int32_t *state_indices,
                       int64_t n_slots, void *o, int N, int H, int K, int V, float scale,
                       int dtype, void *stream);

/*
 * Size of the fixed scratch array behind kda_chunk_fwd_noalloc: 64 MiB.
 */
#define KDA_NOALLOC_WORKSPACE_BYTES (64u * 1024u * 1024u)

/*
 * kda_chunk_fwd for callers that cannot allocate device memory.  (The pages
 * describing KDA have no counterpart of this call; it exists for library
 * users.)  Some hosts give a kernel library only its input and output
 * buffers -- an inference server's plugin interface that owns all device
 * memory through its own pool, or a latency-critical path where a
 * cudaMalloc, which can synchronise the device, is not allowed.  This call
 * takes the arguments of kda_chunk_fwd minus the workspace and allocates
 * nothing: its scratch space is a fixed array of
 * KDA_NOALLOC_WORKSPACE_BYTES inside the library's device image, which every
 * GPU that loads the library holds until the process exits.
 *
 *   - The first call on a device (with that device current) looks up the
 *     array's device address (cudaGetSymbolAddress) and keeps it with the
 *     CUDA context it was taken in; make that first call before any stream
 *     capture on that device.  The lookup is repeated only when the current
 *     context differs (a cudaDeviceReset gives the device a new primary
 *     context, in which the array has a new address); after such a reset,
 *     make one call before capturing again.
 *   - Sizes whose kda_chunk_workspace_bytes(...) exceeds
 *     KDA_NOALLOC_WORKSPACE_BYTES return KDA_ERR_WORKSPACE and enqueue
 *     nothing; other argument errors are those of kda_chunk_fwd.
 *     KDA_CHUNK_GATED in flags is ignored (this is the forward from
 *     activated g and beta).
 *   - Every call, from any stream or thread, uses the same array.  Calls
 *     whose work overlaps on the GPU race and corrupt each other's results:
 *     order them (one stream, or events).  Nothing needs clearing between
 *     calls.
 *   - kda_workspace_status() is not available for this call (the workspace
 *     is not visible to the caller); bad cu_seqlens or slots still skip the
 *     offending sequences.
 */
int kda_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const float *g,
                          const float *beta, const float *initial_state, float *final_state,
                          const int32_t *state_indices, int64_t n_slots, void *o,
                          const int32_t *cu_seqlens, int n_seqs, int64_t total_tokens, int H,
                          int K, int V, float scale, int dtype, int flags, void *stream);

/*
 * Short causal convolution of the fused q/k/v projection (model file,
 * KimiShortConvolution: causal_conv1d_fn in prefill, causal_conv1d_update
 * in decode).  Depthwise over D channels with ks taps (2 <= ks <= 8):
 *   y[t, d] = act( sum_{i<ks} weight[i, d] * x[t - (ks - 1) + i, d] )
 * where positions before a sequence's start read its conv state (its ks - 1
 * previous inputs; zeros without an initial state).  act is SiLU
 * (KDA_CONV_SILU, x * sigmoid(x)) or none (KDA_CONV_NONE).
 *
 *   x, y        [T, D] (prefill) / [N, D] (update), dtype; D % 8 == 0
 *   weight      [ks, D] dtype (the model's conv weight, tap-major)
 *   conv states [N or slots, ks - 1, D] dtype: per sequence, or slots of a
 *               pool picked by state_indices (int32 [N])
 *
 * Prefill: cu_seqlens int32 [N+1] (or NULL: N equal-length sequences);
 * initial_states NULL = zeros (the model passes has_initial_state = 0);
 * final_states (NULL = not written) receives each sequence's last ks - 1
 * inputs and may be the same pool as initial_states.  cu_seqlens must be
 * non-decreasing within [0, T]; malformed entries give undefined outputs for
 * those tokens but no access outside the buffers, and leave the state alone.
 * Update: one token per sequence; the window is [state ; x] and the state
 * shifts by one token in place; a slot outside [0, n_slots) gives NaN
 * outputs and leaves the pool untouched.  y must not overlap x or a state;
 * sequences must not share a slot.  x, y, weight and the states are 16-byte
 * aligned.  A prefill whose staged copy never lands (a bounded wait expired)
 * writes NaN to the affected outputs.
 */
#define KDA_CONV_NONE 0
#define KDA_CONV_SILU 1
int kda_short_conv_fwd(const void *x, const void *weight, void *y, const int32_t *cu_seqlens,
                       int n_seqs, int64_t total_tokens, int D, int ks, int activation,
                       const void *initial_states, void *final_states,
                       const int32_t *state_indices, int64_t n_slots, int dtype, void *stream);
int kda_short_conv_update(const void *x, const void *weight, void *y, void *state_pool,
                          const int32_t *state_indices, int64_t n_slots, int N, int D, int ks,
                          int activation, int dtype, void *stream);

/*
 * Short conv with a speculative verify width (the model's update branch with
 * S > 1 tokens per sequence, conv_state_indices from the per-sequence state
 * blocks and num_accepted_tokens: Ascend model file,
 * KimiShortConvolution.forward and KimiDeltaAttention._forward_core).
 *
 *   x, y          [N, S, D] dtype;  weight [ks, D];  state_pool [slots, ks - 1, D]
 *   state_indices device int32 [N, S]: the conv state after token t of
 *                 sequence n is written to slot state_indices[n][t]
 *   num_accepted  device int32 [N] or NULL: sequence n starts from slot
 *                 state_indices[n][num_accepted[n] - 1] (NULL: [n][0])
 *
 * The same slot convention as kda_recurrent_multi_step.  A count outside
 * [1, S] or a slot outside [0, n_slots) gives the sequence NaN outputs and
 * leaves the pool untouched; slots of different sequences must not overlap.
 * S = 1 with num_accepted = NULL is kda_short_conv_update with
 * state_indices.
 */
int kda_short_conv_multi_update(const void *x, const void *weight, void *y, void *state_pool,
                                const int32_t *state_indices, const int32_t *num_accepted,
                                int64_t n_slots, int N, int S, int D, int ks, int activation,
                                int dtype, void *stream);

/*
 * Speculative (multi-token) decode: S tokens per sequence run in order
 * through the recurrence (the model's decode call with a verify width S:
 * model file, _decode_fused_kda / _decode_gdr with ssm_state_indices of
 * batch x S entries and num_accepted_tokens).
 *
 *   q, k, g       [N, S, H, K]   v, o [N, S, H, V]   beta [N, S, H]
 *   state_indices device int32 [N, S]: the state after token t of sequence
 *                 n is written to slot state_indices[n][t]
 *   num_accepted  device int32 [N] or NULL: sequence n starts from slot
 *                 state_indices[n][num_accepted[n] - 1] (NULL: from
 *                 state_indices[n][0]), the state left by the previous
 *                 verify step after its last accepted token
 *
 * A sequence with a slot outside [0, n_slots) or num_accepted outside
 * [1, S] leaves the pool untouched and gets NaN outputs.  Slots of
 * different sequences must not overlap.  S = 1 with num_accepted = NULL is
 * kda_recurrent_step.  The state is read once and written S times.
 */
int kda_recurrent_multi_step(const void *q, const void *k, const void *v, const float *g,
                             const float *beta, float *state_pool, const int32_t *state_indices,
                             const int32_t *num_accepted, int64_t n_slots, void *o, int N, int S,
                             int H, int K, int V, float scale, int dtype, void *stream);

/*
 * Gated entry points: the model's gate activation computed in-kernel
 * (Ascend model file, _prefill_torch_kda and the decode branch of
 * KimiDeltaAttention.forward).  Instead of activated g and beta they take
 *
 *   raw_gate    [T, H, K] (prefill) / [N, H, K] (decode), in the q dtype
 *   raw_beta    [T, H] / [N, H], in the q dtype
 *   a_log       device fp32 [H]      (the model's A_log)
 *   dt_bias     device fp32 [H, K]   (the model's flat dt_bias, per head)
 *   lower_bound, use_lower_bound
 *
 * and use, per element,
 *   x    = raw_gate + dt_bias[h][k]
 *   g    = lower_bound * sigmoid(exp(a_log[h]) * x)   if use_lower_bound
 *        = -exp(a_log[h]) * softplus(x)               otherwise
 *   beta = sigmoid(raw_beta)
 * with softplus(x) = max(x, 0) + log1p(exp(-|x|)).  Everything else --
 * arguments, layouts, aliasing, errors -- is as for kda_chunk_fwd /
 * kda_recurrent_step.  The tensor-core path reads the raw bf16 gate and
 * activates it on chip (half the gate bytes of an fp32 g); the fp32 path
 * activates it into the workspace first.  Size the workspace with
 * kda_chunk_workspace_bytes(..., flags | KDA_CHUNK_GATED).  Any decay the
 * gate produces is supported on every path: on the tensor-core path chunks
 * with strong decay take the strong-decay prep and, beyond about -5 per
 * token, exact pairwise exponentials on the diagonal (KDA_WS_STRONG_DECAY,
 * KDA_WS_EXACT_DECAY).
 *
 * Output epilogue (model file, KimiDeltaAttention._project_out), optional:
 *   out_gate    [T, H, V] / [N, H, V] in the q dtype, or NULL for none
 *   norm_weight device fp32 [V];  norm_eps > 0
 * replaces each output row of V values by
 *   o / sqrt(mean(o^2) + norm_eps) * norm_weight * sigmoid(out_gate).
 * Decode applies it in the step.  The chunked forward applies it as a final
 * pass over the stored o (kda_output_gate_norm) when its scan runs alongside
 * the intra-chunk phase (see kda_chunk_fwd); otherwise inside its state scan
 * where it can (tensor-core path, one CTA per 32 value columns, out_gate
 * 16-byte aligned, at most 64 (sequence, head) pairs: the row's four CTAs
 * exchange their sums of squares through the workspace, and the grid is
 * launched cooperatively, so it must fit the GPU at once), normalising the
 * unrounded o; else as the final pass.  The two agree within the rounding of
 * o to its dtype.
 */
int kda_chunk_fwd_gated(const void *q, const void *k, const void *v, const void *raw_gate,
                        const void *raw_beta, const float *a_log, const float *dt_bias,
                        float lower_bound, int use_lower_bound, const void *out_gate,
                        const float *norm_weight, float norm_eps, const float *initial_state,
                        float *final_state, const int32_t *state_indices, int64_t n_slots,
                        void *o, const int32_t *cu_seqlens, int n_seqs, int64_t total_tokens,
                        int H, int K, int V, float scale, int dtype, int flags, void *workspace,
                        size_t workspace_bytes, void *stream);

int kda_recurrent_step_gated(const void *q, const void *k, const void *v, const void *raw_gate,
                             const void *raw_beta, const float *a_log, const float *dt_bias,
                             float lower_bound, int use_lower_bound, const void *out_gate,
                             const float *norm_weight, float norm_eps, float *state_pool,
                             const int32_t *state_indices, int64_t n_slots, void *o, int N,
                             int H, int K, int V, float scale, int dtype, void *stream);

/*
 * kda_recurrent_multi_step from the model's raw gates, with the optional
 * output epilogue: the speculative decode as the model's fused decode runs it
 * (raw decay and beta, num_accepted_tokens, per-token state slots).
 *   raw_gate [N, S, H, K] and raw_beta [N, S, H] in the q dtype;
 *   out_gate [N, S, H, V] in the q dtype or NULL.
 * The gate and the epilogue are as for kda_recurrent_step_gated, the slots
 * and counts as for kda_recurrent_multi_step.
 */
int kda_recurrent_multi_step_gated(const void *q, const void *k, const void *v,
                                   const void *raw_gate, const void *raw_beta, const float *a_log,
                                   const float *dt_bias, float lower_bound, int use_lower_bound,
                                   const void *out_gate, const float *norm_weight, float norm_eps,
                                   float *state_pool, const int32_t *state_indices,
                                   const int32_t *num_accepted, int64_t n_slots, void *o, int N,
                                   int S, int H, int K, int V, float scale, int dtype, void *stream);

/*
 * The output epilogue alone, in place on o [rows, V] (rows = tokens x heads,
 * V = 128, dtype as q): each row becomes
 *   o / sqrt(mean(o^2) + eps) * weight * sigmoid(gate)
 * with gate [rows, V] (same dtype) and weight [V] fp32 (model file,
 * KimiDeltaAttention._project_out: o_norm, then the sigmoid gate).  The row
 * statistics are taken in fp32 from the stored o.  rows = 0 is a no-op.
 */
int kda_output_gate_norm(void *o, const void *gate, const float *weight, float eps,
                         int64_t rows, int V, int dtype, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
