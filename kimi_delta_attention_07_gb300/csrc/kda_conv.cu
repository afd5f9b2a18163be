// Short causal convolution of the model's fused q/k/v projection (Ascend
// model file, KimiShortConvolution: causal_conv1d_fn in prefill,
// causal_conv1d_update in decode).  Per channel d, over the last ks inputs:
//   y[t, d] = act( sum_{i<ks} w[i, d] x[t - (ks - 1) + i, d] )
// with positions before a sequence's start read from its conv state (the
// ks - 1 previous inputs, or zeros).  Depthwise, so HBM bound.  The prefill
// streams 4 KB row segments of a run of tokens into shared memory with bulk
// copies (double-buffered, one CTA per SM) while each thread slides a window
// over its 16-byte column of them in registers.
#include <algorithm>

#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

constexpr int kConvThreads = 256;

// Eight consecutive channels kept raw (one 16-byte bf16 vector or two fp32
// vectors) so that a thread can issue all of its row loads before using any.
template <typename T>
struct Row8;
template <>
struct Row8<__nv_bfloat16> {
    uint4 u;
    __device__ __forceinline__ void load(const __nv_bfloat16 *p) {
        u = __ldg(reinterpret_cast<const uint4 *>(p));
    }
    __device__ __forceinline__ void to_f32(float (&x)[8]) const {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {  // a bf16 is the top half of an fp32
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
};
template <>
struct Row8<float> {
    float4 a, b;
    __device__ __forceinline__ void load(const float *p) {
        a = __ldg(reinterpret_cast<const float4 *>(p));
        b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    }
    __device__ __forceinline__ void to_f32(float (&x)[8]) const {
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    }
};

template <typename T>
__device__ __forceinline__ void load8(const T *p, float (&x)[8]) {
    Row8<T> r;
    r.load(p);
    r.to_f32(x);
}

template <typename T>
__device__ __forceinline__ void store8(T *p, const float (&x)[8]);
template <>
__device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16 *p, const float (&x)[8]) {
    uint4 u;
    uint32_t *w = reinterpret_cast<uint32_t *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 h2 = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
        w[i] = *reinterpret_cast<const uint32_t *>(&h2);
    }
    *reinterpret_cast<uint4 *>(p) = u;
}
template <>
__device__ __forceinline__ void store8<float>(float *p, const float (&x)[8]) {
    *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
    *reinterpret_cast<float4 *>(p + 4) = make_float4(x[4], x[5], x[6], x[7]);
}

// SiLU y * sigmoid(y) = y / (1 + 2^(-y log2 e)) on the SFU (approximate
// base-2 exponential and reciprocal, subnormals flushed: an exponential that
// underflows leaves y, one that overflows gives -0).  The depthwise conv has
// about ten ALU operations per element against 4 bytes of traffic, so the
// instruction count sets its speed next to HBM.
__device__ __forceinline__ float ex2_ftz(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ float rcp_ftz(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ float conv_act(float y, int activation) {
    constexpr float kLog2e = 1.4426950408889634f;
    return activation == KDA_CONV_SILU ? y * rcp_ftz(1.0f + ex2_ftz(-kLog2e * y)) : y;
}

// the sequence owning token t (largest n with cu[n] <= t)
__device__ __forceinline__ int owner(const int32_t *cu, int n_seqs, int64_t t) {
    int lo = 0, hi = n_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// sequence n's token range [s, e): from cu_seqlens, or n_seqs equal lengths
__device__ __forceinline__ void seq_range(const int32_t *cu, int n_seqs, int64_t total, int n,
                                          int64_t &s, int64_t &e) {
    if (cu) {
        s = cu[n];
        e = cu[n + 1];
    } else {
        const int64_t len = total / n_seqs;
        s = (int64_t)n * len;
        e = s + len;
    }
}

struct ConvArgs {
    const void *x, *weight;
    void *y;
    const int32_t *cu_seqlens;
    const void *initial_states;  // [N or slots, ks - 1, D] or nullptr (zeros)
    void *final_states;          // [N or slots, ks - 1, D] or nullptr
    const int32_t *state_indices;
    int64_t n_slots, total_tokens;
    int n_seqs, D, ks, activation;
    int fuse_final;  // the prefill kernel writes final_states (which does not alias initial_states)
};

// 16 bytes of a row: 8 bf16 or 4 fp32 channels
template <typename T>
struct Vec16 {
    static constexpr int N = 16 / (int)sizeof(T);
};
__device__ __forceinline__ void unpack16(const uint4 u, float (&x)[8]) {  // bf16
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ void unpack16(const uint4 u, float (&x)[4]) {  // fp32
    x[0] = __uint_as_float(u.x); x[1] = __uint_as_float(u.y);
    x[2] = __uint_as_float(u.z); x[3] = __uint_as_float(u.w);
}
__device__ __forceinline__ uint4 pack16(const float (&x)[8]) {
    uint4 u;
    uint32_t *w = reinterpret_cast<uint32_t *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 h2 = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
        w[i] = *reinterpret_cast<const uint32_t *>(&h2);
    }
    return u;
}
__device__ __forceinline__ uint4 pack16(const float (&x)[4]) {
    return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                      __float_as_uint(x[3]));
}
__device__ __forceinline__ uint4 ldg16(const void *p) {
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

constexpr int kSegThreads = 256;               // threads across one row segment
constexpr int kSegBytes = 16 * kSegThreads;    // one row segment: 16 bytes per thread
constexpr int kPipeGroups = 2;                 // thread groups splitting the item's tokens
constexpr int kPipeThreads = kSegThreads * kPipeGroups;

// Tokens per work item: the longest even tile whose two stages fit in
// ~220 KB (24 for KS = 4).  Longer tiles spread the per-item work (window
// fill, waits, sequence lookup) over more tokens; measured on the 4k x 12288
// projection, two stages of long tiles beat more stages of short ones.
template <int KS>
__host__ __device__ constexpr int pipe_tile() {
    return (28 - KS) & ~1;
}
template <int KS>
__host__ __device__ constexpr int pipe_rows() {
    return pipe_tile<KS>() + KS - 1;  // the tile and the window's reach before it
}
template <int KS>
__host__ __device__ constexpr int pipe_stages() {
    return (220 * 1024) / (pipe_rows<KS>() * kSegBytes) < 6 ? (220 * 1024) / (pipe_rows<KS>() * kSegBytes)
                                                             : 6;
}
template <int KS>
__host__ __device__ constexpr int pipe_smem() {
    return pipe_stages<KS>() * pipe_rows<KS>() * kSegBytes + 128;  // stages + full/empty barriers
}

// Conv state row j (0..KS-2, oldest first) of sequence n, or zeros.
template <typename T, int KS, int C>
__device__ __forceinline__ void history16(const ConvArgs &a, int n, int64_t j, int d0,
                                          float (&v)[C]) {
    const T *init = reinterpret_cast<const T *>(a.initial_states);
    const int64_t slot = a.state_indices ? (int64_t)a.state_indices[n] : (int64_t)n;
    if (init && slot >= 0 && slot < a.n_slots && j >= 0 && j < KS - 1) {
        unpack16(ldg16(init + (slot * (KS - 1) + j) * a.D + d0), v);
    } else {
#pragma unroll
        for (int c = 0; c < C; ++c) v[c] = 0.0f;
    }
}

// Work item = (channel segment, token tile), segment-major; each CTA takes a
// contiguous run of items, so it keeps one segment's weights in registers
// for most of its run, and the window rows a tile reaches back into were
// fetched by the same CTA one item earlier and come from L2.  Rows
// t0 - (KS - 1) .. t0 + cnt - 1 of the segment land in smem rows 0 .. ROWS - 1
// (rows before token 0 are not fetched).  Each of the two thread groups takes
// half of the tile's tokens; a group whose tokens and window lie inside one
// sequence slides the window in registers, any other (a sequence starts in
// its range, or its window reaches into a conv state) takes the short
// per-token path.  Item k uses stage k % S; the stage is released by one
// arrival per warp on its empty barrier, and thread 0 waits for that alone
// before fetching item k + S into it, so no warp waits for another.  A fetch that never lands
// (a bounded wait expires) turns every later output of the warp into NaN.
template <typename T, int KS>
__global__ void __launch_bounds__(kPipeThreads, 1) conv_prefill_kernel(const ConvArgs a) {
    using namespace tc;
    constexpr int C = Vec16<T>::N;
    constexpr int ROWS = pipe_rows<KS>();
    constexpr int STAGE = ROWS * kSegBytes;
    constexpr int S = pipe_stages<KS>();
    constexpr int kPipeTile = pipe_tile<KS>();
    constexpr int TG = kPipeTile / kPipeGroups;  // tokens per thread
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + S * STAGE);
    uint64_t *empty = full + S;
    constexpr int kWarps = kPipeThreads / 32;
    const int tid = threadIdx.x;
    const int col = tid % kSegThreads, grp = tid / kSegThreads;
    const int seg_ch = kSegThreads * C;  // channels per segment
    const int segs = (a.D + seg_ch - 1) / seg_ch;
    const int64_t tiles = (a.total_tokens + kPipeTile - 1) / kPipeTile;
    const int64_t items = tiles * segs;
    const char *xb = reinterpret_cast<const char *>(a.x);
    T *y = reinterpret_cast<T *>(a.y);
    const int64_t row_bytes = (int64_t)a.D * sizeof(T);

    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();

    // local item k of this CTA is first + k
    const int64_t per = (items + gridDim.x - 1) / gridDim.x;
    const int64_t first = (int64_t)blockIdx.x * per;
    const int64_t n_local = max(min(per, items - first), (int64_t)0);
    auto issue = [&](int64_t k, int stage) {  // thread 0: fetch local item k into a stage
        const int64_t item = first + k;
        const int seg = (int)(item / tiles);
        const int64_t t0 = (item - (int64_t)seg * tiles) * kPipeTile;
        const int64_t t_end = min(t0 + kPipeTile, a.total_tokens);
        const int64_t h0 = max(t0 - (KS - 1), (int64_t)0);
        const int c0 = seg * seg_ch;
        const uint32_t bytes = (uint32_t)(min(seg_ch, a.D - c0) * (int)sizeof(T));
        unsigned char *st = smem + stage * STAGE;
        fence_async_smem();
        mbar_arrive_expect_tx(&full[stage], bytes * (uint32_t)(t_end - h0));
        for (int64_t tau = h0; tau < t_end; ++tau)
            bulk_g2s(st + (tau - t0 + KS - 1) * kSegBytes, xb + tau * row_bytes + (int64_t)c0 * sizeof(T),
                     bytes, &full[stage]);
    };
    if (tid == 0)
        for (int i = 0; i < S && i < n_local; ++i) issue(i, i);

    // Final states, fused: a token among its sequence's last KS - 1 is
    // copied to its final-state row by the thread that convolves it (below);
    // the rows a sequence shorter than KS - 1 takes from its initial state
    // (or zeros) are copied here, while the first fetches are in flight.
    T *fin = reinterpret_cast<T *>(a.final_states);
    const T *init = reinterpret_cast<const T *>(a.initial_states);
    if (a.fuse_final) {
        for (int n2 = blockIdx.x; n2 < a.n_seqs; n2 += gridDim.x) {
            int64_t s2, e2;
            seq_range(a.cu_seqlens, a.n_seqs, a.total_tokens, n2, s2, e2);
            const int64_t L = e2 - s2;
            const int64_t slot = a.state_indices ? (int64_t)a.state_indices[n2] : (int64_t)n2;
            if (L < 0 || L >= KS - 1 || slot < 0 || slot >= a.n_slots) continue;
            for (int r = 0; r < KS - 1 - L; ++r)
                for (int c = tid * C; c < a.D; c += kPipeThreads * C) {
                    const uint4 v = init ? ldg16(init + (slot * (KS - 1) + L + r) * a.D + c)
                                         : make_uint4(0, 0, 0, 0);
                    *reinterpret_cast<uint4 *>(fin + (slot * (KS - 1) + r) * a.D + c) = v;
                }
        }
    }
    // token t, when among the last KS - 1 of its sequence (ends at e), to its final row
    auto to_final = [&](int n_t, int64_t t, int64_t e_t, const uint4 raw, int d0) {
        const int64_t r = t - (e_t - (KS - 1));
        const int64_t slot = a.state_indices ? (int64_t)a.state_indices[n_t] : (int64_t)n_t;
        if (r >= 0 && r < KS - 1 && t < e_t && slot >= 0 && slot < a.n_slots)
            *reinterpret_cast<uint4 *>(fin + (slot * (KS - 1) + r) * a.D + d0) = raw;
    };

    float wt[KS][C];
    int w_seg = -1;
    bool failed = false;                   // warp-uniform
    int64_t issued = min(n_local, (int64_t)S);  // thread 0's count of fetched items
    int stage = 0;
    uint32_t phase = 0;  // parity of the stage's current use
    int seg = (int)(first / tiles);  // the current item's (segment, tile), stepped
    int64_t tile = first - (int64_t)seg * tiles;
    for (int64_t k = 0; k < n_local; ++k, ++tile) {
        if (tile == tiles) {
            tile = 0;
            ++seg;
        }
        const int64_t t0 = tile * kPipeTile;
        const int64_t t_end = min(t0 + kPipeTile, a.total_tokens);
        const int64_t ta = t0 + grp * TG, tb = min(ta + TG, t_end);  // this group's tokens
        const int d0 = seg * seg_ch + col * C;
        const bool active = d0 < a.D && ta < tb;
        if (active && seg != w_seg) {
#pragma unroll
            for (int i = 0; i < KS; ++i)
                unpack16(ldg16(reinterpret_cast<const T *>(a.weight) + (int64_t)i * a.D + d0), wt[i]);
            w_seg = seg;
        }
        int n = 0;
        int64_t s = 0, e = 0;
        if (active) {  // the sequence of the group's first token (overlaps the copy's flight)
            n = a.cu_seqlens ? owner(a.cu_seqlens, a.n_seqs, ta) : (int)(ta / (a.total_tokens / a.n_seqs));
            seq_range(a.cu_seqlens, a.n_seqs, a.total_tokens, n, s, e);
        }
        if (!failed) failed = !mbar_wait(&full[stage], phase, 400000000LL);
        failed = __any_sync(0xffffffffu, failed);
        const bool landed = !failed;
        // staged row of token tau (t0 - (KS - 1) <= tau < t_end, tau >= 0)
        const unsigned char *colp = smem + stage * STAGE + col * 16;
        auto staged_raw = [&](int64_t tau) {
            return *reinterpret_cast<const uint4 *>(colp + (int)(tau - t0 + KS - 1) * kSegBytes);
        };
        auto staged = [&](int64_t tau, float(&v)[C]) { unpack16(staged_raw(tau), v); };
        if (active && landed) {
            const int64_t w0 = ta - (KS - 1);
            if (w0 >= s && w0 >= 0 && tb <= e && tb - ta == TG) {  // one sequence, staged window
                float win[KS - 1][C];
#pragma unroll
                for (int r = 0; r < KS - 1; ++r) staged(w0 + r, win[r]);
                uint4 *yp = reinterpret_cast<uint4 *>(y + ta * a.D + d0);
                const int ystep = a.D / C;  // one row, in 16-byte units
#pragma unroll
                for (int r = 0; r < TG; ++r) {
                    float cur[C], acc[C];
                    staged(ta + r, cur);
#pragma unroll
                    for (int c = 0; c < C; ++c) acc[c] = wt[KS - 1][c] * cur[c];
#pragma unroll
                    for (int i = 0; i < KS - 1; ++i)
#pragma unroll
                        for (int c = 0; c < C; ++c) acc[c] = fmaf(wt[i][c], win[i][c], acc[c]);
#pragma unroll
                    for (int c = 0; c < C; ++c) acc[c] = conv_act(acc[c], a.activation);
                    yp[r * ystep] = pack16(acc);
#pragma unroll
                    for (int i = 0; i + 1 < KS - 1; ++i)
#pragma unroll
                        for (int c = 0; c < C; ++c) win[i][c] = win[i + 1][c];
#pragma unroll
                    for (int c = 0; c < C; ++c) win[KS - 2][c] = cur[c];
                }
                if (a.fuse_final && tb > e - (KS - 1))
                    for (int64_t t = max(ta, e - (KS - 1)); t < tb; ++t) to_final(n, t, e, staged_raw(t), d0);
            } else {
#pragma unroll 1
                for (int64_t t = ta; t < tb; ++t) {
                    while (t >= e && n + 1 < a.n_seqs) {  // a new sequence starts here
                        ++n;
                        seq_range(a.cu_seqlens, a.n_seqs, a.total_tokens, n, s, e);
                    }
                    float acc[C];
#pragma unroll
                    for (int c = 0; c < C; ++c) acc[c] = 0.0f;
#pragma unroll
                    for (int i = 0; i < KS; ++i) {
                        const int64_t tau = t - (KS - 1) + i;
                        float v[C];
                        if (tau >= s && tau >= 0) staged(tau, v);
                        else history16<T, KS, C>(a, n, tau - s + (KS - 1), d0, v);
#pragma unroll
                        for (int c = 0; c < C; ++c) acc[c] = fmaf(wt[i][c], v[c], acc[c]);
                    }
#pragma unroll
                    for (int c = 0; c < C; ++c) acc[c] = conv_act(acc[c], a.activation);
                    *reinterpret_cast<uint4 *>(y + t * a.D + d0) = pack16(acc);
                    if (a.fuse_final) to_final(n, t, e, staged_raw(t), d0);
                }
            }
        } else if (active) {  // the copy never landed: mark this group's outputs
            float nan[C];
#pragma unroll
            for (int c = 0; c < C; ++c) nan[c] = __int_as_float(0x7fc00000);
            for (int64_t t = ta; t < tb; ++t) *reinterpret_cast<uint4 *>(y + t * a.D + d0) = pack16(nan);
        }
        __syncwarp();
        if ((tid & 31) == 0) mbar_arrive(&empty[stage]);  // this warp is done with the stage
        if (tid == 0 && !failed && k + S < n_local) {
            if (mbar_wait(&empty[stage], phase, 400000000LL)) {
                issue(k + S, stage);
                issued = k + S + 1;
            } else {
                failed = true;  // thread 0 stops fetching; its warp's later outputs become NaN
            }
        }
        failed = __shfl_sync(0xffffffffu, failed ? 1 : 0, 0) != 0 || failed;
        if (++stage == S) {
            stage = 0;
            phase ^= 1u;
        }
    }
    // let every fetch this CTA issued land before exiting (a no-op unless a
    // wait failed: a warp that consumed all items has seen them all land)
    if (tid == 0) {
        for (int64_t q = max(issued - S, (int64_t)0); q < issued; ++q)
            mbar_wait(&full[q % S], (uint32_t)((q / S) & 1), 400000000LL);
    }
}

// Final state of each sequence: its last ks - 1 inputs (reaching into the
// initial state when the sequence is shorter).  One thread owns all ks - 1
// rows of its 8 channels and reads them all before writing, so the state may
// be updated in place.
template <typename T, int KS>
__global__ void __launch_bounds__(kConvThreads) conv_final_state_kernel(const ConvArgs a) {
    const int chunks = a.D / 8;
    const int64_t total = (int64_t)a.n_seqs * chunks;
    const T *x = reinterpret_cast<const T *>(a.x);
    const T *init = reinterpret_cast<const T *>(a.initial_states);
    T *fin = reinterpret_cast<T *>(a.final_states);
    for (int64_t i = blockIdx.x * (int64_t)kConvThreads + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * kConvThreads) {
        const int n = (int)(i / chunks);
        const int d0 = (int)(i - (int64_t)n * chunks) * 8;
        int64_t s, e;
        seq_range(a.cu_seqlens, a.n_seqs, a.total_tokens, n, s, e);
        const int64_t slot = a.state_indices ? (int64_t)a.state_indices[n] : (int64_t)n;
        // a slot out of range, or a malformed range, leaves the state alone
        if (slot < 0 || slot >= a.n_slots || s < 0 || e < s || e > a.total_tokens) continue;
        const int64_t L = e - s;
        float rows[KS - 1][8];
#pragma unroll
        for (int r = 0; r < KS - 1; ++r) {
            const int64_t j = L + r;  // index into [history (ks - 1 rows) ; sequence]
            if (j >= KS - 1) {
                load8(x + (s + j - (KS - 1)) * a.D + d0, rows[r]);
            } else if (init) {
                load8(init + (slot * (KS - 1) + j) * a.D + d0, rows[r]);
            } else {
#pragma unroll
                for (int c = 0; c < 8; ++c) rows[r][c] = 0.0f;
            }
        }
#pragma unroll
        for (int r = 0; r < KS - 1; ++r) store8(fin + (slot * (KS - 1) + r) * a.D + d0, rows[r]);
    }
}

// One decode token per sequence: window = [state ; x], state shifted in place.
// One thread per (sequence, 8 channels): all window and weight loads are
// issued before the first use.
template <typename T, int KS>
__global__ void __launch_bounds__(kConvThreads)
    conv_update_kernel(const T *__restrict__ x, const T *__restrict__ w, T *__restrict__ y,
                       T *__restrict__ pool, const int32_t *__restrict__ state_indices,
                       int64_t n_slots, int N, int D, int activation) {
    const int chunks = D / 8;
    const int64_t total = (int64_t)N * chunks;
    for (int64_t i = blockIdx.x * (int64_t)kConvThreads + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * kConvThreads) {
        const int n = (int)(i / chunks);
        const int d0 = (int)(i - (int64_t)n * chunks) * 8;
        const int64_t slot = state_indices ? (int64_t)state_indices[n] : (int64_t)n;
        float acc[8];
        if (slot < 0 || slot >= n_slots) {  // invalid slot: NaN output, state untouched
#pragma unroll
            for (int c = 0; c < 8; ++c) acc[c] = __int_as_float(0x7fc00000);
            store8(y + (int64_t)n * D + d0, acc);
            continue;
        }
        T *st = pool + slot * (KS - 1) * (int64_t)D + d0;
        Row8<T> raw[KS], wr[KS];
#pragma unroll
        for (int r = 0; r < KS - 1; ++r) raw[r].load(st + (int64_t)r * D);
        raw[KS - 1].load(x + (int64_t)n * D + d0);
#pragma unroll
        for (int k = 0; k < KS; ++k) wr[k].load(w + (int64_t)k * D + d0);
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] = 0.0f;
#pragma unroll
        for (int k = 0; k < KS; ++k) {
            float v[8], wv[8];
            raw[k].to_f32(v);
            wr[k].to_f32(wv);
#pragma unroll
            for (int c = 0; c < 8; ++c) acc[c] = fmaf(wv[c], v[c], acc[c]);
            if (k > 0) store8(st + (int64_t)(k - 1) * D, v);  // shift the state by one row
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] = conv_act(acc[c], activation);
        store8(y + (int64_t)n * D + d0, acc);
    }
}

// S tokens per sequence (a speculative verify width): the window starts from
// the conv state in slot idx[n][a - 1] (a = the sequence's accepted count, 1
// without counts) and the state after token t goes to slot idx[n][t].  The
// start state is in registers before the first write, so it may be one of the
// destination slots.  A count outside [1, S] or a slot outside [0, n_slots)
// gives the sequence NaN outputs and leaves the pool untouched.
template <typename T, int KS>
__global__ void __launch_bounds__(kConvThreads)
    conv_multi_update_kernel(const T *__restrict__ x, const T *__restrict__ w, T *__restrict__ y,
                             T *__restrict__ pool, const int32_t *__restrict__ idx,
                             const int32_t *__restrict__ accepted, int64_t n_slots, int N, int S,
                             int D, int activation) {
    const int chunks = D / 8;
    const int64_t total = (int64_t)N * chunks;
    for (int64_t i = blockIdx.x * (int64_t)kConvThreads + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * kConvThreads) {
        const int n = (int)(i / chunks);
        const int d0 = (int)(i - (int64_t)n * chunks) * 8;
        const int32_t *sl = idx + (int64_t)n * S;
        const int a = accepted ? accepted[n] : 1;
        bool valid = a >= 1 && a <= S;
        for (int t = 0; t < S; ++t) valid = valid && sl[t] >= 0 && sl[t] < n_slots;
        if (!valid) {
            float nan8[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) nan8[c] = __int_as_float(0x7fc00000);
            for (int t = 0; t < S; ++t) store8(y + ((int64_t)n * S + t) * D + d0, nan8);
            continue;
        }
        Row8<T> raw[KS - 1], wr[KS];
        const T *st0 = pool + (int64_t)sl[a - 1] * (KS - 1) * D + d0;
#pragma unroll
        for (int r = 0; r < KS - 1; ++r) raw[r].load(st0 + (int64_t)r * D);
#pragma unroll
        for (int k = 0; k < KS; ++k) wr[k].load(w + (int64_t)k * D + d0);
        float win[KS - 1][8], wt[KS][8];
#pragma unroll
        for (int r = 0; r < KS - 1; ++r) raw[r].to_f32(win[r]);
#pragma unroll
        for (int k = 0; k < KS; ++k) wr[k].to_f32(wt[k]);
        for (int t = 0; t < S; ++t) {
            float cur[8], acc[8];
            load8(x + ((int64_t)n * S + t) * D + d0, cur);
#pragma unroll
            for (int c = 0; c < 8; ++c) acc[c] = 0.0f;
#pragma unroll
            for (int k = 0; k < KS - 1; ++k)  // oldest tap first, as the one-token update
#pragma unroll
                for (int c = 0; c < 8; ++c) acc[c] = fmaf(wt[k][c], win[k][c], acc[c]);
#pragma unroll
            for (int c = 0; c < 8; ++c) acc[c] = fmaf(wt[KS - 1][c], cur[c], acc[c]);
#pragma unroll
            for (int c = 0; c < 8; ++c) acc[c] = conv_act(acc[c], activation);
            store8(y + ((int64_t)n * S + t) * D + d0, acc);
#pragma unroll
            for (int k = 0; k + 1 < KS - 1; ++k)
#pragma unroll
                for (int c = 0; c < 8; ++c) win[k][c] = win[k + 1][c];
#pragma unroll
            for (int c = 0; c < 8; ++c) win[KS - 2][c] = cur[c];
            T *dst = pool + (int64_t)sl[t] * (KS - 1) * D + d0;
#pragma unroll
            for (int r = 0; r < KS - 1; ++r) store8(dst + (int64_t)r * D, win[r]);
        }
    }
}

template <int V_>
struct KsTag {
    static constexpr int value = V_;
};
// f(KsTag<ks>) for 2 <= ks <= 8 (validated by the caller)
template <typename F>
void dispatch_ks(int ks, F &&f) {
    switch (ks) {
        case 2: f(KsTag<2>{}); break;
        case 3: f(KsTag<3>{}); break;
        case 4: f(KsTag<4>{}); break;
        case 5: f(KsTag<5>{}); break;
        case 6: f(KsTag<6>{}); break;
        case 7: f(KsTag<7>{}); break;
        default: f(KsTag<8>{}); break;
    }
}

int grid_for(int64_t work) {
    return (int)std::min<int64_t>(std::max<int64_t>((work + kConvThreads - 1) / kConvThreads, 1), 152 * 32);
}

}  // namespace

cudaError_t launch_short_conv_prefill(const void *x, const void *weight, void *y,
                                      const int32_t *cu_seqlens, int n_seqs, int64_t total_tokens,
                                      int D, int ks, int activation, const void *initial_states,
                                      void *final_states, const int32_t *state_indices,
                                      int64_t n_slots, int dtype, cudaStream_t stream) {
    // the prefill kernel writes the final states itself unless they are the
    // initial states updated in place (every read of those must come first)
    const bool fuse = final_states && total_tokens > 0 && initial_states != final_states;
    ConvArgs a{x, weight, y, cu_seqlens, initial_states, final_states, state_indices,
               n_slots, total_tokens, n_seqs, D, ks, activation, fuse ? 1 : 0};
    if (total_tokens > 0) {
        auto go = [&](auto ks_tag) {
            constexpr int KS = decltype(ks_tag)::value;
            const int seg_ch = kSegThreads * (dtype == KDA_BF16 ? 8 : 4);
            constexpr int kPipeTile = pipe_tile<KS>();
            const int64_t items = (total_tokens + kPipeTile - 1) / kPipeTile * ((D + seg_ch - 1) / seg_ch);
            const int64_t per = (items + sm_count() - 1) / sm_count();
            const int grid = (int)((items + per - 1) / per);  // every CTA has items
            const int smem = pipe_smem<KS>();
            if (dtype == KDA_BF16) {
                auto kern = conv_prefill_kernel<__nv_bfloat16, KS>;
                cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
                kern<<<grid, kPipeThreads, smem, stream>>>(a);
            } else {
                auto kern = conv_prefill_kernel<float, KS>;
                cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
                kern<<<grid, kPipeThreads, smem, stream>>>(a);
            }
        };
        dispatch_ks(ks, go);
    }
    if (final_states && !fuse) {  // after the outputs: the initial state, updated in place
        const int grid = grid_for((int64_t)n_seqs * (D / 8));
        auto go = [&](auto ks_tag) {
            constexpr int KS = decltype(ks_tag)::value;
            if (dtype == KDA_BF16)
                conv_final_state_kernel<__nv_bfloat16, KS><<<grid, kConvThreads, 0, stream>>>(a);
            else
                conv_final_state_kernel<float, KS><<<grid, kConvThreads, 0, stream>>>(a);
        };
        dispatch_ks(ks, go);
    }
    return cudaGetLastError();
}

cudaError_t launch_short_conv_update(const void *x, const void *weight, void *y, void *pool,
                                     const int32_t *state_indices, int64_t n_slots, int N, int D,
                                     int ks, int activation, int dtype, cudaStream_t stream) {
    auto go = [&](auto ks_tag) {
        constexpr int KS = decltype(ks_tag)::value;
        const int grid = grid_for((int64_t)N * (D / 8));
        if (dtype == KDA_BF16)
            conv_update_kernel<__nv_bfloat16, KS><<<grid, kConvThreads, 0, stream>>>(
                (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)weight, (__nv_bfloat16 *)y,
                (__nv_bfloat16 *)pool, state_indices, n_slots, N, D, activation);
        else
            conv_update_kernel<float, KS><<<grid, kConvThreads, 0, stream>>>(
                (const float *)x, (const float *)weight, (float *)y, (float *)pool, state_indices,
                n_slots, N, D, activation);
    };
    dispatch_ks(ks, go);
    return cudaGetLastError();
}

cudaError_t launch_short_conv_multi_update(const void *x, const void *weight, void *y, void *pool,
                                           const int32_t *state_indices, const int32_t *num_accepted,
                                           int64_t n_slots, int N, int S, int D, int ks, int activation,
                                           int dtype, cudaStream_t stream) {
    const int grid = grid_for((int64_t)N * (D / 8));
    auto go = [&](auto ks_tag) {
        constexpr int KS = decltype(ks_tag)::value;
        if (dtype == KDA_BF16)
            conv_multi_update_kernel<__nv_bfloat16, KS><<<grid, kConvThreads, 0, stream>>>(
                (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)weight, (__nv_bfloat16 *)y,
                (__nv_bfloat16 *)pool, state_indices, num_accepted, n_slots, N, S, D, activation);
        else
            conv_multi_update_kernel<float, KS><<<grid, kConvThreads, 0, stream>>>(
                (const float *)x, (const float *)weight, (float *)y, (float *)pool, state_indices,
                num_accepted, n_slots, N, S, D, activation);
    };
    dispatch_ks(ks, go);
    return cudaGetLastError();
}

}  // namespace kda
