// Decode step of Kimi Delta Attention on a pooled fp32 state, in place.
//
// One token per sequence (Ascend model file, KimiDeltaAttention._decode_gdr
// and _decode_fused_kda; nnterp "kimi_linear" page, the token-by-token form).
// For each (sequence n, head h) and each state row v (the pool stores S^T,
// [V][K], key dim contiguous):
//
//   s      = S^T[v, :] * exp(g)                 decayed row
//   a      = s . k_hat,   b = s . q_hat          (q_hat carries the scale)
//   u      = beta * (v_v - a)
//   S^T[v] = s + u * k_hat                       written back
//   o_v    = b + u * (k_hat . q_hat)            = (S_new^T q_hat)_v
//
// The state is streamed once in and once out (HBM bound): each warp owns
// whole 512-byte rows, a lane holds 4 consecutive key channels (one 128-bit
// load and one 128-bit store per lane per row), and the two dot products per
// row are summed over the lanes (for a whole head per CTA, all of a warp's
// rows at once by one reduce-scatter; see whole_head_token).  Rows of one head
// are split over CTAs when there are too few (sequence, head) pairs to fill
// the GPU.  The gated variant activates the model's raw gate and beta on the
// way in (see GateArgs); the epilogue variant (one CTA per head) normalises
// each head's output row and applies the output gate before storing it (see
// EpiArgs).
#include <string.h>

#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kDecodeThreads = 256;  // 8 warps
constexpr int kWarps = kDecodeThreads / 32;
constexpr int kMaxRowsPerWarp = kHeadDim / kWarps;  // 16: a whole head per CTA
constexpr int kTokBlk = 8;  // speculative decode: tokens per block of gate tables
constexpr int kTabPer = kTokBlk * kHeadDim / kDecodeThreads;  // table entries per thread

// One butterfly level of a reduce-scatter over the warp: a lane holding N
// partial sums passes the half its partner keeps (across lane bit N/2) and
// adds the partner's share of the half it keeps.
template <int N>
__device__ __forceinline__ void scatter_level(float (&p)[16], int lane) {
    constexpr int M = N / 2;
    const bool hi = (lane & M) != 0;
#pragma unroll
    for (int i = 0; i < M; ++i) {
        const float send = hi ? p[i] : p[i + M];
        const float keep = hi ? p[i + M] : p[i];
        p[i] = keep + __shfl_xor_sync(0xffffffffu, send, M);
    }
}

// One token's update of a warp's 16 state rows when its CTA holds a whole
// head (row j of the warp is head row warp + 8 j; dst points at lane's four
// key channels of row 0 in the destination).  The 32 dot products of the
// rows, a_j = s_j . k_hat and c_j = s_j . q_hat, are summed over the lanes by
// a reduce-scatter: at each butterfly level a lane keeps half of its partial
// sums and hands the other half to its partner, so lane l ends with the whole
// sum of product l (a_l below 16, c_{l-16} above) after 31 shuffles, where
// one lane-wide reduction per product takes 160.  Returns u_j on lane j < 16
// and o_j = c_j + u_j (k_hat . q_hat) on lane 16 + j.
__device__ __forceinline__ float whole_head_token(float4 (&s)[kMaxRowsPerWarp], float4 dec,
                                                  float4 kh, float4 qh, float kq, float b,
                                                  float vrow, float *dst, int lane) {
    float p[16];
    const bool hi = (lane & 16) != 0;  // the first level pairs a_j with c_j of the same row
#pragma unroll
    for (int j = 0; j < kMaxRowsPerWarp; ++j) {
        float4 x = s[j];
        x.x *= dec.x; x.y *= dec.y; x.z *= dec.z; x.w *= dec.w;
        s[j] = x;
        const float a = x.x * kh.x + x.y * kh.y + x.z * kh.z + x.w * kh.w;
        const float c = x.x * qh.x + x.y * qh.y + x.z * qh.z + x.w * qh.w;
        p[j] = (hi ? c : a) + __shfl_xor_sync(0xffffffffu, hi ? a : c, 16);
    }
    scatter_level<16>(p, lane);
    scatter_level<8>(p, lane);
    scatter_level<4>(p, lane);
    scatter_level<2>(p, lane);
    const float u = b * (vrow - p[0]);  // lanes 0-15 (vrow: v of row `lane`)
    const float uo = __shfl_sync(0xffffffffu, u, lane & 15);
#pragma unroll
    for (int j = 0; j < kMaxRowsPerWarp; ++j) {
        const float uj = __shfl_sync(0xffffffffu, u, j);
        float4 x = s[j];
        x.x += uj * kh.x; x.y += uj * kh.y; x.z += uj * kh.z; x.w += uj * kh.w;
        s[j] = x;
        *reinterpret_cast<float4 *>(dst + (int64_t)(kWarps * j) * kHeadDim) = x;
    }
    return hi ? p[0] + uo * kq : u;
}

// One token per sequence (the common decode step).
template <typename T, bool GATED, bool EPI>
__global__ void __launch_bounds__(kDecodeThreads, 2)
    recurrent_step_kernel(const T *__restrict__ q, const T *__restrict__ k,
                          const T *__restrict__ v, const float *__restrict__ g,
                          const float *__restrict__ beta, const GateArgs gate, const EpiArgs epi,
                          float *__restrict__ pool, const int32_t *__restrict__ state_indices,
                          int64_t n_slots, T *__restrict__ o, int H, int rows_per_cta,
                          float scale) {
    __shared__ float s_part[kWarps];  // epilogue: per-warp sums of o^2
    const int pair = blockIdx.x;  // n * H + h
    const int n = pair / H;
    const int h = pair - n * H;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int row0 = blockIdx.y * rows_per_cta;
    const int rpw = rows_per_cta / kWarps;  // rows of this warp: row0 + warp + 8 j

    const int64_t slot = state_indices ? (int64_t)state_indices[n] : (int64_t)n;
    const int64_t io_k = (int64_t)pair * kHeadDim;  // offset of q/k/g/v/o rows of (n, h)

    if (slot < 0 || slot >= n_slots) {
        // invalid slot: the pool is not touched and this head's output is NaN
        for (int r = threadIdx.x; r < rows_per_cta; r += kDecodeThreads)
            o[io_k + row0 + r] = from_f32<T>(__int_as_float(0x7fc00000));
        return;
    }

    // The token's inputs are requested before the state rows, so that the
    // decays and norms are ready when the rows arrive; lane j fetches v of the
    // warp's row j.
    const float4 q4 = load4(q + io_k + 4 * lane);
    const float4 k4 = load4(k + io_k + 4 * lane);
    float4 g4, r4, c4;
    float braw, gs = 0.0f;
    if (GATED) {
        r4 = load4(reinterpret_cast<const T *>(gate.raw_gate) + io_k + 4 * lane);
        c4 = load4(gate.dt_bias + (int64_t)h * kHeadDim + 4 * lane);
        gs = expf(gate.a_log[h]);
        braw = to_f32(reinterpret_cast<const T *>(gate.raw_beta)[pair]);
    } else {
        g4 = load4(g + io_k + 4 * lane);
        braw = beta[pair];
    }
    const float vrow = lane < rpw ? to_f32(v[io_k + row0 + warp + kWarps * lane]) : 0.0f;
    float gate_o = 0.0f, w_o = 0.0f;  // epilogue: output gate and norm weight of row `lane`
    if (EPI && lane < rpw) {
        const int r = row0 + warp + kWarps * lane;
        gate_o = to_f32(reinterpret_cast<const T *>(epi.out_gate)[io_k + r]);
        w_o = epi.weight[r];
    }
    float *S = pool + ((slot * H + h) * (int64_t)kHeadDim) * kHeadDim;  // [V][K] of (slot, h)
    float4 s[kMaxRowsPerWarp];
#pragma unroll
    for (int j = 0; j < kMaxRowsPerWarp; ++j)
        if (j < rpw)
            s[j] = *reinterpret_cast<const float4 *>(S + (int64_t)(row0 + warp + kWarps * j) * kHeadDim + 4 * lane);

    // L2 norms of q and k over the key dim (eps inside the root), scale on q.
    float b;
    if (GATED) {
        const bool lb = gate.use_lower_bound != 0;
        g4 = make_float4(gate_decay(r4.x + c4.x, gs, gate.lower_bound, lb),
                         gate_decay(r4.y + c4.y, gs, gate.lower_bound, lb),
                         gate_decay(r4.z + c4.z, gs, gate.lower_bound, lb),
                         gate_decay(r4.w + c4.w, gs, gate.lower_bound, lb));
        b = gate_beta(braw);
    } else {
        b = braw;
    }
    const float sq = warp_sum(q4.x * q4.x + q4.y * q4.y + q4.z * q4.z + q4.w * q4.w);
    const float sk = warp_sum(k4.x * k4.x + k4.y * k4.y + k4.z * k4.z + k4.w * k4.w);
    const float rq = scale / sqrtf(sq + 1e-6f);
    const float rk = 1.0f / sqrtf(sk + 1e-6f);
    const float4 qh = make_float4(q4.x * rq, q4.y * rq, q4.z * rq, q4.w * rq);
    const float4 kh = make_float4(k4.x * rk, k4.y * rk, k4.z * rk, k4.w * rk);
    const float4 dec = make_float4(expf(g4.x), expf(g4.y), expf(g4.z), expf(g4.w));
    const float kq = warp_sum(kh.x * qh.x + kh.y * qh.y + kh.z * qh.z + kh.w * qh.w);

    float my_o = 0.0f, ss = 0.0f;  // epilogue: o of row `lane`, sum of o^2 over the warp's rows
    if (rpw == kMaxRowsPerWarp) {
        const float ov = whole_head_token(s, dec, kh, qh, kq, b, vrow,
                                          S + (int64_t)(row0 + warp) * kHeadDim + 4 * lane, lane);
        if (EPI) {
            my_o = __shfl_sync(0xffffffffu, ov, (lane & 15) + 16);  // lanes 0-15: o of row `lane`
            ss = warp_sum(lane < 16 ? my_o * my_o : 0.0f);
        } else if (lane >= 16) {
            o[io_k + row0 + warp + kWarps * (lane - 16)] = from_f32<T>(ov);
        }
    } else {
#pragma unroll
        for (int j = 0; j < kMaxRowsPerWarp; ++j) {
            if (j >= rpw) break;
            const int r = row0 + warp + kWarps * j;
            float4 x = s[j];
            x.x *= dec.x; x.y *= dec.y; x.z *= dec.z; x.w *= dec.w;
            float a = x.x * kh.x + x.y * kh.y + x.z * kh.z + x.w * kh.w;
            float c = x.x * qh.x + x.y * qh.y + x.z * qh.z + x.w * qh.w;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                a += __shfl_xor_sync(0xffffffffu, a, off);
                c += __shfl_xor_sync(0xffffffffu, c, off);
            }
            const float u = b * (__shfl_sync(0xffffffffu, vrow, j) - a);
            x.x += u * kh.x; x.y += u * kh.y; x.z += u * kh.z; x.w += u * kh.w;
            *reinterpret_cast<float4 *>(S + (int64_t)r * kHeadDim + 4 * lane) = x;
            const float ov = c + u * kq;
            if (EPI) {
                ss = fmaf(ov, ov, ss);
                if (lane == j) my_o = ov;
            } else if (lane == 0) {
                o[io_k + r] = from_f32<T>(ov);
            }
        }
    }
    if (EPI) {  // rows_per_cta == 128: this CTA holds the head's whole output row
        if (lane == 0) s_part[warp] = ss;
        __syncthreads();
        float tot = 0.0f;
#pragma unroll
        for (int w2 = 0; w2 < kWarps; ++w2) tot += s_part[w2];
        const float rn = 1.0f / sqrtf(tot * (1.0f / kHeadDim) + epi.eps);
        if (lane < rpw)
            o[io_k + row0 + warp + kWarps * lane] = from_f32<T>(my_o * rn * w_o * gate_beta(gate_o));
    }
}

// Speculative decode: S tokens per sequence, per-token destination slots,
// the starting slot picked by the accepted count (see launch_recurrent_step).
template <typename T, bool GATED, bool EPI>
__global__ void __launch_bounds__(kDecodeThreads, 2)
    recurrent_multi_step_kernel(const T *__restrict__ q, const T *__restrict__ k,
                                const T *__restrict__ v, const float *__restrict__ g,
                                const float *__restrict__ beta, const GateArgs gate,
                                const EpiArgs epi, float *__restrict__ pool,
                                const int32_t *__restrict__ state_indices,
                                const int32_t *__restrict__ num_accepted, int64_t n_slots,
                                T *__restrict__ o, int S, int H, int rows_per_cta, float scale) {
    // Tokens go in blocks of up to kTokBlk.  At the start of a block the CTA
    // activates the block's raw gates (GATED: e^g of every key channel) and
    // output gates (EPI: sigmoid) into shared tables, behind one barrier; the
    // tokens then run without a barrier, the epilogue keeping each token's raw
    // output row and per-warp sums of o^2 in shared memory until the block's
    // end, where one barrier lets the CTA finish the block's rows.
    __shared__ __align__(16) float s_dec[GATED ? kTokBlk : 1][kHeadDim];
    __shared__ float s_og[EPI ? kTokBlk : 1][kHeadDim];    // sigmoid(out_gate)
    __shared__ float s_o[EPI ? kTokBlk : 1][kHeadDim];     // o before the epilogue
    __shared__ float s_part[EPI ? kTokBlk : 1][kWarps];    // per-warp sums of o^2
    const int pair = blockIdx.x;  // n * H + h
    const int n = pair / H;
    const int h = pair - n * H;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int row0 = blockIdx.y * rows_per_cta;
    const int rpw = rows_per_cta / kWarps;  // rows of this warp: row0 + warp + 8 j
    // token t of sequence n, head h: q/k/g/v/o rows at ((n S + t) H + h) * K
    auto io_of = [&](int t) { return ((int64_t)(n * S + t) * H + h) * kHeadDim; };
    auto slot_of = [&](int t) {  // the slot the state after token t goes to
        return state_indices ? (int64_t)state_indices[(int64_t)n * S + t] : (int64_t)n;
    };

    // Every slot of the sequence, and the number of accepted tokens, is checked
    // before anything is written.
    const int acc = num_accepted ? num_accepted[n] : 1;
    bool valid = acc >= 1 && acc <= S;
    for (int t = 0; t < S && valid; ++t) {
        const int64_t sl = slot_of(t);
        valid = sl >= 0 && sl < n_slots;
    }
    if (!valid) {
        // the pool is not touched and this head's outputs are NaN
        for (int t = 0; t < S; ++t)
            for (int r = threadIdx.x; r < rows_per_cta; r += kDecodeThreads)
                o[io_of(t) + row0 + r] = from_f32<T>(__int_as_float(0x7fc00000));
        return;
    }
    const int64_t slot_in = slot_of(acc - 1);

    // The raw gates of a block of tokens (kTabPer entries of the tables per
    // thread), and their activation into the tables.
    struct TabIn {
        float gx[kTabPer];  // GATED: raw gate + dt_bias
        float og[kTabPer];  // EPI: raw output gate
    };
    auto tab_load = [&](int t0, int nb) {
        TabIn in;
#pragma unroll
        for (int u = 0; u < kTabPer; ++u) {
            const int i = threadIdx.x + u * kDecodeThreads;
            in.gx[u] = 0.0f;
            in.og[u] = 0.0f;
            if (i < nb * kHeadDim) {
                const int tt = i / kHeadDim, c = i % kHeadDim;
                const int64_t e = io_of(t0 + tt) + c;
                if (GATED)
                    in.gx[u] = to_f32(reinterpret_cast<const T *>(gate.raw_gate)[e]) +
                               gate.dt_bias[(int64_t)h * kHeadDim + c];
                if (EPI) in.og[u] = to_f32(reinterpret_cast<const T *>(epi.out_gate)[e]);
            }
        }
        return in;
    };
    auto tab_store = [&](const TabIn &in, int nb, float gscale) {
#pragma unroll
        for (int u = 0; u < kTabPer; ++u) {
            const int i = threadIdx.x + u * kDecodeThreads;
            if (i < nb * kHeadDim) {
                const int tt = i / kHeadDim, c = i % kHeadDim;
                if (GATED)
                    s_dec[GATED ? tt : 0][c] =
                        expf(gate_decay(in.gx[u], gscale, gate.lower_bound, gate.use_lower_bound != 0));
                if (EPI) s_og[EPI ? tt : 0][c] = gate_beta(in.og[u]);
            }
        }
    };
    // The first block's raw gates are requested before the state, so that the
    // tables are in place (behind the block's barrier) while the state rows
    // are still on their way.
    TabIn tab;
    if (GATED || EPI) tab = tab_load(0, min(kTokBlk, S));

    // This warp's state rows; they stay in registers across the tokens.
    const float *S0 = pool + ((slot_in * H + h) * (int64_t)kHeadDim) * kHeadDim;  // [V][K]
    float4 s[kMaxRowsPerWarp];
#pragma unroll
    for (int j = 0; j < kMaxRowsPerWarp; ++j)
        if (j < rpw)
            s[j] = *reinterpret_cast<const float4 *>(S0 + (int64_t)(row0 + warp + kWarps * j) * kHeadDim + 4 * lane);

    // A token's inputs, fetched one token ahead so that their latency overlaps
    // the previous token's row updates.
    struct TokIn {
        float4 q4, k4, g4;  // g4: g (not GATED)
        float vrow, b;      // vrow: v of the warp's row `lane`; b: beta (raw when GATED)
    };
    auto fetch = [&](int t) {
        TokIn in;
        const int64_t io_k = io_of(t);
        const int64_t pt = (int64_t)(n * S + t) * H + h;  // beta / raw beta index
        in.vrow = lane < rpw ? to_f32(v[io_k + row0 + warp + kWarps * lane]) : 0.0f;
        in.q4 = load4(q + io_k + 4 * lane);
        in.k4 = load4(k + io_k + 4 * lane);
        if (GATED) {
            in.b = to_f32(reinterpret_cast<const T *>(gate.raw_beta)[pt]);
        } else {
            in.g4 = load4(g + io_k + 4 * lane);
            in.b = beta[pt];
        }
        return in;
    };
    TokIn nxt = fetch(0);
    const float gscale = GATED ? expf(gate.a_log[h]) : 0.0f;
    for (int t0 = 0; t0 < S; t0 += kTokBlk) {
        const int nb = min(kTokBlk, S - t0);
        if (GATED || EPI) {  // the tables of tokens t0 .. t0 + nb - 1
            if (t0 > 0) {
                __syncthreads();  // every thread is done with the previous block's tables
                tab = tab_load(t0, nb);
            }
            tab_store(tab, nb, gscale);
            __syncthreads();
        }
        for (int tt = 0; tt < nb; ++tt) {
            const int t = t0 + tt;
            const TokIn cur = nxt;
            if (t + 1 < S) nxt = fetch(t + 1);
            const int64_t io_k = io_of(t);
            const float vrow = cur.vrow;
            const float4 q4 = cur.q4, k4 = cur.k4;
            float4 dec;
            float b;
            if (GATED) {
                dec = *reinterpret_cast<const float4 *>(&s_dec[GATED ? tt : 0][4 * lane]);
                b = gate_beta(cur.b);
            } else {
                dec = make_float4(expf(cur.g4.x), expf(cur.g4.y), expf(cur.g4.z), expf(cur.g4.w));
                b = cur.b;
            }
            const float sq = warp_sum(q4.x * q4.x + q4.y * q4.y + q4.z * q4.z + q4.w * q4.w);
            const float sk = warp_sum(k4.x * k4.x + k4.y * k4.y + k4.z * k4.z + k4.w * k4.w);
            const float rq = scale / sqrtf(sq + 1e-6f);
            const float rk = 1.0f / sqrtf(sk + 1e-6f);
            const float4 qh = make_float4(q4.x * rq, q4.y * rq, q4.z * rq, q4.w * rq);
            const float4 kh = make_float4(k4.x * rk, k4.y * rk, k4.z * rk, k4.w * rk);
            const float kq = warp_sum(kh.x * qh.x + kh.y * qh.y + kh.z * qh.z + kh.w * qh.w);

            float *Sd = pool + ((slot_of(t) * H + h) * (int64_t)kHeadDim) * kHeadDim;  // destination
            if (rpw == kMaxRowsPerWarp) {
                const float ov = whole_head_token(s, dec, kh, qh, kq, b, vrow,
                                                  Sd + (int64_t)(row0 + warp) * kHeadDim + 4 * lane, lane);
                if (EPI) {  // rows_per_cta == 128: this CTA holds the head's whole output row
                    const float my_o = __shfl_sync(0xffffffffu, ov, (lane & 15) + 16);  // o of row `lane`
                    const float ss = warp_sum(lane < 16 ? my_o * my_o : 0.0f);
                    if (lane < 16) s_o[EPI ? tt : 0][warp + kWarps * lane] = my_o;
                    if (lane == 0) s_part[EPI ? tt : 0][warp] = ss;
                } else if (lane >= 16) {
                    o[io_k + row0 + warp + kWarps * (lane - 16)] = from_f32<T>(ov);
                }
                continue;
            }
#pragma unroll
            for (int j = 0; j < kMaxRowsPerWarp; ++j) {  // (never with the epilogue)
                if (j >= rpw) break;
                const int r = row0 + warp + kWarps * j;
                float4 x = s[j];
                x.x *= dec.x; x.y *= dec.y; x.z *= dec.z; x.w *= dec.w;
                float a = x.x * kh.x + x.y * kh.y + x.z * kh.z + x.w * kh.w;
                float c = x.x * qh.x + x.y * qh.y + x.z * qh.z + x.w * qh.w;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    a += __shfl_xor_sync(0xffffffffu, a, off);
                    c += __shfl_xor_sync(0xffffffffu, c, off);
                }
                const float u = b * (__shfl_sync(0xffffffffu, vrow, j) - a);
                x.x += u * kh.x; x.y += u * kh.y; x.z += u * kh.z; x.w += u * kh.w;
                s[j] = x;
                *reinterpret_cast<float4 *>(Sd + (int64_t)r * kHeadDim + 4 * lane) = x;
                if (lane == 0) o[io_k + r] = from_f32<T>(c + u * kq);
            }
        }
        if (EPI) {  // the block's output rows, normalised and gated
            __syncthreads();
            for (int i = threadIdx.x; i < nb * kHeadDim; i += kDecodeThreads) {
                const int tt = i / kHeadDim, r = i % kHeadDim;
                float tot = 0.0f;
#pragma unroll
                for (int w2 = 0; w2 < kWarps; ++w2) tot += s_part[EPI ? tt : 0][w2];
                const float rn = 1.0f / sqrtf(tot * (1.0f / kHeadDim) + epi.eps);
                o[io_of(t0 + tt) + r] =
                    from_f32<T>(s_o[EPI ? tt : 0][r] * rn * epi.weight[r] * s_og[EPI ? tt : 0][r]);
            }
        }
    }
}

}  // namespace

struct StepLaunch {
    dim3 grid;
    const void *q, *k, *v;
    const float *g, *beta;
    GateArgs gate;
    EpiArgs epi;
    float *pool;
    const int32_t *state_indices, *num_accepted;
    int64_t n_slots;
    void *o;
    int S, H, rows;
    float scale;
    cudaStream_t stream;
};

template <typename T, bool GATED, bool EPI>
void launch_step3(const StepLaunch &a) {
    if (a.S == 1 && !a.num_accepted)
        recurrent_step_kernel<T, GATED, EPI><<<a.grid, kDecodeThreads, 0, a.stream>>>(
            (const T *)a.q, (const T *)a.k, (const T *)a.v, a.g, a.beta, a.gate, a.epi, a.pool,
            a.state_indices, a.n_slots, (T *)a.o, a.H, a.rows, a.scale);
    else
        recurrent_multi_step_kernel<T, GATED, EPI><<<a.grid, kDecodeThreads, 0, a.stream>>>(
            (const T *)a.q, (const T *)a.k, (const T *)a.v, a.g, a.beta, a.gate, a.epi, a.pool,
            a.state_indices, a.num_accepted, a.n_slots, (T *)a.o, a.S, a.H, a.rows, a.scale);
}

template <typename T>
void launch_step(bool gated, bool epi_on, const StepLaunch &a) {
    if (gated) {
        if (epi_on) launch_step3<T, true, true>(a);
        else launch_step3<T, true, false>(a);
    } else {
        if (epi_on) launch_step3<T, false, true>(a);
        else launch_step3<T, false, false>(a);
    }
}

cudaError_t launch_recurrent_step(const void *q, const void *k, const void *v, const float *g,
                                  const float *beta, const GateArgs *gate, const EpiArgs *epi,
                                  float *pool, const int32_t *state_indices,
                                  const int32_t *num_accepted, int64_t n_slots, void *o, int N,
                                  int S, int H, float scale, int dtype, cudaStream_t stream) {
    const int64_t pairs = (int64_t)N * H;
    // Split a head's 128 rows over more CTAs when there are few heads in flight,
    // so that at least ~4 CTAs per SM are resident.
    int rows = kHeadDim;  // a multiple of 8 warps, at most 16 rows per warp
    const bool epi_on = epi && epi->out_gate;
    while (!epi_on && rows > 16 && pairs * (kHeadDim / rows) < 152 * 8) rows >>= 1;
    const dim3 grid((unsigned)pairs, kHeadDim / rows);
    StepLaunch a;
    memset(&a, 0, sizeof(a));
    a.grid = grid;
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta;
    if (gate) a.gate = *gate;
    if (epi_on) a.epi = *epi;
    a.pool = pool;
    a.state_indices = state_indices;
    a.num_accepted = num_accepted;
    a.n_slots = n_slots;
    a.o = o;
    a.S = S; a.H = H; a.rows = rows;
    a.scale = scale;
    a.stream = stream;
    if (dtype == KDA_BF16) launch_step<__nv_bfloat16>(gate != nullptr, epi_on, a);
    else launch_step<float>(gate != nullptr, epi_on, a);
    return cudaGetLastError();
}

}  // namespace kda
