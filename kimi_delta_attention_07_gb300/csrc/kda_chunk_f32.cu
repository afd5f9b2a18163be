// fp32 CUDA-core chunked KDA: the precise path (fp32 inputs, or bf16 inputs
// with KDA_CHUNK_PRECISE).
//
// Chunked form of the Ascend model file's _torch_chunk_kda, split in two
// kernels around a per-(chunk, head) record in the workspace:
//
//   prep (parallel over chunks x heads):
//     q_hat = scale * l2norm(q), k_hat = l2norm(k)           (fp32)
//     G     = cumulative sum of g inside the chunk, per key channel
//     L[r,j] = beta_r sum_d k_hat[r,d] k_hat[j,d] exp(G[r,d]-G[j,d]),   j < r
//     A[r,j] =        sum_d q_hat[r,d] k_hat[j,d] exp(G[r,d]-G[j,d]),   j <= r
//     X = (I + L)^-1 by forward substitution;  T = X diag(beta)
//     W = T (exp(G) * k_hat),  U = T v,  QG = q_hat * exp(G),
//     KD = k_hat * exp(G_last - G),  gC = exp(G_last)
//   scan (sequential over the chunks of a sequence; parallel over sequences,
//   heads and 32-wide blocks of value columns):
//     Vn = U - W S;   o = QG S + A Vn;   S = diag(gC) S + KD^T Vn
//
// Every exponent above is <= 0 (G is non-increasing when g <= 0), so no
// factorisation into exp(+G) * exp(-G) is used here: the pairwise
// exponentials are taken directly, which keeps this path exact in fp32 for
// any decay.  Padded tail rows carry q = k = v = 0, g = 0, beta = 0 and so
// change nothing.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int C = kChunk;     // 64
constexpr int D = kHeadDim;   // 128 (K = V)
constexpr int DP = D + 1;     // padded row stride of [64][128] tiles in shared memory
constexpr int CP = C + 1;     // padded row stride of [64][64] tiles
constexpr int BV = 32;        // value columns per scan CTA
constexpr int BVP = BV + 1;

// ---------------------------------------------------------------------------
// prep
// ---------------------------------------------------------------------------
constexpr size_t kPrepSmemFloats = 3 * C * DP + 2 * C * CP + C;

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
    chunk_prep_f32_kernel(const T *__restrict__ q, const T *__restrict__ k,
                          const T *__restrict__ v, const float *__restrict__ g,
                          const float *__restrict__ beta, int n_seqs, int H, float scale,
                          void *workspace, WsLayout L) {
    extern __shared__ float smem[];
    float *sQ = smem;              // [C][DP] q_hat (later: v)
    float *sK = sQ + C * DP;       // [C][DP] k_hat (later: exp(G) k_hat)
    float *sG = sK + C * DP;       // [C][DP] g, then G
    float *sL = sG + C * DP;       // [C][CP] L (strictly lower, beta-scaled rows)
    float *sX = sL + C * CP;       // [C][CP] X = (I + L)^-1, then T
    float *sB = sX + C * CP;       // [C] beta

    const int32_t *chunk_off = ws_at<const int32_t>(workspace, L.chunk_off_off);
    const int c = blockIdx.x, h = blockIdx.y;
    if (c >= chunk_off[n_seqs]) return;
    const int n = owner_of_chunk(chunk_off, n_seqs, c);
    const int j_in_seq = c - chunk_off[n];
    const int64_t tok0 = (int64_t)ws_at<const int32_t>(workspace, L.seq_start_off)[n] + (int64_t)j_in_seq * C;
    const int valid = min(C, ws_at<const int32_t>(workspace, L.seq_len_off)[n] - j_in_seq * C);
    float *rec = ws_at<float>(workspace, L.records_off + ((size_t)c * H + h) * F32Rec::bytes);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // 1. load rows, L2-normalise q and k (eps inside the root), scale q.
    for (int r = warp; r < C; r += kThreads / 32) {
        float4 q4 = make_float4(0, 0, 0, 0), k4 = q4, g4 = q4;
        if (r < valid) {
            const int64_t off = ((tok0 + r) * H + h) * (int64_t)D + 4 * lane;
            q4 = load4(q + off);
            k4 = load4(k + off);
            g4 = load4(g + off);
        }
        const float sq = warp_sum(q4.x * q4.x + q4.y * q4.y + q4.z * q4.z + q4.w * q4.w);
        const float sk = warp_sum(k4.x * k4.x + k4.y * k4.y + k4.z * k4.z + k4.w * k4.w);
        const float rq = scale / sqrtf(sq + 1e-6f), rk = 1.0f / sqrtf(sk + 1e-6f);
        float *dq = sQ + r * DP + 4 * lane, *dk = sK + r * DP + 4 * lane, *dg = sG + r * DP + 4 * lane;
        dq[0] = q4.x * rq; dq[1] = q4.y * rq; dq[2] = q4.z * rq; dq[3] = q4.w * rq;
        dk[0] = k4.x * rk; dk[1] = k4.y * rk; dk[2] = k4.z * rk; dk[3] = k4.w * rk;
        dg[0] = g4.x; dg[1] = g4.y; dg[2] = g4.z; dg[3] = g4.w;
    }
    if (tid < C) sB[tid] = tid < valid ? beta[(tok0 + tid) * H + h] : 0.0f;
    __syncthreads();

    // 2. cumulative log-decay per key channel.
    if (tid < D) {
        float run = 0.0f;
        for (int r = 0; r < C; ++r) {
            run += sG[r * DP + tid];
            sG[r * DP + tid] = run;
        }
    }
    __syncthreads();

    // 3. L (strictly lower, rows scaled by beta) and A (lower, diagonal kept),
    //    over the 16x16 tiles on or below the diagonal.
    float *gA = rec + F32Rec::A;
    {
        const int tr = tid >> 4, tj = tid & 15;
        for (int br = 0; br < 4; ++br) {
            for (int bj = 0; bj < 4; ++bj) {
                const int r = 16 * br + tr, j = 16 * bj + tj;
                float accL = 0.0f, accA = 0.0f;
                if (bj <= br && j <= r) {
                    const float *kr = sK + r * DP, *qr = sQ + r * DP, *gr = sG + r * DP;
                    const float *kj = sK + j * DP, *gj = sG + j * DP;
#pragma unroll 8
                    for (int d = 0; d < D; ++d) {
                        const float e = __expf(gr[d] - gj[d]) * kj[d];
                        accL = fmaf(kr[d], e, accL);
                        accA = fmaf(qr[d], e, accA);
                    }
                }
                sL[r * CP + j] = (j < r) ? sB[r] * accL : 0.0f;
                gA[r * C + j] = (j <= r) ? accA : 0.0f;
            }
        }
    }
    __syncthreads();

    // 4. X = (I + L)^-1, row by row: X[r,:] = e_r - sum_{m<r} L[r,m] X[m,:].
    //    Thread (col, part) sums the m = part (mod 4) terms of column col.
    {
        const int col = tid >> 2, part = tid & 3;
        for (int r = 0; r < C; ++r) {
            float acc = 0.0f;
            for (int m = col + part; m < r; m += 4) acc = fmaf(sL[r * CP + m], sX[m * CP + col], acc);
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            if (part == 0) sX[r * CP + col] = (col == r) ? 1.0f : (col < r ? -acc : 0.0f);
            __syncthreads();
        }
        // T = X diag(beta)
        for (int i = tid; i < C * C; i += kThreads) {
            const int r = i / C, cc = i % C;
            sX[r * CP + cc] *= sB[cc];
        }
    }

    // 5. QG, KD, gC to the record; replace k_hat by exp(G) k_hat for W.
    {
        float *gQG = rec + F32Rec::QG, *gKD = rec + F32Rec::KD, *gGC = rec + F32Rec::GC;
        const float *Glast = sG + (C - 1) * DP;
        for (int i = tid; i < C * D; i += kThreads) {
            const int r = i / D, d = i % D;
            const float G = sG[r * DP + d];
            const float kh = sK[r * DP + d];
            gQG[i] = sQ[r * DP + d] * __expf(G);
            gKD[i] = kh * __expf(Glast[d] - G);
            sK[r * DP + d] = kh * __expf(G);
        }
        if (tid < D) gGC[tid] = __expf(Glast[tid]);
    }
    __syncthreads();

    // 6. v rows into sQ (q_hat no longer needed).
    for (int r = warp; r < C; r += kThreads / 32) {
        float4 v4 = make_float4(0, 0, 0, 0);
        if (r < valid) v4 = load4(v + ((tok0 + r) * H + h) * (int64_t)D + 4 * lane);
        float *dv = sQ + r * DP + 4 * lane;
        dv[0] = v4.x; dv[1] = v4.y; dv[2] = v4.z; dv[3] = v4.w;
    }
    __syncthreads();

    // 7. W = T (exp(G) k_hat), U = T v  (T lower triangular).
    {
        float *gW = rec + F32Rec::W, *gU = rec + F32Rec::U;
        const int d = tid & (D - 1);
        for (int r = tid >> 7; r < C; r += kThreads / D) {
            float w = 0.0f, u = 0.0f;
            const float *tr = sX + r * CP;
            for (int j = 0; j <= r; ++j) {
                const float t = tr[j];
                w = fmaf(t, sK[j * DP + d], w);
                u = fmaf(t, sQ[j * DP + d], u);
            }
            gW[r * D + d] = w;
            gU[r * D + d] = u;
        }
    }
}

// ---------------------------------------------------------------------------
// scan
// ---------------------------------------------------------------------------
constexpr size_t kScanSmemFloats = D * BVP + 3 * C * DP + C * CP + C * BVP + D;

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
    chunk_scan_f32_kernel(const float *__restrict__ initial_state, float *__restrict__ final_state,
                          const int32_t *__restrict__ state_indices, T *__restrict__ o,
                          int n_seqs, int H, void *workspace, WsLayout L) {
    extern __shared__ float smem[];
    float *sS = smem;              // [D][BVP] state block: S[d][v], v in this CTA's columns
    float *sW = sS + D * BVP;      // [C][DP]
    float *sQG = sW + C * DP;      // [C][DP]
    float *sKD = sQG + C * DP;     // [C][DP]
    float *sA = sKD + C * DP;      // [C][CP]
    float *sVn = sA + C * CP;      // [C][BVP]
    float *sGC = sVn + C * BVP;    // [D]

    const int n = blockIdx.x, h = blockIdx.y, v0 = blockIdx.z * BV;
    const int tid = threadIdx.x;
    const int32_t start = ws_at<const int32_t>(workspace, L.seq_start_off)[n];
    if (start < 0) return;  // sequence skipped (bad cu_seqlens or slot)
    const int len = ws_at<const int32_t>(workspace, L.seq_len_off)[n];
    const int c0 = ws_at<const int32_t>(workspace, L.chunk_off_off)[n];
    const int nck = (len + C - 1) / C;
    const int64_t slot = state_indices ? (int64_t)state_indices[n] : (int64_t)n;
    const int64_t st_off = (slot * H + h) * (int64_t)D * D;  // [V][K] block of (slot, h)

    // initial state (stored [V][K]) -> sS[d][v]
    for (int i = tid; i < D * BV; i += kThreads) {
        const int vv = i / D, d = i % D;
        sS[d * BVP + vv] = initial_state ? initial_state[st_off + (int64_t)(v0 + vv) * D + d] : 0.0f;
    }

    for (int ck = 0; ck < nck; ++ck) {
        const float *rec = ws_at<const float>(workspace, L.records_off + ((size_t)(c0 + ck) * H + h) * F32Rec::bytes);
        const int valid = min(C, len - ck * C);
        const int64_t tok0 = (int64_t)start + (int64_t)ck * C;
        __syncthreads();  // previous chunk finished with the shared tiles
        for (int i = tid; i < C * D / 4; i += kThreads) {
            const int r = (4 * i) / D, d = (4 * i) % D;
            const float4 w4 = load4(rec + F32Rec::W + 4 * i);
            const float4 q4 = load4(rec + F32Rec::QG + 4 * i);
            const float4 k4 = load4(rec + F32Rec::KD + 4 * i);
            float *pw = sW + r * DP + d, *pq = sQG + r * DP + d, *pk = sKD + r * DP + d;
            pw[0] = w4.x; pw[1] = w4.y; pw[2] = w4.z; pw[3] = w4.w;
            pq[0] = q4.x; pq[1] = q4.y; pq[2] = q4.z; pq[3] = q4.w;
            pk[0] = k4.x; pk[1] = k4.y; pk[2] = k4.z; pk[3] = k4.w;
        }
        for (int i = tid; i < C * C; i += kThreads) sA[(i / C) * CP + i % C] = rec[F32Rec::A + i];
        if (tid < D) sGC[tid] = rec[F32Rec::GC + tid];
        __syncthreads();

        // Vn = U - W S  and  P = QG S   (thread: row r, 8 columns)
        const int r = tid >> 2, cb = (tid & 3) * 8;
        float ws[8], qs[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) ws[x] = qs[x] = 0.0f;
        for (int d = 0; d < D; ++d) {
            const float w = sW[r * DP + d], qg = sQG[r * DP + d];
            const float *srow = sS + d * BVP + cb;
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                ws[x] = fmaf(w, srow[x], ws[x]);
                qs[x] = fmaf(qg, srow[x], qs[x]);
            }
        }
        const float *gU = rec + F32Rec::U + r * D + v0 + cb;
#pragma unroll
        for (int x = 0; x < 8; ++x) sVn[r * BVP + cb + x] = gU[x] - ws[x];
        __syncthreads();

        // o = P + A Vn  (A lower triangular)
        for (int j = 0; j <= r; ++j) {
            const float a = sA[r * CP + j];
#pragma unroll
            for (int x = 0; x < 8; ++x) qs[x] = fmaf(a, sVn[j * BVP + cb + x], qs[x]);
        }
        if (r < valid) {
            T *orow = o + ((tok0 + r) * H + h) * (int64_t)D + v0 + cb;
#pragma unroll
            for (int x = 0; x < 8; ++x) orow[x] = from_f32<T>(qs[x]);
        }

        // S = diag(gC) S + KD^T Vn   (thread: key channel d, 16 columns)
        {
            const int d = tid >> 1, vb = (tid & 1) * 16;
            float acc[16];
            const float gc = sGC[d];
#pragma unroll
            for (int x = 0; x < 16; ++x) acc[x] = gc * sS[d * BVP + vb + x];
            for (int j = 0; j < C; ++j) {
                const float kd = sKD[j * DP + d];
#pragma unroll
                for (int x = 0; x < 16; ++x) acc[x] = fmaf(kd, sVn[j * BVP + vb + x], acc[x]);
            }
            __syncthreads();  // every thread is done reading the old sS
#pragma unroll
            for (int x = 0; x < 16; ++x) sS[d * BVP + vb + x] = acc[x];
        }
    }
    __syncthreads();
    if (final_state) {
        for (int i = tid; i < D * BV; i += kThreads) {
            const int vv = i / D, d = i % D;
            final_state[st_off + (int64_t)(v0 + vv) * D + d] = sS[d * BVP + vv];
        }
    }
}

}  // namespace

cudaError_t launch_chunk_prep_f32(const void *q, const void *k, const void *v, const float *g,
                                  const float *beta, int dtype, int n_seqs, int64_t total_tokens,
                                  int H, float scale, void *workspace, cudaStream_t stream) {
    const WsLayout L = ws_layout(total_tokens, n_seqs, H, F32Rec::bytes);
    const size_t smem = kPrepSmemFloats * sizeof(float);
    const dim3 grid((unsigned)max_chunks(total_tokens, n_seqs), (unsigned)H);
    if (dtype == KDA_BF16) {
        auto kern = chunk_prep_f32_kernel<__nv_bfloat16>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        kern<<<grid, kThreads, smem, stream>>>((const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k,
                                               (const __nv_bfloat16 *)v, g, beta, n_seqs, H, scale,
                                               workspace, L);
    } else {
        auto kern = chunk_prep_f32_kernel<float>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        kern<<<grid, kThreads, smem, stream>>>((const float *)q, (const float *)k,
                                               (const float *)v, g, beta, n_seqs, H, scale,
                                               workspace, L);
    }
    return cudaGetLastError();
}

cudaError_t launch_chunk_scan_f32(const float *initial_state, float *final_state,
                                  const int32_t *state_indices, void *o, int dtype, int n_seqs,
                                  int64_t total_tokens, int H, void *workspace,
                                  cudaStream_t stream) {
    const WsLayout L = ws_layout(total_tokens, n_seqs, H, F32Rec::bytes);
    const size_t smem = kScanSmemFloats * sizeof(float);
    const dim3 grid((unsigned)n_seqs, (unsigned)H, D / BV);
    if (dtype == KDA_BF16) {
        auto kern = chunk_scan_f32_kernel<__nv_bfloat16>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        kern<<<grid, kThreads, smem, stream>>>(initial_state, final_state, state_indices,
                                               (__nv_bfloat16 *)o, n_seqs, H, workspace, L);
    } else {
        auto kern = chunk_scan_f32_kernel<float>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        kern<<<grid, kThreads, smem, stream>>>(initial_state, final_state, state_indices,
                                               (float *)o, n_seqs, H, workspace, L);
    }
    return cudaGetLastError();
}

}  // namespace kda
