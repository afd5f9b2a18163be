// Tensor-core (tcgen05) chunked KDA for bf16 inputs: bf16 MMA operands, fp32
// accumulation in TMEM, fp32 recurrent state.
//
// Same two phases as the fp32 path (chunked form of the Ascend model file's
// _torch_chunk_kda), with every dense contraction on the 5th-generation
// tensor cores:
//
// prep, one CTA per (chunk, head), 8 warps:
//   * q_hat = scale * l2norm(q), k_hat = l2norm(k) (fp32), G = cumsum(g).
//   * Causal scores A[r,j] and the interaction matrix L[r,j] as ONE M=128 MMA
//     per 16-column block b of the chunk: rows 0..63 of the A operand are
//     q_hat_r * exp(G_r - G_ref), rows 64..127 k_hat_r * exp(G_r - G_ref),
//     the B operand is k_hat_j * exp(G_ref - G_j) for the 16 keys j of the
//     block, with the reference G_ref = G at the block's first token.  For
//     every kept pair (j <= r) the row factor is <= 1 and the column factor is
//     at most exp(15 * max|g|), so the factorisation cannot overflow for
//     per-token decays down to about -5.3 (the column exponent is clamped at
//     80 beyond that, and only masked pairs can then be affected).
//   * X = (I + beta L)^-1 by forward substitution in fp32; T = X diag(beta).
//   * W^T = (exp(G) k_hat)^T T^T and U^T = v^T T^T as M=128 (key / value
//     dim) x N=64 x K=64 MMAs.
//   * The record handed to the scan holds the MMA operands of the scan,
//     already in the 128-byte-swizzled K-major shared-memory layout, so the
//     scan moves them with one bulk copy per chunk:
//       WQ  [128][128]: rows 0..63 W, rows 64..127 QG = q_hat exp(G)
//       KDT [128][64] : KD^T, KD = k_hat exp(G_last - G)
//       A   [64][64]  : causal scores (scale folded into q_hat)
//       gC  [128] fp32: exp(G_last);   U [64][128] bf16 row-major.
//
// scan, one CTA per (sequence, head, 32 value columns), 4 warps:
//   per chunk (records double-buffered by cp.async.bulk):
//     D1  = WQ * S            (M=128, N=32, K=128)  rows 0..63: W S
//     Vn  = U - D1[0:64]      (fp32, written as a bf16 K-major operand)
//     D1 += [* ; A] * Vn      (rows 64..127 become o = QG S + A Vn)
//     D3  = KD^T * Vn         (M=128, N=32, K=64)
//     S   = diag(gC) S + D3   (fp32, one key row per thread, in registers)
//   The 128-row A operand of the second MMA starts 8 KB before the A tile in
//   the staged record (its rows 0..63 are the tail of KD^T and only feed D1
//   rows that were already consumed).
#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int C = kChunk;    // 64
constexpr int D = kHeadDim;  // 128
constexpr int kStatusTimeout = 4;

// ---------------------------------------------------------------------------
// prep
// ---------------------------------------------------------------------------
constexpr int kPrepThreads = 256;
constexpr uint32_t kPrepTmemCols = 128;
// shared memory plan (offsets from a 1024-aligned base)
constexpr int P_G = 0;                    // fp32 [64][128] cumulative log-decay   32 KB
constexpr int P_Z = P_G + C * D * 4;      // 32 KB: A_b operand -> L,X fp32 -> E^T,V^T operands
constexpr int P_C = P_Z + 32768;          // 4 x [16][128] bf16 column-factor operands 16 KB
constexpr int P_T = P_C + 16384;          // [64][64] bf16 T operand 8 KB
constexpr int P_MISC = P_T + 8192;        // rq, rk, beta (fp32 x 64 each), barrier, tmem base
constexpr int P_BYTES = P_MISC + 3 * 64 * 4 + 64;
constexpr int P_SMEM = P_BYTES + 1024;    // slack for 1024-byte alignment

__device__ __forceinline__ void st_bf16(unsigned char *base, uint32_t off, float x) {
    *reinterpret_cast<__nv_bfloat16 *>(base + off) = __float2bfloat16_rn(x);
}

__global__ void __launch_bounds__(kPrepThreads, 2)
    chunk_prep_tc_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                         const __nv_bfloat16 *__restrict__ v, const float *__restrict__ g,
                         const float *__restrict__ beta, int n_seqs, int H, float scale,
                         void *workspace, WsLayout L) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    float *sG = reinterpret_cast<float *>(sm + P_G);
    unsigned char *sZ = sm + P_Z;
    unsigned char *sC = sm + P_C;
    unsigned char *sT = sm + P_T;
    float *sRq = reinterpret_cast<float *>(sm + P_MISC);
    float *sRk = sRq + 64;
    float *sB = sRk + 64;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sB + 64);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 1);

    const int32_t *chunk_off = ws_at<const int32_t>(workspace, L.chunk_off_off);
    const int c = blockIdx.x, h = blockIdx.y;
    if (c >= chunk_off[n_seqs]) return;
    const int n = owner_of_chunk(chunk_off, n_seqs, c);
    const int jc = c - chunk_off[n];
    const int64_t tok0 = (int64_t)ws_at<const int32_t>(workspace, L.seq_start_off)[n] + (int64_t)jc * C;
    const int valid = min(C, ws_at<const int32_t>(workspace, L.seq_len_off)[n] - jc * C);
    unsigned char *rec = ws_at<unsigned char>(workspace, L.records_off + ((size_t)c * H + h) * TcRec::bytes);
    int32_t *status = ws_at<int32_t>(workspace, L.status_off);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (warp == 0) tmem_alloc(tmem_slot, kPrepTmemCols);
    if (tid == 32) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }

    // 1. cumulative log-decay (threads 0..127, one key channel each) and the
    //    row norms of q and k (warps 4..7), beta.
    if (tid < D) {
        float run = 0.0f;
        const float *gp = g + (tok0 * H + h) * (int64_t)D + tid;
#pragma unroll 8
        for (int r = 0; r < C; ++r) {
            run += (r < valid) ? gp[(int64_t)r * H * D] : 0.0f;
            sG[r * D + tid] = run;
        }
    } else {
        for (int r = warp - 4; r < C; r += 4) {
            float4 q4 = make_float4(0, 0, 0, 0), k4 = q4;
            if (r < valid) {
                const int64_t off = ((tok0 + r) * H + h) * (int64_t)D + 4 * lane;
                q4 = load4(q + off);
                k4 = load4(k + off);
            }
            const float sq = warp_sum(q4.x * q4.x + q4.y * q4.y + q4.z * q4.z + q4.w * q4.w);
            const float sk = warp_sum(k4.x * k4.x + k4.y * k4.y + k4.z * k4.z + k4.w * k4.w);
            if (lane == 0) {
                sRq[r] = scale / sqrtf(sq + 1e-6f);
                sRk[r] = 1.0f / sqrtf(sk + 1e-6f);
            }
        }
        if (tid - D < C) {
            const int r = tid - D;
            sB[r] = r < valid ? beta[(tok0 + r) * H + h] : 0.0f;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // 2. QG (WQ rows 64..127), KD^T, column-factor operands, gC.
    {
        const int d = tid & (D - 1);
        const float Gl = sG[(C - 1) * D + d];
        for (int r = tid >> 7; r < C; r += 2) {
            float qv = 0.0f, kv = 0.0f;
            if (r < valid) {
                const int64_t off = ((tok0 + r) * H + h) * (int64_t)D + d;
                qv = __bfloat162float(q[off]);
                kv = __bfloat162float(k[off]);
            }
            const float qh = qv * sRq[r], kh = kv * sRk[r];
            const float G = sG[r * D + d];
            const float Gb = sG[(r & ~15) * D + d];
            st_bf16(rec, TcRec::WQ + sw128_off(64 + r, d, 128), qh * __expf(G));
            st_bf16(rec, TcRec::KDT + sw128_off(d, r, 128), kh * __expf(Gl - G));
            st_bf16(sC, (uint32_t)((r >> 4) * 4096) + sw128_off(r & 15, d, 16),
                    kh * __expf(fminf(Gb - G, 80.0f)));
        }
        if (tid < D) reinterpret_cast<float *>(rec + TcRec::GC)[tid] = __expf(Gl);
    }

    // 3. A and L, one 16-column block at a time (A operand rebuilt in Z).
    bool ok = true;
    uint32_t phase = 0;
    for (int b = 0; b < 4; ++b) {
        const int d = tid & (D - 1);
        for (int r = tid >> 7; r < C; r += 2) {
            float qa = 0.0f, ka = 0.0f;
            if (r >= 16 * b && r < valid) {
                const int64_t off = ((tok0 + r) * H + h) * (int64_t)D + d;
                const float e = __expf(sG[r * D + d] - sG[16 * b * D + d]);
                qa = __bfloat162float(q[off]) * sRq[r] * e;
                ka = __bfloat162float(k[off]) * sRk[r] * e;
            }
            st_bf16(sZ, sw128_off(r, d, 128), qa);
            st_bf16(sZ, sw128_off(64 + r, d, 128), ka);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            mma_tile<128, 16, 128>(tmem + 16 * b, smem_u32(sZ), 128, smem_u32(sC + b * 4096), 16,
                                   false);
            mma_commit(bar);
        }
        ok = mbar_wait(bar, phase) && ok;
        phase ^= 1;
        tc_fence_after();
    }
    if (!__syncthreads_and(ok)) {
        if (tid == 0) atomicOr(status, kStatusTimeout);
        goto done;
    }

    // 4. read A (lanes 0..63) to the record and L (lanes 64..127) to shared fp32.
    {
        float *sL = reinterpret_cast<float *>(sZ);
        const int quarter = warp & 3, col0 = (warp >> 2) * 32;
        const int row = 32 * quarter + lane;
        float x[32];
        tmem_ld32(tmem + ((uint32_t)(32 * quarter) << 16) + col0, x);
        tmem_ld_wait();
        if (row < C) {
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int j = col0 + jj;
                st_bf16(rec, TcRec::A + sw128_off(row, j, 64), j <= row ? x[jj] : 0.0f);
            }
        } else {
            const int r = row - C;
            const float br = sB[r];
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int j = col0 + jj;
                sL[r * C + j] = j < r ? br * x[jj] : 0.0f;
            }
        }
    }
    tc_fence_before();
    __syncthreads();

    // 5. X = (I + L)^-1 row by row; T = X diag(beta) as a bf16 operand.
    {
        const float *sL = reinterpret_cast<const float *>(sZ);
        float *sX = reinterpret_cast<float *>(sZ) + C * C;
        const int col = tid >> 2, part = tid & 3;
        for (int r = 0; r < C; ++r) {
            float acc = 0.0f;
            for (int m = col + part; m < r; m += 4) acc = fmaf(sL[r * C + m], sX[m * C + col], acc);
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            if (part == 0) sX[r * C + col] = (col == r) ? 1.0f : (col < r ? -acc : 0.0f);
            __syncthreads();
        }
        for (int i = tid; i < C * C; i += kPrepThreads) {
            const int r = i / C, cc = i % C;
            st_bf16(sT, sw128_off(r, cc, 64), sX[r * C + cc] * sB[cc]);
        }
    }
    __syncthreads();

    // 6. E^T = (exp(G) k_hat)^T and V^T operands (in Z), then W^T, U^T MMAs.
    {
        unsigned char *sE = sZ, *sV = sZ + 16384;
        const int d = tid & (D - 1);
        for (int j = tid >> 7; j < C; j += 2) {
            float kv = 0.0f, vv = 0.0f;
            if (j < valid) {
                const int64_t off = ((tok0 + j) * H + h) * (int64_t)D + d;
                kv = __bfloat162float(k[off]);
                vv = __bfloat162float(v[off]);
            }
            st_bf16(sE, sw128_off(d, j, 128), kv * sRk[j] * __expf(sG[j * D + d]));
            st_bf16(sV, sw128_off(d, j, 128), vv);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            mma_tile<128, 64, 64>(tmem + 0, smem_u32(sE), 128, smem_u32(sT), 64, false);
            mma_tile<128, 64, 64>(tmem + 64, smem_u32(sV), 128, smem_u32(sT), 64, false);
            mma_commit(bar);
        }
        ok = mbar_wait(bar, phase);
        tc_fence_after();
    }
    if (!__syncthreads_and(ok)) {
        if (tid == 0) atomicOr(status, kStatusTimeout);
        goto done;
    }

    // 7. W (WQ rows 0..63) and U to the record.
    {
        const int quarter = warp & 3, col0 = (warp >> 2) * 32;
        const int lrow = 32 * quarter + lane;  // key dim d for W, value dim for U
        const uint32_t ta = tmem + ((uint32_t)(32 * quarter) << 16);
        float x[32];
        tmem_ld32(ta + col0, x);
        tmem_ld_wait();
#pragma unroll
        for (int ii = 0; ii < 32; ++ii) st_bf16(rec, TcRec::WQ + sw128_off(col0 + ii, lrow, 128), x[ii]);
        tmem_ld32(ta + 64 + col0, x);
        tmem_ld_wait();
        __nv_bfloat16 *U = reinterpret_cast<__nv_bfloat16 *>(rec + TcRec::U);
#pragma unroll
        for (int ii = 0; ii < 32; ++ii) U[(col0 + ii) * D + lrow] = __float2bfloat16_rn(x[ii]);
    }

done:
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kPrepTmemCols);
}

// ---------------------------------------------------------------------------
// scan
// ---------------------------------------------------------------------------
constexpr int kScanThreads = 128;
constexpr int BV = 32;
constexpr uint32_t kScanTmemCols = 64;
constexpr uint32_t kStageBytes = TcRec::U;  // WQ | KDT | A | gC, copied in one piece
constexpr int S_STAGE = 58368;              // kStageBytes rounded up to 1024
constexpr int S_SOP = 2 * S_STAGE;          // S^T operand [32][128] bf16, 8 KB
constexpr int S_VOP = S_SOP + 8192;         // Vn^T operand [32][64] bf16, 4 KB
constexpr int S_BAR = S_VOP + 4096;         // full[2], mma
constexpr int S_BYTES = S_BAR + 64;
constexpr int S_SMEM = S_BYTES + 1024;
static_assert(kStageBytes <= (uint32_t)S_STAGE, "stage too small");
static_assert(kStageBytes % 16 == 0, "bulk copy size");

__global__ void __launch_bounds__(kScanThreads, 1)
    chunk_scan_tc_kernel(const float *__restrict__ initial_state, float *__restrict__ final_state,
                         const int32_t *__restrict__ state_indices, __nv_bfloat16 *__restrict__ o,
                         int n_seqs, int H, void *workspace, WsLayout L) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char *sS = sm + S_SOP;
    unsigned char *sVn = sm + S_VOP;
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + S_BAR);
    uint64_t *mbar = full + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mbar + 1);

    const int n = blockIdx.x, h = blockIdx.y, v0 = blockIdx.z * BV;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int32_t start = ws_at<const int32_t>(workspace, L.seq_start_off)[n];
    if (start < 0) return;  // sequence skipped (bad cu_seqlens or slot)
    const int len = ws_at<const int32_t>(workspace, L.seq_len_off)[n];
    const int c0 = ws_at<const int32_t>(workspace, L.chunk_off_off)[n];
    const int nck = (len + C - 1) / C;
    const int64_t slot = state_indices ? (int64_t)state_indices[n] : (int64_t)n;
    const int64_t st_off = (slot * H + h) * (int64_t)D * D;  // [V][K] block of (slot, h)
    int32_t *status = ws_at<int32_t>(workspace, L.status_off);
    const unsigned char *recs = ws_at<const unsigned char>(workspace, L.records_off);
    auto rec_of = [&](int ck) { return recs + ((size_t)(c0 + ck) * H + h) * TcRec::bytes; };

    if (warp == 0) tmem_alloc(tmem_slot, kScanTmemCols);
    if (tid == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_init(mbar, 1);
        fence_mbar_init();
    }
    // state row d = tid, columns v0 .. v0+31, fp32 in registers
    float S[BV];
#pragma unroll
    for (int x = 0; x < BV; ++x)
        S[x] = initial_state ? initial_state[st_off + (int64_t)(v0 + x) * D + tid] : 0.0f;
#pragma unroll
    for (int x = 0; x < BV; ++x) st_bf16(sS, sw128_off(x, tid, BV), S[x]);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tD1 = tmem, tD3 = tmem + 32;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;

    bool issued[2] = {false, false};
    if (tid == 0 && nck > 0) {
        mbar_arrive_expect_tx(&full[0], kStageBytes);
        bulk_g2s(sm, rec_of(0), kStageBytes, &full[0]);
        issued[0] = true;
    }
    uint32_t mphase = 0;
    bool ok = true;
    for (int ck = 0; ck < nck; ++ck) {
        const int stage = ck & 1;
        unsigned char *st = sm + stage * S_STAGE;
        if (tid == 0 && ck + 1 < nck) {  // the other stage was released at the end of ck-1
            mbar_arrive_expect_tx(&full[stage ^ 1], kStageBytes);
            bulk_g2s(sm + (stage ^ 1) * S_STAGE, rec_of(ck + 1), kStageBytes, &full[stage ^ 1]);
            issued[stage ^ 1] = true;
        }
        const int valid = min(C, len - ck * C);
        const int64_t tok0 = (int64_t)start + (int64_t)ck * C;
        // U row for this thread's chunk row (threads 0..63), fetched while waiting
        uint4 u4[4];
        if (tid < C) {
            const uint4 *up = reinterpret_cast<const uint4 *>(rec_of(ck) + TcRec::U + (tid * D + v0) * 2);
#pragma unroll
            for (int x = 0; x < 4; ++x) u4[x] = up[x];
        }
        ok = mbar_wait(&full[stage], (ck >> 1) & 1) && ok;
        if (tid == 0) issued[stage] = false;
        if (!__syncthreads_and(ok)) break;

        // D1 = WQ * S
        if (tid == 0) {
            tc_fence_after();
            mma_tile<128, BV, 128>(tD1, smem_u32(st + TcRec::WQ), 128, smem_u32(sS), BV, false);
            mma_commit(mbar);
        }
        ok = mbar_wait(mbar, mphase) && ok;
        mphase ^= 1;
        tc_fence_after();
        if (warp < 2) {  // rows 0..63: Vn = U - W S
            float x[32];
            tmem_ld32(tD1 + lane_base, x);
            tmem_ld_wait();
            const __nv_bfloat16 *ub = reinterpret_cast<const __nv_bfloat16 *>(u4);
#pragma unroll
            for (int vv = 0; vv < BV; ++vv)
                st_bf16(sVn, sw128_off(vv, tid, BV), __bfloat162float(ub[vv]) - x[vv]);
        }
        fence_async_smem();
        tc_fence_before();
        if (!__syncthreads_and(ok)) break;

        // D1 += [* ; A] * Vn ;  D3 = KD^T * Vn
        if (tid == 0) {
            tc_fence_after();
            mma_tile<128, BV, 64>(tD1, smem_u32(st + TcRec::A) - 8192, 128, smem_u32(sVn), BV, true);
            mma_tile<128, BV, 64>(tD3, smem_u32(st + TcRec::KDT), 128, smem_u32(sVn), BV, false);
            mma_commit(mbar);
        }
        ok = mbar_wait(mbar, mphase) && ok;
        mphase ^= 1;
        tc_fence_after();
        if (warp >= 2) {  // rows 64..127: o
            float x[32];
            tmem_ld32(tD1 + lane_base, x);
            tmem_ld_wait();
            const int r = tid - 64;
            if (r < valid) {
                uint4 pk[4];
                __nv_bfloat16 *pb = reinterpret_cast<__nv_bfloat16 *>(pk);
#pragma unroll
                for (int vv = 0; vv < BV; ++vv) pb[vv] = __float2bfloat16_rn(x[vv]);
                uint4 *op = reinterpret_cast<uint4 *>(o + ((tok0 + r) * H + h) * (int64_t)D + v0);
#pragma unroll
                for (int x4 = 0; x4 < 4; ++x4) op[x4] = pk[x4];
            }
        }
        {  // S = diag(gC) S + KD^T Vn
            float x[32];
            tmem_ld32(tD3 + lane_base, x);
            tmem_ld_wait();
            const float gc = reinterpret_cast<const float *>(st + TcRec::GC)[tid];
#pragma unroll
            for (int vv = 0; vv < BV; ++vv) {
                S[vv] = fmaf(gc, S[vv], x[vv]);
                st_bf16(sS, sw128_off(vv, tid, BV), S[vv]);
            }
        }
        fence_async_smem();
        tc_fence_before();
        if (!__syncthreads_and(ok)) break;
    }
    if (!ok) {
        if (tid == 0) {
            atomicOr(status, kStatusTimeout);
            // let copies still in flight land before the shared memory is released
            for (int s = 0; s < 2; ++s)
                if (issued[s]) mbar_wait(&full[s], 0, 400000000LL) || mbar_wait(&full[s], 1, 400000000LL);
        }
    } else if (final_state) {
#pragma unroll
        for (int x = 0; x < BV; ++x) final_state[st_off + (int64_t)(v0 + x) * D + tid] = S[x];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kScanTmemCols);
}

}  // namespace

cudaError_t launch_chunk_prep_tc(const void *q, const void *k, const void *v, const float *g,
                                 const float *beta, int n_seqs, int64_t total_tokens, int H,
                                 float scale, void *workspace, cudaStream_t stream) {
    const WsLayout L = ws_layout(total_tokens, n_seqs, H, TcRec::bytes);
    const dim3 grid((unsigned)max_chunks(total_tokens, n_seqs), (unsigned)H);
    cudaFuncSetAttribute(chunk_prep_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM);
    chunk_prep_tc_kernel<<<grid, kPrepThreads, P_SMEM, stream>>>(
        (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k, (const __nv_bfloat16 *)v, g, beta,
        n_seqs, H, scale, workspace, L);
    return cudaGetLastError();
}

cudaError_t launch_chunk_scan_tc(const float *initial_state, float *final_state,
                                 const int32_t *state_indices, void *o, int n_seqs,
                                 int64_t total_tokens, int H, void *workspace,
                                 cudaStream_t stream) {
    const WsLayout L = ws_layout(total_tokens, n_seqs, H, TcRec::bytes);
    const dim3 grid((unsigned)n_seqs, (unsigned)H, D / BV);
    cudaFuncSetAttribute(chunk_scan_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, S_SMEM);
    chunk_scan_tc_kernel<<<grid, kScanThreads, S_SMEM, stream>>>(
        initial_state, final_state, state_indices, (__nv_bfloat16 *)o, n_seqs, H, workspace, L);
    return cudaGetLastError();
}

}  // namespace kda
