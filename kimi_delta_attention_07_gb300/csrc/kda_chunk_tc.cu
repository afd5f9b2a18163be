// Tensor-core (tcgen05) chunked KDA for bf16 inputs: bf16 MMA operands, fp32
// accumulation in TMEM, fp32 recurrent state.
//
// Same two phases as the fp32 path (chunked form of the Ascend model file's
// _torch_chunk_kda), with every dense contraction on the 5th-generation
// tensor cores.
//
// prep -- persistent, one CTA per SM walking the (chunk, head) items; the raw
// q, k, v, g rows of the next item are bulk-copied into a second shared
// buffer while the current item is computed:
//   * q_hat = scale * l2norm(q), k_hat = l2norm(k) (fp32), G = cumsum(g).
//   * G is replaced in place by l_r = exp(G_r - G_{16 br}) (br = r's 16-row
//     block) and per-channel block factors rho_b = exp(G_{16b}) and
//     tau_{br,b} = exp(G_{16br} - G_{16b}); every exponent is <= 0, and
//     exp(G_r - G_{16b}) = l_r * tau_{br,b}, exp(G_r) = l_r * rho_br.
//   * Causal scores A[r,j] and the interaction matrix L[r,j] as ONE M=128 MMA
//     per 16-column block b: rows 0..63 of the A operand are
//     q_hat_r * exp(G_r - G_16b), rows 64..127 k_hat_r * exp(G_r - G_16b)
//     (zero for r < 16b), the B operand is k_hat_j * exp(G_16b - G_j) for the
//     16 keys of block b.  For every kept pair (j <= r) the row factor is
//     <= 1 and the column factor at most exp(15 * max|g|); the column
//     exponent is clamped at 80, which only matters for per-token decays
//     below about -5.3 and then only for masked pairs.
//   * X = (I + beta L)^-1 blockwise in fp32 (16x16 diagonal blocks by forward
//     substitution, one warp each, then three levels of 16x16 products);
//     T = X diag(beta).
//   * W = T (exp(G) k_hat) and U = T v as M=128 x N=128 x K=64 MMAs whose A
//     operand is [T ; scratch] (rows 64..127 unused), so each thread of
//     TMEM lanes 0..63 holds whole rows of W and U.
//   * Record written with 16-byte stores, laid out as the scan's shared-
//     memory image (128-byte-swizzled K-major operands), see TcRec.
//
// scan, one CTA per (sequence, head, 32 value columns), 4 warps, records in a
// 3-stage cp.async.bulk ring:
//     D1  = WQ * S            (M=128, N=32, K=128)  rows 0..63: W S
//     Vn  = U - D1[0:64]      (fp32, written as a bf16 K-major operand)
//     D1 += [* ; A] * Vn      (rows 64..127 become o = QG S + A Vn)
//     D3  = KD^T * Vn         (M=128, N=32, K=64)
//     S   = diag(gC) S + D3   (fp32, one key row per thread, in registers)
//   The 128-row A operand of the second MMA starts 8 KB before the A tile in
//   the staged record (its rows 0..63 are the tail of KD^T and only feed D1
//   rows that were already consumed).
#include <cuda.h>  // CUtensorMap (the encoder is fetched through the runtime)
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int C = kChunk;    // 64
constexpr int D = kHeadDim;  // 128
constexpr int kStatusTimeout = 4;

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&p);
}

__device__ __forceinline__ uint4 pack8(const float (&x)[8]) {
    return make_uint4(pack2(x[0], x[1]), pack2(x[2], x[3]), pack2(x[4], x[5]), pack2(x[6], x[7]));
}

// 8 consecutive bf16 (16 bytes) -> fp32
__device__ __forceinline__ void unpack8(uint4 raw, float (&x)[8]) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 p = *reinterpret_cast<const __nv_bfloat162 *>(&w[i]);
        const float2 f = __bfloat1622float2(p);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}

__device__ __forceinline__ void load8f(const float *p, float (&x)[8]) {
    const float4 a = *reinterpret_cast<const float4 *>(p);
    const float4 b = *reinterpret_cast<const float4 *>(p + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

__device__ __forceinline__ void store8f(float *p, const float (&x)[8]) {
    *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
    *reinterpret_cast<float4 *>(p + 4) = make_float4(x[4], x[5], x[6], x[7]);
}

// ---------------------------------------------------------------------------
// prep
// ---------------------------------------------------------------------------
constexpr int kPrepThreads = 256;
constexpr uint32_t kPrepTmemCols = 256;
// one item's raw rows (double-buffered)
constexpr int R_Q = 0;          // bf16 [64][128]; after the A/L MMAs: X fp32 [64][64]
constexpr int R_K = 16384;      // bf16 [64][128]
constexpr int R_V = 32768;      // bf16 [64][128]
constexpr int R_G = 49152;      // fp32 [64][128]: g -> G -> l
constexpr int R_BYTES = 81920;
constexpr int P_Z = 2 * R_BYTES;          // 32 KB: A_b operand | L fp32 (stride 68) | E^T, V^T
constexpr int P_C = P_Z + 32768;          // 16 KB: column-factor operands | [T ; temps]
constexpr int P_RQ = P_C + 16384;         // fp32 [64]
constexpr int P_RK = P_RQ + 256;          // fp32 [64]
constexpr int P_BETA = P_RK + 256;        // fp32 [64]
constexpr int P_GREF = P_BETA + 256;      // fp32 [5][128]: G at rows 0, 16, 32, 48, 63
constexpr int P_RHO = P_GREF + 5 * 512;   // fp32 [4][128]: exp(G_16b)
constexpr int P_TAU = P_RHO + 4 * 512;    // fp32 [6][128]: exp(G_16br - G_16b), br > b
constexpr int P_BAR = P_TAU + 6 * 512;    // full[2], mma barrier, tmem slot
constexpr int P_BYTES = P_BAR + 64;
constexpr int P_SMEM = P_BYTES + 1024;
constexpr int LSTRIDE = 68;               // row stride (floats) of L in shared memory
static_assert(C * LSTRIDE * 4 <= 17408 && 22528 + 6 * 16 * 20 * 4 <= 32768, "Z scratch does not fit");

__device__ __forceinline__ int tau_index(int br, int b) { return br * (br - 1) / 2 + b; }

struct PrepItem {
    int64_t tok0;
    int valid, h, c;
};

__device__ __forceinline__ PrepItem prep_item(int item, int H, const int32_t *chunk_off,
                                              const int32_t *seq_start, const int32_t *seq_len,
                                              int n_seqs) {
    PrepItem it;
    it.c = item / H;
    it.h = item - it.c * H;
    const int n = owner_of_chunk(chunk_off, n_seqs, it.c);
    const int jc = it.c - chunk_off[n];
    it.tok0 = (int64_t)seq_start[n] + (int64_t)jc * C;
    it.valid = min(C, seq_len[n] - jc * C);
    return it;
}


// Raw rows of one (chunk, head) item: q, k, v ([T, H, 128] bf16) and g
// ([T, H, 128] fp32) through 3-D tensor maps {128, H, T}; one 128 x 1 x 64
// box each, rows past the end of the tensor arrive as zeros.
struct RawMaps {
    CUtensorMap q, k, v, g;
};

__device__ __forceinline__ void load_raw(unsigned char *buf, const RawMaps &m, int h, int64_t tok0,
                                         uint64_t *bar) {
    mbar_arrive_expect_tx(bar, (uint32_t)R_BYTES);
    tma_load_3d(buf + R_Q, &m.q, 0, h, (int)tok0, bar);
    tma_load_3d(buf + R_K, &m.k, 0, h, (int)tok0, bar);
    tma_load_3d(buf + R_V, &m.v, 0, h, (int)tok0, bar);
    tma_load_3d(buf + R_G, &m.g, 0, h, (int)tok0, bar);
}

// 16x16 fp32 matrices of the inverse live with a row stride of 20 floats
// (16-byte aligned rows, conflict-free row reads across 8 rows).
constexpr int MS = 20;
constexpr int MBLK = 16 * MS;  // floats per 16x16 matrix

// Four outputs (row i, columns 4cg..4cg+3) of P = A * B for 16x16 matrices;
// A read with stride lda, B with stride MS.
__device__ __forceinline__ float4 mm16_row4(const float *A, int lda, const float *B, int i, int cg) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
        const float a = A[i * lda + kk];
        const float4 b = *reinterpret_cast<const float4 *>(B + kk * MS + 4 * cg);
        acc.x = fmaf(a, b.x, acc.x);
        acc.y = fmaf(a, b.y, acc.y);
        acc.z = fmaf(a, b.z, acc.z);
        acc.w = fmaf(a, b.w, acc.w);
    }
    return acc;
}

__global__ void __launch_bounds__(kPrepThreads, 1)
    chunk_prep_tc_kernel(const __grid_constant__ RawMaps maps, const float *__restrict__ beta,
                         int n_seqs, int H, float scale, void *workspace, WsLayout L) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char *sZ = sm + P_Z;
    unsigned char *sC = sm + P_C;
    float *sRq = reinterpret_cast<float *>(sm + P_RQ);
    float *sRk = reinterpret_cast<float *>(sm + P_RK);
    float *sB = reinterpret_cast<float *>(sm + P_BETA);
    float *sGref = reinterpret_cast<float *>(sm + P_GREF);
    float *sRho = reinterpret_cast<float *>(sm + P_RHO);
    float *sTau = reinterpret_cast<float *>(sm + P_TAU);
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + P_BAR);
    uint64_t *mbar = full + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mbar + 1);

    const int32_t *chunk_off = ws_at<const int32_t>(workspace, L.chunk_off_off);
    const int32_t *seq_start = ws_at<const int32_t>(workspace, L.seq_start_off);
    const int32_t *seq_len = ws_at<const int32_t>(workspace, L.seq_len_off);
    int32_t *status = ws_at<int32_t>(workspace, L.status_off);
    const int n_items = chunk_off[n_seqs] * H;
    if ((int)blockIdx.x >= n_items) return;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (warp == 0) tmem_alloc(tmem_slot, kPrepTmemCols);
    if (tid == 32) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_init(mbar, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // first item
    PrepItem nxt = prep_item(blockIdx.x, H, chunk_off, seq_start, seq_len, n_seqs);
    if (tid == 0) load_raw(sm, maps, nxt.h, nxt.tok0, &full[0]);
    float beta_next = 0.0f;
    if (tid < nxt.valid) beta_next = beta[(nxt.tok0 + tid) * H + nxt.h];

    uint32_t mphase = 0;
    bool ok = true;
    int m = 0;
    KDA_PHASE_START();
    for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++m) {
        const PrepItem cur = nxt;
        const int buf = m & 1;
        unsigned char *raw = sm + buf * R_BYTES;
        const __nv_bfloat16 *sQr = reinterpret_cast<const __nv_bfloat16 *>(raw + R_Q);
        const __nv_bfloat16 *sKr = reinterpret_cast<const __nv_bfloat16 *>(raw + R_K);
        const __nv_bfloat16 *sVr = reinterpret_cast<const __nv_bfloat16 *>(raw + R_V);
        float *sG = reinterpret_cast<float *>(raw + R_G);
        float *sX = reinterpret_cast<float *>(raw + R_Q);  // after the q rows are consumed
        unsigned char *rec = ws_at<unsigned char>(workspace, L.records_off + ((size_t)cur.c * H + cur.h) * TcRec::bytes);
        const int valid = cur.valid;
        if (tid < C) sB[tid] = tid < valid ? beta_next : 0.0f;

        const int nitem = item + gridDim.x;
        if (nitem < n_items) nxt = prep_item(nitem, H, chunk_off, seq_start, seq_len, n_seqs);
        ok = mbar_wait(&full[buf], (m >> 1) & 1) && ok;
        // zero the rows past the end of the sequence (not copied)
        for (int i = tid; i < (C - valid) * 16; i += kPrepThreads) {
            const int r = valid + i / 16, c16 = i % 16;
            const uint4 z = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4 *>(raw + R_Q + r * 256 + c16 * 16) = z;
            *reinterpret_cast<uint4 *>(raw + R_K + r * 256 + c16 * 16) = z;
            *reinterpret_cast<uint4 *>(raw + R_V + r * 256 + c16 * 16) = z;
            *reinterpret_cast<uint4 *>(raw + R_G + r * 512 + c16 * 32) = z;
            *reinterpret_cast<uint4 *>(raw + R_G + r * 512 + c16 * 32 + 16) = z;
        }
        if (!__syncthreads_and(ok)) break;
        KDA_PHASE(0, 0);
        // prefetch the next item into the other buffer (its last reader was item m-1)
        if (nitem < n_items) {
            if (tid == 0) {
                fence_async_smem();
                load_raw(sm + (buf ^ 1) * R_BYTES, maps, nxt.h, nxt.tok0, &full[buf ^ 1]);
            }
            if (tid < nxt.valid) beta_next = beta[(nxt.tok0 + tid) * H + nxt.h];
        }

        KDA_PHASE(0, 1);
        // 1. row norms of q and k (16 lanes per row, 8 channels each); cumulative
        //    log-decay in place (two halves).
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int r = 16 * it + (tid >> 4), c16 = tid & 15;
            float a[8], b[8];
            unpack8(*reinterpret_cast<const uint4 *>(sQr + r * D + 8 * c16), a);
            unpack8(*reinterpret_cast<const uint4 *>(sKr + r * D + 8 * c16), b);
            float sq = 0.f, sk = 0.f;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                sq = fmaf(a[t], a[t], sq);
                sk = fmaf(b[t], b[t], sk);
            }
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, o);
                sk += __shfl_xor_sync(0xffffffffu, sk, o);
            }
            if (c16 == 0) {
                sRq[r] = scale / sqrtf(sq + 1e-6f);
                sRk[r] = 1.0f / sqrtf(sk + 1e-6f);
            }
        }
        {
            const int d = tid & (D - 1), r0 = (tid >> 7) * 32;
            float x[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) x[i] = sG[(r0 + i) * D + d];
#pragma unroll
            for (int i = 1; i < 32; ++i) x[i] += x[i - 1];
            if (!r0) {
#pragma unroll
                for (int i = 0; i < 32; ++i) sG[i * D + d] = x[i];
            }
            __syncthreads();
            if (r0) {
                const float base = sG[31 * D + d];
#pragma unroll
                for (int i = 0; i < 32; ++i) sG[(r0 + i) * D + d] = x[i] + base;
            }
        }
        __syncthreads();
        // reference rows and block factors (threads 0..127: one key channel each)
        if (tid < D) {
            const int d = tid;
            float gb[4];
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                gb[b] = sG[16 * b * D + d];
                sGref[b * D + d] = gb[b];
                sRho[b * D + d] = __expf(gb[b]);
            }
            sGref[4 * D + d] = sG[(C - 1) * D + d];
#pragma unroll
            for (int br = 1; br < 4; ++br)
#pragma unroll
                for (int b = 0; b < br; ++b) sTau[tau_index(br, b) * D + d] = __expf(gb[br] - gb[b]);
            reinterpret_cast<float *>(rec + TcRec::GC)[d] = __expf(sG[(C - 1) * D + d]);
        }
        __syncthreads();

        KDA_PHASE(0, 2);
        // 2a. KD^T = (k_hat exp(G_last - G))^T, in 16-byte chunks of 8 chunk rows.
        for (int qi = tid; qi < 8 * D; qi += kPrepThreads) {
            const int c8 = qi >> 7, d = qi & (D - 1);
            const float gl = sGref[4 * D + d];
            float x[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const int r = 8 * c8 + t;
                x[t] = __bfloat162float(sKr[r * D + d]) * sRk[r] * __expf(gl - sG[r * D + d]);
            }
            *reinterpret_cast<uint4 *>(rec + TcRec::KDT + sw128_off(d, 8 * c8, 128)) = pack8(x);
        }
        __syncthreads();
        KDA_PHASE(0, 3);
        // 2b. per (row, 8 channels): QG, column factors, then G -> l in place.
        for (int qi = tid; qi < C * 16; qi += kPrepThreads) {
            const int r = qi >> 4, d0 = (qi & 15) * 8, br = r >> 4;
            float G8[8], Gb8[8], rho8[8], qv[8], kv[8];
            load8f(sG + r * D + d0, G8);
            load8f(sGref + br * D + d0, Gb8);
            load8f(sRho + br * D + d0, rho8);
            unpack8(*reinterpret_cast<const uint4 *>(sQr + r * D + d0), qv);
            unpack8(*reinterpret_cast<const uint4 *>(sKr + r * D + d0), kv);
            const float rq = sRq[r], rk = sRk[r];
            float qg[8], cf[8], l8[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                l8[t] = __expf(G8[t] - Gb8[t]);
                qg[t] = qv[t] * rq * l8[t] * rho8[t];
                cf[t] = kv[t] * rk * __expf(fminf(Gb8[t] - G8[t], 80.0f));
            }
            *reinterpret_cast<uint4 *>(rec + TcRec::WQ + sw128_off(64 + r, d0, 128)) = pack8(qg);
            *reinterpret_cast<uint4 *>(sC + br * 4096 + sw128_off(r & 15, d0, 16)) = pack8(cf);
            store8f(sG + r * D + d0, l8);
        }

        KDA_PHASE(0, 4);
        // 3. A and L: one M=128 x N=16 x K=128 MMA per 16-column block.
        for (int b = 0; b < 4; ++b) {
            __syncthreads();  // l complete (b = 0) / previous MMA done with Z (b > 0)
            for (int qi = tid; qi < C * 16; qi += kPrepThreads) {
                const int r = qi >> 4, d0 = (qi & 15) * 8, br = r >> 4;
                float qa[8], ka[8];
                if (r < 16 * b) {
#pragma unroll
                    for (int t = 0; t < 8; ++t) qa[t] = ka[t] = 0.0f;
                } else {
                    float l8[8], qv[8], kv[8];
                    load8f(sG + r * D + d0, l8);
                    if (br != b) {
                        float t8[8];
                        load8f(sTau + tau_index(br, b) * D + d0, t8);
#pragma unroll
                        for (int t = 0; t < 8; ++t) l8[t] *= t8[t];
                    }
                    unpack8(*reinterpret_cast<const uint4 *>(sQr + r * D + d0), qv);
                    unpack8(*reinterpret_cast<const uint4 *>(sKr + r * D + d0), kv);
                    const float rq = sRq[r], rk = sRk[r];
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        qa[t] = qv[t] * rq * l8[t];
                        ka[t] = kv[t] * rk * l8[t];
                    }
                }
                *reinterpret_cast<uint4 *>(sZ + sw128_off(r, d0, 128)) = pack8(qa);
                *reinterpret_cast<uint4 *>(sZ + sw128_off(64 + r, d0, 128)) = pack8(ka);
            }
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
            if (tid == 0) {
                tc_fence_after();
                mma_tile<128, 16, 128, 128, 16>(tmem + 16 * b, smem_u32(sZ), smem_u32(sC + b * 4096), false);
                mma_commit(mbar);
            }
            ok = mbar_wait(mbar, mphase) && ok;
            mphase ^= 1;
            tc_fence_after();
        }
        if (!__syncthreads_and(ok)) break;

        KDA_PHASE(0, 5);
        // 4. A rows (TMEM lanes 0..63) to the record; beta-scaled L rows
        //    (lanes 64..127) to shared fp32.
        {
            float *sL = reinterpret_cast<float *>(sZ);
            const int quarter = warp & 3, col0 = (warp >> 2) * 32;
            const int row = 32 * quarter + lane;
            float x[32];
            tmem_ld32(tmem + ((uint32_t)(32 * quarter) << 16) + col0, x);
            tmem_ld_wait();
            if (row < C) {
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    float y[8];
#pragma unroll
                    for (int t = 0; t < 8; ++t) y[t] = (col0 + 8 * c8 + t <= row) ? x[8 * c8 + t] : 0.0f;
                    *reinterpret_cast<uint4 *>(rec + TcRec::A + sw128_off(row, col0 + 8 * c8, 64)) = pack8(y);
                }
            } else {
                const int r = row - C;
                const float bet = sB[r];
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) {
                    float4 y;
                    const int j = col0 + 4 * c4;
                    y.x = (j + 0 < r) ? bet * x[4 * c4 + 0] : 0.0f;
                    y.y = (j + 1 < r) ? bet * x[4 * c4 + 1] : 0.0f;
                    y.z = (j + 2 < r) ? bet * x[4 * c4 + 2] : 0.0f;
                    y.w = (j + 3 < r) ? bet * x[4 * c4 + 3] : 0.0f;
                    *reinterpret_cast<float4 *>(sL + r * LSTRIDE + j) = y;
                }
            }
        }
        tc_fence_before();
        __syncthreads();

        KDA_PHASE(0, 6);
        // 5. X = (I + L)^-1, L strictly lower (beta-scaled rows), in 16x16 blocks:
        //    diagonal blocks X_bb = (I + N)^-1 = (I - N)(I + N^2)(I + N^4)(I + N^8)
        //    (N = L_bb is nilpotent); then with M = X_D L_off (strictly block
        //    lower, M^4 = 0): (I + L)^-1 = (I - M + M^2 - M^3) X_D.
        //    T = X diag(beta) -> bf16 operand at sC.
        {
            const float *sL = reinterpret_cast<const float *>(sZ);
            float *T1 = reinterpret_cast<float *>(sC);              // 4 blocks each (5 KB)
            float *T2 = T1 + 4 * MBLK;
            float *T3 = T2 + 4 * MBLK;
            float *T4 = reinterpret_cast<float *>(sZ) + 64 * LSTRIDE;  // after L in Z
            const int bb = tid >> 6, i = (tid & 63) >> 2, cg = tid & 3;
            const int o = 16 * bb;
            const float *N = sL + o * LSTRIDE + o;                   // L_bb, stride LSTRIDE
            auto put = [](float *M_, int i_, int cg_, float4 x) {
                *reinterpret_cast<float4 *>(M_ + i_ * MS + 4 * cg_) = x;
            };
            auto get = [](const float *M_, int i_, int cg_) {
                return *reinterpret_cast<const float4 *>(M_ + i_ * MS + 4 * cg_);
            };
            // P2 = N N  -> T1 ; N as a MS-stride copy -> T4 (for products with N on the right)
            {
                float4 nn;
                nn.x = N[i * LSTRIDE + 4 * cg + 0]; nn.y = N[i * LSTRIDE + 4 * cg + 1];
                nn.z = N[i * LSTRIDE + 4 * cg + 2]; nn.w = N[i * LSTRIDE + 4 * cg + 3];
                put(T4 + bb * MBLK, i, cg, nn);
            }
            __syncthreads();
            put(T1 + bb * MBLK, i, cg, mm16_row4(N, LSTRIDE, T4 + bb * MBLK, i, cg));
            __syncthreads();
            // P4 = P2 P2 -> T2 ;  Y1 = I - N + P2 - N P2 -> T3
            {
                const float4 p4 = mm16_row4(T1 + bb * MBLK, MS, T1 + bb * MBLK, i, cg);
                const float4 np2 = mm16_row4(N, LSTRIDE, T1 + bb * MBLK, i, cg);
                const float4 p2 = get(T1 + bb * MBLK, i, cg);
                const float4 n4 = get(T4 + bb * MBLK, i, cg);
                float4 y;
                y.x = (i == 4 * cg + 0 ? 1.f : 0.f) - n4.x + p2.x - np2.x;
                y.y = (i == 4 * cg + 1 ? 1.f : 0.f) - n4.y + p2.y - np2.y;
                y.z = (i == 4 * cg + 2 ? 1.f : 0.f) - n4.z + p2.z - np2.z;
                y.w = (i == 4 * cg + 3 ? 1.f : 0.f) - n4.w + p2.w - np2.w;
                put(T2 + bb * MBLK, i, cg, p4);
                put(T3 + bb * MBLK, i, cg, y);
            }
            __syncthreads();
            // P8 = P4 P4 -> T1 ;  Y2 = Y1 + Y1 P4 -> T4
            {
                const float4 p8 = mm16_row4(T2 + bb * MBLK, MS, T2 + bb * MBLK, i, cg);
                const float4 yp = mm16_row4(T3 + bb * MBLK, MS, T2 + bb * MBLK, i, cg);
                const float4 y1 = get(T3 + bb * MBLK, i, cg);
                put(T1 + bb * MBLK, i, cg, p8);
                put(T4 + bb * MBLK, i, cg, make_float4(y1.x + yp.x, y1.y + yp.y, y1.z + yp.z, y1.w + yp.w));
            }
            __syncthreads();
            // X_bb = Y2 + Y2 P8 -> sX diagonal block (stride 64) and T2 (stride MS)
            {
                const float4 yp = mm16_row4(T4 + bb * MBLK, MS, T1 + bb * MBLK, i, cg);
                const float4 y2 = get(T4 + bb * MBLK, i, cg);
                const float4 xd = make_float4(y2.x + yp.x, y2.y + yp.y, y2.z + yp.z, y2.w + yp.w);
                *reinterpret_cast<float4 *>(sX + (o + i) * C + o + 4 * cg) = xd;
                put(T2 + bb * MBLK, i, cg, xd);
            }
            __syncthreads();
            KDA_PHASE(0, 7);
            // Off-diagonal part.  Block pairs (a, b), a > b, indexed p = 0..5:
            // (1,0) (2,0) (2,1) (3,0) (3,1) (3,2).  X_D blocks are in T2 (stride MS).
            // Scratch: Z holds L in bytes [0, 17408) and the Y2 blocks in
            // [17408, 22528); M goes after them, [22528, 30208).
            const float *XD = T2;
            float *Mb = reinterpret_cast<float *>(sZ + 22528);  // M_ab = X_aa L_ab, 6 blocks
            float *M2 = T1;          // (M^2)_ab for (2,0) (3,1) (3,0)
            float *M3 = T3;          // (M^3)_30
            auto pair_a = [](int p) { return p < 1 ? 1 : (p < 3 ? 2 : 3); };
            auto pair_b = [](int p, int a) { return p - a * (a - 1) / 2; };
            for (int sl = tid; sl < 6 * 64; sl += kPrepThreads) {
                const int p = sl >> 6, ii = (sl & 63) >> 2, cc = sl & 3;
                const int a = pair_a(p), b = pair_b(p, a);
                // X_aa (stride MS) times L_ab (stride LSTRIDE, needs a MS copy of B):
                // compute directly: sum_k X_aa[ii][k] L[16a+k][16b + 4cc..]
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int kk = 0; kk < 16; ++kk) {
                    const float x = XD[a * MBLK + ii * MS + kk];
                    const float4 l = *reinterpret_cast<const float4 *>(sL + (16 * a + kk) * LSTRIDE + 16 * b + 4 * cc);
                    acc.x = fmaf(x, l.x, acc.x); acc.y = fmaf(x, l.y, acc.y);
                    acc.z = fmaf(x, l.z, acc.z); acc.w = fmaf(x, l.w, acc.w);
                }
                put(Mb + p * MBLK, ii, cc, acc);
            }
            __syncthreads();
            // M^2: (2,0) = M21 M10 ; (3,1) = M32 M21 ; (3,0) = M31 M10 + M32 M20
            for (int sl = tid; sl < 3 * 64; sl += kPrepThreads) {
                const int p = sl >> 6, ii = (sl & 63) >> 2, cc = sl & 3;
                float4 acc;
                if (p == 0) acc = mm16_row4(Mb + 2 * MBLK, MS, Mb + 0 * MBLK, ii, cc);
                else if (p == 1) acc = mm16_row4(Mb + 5 * MBLK, MS, Mb + 2 * MBLK, ii, cc);
                else {
                    const float4 a1 = mm16_row4(Mb + 4 * MBLK, MS, Mb + 0 * MBLK, ii, cc);
                    const float4 a2 = mm16_row4(Mb + 5 * MBLK, MS, Mb + 1 * MBLK, ii, cc);
                    acc = make_float4(a1.x + a2.x, a1.y + a2.y, a1.z + a2.z, a1.w + a2.w);
                }
                put(M2 + p * MBLK, ii, cc, acc);
            }
            __syncthreads();
            // M^3: (3,0) = M32 (M^2)_20
            if (tid < 64) put(M3, (tid & 63) >> 2, tid & 3, mm16_row4(Mb + 5 * MBLK, MS, M2 + 0 * MBLK, (tid & 63) >> 2, tid & 3));
            __syncthreads();
            // X_ab = (-M + M^2 - M^3)_ab X_bb
            for (int sl = tid; sl < 6 * 64; sl += kPrepThreads) {
                const int p = sl >> 6, ii = (sl & 63) >> 2, cc = sl & 3;
                const int a = pair_a(p), b = pair_b(p, a);
                const int p2 = (p == 1) ? 0 : (p == 4) ? 1 : (p == 3) ? 2 : -1;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int kk = 0; kk < 16; ++kk) {
                    float z = -Mb[p * MBLK + ii * MS + kk];
                    if (p2 >= 0) z += M2[p2 * MBLK + ii * MS + kk];
                    if (p == 3) z -= M3[ii * MS + kk];
                    const float4 xb = *reinterpret_cast<const float4 *>(XD + b * MBLK + kk * MS + 4 * cc);
                    acc.x = fmaf(z, xb.x, acc.x); acc.y = fmaf(z, xb.y, acc.y);
                    acc.z = fmaf(z, xb.z, acc.z); acc.w = fmaf(z, xb.w, acc.w);
                }
                *reinterpret_cast<float4 *>(sX + (16 * a + ii) * C + 16 * b + 4 * cc) = acc;
            }
            __syncthreads();
            // T = X diag(beta), lower triangle, as a K-major [i][j] bf16 operand
            for (int qi = tid; qi < C * 8; qi += kPrepThreads) {
                const int ri = qi >> 3, j0 = (qi & 7) * 8;
                float y[8];
#pragma unroll
                for (int t = 0; t < 8; ++t) y[t] = (j0 + t <= ri) ? sX[ri * C + j0 + t] * sB[j0 + t] : 0.0f;
                *reinterpret_cast<uint4 *>(sC + sw128_off(ri, j0, 64)) = pack8(y);
            }
        }
        __syncthreads();

        KDA_PHASE(0, 8);
        // 6. E^T = (exp(G) k_hat)^T and V^T operands in Z; W = T E, U = T V.
        for (int qi = tid; qi < 8 * D; qi += kPrepThreads) {
            const int c8 = qi >> 7, d = qi & (D - 1);
            const float rho = sRho[(c8 >> 1) * D + d];
            float e[8], vv[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const int j = 8 * c8 + t;
                e[t] = __bfloat162float(sKr[j * D + d]) * sRk[j] * sG[j * D + d] * rho;
                vv[t] = __bfloat162float(sVr[j * D + d]);
            }
            *reinterpret_cast<uint4 *>(sZ + sw128_off(d, 8 * c8, 128)) = pack8(e);
            *reinterpret_cast<uint4 *>(sZ + 16384 + sw128_off(d, 8 * c8, 128)) = pack8(vv);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            mma_tile<128, 128, 64, 128, 128>(tmem + 0, smem_u32(sC), smem_u32(sZ), false);
            mma_tile<128, 128, 64, 128, 128>(tmem + 128, smem_u32(sC), smem_u32(sZ + 16384), false);
            mma_commit(mbar);
        }
        ok = mbar_wait(mbar, mphase) && ok;
        mphase ^= 1;
        tc_fence_after();
        if (!__syncthreads_and(ok)) break;

        KDA_PHASE(0, 9);
        // 7. W rows (WQ rows 0..63) and U to the record: TMEM lanes 0..63.
        if ((warp & 3) < 2) {
            const int i = 32 * (warp & 3) + lane, half = warp >> 2;
            const uint32_t ta = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                float x[32];
                const int c0 = 64 * half + 32 * part;
                tmem_ld32(ta + c0, x);
                tmem_ld_wait();
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    float y[8];
#pragma unroll
                    for (int t = 0; t < 8; ++t) y[t] = x[8 * c8 + t];
                    *reinterpret_cast<uint4 *>(rec + TcRec::WQ + sw128_off(i, c0 + 8 * c8, 128)) = pack8(y);
                }
                tmem_ld32(ta + 128 + c0, x);
                tmem_ld_wait();
                unsigned char *ub = rec + TcRec::U + (c0 >> 5) * TcRec::UBLK + i * 64;
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    float y[8];
#pragma unroll
                    for (int t = 0; t < 8; ++t) y[t] = x[8 * c8 + t];
                    *reinterpret_cast<uint4 *>(ub + 16 * c8) = pack8(y);
                }
            }
        }
        tc_fence_before();
        __syncthreads();
        KDA_PHASE(0, 10);
    }
    if (!ok) {
        if (tid == 0) {
            atomicOr(status, kStatusTimeout);
            // let copies still in flight land before the shared memory is released
            mbar_wait(&full[0], 0, 400000000LL) || mbar_wait(&full[0], 1, 400000000LL);
            mbar_wait(&full[1], 0, 400000000LL) || mbar_wait(&full[1], 1, 400000000LL);
        }
        __syncthreads();
    }
    if (warp == 0) tmem_dealloc(tmem, kPrepTmemCols);
}

// ---------------------------------------------------------------------------
// scan
// ---------------------------------------------------------------------------
constexpr int kScanThreads = 128;
constexpr int BV = 32;
constexpr uint32_t kScanTmemCols = 64;
constexpr int kStages = 3;
constexpr uint32_t kImageBytes = TcRec::U;                   // WQ | KDT | A | gC
constexpr uint32_t kStageBytes = kImageBytes + TcRec::UBLK;  // + this CTA's U block
constexpr int S_STAGE = 62464;                               // kStageBytes rounded up to 1024
constexpr int S_SOP = kStages * S_STAGE;                     // S^T operand [32][128] bf16, 8 KB
constexpr int S_VOP = S_SOP + 8192;                          // Vn^T operand [32][64] bf16, 4 KB
constexpr int S_BAR = S_VOP + 4096;                          // full[kStages], mma
constexpr int S_BYTES = S_BAR + 64;
constexpr int S_SMEM = S_BYTES + 1024;
static_assert(kStageBytes <= (uint32_t)S_STAGE, "stage too small");
static_assert(kImageBytes % 16 == 0 && TcRec::UBLK % 16 == 0, "bulk copy size");

// Write this thread's 32 values x[v] as column `col` of a K-major SW128 bf16
// operand with 32 rows: neighbouring lanes (col even / odd) swap one value so
// that each 32-bit store holds two adjacent columns of one row.  Whole warps.
__device__ __forceinline__ void store_col_pairs(unsigned char *op, int col, const float (&x)[32]) {
    const int odd = col & 1;
    const int ce = col & ~1;
    const int kk = ce & 63;
    // element (row, ce) of the 32-row tile sits at
    //   (ce / 64) * 4096 + row * 128 + (((kk / 8) ^ (row % 8)) * 16) + (kk % 8) * 2;
    // for row = 2m + odd, (row % 8) = ((2m) % 8) | odd, hence the hoisted terms
    unsigned char *base = op + (ce >> 6) * 4096 + odd * 128 + ((kk & 7) << 1);
    const int cx = (kk >> 3) ^ odd;
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        const float send = odd ? x[2 * m] : x[2 * m + 1];
        const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
        const float lo = odd ? recv : x[2 * m];
        const float hi = odd ? x[2 * m + 1] : recv;
        *reinterpret_cast<uint32_t *>(base + 256 * m + ((cx ^ ((2 * m) & 7)) << 4)) = pack2(lo, hi);
    }
}

__global__ void __launch_bounds__(kScanThreads, 1)
    chunk_scan_tc_kernel(const float *__restrict__ initial_state, float *__restrict__ final_state,
                         const int32_t *__restrict__ state_indices, __nv_bfloat16 *__restrict__ o,
                         int n_seqs, int H, void *workspace, WsLayout L) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    unsigned char *sS = sm + S_SOP;
    unsigned char *sVn = sm + S_VOP;
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + S_BAR);
    uint64_t *mbar = full + kStages;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mbar + 1);

    const int n = blockIdx.x, h = blockIdx.y, vb = blockIdx.z, v0 = vb * BV;
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
    auto issue = [&](int ck) {  // thread 32 (not the MMA-issuing thread)
        const int s = ck % kStages;
        unsigned char *dst = sm + s * S_STAGE;
        mbar_arrive_expect_tx(&full[s], kStageBytes);
        bulk_g2s(dst, rec_of(ck), kImageBytes, &full[s]);
        bulk_g2s(dst + kImageBytes, rec_of(ck) + TcRec::U + vb * TcRec::UBLK, TcRec::UBLK, &full[s]);
    };

    if (warp == 0) tmem_alloc(tmem_slot, kScanTmemCols);
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
        mbar_init(mbar, 1);
        fence_mbar_init();
    }
    // state row d = tid, columns v0 .. v0+31, fp32 in registers
    float S[BV];
#pragma unroll
    for (int x = 0; x < BV; ++x)
        S[x] = initial_state ? initial_state[st_off + (int64_t)(v0 + x) * D + tid] : 0.0f;
    store_col_pairs(sS, tid, S);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tD1 = tmem, tD3 = tmem + 32;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;

    if (tid == 32) {
        for (int ck = 0; ck < kStages - 1 && ck < nck; ++ck) issue(ck);
    }
    uint32_t mphase = 0;
    bool ok = true;
    KDA_PHASE_START();
    for (int ck = 0; ck < nck; ++ck) {
        const int stage = ck % kStages;
        unsigned char *st = sm + stage * S_STAGE;
        if (tid == 32 && ck + kStages - 1 < nck) issue(ck + kStages - 1);  // its stage was freed by ck-1
        const int valid = min(C, len - ck * C);
        const int64_t tok0 = (int64_t)start + (int64_t)ck * C;
        KDA_PHASE(1, 0);
        ok = mbar_wait(&full[stage], (uint32_t)((ck / kStages) & 1)) && ok;
        if (!__syncthreads_and(ok)) break;
        KDA_PHASE(1, 1);

        // D1 = WQ * S
        if (tid == 0) {
            tc_fence_after();
            mma_tile<128, BV, 128, 128, BV>(tD1, smem_u32(st + TcRec::WQ), smem_u32(sS), false);
            mma_commit(mbar);
        }
        KDA_PHASE(1, 2);
        ok = mbar_wait(mbar, mphase) && ok;
        mphase ^= 1;
        tc_fence_after();
        KDA_PHASE(1, 3);
        if (warp < 2) {  // rows 0..63: Vn = U - W S
            float x[32], u[32];
            tmem_ld32(tD1 + lane_base, x);
            const uint4 *up = reinterpret_cast<const uint4 *>(st + kImageBytes + tid * 64);
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
                float y[8];
                unpack8(up[c8], y);
#pragma unroll
                for (int t = 0; t < 8; ++t) u[8 * c8 + t] = y[t];
            }
            tmem_ld_wait();
#pragma unroll
            for (int vv = 0; vv < BV; ++vv) x[vv] = u[vv] - x[vv];
            store_col_pairs(sVn, tid, x);
        }
        KDA_PHASE(1, 4);
        fence_async_smem();
        tc_fence_before();
        if (!__syncthreads_and(ok)) break;
        KDA_PHASE(1, 5);

        // D1 += [* ; A] * Vn ;  D3 = KD^T * Vn
        if (tid == 0) {
            tc_fence_after();
            mma_tile<128, BV, 64, 128, BV>(tD1, smem_u32(st + TcRec::A) - 8192, smem_u32(sVn), true);
            mma_tile<128, BV, 64, 128, BV>(tD3, smem_u32(st + TcRec::KDT), smem_u32(sVn), false);
            mma_commit(mbar);
        }
        KDA_PHASE(1, 6);
        ok = mbar_wait(mbar, mphase) && ok;
        mphase ^= 1;
        tc_fence_after();
        KDA_PHASE(1, 7);
        if (warp >= 2) {  // rows 64..127: o
            float x[32];
            tmem_ld32(tD1 + lane_base, x);
            tmem_ld_wait();
            const int r = tid - 64;
            if (r < valid) {
                uint4 *op = reinterpret_cast<uint4 *>(o + ((tok0 + r) * H + h) * (int64_t)D + v0);
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    float y[8];
#pragma unroll
                    for (int t = 0; t < 8; ++t) y[t] = x[8 * c8 + t];
                    op[c8] = pack8(y);
                }
            }
        }
        {  // S = diag(gC) S + KD^T Vn
            float x[32];
            tmem_ld32(tD3 + lane_base, x);
            const float gc = reinterpret_cast<const float *>(st + TcRec::GC)[tid];
            tmem_ld_wait();
#pragma unroll
            for (int vv = 0; vv < BV; ++vv) S[vv] = fmaf(gc, S[vv], x[vv]);
            store_col_pairs(sS, tid, S);
        }
        KDA_PHASE(1, 8);
        fence_async_smem();
        tc_fence_before();
        if (!__syncthreads_and(ok)) break;
        KDA_PHASE(1, 9);
    }
    if (!ok) {
        if (tid == 32) {
            atomicOr(status, kStatusTimeout);
            // let copies still in flight land before the shared memory is released
            for (int s = 0; s < kStages; ++s)
                mbar_wait(&full[s], 0, 400000000LL) || mbar_wait(&full[s], 1, 400000000LL);
        }
    } else if (final_state) {
#pragma unroll
        for (int x = 0; x < BV; ++x) final_state[st_off + (int64_t)(v0 + x) * D + tid] = S[x];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kScanTmemCols);
}

int sm_count() {
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

}  // namespace

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
        cudaGetLastError();
    });
    return fn;
}

// 3-D map {128, H, T} over a [T, H, 128] tensor; box 128 x 1 x 64.
bool encode_rows(CUtensorMap *m, const void *base, CUtensorMapDataType dt, size_t elem, int H,
                 int64_t T) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t strides[2] = {(cuuint64_t)(D * elem), (cuuint64_t)(D * elem) * (cuuint64_t)H};
    const cuuint32_t box[3] = {(cuuint32_t)D, 1, (cuuint32_t)C};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_chunk_prep_tc(const void *q, const void *k, const void *v, const float *g,
                                 const float *beta, int n_seqs, int64_t total_tokens, int H,
                                 float scale, void *workspace, cudaStream_t stream) {
    const WsLayout L = ws_layout(total_tokens, n_seqs, H, TcRec::bytes);
    const int64_t items_max = max_chunks(total_tokens, n_seqs) * (int64_t)H;
    const int grid = (int)std::min<int64_t>(items_max, (int64_t)sm_count());
    RawMaps maps;
    memset(&maps, 0, sizeof(maps));
    if (total_tokens > 0) {
        if (!encode_rows(&maps.q, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, total_tokens) ||
            !encode_rows(&maps.k, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, total_tokens) ||
            !encode_rows(&maps.v, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, total_tokens) ||
            !encode_rows(&maps.g, g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, H, total_tokens))
            return cudaErrorInvalidValue;
    }
    cudaFuncSetAttribute(chunk_prep_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM);
    chunk_prep_tc_kernel<<<grid, kPrepThreads, P_SMEM, stream>>>(maps, beta, n_seqs, H, scale,
                                                                  workspace, L);
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

#ifdef KDA_PHASE_TRACE
extern "C" int kda_phase_read(unsigned long long *out) {
    return (int)cudaMemcpyFromSymbol(out, kda_phase_cycles, sizeof(unsigned long long) * 64);
}
extern "C" int kda_phase_reset() {
    unsigned long long z[64] = {0};
    return (int)cudaMemcpyToSymbol(kda_phase_cycles, z, sizeof(z));
}
#endif
